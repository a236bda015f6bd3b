// Per-call bf16 split of the cores read by the tensor-core chunk kernels:
// G1 and G2 become two bf16 planes each, hi = bf16(x) and lo = bf16(x - hi),
// in the cores' own layouts ([m1][n1][R1] and [m2][R1][n2 R2]), so that the
// chunk kernels stage them with plain copies and load ldmatrix fragments with
// no per-use conversion (the three-term products of tt_mma.cuh).
#include "tt_internal.cuh"
#include "tt_mma.cuh"

namespace tt {

__global__ void __launch_bounds__(256) k_split_cores(const float4* __restrict__ g1, int64_t n1,
                                                     const float4* __restrict__ g2, int64_t n2,
                                                     uint2* __restrict__ g1h, uint2* __restrict__ g1l,
                                                     uint2* __restrict__ g2h, uint2* __restrict__ g2l) {
  const int64_t total = n1 + n2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const bool first = i < n1;
    const int64_t j = first ? i : i - n1;
    const float4 v = first ? __ldg(g1 + j) : __ldg(g2 + j);
    uint32_t h0, l0, h1, l1;
    split_bf16x2(v.x, v.y, h0, l0);
    split_bf16x2(v.z, v.w, h1, l1);
    (first ? g1h : g2h)[j] = make_uint2(h0, h1);
    (first ? g1l : g2l)[j] = make_uint2(l0, l1);
  }
}

int launch_split(const Shape& s, const WS& w, const float* const cores[3], cudaStream_t st) {
  if (!w.g2l) return TT_EMB_OK;
  const int64_t n1 = s.m1 * s.n1 * s.R1 / 4, n2 = s.m2 * s.R1 * s.n2 * s.R2 / 4;
  int grid = (int)ceil_div(n1 + n2, 256);
  if (grid > sm_count() * 8) grid = sm_count() * 8;
  TT_TIMED("k_split", st, (k_split_cores<<<grid, 256, 0, st>>>(
                              reinterpret_cast<const float4*>(cores[0]), n1,
                              reinterpret_cast<const float4*>(cores[1]), n2,
                              reinterpret_cast<uint2*>(w.g1h), reinterpret_cast<uint2*>(w.g1l),
                              reinterpret_cast<uint2*>(w.g2h), reinterpret_cast<uint2*>(w.g2l))));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
