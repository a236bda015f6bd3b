// Per-call bf16 split of the cores read by the tensor-core chunk kernels:
// G1, G2 and G3 become two bf16 planes each, hi = bf16(x) and lo = bf16(x - hi),
// in the cores' own layouts ([m1][n1][R1], [m2][R1][n2 R2], [m3][R2][n3]), and G3
// also transposed per i3 ([m3][n3][R2]), so that the chunk kernels stage them
// with plain copies and load fragments with no per-use conversion (the
// three-term products of tt_mma.cuh).
#include "tt_internal.cuh"
#include "tt_mma.cuh"

namespace tt {

// With `reuse` set, the launch returns at once when the planes already hold
// these cores: the control block records the source addresses of the last
// completed split (written by the chunk kernel that runs after it, so that no
// block of this launch can see a record that this launch has not finished),
// and every grouping run clears that record.
__global__ void __launch_bounds__(256) k_split_cores(const float4* __restrict__ g1, int64_t n1,
                                                     const float4* __restrict__ g2, int64_t n2,
                                                     uint2* __restrict__ g1h, uint2* __restrict__ g1l,
                                                     uint2* __restrict__ g2h, uint2* __restrict__ g2l,
                                                     const float* __restrict__ g3, int64_t g3_count,
                                                     int R2, int N3, uint16_t* __restrict__ g3h,
                                                     uint16_t* __restrict__ g3l, uint16_t* __restrict__ g3th,
                                                     uint16_t* __restrict__ g3tl, Ctl* ctl, int reuse) {
  if (reuse && ctl->split_valid && ctl->split_src[0] == (unsigned long long)g1 &&
      ctl->split_src[1] == (unsigned long long)g2 && ctl->split_src[2] == (unsigned long long)g3)
    return;
  // G3 (small): element-wise, natural and transposed planes
  {
    const int64_t n3 = g3_count;
    const int64_t stride3 = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n3; e += stride3) {
      const float x = __ldg(g3 + e);
      const __nv_bfloat16 h = __float2bfloat16_rn(x);
      const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
      g3h[e] = *reinterpret_cast<const uint16_t*>(&h);
      g3l[e] = *reinterpret_cast<const uint16_t*>(&l);
      // e = (i3 R2 + r2) n3 + j3  ->  (i3 n3 + j3) R2 + r2
      const int64_t i3 = e / (R2 * N3), rem = e - i3 * (R2 * N3);
      const int64_t r2 = rem / N3, j3 = rem - r2 * N3;
      const int64_t t = (i3 * N3 + j3) * R2 + r2;
      g3th[t] = *reinterpret_cast<const uint16_t*>(&h);
      g3tl[t] = *reinterpret_cast<const uint16_t*>(&l);
    }
  }
  // G1 and G2: grid-stride, four independent 16-byte loads per thread and step
  const int64_t total = n1 + n2;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total) v[u] = i < n1 ? __ldg(g1 + i) : __ldg(g2 + (i - n1));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total) {
        uint32_t h0, l0, h1, l1;
        split_bf16x2(v[u].x, v[u].y, h0, l0);
        split_bf16x2(v[u].z, v[u].w, h1, l1);
        const bool first = i < n1;
        const int64_t j = first ? i : i - n1;
        (first ? g1h : g2h)[j] = make_uint2(h0, h1);
        (first ? g1l : g2l)[j] = make_uint2(l0, l1);
      }
    }
  }
}

int launch_split(const Shape& s, const WS& w, const float* const cores[3], int reuse, cudaStream_t st) {
  if (!w.g2l) return TT_EMB_OK;
  const int64_t n1 = s.m1 * s.n1 * s.R1 / 4, n2 = s.m2 * s.R1 * s.n2 * s.R2 / 4;
  int grid = (int)ceil_div(n1 + n2, 4 * 256);
  if (grid > sm_count() * 2) grid = sm_count() * 2;
  if (grid < 1) grid = 1;
  TT_TIMED("k_split", st, (k_split_cores<<<grid, 256, 0, st>>>(
                              reinterpret_cast<const float4*>(cores[0]), n1,
                              reinterpret_cast<const float4*>(cores[1]), n2,
                              reinterpret_cast<uint2*>(w.g1h), reinterpret_cast<uint2*>(w.g1l),
                              reinterpret_cast<uint2*>(w.g2h), reinterpret_cast<uint2*>(w.g2l),
                              cores[2], s.m3 * s.R2 * s.n3, s.R2, s.n3, w.g3h, w.g3l, w.g3th, w.g3tl,
                              w.ctl, reuse)));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
