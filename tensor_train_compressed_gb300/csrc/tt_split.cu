// Per-call bf16 split of the cores read by the tensor-core chunk kernels
// (three-term products of tt_mma.cuh): the split launch of the forward.
#include "tt_split.cuh"

namespace tt {

// With `reuse` set, the launch returns at once when the planes already hold
// these cores (the record is cleared by every grouping run).
__global__ void __launch_bounds__(256) k_split_cores(SplitArgs a, Ctl* ctl, int reuse) {
  if (reuse && split_current(a, ctl)) return;
  split_cores_body(a);
}

SplitArgs make_split_args(const Shape& s, const WS& w, const float* const cores[3]) {
  SplitArgs a;
  a.g1 = reinterpret_cast<const float4*>(cores[0]);
  a.n1 = s.m1 * s.n1 * s.R1 / 4;
  a.g2 = reinterpret_cast<const float4*>(cores[1]);
  a.n2 = s.m2 * s.R1 * s.n2 * s.R2 / 4;
  a.g1h = reinterpret_cast<uint2*>(w.g1h);
  a.g1l = reinterpret_cast<uint2*>(w.g1l);
  a.g2h = reinterpret_cast<uint2*>(w.g2h);
  a.g2l = reinterpret_cast<uint2*>(w.g2l);
  a.g3 = cores[2];
  a.g3_count = s.m3 * s.R2 * s.n3;
  a.R2 = s.R2;
  a.N3 = s.n3;
  a.g3h = w.g3h;
  a.g3l = w.g3l;
  a.g3th = w.g3th;
  a.g3tl = w.g3tl;
  return a;
}

// One pass of four float4 per thread over G1 and G2, at most 8 CTAs per SM.
int split_grid(const SplitArgs& a) {
  if (!a.g2l) return 0;
  int64_t grid = ceil_div(a.n1 + a.n2, 4 * 256);
  const int64_t g3 = ceil_div(a.g3_count, 256);
  if (grid < g3) grid = g3;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (grid > cap) grid = cap;
  return grid < 1 ? 1 : (int)grid;
}

int launch_split(const Shape& s, const WS& w, const float* const cores[3], int reuse, cudaStream_t st) {
  if (!w.g2l) return TT_EMB_OK;
  const SplitArgs a = make_split_args(s, w, cores);
  TT_TIMED("k_split", st, (k_split_cores<<<split_grid(a), 256, 0, st>>>(a, w.ctl, reuse)));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
