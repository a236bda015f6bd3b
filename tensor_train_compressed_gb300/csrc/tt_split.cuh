// bf16 split of the cores read by the tensor-core chunk kernels (device part,
// shared by the split launch of the forward and the backward's preparation
// kernel): G1, G2 and G3 become two bf16 planes each, hi = bf16(x) and
// lo = bf16(x - hi), in the cores' own layouts ([m1][n1][R1], [m2][R1][n2 R2],
// [m3][R2][n3]), and G3 also transposed per i3 ([m3][n3][R2]).
#pragma once
#include "tt_internal.cuh"
#include "tt_mma.cuh"

namespace tt {

struct SplitArgs {
  const float4* g1;
  int64_t n1;             // float4 of G1
  const float4* g2;
  int64_t n2;             // float4 of G2
  uint2 *g1h, *g1l, *g2h, *g2l;
  const float* g3;
  int64_t g3_count;       // floats of G3
  int R2, N3;
  uint16_t *g3h, *g3l, *g3th, *g3tl;   // null: the shape has no split planes
};

// True when the planes already hold these cores: the control block records the
// source addresses of the last completed split (written by a chunk kernel that
// runs after it, so that no block of a splitting launch can see a record that
// the launch has not finished).
__device__ __forceinline__ bool split_current(const SplitArgs& a, const Ctl* ctl) {
  return ctl->split_valid && ctl->split_src[0] == (unsigned long long)a.g1 &&
         ctl->split_src[1] == (unsigned long long)a.g2 &&
         ctl->split_src[2] == (unsigned long long)a.g3;
}

// Grid-stride split over all threads of the launch.
__device__ __forceinline__ void split_cores_body(const SplitArgs& a) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // G3 (small): element-wise, natural and transposed planes
  for (int64_t e = t0; e < a.g3_count; e += stride) {
    const float x = __ldg(a.g3 + e);
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
    a.g3h[e] = *reinterpret_cast<const uint16_t*>(&h);
    a.g3l[e] = *reinterpret_cast<const uint16_t*>(&l);
    // e = (i3 R2 + r2) n3 + j3  ->  (i3 n3 + j3) R2 + r2
    const int64_t i3 = e / (a.R2 * a.N3), rem = e - i3 * (a.R2 * a.N3);
    const int64_t r2 = rem / a.N3, j3 = rem - r2 * a.N3;
    const int64_t t = (i3 * a.N3 + j3) * a.R2 + r2;
    a.g3th[t] = *reinterpret_cast<const uint16_t*>(&h);
    a.g3tl[t] = *reinterpret_cast<const uint16_t*>(&l);
  }
  // G1 and G2: four independent 16-byte loads per thread and step
  const int64_t total = a.n1 + a.n2;
  for (int64_t i0 = t0; i0 < total; i0 += 4 * stride) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total) v[u] = i < a.n1 ? __ldg(a.g1 + i) : __ldg(a.g2 + (i - a.n1));
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      if (i < total) {
        uint32_t h0, l0, h1, l1;
        split_bf16x2(v[u].x, v[u].y, h0, l0);
        split_bf16x2(v[u].z, v[u].w, h1, l1);
        const bool first = i < a.n1;
        const int64_t j = first ? i : i - a.n1;
        (first ? a.g1h : a.g2h)[j] = make_uint2(h0, h1);
        (first ? a.g1l : a.g2l)[j] = make_uint2(l0, l1);
      }
    }
  }
}

SplitArgs make_split_args(const Shape& s, const WS& w, const float* const cores[3]);
// CTAs of 256 threads that a split of this shape wants (0 without split planes)
int split_grid(const SplitArgs& a);

}  // namespace tt
