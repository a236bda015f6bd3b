// Warp-level tensor-core tiles for the fp32 contractions of the chunk kernels.
//
// Every contraction of the TT chain in a work chunk is a small dense GEMM
// (prefix partials: (4 np) x (n2 R2) x R1; rows: (n1 n2) x (2 n3) x R2 per pair
// of rows of one prefix).  They run as m16n8k8 TF32 tensor-core tiles
// (mma.sync, fp32 accumulate) with each fp32 operand split into two TF32
// terms, x = hi + lo with hi = x rounded to TF32 (10 explicit mantissa bits)
// and lo = x - hi (exact in fp32).  The product is taken as
//   a.b ~ a_lo.b_hi + a_hi.b_lo + a_hi.b_hi,
// dropping only a_lo.b_lo (relative size 2^-22) and the truncation of lo to
// TF32 by the tensor core (2^-21), so each product keeps fp32-level accuracy
// while the tensor pipe does the multiply-adds (about four times the FP32
// FMA rate per SM, measured) and the FMA issue slots stay free.
//
// Fragment layout of mma.m16n8k8 (row.col, tf32), g = lane / 4, t = lane % 4:
//   A (16 x 8):  a0 = A[g][t], a1 = A[g+8][t], a2 = A[g][t+4], a3 = A[g+8][t+4]
//   B (8 x 8):   b0 = B[t][g], b1 = B[t+4][g]
//   C (16 x 8):  c0 = C[g][2t], c1 = C[g][2t+1], c2 = C[g+8][2t], c3 = C[g+8][2t+1]
#pragma once

#include <cstdint>

namespace tt {

struct Tf32x2 {
  uint32_t hi, lo;
};

__device__ __forceinline__ Tf32x2 split_tf32(float x) {
  uint32_t h;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(h) : "f"(x));
  Tf32x2 r;
  r.hi = h;
  r.lo = __float_as_uint(x - __uint_as_float(h));
  return r;
}

__device__ __forceinline__ void mma_tf32(float c[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// A fragment (16 x 8) of one k-step, split.
struct FragA {
  Tf32x2 v[4];
};
// B fragment (8 x 8) of one k-step, split.
struct FragB {
  Tf32x2 v[2];
};

// A[m][k] at A[m * lda + k] for rows m < 8 and at A[off8 + (m - 8) * lda + k]
// for rows 8 .. 15; columns k0 .. k0+7.
__device__ __forceinline__ FragA load_a(const float* A, int lda, int off8, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const float* r0 = A + g * lda + t;
  const float* r8 = A + off8 + g * lda + t;
  FragA f;
  f.v[0] = split_tf32(r0[0]);
  f.v[1] = split_tf32(r8[0]);
  f.v[2] = split_tf32(r0[4]);
  f.v[3] = split_tf32(r8[4]);
  return f;
}
// B[k][n] at B[k * ldb + n]; rows k0 .. k0+7, columns n0 .. n0+7.
__device__ __forceinline__ FragB load_b(const float* B, int ldb, int lane) {
  const int g = lane >> 2, t = lane & 3;
  FragB f;
  f.v[0] = split_tf32(B[t * ldb + g]);
  f.v[1] = split_tf32(B[(t + 4) * ldb + g]);
  return f;
}

// A[m][k] at A[m + k * ldk] (column-major), rows 0 .. 15, columns 0 .. 7.
__device__ __forceinline__ FragA load_a_cm(const float* A, int ldk, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const float* c0 = A + g + t * ldk;
  const float* c4 = A + g + (t + 4) * ldk;
  FragA f;
  f.v[0] = split_tf32(c0[0]);
  f.v[1] = split_tf32(c0[8]);
  f.v[2] = split_tf32(c4[0]);
  f.v[3] = split_tf32(c4[8]);
  return f;
}

// c += a.b with the three-term split (small terms first).
__device__ __forceinline__ void mma_3xtf32(float c[4], const FragA& a, const FragB& b) {
  mma_tf32(c, a.v[0].lo, a.v[1].lo, a.v[2].lo, a.v[3].lo, b.v[0].hi, b.v[1].hi);
  mma_tf32(c, a.v[0].hi, a.v[1].hi, a.v[2].hi, a.v[3].hi, b.v[0].lo, b.v[1].lo);
  mma_tf32(c, a.v[0].hi, a.v[1].hi, a.v[2].hi, a.v[3].hi, b.v[0].hi, b.v[1].hi);
}

// Same product with the hi.hi term and the two small terms in separate
// accumulators (two independent dependency chains).
__device__ __forceinline__ void mma_3xtf32_2(float big[4], float small[4], const FragA& a,
                                             const FragB& b) {
  mma_tf32(small, a.v[0].lo, a.v[1].lo, a.v[2].lo, a.v[3].lo, b.v[0].hi, b.v[1].hi);
  mma_tf32(big, a.v[0].hi, a.v[1].hi, a.v[2].hi, a.v[3].hi, b.v[0].hi, b.v[1].hi);
  mma_tf32(small, a.v[0].hi, a.v[1].hi, a.v[2].hi, a.v[3].hi, b.v[0].lo, b.v[1].lo);
}

// Float pair atomically added to global memory (no return value).
__device__ __forceinline__ void red_add_f2(float* p, float x, float y) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(x), "f"(y) : "memory");
}

}  // namespace tt
