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
#include <cuda_bf16.h>

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

// ---------------------------------------------------------------------------
// bf16 three-term tiles for the prefix-level products.  Operands are stored as
// two bf16 planes, hi = x rounded to bf16 and lo = (x - hi) rounded to bf16
// (|x - hi - lo| <= 2^-18 |x|), and multiplied as a_lo.b_hi + a_hi.b_lo +
// a_hi.b_hi with mma.m16n8k16 (fp32 accumulate): relative error about 1e-5
// per product against fp32's 6e-8, at twice the multiply-adds per tensor
// instruction of TF32 and with no per-use splitting.  Fragments come straight
// from shared memory by ldmatrix (8 x 8 b16 matrices, one 16-byte row address
// per lane), with .trans for an operand stored along the other axis, so one
// plane layout serves both products that read it.  Rows of every plane are
// padded to an odd multiple of 16 bytes (conflict-free ldmatrix).

__device__ __forceinline__ void ldsm_x4(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t r[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t r[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t r[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}

// Byte address of this lane's row for the 16 x 16 A fragment (rows m0.., k0..):
// of a [m][k] plane (plain load) or a [k][m] plane (transposed load); ld in
// bf16 elements, base a shared-memory byte address.
__device__ __forceinline__ uint32_t a_addr_mk(uint32_t base, int ld, int m0, int k0, int lane) {
  const int i = lane >> 3, r = lane & 7;
  return base + 2u * (uint32_t)((m0 + 8 * (i & 1) + r) * ld + k0 + 8 * (i >> 1));
}
__device__ __forceinline__ uint32_t a_addr_km(uint32_t base, int ld, int m0, int k0, int lane) {
  const int i = lane >> 3, r = lane & 7;
  return base + 2u * (uint32_t)((k0 + 8 * (i >> 1) + r) * ld + m0 + 8 * (i & 1));
}
// B fragments of the two n-tiles n0.., n0+8.. (k0 .. k0+15): regs {0,1} and {2,3};
// of a [k][n] plane (transposed load) or a [n][k] plane (plain load).
__device__ __forceinline__ uint32_t b2_addr_kn(uint32_t base, int ld, int k0, int n0, int lane) {
  const int i = lane >> 3, r = lane & 7;
  return base + 2u * (uint32_t)((k0 + 8 * (i & 1) + r) * ld + n0 + 8 * (i >> 1));
}
__device__ __forceinline__ uint32_t b2_addr_nk(uint32_t base, int ld, int k0, int n0, int lane) {
  const int i = lane >> 3, r = lane & 7;
  return base + 2u * (uint32_t)((n0 + 8 * (i >> 1) + r) * ld + k0 + 8 * (i & 1));
}
// B fragment of one n-tile of a [n][k] plane (x2 load: lanes 0-15 give the rows).
__device__ __forceinline__ uint32_t b1_addr_nk(uint32_t base, int ld, int k0, int n0, int lane) {
  const int i = (lane >> 3) & 1, r = lane & 7;
  return base + 2u * (uint32_t)((n0 + r) * ld + k0 + 8 * i);
}

__device__ __forceinline__ void mma_bf16(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// m16n8k8 bf16 tile (A fragment 2 registers, B fragment 1)
__device__ __forceinline__ void mma_bf16_k8(float c[4], uint32_t a0, uint32_t a1, uint32_t b0) {
  asm("mma.sync.aligned.m16n8k8.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(b0));
}
// c += a.b, three-term bf16 split (small terms first)
__device__ __forceinline__ void mma_bf16x3(float c[4], const uint32_t ah[4], const uint32_t al[4],
                                           uint32_t bh0, uint32_t bh1, uint32_t bl0, uint32_t bl1) {
  mma_bf16(c, al, bh0, bh1);
  mma_bf16(c, ah, bl0, bl1);
  mma_bf16(c, ah, bh0, bh1);
}

// (x, y) -> packed bf16x2 words of the hi and lo planes
__device__ __forceinline__ void split_bf16x2(float x, float y, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x - hf.x, y - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Float pair atomically added to global memory (no return value).
__device__ __forceinline__ void red_add_f2(float* p, float x, float y) {
  asm volatile("red.global.add.v2.f32 [%0], {%1, %2};" ::"l"(p), "f"(x), "f"(y) : "memory");
}

}  // namespace tt
