// Register-tiled building blocks shared by the forward and backward chunk
// kernels for n1 = n3 = 4 and R1 = R2 = R (the shapes of the benchmark tables).
#pragma once

#include "tt_internal.cuh"

namespace tt {

// Prefixes per chunk of the tiled kernels (shared by the grouping, the forward
// and the backward: the backward sizes its shared memory for this many).
constexpr int kCP_8_32 = 8, kCP_8_64 = 4, kCP_4_16 = 16;

// Register-tiled chunk kernel for n1 = n3 = 4 and R1 = R2 = R (the shapes of the
// benchmark tables).  Shared memory per CTA:
//   G2s  [R][N2*R]          the chunk's G2 slice (all its prefixes share i2)
//   P1t  [CP][R][4]         G1[i1_p] transposed, a-major
//   P2   [CP][4*N2][R+4]    prefix partials, rows padded by 4 floats and the
//                           per-prefix block by 4 more, so that the 128-bit
//                           loads of stage 3 are free of bank conflicts
//   G3s  [RB][R*4+4]        G3 slices of a batch of RB rows, padded likewise
// Stage 2 is a (4*np) x (N2*R) x R GEMM: each thread owns the 4 j1 rows of one
// prefix and C columns (C chosen from np so that ~256 threads are busy).
// Stage 3 gives each warp one block of 4 j12 values and each lane one row.
template <int N2, int R, int CP>
struct TileCfg {
  static constexpr int N1 = 4, N3 = 4, kN2 = N2, kR = R;
  static constexpr int NC = N2 * R;                 // stage-2 columns (j2, b)
  static constexpr int NB = N1 * N2 / 4;            // j12 blocks of 4
  static constexpr int P2S = R + 4;                 // padded P2 row stride
  static constexpr int P2P = N1 * N2 * P2S + 4;     // padded P2 block per prefix
  static constexpr int RB = 32 * (8 / NB);          // rows per stage-3 batch
  static constexpr int G3S = R * N3 + 4;            // padded G3 row stride
  static constexpr int D = N1 * N2 * N3;
  static constexpr int F_G2 = R * NC;
  static constexpr int F_P1 = CP * R * N1;
  static constexpr int F_P2 = CP * P2P;
  static constexpr int F_G3 = RB * G3S;
  static constexpr int SMEM = 4 * (F_G2 + F_P1 + F_P2 + F_G3);
  static constexpr int MIN_BLOCKS = SMEM <= 110 * 1024 ? 2 : 1;
  static_assert(NB == 4 || NB == 8, "j12 blocks must fill 8 warps");
  static_assert(R % 4 == 0, "R must be a multiple of 4");
};

template <class T, int C>
__device__ __forceinline__ void tiled_stage2(const float* __restrict__ G2s,
                                             const float* __restrict__ P1t,
                                             float* __restrict__ P2, int np,
                                             int ltid = -1, int nthreads = -1) {
  if (ltid < 0) ltid = threadIdx.x;
  if (nthreads < 0) nthreads = blockDim.x;
  constexpr int R = T::kR;
  constexpr int NC = T::NC;
  constexpr int G = NC / C;                 // column groups per prefix
  for (int item = ltid; item < np * G; item += nthreads) {
    const int p = item / G, cg = item - p * G;
    float acc[4][C];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < C; ++c) acc[i][c] = 0.f;
    const float* ap = P1t + p * (R * 4);
#pragma unroll 8
    for (int k = 0; k < R; ++k) {
      const float4 av = *reinterpret_cast<const float4*>(ap + k * 4);
      float bv[C];
      const float* brow = G2s + k * NC;
      if constexpr (C >= 4) {
#pragma unroll
        for (int q = 0; q < C / 4; ++q) {
          const float4 v = *reinterpret_cast<const float4*>(brow + q * (NC * 4 / C) + 4 * cg);
          bv[4 * q] = v.x; bv[4 * q + 1] = v.y; bv[4 * q + 2] = v.z; bv[4 * q + 3] = v.w;
        }
      } else if constexpr (C == 2) {
        const float2 v = *reinterpret_cast<const float2*>(brow + 2 * cg);
        bv[0] = v.x; bv[1] = v.y;
      } else {
        bv[0] = brow[cg];
      }
#pragma unroll
      for (int c = 0; c < C; ++c) {
        acc[0][c] = fmaf(av.x, bv[c], acc[0][c]);
        acc[1][c] = fmaf(av.y, bv[c], acc[1][c]);
        acc[2][c] = fmaf(av.z, bv[c], acc[2][c]);
        acc[3][c] = fmaf(av.w, bv[c], acc[3][c]);
      }
    }
    float* pp = P2 + p * T::P2P;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if constexpr (C >= 4) {
#pragma unroll
        for (int q = 0; q < C / 4; ++q) {
          const int n = q * (NC * 4 / C) + 4 * cg;    // 4 consecutive columns, same j2
          const int j2 = n / R, b = n - j2 * R;
          *reinterpret_cast<float4*>(pp + (i * T::kN2 + j2) * T::P2S + b) =
              make_float4(acc[i][4 * q], acc[i][4 * q + 1], acc[i][4 * q + 2], acc[i][4 * q + 3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < C; ++c) {
          const int n = C * cg + c;
          const int j2 = n / R, b = n - j2 * R;
          pp[(i * T::kN2 + j2) * T::P2S + b] = acc[i][c];
        }
      }
    }
  }
}

// P2 for the np prefixes of a chunk, with C chosen so that ~256 threads work.
template <class T>
__device__ __forceinline__ void tiled_stage2_any(const float* __restrict__ G2s,
                                                 const float* __restrict__ P1t,
                                                 float* __restrict__ P2, int np) {
  const int need = (np * T::NC + 255) / 256;
  if (need <= 1) tiled_stage2<T, 1>(G2s, P1t, P2, np);
  else if (need <= 2) tiled_stage2<T, 2>(G2s, P1t, P2, np);
  else if (need <= 4) tiled_stage2<T, 4>(G2s, P1t, P2, np);
  else if (need <= 8) tiled_stage2<T, 8>(G2s, P1t, P2, np);
  else tiled_stage2<T, 16>(G2s, P1t, P2, np);
}

// ---------------------------------------------------------------------------
// mbarrier + bulk-copy (TMA, 1-D) helpers.  Every wait is capped: after
// kWaitCap polls it sets the timeout bit and gives up.
constexpr long long kWaitCap = 1ll << 24;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
// 16-byte asynchronous global -> shared copy (cp.async, L2 only); its
// completion is tracked per thread (cp_async_arrive_noinc).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
// Arrive on `bar` once all cp.async copies this thread issued so far have
// landed; the arrival is part of the barrier's initial count (no increment).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Stage the chunk's G2 slice and the transposed G1 rows of its prefixes;
// `while_in_flight` runs once the slice's copies are issued.
template <class T, class F = void (*)()>
__device__ __forceinline__ void tiled_load_g2_p1(const float* __restrict__ G1,
                                                 const float* __restrict__ G2,
                                                 const int32_t* __restrict__ pair_i1, int i2,
                                                 int p0, int np, float* G2s, float* P1t,
                                                 F while_in_flight = [] {}) {
  constexpr int R = T::kR;
  const int tid = threadIdx.x;
  const float4* g2 = reinterpret_cast<const float4*>(G2 + (size_t)i2 * T::F_G2);
  float4* d = reinterpret_cast<float4*>(G2s);
  // the G2 slice by 16-byte asynchronous copies, all in flight at once, while
  // the G1 rows (transposed on the way) take the register path
  for (int e = tid; e < T::F_G2 / 4; e += 256) cp_async16(d + e, g2 + e);
  while_in_flight();
  for (int e = tid; e < np * R * 4; e += 256) {
    const int p = e / (R * 4), rem = e - p * (R * 4);
    const int j1 = rem / R, k = rem - j1 * R;        // coalesced read of G1[i1][0][j1][k]
    P1t[p * (R * 4) + k * 4 + j1] = __ldg(G1 + (size_t)pair_i1[p0 + p] * (R * 4) + rem);
  }
  cp_async_wait_all();
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, Ctl* ctl) {
  for (long long i = 0; i < kWaitCap; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  set_status(ctl, kStTimeout);
  return false;
}
// global -> shared bulk copy completing on `bar` (16-byte aligned, size % 16 == 0)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// Decoded work-chunk descriptor: rows [x0, x1), prefixes [p0, p1]; `whole` is
// set when the chunk starts at the first row of its first prefix.
struct ChunkDesc {
  int x0, x1, p0, p1;
  bool whole;
  bool cont;   // the next chunk (row order) is a later piece of this chunk's last prefix
};
__device__ __forceinline__ ChunkDesc load_chunk(const int2* __restrict__ desc, int c) {
  const int2 a = desc[c], b = desc[c + 1];
  ChunkDesc d;
  d.x0 = a.x;
  d.x1 = b.x;
  d.p0 = a.y & 0x7fffffff;
  d.whole = a.y < 0;
  // the next chunk starts a new prefix, or continues (a piece of) this one
  d.p1 = (b.y & 0x7fffffff) - (b.y < 0 ? 1 : 0);
  d.cont = b.y >= 0;
  return d;
}
// Lane 0 of the calling warp claims the next work chunk; broadcast to the warp.
__device__ __forceinline__ int claim_chunk(uint32_t* ctr) {
  int c = 0;
  if ((threadIdx.x & 31) == 0) c = (int)atomicAdd(ctr, 1u);
  return __shfl_sync(0xffffffffu, c, 0);
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Stage 2 for chunks of one or two prefixes, from G1 rows in their natural
// [j1][a] layout: the R-long reduction is split over KQ lanes (8/16 lanes
// apart, so the 128-bit G2 loads of a phase stay conflict-free) and summed by
// shuffles.  KQ = 4 for one prefix, 2 for two: 256 threads either way.
template <class T, int KQ>
__device__ __forceinline__ void tiled_stage2_splitk(const float* __restrict__ G2s,
                                                    const float* __restrict__ P1n,
                                                    float* __restrict__ P2, int np, int nthreads,
                                                    int ltid) {
  constexpr int R = T::kR, NC = T::NC, CPW = 32 / KQ;   // column groups per warp
  constexpr int KS = R / KQ;
  const int lane = threadIdx.x & 31;
  const int kq = lane / CPW, cgl = lane - kq * CPW;
  const int total = np * (NC / 4) * KQ;
  for (int base = 0; base < total; base += nthreads) {
    const int wi = (base + ltid) >> 5;                 // warp-item
    const int cgall = wi * CPW + cgl;                   // over all prefixes
    const bool valid = base + ltid < total;
    const int p = cgall / (NC / 4), cg = cgall - p * (NC / 4);
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    if (valid) {
      const float* ap = P1n + p * (4 * R);
#pragma unroll 4
      for (int k = kq * KS; k < (kq + 1) * KS; ++k) {
        const float4 bv = *reinterpret_cast<const float4*>(G2s + k * NC + 4 * cg);
        const float a0 = ap[k], a1 = ap[R + k], a2 = ap[2 * R + k], a3 = ap[3 * R + k];
        acc[0][0] = fmaf(a0, bv.x, acc[0][0]); acc[0][1] = fmaf(a0, bv.y, acc[0][1]);
        acc[0][2] = fmaf(a0, bv.z, acc[0][2]); acc[0][3] = fmaf(a0, bv.w, acc[0][3]);
        acc[1][0] = fmaf(a1, bv.x, acc[1][0]); acc[1][1] = fmaf(a1, bv.y, acc[1][1]);
        acc[1][2] = fmaf(a1, bv.z, acc[1][2]); acc[1][3] = fmaf(a1, bv.w, acc[1][3]);
        acc[2][0] = fmaf(a2, bv.x, acc[2][0]); acc[2][1] = fmaf(a2, bv.y, acc[2][1]);
        acc[2][2] = fmaf(a2, bv.z, acc[2][2]); acc[2][3] = fmaf(a2, bv.w, acc[2][3]);
        acc[3][0] = fmaf(a3, bv.x, acc[3][0]); acc[3][1] = fmaf(a3, bv.y, acc[3][1]);
        acc[3][2] = fmaf(a3, bv.z, acc[3][2]); acc[3][3] = fmaf(a3, bv.w, acc[3][3]);
      }
    }
#pragma unroll
    for (int o = CPW; o < 32; o <<= 1)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += __shfl_xor_sync(0xffffffffu, acc[i][j], o);
    if (valid && kq == 0) {
      const int n = 4 * cg, j2 = n / R, b = n - j2 * R;
      float* pp = P2 + p * T::P2P + j2 * T::P2S + b;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(pp + i * T::kN2 * T::P2S) =
            make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
  }
}

// Stage 2 from G1 rows in natural layout P1n; for np >= 3 they are first
// transposed into P1t ([p][a][j1], 4*R*np floats) so that the A operand of a
// k step is one 128-bit broadcast load.  Ends with the 256 compute threads
// synchronised (named barrier 1).
template <class T>
__device__ __forceinline__ void stage2_natural(const float* __restrict__ G2s,
                                               const float* __restrict__ P1n,
                                               float* __restrict__ P1t,
                                               float* __restrict__ P2, int np, int ltid = -1,
                                               int bar_id = 1) {
  constexpr int R = T::kR;
  if (ltid < 0) ltid = threadIdx.x;
  const int need = (np * T::NC + 255) / 256;    // column groups of 4 per thread for ~256 items
  if (np == 1) {
    tiled_stage2_splitk<T, 4>(G2s, P1n, P2, np, 256, ltid);
  } else if (np == 2) {
    tiled_stage2_splitk<T, 2>(G2s, P1n, P2, np, 256, ltid);
  } else {
    for (int e = ltid; e < np * 4 * R; e += 256) {
      const int p = e / (4 * R), rem = e - p * (4 * R);
      const int j1 = rem / R, k = rem - j1 * R;
      P1t[p * 4 * R + k * 4 + j1] = P1n[e];
    }
    named_sync(bar_id, 256);
    if (need <= 4) tiled_stage2<T, 4>(G2s, P1t, P2, np, ltid, 256);
    else if (need <= 8) tiled_stage2<T, 8>(G2s, P1t, P2, np, ltid, 256);
    else tiled_stage2<T, 16>(G2s, P1t, P2, np, ltid, 256);
  }
  named_sync(bar_id, 256);
}


}  // namespace tt
