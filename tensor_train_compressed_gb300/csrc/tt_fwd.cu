// Forward TT embedding bag: prefix partials, unique rows, bag pooling.
//
// FlowTT (summary card, key innovations and approach; abstract): each shared
// prefix of the contraction chain is formed once and kept on chip while every
// row that extends it is formed.  Per work chunk (a run of unique (i1, i2)
// prefixes with the same i2, or a piece of one large prefix):
//
//   stage 2   P2[p] = G1[i1_p] . G2[i2]     (n1 x R1).(R1 x n2*R2), in shared memory
//   stage 3   row[x] = P2[p(x)] . G3[i3_x]  (n1*n2 x R2).(R2 x n3) = D values
//
// Rows go to a unique-row buffer in the workspace (L2-resident at the sizes
// used here); k_pool then sums each bag's rows with coalesced float4 loads
// and stores (sum pooling of the TT-EmbeddingBag, TT-Rec abstract).
// Persistent CTAs take chunks from an atomic counter (dynamic load
// balancing under Zipf skew, FlowTT summary card, key innovations).
#include "tt_internal.cuh"

namespace tt {

struct FwdArgs {
  Shape s;
  WS w;
  const float* G1;
  const float* G2;
  const float* G3;
};

// Shape-generic chunk kernel (any shape within the shared-memory limit).
__global__ void __launch_bounds__(256) k_fwd_generic(FwdArgs a) {
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  __shared__ int c_sh;
  const Shape& s = a.s;
  const int tid = threadIdx.x;
  const int g2n = s.R1 * s.n2 * s.R2;
  const int p1n = s.n1 * s.R1;
  const int n2R2 = s.n2 * s.R2;
  const int p2n = s.n1 * n2R2;
  const int n3 = s.n3, R1 = s.R1, R2 = s.R2, D = s.D;
  float* G2s = sm;
  const int n_chunks = a.w.ctl->n_chunks;
  for (;;) {
    if (tid == 0) c_sh = (int)atomicAdd(&a.w.ctl->fwd_chunk_ctr, 1u);
    __syncthreads();
    const int c = c_sh;
    if (c >= n_chunks) break;
    const int x0 = a.w.chunk_start[c], x1 = a.w.chunk_start[c + 1];
    const int p0 = a.w.row_pair[x0], p1 = a.w.row_pair[x1 - 1];
    const int np = p1 - p0 + 1;
    float* P1s = G2s + g2n;
    float* P2s = P1s + np * p1n;
    const int i2 = a.w.pair_i2[p0];
    const float* g2 = a.G2 + (size_t)i2 * g2n;
    for (int e = tid; e < g2n; e += blockDim.x) G2s[e] = __ldg(g2 + e);
    for (int e = tid; e < np * p1n; e += blockDim.x) {
      const int p = e / p1n;
      P1s[e] = __ldg(a.G1 + (size_t)a.w.pair_i1[p0 + p] * p1n + (e - p * p1n));
    }
    __syncthreads();
    for (int e = tid; e < np * p2n; e += blockDim.x) {
      const int p = e / p2n, rem = e - p * p2n;
      const int j1 = rem / n2R2, j2b = rem - j1 * n2R2;
      const float* pa = P1s + p * p1n + j1 * R1;
      float acc = 0.f;
      for (int aa = 0; aa < R1; ++aa) acc = fmaf(pa[aa], G2s[aa * n2R2 + j2b], acc);
      P2s[e] = acc;
    }
    __syncthreads();
    const int nx = x1 - x0;
    for (int e = tid; e < nx * D; e += blockDim.x) {
      const int xi = e / D, j = e - xi * D;
      const int x = x0 + xi;
      const int j12 = j / n3, j3 = j - j12 * n3;
      const float* pp = P2s + (a.w.row_pair[x] - p0) * p2n + j12 * R2;
      const float* g3 = a.G3 + (size_t)a.w.row_i3[x] * R2 * n3 + j3;
      float acc = 0.f;
      for (int b = 0; b < R2; ++b) acc = fmaf(pp[b], __ldg(g3 + b * n3), acc);
      a.w.rowbuf[(size_t)x * D + j] = acc;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
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
                                             float* __restrict__ P2, int np) {
  constexpr int R = T::kR;
  constexpr int NC = T::NC;
  constexpr int G = NC / C;                 // column groups per prefix
  for (int item = threadIdx.x; item < np * G; item += blockDim.x) {
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

template <int N2, int R, int CP>
__global__ void __launch_bounds__(256, TileCfg<N2, R, CP>::MIN_BLOCKS) k_fwd_tiled(FwdArgs a) {
  using T = TileCfg<N2, R, CP>;
  extern __shared__ float4 sm4[];
  float* G2s = reinterpret_cast<float*>(sm4);
  float* P1t = G2s + T::F_G2;
  float* P2 = P1t + T::F_P1;
  float* G3s = P2 + T::F_P2;
  __shared__ int c_sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_chunks = a.w.ctl->n_chunks;
  for (;;) {
    if (tid == 0) c_sh = (int)atomicAdd(&a.w.ctl->fwd_chunk_ctr, 1u);
    __syncthreads();
    const int c = c_sh;
    if (c >= n_chunks) break;
    const int x0 = a.w.chunk_start[c], x1 = a.w.chunk_start[c + 1];
    const int p0 = a.w.row_pair[x0], p1 = a.w.row_pair[x1 - 1];
    const int np = p1 - p0 + 1;
    const int i2 = a.w.pair_i2[p0];
    {
      const float4* g2 = reinterpret_cast<const float4*>(a.G2 + (size_t)i2 * T::F_G2);
      float4* d = reinterpret_cast<float4*>(G2s);
#pragma unroll 4
      for (int e = tid; e < T::F_G2 / 4; e += 256) d[e] = __ldg(g2 + e);
    }
    for (int e = tid; e < np * R * 4; e += 256) {
      const int p = e / (R * 4), rem = e - p * (R * 4);
      const int j1 = rem / R, k = rem - j1 * R;         // coalesced read of G1[i1][0][j1][k]
      P1t[p * (R * 4) + k * 4 + j1] = __ldg(a.G1 + (size_t)a.w.pair_i1[p0 + p] * (R * 4) + rem);
    }
    __syncthreads();
    // stage 2: C = columns per thread, so that np * NC / C ~ 256 items
    {
      const int need = (np * T::NC + 255) / 256;
      if (need <= 1) tiled_stage2<T, 1>(G2s, P1t, P2, np);
      else if (need <= 2) tiled_stage2<T, 2>(G2s, P1t, P2, np);
      else if (need <= 4) tiled_stage2<T, 4>(G2s, P1t, P2, np);
      else if (need <= 8) tiled_stage2<T, 8>(G2s, P1t, P2, np);
      else tiled_stage2<T, 16>(G2s, P1t, P2, np);
    }
    // stage 3 in batches of RB rows
    const int blk = warp % T::NB, rgrp = warp / T::NB;
    for (int xb = x0; xb < x1; xb += T::RB) {
      const int nb = min(T::RB, x1 - xb);
      __syncthreads();   // P2 complete (first batch) / G3s free (later batches)
      constexpr int Q = R;   // float4 per G3 slice (R*4 floats)
      for (int e = tid; e < nb * Q; e += 256) {
        const int r = e / Q, q = e - r * Q;
        const float4 v = __ldg(reinterpret_cast<const float4*>(
                                   a.G3 + (size_t)a.w.row_i3[xb + r] * (R * 4)) + q);
        *reinterpret_cast<float4*>(G3s + r * T::G3S + 4 * q) = v;
      }
      __syncthreads();
      const int r = rgrp * 32 + lane;
      if (r < nb) {
        const int x = xb + r;
        const float* pp = P2 + (a.w.row_pair[x] - p0) * T::P2P + (blk * 4) * T::P2S;
        const float* gg = G3s + r * T::G3S;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 2
        for (int b = 0; b < R; b += 4) {
          float4 pv[4], gv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) pv[i] = *reinterpret_cast<const float4*>(pp + i * T::P2S + b);
#pragma unroll
          for (int t = 0; t < 4; ++t) gv[t] = *reinterpret_cast<const float4*>(gg + (b + t) * 4);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float pw[4] = {pv[i].x, pv[i].y, pv[i].z, pv[i].w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              acc[i][0] = fmaf(pw[t], gv[t].x, acc[i][0]);
              acc[i][1] = fmaf(pw[t], gv[t].y, acc[i][1]);
              acc[i][2] = fmaf(pw[t], gv[t].z, acc[i][2]);
              acc[i][3] = fmaf(pw[t], gv[t].w, acc[i][3]);
            }
          }
        }
        float4* o = reinterpret_cast<float4*>(a.w.rowbuf + (size_t)x * T::D + blk * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      }
    }
    __syncthreads();
  }
}

// out[b] = sum of the unique rows of bag b's lookups; one warp per bag.
__global__ void __launch_bounds__(256) k_pool(const int64_t* __restrict__ offsets, int64_t B,
                                              int64_t nnz, const int32_t* __restrict__ uid,
                                              const float* __restrict__ rowbuf, int D,
                                              float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < B; b += warps) {
    int64_t l0 = offsets[b], l1 = offsets[b + 1];
    l0 = l0 < 0 ? 0 : (l0 > nnz ? nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > nnz ? nnz : l1);
    if ((D & 3) == 0) {
      const int D4 = D >> 2;
      const float4* rb = reinterpret_cast<const float4*>(rowbuf);
      float4* o = reinterpret_cast<float4*>(out + b * (int64_t)D);
      for (int c = lane; c < D4; c += 32) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        int64_t l = l0;
        for (; l + 4 <= l1; l += 4) {
          const int u0 = uid[l], u1 = uid[l + 1], u2 = uid[l + 2], u3 = uid[l + 3];
          const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 v0 = u0 >= 0 ? rb[(int64_t)u0 * D4 + c] : z;
          const float4 v1 = u1 >= 0 ? rb[(int64_t)u1 * D4 + c] : z;
          const float4 v2 = u2 >= 0 ? rb[(int64_t)u2 * D4 + c] : z;
          const float4 v3 = u3 >= 0 ? rb[(int64_t)u3 * D4 + c] : z;
          acc.x += v0.x; acc.y += v0.y; acc.z += v0.z; acc.w += v0.w;
          acc.x += v1.x; acc.y += v1.y; acc.z += v1.z; acc.w += v1.w;
          acc.x += v2.x; acc.y += v2.y; acc.z += v2.z; acc.w += v2.w;
          acc.x += v3.x; acc.y += v3.y; acc.z += v3.z; acc.w += v3.w;
        }
        for (; l < l1; ++l) {
          const int u = uid[l];
          if (u >= 0) {
            const float4 v = rb[(int64_t)u * D4 + c];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
          }
        }
        o[c] = acc;
      }
    } else {
      for (int j = lane; j < D; j += 32) {
        float acc = 0.f;
        for (int64_t l = l0; l < l1; ++l) {
          const int u = uid[l];
          if (u >= 0) acc += rowbuf[(int64_t)u * D + j];
        }
        out[b * (int64_t)D + j] = acc;
      }
    }
  }
}

static size_t fwd_generic_smem(const Shape& s, int CP) {
  return sizeof(float) * ((size_t)s.R1 * s.n2 * s.R2 +
                          (size_t)CP * (s.n1 * s.R1 + s.n1 * s.n2 * s.R2));
}

// Which chunk kernel serves a shape, and its chunking parameters.
enum FwdKind { kFwdGeneric = 0, kFwdTiled_8_32, kFwdTiled_8_64, kFwdTiled_4_16 };

static FwdKind fwd_kind(const Shape& s) {
  if (s.n1 != 4 || s.n3 != 4 || s.R1 != s.R2) return kFwdGeneric;
  if (s.n2 == 8 && s.R1 == 32) return kFwdTiled_8_32;
  if (s.n2 == 8 && s.R1 == 64) return kFwdTiled_8_64;
  if (s.n2 == 4 && s.R1 == 16) return kFwdTiled_4_16;
  return kFwdGeneric;
}

constexpr int kCP_8_32 = 12, kCP_8_64 = 4, kCP_4_16 = 16;

int forward_chunk_params(const Shape& s, int* pairs_per_chunk, int* rows_per_chunk) {
  const int64_t g2n = (int64_t)s.R1 * s.n2 * s.R2;
  const int64_t per = (int64_t)s.n1 * s.R1 + (int64_t)s.n1 * s.n2 * s.R2;
  if (g2n + per + (int64_t)s.n1 * s.n2 * s.R2 > kMaxSmemFloats) return TT_EMB_ERR_UNSUPPORTED;
  int64_t cp = (kMaxSmemFloats - g2n) / per;
  if (cp > 16) cp = 16;
  if (cp < 1) cp = 1;
  switch (fwd_kind(s)) {
    case kFwdTiled_8_32: cp = kCP_8_32; break;
    case kFwdTiled_8_64: cp = kCP_8_64; break;
    case kFwdTiled_4_16: cp = kCP_4_16; break;
    default: break;
  }
  *pairs_per_chunk = (int)cp;
  *rows_per_chunk = 32;
  return TT_EMB_OK;
}

static int persistent_grid(const void* fn, int threads, size_t smem) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return per_sm * sm_count();
}

template <int N2, int R, int CP>
static void launch_tiled(const FwdArgs& fa, cudaStream_t st) {
  using T = TileCfg<N2, R, CP>;
  static int grid = 0;
  if (grid == 0) {
    cudaFuncSetAttribute(k_fwd_tiled<N2, R, CP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         T::SMEM);
    grid = persistent_grid((const void*)k_fwd_tiled<N2, R, CP>, 256, T::SMEM);
  }
  TT_TIMED("k_fwd_tiled", st, (k_fwd_tiled<N2, R, CP><<<grid, 256, T::SMEM, st>>>(fa)));
}

int launch_forward(const Shape& s, const Layout& L, const WS& w, const float* const cores[3],
                   const int64_t* offsets, int64_t nnz, int64_t num_bags, float* out,
                   cudaStream_t st) {
  (void)L;
  int CP = 0, CR = 0;
  int rc = forward_chunk_params(s, &CP, &CR);
  if (rc) return rc;
  FwdArgs fa;
  fa.s = s;
  fa.w = w;
  fa.G1 = cores[0];
  fa.G2 = cores[1];
  fa.G3 = cores[2];
  switch (fwd_kind(s)) {
    case kFwdTiled_8_32: launch_tiled<8, 32, kCP_8_32>(fa, st); break;
    case kFwdTiled_8_64: launch_tiled<8, 64, kCP_8_64>(fa, st); break;
    case kFwdTiled_4_16: launch_tiled<4, 16, kCP_4_16>(fa, st); break;
    default: {
      const size_t smem = fwd_generic_smem(s, CP);
      static int grid = 0;
      if (grid == 0) {
        cudaFuncSetAttribute(k_fwd_generic, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kMaxSmemFloats * (int)sizeof(float));
        grid = persistent_grid((const void*)k_fwd_generic, 256, kMaxSmemFloats * sizeof(float));
      }
      TT_TIMED("k_fwd_generic", st, (k_fwd_generic<<<grid, 256, smem, st>>>(fa)));
    }
  }
  if (num_bags > 0) {
    int grid = (int)ceil_div(num_bags, 8);
    const int cap = sm_count() * 16;
    if (grid > cap) grid = cap;
    TT_TIMED("k_pool", st, (k_pool<<<grid, 256, 0, st>>>(offsets, num_bags, nnz, w.uid, w.rowbuf, s.D, out)));
  }
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
