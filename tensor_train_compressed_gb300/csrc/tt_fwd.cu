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
#include "tt_tile.cuh"
#include "tt_mma.cuh"

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

// Chunk metadata from the descriptors the grouping writes: rows x0 .. x1-1,
// prefixes p0 .. p0+np-1, their i2.  Two dependent round trips (descriptors,
// then i2); c >= n_chunks gives x0 = x1 (the end).
struct TiledMeta {
  int c, x0, x1, p0, np, i2, tab;
};
__device__ __forceinline__ TiledMeta tiled_meta(const WS& w, int c, int n_chunks) {
  TiledMeta m{c, 0, 0, 0, 0, 0, 0};
  if (c >= n_chunks) return m;
  const int2 d0 = w.chunk_desc[c], d1 = w.chunk_desc[c + 1];
  m.x0 = d0.x;
  m.x1 = d1.x;
  m.p0 = d0.y & 0x7fffffff;
  // the chunk's last prefix: the next chunk's, unless that one starts a new prefix
  const int pn = d1.y & 0x7fffffff;
  const int p1 = (d1.y < 0) ? pn - 1 : pn;
  m.np = p1 - m.p0 + 1;
  m.i2 = w.pair_i2[m.p0];
  return m;
}

// The tables of one launch of the tiled chunk kernel (one table for a plain
// forward; up to kMaxTables for tt_emb_forward_tables, all of one (n, R)).
// Chunks are claimed from the first table's counter and numbered across the
// tables in order, so that one persistent grid balances all of them.
struct TiledTables {
  FwdArgs t[kMaxTables];
  int T;
};

// Table and table-local metadata of global chunk cg (cbase: first global chunk
// of every table, cbase[T] = all chunks).
__device__ __forceinline__ TiledMeta tiled_meta_tables(const TiledTables& tabs, const int* cbase,
                                                       int cg) {
  int t = 0;
  while (t + 1 < tabs.T && cg >= cbase[t + 1]) ++t;
  if (cg >= cbase[tabs.T]) {
    TiledMeta m{cg, 0, 0, 0, 0, 0, 0};
    return m;
  }
  TiledMeta m = tiled_meta(tabs.t[t].w, cg - cbase[t], cbase[t + 1] - cbase[t]);
  m.c = cg;
  m.tab = t;
  return m;
}

template <int N2, int R, int CP>
__global__ void __launch_bounds__(256, TileCfg<N2, R, CP>::MIN_BLOCKS)
    k_fwd_tiled(const __grid_constant__ TiledTables tabs) {
  using T = TileCfg<N2, R, CP>;
  extern __shared__ float4 sm4[];
  float* G2s = reinterpret_cast<float*>(sm4);
  float* P1t = G2s + T::F_G2;
  float* P2 = P1t + T::F_P1;
  float* G3s = P2 + T::F_P2;
  __shared__ TiledMeta meta[2];
  __shared__ int rp_sh[T::RB];          // prefix of every row of the stage-3 batch
  __shared__ int cbase[kMaxTables + 1];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t* ctr = &tabs.t[0].w.ctl->fwd_chunk_ctr;
  if (tid == 0) {
    int acc = 0;
    for (int t = 0; t < tabs.T; ++t) {
      cbase[t] = acc;
      acc += tabs.t[t].w.ctl->n_chunks;
    }
    cbase[tabs.T] = acc;
    meta[0] = tiled_meta_tables(tabs, cbase, (int)atomicAdd(ctr, 1u));
  }
  __syncthreads();
  const int n_chunks = cbase[tabs.T];
  for (int it = 0;; ++it) {
    const TiledMeta m = meta[it & 1];
    if (m.c >= n_chunks) break;
    const FwdArgs& a = tabs.t[m.tab];
    const int x0 = m.x0, x1 = m.x1, p0 = m.p0, np = m.np;
    // the G2 slice and G1 rows of this chunk; thread 0 claims the next chunk and
    // loads its metadata while the copies are in flight
    tiled_load_g2_p1<T>(a.G1, a.G2, a.w.pair_i1, m.i2, p0, np, G2s, P1t, [&]() {
      if (tid == 0) meta[(it + 1) & 1] = tiled_meta_tables(tabs, cbase, (int)atomicAdd(ctr, 1u));
    });
    __syncthreads();
    tiled_stage2_any<T>(G2s, P1t, P2, np);
    // stage 3 in batches of RB rows
    const int blk = warp % T::NB, rgrp = warp / T::NB;
    for (int xb = x0; xb < x1; xb += T::RB) {
      const int nb = min(T::RB, x1 - xb);
      __syncthreads();   // P2 complete (first batch) / G3s free (later batches)
      constexpr int Q = R;   // float4 per G3 slice (R*4 floats)
      for (int e = tid; e < nb * Q; e += 256) {   // asynchronous 16-byte copies, all in flight
        const int r = e / Q, q = e - r * Q;
        cp_async16(G3s + r * T::G3S + 4 * q,
                   reinterpret_cast<const float4*>(a.G3 + (size_t)a.w.row_i3[xb + r] * (R * 4)) + q);
      }
      if (tid < nb) rp_sh[tid] = a.w.row_pair[xb + tid] - p0;
      cp_async_wait_all();
      __syncthreads();
      const int r = rgrp * 32 + lane;
      if (r < nb) {
        const int x = xb + r;
        const float* pp = P2 + rp_sh[r] * T::P2P + (blk * 4) * T::P2S;
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

// ---------------------------------------------------------------------------
// Tensor-core chunk kernel for n1 = n3 = 4, n2 = 8, R1 = R2 = 32 (D = 128).
// Warp 8 is a producer: it claims the next chunk, writes the chunk's metadata
// (the list of row pairs) and stages the G2 slice, the G1 rows and up to ROWMAX
// G3 rows into the free one of two stage buffers with 16-byte cp.async copies
// (one 512-byte warp instruction per row slice, into padded rows), each lane
// signalling the buffer's "full" mbarrier when its copies have landed.
// Warps 0-7 consume with m16n8k8 TF32 tiles (three-term split, fp32 accuracy;
// tt_mma.cuh):
//   stage 2  P2 = [G1 rows of the chunk's prefixes] . G2[i2]   (4 np) x 256 x 32
//   stage 3  for each pair of rows of one prefix:
//            P2[p] . [G3[i3_a] | G3[i3_b]]                     32 x 8 x 32
//            (a prefix with an odd row count pairs its last row with itself and
//            drops the copy)
// and release the buffer through its "empty" mbarrier, so that the staging of
// chunk i+1 overlaps the math of chunk i.  All shared-memory strides are
// padded so that every fragment load and store is free of bank conflicts.
template <int CW>
struct MmaFwd {
  static constexpr int CP = kCP_8_32, R = 32, NC = 256, D = 128;
  static constexpr int ROWMAX = 64;                  // G3 rows staged per chunk
  static constexpr int MAXROWS = CP * 32;            // rows of one chunk (CP prefixes x 32)
  static constexpr int MAXPAIRS = MAXROWS / 2 + CP;
  // G2 and G1 are staged as bf16 hi / lo planes (k_split_cores): G2 rows (r1)
  // of 264 bf16 (528 B), G1 rows ((p, j1)) of 40 bf16 (80 B)
  static constexpr int G2LD = NC + 8, G1LD = R + 8;
  static constexpr int G2PLANE = R * G2LD * 2, G1PLANE = 4 * CP * G1LD * 2;   // bytes
  // staged G3 rows as bf16 planes of G3 transposed per row: [j3][r2], 80-byte
  // j3 rows (row ROWMAX stays zero); P2 as bf16 planes [p][j1][j2][r2]: j2 rows
  // of 80 B, j1 blocks of 656 B, prefixes 2624 B apart
  static constexpr int GTROW = 4 * (R + 8) * 2, GTPLANE = (ROWMAX + 1) * GTROW;
  static constexpr int PB = 80, PA = 8 * PB + 16, PPB = 4 * PA, P2PLANE = CP * PPB;
  static constexpr int F_G2 = G2PLANE / 2, F_P1 = G1PLANE / 2, F_G3 = GTPLANE / 2;   // floats
  static constexpr int STAGE_F = F_G2 + F_P1 + F_G3;
  static constexpr int F_P2 = P2PLANE / 2;
  // L2 checkpoint slot of one prefix partial: the hi and lo planes of its P2
  // (one prefix of the P2 layout, padding included)
  static constexpr int CKB = 2 * PPB;
  struct Meta {
    int x0, x1, p0, np, npairs, end;
    int ck;               // checkpoint role: s + 1 writes slot s, -(s + 1) reads it, 0 none
    int nst;              // G3 rows staged (the chunk's first ROWMAX rows)
    int pair[MAXPAIRS];   // first row | (second row valid) << 8 | chunk-local prefix << 9
    int g3i[ROWMAX];      // i3 of the staged rows (read by the G3 stager)
  };
  static constexpr int NCW = NC / CW;                // stage-2 columns per consumer warp
  // consumers, lead producer, NCOPY G2 copiers and NSTAGE G3 stagers sharing
  // a stage's copies row by row (one warp issuing all of them paces the pipeline)
  static constexpr int NCOPY = 2, NSTAGE = 2;
  static constexpr int THREADS = 32 * (CW + 1 + NCOPY + NSTAGE);
  static constexpr int SMEM = 4 * (2 * STAGE_F + F_P2) + 2 * (int)sizeof(Meta) + 8 * 8 + 16;
  static_assert(CW == 8 || CW == 16, "8 or 16 consumer warps");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(MAXROWS <= 256 && CP <= 8 && 4 * CP <= 32, "pair encoding and G1 staging");
};

// P2 rows (p, j1) = 16 MT tiles x 256 columns (j2, r2); consumer warp w owns
// columns 32 w .. 32 w + 31.  bf16 three-term tiles from the staged planes:
// A = G1 rows [(p, j1)][r1] (plain ldmatrix), B = G2 [r1][(j2, r2)] (transposed).
template <int CW, int MT>
__device__ __forceinline__ void mma_fwd_stage2(const float* __restrict__ G2s,
                                               const float* __restrict__ P1n,
                                               float* __restrict__ P2, int warp, int lane) {
  using C = MmaFwd<CW>;
  static_assert(C::NCW == 32, "eight consumer warps");
  const int g = lane >> 2, t = lane & 3;
  const uint32_t g2h = smem_addr(G2s), g2l = g2h + C::G2PLANE;
  const uint32_t g1h = smem_addr(P1n), g1l = g1h + C::G1PLANE;
  float acc[MT][4][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
  const int col0 = warp * C::NCW;
#pragma unroll
  for (int ks = 0; ks < C::R / 16; ++ks) {
    uint32_t ah[MT][4], al[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      ldsm_x4(ah[mt], a_addr_mk(g1h, C::G1LD, 16 * mt, 16 * ks, lane));
      ldsm_x4(al[mt], a_addr_mk(g1l, C::G1LD, 16 * mt, 16 * ks, lane));
    }
#pragma unroll
    for (int np2 = 0; np2 < 2; ++np2) {
      uint32_t bh[4], bl[4];
      ldsm_x4_t(bh, b2_addr_kn(g2h, C::G2LD, 16 * ks, col0 + 16 * np2, lane));
      ldsm_x4_t(bl, b2_addr_kn(g2l, C::G2LD, 16 * ks, col0 + 16 * np2, lane));
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          mma_bf16x3(acc[mt][2 * np2 + h], ah[mt], al[mt], bh[2 * h], bh[2 * h + 1], bl[2 * h], bl[2 * h + 1]);
    }
  }
  // row (p, j1) = 16 mt + g (+8), columns (j2, r2) = (warp, 8 nt + 2t (+1))
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = 16 * mt + g + 8 * h;
      char* dst = reinterpret_cast<char*>(P2) + (row >> 2) * C::PPB + (row & 3) * C::PA + warp * C::PB + 4 * t;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        uint32_t hi, lo;
        split_bf16x2(acc[mt][nt][2 * h], acc[mt][nt][2 * h + 1], hi, lo);
        *reinterpret_cast<uint32_t*>(dst + 16 * nt) = hi;
        *reinterpret_cast<uint32_t*>(dst + 16 * nt + C::P2PLANE) = lo;
      }
    }
}

// Rows of the chunk, by pairs.  Consumer warp w takes m-tile w % 2 (j12 =
// 16 (w % 2) .. +15) of a contiguous share of the pairs, so that consecutive
// pairs of one prefix reuse the warp's P2 fragments.  bf16 m16n8k16 tiles:
// A[j12][r2] = P2 planes (plain ldmatrix), B[r2][(row of pair, j3)] from the
// staged G3 planes [j3][r2] per row (plain ldmatrix, rows (row, j3); a missing
// second row reads the zero row), or, for rows past the first ROWMAX, 32-bit
// pairs loaded from the global split planes.
template <int CW>
__device__ __forceinline__ void mma_fwd_stage3(const typename MmaFwd<CW>::Meta& m, uint32_t P2h,
                                               uint32_t G3h, const uint16_t* __restrict__ g3th,
                                               const uint16_t* __restrict__ g3tl,
                                               const int32_t* __restrict__ row_i3, float* __restrict__ rowbuf,
                                               int warp, int lane) {
  using C = MmaFwd<CW>;
  constexpr int SH = CW / 2;                        // warps per m-tile
  const int g = lane >> 2, t = lane & 3;
  const int mt = warp & 1, share = warp >> 1;
  const int npairs = m.npairs, x0 = m.x0;
  const int q0 = npairs * share / SH, q1 = npairs * (share + 1) / SH;
  const int li = lane >> 3, lr = lane & 7;
  int cur_p = -1;
  uint32_t ah[2][4], al[2][4];
  for (int q = q0; q < q1; ++q) {
    const int e = m.pair[q];
    const int r0 = e & 255, has2 = (e >> 8) & 1, p = e >> 9;
    if (p != cur_p) {
      cur_p = p;
      // matrix li: rows j12 = 16 mt + 8 (li & 1) + lr (j1 = 2 mt + (li & 1), j2 = lr),
      // columns r2 = 16 ks + 8 (li >> 1)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint32_t aa = P2h + p * C::PPB + (2 * mt + (li & 1)) * C::PA + lr * C::PB +
                            2 * (16 * ks + 8 * (li >> 1));
        ldsm_x4(ah[ks], aa);
        ldsm_x4(al[ks], aa + C::P2PLANE);
      }
    }
    float big[4] = {0.f, 0.f, 0.f, 0.f}, small[4] = {0.f, 0.f, 0.f, 0.f};
    if (r0 + 1 < C::ROWMAX) {
      // B rows n = (row of pair, j3) = lr, k columns r2 = 16 ks + 8 ((lane >> 3) & 1)
      const int xr = (lr >> 2) == 0 ? r0 : (has2 ? r0 + 1 : C::ROWMAX);
      const uint32_t bb = G3h + xr * C::GTROW + (lr & 3) * 80 + 16 * (li & 1);
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        uint32_t bh[2], bl[2];
        ldsm_x2(bh, bb + 32 * ks);
        ldsm_x2(bl, bb + 32 * ks + C::GTPLANE);
        mma_bf16(small, al[ks], bh[0], bh[1]);
        mma_bf16(big, ah[ks], bh[0], bh[1]);
        mma_bf16(small, ah[ks], bl[0], bl[1]);
      }
    } else {
      // b0 = {B[k = 2t][n = g], B[2t+1][g]}, b1 = same at k + 8; n = (row g / 4, j3 = g % 4)
      const int xr = r0 + (g >> 2);
      const bool live = (g >> 2) == 0 || has2;
      const size_t base = live ? ((size_t)__ldg(row_i3 + x0 + xr) * 4 + (g & 3)) * C::R : 0;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const size_t k0 = base + 16 * ks + 2 * t;
        const uint32_t bh0 = live ? __ldg(reinterpret_cast<const uint32_t*>(g3th + k0)) : 0u;
        const uint32_t bh1 = live ? __ldg(reinterpret_cast<const uint32_t*>(g3th + k0 + 8)) : 0u;
        const uint32_t bl0 = live ? __ldg(reinterpret_cast<const uint32_t*>(g3tl + k0)) : 0u;
        const uint32_t bl1 = live ? __ldg(reinterpret_cast<const uint32_t*>(g3tl + k0 + 8)) : 0u;
        mma_bf16(small, al[ks], bh0, bh1);
        mma_bf16(big, ah[ks], bh0, bh1);
        mma_bf16(small, ah[ks], bl0, bl1);
      }
    }
    // C[j12][(row of pair, j3)]: this lane holds j3 = 2 (t % 2), +1 of row t / 2
    if (t < 2 || has2) {
      float* o = rowbuf + (size_t)(x0 + r0 + (t >> 1)) * C::D + (16 * mt + g) * 4 + 2 * (t & 1);
      *reinterpret_cast<float2*>(o) = make_float2(small[0] + big[0], small[1] + big[1]);
      *reinterpret_cast<float2*>(o + 32) = make_float2(small[2] + big[2], small[3] + big[3]);
    }
  }
}

template <int CW>
__global__ void __launch_bounds__(MmaFwd<CW>::THREADS, 1) k_fwd_mma(FwdArgs a) {
  using C = MmaFwd<CW>;
  using Meta = typename C::Meta;
  extern __shared__ float4 sm4[];
  float* base = reinterpret_cast<float*>(sm4);
  float* P2 = base + 2 * C::STAGE_F;
  Meta* meta = reinterpret_cast<Meta*>(P2 + C::F_P2);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + 2);
  uint64_t* empty = full + 2;
  uint64_t* go = empty + 2;                          // lead producer -> G2 copier, per stage
  uint64_t* go3 = go + 2;                            // lead producer -> G3 stager, per stage
  volatile int* slot = reinterpret_cast<volatile int*>(go3 + 2);  // the stage's i2, or -1: stop
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    // full: the copy arrivals of the producer warps' lanes + the lead's metadata
    // arrival
    mbar_init(&full[0], 32 * (1 + C::NCOPY + C::NSTAGE) + 1);
    mbar_init(&full[1], 32 * (1 + C::NCOPY + C::NSTAGE) + 1);
    mbar_init(&empty[0], 1);
    mbar_init(&empty[1], 1);
    mbar_init(&go[0], 1);
    mbar_init(&go[1], 1);
    mbar_init(&go3[0], 1);
    mbar_init(&go3[1], 1);
    mbar_init_fence();
    if (blockIdx.x == 0) mark_split(a.w.ctl, a.G1, a.G2, a.G3);
  }
  // the zero row (row ROWMAX) of the staged G3 planes of both stages
  for (int e = tid; e < 2 * 2 * (C::GTROW / 16); e += C::THREADS) {
    const int st = e / (2 * (C::GTROW / 16)), rem = e - st * 2 * (C::GTROW / 16);
    const int plane = rem / (C::GTROW / 16), q = rem - plane * (C::GTROW / 16);
    char* row = reinterpret_cast<char*>(base + st * C::STAGE_F + C::F_G2 + C::F_P1) + plane * C::GTPLANE +
                C::ROWMAX * C::GTROW;
    *reinterpret_cast<uint4*>(row + 16 * q) = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  const int n_chunks = a.w.ctl->n_chunks;
  // L2 checkpoint of prefix partials: a hot prefix is split into CR-row pieces;
  // its first piece writes its P2 planes to a slot (owner word: CAS from 0 to
  // prefix + 1) and sets the slot's ready word to prefix + 1; a later piece that
  // finds the ready word set loads P2 from the slot instead of forming it again,
  // and recomputes it otherwise (nothing ever waits for a slot).  The claim
  // order puts later pieces after all other chunks, so their first piece is
  // usually done.  Slots lie in the unique-row buffer past the batch's unique
  // rows (below its zero row); their words are zeroed by every grouping.
  const int64_t U_r = a.w.ctl->U_r;
  const int64_t ck_fit = (a.w.rowbuf_rows - U_r) * (int64_t)C::D * 4 / C::CKB;
  const int n_slots = (int)(ck_fit < 0 ? 0 : (ck_fit > kCkptSlots ? kCkptSlots : ck_fit));
  char* ck_data = reinterpret_cast<char*>(a.w.rowbuf + (size_t)U_r * C::D);
  uint32_t* ck_owner = a.w.ckpt;
  uint32_t* ck_ready = a.w.ckpt + kCkptSlots;

  if (warp >= CW + 1 + C::NCOPY) {
    // ---------------- G3 stagers: stage the chunk's first ROWMAX G3 rows (the
    // transposed split planes; the lead producer lists their i3 in the stage's
    // metadata), stager h the rows h, h + NSTAGE, ..., per row lane = plane |
    // j3 | 16-byte piece
    const int h = warp - (CW + 1 + C::NCOPY);
    for (int it = 0;; ++it) {
      const int s = it & 1;
      if (!mbar_wait(&go3[s], ((uint32_t)it >> 1) & 1, a.w.ctl)) break;
      const int i2 = slot[s];
      if (i2 != -1) {
        const Meta& mg = meta[s];
        const int nst = mg.nst;
        char* G3s = reinterpret_cast<char*>(base + s * C::STAGE_F + C::F_G2 + C::F_P1);
        const int plane = lane >> 4, j3 = (lane >> 2) & 3, q = lane & 3;
        const uint16_t* src = plane ? a.w.g3tl : a.w.g3th;
        for (int r0 = h; r0 < nst; r0 += 8 * C::NSTAGE) {
#pragma unroll
          for (int u = 0; u < 8 * C::NSTAGE; u += C::NSTAGE)
            if (r0 + u < nst)
              cp_async16(G3s + plane * C::GTPLANE + (r0 + u) * C::GTROW + j3 * 80 + 16 * q,
                         src + ((size_t)mg.g3i[r0 + u] * 4 + j3) * C::R + 8 * q);
        }
      }
      cp_async_arrive_noinc(&full[s]);
      if (i2 == -1) break;
    }
    cp_async_wait_all();
    return;
  }

  if (warp >= CW + 1) {
    // ---------------- G2 copiers: stage the G2 planes of the chunks the lead
    // producer hands over, one stage at a time; the 64 rows of the two planes
    // (hi, lo) are dealt to the copiers, copier h taking rows h, h + NCOPY, ...
    const int h = warp - (CW + 1);
    for (int it = 0;; ++it) {
      const int s = it & 1;
      if (!mbar_wait(&go[s], ((uint32_t)it >> 1) & 1, a.w.ctl)) break;
      const int i2 = slot[s];        // the G2 slice, -1: stop, -2 - k: checkpoint slot k
      if (i2 >= 0) {
        const size_t at = (size_t)i2 * C::R * C::NC;
        char* dst = reinterpret_cast<char*>(base + s * C::STAGE_F);
#pragma unroll 8
        for (int pr = h; pr < 2 * C::R; pr += C::NCOPY) {   // lane: 16-byte piece of a 512-byte row
          const int plane = pr / C::R, row = pr - plane * C::R;
          cp_async16(dst + plane * C::G2PLANE + row * (2 * C::G2LD) + 16 * lane,
                     (plane ? a.w.g2l : a.w.g2h) + at + row * C::NC + 8 * lane);
        }
      } else if (i2 <= -2) {
        // a checkpointed P2 into the stage's G2 area, in the P2 layout (planes
        // P2PLANE apart), where the consumers' stage 3 reads it
        const char* src = ck_data + (size_t)(-2 - i2) * C::CKB;
        char* dst = reinterpret_cast<char*>(base + s * C::STAGE_F);
        for (int e = lane + 32 * h; e < C::CKB / 16; e += 32 * C::NCOPY) {
          const int plane = e / (C::PPB / 16), q = e - plane * (C::PPB / 16);
          cp_async16(dst + plane * C::P2PLANE + 16 * q, src + plane * C::PPB + 16 * q);
        }
      }
      cp_async_arrive_noinc(&full[s]);
      if (i2 == -1) break;
    }
    cp_async_wait_all();
    return;
  }

  if (warp == CW) {
    // ---------------- lead producer.  Software-pipelined: while chunk i is staged,
    // the metadata loads of chunk i+1 and the claim of chunk i+2 are in flight.
    // The G2 copier is released for a stage only once that stage is free.
    auto release = [&](int s, int i2) {
      __syncwarp();
      if (lane == 0) {
        slot[s] = i2;
        mbar_arrive(&go[s]);
        mbar_arrive(&go3[s]);
      }
    };
    // The metadata of a chunk, as loaded (every field a plain load or
    // register arithmetic, so that issuing them does not wait for any)
    struct PMeta {
      int x0, x1, p0, np, nst, i2;
      int g30, g31;    // i3 of staged rows lane, lane + 32
      int gi1, prs;    // lane < np: i1 and first row of prefix p0 + lane (else prs = x1)
    };
    auto load_meta = [&](const ChunkDesc& d, PMeta& pm) {
      pm.x0 = d.x0;
      pm.x1 = d.x1;
      pm.p0 = d.p0;
      pm.np = d.p1 - d.p0 + 1;
      const int rows = d.x1 - d.x0;
      pm.nst = min(rows, C::ROWMAX);
      pm.g30 = lane < pm.nst ? a.w.row_i3[d.x0 + lane] : 0;
      pm.g31 = lane + 32 < pm.nst ? a.w.row_i3[d.x0 + lane + 32] : 0;
      pm.gi1 = 0;
      pm.prs = d.x1;
      if (lane < pm.np) {
        pm.gi1 = a.w.pair_i1[d.p0 + lane];
        pm.prs = a.w.pair_row_start[d.p0 + lane];
      }
      pm.i2 = a.w.pair_i2[d.p0];
    };
    // The c-th claim takes chunk chunk_order[c].  Every dependent step of a
    // chunk's bookkeeping gets one iteration of slack: the claim of chunk k + 3
    // is issued at the start of iteration k and read at its end, when the load
    // of its order entry is issued; chunk k + 2's descriptor is loaded late in
    // iteration k from that entry, chunk k + 1's metadata at its start, and
    // chunk k + 1's checkpoint role (ready check or slot claim) is decided from
    // its descriptor during iteration k.
    const int32_t* order = a.w.chunk_order;
    uint32_t* ctr = &a.w.ctl->fwd_chunk_ctr;
    int c = claim_chunk(ctr), cn = claim_chunk(ctr), cnn = claim_chunk(ctr);
    ChunkDesc d0{}, dn{};
    if (c < n_chunks) d0 = load_chunk(a.w.chunk_desc, order[c]);
    if (cn < n_chunks) dn = load_chunk(a.w.chunk_desc, order[cn]);
    int onn = cnn < n_chunks ? order[cnn] : 0;
    PMeta cur{}, nxt{};
    if (c < n_chunks) load_meta(d0, cur);
    // checkpoint role of one chunk: 0 none, s + 1 writes slot s, -(s + 1) reads it
    // (lane 0 issues the check; `resolve` reads its result)
    auto role_issue = [&](const ChunkDesc& d, int& kind, int& sl, uint32_t& v) {
      kind = 0;
      sl = 0;
      v = 0;
      if (n_slots > 0 && d.p1 == d.p0) {
        sl = d.p0 % n_slots;
        if (!d.whole) {                 // a later piece: reuse the slot if it is ready
          kind = 1;
          if (lane == 0) v = ld_acquire_u32(ck_ready + sl);
        } else if (d.cont) {            // the first piece of a hot prefix: checkpoint its P2
          kind = 2;
          if (lane == 0) v = atomicCAS(ck_owner + sl, 0u, (uint32_t)d.p0 + 1u);
        }
      }
    };
    auto role_resolve = [&](const ChunkDesc& d, int kind, int sl, uint32_t v) {
      v = __shfl_sync(0xffffffffu, v, 0);
      if (kind == 1 && v == (uint32_t)d.p0 + 1u) return -(sl + 1);
      if (kind == 2 && v == 0u) return sl + 1;
      return 0;
    };
    int ck_cur = 0;
    if (c < n_chunks) {
      int kind, sl;
      uint32_t v;
      role_issue(d0, kind, sl, v);
      ck_cur = role_resolve(d0, kind, sl, v);
    }
    for (int it = 0;; ++it) {
      const int s = it & 1;
      const uint32_t use = (uint32_t)it >> 1;
      Meta& m = meta[s];
      if (c >= n_chunks) {
        const bool ok = use == 0 || mbar_wait(&empty[s], (use - 1) & 1, a.w.ctl);
        release(s, -1);
        if (!ok) break;
        if (lane == 0) m.end = 1;
        __syncwarp();
        cp_async_arrive_noinc(&full[s]);
        if (lane == 0) mbar_arrive(&full[s]);
        break;
      }
      if (cn < n_chunks) load_meta(dn, nxt);
      uint32_t tk = 0;
      if (lane == 0) tk = atomicAdd(ctr, 1u);
      int kind_n = 0, sl_n = 0;
      uint32_t v_n = 0;
      if (cn < n_chunks) role_issue(dn, kind_n, sl_n, v_n);
      if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, a.w.ctl)) {
        release(s, -1);
        break;
      }
      const int ck = ck_cur;
      if (ck < 0 && lane == 0) atomicAdd(&a.w.ctl->ckpt_reused, 1);
      // the i3 of the rows the G3 stager stages for this chunk
      if (lane < cur.nst) m.g3i[lane] = cur.g30;
      if (lane + 32 < cur.nst) m.g3i[lane + 32] = cur.g31;
      if (lane == 0) m.nst = cur.nst;
      release(s, ck < 0 ? -1 + ck : cur.i2);   // -2 - slot: the copier loads the checkpoint
      float* G2s = base + s * C::STAGE_F;
      float* P1n = G2s + C::F_G2;
      // G1[i1_p] planes: per prefix, lane = plane | j1 | piece (not for a reused P2)
#pragma unroll
      for (int pp = 0; pp < C::CP; ++pp) {
        const int i1 = __shfl_sync(0xffffffffu, cur.gi1, pp);
        const int plane = lane >> 4, j1 = (lane >> 2) & 3, q = lane & 3;
        if (pp < cur.np && ck >= 0)
          cp_async16(reinterpret_cast<char*>(P1n) + plane * C::G1PLANE + (4 * pp + j1) * (2 * C::G1LD) + 16 * q,
                     (plane ? a.w.g1l : a.w.g1h) + ((size_t)i1 * 4 + j1) * C::R + 8 * q);
      }
      cp_async_arrive_noinc(&full[s]);
      // pairs: a row starts a pair when its offset within its prefix is even;
      // the list follows row order (prefix after prefix)
      int rsq[C::CP];
#pragma unroll
      for (int j = 0; j < C::CP; ++j)   // chunk-local first row of each prefix (rows past the last)
        rsq[j] = max(__shfl_sync(0xffffffffu, cur.prs, j), cur.x0) - cur.x0;
      const int rows = cur.x1 - cur.x0;
      int npairs = 0;
      for (int rb = 0; rb < rows; rb += 32) {
        const int r = rb + lane;
        int q = -1, qs = 0, qe = rows;
#pragma unroll
        for (int j = 0; j < C::CP; ++j) {
          if (rsq[j] <= r) {
            ++q;
            qs = rsq[j];
          } else {
            qe = min(qe, rsq[j]);
          }
        }
        const bool start = r < rows && ((r - qs) & 1) == 0;
        const unsigned bal = __ballot_sync(0xffffffffu, start);
        if (start)
          m.pair[npairs + __popc(bal & ((1u << lane) - 1u))] = r | ((r + 1 < qe) ? 256 : 0) | (q << 9);
        npairs += __popc(bal);
      }
      __syncwarp();
      if (lane == 0) {
        m.x0 = cur.x0;
        m.x1 = cur.x1;
        m.p0 = cur.p0;
        m.np = cur.np;
        m.npairs = npairs;
        m.end = 0;
        m.ck = ck;
        mbar_arrive(&full[s]);
      }
      ChunkDesc dnn{};
      if (cnn < n_chunks) dnn = load_chunk(a.w.chunk_desc, onn);
      const int ck_nxt = cn < n_chunks ? role_resolve(dn, kind_n, sl_n, v_n) : 0;
      const int c3 = __shfl_sync(0xffffffffu, (int)tk, 0);
      const int onew = c3 < n_chunks ? order[c3] : 0;
      c = cn;
      cur = nxt;
      ck_cur = ck_nxt;
      cn = cnn;
      dn = dnn;
      cnn = c3;
      onn = onew;
    }
    cp_async_wait_all();
    return;
  }

  // ---------------- consumers: warps 0 .. CW-1
  for (int k = 0;; ++k) {
    const int s = k & 1;
    if (!mbar_wait(&full[s], ((uint32_t)k >> 1) & 1, a.w.ctl)) break;
    const Meta& m = meta[s];
    if (m.end) break;
    const float* G2s = base + s * C::STAGE_F;
    const float* P1n = G2s + C::F_G2;
    const float* G3s = P1n + C::F_P1;
    const int ck = m.ck;
    if (ck >= 0) {
      if (m.np > 4) mma_fwd_stage2<CW, 2>(G2s, P1n, P2, warp, lane);
      else mma_fwd_stage2<CW, 1>(G2s, P1n, P2, warp, lane);
      named_sync(1, 32 * CW);
      if (ck > 0) {                 // checkpoint: the prefix's P2 planes to slot ck - 1
        char* dst = ck_data + (size_t)(ck - 1) * C::CKB;
        for (int e = tid; e < C::CKB / 16; e += 32 * CW) {
          const int plane = e / (C::PPB / 16), q = e - plane * (C::PPB / 16);
          *reinterpret_cast<uint4*>(dst + plane * C::PPB + 16 * q) =
              *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(P2) + plane * C::P2PLANE + 16 * q);
        }
      }
      mma_fwd_stage3<CW>(m, smem_addr(P2), smem_addr(G3s), a.w.g3th, a.w.g3tl, a.w.row_i3, a.w.rowbuf, warp, lane);
    } else {                        // P2 from the checkpoint, staged in the G2 area
      mma_fwd_stage3<CW>(m, smem_addr(G2s), smem_addr(G3s), a.w.g3th, a.w.g3tl, a.w.row_i3, a.w.rowbuf, warp, lane);
    }
    named_sync(1, 32 * CW);
    if (ck > 0 && tid == 0) {       // the slot's planes are written: publish them
      __threadfence();
      st_release_u32(ck_ready + ck - 1, (uint32_t)m.p0 + 1u);
    }
    if (tid == 0) mbar_arrive(&empty[s]);
  }
}

// out[b] = pooled unique rows of bag b's lookups; one warp per bag.  The
// lanes fetch up to 32 of the bag's unique-row ids (and weights) at once; each
// lane then sums its float4 column of those rows, 8 loads in flight.  MODE
// (PoolMode): plain sum, sum with each row scaled by its lookup's per-sample
// weight, or the sum divided by the bag's length (empty bags give zeros).
// The bag of every lookup is written on the way (bag_of, for the backward).

// The weight of lookup l (MODE kPoolWeighted), 0 for an out-of-range lookup.
template <int MODE>
__device__ __forceinline__ float pool_weight(const float* __restrict__ psw, int64_t l, int32_t u) {
  return (MODE == kPoolWeighted && u >= 0) ? psw[l] : 1.f;
}

template <int MODE>
__device__ __forceinline__ void pool_mean(float4& acc, int64_t len) {
  if (MODE == kPoolMean && len > 0) {
    const float f = (float)len;
    acc.x /= f; acc.y /= f; acc.z /= f; acc.w /= f;
  }
}

template <int MODE>
__global__ void __launch_bounds__(256) k_pool(const int64_t* __restrict__ offsets, int64_t B,
                                              int64_t nnz, const int32_t* __restrict__ uid,
                                              const float* __restrict__ psw,
                                              const float* __restrict__ rowbuf, int D,
                                              float* __restrict__ out, int32_t* __restrict__ bag_of) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < B; b += warps) {
    int64_t l0 = offsets[b], l1 = offsets[b + 1];
    l0 = l0 < 0 ? 0 : (l0 > nnz ? nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > nnz ? nnz : l1);
    for (int64_t l = l0 + lane; l < l1; l += 32) bag_of[l] = (int32_t)b;
    if ((D & 3) == 0) {
      const int cols = D >> 2;
      const float4* rb4 = reinterpret_cast<const float4*>(rowbuf);
      for (int c0 = 0; c0 < cols; c0 += 32) {
        const int c = c0 + lane;
        const bool live = c < cols;
        float4 acc = z4;
        for (int64_t lb = l0; lb < l1; lb += 32) {
          const int cnt = (int)(l1 - lb < 32 ? l1 - lb : 32);
          const int32_t my_u = lane < cnt ? uid[lb + lane] : -1;
          const float my_w = lane < cnt ? pool_weight<MODE>(psw, lb + lane, my_u) : 0.f;
          int j = 0;
          for (; j + 8 <= cnt; j += 8) {
            float4 v[8];
            float wt[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const int32_t u = __shfl_sync(0xffffffffu, my_u, j + t);
              wt[t] = __shfl_sync(0xffffffffu, my_w, j + t);
              v[t] = (live && u >= 0) ? rb4[(int64_t)u * cols + c] : z4;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              if (MODE == kPoolWeighted) f4fma(acc, wt[t], v[t]);
              else f4add(acc, v[t]);
            }
          }
          for (; j < cnt; ++j) {
            const int32_t u = __shfl_sync(0xffffffffu, my_u, j);
            const float wj = __shfl_sync(0xffffffffu, my_w, j);
            if (live && u >= 0) {
              if (MODE == kPoolWeighted) f4fma(acc, wj, rb4[(int64_t)u * cols + c]);
              else f4add(acc, rb4[(int64_t)u * cols + c]);
            }
          }
        }
        pool_mean<MODE>(acc, l1 - l0);
        if (live) reinterpret_cast<float4*>(out + b * (int64_t)D)[c] = acc;
      }
    } else {
      for (int j = lane; j < D; j += 32) {
        float acc = 0.f;
        for (int64_t l = l0; l < l1; ++l) {
          const int u = uid[l];
          if (u >= 0) {
            if (MODE == kPoolWeighted) acc = fmaf(psw[l], rowbuf[(int64_t)u * D + j], acc);
            else acc += rowbuf[(int64_t)u * D + j];
          }
        }
        if (MODE == kPoolMean && l1 > l0) acc /= (float)(l1 - l0);
        out[b * (int64_t)D + j] = acc;
      }
    }
  }
}

// Pooling for D = 128: every lane owns one float4 column, so the inner loop
// needs no column checks; lookups with an out-of-range index point at the zero
// row `zrow` (weight 0); full batches of 8 row loads run unpredicated.
constexpr int kPoolThreads = 128, kPoolCtasPerSm = 9;
template <int MODE>
__global__ void __launch_bounds__(kPoolThreads, MODE == kPoolWeighted ? 1 : kPoolCtasPerSm) k_pool128(const int64_t* __restrict__ offsets, int64_t B64,
                                                    int64_t nnz64, const int32_t* __restrict__ uid,
                                                    const float* __restrict__ psw,
                                                    const float4* __restrict__ rb4, int32_t zrow,
                                                    float4* __restrict__ out,
                                                    int32_t* __restrict__ bag_of) {
  // bags < 2^31 and lookups < 2^30, so positions fit in 32 bits (fewer
  // registers: 36 warps per SM instead of 32); an offset is read by its low word
  // (little-endian) and clamped to [0, nnz], which keeps every access in
  // bounds even for offsets the grouping reported as bad
  const int B = (int)B64, nnz = (int)nnz64;
  const int32_t* __restrict__ off32 = reinterpret_cast<const int32_t*>(offsets);
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  for (int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < B; b += warps) {
    int l0 = off32[2 * (int64_t)b], l1 = off32[2 * (int64_t)b + 2];
    l0 = l0 < 0 ? 0 : (l0 > nnz ? nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > nnz ? nnz : l1);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int lb = l0; lb < l1; lb += 32) {
      const int cnt = l1 - lb < 32 ? l1 - lb : 32;
      int32_t my_u = lane < cnt ? uid[lb + lane] : zrow;
      if (lane < cnt) bag_of[lb + lane] = b;
      float my_w = 0.f;
      if (MODE == kPoolWeighted) my_w = (lane < cnt && my_u >= 0) ? psw[lb + lane] : 0.f;
      my_u = my_u < 0 ? zrow : my_u;
      int j = 0;
      for (; j + 8 <= cnt; j += 8) {
        float4 v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) v[t] = rb4[(int64_t)__shfl_sync(0xffffffffu, my_u, j + t) * 32 + lane];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (MODE == kPoolWeighted) f4fma(acc, __shfl_sync(0xffffffffu, my_w, j + t), v[t]);
          else f4add(acc, v[t]);
        }
      }
      for (; j < cnt; ++j) {
        const float4 v = rb4[(int64_t)__shfl_sync(0xffffffffu, my_u, j) * 32 + lane];
        if (MODE == kPoolWeighted) f4fma(acc, __shfl_sync(0xffffffffu, my_w, j), v);
        else f4add(acc, v);
      }
    }
    pool_mean<MODE>(acc, l1 - l0);
    out[(int64_t)b * 32 + lane] = acc;
  }
}

static size_t fwd_generic_smem(const Shape& s, int CP) {
  return sizeof(float) * ((size_t)s.R1 * s.n2 * s.R2 +
                          (size_t)CP * (s.n1 * s.R1 + s.n1 * s.n2 * s.R2));
}

// Which chunk kernel serves a shape, and its chunking parameters.
enum FwdKind { kFwdGeneric = 0, kFwdMma_8_32, kFwdMma_8_64, kFwdTiled_4_16 };

static FwdKind fwd_kind(const Shape& s) {
  if (tc_shape(s)) return kFwdMma_8_32;
  if (tc64_shape(s)) return kFwdMma_8_64;
  if (s.n1 == 4 && s.n3 == 4 && s.n2 == 4 && s.R1 == 16 && s.R2 == 16) return kFwdTiled_4_16;
  return kFwdGeneric;
}

int forward_chunk_params(const Shape& s, int* pairs_per_chunk, int* rows_per_chunk) {
  const int64_t g2n = (int64_t)s.R1 * s.n2 * s.R2;
  const int64_t per = (int64_t)s.n1 * s.R1 + (int64_t)s.n1 * s.n2 * s.R2;
  if (g2n + per + (int64_t)s.n1 * s.n2 * s.R2 > kMaxSmemFloats) return TT_EMB_ERR_UNSUPPORTED;
  int64_t cp = (kMaxSmemFloats - g2n) / per;
  if (cp > 16) cp = 16;
  if (cp < 1) cp = 1;
  switch (fwd_kind(s)) {
    case kFwdMma_8_32: cp = kCP_8_32; break;
    case kFwdMma_8_64: cp = kCP_8_64; break;
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

template <int CW>
static void launch_fwd_mma(const FwdArgs& fa, cudaStream_t st) {
  using C = MmaFwd<CW>;
  static int grid = 0;
  if (grid == 0) {
    cudaFuncSetAttribute(k_fwd_mma<CW>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    grid = persistent_grid((const void*)k_fwd_mma<CW>, C::THREADS, C::SMEM);
  }
  TT_TIMED("k_fwd_mma", st, (k_fwd_mma<CW><<<grid, C::THREADS, C::SMEM, st>>>(fa)));
}

template <int N2, int R, int CP>
static void launch_tiled(const TiledTables& tt, cudaStream_t st) {
  using T = TileCfg<N2, R, CP>;
  static int grid = 0;
  if (grid == 0) {
    cudaFuncSetAttribute(k_fwd_tiled<N2, R, CP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         T::SMEM);
    grid = persistent_grid((const void*)k_fwd_tiled<N2, R, CP>, 256, T::SMEM);
  }
  TT_TIMED("k_fwd_tiled", st, (k_fwd_tiled<N2, R, CP><<<grid, 256, T::SMEM, st>>>(tt)));
}


int launch_rows(const Shape& s, const WS& w, const float* const cores[3], int presplit,
                cudaStream_t st) {
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
    case kFwdMma_8_32:
      if (!presplit) {
        rc = launch_split(s, w, cores, 0, st);
        if (rc) return rc;
      }
      launch_fwd_mma<8>(fa, st);
      break;
    case kFwdMma_8_64: {
      if (!presplit) {
        rc = launch_split(s, w, cores, 0, st);
        if (rc) return rc;
      }
      const float* const* c3 = cores;
      return launch_fwd_mma64(1, &w, &c3, st);
    }
    case kFwdTiled_4_16: {
      TiledTables tt;
      tt.t[0] = fa;
      tt.T = 1;
      launch_tiled<4, 16, kCP_4_16>(tt, st);
      break;
    }
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
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

template <int MODE>
static void launch_pool_mode(const Shape& s, const Layout& L, const WS& w, const int64_t* offsets,
                             int64_t nnz, int64_t num_bags, const float* psw, float* out,
                             cudaStream_t st) {
  int grid = (int)ceil_div(num_bags, 8);
  const int cap = sm_count() * 16;
  if (grid > cap) grid = cap;
  if (s.D == 128) {
    // two full waves of 4-warp CTAs, each warp taking bags by grid stride
    grid = (int)ceil_div(num_bags, kPoolThreads / 32);
    const int cap128 = sm_count() * kPoolCtasPerSm * 2;
    if (grid > cap128) grid = cap128;
    TT_TIMED("k_pool", st, (k_pool128<MODE><<<grid, kPoolThreads, 0, st>>>(
                               offsets, num_bags, nnz, w.uid, psw,
                               reinterpret_cast<const float4*>(w.rowbuf), (int32_t)L.rowbuf_rows,
                               reinterpret_cast<float4*>(out), w.bag_of)));
  } else {
    TT_TIMED("k_pool", st, (k_pool<MODE><<<grid, 256, 0, st>>>(offsets, num_bags, nnz, w.uid, psw,
                                                                w.rowbuf, s.D, out, w.bag_of)));
  }
}

int launch_forward(const Shape& s, const Layout& L, const WS& w, const float* const cores[3],
                   const int64_t* offsets, int64_t nnz, int64_t num_bags, const Pooling& pool,
                   int presplit, float* out, cudaStream_t st) {
  int rc = launch_rows(s, w, cores, presplit, st);
  if (rc) return rc;
  if (num_bags > 0) {
    switch (pool.mode) {
      case kPoolWeighted:
        launch_pool_mode<kPoolWeighted>(s, L, w, offsets, nnz, num_bags, pool.psw, out, st);
        break;
      case kPoolMean:
        launch_pool_mode<kPoolMean>(s, L, w, offsets, nnz, num_bags, nullptr, out, st);
        break;
      default: launch_pool_mode<kPoolSum>(s, L, w, offsets, nnz, num_bags, nullptr, out, st);
    }
  }
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

// Sum pooling of several tables (D = 128) in one launch: bags are numbered
// across the tables (bag_base[t] = first bag of table t), each warp takes bags
// by grid stride and pools them as k_pool128<kPoolSum> does (4-warp CTAs,
// 32-bit positions, offsets read by their low word and clamped).
struct PoolTables {
  const int64_t* offsets[kMaxTables];
  int32_t nnz[kMaxTables];
  const int32_t* uid[kMaxTables];
  const float4* rb4[kMaxTables];
  int32_t zrow[kMaxTables];
  float4* out[kMaxTables];
  int32_t* bag_of[kMaxTables];
  int32_t bag_base[kMaxTables + 1];
  int T;
};

__global__ void __launch_bounds__(kPoolThreads, kPoolCtasPerSm)
    k_pool128_tables(const __grid_constant__ PoolTables pt) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int total = pt.bag_base[pt.T];
  for (int g = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); g < total; g += warps) {
    int t = 0;
    while (t + 1 < pt.T && g >= pt.bag_base[t + 1]) ++t;
    const int b = g - pt.bag_base[t], nnz = pt.nnz[t];
    const int32_t* off32 = reinterpret_cast<const int32_t*>(pt.offsets[t]);
    int l0 = off32[2 * (int64_t)b], l1 = off32[2 * (int64_t)b + 2];
    l0 = l0 < 0 ? 0 : (l0 > nnz ? nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > nnz ? nnz : l1);
    const int32_t* uid = pt.uid[t];
    const float4* rb4 = pt.rb4[t];
    const int32_t zrow = pt.zrow[t];
    int32_t* bag_of = pt.bag_of[t];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int lb = l0; lb < l1; lb += 32) {
      const int cnt = l1 - lb < 32 ? l1 - lb : 32;
      int32_t my_u = lane < cnt ? uid[lb + lane] : zrow;
      if (lane < cnt) bag_of[lb + lane] = b;
      my_u = my_u < 0 ? zrow : my_u;
      int j = 0;
      for (; j + 8 <= cnt; j += 8) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) v[u] = rb4[(int64_t)__shfl_sync(0xffffffffu, my_u, j + u) * 32 + lane];
#pragma unroll
        for (int u = 0; u < 8; ++u) f4add(acc, v[u]);
      }
      for (; j < cnt; ++j) f4add(acc, rb4[(int64_t)__shfl_sync(0xffffffffu, my_u, j) * 32 + lane]);
    }
    pt.out[t][(int64_t)b * 32 + lane] = acc;
  }
}

int launch_forward_tables(int T, const Shape* s, const Layout* L, const WS* w,
                          const float* const* const* cores, const int64_t* const* offsets,
                          const int64_t* nnz, const int64_t* num_bags, float* const* out,
                          int presplit, cudaStream_t st) {
  const FwdKind kind = fwd_kind(s[0]);
  if (kind != kFwdMma_8_64 && kind != kFwdTiled_4_16) {
    for (int t = 0; t < T; ++t) {
      if (nnz[t] == 0) continue;
      const Pooling pool{kPoolSum, nullptr};
      const int rc = launch_forward(s[t], L[t], w[t], cores[t], offsets[t], nnz[t], num_bags[t],
                                    pool, presplit, out[t], st);
      if (rc) return rc;
    }
    return TT_EMB_OK;
  }
  if (kind == kFwdMma_8_64) {
    // the split of every table with lookups, then one launch over all their chunks
    WS wt[kMaxTables];
    const float* const* ct[kMaxTables];
    int n = 0;
    for (int t = 0; t < T; ++t) {
      if (nnz[t] == 0) continue;
      if (!presplit) {
        const int rc = launch_split(s[t], w[t], cores[t], 0, st);
        if (rc) return rc;
      }
      wt[n] = w[t];
      ct[n++] = cores[t];
    }
    if (n > 0) {
      const int rc = launch_fwd_mma64(n, wt, ct, st);
      if (rc) return rc;
    }
  } else {
    TiledTables tt;
    tt.T = 0;
    for (int t = 0; t < T; ++t) {
      if (nnz[t] == 0) continue;
      FwdArgs& fa = tt.t[tt.T++];
      fa.s = s[t];
      fa.w = w[t];
      fa.G1 = cores[t][0];
      fa.G2 = cores[t][1];
      fa.G3 = cores[t][2];
    }
    if (tt.T > 0) launch_tiled<4, 16, kCP_4_16>(tt, st);
  }
  if (s[0].D == 128) {
    // the pooling of every table with lookups in one launch
    PoolTables pt;
    pt.T = 0;
    pt.bag_base[0] = 0;
    for (int t = 0; t < T; ++t) {
      if (nnz[t] == 0 || num_bags[t] == 0) continue;
      const int k = pt.T++;
      pt.offsets[k] = offsets[t];
      pt.nnz[k] = (int32_t)nnz[t];
      pt.uid[k] = w[t].uid;
      pt.rb4[k] = reinterpret_cast<const float4*>(w[t].rowbuf);
      pt.zrow[k] = (int32_t)L[t].rowbuf_rows;
      pt.out[k] = reinterpret_cast<float4*>(out[t]);
      pt.bag_of[k] = w[t].bag_of;
      pt.bag_base[k + 1] = pt.bag_base[k] + (int32_t)num_bags[t];
    }
    if (pt.T > 0) {
      // two full waves of 4-warp CTAs, as for one table
      int grid = (int)ceil_div(pt.bag_base[pt.T], kPoolThreads / 32);
      const int cap = sm_count() * kPoolCtasPerSm * 2;
      if (grid > cap) grid = cap;
      TT_TIMED("k_pool", st, (k_pool128_tables<<<grid, kPoolThreads, 0, st>>>(pt)));
    }
  } else {
    for (int t = 0; t < T; ++t)
      if (nnz[t] > 0 && num_bags[t] > 0)
        launch_pool_mode<kPoolSum>(s[t], L[t], w[t], offsets[t], nnz[t], num_bags[t], nullptr,
                                   out[t], st);
  }
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
