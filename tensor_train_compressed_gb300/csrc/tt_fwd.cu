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
    tiled_load_g2_p1<T>(a.G1, a.G2, a.w.pair_i1, i2, p0, np, G2s, P1t);
    __syncthreads();
    tiled_stage2_any<T>(G2s, P1t, P2, np);
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

// ---------------------------------------------------------------------------
// Warp-specialised chunk kernel (n1 = n3 = 4, R1 = R2 = R, G2 slice small enough
// to double-buffer).  Warp 8 is a producer: it claims the next chunk, writes the
// chunk's metadata and issues bulk copies (TMA, 1-D) of the G2 slice, the G1
// rows and up to ROWMAX G3 rows into the free one of two stage buffers,
// completing on that buffer's "full" mbarrier.  Warps 0-7 consume: stage 2
// (P2 in shared memory), stage 3 (rows), then release the buffer through its
// "empty" mbarrier.  Staging of chunk i+1 thus overlaps the math of chunk i.
template <int N2, int R, int CP, int GROUPS = 1>
struct WsCfg {
  using T = TileCfg<N2, R, CP>;
  static constexpr int THREADS = GROUPS * 256 + 32;
  static constexpr int ROWMAX = 64;
  static constexpr int F_P1 = CP * 4 * R;            // G1 rows, natural [p][j1][a]
  static constexpr int F_G3 = ROWMAX * T::G3S;
  static constexpr int STAGE_F = T::F_G2 + F_P1 + F_G3;
  struct Meta {
    int x0, x1, p0, np, end, pad[3];
    int rp[ROWMAX];                                   // prefix (chunk-local) of each staged row
  };
  static constexpr int SMEM =
      4 * (2 * STAGE_F + GROUPS * (T::F_P2 + F_P1)) + 2 * (int)sizeof(Meta) + 4 * 8;
  static_assert(T::NB == 8, "one compute warp per j12 block");
  static_assert(GROUPS == 1 || GROUPS == 2, "one or two consumer groups");
  static_assert(ROWMAX <= 64 && CP <= 32, "the producer stages with two rows per lane");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

// acc[i][j3] = sum over b in [b0, b0 + NBV) of P2[j12 = 4 blk + i][b] G3[b][j3]
template <class T, bool kGlobalG3, int NBV = T::kR>
__device__ __forceinline__ void row_dot(const float* __restrict__ pp,
                                        const float* __restrict__ gg, float acc[4][4],
                                        int b0 = 0) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 2
  for (int b = b0; b < b0 + NBV; b += 4) {
    float4 pv[4], gv[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pv[i] = *reinterpret_cast<const float4*>(pp + i * T::P2S + b);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if constexpr (kGlobalG3) gv[t] = __ldg(reinterpret_cast<const float4*>(gg + (b + t) * 4));
      else gv[t] = *reinterpret_cast<const float4*>(gg + (b + t) * 4);
    }
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
}

template <class T, int SPLIT>
__device__ __forceinline__ void stage3_split(const float* __restrict__ P2,
                                             const float* __restrict__ G3s,
                                             const int* __restrict__ rp, float* __restrict__ rowbuf,
                                             int x0, int rows, int blk, int lane) {
  constexpr int NBV = T::kR / SPLIT;
  const int r = lane / SPLIT, q = lane % SPLIT;
  float acc[4][4];
  if (r < rows) {
    const float* pp = P2 + rp[r] * T::P2P + (blk * 4) * T::P2S;
    row_dot<T, false, NBV>(pp, G3s + r * T::G3S, acc, q * NBV);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  }
#pragma unroll
  for (int o = 1; o < SPLIT; o <<= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] += __shfl_xor_sync(0xffffffffu, acc[i][j], o);
  if (r < rows) {
    float4* out = reinterpret_cast<float4*>(rowbuf + (size_t)(x0 + r) * T::D + blk * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i % SPLIT == q) out[i] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
}

// With GROUPS = 2 there are two consumer groups of 8 warps: group g owns stage
// buffer g (and its own P2), so the producer's stages alternate between the
// groups and two chunks are in flight per SM.
template <int N2, int R, int CP, int GROUPS>
__global__ void __launch_bounds__(WsCfg<N2, R, CP, GROUPS>::THREADS, 1) k_fwd_ws(FwdArgs a) {
  using W = WsCfg<N2, R, CP, GROUPS>;
  using T = typename W::T;
  using Meta = typename W::Meta;
  extern __shared__ float4 sm4[];
  float* base = reinterpret_cast<float*>(sm4);
  float* P2all = base + 2 * W::STAGE_F;
  float* P1tall = P2all + GROUPS * T::F_P2;
  Meta* meta = reinterpret_cast<Meta*>(P1tall + GROUPS * W::F_P1);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + 2);
  uint64_t* empty = full + 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&empty[0], 1);
    mbar_init(&empty[1], 1);
    mbar_init_fence();
  }
  __syncthreads();
  const int n_chunks = a.w.ctl->n_chunks;

  if (warp == 8 * GROUPS) {
    // ---------------- producer: claims one chunk ahead, so that the claim and
    // the descriptor load of chunk i+1 overlap the staging of chunk i
    auto end_stage = [&](int it) {          // end marker into the stage of iteration it
      const int s = it & 1;
      const uint32_t use = (uint32_t)it >> 1;
      if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, a.w.ctl)) return;
      if (lane == 0) {
        meta[s].end = 1;
        mbar_arrive(&full[s]);
      }
    };
    int c = claim_chunk(&a.w.ctl->fwd_chunk_ctr);
    ChunkDesc d{};
    if (c < n_chunks) d = load_chunk(a.w.chunk_desc, c);
    for (int it = 0;; ++it) {
      const int s = it & 1;
      const uint32_t use = (uint32_t)it >> 1;
      Meta& m = meta[s];
      if (c >= n_chunks) {
        end_stage(it);
        if (GROUPS == 2) end_stage(it + 1);   // the other group's stage too
        break;
      }
      const int x0 = d.x0, x1 = d.x1, p0 = d.p0;
      const int np = d.p1 - p0 + 1;
      const int nst = min(x1 - x0, W::ROWMAX);
      // metadata of this chunk (loads in flight while the stage frees up)
      int rp0 = 0, rp1 = 0, g30 = 0, g31 = 0, gi1 = 0;
      if (lane < nst) {
        rp0 = a.w.row_pair[x0 + lane] - p0;
        g30 = a.w.row_i3[x0 + lane];
      }
      if (lane + 32 < nst) {
        rp1 = a.w.row_pair[x0 + lane + 32] - p0;
        g31 = a.w.row_i3[x0 + lane + 32];
      }
      if (lane < np) gi1 = a.w.pair_i1[p0 + lane];
      const int i2 = a.w.pair_i2[p0];
      // claim the next chunk and fetch its descriptor
      const int cn = claim_chunk(&a.w.ctl->fwd_chunk_ctr);
      ChunkDesc dn{};
      if (cn < n_chunks) dn = load_chunk(a.w.chunk_desc, cn);
      if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, a.w.ctl)) break;
      float* G2s = base + s * W::STAGE_F;
      float* P1n = G2s + T::F_G2;
      float* G3s = P1n + W::F_P1;
      if (lane < nst) m.rp[lane] = rp0;
      if (lane + 32 < nst) m.rp[lane + 32] = rp1;
      __syncwarp();
      if (lane == 0) {
        m.x0 = x0;
        m.x1 = x1;
        m.p0 = p0;
        m.np = np;
        m.end = 0;
        const uint32_t bytes = 4u * (T::F_G2 + np * 4 * R + nst * 4 * R);
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(G2s, a.G2 + (size_t)i2 * T::F_G2, 4u * T::F_G2, &full[s]);
      }
      __syncwarp();
      if (lane < np) bulk_g2s(P1n + lane * 4 * R, a.G1 + (size_t)gi1 * 4 * R, 16u * R, &full[s]);
      if (lane < nst) bulk_g2s(G3s + lane * T::G3S, a.G3 + (size_t)g30 * 4 * R, 16u * R, &full[s]);
      if (lane + 32 < nst)
        bulk_g2s(G3s + (lane + 32) * T::G3S, a.G3 + (size_t)g31 * 4 * R, 16u * R, &full[s]);
      c = cn;
      d = dn;
    }
    return;
  }

  // ---------------- consumers: group g = warps 8g .. 8g+7
  const int g = warp >> 3, ltid = tid - 256 * g, blk = warp & 7;
  const int bar_id = 1 + g;
  float* P2 = P2all + g * T::F_P2;
  float* P1t = P1tall + g * W::F_P1;
  for (int k = 0;; ++k) {
    // GROUPS == 1: both stages in turn; GROUPS == 2: stage g only
    const int s = GROUPS == 1 ? (k & 1) : g;
    const uint32_t parity = GROUPS == 1 ? (((uint32_t)k >> 1) & 1) : ((uint32_t)k & 1);
    if (!mbar_wait(&full[s], parity, a.w.ctl)) break;
    const Meta& m = meta[s];
    if (m.end) break;
    const int x0 = m.x0, x1 = m.x1, p0 = m.p0, np = m.np;
    const float* G2s = base + s * W::STAGE_F;
    const float* P1n = G2s + T::F_G2;
    const float* G3s = P1n + W::F_P1;
    stage2_natural<T>(G2s, P1n, P1t, P2, np, ltid, bar_id);
    const int rows = x1 - x0;
    if (rows <= 16) {
      // few rows: SPLIT lanes share a row, each over R/SPLIT of the b sum
      if (rows <= 8) stage3_split<T, 4>(P2, G3s, m.rp, a.w.rowbuf, x0, rows, blk, lane);
      else stage3_split<T, 2>(P2, G3s, m.rp, a.w.rowbuf, x0, rows, blk, lane);
    } else {
      for (int r = lane; r < rows; r += 32) {
        const int x = x0 + r;
        float acc[4][4];
        if (r < W::ROWMAX) {
          const float* pp = P2 + m.rp[r] * T::P2P + (blk * 4) * T::P2S;
          row_dot<T, false>(pp, G3s + r * T::G3S, acc);
        } else {
          const float* pp = P2 + (a.w.row_pair[x] - p0) * T::P2P + (blk * 4) * T::P2S;
          row_dot<T, true>(pp, a.G3 + (size_t)a.w.row_i3[x] * 4 * R, acc);
        }
        float4* o = reinterpret_cast<float4*>(a.w.rowbuf + (size_t)x * T::D + blk * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      }
    }
    named_sync(bar_id, 256);
    if (ltid == 0) mbar_arrive(&empty[s]);
  }
}

// out[b] = sum of the unique rows of bag b's lookups; one warp per bag.  The
// lanes fetch up to 32 of the bag's unique-row ids at once; each lane then sums
// its float4 column of those rows, 8 loads in flight.

__global__ void __launch_bounds__(256) k_pool(const int64_t* __restrict__ offsets, int64_t B,
                                              int64_t nnz, const int32_t* __restrict__ uid,
                                              const float* __restrict__ rowbuf, int D,
                                              float* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < B; b += warps) {
    int64_t l0 = offsets[b], l1 = offsets[b + 1];
    l0 = l0 < 0 ? 0 : (l0 > nnz ? nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > nnz ? nnz : l1);
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
          int j = 0;
          for (; j + 8 <= cnt; j += 8) {
            float4 v[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
              const int32_t u = __shfl_sync(0xffffffffu, my_u, j + t);
              v[t] = (live && u >= 0) ? rb4[(int64_t)u * cols + c] : z4;
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) f4add(acc, v[t]);
          }
          for (; j < cnt; ++j) {
            const int32_t u = __shfl_sync(0xffffffffu, my_u, j);
            if (live && u >= 0) f4add(acc, rb4[(int64_t)u * cols + c]);
          }
        }
        if (live) reinterpret_cast<float4*>(out + b * (int64_t)D)[c] = acc;
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

// Pooling for D = 128: every lane owns one float4 column, so the inner loop
// needs no column checks; lookups with an out-of-range index point at the zero
// row `zrow`; full batches of 8 row loads run unpredicated.
__global__ void __launch_bounds__(256) k_pool128(const int64_t* __restrict__ offsets, int64_t B,
                                                 int64_t nnz, const int32_t* __restrict__ uid,
                                                 const float4* __restrict__ rb4, int32_t zrow,
                                                 float4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < B; b += warps) {
    int64_t l0 = offsets[b], l1 = offsets[b + 1];
    l0 = l0 < 0 ? 0 : (l0 > nnz ? nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > nnz ? nnz : l1);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t lb = l0; lb < l1; lb += 32) {
      const int cnt = (int)(l1 - lb < 32 ? l1 - lb : 32);
      int32_t my_u = lane < cnt ? uid[lb + lane] : zrow;
      my_u = my_u < 0 ? zrow : my_u;
      int j = 0;
      for (; j + 8 <= cnt; j += 8) {
        float4 v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) v[t] = rb4[(int64_t)__shfl_sync(0xffffffffu, my_u, j + t) * 32 + lane];
#pragma unroll
        for (int t = 0; t < 8; ++t) f4add(acc, v[t]);
      }
      for (; j < cnt; ++j) f4add(acc, rb4[(int64_t)__shfl_sync(0xffffffffu, my_u, j) * 32 + lane]);
    }
    out[b * 32 + lane] = acc;
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

template <int N2, int R, int CP, int GROUPS>
static void launch_ws(const FwdArgs& fa, cudaStream_t st) {
  using W = WsCfg<N2, R, CP, GROUPS>;
  static int grid = 0;
  if (grid == 0) {
    cudaFuncSetAttribute(k_fwd_ws<N2, R, CP, GROUPS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         W::SMEM);
    grid = persistent_grid((const void*)k_fwd_ws<N2, R, CP, GROUPS>, W::THREADS, W::SMEM);
  }
  TT_TIMED("k_fwd_ws", st, (k_fwd_ws<N2, R, CP, GROUPS><<<grid, W::THREADS, W::SMEM, st>>>(fa)));
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
    case kFwdTiled_8_32: launch_ws<8, 32, kCP_8_32, 1>(fa, st); break;
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
    if (s.D == 128) {
      TT_TIMED("k_pool", st, (k_pool128<<<grid, 256, 0, st>>>(
                                 offsets, num_bags, nnz, w.uid, reinterpret_cast<const float4*>(w.rowbuf),
                                 (int32_t)L.rowbuf_rows, reinterpret_cast<float4*>(out))));
    } else {
      TT_TIMED("k_pool", st, (k_pool<<<grid, 256, 0, st>>>(offsets, num_bags, nnz, w.uid, w.rowbuf, s.D, out)));
    }
  }
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
