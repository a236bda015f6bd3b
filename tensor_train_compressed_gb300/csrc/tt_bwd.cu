// Backward TT embedding bag into the three cores, and the SGD update.
//
// The gradient of <grad_out, out> (FlowTT reports training latency, so the
// cores are trained; summary card, evaluation; abstract).  With the grouping
// of the forward:
//
//   S[x]          = sum of grad_out[bag(l)] over the lookups l of unique row x
//   dG3[i3_x]    += P2[p(x)]^T . S[x]              (R2 x n1n2).(n1n2 x n3)
//   dP2[p]        = sum_x S[x] . G3[i3_x]^T         (n1n2 x n3).(n3 x R2)
//   dG2[i2]      += P1[p]^T . dP2[p]               (R1 x n1).(n1 x n2R2)
//   dG1[i1_p]    += dP2[p] . G2[i2]^T              (n1 x n2R2).(n2R2 x R1)
//
// P2 is recomputed per chunk from the cores (it is never stored).  S is
// gathered slice by slice over the sorted lookups; a row that crosses a slice
// boundary is accumulated with atomics into a zeroed row, all others are
// stored once.  Core gradients are accumulated with float atomics.
#include "tt_internal.cuh"
#include "tt_tile.cuh"

namespace tt {

// Zero the S rows that more than one gather slice will add into, write the bag
// of every lookup (CSR offsets, one warp per bag, clamped so that bad offsets
// stay in bounds) and reset the backward chunk counter.
__global__ void __launch_bounds__(256) k_s_zero(WS w, int D, const int64_t* __restrict__ offsets,
                                                int64_t B, int64_t nnz, int span) {
  if (blockIdx.x == 0 && threadIdx.x == 0) w.ctl->bwd_chunk_ctr = 0;
  const int U = w.ctl->U_r;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int64_t u = gw; u < U; u += warps) {
    const int32_t s0 = w.row_start[u], s1 = w.row_start[u + 1];
    if (s0 / span != (s1 - 1) / span) {
      float* r = w.rowbuf + u * (int64_t)D;
      for (int j = lane; j < D; j += 32) r[j] = 0.f;
    }
  }
  for (int64_t b = gw; b < B; b += warps) {
    int64_t l0 = offsets[b], l1 = offsets[b + 1];
    l0 = l0 < 0 ? 0 : (l0 > nnz ? nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > nnz ? nnz : l1);
    for (int64_t l = l0 + lane; l < l1; l += 32) w.bag_of[l] = (int32_t)b;
  }
}

__device__ __forceinline__ void s_flush(const WS& w, int32_t u, int64_t k0, int c, int D,
                                        float4 acc, bool vec, float accs) {
  const int32_t s0 = w.row_start[u], s1 = w.row_start[u + 1];
  const bool shared_row = s0 < k0 || s1 > k0 + kSSlice;
  if (vec) {
    float4* dst = reinterpret_cast<float4*>(w.rowbuf + u * (int64_t)D) + c;
    if (shared_row) atomicAdd(dst, acc);
    else *dst = acc;
  } else {
    float* dst = w.rowbuf + u * (int64_t)D + c;
    if (shared_row) atomicAdd(dst, accs);
    else *dst = accs;
  }
}

// S[x] for every unique row: one warp per slice of kSSlice sorted lookups.  The
// lanes fetch the slice's (unique row, bag) pairs in parallel, 32 at a time; the
// output-gradient rows are then summed with 8 loads in flight, flushing at every
// change of unique row.
__global__ void __launch_bounds__(256) k_s_gather(WS w, const float* __restrict__ grad_out,
                                                  int64_t B, int D) {
  const int lane = threadIdx.x & 31;
  const int64_t nv = w.ctl->n_valid;
  const int64_t k0 = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kSSlice;
  if (k0 >= nv) return;
  const int64_t k1 = k0 + kSSlice < nv ? k0 + kSSlice : nv;
  const bool vec = (D & 3) == 0;
  const int cols = vec ? (D >> 2) : D;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < cols; c0 += 32) {
    const int c = c0 + lane;
    const bool live = c < cols;
    float4 acc = z4;
    float accs = 0.f;
    int32_t cur = -1;
    for (int64_t kb = k0; kb < k1; kb += 32) {
      const int cnt = (int)(k1 - kb < 32 ? k1 - kb : 32);
      int32_t my_u = -1, my_b = 0;
      if (lane < cnt) {
        const int32_t l = w.perm[kb + lane];
        my_u = w.uid[l];
        const int32_t bb = w.bag_of[l];
        my_b = bb < 0 ? 0 : (bb >= B ? (int32_t)(B - 1) : bb);
      }
      for (int j = 0; j < cnt; j += 8) {
        int32_t uj[8];
        float4 g[8];
        float gs[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int jj = (j + t) & 31;
          uj[t] = __shfl_sync(0xffffffffu, my_u, jj);
          const int32_t bj = __shfl_sync(0xffffffffu, my_b, jj);
          const bool use = live && (j + t) < cnt;
          g[t] = z4;
          gs[t] = 0.f;
          if (use) {
            if (vec) g[t] = __ldg(reinterpret_cast<const float4*>(grad_out + bj * (int64_t)D) + c);
            else gs[t] = __ldg(grad_out + bj * (int64_t)D + c);
          }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (j + t >= cnt) break;
          if (uj[t] != cur) {
            if (cur >= 0 && live) s_flush(w, cur, k0, c, D, acc, vec, accs);
            acc = z4;
            accs = 0.f;
            cur = uj[t];
          }
          acc.x += g[t].x; acc.y += g[t].y; acc.z += g[t].z; acc.w += g[t].w;
          accs += gs[t];
        }
      }
    }
    if (cur >= 0 && live) s_flush(w, cur, k0, c, D, acc, vec, accs);
  }
}

// S[x] with the partial sums of rows that cross warp boundaries merged inside
// the CTA: a CTA covers kSCta = 8 x kSSlice sorted positions; each warp sums
// the runs of its kSSlice positions (8 output-gradient rows in flight), stores
// the runs that start and end inside its range, and leaves its first and last
// run in shared memory; one warp then merges those in position order and
// stores each merged row, or adds it with float atomics (into a row zeroed by
// k_s_zero) when the row also crosses the CTA's range.  D % 4 == 0.
constexpr int kSCta = 8 * kSSlice;

__device__ __forceinline__ void s_merge_flush(const WS& w, int32_t u, int64_t K0, const float4& m,
                                              int lane) {
  const int32_t s0 = w.row_start[u], s1 = w.row_start[u + 1];
  float4* dst = reinterpret_cast<float4*>(w.rowbuf) + (int64_t)u * 32 + lane;
  if (s0 < K0 || s1 > K0 + kSCta) atomicAdd(dst, m);
  else *dst = m;
}

// D = 128: every lane owns one float4 column of the rows.
__global__ void __launch_bounds__(256) k_s_gather_cta(WS w, const float* __restrict__ grad_out,
                                                      int64_t B) {
  __shared__ float4 part[8][2][32];
  __shared__ int part_u[8][2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nv = w.ctl->n_valid;
  const int64_t K0 = (int64_t)blockIdx.x * kSCta;
  if (K0 >= nv) return;                                // uniform over the CTA
  const int64_t K1 = K0 + kSCta < nv ? K0 + kSCta : nv;
  const int64_t k0 = K0 + (int64_t)warp * kSSlice;
  const int64_t k1 = k0 + kSSlice < K1 ? k0 + kSSlice : K1;
  const float4* g4 = reinterpret_cast<const float4*>(grad_out);
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 acc = z4;
  int32_t cur = -1, first_u = -1;
  bool first_open = true;                              // the warp's first run is still open
  if (lane < 2) part_u[warp][lane] = -1;
  auto close_run = [&]() {
    if (cur < 0) return;
    if (first_open) {                                  // the first run: keep for the merge
      part[warp][0][lane] = acc;
      first_u = cur;
      first_open = false;
    } else {                                           // a run inside the warp's range
      reinterpret_cast<float4*>(w.rowbuf)[(int64_t)cur * 32 + lane] = acc;
    }
  };
  for (int64_t kb = k0; kb < k1; kb += 32) {
    const int cnt = (int)(k1 - kb < 32 ? k1 - kb : 32);
    int32_t my_u = -1, my_b = 0;
    if (lane < cnt) {
      const int32_t l = w.perm[kb + lane];
      my_u = w.uid[l];
      const int32_t bb = w.bag_of[l];
      my_b = bb < 0 ? 0 : (bb >= B ? (int32_t)(B - 1) : bb);
    }
    int j = 0;
    for (; j + 8 <= cnt; j += 8) {
      int32_t uj[8];
      float4 g[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        uj[t] = __shfl_sync(0xffffffffu, my_u, j + t);
        g[t] = __ldg(g4 + (int64_t)__shfl_sync(0xffffffffu, my_b, j + t) * 32 + lane);
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (uj[t] != cur) {
          close_run();
          acc = z4;
          cur = uj[t];
        }
        f4add(acc, g[t]);
      }
    }
    for (; j < cnt; ++j) {
      const int32_t u = __shfl_sync(0xffffffffu, my_u, j);
      const float4 g = __ldg(g4 + (int64_t)__shfl_sync(0xffffffffu, my_b, j) * 32 + lane);
      if (u != cur) {
        close_run();
        acc = z4;
        cur = u;
      }
      f4add(acc, g);
    }
  }
  // the last run (or the only one)
  if (cur >= 0) {
    if (first_open) {
      part[warp][0][lane] = acc;
      first_u = cur;
    } else {
      part[warp][1][lane] = acc;
      if (lane == 0) part_u[warp][1] = cur;
    }
  }
  if (lane == 0) part_u[warp][0] = first_u;
  __syncthreads();
  if (warp == 0) {
    int32_t mu = -1;
    float4 m = z4;
    for (int ww = 0; ww < 8; ++ww)
      for (int e = 0; e < 2; ++e) {
        const int32_t u = part_u[ww][e];
        if (u < 0) continue;
        if (u != mu) {
          if (mu >= 0) s_merge_flush(w, mu, K0, m, lane);
          mu = u;
          m = z4;
        }
        f4add(m, part[ww][e][lane]);
      }
    if (mu >= 0) s_merge_flush(w, mu, K0, m, lane);
  }
}

struct BwdArgs {
  Shape s;
  WS w;
  const float* G1;
  const float* G2;
  const float* G3;
  float* dG1;
  float* dG2;
  float* dG3;
  int dG2_in_smem;   // accumulate the chunk's dG2[i2] in shared memory first
};

// Shape-generic backward chunk kernel; prefixes of a chunk are handled one by one.
__global__ void __launch_bounds__(256) k_bwd_generic(BwdArgs a) {
  extern __shared__ float4 sm4[];
  float* sm = reinterpret_cast<float*>(sm4);
  __shared__ int c_sh;
  const Shape& s = a.s;
  const int tid = threadIdx.x;
  const int g2n = s.R1 * s.n2 * s.R2;
  const int p1n = s.n1 * s.R1;
  const int n2R2 = s.n2 * s.R2;
  const int p2n = s.n1 * n2R2;
  const int n12 = s.n1 * s.n2;
  const int n1 = s.n1, n2 = s.n2, n3 = s.n3, R1 = s.R1, R2 = s.R2, D = s.D;
  float* G2s = sm;
  float* P1s = G2s + g2n;
  float* P2s = P1s + p1n;
  float* dP2s = P2s + p2n;
  float* dG2s = dP2s + p2n;   // only if a.dG2_in_smem
  const int n_chunks = a.w.ctl->n_chunks;
  for (;;) {
    if (tid == 0) c_sh = (int)atomicAdd(&a.w.ctl->bwd_chunk_ctr, 1u);
    __syncthreads();
    const int c = c_sh;
    if (c >= n_chunks) break;
    const int x0 = a.w.chunk_start[c], x1 = a.w.chunk_start[c + 1];
    const int p0 = a.w.row_pair[x0], p1 = a.w.row_pair[x1 - 1];
    const int i2 = a.w.pair_i2[p0];
    const float* g2 = a.G2 + (size_t)i2 * g2n;
    for (int e = tid; e < g2n; e += blockDim.x) {
      G2s[e] = __ldg(g2 + e);
      if (a.dG2_in_smem) dG2s[e] = 0.f;
    }
    for (int p = p0; p <= p1; ++p) {
      const int i1 = a.w.pair_i1[p];
      for (int e = tid; e < p1n; e += blockDim.x) P1s[e] = __ldg(a.G1 + (size_t)i1 * p1n + e);
      __syncthreads();
      for (int e = tid; e < p2n; e += blockDim.x) {
        const int j1 = e / n2R2, j2b = e - j1 * n2R2;
        float acc = 0.f;
        for (int aa = 0; aa < R1; ++aa) acc = fmaf(P1s[j1 * R1 + aa], G2s[aa * n2R2 + j2b], acc);
        P2s[e] = acc;
      }
      __syncthreads();
      const int pr0 = a.w.pair_row_start[p], pr1 = a.w.pair_row_start[p + 1];
      const int xa = pr0 > x0 ? pr0 : x0, xb = pr1 < x1 ? pr1 : x1;
      // dG3 contributions of the prefix's rows in this chunk
      for (int e = tid; e < (xb - xa) * R2 * n3; e += blockDim.x) {
        const int xi = e / (R2 * n3), rem = e - xi * (R2 * n3);
        const int b = rem / n3, j3 = rem - b * n3;
        const int x = xa + xi;
        const float* S = a.w.rowbuf + (size_t)x * D + j3;
        float acc = 0.f;
        for (int j12 = 0; j12 < n12; ++j12) acc = fmaf(P2s[j12 * R2 + b], S[j12 * n3], acc);
        atomicAdd(a.dG3 + ((size_t)a.w.row_i3[x] * R2 + b) * n3 + j3, acc);
      }
      // dP2 of the prefix from the same rows
      for (int e = tid; e < p2n; e += blockDim.x) {
        const int j12 = e / R2, b = e - j12 * R2;
        float acc = 0.f;
        for (int x = xa; x < xb; ++x) {
          const float* S = a.w.rowbuf + (size_t)x * D + j12 * n3;
          const float* g3 = a.G3 + ((size_t)a.w.row_i3[x] * R2 + b) * n3;
          for (int j3 = 0; j3 < n3; ++j3) acc = fmaf(S[j3], __ldg(g3 + j3), acc);
        }
        dP2s[e] = acc;
      }
      __syncthreads();
      // dG2[i2][a][j2][b] += sum_j1 P1[j1][a] dP2[j1][j2][b]
      for (int e = tid; e < g2n; e += blockDim.x) {
        const int aa = e / n2R2, j2b = e - aa * n2R2;
        float acc = 0.f;
        for (int j1 = 0; j1 < n1; ++j1) acc = fmaf(P1s[j1 * R1 + aa], dP2s[j1 * n2R2 + j2b], acc);
        if (a.dG2_in_smem) dG2s[e] += acc;
        else atomicAdd(a.dG2 + (size_t)i2 * g2n + e, acc);
      }
      // dG1[i1][j1][a] += sum_{j2,b} dP2[j1][j2][b] G2[a][j2][b]
      for (int e = tid; e < p1n; e += blockDim.x) {
        const int j1 = e / R1, aa = e - j1 * R1;
        float acc = 0.f;
        for (int j2b = 0; j2b < n2R2; ++j2b)
          acc = fmaf(dP2s[j1 * n2R2 + j2b], G2s[aa * n2R2 + j2b], acc);
        atomicAdd(a.dG1 + (size_t)i1 * p1n + e, acc);
      }
      __syncthreads();
    }
    if (a.dG2_in_smem) {
      for (int e = tid; e < g2n; e += blockDim.x) atomicAdd(a.dG2 + (size_t)i2 * g2n + e, dG2s[e]);
    }
    __syncthreads();
  }
  (void)n2;
}

// ---------------------------------------------------------------------------
// Warp-specialised backward chunk kernel (n1 = n3 = 4, R1 = R2 = R).  Warp 8 is a
// producer: for the next chunk it writes the metadata and bulk-copies (TMA,
// 1-D) the G2 slice, the G1 rows and the S and G3 rows of the first RB rows into
// the free one of two stage buffers.  Warps 0-7 consume: P2 (stage 2), then per
// batch of RB rows dG3 (float4 atomics) and dP2 (shared memory), then
// dG2 = P1^T dP2 and dG1 = dP2 G2^T.  A chunk that starts a hot prefix takes all
// of that prefix's rows (later batches are loaded by the consumers into the
// already consumed row area); chunks holding its later pieces are skipped.
template <int N2, int R, int CP>
struct BwsCfg {
  using T = TileCfg<N2, R, CP>;
  static constexpr int RB = 32;
  static constexpr int SS = T::D + 4;                 // padded S row (floats)
  static constexpr int GS = 4 * R + 4;                // padded G3 row, natural [b][j3]
  static constexpr int F_P1 = CP * 4 * R;             // natural [p][j1][a]
  static constexpr int STAGE_F = T::F_G2 + F_P1 + RB * (SS + GS);
  struct Meta {
    int x0, x1, p0, np, end, nst, i2, pad;
    int rp[RB];
    int ri3[RB];
    int pi1[CP + (CP & 1)];   // even count keeps the barriers that follow 8-byte aligned
  };
  static constexpr int SMEM = 4 * (2 * STAGE_F + 2 * T::F_P2) + 2 * (int)sizeof(Meta) + 4 * 8;
  static_assert(RB * R <= 4 * 256, "in-place G3 transpose: 4 float4 per thread");
  static constexpr int TILES = T::NB * (R / 4);
  static constexpr int RG = 256 / TILES;
  static_assert(T::NB == 8 && 256 % TILES == 0 && RB % RG == 0, "mappings");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

template <class T, class C, int SPLIT>
__device__ __forceinline__ void bwd_dg3(const float* __restrict__ P2, const float* __restrict__ Ss,
                                        const int* __restrict__ rp, const int* __restrict__ ri3,
                                        float* __restrict__ dG3, int nb, int warp, int lane) {
  constexpr int R = T::kR, NJ = 4 * T::kN2 / SPLIT;
  const int r = lane / SPLIT, q = lane % SPLIT;
  for (int bb = warp; bb < R / 4; bb += 8) {
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    if (r < nb) {
      const float* pp = P2 + rp[r] * T::P2P + 4 * bb;
      const float* ss = Ss + r * C::SS;
#pragma unroll 8
      for (int j12 = q * NJ; j12 < (q + 1) * NJ; ++j12) {
        const float4 pv = *reinterpret_cast<const float4*>(pp + j12 * T::P2S);
        const float4 sv = *reinterpret_cast<const float4*>(ss + 4 * j12);
        const float pw[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[i][0] = fmaf(pw[i], sv.x, acc[i][0]);
          acc[i][1] = fmaf(pw[i], sv.y, acc[i][1]);
          acc[i][2] = fmaf(pw[i], sv.z, acc[i][2]);
          acc[i][3] = fmaf(pw[i], sv.w, acc[i][3]);
        }
      }
    }
#pragma unroll
    for (int o = 1; o < SPLIT; o <<= 1)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += __shfl_xor_sync(0xffffffffu, acc[i][j], o);
    if (r < nb) {
      float4* dst = reinterpret_cast<float4*>(dG3 + ((size_t)ri3[r] * R + 4 * bb) * 4);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (i % SPLIT == q)
          atomicAdd(dst + i, make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
    }
  }
}

template <int N2, int R, int CP>
__global__ void __launch_bounds__(288, 1) k_bwd_ws(BwdArgs a) {
  using C = BwsCfg<N2, R, CP>;
  using T = typename C::T;
  using Meta = typename C::Meta;
  constexpr int NC = T::NC, P2S = T::P2S, P2P = T::P2P, D = T::D;
  extern __shared__ float4 sm4[];
  float* base = reinterpret_cast<float*>(sm4);
  float* P2 = base + 2 * C::STAGE_F;
  float* dP2 = P2 + T::F_P2;
  float* P1t = dP2;     // transposed G1 rows live in the dP2 area until stage 2 is done
  Meta* meta = reinterpret_cast<Meta*>(dP2 + T::F_P2);
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

  if (warp == 8) {
    // ---------------- producer: claims one chunk ahead (see the forward kernel);
    // chunks holding a later piece of a hot prefix are skipped
    auto next_chunk = [&](ChunkDesc& d) {
      for (;;) {
        const int c = claim_chunk(&a.w.ctl->bwd_chunk_ctr);
        if (c >= n_chunks) return c;
        d = load_chunk(a.w.chunk_desc, c);
        if (d.whole) return c;
      }
    };
    ChunkDesc d{};
    int c = next_chunk(d);
    for (int it = 0;; ++it) {
      const int s = it & 1;
      const uint32_t use = (uint32_t)it >> 1;
      Meta& m = meta[s];
      if (c >= n_chunks) {
        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, a.w.ctl)) break;
        if (lane == 0) {
          m.end = 1;
          mbar_arrive(&full[s]);
        }
        break;
      }
      const int x0 = d.x0, p0 = d.p0, p1 = d.p1;
      const int x1 = p1 == p0 ? a.w.pair_row_start[p0 + 1] : d.x1;   // a whole hot prefix
      const int np = p1 - p0 + 1;
      const int nst = min(x1 - x0, C::RB);
      int rp = 0, g3 = 0, gi1 = 0;
      if (lane < nst) {
        rp = a.w.row_pair[x0 + lane] - p0;
        g3 = a.w.row_i3[x0 + lane];
      }
      if (lane < np) gi1 = a.w.pair_i1[p0 + lane];
      const int i2 = a.w.pair_i2[p0];
      ChunkDesc dn{};
      const int cn = next_chunk(dn);
      if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, a.w.ctl)) break;
      float* G2s = base + s * C::STAGE_F;
      float* P1n = G2s + T::F_G2;
      float* Ss = P1n + C::F_P1;
      float* G3s = Ss + C::RB * C::SS;
      if (lane < nst) {
        m.rp[lane] = rp;
        m.ri3[lane] = g3;
      }
      if (lane < np) m.pi1[lane] = gi1;
      __syncwarp();
      if (lane == 0) {
        m.x0 = x0;
        m.x1 = x1;
        m.p0 = p0;
        m.np = np;
        m.nst = nst;
        m.i2 = i2;
        m.end = 0;
        const uint32_t bytes = 4u * (T::F_G2 + np * 4 * R + nst * (D + 4 * R));
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(G2s, a.G2 + (size_t)i2 * T::F_G2, 4u * T::F_G2, &full[s]);
      }
      __syncwarp();
      if (lane < np) bulk_g2s(P1n + lane * 4 * R, a.G1 + (size_t)gi1 * 4 * R, 16u * R, &full[s]);
      if (lane < nst) {
        bulk_g2s(Ss + lane * C::SS, a.w.rowbuf + (size_t)(x0 + lane) * D, 4u * D, &full[s]);
        bulk_g2s(G3s + lane * C::GS, a.G3 + (size_t)g3 * 4 * R, 16u * R, &full[s]);
      }
      c = cn;
      d = dn;
    }
    return;
  }

  // ---------------- consumers (warps 0-7)
  for (int it = 0;; ++it) {
    const int s = it & 1;
    if (!mbar_wait(&full[s], ((uint32_t)it >> 1) & 1, a.w.ctl)) break;
    Meta& m = meta[s];
    if (m.end) break;
    const int x0 = m.x0, x1 = m.x1, p0 = m.p0, np = m.np;
    const float* G2s = base + s * C::STAGE_F;
    const float* P1n = G2s + T::F_G2;
    float* Ss = const_cast<float*>(P1n) + C::F_P1;
    float* G3s = Ss + C::RB * C::SS;
    stage2_natural<T>(G2s, P1n, P1t, P2, np);
    for (int e = tid; e < np * P2P; e += 256) dP2[e] = 0.f;

    for (int xb = x0; xb < x1; xb += C::RB) {
      const int nb = min(C::RB, x1 - xb);
      if (xb != x0) {
        // later batches of a hot prefix: the consumers load them into the row area
        named_sync(1, 256);
        if (tid < nb) {
          m.rp[tid] = a.w.row_pair[xb + tid] - p0;
          m.ri3[tid] = a.w.row_i3[xb + tid];
        }
        for (int e = tid; e < nb * (D / 4); e += 256) {
          const int r = e / (D / 4), q = e - r * (D / 4);
          *reinterpret_cast<float4*>(Ss + r * C::SS + 4 * q) =
              reinterpret_cast<const float4*>(a.w.rowbuf + (size_t)(xb + r) * D)[q];
        }
        // G3 rows straight into the transposed [j3][b] layout
        for (int e = tid; e < nb * R; e += 256) {
          const int r = e / R, b = e - r * R;
          const float4 v = __ldg(
              reinterpret_cast<const float4*>(a.G3 + (size_t)a.w.row_i3[xb + r] * 4 * R) + b);
          float* g = G3s + r * C::GS + b;
          g[0] = v.x;
          g[R] = v.y;
          g[2 * R] = v.z;
          g[3 * R] = v.w;
        }
        named_sync(1, 256);
      } else {
        // the staged G3 rows, in place from [b][j3] to [j3][b] (so that the dP2 tiles read
        // 4 consecutive b per 128-bit load)
        float4 v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = tid + 256 * q;
          if (e < nb * R) v[q] = *reinterpret_cast<const float4*>(G3s + (e / R) * C::GS + 4 * (e % R));
        }
        named_sync(1, 256);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = tid + 256 * q;
          if (e < nb * R) {
            float* g = G3s + (e / R) * C::GS + (e % R);
            g[0] = v[q].x;
            g[R] = v[q].y;
            g[2 * R] = v[q].z;
            g[3 * R] = v[q].w;
          }
        }
        named_sync(1, 256);
      }
      // dG3[i3][b][j3] += sum_j12 P2[j12][b] S[j12][j3]: warp = block of 4 b, lane = row
      // (batches of <= 16 / <= 8 rows: 2 / 4 lanes per row split the j12 sum)
      if (nb <= 8) bwd_dg3<T, C, 4>(P2, Ss, m.rp, m.ri3, a.dG3, nb, warp, lane);
      else if (nb <= 16) bwd_dg3<T, C, 2>(P2, Ss, m.rp, m.ri3, a.dG3, nb, warp, lane);
      else bwd_dg3<T, C, 1>(P2, Ss, m.rp, m.ri3, a.dG3, nb, warp, lane);
      // dP2[p][j12][b] += sum_j3 S[j12][j3] G3[b][j3]: tile (4 j12 x 4 b) per thread,
      // row groups walk their rows and flush at every change of prefix
      {
        const int tile = tid % C::TILES, rg = tid / C::TILES;
        const int jb = tile / (R / 4), bq = tile - jb * (R / 4);
        const int r0 = (rg * nb) / C::RG, r1 = ((rg + 1) * nb) / C::RG;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        int cur = -1;
        for (int r = r0; r < r1; ++r) {
          const int pl = m.rp[r];
          if (pl != cur) {
            if (cur >= 0) {
              float* d = dP2 + cur * P2P + (4 * jb) * P2S + 4 * bq;
#pragma unroll
              for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  atomicAdd(d + i * P2S + j, acc[i][j]);
                  acc[i][j] = 0.f;
                }
            }
            cur = pl;
          }
          float4 sv[4], gv[4];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            sv[i] = *reinterpret_cast<const float4*>(Ss + r * C::SS + (4 * jb + i) * 4);
#pragma unroll
          for (int j3 = 0; j3 < 4; ++j3)
            gv[j3] = *reinterpret_cast<const float4*>(G3s + r * C::GS + j3 * R + 4 * bq);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float s4[4] = {sv[i].x, sv[i].y, sv[i].z, sv[i].w};
#pragma unroll
            for (int j3 = 0; j3 < 4; ++j3) {
              acc[i][0] = fmaf(s4[j3], gv[j3].x, acc[i][0]);
              acc[i][1] = fmaf(s4[j3], gv[j3].y, acc[i][1]);
              acc[i][2] = fmaf(s4[j3], gv[j3].z, acc[i][2]);
              acc[i][3] = fmaf(s4[j3], gv[j3].w, acc[i][3]);
            }
          }
        }
        if (cur >= 0) {
          float* d = dP2 + cur * P2P + (4 * jb) * P2S + 4 * bq;
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) atomicAdd(d + i * P2S + j, acc[i][j]);
        }
      }
    }
    named_sync(1, 256);
    // dG2[i2][a][n] += sum_{p, j1} P1[p][j1][a] dP2[p][j1][n]: warp = block of 4 a,
    // lane = 4-column groups at stride 128
    const int i2 = m.i2;
    {
      constexpr int Q = NC / 128;
      for (int ab = warp; ab < R / 4; ab += 8) {
        float acc[4][4 * Q];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4 * Q; ++j) acc[i][j] = 0.f;
        for (int p = 0; p < np; ++p) {
#pragma unroll
          for (int j1 = 0; j1 < 4; ++j1) {
            const float4 a4 = *reinterpret_cast<const float4*>(P1n + p * 4 * R + j1 * R + 4 * ab);
            const float aw[4] = {a4.x, a4.y, a4.z, a4.w};
            float bv[4 * Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) {
              const int n = q * 128 + 4 * lane;
              const int j2 = n / R, b = n - j2 * R;
              const float4 v = *reinterpret_cast<const float4*>(
                  dP2 + p * P2P + (j1 * N2 + j2) * P2S + b);
              bv[4 * q] = v.x; bv[4 * q + 1] = v.y; bv[4 * q + 2] = v.z; bv[4 * q + 3] = v.w;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int j = 0; j < 4 * Q; ++j) acc[i][j] = fmaf(aw[i], bv[j], acc[i][j]);
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            float4* dst = reinterpret_cast<float4*>(
                a.dG2 + (size_t)i2 * T::F_G2 + (size_t)(4 * ab + i) * NC + q * 128 + 4 * lane);
            atomicAdd(dst, make_float4(acc[i][4 * q], acc[i][4 * q + 1], acc[i][4 * q + 2],
                                       acc[i][4 * q + 3]));
          }
      }
    }
    // dG1[i1_p][j1][a] += sum_n dP2[p][j1][n] G2[a][n]: item = (prefix, 4 a, n-slice);
    // the 8 n-slices of an item sit in 8 adjacent lanes and are summed by shuffles
    {
      constexpr int AQ = R / 4;
      const int items = np * AQ * 8;
      for (int b0 = 0; b0 < items; b0 += 256) {
        const int item = b0 + tid;
        const bool valid = item < items;
        const int ns = item & 7, g = item >> 3;
        const int p = g / AQ, aq = g - p * AQ;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
        if (valid) {
          for (int sgrp = 0; sgrp < NC / 32; ++sgrp) {
            const int n = 32 * sgrp + 4 * ns;
            const int j2 = n / R, b = n - j2 * R;
            float4 dv[4], gv[4];
#pragma unroll
            for (int j1 = 0; j1 < 4; ++j1)
              dv[j1] = *reinterpret_cast<const float4*>(dP2 + p * P2P + (j1 * N2 + j2) * P2S + b);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              gv[i] = *reinterpret_cast<const float4*>(G2s + (4 * aq + i) * NC + n);
#pragma unroll
            for (int j1 = 0; j1 < 4; ++j1)
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                float v = acc[j1][i];
                v = fmaf(dv[j1].x, gv[i].x, v);
                v = fmaf(dv[j1].y, gv[i].y, v);
                v = fmaf(dv[j1].z, gv[i].z, v);
                v = fmaf(dv[j1].w, gv[i].w, v);
                acc[j1][i] = v;
              }
          }
        }
#pragma unroll
        for (int j1 = 0; j1 < 4; ++j1)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float v = acc[j1][i];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            acc[j1][i] = v;
          }
        if (valid && ns == 0) {
          const int i1 = m.pi1[p];
#pragma unroll
          for (int j1 = 0; j1 < 4; ++j1)
            atomicAdd(reinterpret_cast<float4*>(a.dG1 + ((size_t)i1 * 4 + j1) * R + 4 * aq),
                      make_float4(acc[j1][0], acc[j1][1], acc[j1][2], acc[j1][3]));
        }
      }
    }
    named_sync(1, 256);
    if (tid == 0) mbar_arrive(&empty[s]);
  }
}

// G_k <- G_k - lr * dG_k for the three cores in one launch (float4 where the
// segment allows), optionally resetting dG_k to zero in the same pass.
struct SgdArgs {
  float* G[3];
  float* dG[3];
  int64_t count[3];
  int64_t start[4];   // prefix of the float4 counts of the segments
  float lr;
  int zero;
};

__global__ void __launch_bounds__(256) k_sgd(SgdArgs a) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < a.start[3]; i += stride) {
    const int k = i < a.start[1] ? 0 : (i < a.start[2] ? 1 : 2);
    const int64_t e = (i - a.start[k]) * 4;
    float* G = a.G[k];
    float* dG = a.dG[k];
    const int64_t n = a.count[k];
    if (e + 4 <= n) {
      float4 g = *reinterpret_cast<float4*>(G + e);
      const float4 d = *reinterpret_cast<const float4*>(dG + e);
      g.x = fmaf(-a.lr, d.x, g.x);
      g.y = fmaf(-a.lr, d.y, g.y);
      g.z = fmaf(-a.lr, d.z, g.z);
      g.w = fmaf(-a.lr, d.w, g.w);
      *reinterpret_cast<float4*>(G + e) = g;
      if (a.zero) *reinterpret_cast<float4*>(dG + e) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      for (int64_t t = e; t < n; ++t) {
        G[t] = fmaf(-a.lr, dG[t], G[t]);
        if (a.zero) dG[t] = 0.f;
      }
    }
  }
}

static int persistent_grid_bwd(const void* fn, int threads, size_t smem) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return per_sm * sm_count();
}

int launch_backward(const Shape& s, const Layout& L, const WS& w, const float* grad_out,
                    const float* const cores[3], const int64_t* offsets, int64_t nnz,
                    int64_t num_bags, float* const core_grads[3], cudaStream_t st) {
  if (nnz == 0) return TT_EMB_OK;
  const int sms = sm_count();
  int grid = (int)ceil_div(L.rowbuf_rows > num_bags ? L.rowbuf_rows : num_bags, 8);
  if (grid > sms * 16) grid = sms * 16;
  if (grid < 1) grid = 1;
  const bool cta_gather = s.D == 128;
  TT_TIMED("k_s_zero", st, (k_s_zero<<<grid, 256, 0, st>>>(w, s.D, offsets, num_bags, nnz,
                                                             cta_gather ? kSCta : kSSlice)));
  const int64_t slices = ceil_div(nnz, kSSlice);
  if (cta_gather) {
    TT_TIMED("k_s_gather", st, (k_s_gather_cta<<<(int)ceil_div(nnz, kSCta), 256, 0, st>>>(
                                   w, grad_out, num_bags)));
  } else {
    TT_TIMED("k_s_gather", st, (k_s_gather<<<(int)ceil_div(slices, 8), 256, 0, st>>>(w, grad_out, num_bags, s.D)));
  }

  BwdArgs ba;
  ba.s = s;
  ba.w = w;
  ba.G1 = cores[0];
  ba.G2 = cores[1];
  ba.G3 = cores[2];
  ba.dG1 = core_grads[0];
  ba.dG2 = core_grads[1];
  ba.dG3 = core_grads[2];
  if (s.n1 == 4 && s.n3 == 4 && s.n2 == 8 && s.R1 == 32 && s.R2 == 32) {
    using C = BwsCfg<8, 32, kCP_8_32>;
    static int grid = 0;
    if (grid == 0) {
      cudaFuncSetAttribute(k_bwd_ws<8, 32, kCP_8_32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::SMEM);
      grid = persistent_grid_bwd((const void*)k_bwd_ws<8, 32, kCP_8_32>, 288, C::SMEM);
    }
    TT_TIMED("k_bwd_ws", st, (k_bwd_ws<8, 32, kCP_8_32><<<grid, 288, C::SMEM, st>>>(ba)));
  } else {
    const size_t g2n = (size_t)s.R1 * s.n2 * s.R2;
    const size_t base = g2n + (size_t)s.n1 * s.R1 + 2 * (size_t)s.n1 * s.n2 * s.R2;
    ba.dG2_in_smem = (base + g2n) <= (size_t)kMaxSmemFloats;
    const size_t smem = sizeof(float) * (base + (ba.dG2_in_smem ? g2n : 0));
    static int grid = 0;
    if (grid == 0) {
      cudaFuncSetAttribute(k_bwd_generic, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxSmemFloats * (int)sizeof(float));
      grid = persistent_grid_bwd((const void*)k_bwd_generic, 256, kMaxSmemFloats * sizeof(float));
    }
    TT_TIMED("k_bwd_generic", st, (k_bwd_generic<<<grid, 256, smem, st>>>(ba)));
  }
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

int launch_sgd(float* const cores[3], float* const grads[3], const Shape& s, float lr,
               int zero_grads, cudaStream_t st) {
  SgdArgs a;
  const int64_t counts[3] = {s.m1 * s.n1 * s.R1, s.m2 * s.R1 * s.n2 * s.R2, s.m3 * s.R2 * s.n3};
  a.start[0] = 0;
  for (int k = 0; k < 3; ++k) {
    a.G[k] = cores[k];
    a.dG[k] = grads[k];
    a.count[k] = counts[k];
    a.start[k + 1] = a.start[k] + ceil_div(counts[k], 4);
  }
  a.lr = lr;
  a.zero = zero_grads ? 1 : 0;
  int grid = (int)ceil_div(a.start[3], 256);
  if (grid > sm_count() * 8) grid = sm_count() * 8;
  if (grid < 1) grid = 1;
  TT_TIMED("k_sgd", st, (k_sgd<<<grid, 256, 0, st>>>(a)));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
