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
#include "tt_mma.cuh"
#include "tt_split.cuh"

namespace tt {

// Preparation of the backward, one launch of one wave:
//  - zero the S rows that more than one gather slice will add into (one thread
//    per unique row; a crossing row, one per slice boundary at most, is zeroed
//    by its thread),
//  - reset the backward chunk counter,
//  - split the cores into their bf16 planes unless they already hold them
//    (tensor-core shapes; sp.g2l is null otherwise).
// (The bag of every lookup is written by the grouping.)
__global__ void __launch_bounds__(256) k_s_zero(WS w, int D, int span, int64_t rows_cap,
                                                SplitArgs sp, int reuse) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t gtid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (reuse && (w.ctl->method == kGroupBitmap || w.ctl->method == kGroupDirect)) {
    // the grouping came from a forward-only call and has no per-row lookup
    // lists (or there is none: a per-lookup forward): report it, and leave the
    // backward's later kernels no lookups and no chunks, so that the core
    // gradients stay as they are
    if (gtid == 0) {
      set_status(w.ctl, kStNoLists);
      w.ctl->n_valid = 0;
      w.ctl->n_chunks = 0;
    }
    return;
  }
  const int64_t U = w.ctl->U_r;
  int32_t s0 = 0, s1 = 0;
  if (gtid < rows_cap) {               // row_start holds rows_cap + 1 entries at least
    s0 = w.row_start[gtid];
    s1 = w.row_start[gtid + 1];
  }
  const bool need_split = sp.g2l && !(reuse && split_current(sp, w.ctl));
  if (blockIdx.x == 0 && threadIdx.x == 0) w.ctl->bwd_chunk_ctr = 0;
  for (int64_t u = gtid; u < U; u += stride) {
    if (u != gtid) {
      s0 = w.row_start[u];
      s1 = w.row_start[u + 1];
    }
    if (s0 / span != (s1 - 1) / span) {
      float* r = w.rowbuf + u * (int64_t)D;
      if ((D & 3) == 0) {
        for (int j = 0; j < D; j += 4) *reinterpret_cast<float4*>(r + j) = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
        for (int j = 0; j < D; ++j) r[j] = 0.f;
      }
    }
  }
  if (need_split) split_cores_body(sp);
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

// The factor with which lookup l's row enters its bag b (PoolMode): its
// per-sample weight, 1 / (length of b), or 1.  S[x] sums grad_out[b] times
// that factor.
template <int MODE>
__device__ __forceinline__ float lookup_factor(const float* __restrict__ psw,
                                               const int64_t* __restrict__ offsets, int64_t nnz,
                                               int32_t l, int32_t b) {
  if (MODE == kPoolWeighted) return psw[l];
  if (MODE == kPoolMean) {
    int64_t l0 = offsets[b], l1 = offsets[b + 1];
    l0 = l0 < 0 ? 0 : (l0 > nnz ? nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > nnz ? nnz : l1);
    return l1 > l0 ? 1.f / (float)(l1 - l0) : 0.f;
  }
  return 1.f;
}

// S[x] for every unique row: one warp per slice of kSSlice sorted lookups.  The
// lanes fetch the slice's (unique row, bag, factor) triples in parallel, 32 at a
// time; the output-gradient rows are then summed with 8 loads in flight,
// flushing at every change of unique row.
template <int MODE>
__global__ void __launch_bounds__(256) k_s_gather(WS w, const float* __restrict__ grad_out,
                                                  int64_t B, int D, const float* __restrict__ psw,
                                                  const int64_t* __restrict__ offsets, int64_t nnz) {
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
      float my_c = 1.f;
      if (lane < cnt) {
        const int32_t l = w.perm[kb + lane];
        my_u = w.uid[l];
        const int32_t bb = w.bag_of[l];
        my_b = bb < 0 ? 0 : (bb >= B ? (int32_t)(B - 1) : bb);
        my_c = lookup_factor<MODE>(psw, offsets, nnz, l, my_b);
      }
      for (int j = 0; j < cnt; j += 8) {
        int32_t uj[8];
        float4 g[8];
        float gs[8], cf[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int jj = (j + t) & 31;
          uj[t] = __shfl_sync(0xffffffffu, my_u, jj);
          const int32_t bj = __shfl_sync(0xffffffffu, my_b, jj);
          cf[t] = __shfl_sync(0xffffffffu, my_c, jj);
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
          if (MODE == kPoolSum) {
            f4add(acc, g[t]);
            accs += gs[t];
          } else {
            f4fma(acc, cf[t], g[t]);
            accs = fmaf(cf[t], gs[t], accs);
          }
        }
      }
    }
    if (cur >= 0 && live) s_flush(w, cur, k0, c, D, acc, vec, accs);
  }
}

// S[x] with the partial sums of rows that cross warp boundaries merged inside
// the CTA: a CTA covers 8 x span sorted positions (span, at most 32 x
// kGatherBatches, chosen per batch so that the grid fills whole waves); each
// warp sums the runs of its span positions (8 output-gradient rows in flight), stores
// the runs that start and end inside its range, and leaves its first and last
// run in shared memory; one warp then merges those in position order and
// stores each merged row, or adds it with float atomics (into a row zeroed by
// k_s_zero) when the row also crosses the CTA's range.  D = 128.
__device__ __forceinline__ void s_merge_flush(const WS& w, int32_t u, int64_t K0, int64_t K1,
                                              const float4& m, int lane) {
  const int32_t s0 = w.row_start[u], s1 = w.row_start[u + 1];
  float4* dst = reinterpret_cast<float4*>(w.rowbuf) + (int64_t)u * 32 + lane;
  if (s0 < K0 || s1 > K1) atomicAdd(dst, m);
  else *dst = m;
}

constexpr int kGatherBatches = 3;   // batches of 32 sorted positions per warp, at most

// D = 128: every lane owns one float4 column of the rows.
template <int MODE>
__global__ void __launch_bounds__(256, MODE == kPoolSum ? 4 : 3) k_s_gather_cta(WS w, const float* __restrict__ grad_out,
                                                         int64_t B, const float* __restrict__ psw,
                                                         const int64_t* __restrict__ offsets,
                                                         int64_t nnz, int span) {
  __shared__ float4 part[8][2][32];
  __shared__ int part_u[8][2];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t nv = w.ctl->n_valid;
  const int64_t cspan = 8 * (int64_t)span;
  const int64_t K0 = (int64_t)blockIdx.x * cspan;
  if (K0 >= nv) return;                                // uniform over the CTA
  const int64_t K1 = K0 + cspan < nv ? K0 + cspan : nv;
  const int64_t k0 = K0 + (int64_t)warp * span;
  const int64_t k1 = k0 + span < K1 ? k0 + span : K1;
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
  // the (unique row, bag, factor) of all 32-position batches of the slice,
  // loaded together: two dependent round trips for the whole slice
  int32_t bu[kGatherBatches], bbag[kGatherBatches], bl[kGatherBatches];
  float bc[kGatherBatches];
#pragma unroll
  for (int h = 0; h < kGatherBatches; ++h) {
    bu[h] = -1;
    bbag[h] = 0;
    bl[h] = -1;
    bc[h] = 1.f;
    if (k0 + 32 * h + lane < k1) bl[h] = w.perm[k0 + 32 * h + lane];
  }
#pragma unroll
  for (int h = 0; h < kGatherBatches; ++h)
    if (bl[h] >= 0) {
      bu[h] = w.uid[bl[h]];
      bbag[h] = w.bag_of[bl[h]];
    }
#pragma unroll
  for (int h = 0; h < kGatherBatches; ++h) {
    bbag[h] = bbag[h] < 0 ? 0 : (bbag[h] >= B ? (int32_t)(B - 1) : bbag[h]);
    if (bl[h] >= 0) bc[h] = lookup_factor<MODE>(psw, offsets, nnz, bl[h], bbag[h]);
  }
#pragma unroll
  for (int h = 0; h < kGatherBatches; ++h) {
    const int64_t kb = k0 + 32 * h;
    if (kb >= k1) break;
    const int cnt = (int)(k1 - kb < 32 ? k1 - kb : 32);
    const int32_t my_u = bu[h], my_b = bbag[h];
    const float my_c = bc[h];
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
        if (MODE == kPoolSum) f4add(acc, g[t]);
        else f4fma(acc, __shfl_sync(0xffffffffu, my_c, j + t), g[t]);
      }
    }
    for (; j < cnt; ++j) {
      const int32_t u = __shfl_sync(0xffffffffu, my_u, j);
      const float4 g = __ldg(g4 + (int64_t)__shfl_sync(0xffffffffu, my_b, j) * 32 + lane);
      const float cj = __shfl_sync(0xffffffffu, my_c, j);
      if (u != cur) {
        close_run();
        acc = z4;
        cur = u;
      }
      if (MODE == kPoolSum) f4add(acc, g);
      else f4fma(acc, cj, g);
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
          if (mu >= 0) s_merge_flush(w, mu, K0, K0 + cspan, m, lane);
          mu = u;
          m = z4;
        }
        f4add(m, part[ww][e][lane]);
      }
    if (mu >= 0) s_merge_flush(w, mu, K0, K0 + cspan, m, lane);
  }
}

// The bag of every lookup, one warp per 32 bags (the forward's pooling writes
// the same array; this serves a grouping that no forward followed).
__global__ void __launch_bounds__(256) k_bag_ids(int32_t* __restrict__ bag_of,
                                                 const int64_t* __restrict__ offsets, int64_t B,
                                                 int64_t nnz) {
  const int lane = threadIdx.x & 31;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t wb = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); wb < B; wb += stride) {
    const int64_t b = wb + lane;
    const int64_t o0 = b < B ? offsets[b] : 0, o1 = b < B ? offsets[b + 1] : 0;
    write_bag_ids(bag_of, wb, B, nnz, o0, o1, lane);
  }
}

int launch_bag_ids(const WS& w, const int64_t* offsets, int64_t num_bags, int64_t nnz,
                   cudaStream_t st) {
  if (num_bags <= 0 || nnz <= 0) return TT_EMB_OK;
  int grid = (int)ceil_div(num_bags, 256);
  if (grid > sm_count() * 8) grid = sm_count() * 8;
  TT_TIMED("k_bag_ids", st, (k_bag_ids<<<grid, 256, 0, st>>>(w.bag_of, offsets, num_bags, nnz)));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

// Gradient of the per-sample weights: dW[l] = <grad_out[bag(l)], row(r_l)>,
// read from the unique rows in the row buffer (filled by the row kernels just
// before); one warp per bag, 4 lookups per step, each lane a float4 column of
// the rows; out-of-range lookups get 0.  Stores are one coalesced write per
// 32 lookups.
__global__ void __launch_bounds__(256) k_psw_grad(const int64_t* __restrict__ offsets, int64_t B,
                                                  int64_t nnz, const int32_t* __restrict__ uid,
                                                  const float* __restrict__ rowbuf, int D,
                                                  const float* __restrict__ grad_out,
                                                  float* __restrict__ dW) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const bool vec = (D & 3) == 0;
  const int cols = vec ? (D >> 2) : D;
  for (int64_t b = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < B; b += warps) {
    int64_t l0 = offsets[b], l1 = offsets[b + 1];
    l0 = l0 < 0 ? 0 : (l0 > nnz ? nnz : l0);
    l1 = l1 < l0 ? l0 : (l1 > nnz ? nnz : l1);
    for (int64_t lb = l0; lb < l1; lb += 32) {
      const int cnt = (int)(l1 - lb < 32 ? l1 - lb : 32);
      const int32_t my_u = lane < cnt ? uid[lb + lane] : -1;
      float my_dw = 0.f;
      for (int j = 0; j < cnt; j += 4) {
        int32_t u[4];
        float part[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          u[t] = __shfl_sync(0xffffffffu, my_u, (j + t) & 31);
          if (j + t >= cnt) u[t] = -1;
          part[t] = 0.f;
        }
        for (int c = lane; c < cols; c += 32) {
          if (vec) {
            const float4 g = reinterpret_cast<const float4*>(grad_out + b * (int64_t)D)[c];
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (u[t] >= 0) {
                const float4 v = reinterpret_cast<const float4*>(rowbuf + (int64_t)u[t] * D)[c];
                part[t] = fmaf(g.x, v.x, fmaf(g.y, v.y, fmaf(g.z, v.z, fmaf(g.w, v.w, part[t]))));
              }
          } else {
            const float g = grad_out[b * (int64_t)D + c];
#pragma unroll
            for (int t = 0; t < 4; ++t)
              if (u[t] >= 0) part[t] = fmaf(g, rowbuf[(int64_t)u[t] * D + c], part[t]);
          }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) part[t] += __shfl_xor_sync(0xffffffffu, part[t], o);
          if (lane == j + t) my_dw = part[t];
        }
      }
      if (lane < cnt) dW[lb + lane] = my_dw;
    }
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
// Tensor-core backward chunk kernel for n1 = n3 = 4, n2 = 8, R1 = R2 = 32 (D = 128).
// Warp 8 is a producer: it claims the next chunk (skipping chunks that hold a
// later piece of a hot prefix: the chunk that starts such a prefix takes all of
// its rows, so that its prefix-level products are formed once), lists the row
// pairs of the first batch and stages the chunk's operands into the free one of
// two stage buffers, all as bf16 hi / lo planes: G2 and G1 (copies of the
// per-call split planes), the first batch's G3 rows (copies of the split G3
// planes, [r2][j3] per row) and its S rows (converted here from the fp32
// unique-row buffer into [j3][(j1, j2)] per row).  Warps 0-7 consume with
// three-term bf16 tensor-core tiles (tt_mma.cuh), fragments by ldmatrix:
//   (1) P2 = [G1 rows] . G2[i2]                     (4 np) x 256 x 32, m16n8k16
//   per batch of RB rows, by pairs of rows of one prefix:
//   (2) dP2[p] += S[x] . G3[i3_x]^T                  32 x 32 x (4 per row), m16n8k8
//   (3) dG3[i3_x] += P2[p]^T . S[x]                  32 x (4 per row) x 32, m16n8k16
//   then
//   (4) dG2[i2] += [G1 rows]^T . dP2                 32 x 256 x (4 np)
//   (5) dG1[i1_p] += dP2[p] . G2[i2]^T               (4 np) x 32 x 256
// A pair's missing second row reads a zero row.  Core gradients are
// accumulated with vector float reductions.
// Longest run of consecutive chunks one claim of the backward chunk kernel takes.
constexpr int kBwdRun = 16;

struct MmaBwd {
  static constexpr int CP = kCP_8_32, R = 32, NC = 256, D = 128;
  static constexpr int RB = 24;                     // rows per batch (row RB of a stage stays zero)
  static constexpr int MAXPAIRS = RB / 2 + CP;      // pairs of one batch
  // bf16 plane geometry (elements / bytes)
  static constexpr int G2LD = NC + 8, G1LD = R + 8, DPLD = NC + 8;
  static constexpr int G2PLANE = R * G2LD * 2, G1PLANE = 4 * CP * G1LD * 2, DPPLANE = 4 * CP * DPLD * 2;
  static constexpr int SROW = 4 * (32 + 8) * 2;     // S plane row: [j3][(j1, j2)], 80-byte j3 rows
  static constexpr int GROW = (4 * R + 32) * 2;     // G3 plane row: [r2][j3], 320 bytes
  static constexpr int SPLANE = (RB + 1) * SROW, GPLANE = (RB + 1) * GROW;
  // P2 planes [p][j1][j2][r2]: j2 rows of 80 B, j1 blocks of 656 B, prefixes 2624 B apart
  static constexpr int PB = 80, PA = 8 * PB + 16, PPB = 4 * PA;
  static constexpr int P2PLANE = CP * PPB;
  // stage layout (bytes)
  static constexpr int OFF_G1 = 2 * G2PLANE, OFF_S = OFF_G1 + 2 * G1PLANE, OFF_G3 = OFF_S + 2 * SPLANE;
  static constexpr int STAGE_B = OFF_G3 + 2 * GPLANE;
  static constexpr int OFF_P2 = 2 * STAGE_B, OFF_DP = OFF_P2 + 2 * P2PLANE, OFF_META = OFF_DP + 2 * DPPLANE;
  struct Meta {
    int x0, x1, p0, np, i2, nb, npairs, end;
    int flush;           // the CTA's next chunk has another i2: reduce dG2[i2] after this one
    int pad[3];
    int rs[CP];          // chunk-local first row of each prefix
    int pi1[CP];
    int ri3[RB];         // i3 of the current batch's rows
    int pair[MAXPAIRS];  // batch-local first row | (second row valid) << 8 | prefix << 9
  };
  static constexpr int THREADS = 288;
  static constexpr int SMEM = OFF_META + 2 * (int)sizeof(Meta) + 4 * 8;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(STAGE_B % 16 == 0 && OFF_S % 16 == 0 && OFF_G3 % 16 == 0 && OFF_META % 16 == 0, "alignment");
  static_assert(RB <= 32 && CP <= 8, "one row per producer lane; pair encoding");
};

// Pairs of the rows [b0, b1) of a chunk, prefix by prefix (rsq[j]: chunk-local
// first row of prefix j, `rows` for j >= np).  One warp; returns the count.
__device__ __forceinline__ int bwd_pairs(int b0, int b1, int rows, const int* rsq, int* pair, int lane) {
  int n = 0;
  for (int rb = b0; rb < b1; rb += 32) {
    const int r = rb + lane;
    int q = -1, qs = 0, qe = rows;
#pragma unroll
    for (int j = 0; j < MmaBwd::CP; ++j) {
      const int v = rsq[j];
      if (v <= r) {
        ++q;
        qs = v;
      } else {
        qe = min(qe, v);
      }
    }
    qs = max(qs, b0);
    qe = min(qe, b1);
    const bool start = r < b1 && ((r - qs) & 1) == 0;
    const unsigned bal = __ballot_sync(0xffffffffu, start);
    if (start) pair[n + __popc(bal & ((1u << lane) - 1u))] = (r - b0) | ((r + 1 < qe) ? 256 : 0) | (q << 9);
    n += __popc(bal);
  }
  return n;
}

// S row x (fp32 [(j1, j2)][j3], lane l's float4 = (j1, j2) = l, j3 = 0..3) -> bf16
// planes [j3][(j1, j2)] of stage row r: eight 2-byte stores.
__device__ __forceinline__ void bwd_store_s(char* Sp, int r, float4 v, int l) {
  using C = MmaBwd;
  const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const __nv_bfloat16 h = __float2bfloat16_rn(x[c]);
    const __nv_bfloat16 lo = __float2bfloat16_rn(x[c] - __bfloat162float(h));
    char* o = Sp + r * C::SROW + c * 80 + 2 * l;
    *reinterpret_cast<__nv_bfloat16*>(o) = h;
    *reinterpret_cast<__nv_bfloat16*>(o + C::SPLANE) = lo;
  }
}

// (1): P2 rows (p, j1) = 16 MT tiles x 256 columns; warp w owns j2 = w.  bf16
// three-term tiles: A = G1 rows (plain ldmatrix), B = G2 [r1][(j2, r2)]
// (transposed).  P2 is kept as bf16 planes for (3).
template <int MT>
__device__ __forceinline__ void mma_bwd_p2(uint32_t g2h, uint32_t g1h, char* __restrict__ P2, int warp,
                                           int lane) {
  using C = MmaBwd;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t g2l = g2h + C::G2PLANE, g1l = g1h + C::G1PLANE;
  float acc[MT][4][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.f;
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
      ldsm_x4_t(bh, b2_addr_kn(g2h, C::G2LD, 16 * ks, 32 * warp + 16 * np2, lane));
      ldsm_x4_t(bl, b2_addr_kn(g2l, C::G2LD, 16 * ks, 32 * warp + 16 * np2, lane));
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
          mma_bf16x3(acc[mt][2 * np2 + h], ah[mt], al[mt], bh[2 * h], bh[2 * h + 1], bl[2 * h], bl[2 * h + 1]);
    }
  }
  // row (p, j1) = 16 mt + g (+8), columns j2 = warp, r2 = 8 nt + 2t (+1)
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = 16 * mt + g + 8 * h;
      char* dst = P2 + (row >> 2) * C::PPB + (row & 3) * C::PA + warp * C::PB + 4 * t;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        uint32_t hi, lo;
        split_bf16x2(acc[mt][nt][2 * h], acc[mt][nt][2 * h + 1], hi, lo);
        *reinterpret_cast<uint32_t*>(dst + 16 * nt) = hi;
        *reinterpret_cast<uint32_t*>(dst + 16 * nt + C::P2PLANE) = lo;
      }
    }
}

// dP2 accumulator of one warp: tile (j12 = 16 mt .. +15) x (r2 = 8 nt .. +7) of
// the current prefix, two pair parities x {hi.hi, small terms}.
struct DP2Acc {
  float c[4][4];
  int p;
};

__device__ __forceinline__ void dp2_flush(DP2Acc& acc, char* __restrict__ dP2, int mt, int nt, int lane) {
  using C = MmaBwd;
  const int g = lane >> 2, t = lane & 3;
  if (acc.p >= 0) {
    float v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (acc.c[1][i] + acc.c[3][i]) + (acc.c[0][i] + acc.c[2][i]);
    // rows j12 = 16 mt + g (+8): j1 = 2 mt (+1), j2 = g; plane row (p, j1), column (j2, r2)
    char* hi = dP2 + 2 * (((4 * acc.p + 2 * mt) * C::DPLD) + g * C::R + 8 * nt + 2 * t);
    uint32_t h0, l0, h1, l1;
    split_bf16x2(v[0], v[1], h0, l0);
    split_bf16x2(v[2], v[3], h1, l1);
    *reinterpret_cast<uint32_t*>(hi) = h0;
    *reinterpret_cast<uint32_t*>(hi + C::DPPLANE) = l0;
    *reinterpret_cast<uint32_t*>(hi + 2 * C::DPLD) = h1;
    *reinterpret_cast<uint32_t*>(hi + 2 * C::DPLD + C::DPPLANE) = l1;
  }
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc.c[u][i] = 0.f;
}

// (2) over the pairs of one batch, four pairs per step, bf16 m16n8k8 tiles:
// A[j12][(row of pair, j3)] from the S planes (transposed ldmatrix, rows
// (row, j3)), B[(row, j3)][r2] = G3[i3_row][r2][j3] (32-bit loads of j3 pairs).
__device__ __forceinline__ void mma_bwd_dp2(const MmaBwd::Meta& m, uint32_t Sh, const char* __restrict__ G3p,
                                            char* __restrict__ dP2, DP2Acc& acc, int warp, int lane) {
  using C = MmaBwd;
  constexpr int U = 4;
  const int g = lane >> 2, t = lane & 3;
  const int mt = warp & 1, nt = warp >> 1;
  const int npairs = m.npairs;
  const int lr = lane & 7, lj = (lane >> 3) & 1;
  for (int q0 = 0; q0 < npairs; q0 += U) {
    int e[U];
#pragma unroll
    for (int u = 0; u < U; ++u) e[u] = q0 + u < npairs ? m.pair[q0 + u] : -1;
    uint32_t ah[U][2], al[U][2], bh[U], bl[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int eu = e[u] < 0 ? e[0] : e[u];
      const int r0 = eu & 255, has2 = (eu >> 8) & 1;
      // ldmatrix rows k = (row of pair, j3): lanes 0-7 (and 8-15) give row lr
      const int xr = (lr >> 2) == 0 ? r0 : (has2 ? r0 + 1 : C::RB);
      const uint32_t aa = Sh + xr * C::SROW + (lr & 3) * 80 + 2 * (16 * mt + 8 * lj);
      ldsm_x2_t(ah[u], aa);
      ldsm_x2_t(al[u], aa + C::SPLANE);
      // B: k = (t / 2, j3 = 2 (t % 2)), n = r2 = 8 nt + g
      const int xb = (t >> 1) == 0 ? r0 : (has2 ? r0 + 1 : C::RB);
      const char* bp = G3p + xb * C::GROW + (8 * nt + g) * 8 + 4 * (t & 1);
      bh[u] = *reinterpret_cast<const uint32_t*>(bp);
      bl[u] = *reinterpret_cast<const uint32_t*>(bp + C::GPLANE);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (e[u] < 0) break;
      const int p = e[u] >> 9;
      if (p != acc.p) {
        dp2_flush(acc, dP2, mt, nt, lane);
        acc.p = p;
      }
      float* big = acc.c[(u & 1) ? 2 : 0];
      float* small = acc.c[(u & 1) ? 3 : 1];
      mma_bf16_k8(small, al[u][0], al[u][1], bh[u]);
      mma_bf16_k8(big, ah[u][0], ah[u][1], bh[u]);
      mma_bf16_k8(small, ah[u][0], ah[u][1], bl[u]);
    }
  }
}

// (3) over the pairs of one batch: warp w takes m-tile w % 2 (r2 = 16 (w % 2) ..
// +15) of a contiguous quarter of the pairs.  bf16 m16n8k16 tiles:
// A[r2][j12] = P2[p][j12][r2] (transposed ldmatrix, cached per prefix),
// B[j12][(row of pair, j3)] from the S planes (plain ldmatrix, rows (row, j3)).
__device__ __forceinline__ void mma_bwd_dg3(const MmaBwd::Meta& m, uint32_t P2h, uint32_t Sh,
                                            float* __restrict__ dG3, int warp, int lane) {
  using C = MmaBwd;
  const int g = lane >> 2, t = lane & 3;
  const int mt = warp & 1, quarter = warp >> 1;
  const int npairs = m.npairs;
  const int q0 = (npairs * quarter) >> 2, q1 = (npairs * (quarter + 1)) >> 2;
  const int li = lane >> 3, lr = lane & 7;
  int cur_p = -1;
  uint32_t ah[2][4], al[2][4];
  for (int q = q0; q < q1; ++q) {
    const int e = m.pair[q];
    const int r0 = e & 255, has2 = (e >> 8) & 1, p = e >> 9;
    if (p != cur_p) {
      cur_p = p;
      // matrix li: k rows j12 = 16 ks + 8 (li >> 1) + lr (j1 = 2 ks + (li >> 1), j2 = lr),
      // m columns r2 = 16 mt + 8 (li & 1)
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const uint32_t aa = P2h + p * C::PPB + (2 * ks + (li >> 1)) * C::PA + lr * C::PB +
                            2 * (16 * mt + 8 * (li & 1));
        ldsm_x4_t(ah[ks], aa);
        ldsm_x4_t(al[ks], aa + C::P2PLANE);
      }
    }
    // B rows n = (row of pair, j3) = lr, k columns j12 = 16 ks + 8 ((lane >> 3) & 1)
    const int xr = (lr >> 2) == 0 ? r0 : (has2 ? r0 + 1 : C::RB);
    const uint32_t bb = Sh + xr * C::SROW + (lr & 3) * 80 + 16 * (li & 1);
    // hi.hi and the two small products in three accumulators (chains of two)
    float big[4] = {0.f, 0.f, 0.f, 0.f}, sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
      uint32_t bh[2], bl[2];
      ldsm_x2(bh, bb + 32 * ks);
      ldsm_x2(bl, bb + 32 * ks + C::SPLANE);
      mma_bf16(sa, al[ks], bh[0], bh[1]);
      mma_bf16(sb, ah[ks], bl[0], bl[1]);
      mma_bf16(big, ah[ks], bh[0], bh[1]);
    }
    // C[r2][(row of pair, j3)]: this lane holds j3 = 2 (t % 2), +1 of row t / 2
    if (t < 2 || has2) {
      float* o = dG3 + (size_t)m.ri3[r0 + (t >> 1)] * (4 * C::R) + (16 * mt + g) * 4 + 2 * (t & 1);
      red_add_f2(o, (sa[0] + sb[0]) + big[0], (sa[1] + sb[1]) + big[1]);
      red_add_f2(o + 32, (sa[2] + sb[2]) + big[2], (sa[3] + sb[3]) + big[3]);
    }
  }
}

// (4): dG2[i2][r1][(j2, r2)] += sum over (p, j1) of G1[i1_p][j1][r1] dP2[p][j1][j2][r2],
// into the warp's accumulators (kept across the CTA's consecutive chunks of one
// i2, reduced into dG2 by dg2_flush); warp w owns columns 32 w .. 32 w + 31.  bf16 tiles: A = G1 rows read transposed
// ([k = (p, j1)][m = r1]), B = dP2 planes [k = (p, j1)][n] (transposed); the k range
// is padded to 16 with rows that the caller has zeroed in both operands.
__device__ __forceinline__ void mma_bwd_dg2(uint32_t g1h, uint32_t dph, float (&acc)[2][4][4], int np,
                                            int warp, int lane) {
  using C = MmaBwd;
  const uint32_t g1l = g1h + C::G1PLANE, dpl = dph + C::DPPLANE;
  const int kk = (np + 3) >> 2;
  for (int ks = 0; ks < kk; ++ks) {
    uint32_t ah[2][4], al[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      ldsm_x4_t(ah[mt], a_addr_km(g1h, C::G1LD, 16 * mt, 16 * ks, lane));
      ldsm_x4_t(al[mt], a_addr_km(g1l, C::G1LD, 16 * mt, 16 * ks, lane));
    }
#pragma unroll
    for (int np2 = 0; np2 < 2; ++np2) {
      uint32_t bh[4], bl[4];
      ldsm_x4_t(bh, b2_addr_kn(dph, C::DPLD, 16 * ks, 32 * warp + 16 * np2, lane));
      ldsm_x4_t(bl, b2_addr_kn(dpl, C::DPLD, 16 * ks, 32 * warp + 16 * np2, lane));
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
          mma_bf16x3(acc[mt][2 * np2 + h], ah[mt], al[mt], bh[2 * h], bh[2 * h + 1], bl[2 * h], bl[2 * h + 1]);
    }
  }
}

// dG2[i2] += the warp's accumulated part of (4) (vector float reductions), then
// the accumulators start again from zero.
__device__ __forceinline__ void dg2_flush(float (&acc)[2][4][4], float* __restrict__ dG2i2, int warp,
                                          int lane) {
  using C = MmaBwd;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float* o = dG2i2 + (size_t)(16 * mt + g + 8 * h) * C::NC + 32 * warp + 2 * t;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        red_add_f2(o + 8 * nt, acc[mt][nt][2 * h], acc[mt][nt][2 * h + 1]);
        acc[mt][nt][2 * h] = acc[mt][nt][2 * h + 1] = 0.f;
      }
    }
}

// (5): dG1[i1_p][j1][r1] += sum over (j2, r2) of dP2[p][j1][j2][r2] G2[r1][(j2, r2)];
// warp w takes the tile (p, j1) = 16 (w % 2) .. +15 x r1 = 8 (w / 2) .. +7.  bf16 tiles:
// A = dP2 planes [m = (p, j1)][k] (plain), B = G2 [n = r1][k = (j2, r2)] (plain).
__device__ __forceinline__ void mma_bwd_dg1(uint32_t dph, uint32_t g2h, const int* __restrict__ pi1,
                                            float* __restrict__ dG1, int np, int warp, int lane) {
  using C = MmaBwd;
  const int g = lane >> 2, t = lane & 3;
  const int mt = warp & 1, nt = warp >> 1;
  if (16 * mt >= 4 * np) return;
  const uint32_t dpl = dph + C::DPPLANE, g2l = g2h + C::G2PLANE;
  float c[2][4];
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int i = 0; i < 4; ++i) c[u][i] = 0.f;
#pragma unroll
  for (int ks = 0; ks < C::NC / 16; ++ks) {
    uint32_t ah[4], al[4], bh[2], bl[2];
    ldsm_x4(ah, a_addr_mk(dph, C::DPLD, 16 * mt, 16 * ks, lane));
    ldsm_x4(al, a_addr_mk(dpl, C::DPLD, 16 * mt, 16 * ks, lane));
    ldsm_x2(bh, b1_addr_nk(g2h, C::G2LD, 16 * ks, 8 * nt, lane));
    ldsm_x2(bl, b1_addr_nk(g2l, C::G2LD, 16 * ks, 8 * nt, lane));
    mma_bf16x3(c[ks & 1], ah, al, bh[0], bh[1], bl[0], bl[1]);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int row = 16 * mt + g + 8 * h, p = row >> 2;
    if (p < np) {
      float* o = dG1 + ((size_t)pi1[p] * 4 + (row & 3)) * C::R + 8 * nt + 2 * t;
      red_add_f2(o, c[0][2 * h] + c[1][2 * h], c[0][2 * h + 1] + c[1][2 * h + 1]);
    }
  }
}

__global__ void __launch_bounds__(MmaBwd::THREADS, 1) k_bwd_mma(BwdArgs a) {
  using C = MmaBwd;
  using Meta = C::Meta;
  extern __shared__ float4 sm4[];
  char* base = reinterpret_cast<char*>(sm4);
  char* P2 = base + C::OFF_P2;                      // bf16 planes
  char* dP2 = base + C::OFF_DP;                     // bf16 planes
  Meta* meta = reinterpret_cast<Meta*>(base + C::OFF_META);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + 2);
  uint64_t* empty = full + 2;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(&full[0], 33);
    mbar_init(&full[1], 33);
    mbar_init(&empty[0], 1);
    mbar_init(&empty[1], 1);
    mbar_init_fence();
    if (blockIdx.x == 0) mark_split(a.w.ctl, a.G1, a.G2, a.G3);
  }
  // the zero row (row RB) of the S and G3 planes of both stages
  for (int e = tid; e < 2 * 4 * (C::SROW / 16); e += C::THREADS) {
    const int st = e / (4 * (C::SROW / 16)), rem = e - st * 4 * (C::SROW / 16);
    const int which = rem / (C::SROW / 16), q = rem - which * (C::SROW / 16);
    char* st0 = base + st * C::STAGE_B;
    char* row = which < 2 ? st0 + C::OFF_S + which * C::SPLANE + C::RB * C::SROW
                          : st0 + C::OFF_G3 + (which - 2) * C::GPLANE + C::RB * C::GROW;
    *reinterpret_cast<uint4*>(row + 16 * q) = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  const int n_chunks = a.w.ctl->n_chunks;

  if (warp == 8) {
    // ---------------- producer (claims one chunk ahead).  Chunks are claimed in
    // runs of consecutive ones, long while many remain and one at a time at the
    // end (guided), so that this CTA's consecutive chunks often share i2 and the
    // consumers keep dG2[i2] in registers across them.
    int run_c = 0, run_end = 0;
    auto claim_next = [&]() {
      if (run_c >= run_end) {
        int k = 1, c0 = 0;
        if (lane == 0) {
          const int seen = (int)ld_relaxed_u32(&a.w.ctl->bwd_chunk_ctr);
          k = (n_chunks - seen) / (2 * (int)gridDim.x);
          k = k < 1 ? 1 : (k > kBwdRun ? kBwdRun : k);
          c0 = (int)atomicAdd(&a.w.ctl->bwd_chunk_ctr, (uint32_t)k);
        }
        run_c = __shfl_sync(0xffffffffu, c0, 0);
        run_end = run_c + __shfl_sync(0xffffffffu, k, 0);
      }
      return run_c++;
    };
    auto next_chunk = [&](ChunkDesc& d) {
      for (;;) {
        const int c = claim_next();
        if (c >= n_chunks) return c;
        d = load_chunk(a.w.chunk_desc, c);
        if (d.whole) return c;
      }
    };
    ChunkDesc d{};
    int c = next_chunk(d);
    int held_i2[2] = {-1, -1};           // the i2 whose G2 slice each stage holds
    for (int it = 0;; ++it) {
      const int s = it & 1;
      const uint32_t use = (uint32_t)it >> 1;
      Meta& m = meta[s];
      if (c >= n_chunks) {
        if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, a.w.ctl)) break;
        if (lane == 0) m.end = 1;
        __syncwarp();
        cp_async_arrive_noinc(&full[s]);
        if (lane == 0) mbar_arrive(&full[s]);
        break;
      }
      const int x0 = d.x0, p0 = d.p0, p1 = d.p1;
      const int x1 = p1 == p0 ? a.w.pair_row_start[p0 + 1] : d.x1;   // a whole hot prefix
      const int np = p1 - p0 + 1, rows = x1 - x0;
      const int nb = min(rows, C::RB);
      int g3 = 0, gi1 = 0, rs = rows;
      if (lane < nb) g3 = a.w.row_i3[x0 + lane];
      if (lane < np) {
        gi1 = a.w.pair_i1[p0 + lane];
        rs = max(a.w.pair_row_start[p0 + lane], x0) - x0;
      }
      const int i2 = a.w.pair_i2[p0];
      // the first batch's S rows: every load issued now, into registers (lane =
      // (j1, j2) float4), stored once the stage is free
      float4 sv[C::RB];
#pragma unroll
      for (int u = 0; u < C::RB; ++u)
        sv[u] = u < nb ? __ldg(reinterpret_cast<const float4*>(a.w.rowbuf + (size_t)(x0 + u) * C::D) + lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      ChunkDesc dn{};
      const int cn = next_chunk(dn);
      const int flush = cn >= n_chunks || a.w.pair_i2[dn.p0] != i2;
      if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1, a.w.ctl)) break;
      char* st = base + s * C::STAGE_B;
      if (held_i2[s] != i2) {           // (a run of one i2 finds it there already)
        held_i2[s] = i2;
        const uint16_t* h2 = a.w.g2h + (size_t)i2 * C::R * C::NC;
        const uint16_t* l2 = a.w.g2l + (size_t)i2 * C::R * C::NC;
#pragma unroll 8
        for (int i = 0; i < 2 * C::R * C::NC / 256; ++i) {
          const int e = i * 32 + lane, plane = e >> 10, row = (e >> 5) & 31, q = e & 31;
          cp_async16(st + plane * C::G2PLANE + row * (2 * C::G2LD) + 16 * q,
                     (plane ? l2 : h2) + row * C::NC + 8 * q);
        }
      }
#pragma unroll
      for (int pp = 0; pp < C::CP; ++pp) {
        const int i1 = __shfl_sync(0xffffffffu, gi1, pp);
        const int plane = lane >> 4, j1 = (lane >> 2) & 3, q = lane & 3;
        if (pp < np)
          cp_async16(st + C::OFF_G1 + plane * C::G1PLANE + (4 * pp + j1) * (2 * C::G1LD) + 16 * q,
                     (plane ? a.w.g1l : a.w.g1h) + ((size_t)i1 * 4 + j1) * C::R + 8 * q);
      }
      // G3 rows: lane = plane | 16-byte piece
      for (int r = 0; r < nb; ++r) {
        const int i3 = __shfl_sync(0xffffffffu, g3, r);
        const int plane = lane >> 4, q = lane & 15;
        cp_async16(st + C::OFF_G3 + plane * C::GPLANE + r * C::GROW + 16 * q,
                   (plane ? a.w.g3l : a.w.g3h) + (size_t)i3 * 4 * C::R + 8 * q);
      }
      cp_async_arrive_noinc(&full[s]);
      // S rows, converted: lane = (j1, j2)
#pragma unroll
      for (int u = 0; u < C::RB; ++u)
        if (u < nb) bwd_store_s(st + C::OFF_S, u, sv[u], lane);
      if (lane < C::CP) {
        m.rs[lane] = rs;
        m.pi1[lane] = gi1;
      }
      if (lane < nb) m.ri3[lane] = g3;
      int rsq[C::CP];
#pragma unroll
      for (int j = 0; j < C::CP; ++j) rsq[j] = __shfl_sync(0xffffffffu, rs, j);
      const int npairs = bwd_pairs(0, nb, rows, rsq, m.pair, lane);
      __syncwarp();
      if (lane == 0) {
        m.x0 = x0;
        m.x1 = x1;
        m.p0 = p0;
        m.np = np;
        m.i2 = i2;
        m.nb = nb;
        m.npairs = npairs;
        m.end = 0;
        m.flush = flush;
        mbar_arrive(&full[s]);
      }
      c = cn;
      d = dn;
    }
    cp_async_wait_all();
    return;
  }

  // ---------------- consumers (warps 0-7)
  float dg2[2][4][4];                    // (4) of the CTA's current run of chunks of one i2
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) dg2[mt][nt][i] = 0.f;
  for (int it = 0;; ++it) {
    const int s = it & 1;
    if (!mbar_wait(&full[s], ((uint32_t)it >> 1) & 1, a.w.ctl)) break;
    Meta& m = meta[s];
    if (m.end) break;
    const int x0 = m.x0, x1 = m.x1, np = m.np, rows = x1 - x0;
    char* st = base + s * C::STAGE_B;
    const uint32_t g2h = smem_addr(st), g1h = smem_addr(st + C::OFF_G1);
    const uint32_t Sh = smem_addr(st + C::OFF_S), P2h = smem_addr(P2), dph = smem_addr(dP2);
    const char* G3p = st + C::OFF_G3;
    // Later batches (rows of the chunk beyond the first RB: a hot prefix's) are
    // staged by the consumers with their loads issued early: the S rows and
    // row i3 of batch k + 1 before batch k is computed, so that only the G3
    // plane pieces (addressed by i3) are loaded while the batch is stored;
    // thread t handles the (row, 16-byte piece) elements t, t + 256 and
    // t + 512 of a batch.
    float4 ns[3];
    int si3[3];
    if (np > 4) mma_bwd_p2<2>(g2h, g1h, P2, warp, lane);
    else mma_bwd_p2<1>(g2h, g1h, P2, warp, lane);
    {
      // rows (p, j1) from 4 np up to the next multiple of 16 enter the k range of (4):
      // zero them in both bf16 operands (G1 rows: 5 pieces of 16 B per plane row;
      // dP2 rows: 33 pieces)
      const int r0 = 4 * np, r1 = 16 * ((np + 3) >> 2);
      const int nz = (r1 - r0) * 2;            // plane rows
      for (int e = tid; e < nz * 38; e += 256) {
        const int pr = e / 38, q = e - pr * 38, plane = pr & 1, row = r0 + (pr >> 1);
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        if (q < 5)
          *reinterpret_cast<uint4*>(st + C::OFF_G1 + plane * C::G1PLANE + row * (2 * C::G1LD) + 16 * q) = z;
        else
          *reinterpret_cast<uint4*>(dP2 + plane * C::DPPLANE + row * (2 * C::DPLD) + 16 * (q - 5)) = z;
      }
    }
    named_sync(1, 256);
    DP2Acc acc;
    acc.p = -1;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc.c[u][i] = 0.f;
    for (int b0 = 0; b0 < rows; b0 += C::RB) {
      if (b0 > 0) {
        // a later batch: store what was loaded during the previous one
        const int nb = min(C::RB, rows - b0);
        named_sync(1, 256);                      // previous batch fully consumed
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int e = tid + 256 * k, r = e >> 5, q = e & 31;
          if (r < nb) {
            bwd_store_s(st + C::OFF_S, r, ns[k], q);
            const int plane = q >> 4, pc = q & 15;
            *reinterpret_cast<uint4*>(const_cast<char*>(G3p) + plane * C::GPLANE + r * C::GROW + 16 * pc) =
                __ldg(reinterpret_cast<const uint4*>((plane ? a.w.g3l : a.w.g3h) + (size_t)si3[k] * 4 * C::R + 8 * pc));
            if (q == 0) m.ri3[r] = si3[k];
          }
        }
        if (warp == 0) {
          const int npairs = bwd_pairs(b0, b0 + nb, rows, m.rs, m.pair, lane);
          if (lane == 0) m.npairs = npairs;
        }
        named_sync(1, 256);
      }
      if (b0 + C::RB < rows) {                   // the next batch's loads
        const int nb0 = b0 + C::RB;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int e = tid + 256 * k, r = e >> 5, q = e & 31;
          if (nb0 + r < rows) {
            ns[k] = __ldg(reinterpret_cast<const float4*>(a.w.rowbuf + (size_t)(x0 + nb0 + r) * C::D) + q);
            si3[k] = __ldg(a.w.row_i3 + x0 + nb0 + r);
          }
        }
      }
      mma_bwd_dg3(m, P2h, Sh, a.dG3, warp, lane);
      mma_bwd_dp2(m, Sh, G3p, dP2, acc, warp, lane);
    }
    dp2_flush(acc, dP2, warp & 1, warp >> 1, lane);
    named_sync(1, 256);
    mma_bwd_dg2(g1h, dph, dg2, np, warp, lane);
    if (m.flush) dg2_flush(dg2, a.dG2 + (size_t)m.i2 * C::R * C::NC, warp, lane);
    mma_bwd_dg1(dph, g2h, m.pi1, a.dG1, np, warp, lane);
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
  // SPLIT: bf16 planes of the updated cores (tensor-core shape: every count is a
  // multiple of 4 and a float4 of G3 is one (i3, r2) row of its n3 = 4 values)
  uint2* hi[3];
  uint2* lo[3];
  uint16_t* g3th;
  uint16_t* g3tl;
  int R2;
};

template <bool SPLIT>
__global__ void __launch_bounds__(256) k_sgd(SgdArgs a) {
  // four float4 per thread and step, all loads issued before the stores (the
  // cores and their gradients never alias); segment pointers chosen by selects.
  // With SPLIT the updated values also go to the bf16 planes of the chunk
  // kernels (the split of tt_split.cuh, element for element)
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  auto seg_g = [&](int k) { return k == 0 ? a.G[0] : (k == 1 ? a.G[1] : a.G[2]); };
  auto seg_d = [&](int k) { return k == 0 ? a.dG[0] : (k == 1 ? a.dG[1] : a.dG[2]); };
  auto seg_n = [&](int k) { return k == 0 ? a.count[0] : (k == 1 ? a.count[1] : a.count[2]); };
  auto seg_s = [&](int k) { return k == 0 ? a.start[0] : (k == 1 ? a.start[1] : a.start[2]); };
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < a.start[3]; i0 += 4 * stride) {
    float4 g[4], d[4];
    int ks[4];
    int64_t es[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t i = i0 + u * stride;
      ks[u] = -1;
      es[u] = 0;
      if (i < a.start[3]) {
        const int k = i < a.start[1] ? 0 : (i < a.start[2] ? 1 : 2);
        const int64_t e = (i - seg_s(k)) * 4;
        ks[u] = k;
        es[u] = e;
        if (e + 4 <= seg_n(k)) {
          g[u] = *reinterpret_cast<const float4*>(seg_g(k) + e);
          d[u] = *reinterpret_cast<const float4*>(seg_d(k) + e);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = ks[u];
      if (k < 0) continue;
      float* G = seg_g(k);
      float* dG = seg_d(k);
      const int64_t e = es[u], n = seg_n(k);
      if (e + 4 <= n) {
        float4 v = g[u];
        v.x = fmaf(-a.lr, d[u].x, v.x);
        v.y = fmaf(-a.lr, d[u].y, v.y);
        v.z = fmaf(-a.lr, d[u].z, v.z);
        v.w = fmaf(-a.lr, d[u].w, v.w);
        *reinterpret_cast<float4*>(G + e) = v;
        if (a.zero) *reinterpret_cast<float4*>(dG + e) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (SPLIT) {
          uint32_t h0, l0, h1, l1;
          split_bf16x2(v.x, v.y, h0, l0);
          split_bf16x2(v.z, v.w, h1, l1);
          const int64_t j = e >> 2;
          (k == 0 ? a.hi[0] : (k == 1 ? a.hi[1] : a.hi[2]))[j] = make_uint2(h0, h1);
          (k == 0 ? a.lo[0] : (k == 1 ? a.lo[1] : a.lo[2]))[j] = make_uint2(l0, l1);
          if (k == 2) {   // row j = i3 R2 + r2 -> transposed (i3 n3 + j3) R2 + r2
            const int64_t i3 = j / a.R2, r2 = j - i3 * a.R2;
            const int64_t t0 = i3 * 4 * a.R2 + r2;
            a.g3th[t0] = (uint16_t)(h0 & 0xffffu);
            a.g3th[t0 + a.R2] = (uint16_t)(h0 >> 16);
            a.g3th[t0 + 2 * a.R2] = (uint16_t)(h1 & 0xffffu);
            a.g3th[t0 + 3 * a.R2] = (uint16_t)(h1 >> 16);
            a.g3tl[t0] = (uint16_t)(l0 & 0xffffu);
            a.g3tl[t0 + a.R2] = (uint16_t)(l0 >> 16);
            a.g3tl[t0 + 2 * a.R2] = (uint16_t)(l1 & 0xffffu);
            a.g3tl[t0 + 3 * a.R2] = (uint16_t)(l1 >> 16);
          }
        }
      } else {
        for (int64_t t = e; t < n; ++t) {
          G[t] = fmaf(-a.lr, dG[t], G[t]);
          if (a.zero) dG[t] = 0.f;
        }
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

template <int MODE>
static void launch_s_gather(const Shape& s, const Layout& L, const WS& w, const float* grad_out,
                            int64_t nnz, int64_t num_bags, const int64_t* offsets, const float* psw,
                            const SplitArgs& sp, int reuse, cudaStream_t st) {
  const bool cta_gather = s.D == 128;
  // CTA gather: positions per warp so that the grid fills whole waves of the
  // resident CTAs (a partial last wave would run a few CTAs on an idle GPU)
  static int gather_res = 0;
  if (gather_res == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_s_gather_cta<MODE>, 256, 0) !=
            cudaSuccess || per_sm < 1)
      per_sm = 1;
    gather_res = per_sm * sm_count();
  }
  const int64_t per_wave = 8ll * 32 * kGatherBatches * gather_res;
  const int64_t waves = nnz > per_wave ? ceil_div(nnz, per_wave) : 1;
  int span = (int)ceil_div(nnz, 8ll * gather_res * waves);
  if (span < 1) span = 1;
  static int zero_wave = 0;
  if (zero_wave == 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_s_zero, 256, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    zero_wave = per_sm * sm_count();
  }
  const int64_t want = ceil_div(L.rowbuf_rows, 256);
  int grid = want < zero_wave ? (int)want : zero_wave;
  if (grid < split_grid(sp)) grid = split_grid(sp);
  if (grid < 1) grid = 1;
  TT_TIMED("k_s_zero", st, (k_s_zero<<<grid, 256, 0, st>>>(w, s.D, cta_gather ? 8 * span : kSSlice,
                                                             L.rowbuf_rows, sp, reuse)));
  if (cta_gather) {
    TT_TIMED("k_s_gather", st, (k_s_gather_cta<MODE><<<(int)ceil_div(nnz, 8ll * span), 256, 0, st>>>(
                                   w, grad_out, num_bags, psw, offsets, nnz, span)));
  } else {
    const int64_t slices = ceil_div(nnz, kSSlice);
    TT_TIMED("k_s_gather", st, (k_s_gather<MODE><<<(int)ceil_div(slices, 8), 256, 0, st>>>(
                                   w, grad_out, num_bags, s.D, psw, offsets, nnz)));
  }
}

int launch_backward(const Shape& s, const Layout& L, const WS& w, const float* grad_out, int reuse,
                    const float* const cores[3], const int64_t* offsets, int64_t nnz,
                    int64_t num_bags, const Pooling& pool, float* const core_grads[3],
                    float* grad_weights, cudaStream_t st) {
  if (nnz == 0) return TT_EMB_OK;
  const int sms = sm_count();
  if (grad_weights) {
    // the unique rows (the row buffer is free until S takes it), then one dot
    // product per lookup; the forward chunk counter is re-armed first
    if (cudaMemsetAsync(&w.ctl->fwd_chunk_ctr, 0, sizeof(uint32_t), st) != cudaSuccess)
      return TT_EMB_ERR_CUDA;
    // and the prefix-partial checkpoints are emptied: these cores may not be
    // the ones the forward checkpointed
    if (cudaMemsetAsync(w.ckpt, 0, sizeof(uint32_t) * 2 * kCkptSlots, st) != cudaSuccess)
      return TT_EMB_ERR_CUDA;
    const int rc = launch_rows(s, w, cores, 0, st);
    if (rc) return rc;
    int grid = (int)ceil_div(num_bags, 8);
    if (grid > sms * 16) grid = sms * 16;
    TT_TIMED("k_psw_grad", st, (k_psw_grad<<<grid, 256, 0, st>>>(offsets, num_bags, nnz, w.uid,
                                                                  w.rowbuf, s.D, grad_out,
                                                                  grad_weights)));
  }
  // the split planes only where the backward's chunk kernel reads them
  SplitArgs sp = make_split_args(s, w, cores);
  if (!tc_shape(s)) sp.g2l = nullptr;
  switch (pool.mode) {
    case kPoolWeighted:
      launch_s_gather<kPoolWeighted>(s, L, w, grad_out, nnz, num_bags, offsets, pool.psw, sp, reuse,
                                     st);
      break;
    case kPoolMean:
      launch_s_gather<kPoolMean>(s, L, w, grad_out, nnz, num_bags, offsets, nullptr, sp, reuse, st);
      break;
    default:
      launch_s_gather<kPoolSum>(s, L, w, grad_out, nnz, num_bags, offsets, nullptr, sp, reuse, st);
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
  if (tc_shape(s)) {
    static int grid = 0;
    if (grid == 0) {
      cudaFuncSetAttribute(k_bwd_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, MmaBwd::SMEM);
      grid = persistent_grid_bwd((const void*)k_bwd_mma, MmaBwd::THREADS, MmaBwd::SMEM);
    }
    TT_TIMED("k_bwd_mma", st, (k_bwd_mma<<<grid, MmaBwd::THREADS, MmaBwd::SMEM, st>>>(ba)));
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

// Plain SGD over three arrays of the given lengths (the cores of a chain are
// updated three at a time).
int launch_sgd_counts(float* const G[3], float* const dG[3], const int64_t counts[3], float lr,
                      int zero_grads, cudaStream_t st) {
  SgdArgs a;
  a.start[0] = 0;
  for (int k = 0; k < 3; ++k) {
    a.G[k] = G[k];
    a.dG[k] = dG[k];
    a.count[k] = counts[k];
    a.start[k + 1] = a.start[k] + ceil_div(counts[k], 4);
    a.hi[k] = a.lo[k] = nullptr;
  }
  a.lr = lr;
  a.zero = zero_grads ? 1 : 0;
  a.g3th = a.g3tl = nullptr;
  a.R2 = 1;
  if (a.start[3] == 0) return TT_EMB_OK;
  int grid = (int)ceil_div(a.start[3], 4 * 256);
  if (grid > sm_count() * 4) grid = sm_count() * 4;
  if (grid < 1) grid = 1;
  TT_TIMED("k_sgd", st, (k_sgd<false><<<grid, 256, 0, st>>>(a)));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

int launch_sgd(float* const cores[3], float* const grads[3], const Shape& s, float lr,
               int zero_grads, const WS* ws, cudaStream_t st) {
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
  const bool split = ws && ws->g2l;
  a.hi[0] = split ? reinterpret_cast<uint2*>(ws->g1h) : nullptr;
  a.lo[0] = split ? reinterpret_cast<uint2*>(ws->g1l) : nullptr;
  a.hi[1] = split ? reinterpret_cast<uint2*>(ws->g2h) : nullptr;
  a.lo[1] = split ? reinterpret_cast<uint2*>(ws->g2l) : nullptr;
  a.hi[2] = split ? reinterpret_cast<uint2*>(ws->g3h) : nullptr;
  a.lo[2] = split ? reinterpret_cast<uint2*>(ws->g3l) : nullptr;
  a.g3th = split ? ws->g3th : nullptr;
  a.g3tl = split ? ws->g3tl : nullptr;
  a.R2 = s.R2;
  int grid = (int)ceil_div(a.start[3], 4 * 256);
  if (grid > sm_count() * 8) grid = sm_count() * 8;   // one pass of four float4 per thread
  if (grid < 1) grid = 1;
  if (split) {
    TT_TIMED("k_sgd", st, (k_sgd<true><<<grid, 256, 0, st>>>(a)));
  } else {
    TT_TIMED("k_sgd", st, (k_sgd<false><<<grid, 256, 0, st>>>(a)));
  }
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
