// Prefix grouping in ONE cooperative launch.
//
// The same grouping as tt_group.cu (index decomposition and checks, LSD radix
// sort of (key << 32 | position) by the (i2, i1, i3) key, unique rows and
// (i1, i2) prefixes, work chunks), for a grid whose CTAs are all resident at
// once (cooperative launch).  Every CTA owns one contiguous segment of
// L = ceil(nnz / G) sorted positions and keeps its items in registers through
// a phase; phases are separated by grid barriers instead of kernel launches,
// and every cross-CTA prefix is read directly from per-CTA counts that the
// preceding barrier made complete (no look-back chains):
//
//   phase 0    keys, offsets check, per-CTA digit counts of pass 0
//   pass p     CTA prefix + digit totals from the counts, stable rank within
//              the CTA, scatter; the counts of pass p+1 are accumulated per
//              destination CTA as the items land
//   segment    run flags and per-CTA run counts | prefix, CSR arrays, uid
//   chunks     chunk flags over the unique rows, per-CTA counts | prefix, chunks
//
// Grid barriers are capped spins: after kSpinCap polls a CTA sets the timeout
// bit and goes on, so a broken barrier cannot hang the GPU.
#include "tt_internal.cuh"

namespace tt {

constexpr int kCoopThreads = 512;
constexpr int kCoopWarps = kCoopThreads / 32;
constexpr int kCoopMaxGrid = 1024;

struct CoopArgs {
  const int64_t* indices;
  int64_t nnz;
  const int64_t* offsets;
  int64_t B;
  Shape s;
  uint32_t sentinel;
  int passes;
  int L;                  // sorted positions per CTA segment
  int CP, CR;             // chunking parameters
  WS w;
  uint32_t* counts;       // [kMaxPasses][G][kRadix] per-CTA digit counts
  int2* seg_counts;       // [G] (rows, prefixes) per CTA
  int* chunk_counts;      // [G] chunk starts per CTA
};

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Sense-reversal grid barrier over the CTAs of a cooperative launch (capped).
__device__ __forceinline__ void grid_barrier(Ctl* ctl) {
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* count = &ctl->pad[0];
    uint32_t* gen = &ctl->pad[1];
    const uint32_t g = ld_acquire_u32(gen);
    __threadfence();
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
      *count = 0;
      __threadfence();
      st_release_u32(gen, g + 1);
    } else {
      long long spins = 0;
      while (ld_acquire_u32(gen) == g) {
        if (++spins > kSpinCap) {
          set_status(ctl, kStTimeout);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();
}

// Block-wide exclusive scan of one uint32 per thread (kCoopThreads threads).
__device__ __forceinline__ uint32_t coop_scan(uint32_t v, uint32_t* total, uint32_t* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  uint32_t pre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kCoopWarps; ++w) {
    const uint32_t c = sm[w];
    if (w < warp) pre += c;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return pre + x - v;
}

// Sum over CTAs cc < c (pre) and over all CTAs (tot) of a per-CTA int2 count.
__device__ __forceinline__ void cta_prefix2(const int2* cnt, int G, int c, int2* pre, int2* tot,
                                            uint32_t* sm) {
  uint32_t pr = 0, pp = 0, tr = 0, tp = 0;
  for (int cc = threadIdx.x; cc < G; cc += kCoopThreads) {
    const int2 v = __ldcg(cnt + cc);
    tr += (uint32_t)v.x;
    tp += (uint32_t)v.y;
    if (cc < c) {
      pr += (uint32_t)v.x;
      pp += (uint32_t)v.y;
    }
  }
  uint32_t t;
  coop_scan(pr, &t, sm);
  pre->x = (int)t;
  coop_scan(pp, &t, sm);
  pre->y = (int)t;
  coop_scan(tr, &t, sm);
  tot->x = (int)t;
  coop_scan(tp, &t, sm);
  tot->y = (int)t;
}

template <int ITEMS>
__global__ void __launch_bounds__(kCoopThreads, 1) k_group_coop(CoopArgs a) {
  __shared__ uint32_t whist[kCoopWarps][kRadix];   // per-warp digit counts, then offsets
  __shared__ uint32_t red[4][kRadix];              // partial (pre, tot) of the two halves
  __shared__ uint32_t scan_sm[kCoopWarps];
  __shared__ int2 wcnt[kCoopWarps];                 // per-warp (rows, prefixes)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x, G = gridDim.x;
  const int64_t seg0 = (int64_t)c * a.L;
  const int64_t seg1 = seg0 + a.L < a.nnz ? seg0 + a.L : a.nnz;
  constexpr int kSpan = 32 * ITEMS;                // positions per warp

  uint64_t word[ITEMS];

  // ------------------------------------------------------------------ phase 0
  {
    uint32_t* cnt0 = &red[0][0];
    for (int i = tid; i < kRadix; i += kCoopThreads) cnt0[i] = 0;
    __syncthreads();
    bool bad = false;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = seg0 + warp * kSpan + it * 32 + lane;
      uint64_t wv = ~0ull;
      if (i < seg1) {
        const int64_t r = a.indices[i];
        uint32_t key = a.sentinel;
        if (r >= 0 && r < a.s.M) key = group_key(r, a.s);
        else bad = true;
        wv = ((uint64_t)key << 32) | (uint64_t)(uint32_t)i;
      }
      word[it] = wv;
      const uint32_t d = i < seg1 ? (uint32_t)(wv >> 32) & (kRadix - 1) : 0x100u;
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (i < seg1 && lane == __ffs(peers) - 1) atomicAdd(&cnt0[d], __popc(peers));
    }
    if (bad) set_status(a.w.ctl, kStIndex);
    bool bad_off = false;
    for (int64_t b = (int64_t)c * kCoopThreads + tid; b <= a.B; b += (int64_t)G * kCoopThreads) {
      const int64_t v = a.offsets[b];
      if (v < 0 || v > a.nnz) bad_off = true;
      if (b == 0 && v != 0) bad_off = true;
      if (b == a.B && v != a.nnz) bad_off = true;
      if (b < a.B && a.offsets[b + 1] < v) bad_off = true;
    }
    if (bad_off) set_status(a.w.ctl, kStOffsets);
    __syncthreads();
    for (int d = tid; d < kRadix; d += kCoopThreads) {
      a.counts[(size_t)c * kRadix + d] = cnt0[d];
      for (int p = 1; p < a.passes; ++p) a.counts[((size_t)p * G + c) * kRadix + d] = 0;
    }
  }
  grid_barrier(a.w.ctl);

  // ------------------------------------------------------------------ radix passes
  const uint64_t* src = nullptr;
  for (int p = 0; p < a.passes; ++p) {
    uint64_t* dst = (p & 1) ? a.w.keysB : a.w.keysA;
    if (p > 0) {
#pragma unroll
      for (int it = 0; it < ITEMS; ++it) {
        const int64_t i = seg0 + warp * kSpan + it * 32 + lane;
        word[it] = i < seg1 ? __ldcg(src + i) : ~0ull;
      }
    }
    for (int i = tid; i < kCoopWarps * kRadix; i += kCoopThreads) (&whist[0][0])[i] = 0;
    // partial sums over the CTAs of this pass's counts: two threads per digit
    {
      const int d = tid & (kRadix - 1), h = tid >> 8;
      const uint32_t* col = a.counts + (size_t)p * G * kRadix + d;
      const int c0 = h ? G / 2 : 0, c1 = h ? G : G / 2;
      uint32_t pre = 0, tot = 0;
#pragma unroll 8
      for (int cc = c0; cc < c1; ++cc) {
        const uint32_t v = __ldcg(col + (size_t)cc * kRadix);
        tot += v;
        pre += cc < c ? v : 0u;
      }
      red[2 * h][d] = pre;
      red[2 * h + 1][d] = tot;
    }
    __syncthreads();
    // stable rank of each item among its warp's items with the same digit
    const int shift = 32 + kRadixBits * p;
    uint32_t rank[ITEMS];
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = seg0 + warp * kSpan + it * 32 + lane;
      const uint32_t d = (uint32_t)(word[it] >> shift) & (kRadix - 1);
      const uint32_t key = i < seg1 ? d : 0x100u;
      const uint32_t peers = __match_any_sync(0xffffffffu, key);
      const int leader = __ffs(peers) - 1;
      uint32_t prev = 0;
      if (lane == leader && i < seg1) {
        prev = whist[warp][d];
        whist[warp][d] = prev + __popc(peers);
      }
      prev = __shfl_sync(0xffffffffu, prev, leader);
      rank[it] = prev + __popc(peers & lanemask_lt());
      __syncwarp();
    }
    __syncthreads();
    // absolute start of every (warp, digit): bucket base + CTA prefix + warp prefix
    {
      const uint32_t tot_d = tid < kRadix ? red[1][tid] + red[3][tid] : 0u;
      uint32_t all;
      const uint32_t bucket = coop_scan(tot_d, &all, scan_sm);
      if (tid < kRadix) {
        const int d = tid;
        uint32_t run = bucket + red[0][d] + red[2][d];
#pragma unroll
        for (int w = 0; w < kCoopWarps; ++w) {
          const uint32_t n = whist[w][d];
          whist[w][d] = run;
          run += n;
        }
      }
      __syncthreads();
    }
    // scatter; count the next pass's digits by destination CTA
    const bool more = p + 1 < a.passes;
    uint32_t* next = a.counts + (size_t)(p + 1) * G * kRadix;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = seg0 + warp * kSpan + it * 32 + lane;
      const bool live = i < seg1;
      uint32_t pos = 0;
      if (live) {
        const uint32_t d = (uint32_t)(word[it] >> shift) & (kRadix - 1);
        pos = whist[warp][d] + rank[it];
        if (pos < (uint64_t)a.nnz) dst[pos] = word[it];
      }
      if (more) {
        const uint32_t d2 = (uint32_t)(word[it] >> (shift + kRadixBits)) & (kRadix - 1);
        const uint32_t dc = pos / (uint32_t)a.L;
        const uint32_t key = live && pos < (uint64_t)a.nnz ? (dc << 8) | d2 : 0xffffffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, key);
        if (key != 0xffffffffu && lane == __ffs(peers) - 1)
          atomicAdd(&next[(size_t)dc * kRadix + d2], __popc(peers));
      }
    }
    src = dst;
    grid_barrier(a.w.ctl);
  }

  // ------------------------------------------------------------------ segmentation
  const uint64_t* sorted = src;
  const uint64_t M = (uint64_t)a.s.M;
  const uint32_t m3 = (uint32_t)a.s.m3;
  uint32_t rbits[ITEMS], pbits[ITEMS];
  {
    uint32_t wr = 0, wp = 0;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = seg0 + warp * kSpan + it * 32 + lane;
      const bool live = i < seg1;
      const uint64_t wv = live ? __ldcg(sorted + i) : ~0ull;
      const uint64_t pv = (live && i > 0) ? __ldcg(sorted + i - 1) : ~0ull;
      word[it] = wv;
      const uint64_t key = wv >> 32, pk = pv >> 32;
      const bool valid = live && key < M;
      const bool rf = valid && (i == 0 || key != pk);
      const bool pf = valid && (i == 0 || (uint32_t)key / m3 != (uint32_t)pk / m3);
      rbits[it] = __ballot_sync(0xffffffffu, rf);
      pbits[it] = __ballot_sync(0xffffffffu, pf);
      wr += __popc(rbits[it]);
      wp += __popc(pbits[it]);
    }
    if (lane == 0) wcnt[warp] = make_int2((int)wr, (int)wp);
    __syncthreads();
    if (tid == 0) {
      int tr = 0, tp = 0;
      for (int w = 0; w < kCoopWarps; ++w) {
        tr += wcnt[w].x;
        tp += wcnt[w].y;
      }
      a.seg_counts[c] = make_int2(tr, tp);
    }
  }
  grid_barrier(a.w.ctl);
  {
    int2 pre, tot;
    cta_prefix2(a.seg_counts, G, c, &pre, &tot, scan_sm);
    int rr = pre.x, pp = pre.y;          // runs before this warp's first position
    for (int w = 0; w < warp; ++w) {
      rr += wcnt[w].x;
      pp += wcnt[w].y;
    }
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = seg0 + warp * kSpan + it * 32 + lane;
      const bool rf = (rbits[it] >> lane) & 1u, pf = (pbits[it] >> lane) & 1u;
      // runs started at or before this position
      const int ri = rr + __popc(rbits[it] & lt) + (rf ? 1 : 0);
      const int pi = pp + __popc(pbits[it] & lt) + (pf ? 1 : 0);
      if (i < seg1) {
        const uint64_t key = word[it] >> 32;
        const int32_t l = (int32_t)(word[it] & 0xffffffffu);
        a.w.perm[i] = l;
        if ((uint64_t)(uint32_t)l < (uint64_t)a.nnz) {
          if (key >= M) {
            a.w.uid[l] = -1;
            if (i == 0) {            // no valid lookup at all
              a.w.ctl->n_valid = 0;
              a.w.ctl->U_r = 0;
              a.w.ctl->U_12 = 0;
              a.w.row_start[0] = 0;
              a.w.pair_row_start[0] = 0;
            }
          } else {
            const uint32_t q = (uint32_t)key / m3;
            if (pf) {
              const uint32_t q2 = q / (uint32_t)a.s.m1;
              a.w.pair_row_start[pi - 1] = ri - 1;
              a.w.pair_i1[pi - 1] = (int32_t)(q - q2 * (uint32_t)a.s.m1);
              a.w.pair_i2[pi - 1] = (int32_t)q2;
            }
            if (rf) {
              a.w.row_start[ri - 1] = (int32_t)i;
              a.w.row_i3[ri - 1] = (int32_t)((uint32_t)key - q * m3);
              a.w.row_pair[ri - 1] = pi - 1;
            }
            a.w.uid[l] = ri - 1;
            const bool last = (i + 1 == a.nnz) || (__ldcg(sorted + i + 1) >> 32) >= M;
            if (last) {
              a.w.ctl->n_valid = (int32_t)(i + 1);
              a.w.ctl->U_r = ri;
              a.w.ctl->U_12 = pi;
              a.w.row_start[ri] = (int32_t)(i + 1);
              a.w.pair_row_start[pi] = ri;
            }
          }
        }
      }
      rr += __popc(rbits[it]);
      pp += __popc(pbits[it]);
    }
  }
  grid_barrier(a.w.ctl);

  // ------------------------------------------------------------------ chunks
  {
    const int U = __ldcg(&a.w.ctl->U_r);
    const int Lr = (U + G - 1) / G;
    const int x0 = c * Lr, x1 = min(x0 + Lr, U);
    // Lr <= L <= kCoopThreads * ITEMS, so ITEMS rounds of the block cover a segment
    uint32_t fl[ITEMS];
    uint32_t mine = 0;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      const int x = x0 + k * kCoopThreads + tid;
      bool f = false;
      if (x < x1) {
        const int32_t p = __ldcg(a.w.row_pair + x);
        const int32_t f0 = __ldcg(a.w.pair_row_start + p);
        const int32_t nr = __ldcg(a.w.pair_row_start + p + 1) - f0;
        if (x != f0) {
          f = ((x - f0) % a.CR) == 0;
        } else if (p == 0) {
          f = true;
        } else {
          const int32_t pf = __ldcg(a.w.pair_row_start + p - 1);
          f = (p % a.CP) == 0 || __ldcg(a.w.pair_i2 + p) != __ldcg(a.w.pair_i2 + p - 1) || nr > a.CR ||
              (f0 - pf) > a.CR;
        }
      }
      fl[k] = f ? 1u : 0u;
      mine += fl[k];
    }
    uint32_t tot;
    coop_scan(mine, &tot, scan_sm);
    if (tid == 0) a.chunk_counts[c] = (int)tot;
    grid_barrier(a.w.ctl);
    int2 pre2, tot2;
    {
      // reuse the int2 prefix helper with a zero second component
      uint32_t pr = 0, tt = 0;
      for (int cc = tid; cc < G; cc += kCoopThreads) {
        const uint32_t v = (uint32_t)__ldcg(a.chunk_counts + cc);
        tt += v;
        if (cc < c) pr += v;
      }
      uint32_t t;
      coop_scan(pr, &t, scan_sm);
      pre2.x = (int)t;
      coop_scan(tt, &t, scan_sm);
      tot2.x = (int)t;
    }
    int base = pre2.x;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      uint32_t t;
      const uint32_t ex = coop_scan(fl[k], &t, scan_sm);
      const int x = x0 + k * kCoopThreads + tid;
      if (fl[k]) {
        const int ci = base + (int)ex;
        const int32_t p = __ldcg(a.w.row_pair + x);
        const bool first = __ldcg(a.w.pair_row_start + p) == x;
        a.w.chunk_start[ci] = x;
        a.w.chunk_desc[ci] = make_int2(x, p | (first ? (int32_t)0x80000000 : 0));
      }
      base += (int)t;
    }
    if (c == 0 && tid == 0) {
      a.w.ctl->n_chunks = tot2.x;
      a.w.chunk_start[tot2.x] = U;
      a.w.chunk_desc[tot2.x] = make_int2(U, __ldcg(&a.w.ctl->U_12) | (int32_t)0x80000000);
    }
  }
}

// Largest ITEMS the cooperative path is compiled for.
constexpr int kCoopItemsMax = 16;

template <int ITEMS>
static int launch_coop_items(const CoopArgs& ca, int G, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kCoopThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  TT_TIMED("k_group_coop", st, (e = cudaLaunchKernelEx(&cfg, k_group_coop<ITEMS>, ca)));
  return e == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

// Grid of the cooperative grouping (all CTAs resident), 0 if unavailable.
int coop_grid() {
  static int grid = -1;
  if (grid < 0) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_group_coop<kCoopItemsMax>,
                                                      kCoopThreads, 0) != cudaSuccess)
      per_sm = 0;
    int coop = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    grid = coop ? per_sm * sm_count() : 0;
    if (grid > kCoopMaxGrid) grid = kCoopMaxGrid;
  }
  return grid;
}

size_t coop_scratch_bytes() {
  return sizeof(uint32_t) * kMaxPasses * kCoopMaxGrid * kRadix + sizeof(int2) * kCoopMaxGrid +
         sizeof(int) * kCoopMaxGrid;
}

// Runs the whole grouping as one cooperative launch if the batch fits the
// register-resident segments; returns TT_EMB_ERR_UNSUPPORTED otherwise (the
// caller then uses the multi-kernel path).
int launch_group_coop(const Shape& s, const Layout& L, const WS& w, void* scratch,
                      const int64_t* indices, int64_t nnz, const int64_t* offsets,
                      int64_t num_bags, int pairs_per_chunk, int rows_per_chunk,
                      cudaStream_t st) {
  const int G = coop_grid();
  if (G < 2 || nnz <= 0) return TT_EMB_ERR_UNSUPPORTED;
  const int64_t Lseg = ceil_div(nnz, G);
  if (Lseg > (int64_t)kCoopThreads * kCoopItemsMax) return TT_EMB_ERR_UNSUPPORTED;
  CoopArgs ca;
  ca.indices = indices;
  ca.nnz = nnz;
  ca.offsets = offsets;
  ca.B = num_bags;
  ca.s = s;
  ca.sentinel = L.key_bits >= 32 ? 0xffffffffu : ((1u << L.key_bits) - 1u);
  ca.passes = L.passes;
  ca.L = (int)Lseg;
  ca.CP = pairs_per_chunk;
  ca.CR = rows_per_chunk;
  ca.w = w;
  char* sc = static_cast<char*>(scratch);
  ca.counts = reinterpret_cast<uint32_t*>(sc);
  ca.seg_counts = reinterpret_cast<int2*>(sc + sizeof(uint32_t) * kMaxPasses * kCoopMaxGrid * kRadix);
  ca.chunk_counts = reinterpret_cast<int*>(reinterpret_cast<char*>(ca.seg_counts) +
                                           sizeof(int2) * kCoopMaxGrid);
  if (Lseg <= kCoopThreads * 4) return launch_coop_items<4>(ca, G, st);
  if (Lseg <= kCoopThreads * 8) return launch_coop_items<8>(ca, G, st);
  return launch_coop_items<16>(ca, G, st);
}

}  // namespace tt
