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
//   pass p     stable rank within the CTA and its digit counts | CTA prefix +
//              digit totals from all CTAs' counts, scatter
//   segment    run flags and per-CTA run counts | prefix, CSR arrays, uid
//   chunks     chunk flags over the unique rows, per-CTA counts | prefix, chunks
//
// Grid barriers are capped spins: after kSpinCap polls a CTA sets the timeout
// bit and goes on, so a broken barrier cannot hang the GPU.
#include "tt_coop.cuh"

namespace tt {

struct CoopArgs {
  Idx indices;
  int64_t nnz;
  const int64_t* offsets;
  int64_t B;
  Shape s;
  uint32_t sentinel;
  int passes;
  int L;                  // sorted positions per CTA segment
  int CP, CR;             // chunking parameters
  WS w;
  uint32_t* counts;       // [kMaxPasses][G][kRadix / 2] per-CTA digit counts, two uint16 a word
  int4* seg_counts;       // [G] (rows, prefixes, valid lookups, 0) per CTA
  int* chunk_counts;      // [G] chunk starts per CTA
  uint32_t* bar;          // grid barrier words (zeroed before the launch)
  unsigned long long* trace;   // [16] phase timestamps of CTA 0 (ns, %globaltimer)
};

template <int ITEMS>
__global__ void __launch_bounds__(kCoopThreads, 1) k_group_coop(CoopArgs a) {
  __shared__ uint32_t whist[kCoopWarps][kRadix];   // per-warp digit counts, then offsets
  __shared__ __align__(16) uint32_t red[kCoopWarps][kRadix];   // per-warp partial digit sums
  __shared__ uint32_t scan_sm[kCoopWarps];
  __shared__ int2 wcnt[kCoopWarps];                 // per-warp (rows, prefixes)
  __shared__ uint4 sum_sm[kCoopWarps];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int c = blockIdx.x, G = gridDim.x;
  int tstep = 0;
  auto stamp = [&]() {
    if (c == 0 && tid == 0 && tstep < 16) a.trace[tstep] = global_ns();
    ++tstep;
  };
  stamp();
  const int64_t seg0 = (int64_t)c * a.L;
  const int64_t seg1 = seg0 + a.L < a.nnz ? seg0 + a.L : a.nnz;
  constexpr int kSpan = 32 * ITEMS;                // positions per warp

  uint64_t word[ITEMS];

  // ------------------------------------------------------------------ phase 0
  {
    // every load of the phase is issued before any arithmetic: the CTA's
    // indices and the bounds of the bag this thread checks
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = seg0 + warp * kSpan + it * 32 + lane;
      word[it] = i < seg1 ? (uint64_t)a.indices.at(i) : 0ull;
    }
    const int64_t bt = (int64_t)c * kCoopThreads + tid;
    int64_t o0 = 0, o1 = 0;
    if (bt <= a.B) o0 = __ldg(a.offsets + bt);
    if (bt < a.B) o1 = __ldg(a.offsets + bt + 1);
    bool bad = false;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = seg0 + warp * kSpan + it * 32 + lane;
      uint64_t wv = ~0ull;
      if (i < seg1) {
        const int64_t r = (int64_t)word[it];
        uint32_t key = a.sentinel;
        if (r >= 0 && r < a.s.M) key = group_key(r, a.s);
        else bad = true;
        wv = ((uint64_t)key << 32) | (uint64_t)(uint32_t)i;
      }
      word[it] = wv;
    }
    if (bad) set_status(a.w.ctl, kStIndex);
    bool bad_off = false;
    for (int64_t b = bt; b <= a.B; b += (int64_t)G * kCoopThreads) {
      int64_t v = o0, v1 = o1;
      if (b != bt) {                       // batches of more than G * 512 bags
        v = a.offsets[b];
        v1 = b < a.B ? a.offsets[b + 1] : 0;
      }
      if (v < 0 || v > a.nnz) bad_off = true;
      if (b == 0 && v != 0) bad_off = true;
      if (b == a.B && v != a.nnz) bad_off = true;
      if (b < a.B && v1 < v) bad_off = true;
    }
    if (bad_off) set_status(a.w.ctl, kStOffsets);
  }

  // ------------------------------------------------------------------ radix passes
  // per pass: stable rank within the CTA -> this CTA's digit counts -> barrier ->
  // CTA prefix and digit totals from all CTAs' counts -> scatter -> barrier
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
    __syncthreads();
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
    // this CTA's digit counts (at most L <= 512 ITEMS < 2^16 each), one 512-byte row
    uint32_t* cnt = a.counts + (size_t)p * G * (kRadix / 2);
    if (tid < kRadix / 2) {
      uint32_t n0 = 0, n1 = 0;
#pragma unroll
      for (int w = 0; w < kCoopWarps; ++w) {
        n0 += whist[w][2 * tid];
        n1 += whist[w][2 * tid + 1];
      }
      cnt[(size_t)c * (kRadix / 2) + tid] = n0 | (n1 << 16);
    }
    grid_barrier(a.bar, a.w.ctl);
    stamp();
    // CTA prefix and total of every digit from all CTAs' rows: warp w reads rows
    // w, w + 16, ..., lane l the 16 bytes of digits 8 l .. 8 l + 7 (a warp load
    // is one whole 512-byte row); the 16 warps' partial sums meet in shared memory
    uint32_t my_pre = 0, my_tot = 0;
    {
      uint32_t pre[8], tot[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) pre[k] = tot[k] = 0u;
      const uint4* rows = reinterpret_cast<const uint4*>(cnt);
#pragma unroll 5
      for (int cc = warp; cc < G; cc += kCoopWarps) {
        const uint4 v = __ldcg(rows + (size_t)cc * (kRadix / 8) + lane);
        const bool before = cc < c;
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t lo = wv[j] & 0xffffu, hi = wv[j] >> 16;
          tot[2 * j] += lo;
          tot[2 * j + 1] += hi;
          pre[2 * j] += before ? lo : 0u;
          pre[2 * j + 1] += before ? hi : 0u;
        }
      }
      uint4* mine = reinterpret_cast<uint4*>(&red[warp][8 * lane]);
      mine[0] = make_uint4(pre[0], pre[1], pre[2], pre[3]);
      mine[1] = make_uint4(pre[4], pre[5], pre[6], pre[7]);
      __syncthreads();
      if (tid < kRadix)
#pragma unroll
        for (int w = 0; w < kCoopWarps; ++w) my_pre += red[w][tid];
      __syncthreads();
      mine[0] = make_uint4(tot[0], tot[1], tot[2], tot[3]);
      mine[1] = make_uint4(tot[4], tot[5], tot[6], tot[7]);
      __syncthreads();
      if (tid < kRadix)
#pragma unroll
        for (int w = 0; w < kCoopWarps; ++w) my_tot += red[w][tid];
    }
    // absolute start of every (warp, digit): bucket base + CTA prefix + warp prefix
    {
      uint32_t all;
      const uint32_t bucket = coop_scan(tid < kRadix ? my_tot : 0u, &all, scan_sm);
      if (tid < kRadix) {
        const int d = tid;
        uint32_t run = bucket + my_pre;
#pragma unroll
        for (int w = 0; w < kCoopWarps; ++w) {
          const uint32_t n = whist[w][d];
          whist[w][d] = run;
          run += n;
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = seg0 + warp * kSpan + it * 32 + lane;
      if (i < seg1) {
        const uint32_t d = (uint32_t)(word[it] >> shift) & (kRadix - 1);
        const uint32_t pos = whist[warp][d] + rank[it];
        if (pos < (uint64_t)a.nnz) dst[pos] = word[it];
      }
    }
    src = dst;
    grid_barrier(a.bar, a.w.ctl);
    stamp();
  }

  // ------------------------------------------------------------------ segmentation
  const uint64_t* sorted = src;
  const uint64_t M = (uint64_t)a.s.M;
  const uint32_t m3 = (uint32_t)a.s.m3;
  uint32_t rbits[ITEMS], pbits[ITEMS];
  {
    uint32_t wr = 0, wp = 0, wv_cnt = 0;
    // one load per position; the word before a position comes from the lane
    // before, from lane 31 of the item before, or (first position of the warp)
    // from one more load
    const int64_t wbase = seg0 + warp * kSpan;
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = wbase + it * 32 + lane;
      word[it] = i < seg1 ? __ldcg(sorted + i) : ~0ull;
    }
    const uint64_t before_warp = (wbase > 0 && wbase < seg1) ? __ldcg(sorted + wbase - 1) : ~0ull;
    uint64_t carry = before_warp;          // the word before this item's lane 0
#pragma unroll
    for (int it = 0; it < ITEMS; ++it) {
      const int64_t i = wbase + it * 32 + lane;
      const bool live = i < seg1;
      const uint64_t wv = word[it];
      const uint64_t up = __shfl_up_sync(0xffffffffu, wv, 1);
      uint64_t pv = lane > 0 ? up : carry;
      carry = __shfl_sync(0xffffffffu, wv, 31);
      if (!live || i == 0) pv = ~0ull;
      const uint64_t key = wv >> 32, pk = pv >> 32;
      const bool valid = live && key < M;
      const bool rf = valid && (i == 0 || key != pk);
      const bool pf = valid && (i == 0 || fdiv((uint32_t)key, a.s.fm3) != fdiv((uint32_t)pk, a.s.fm3));
      rbits[it] = __ballot_sync(0xffffffffu, rf);
      pbits[it] = __ballot_sync(0xffffffffu, pf);
      wr += __popc(rbits[it]);
      wp += __popc(pbits[it]);
      wv_cnt += __popc(__ballot_sync(0xffffffffu, valid));
    }
    if (lane == 0) wcnt[warp] = make_int2((int)wr, (int)wp);
    const uint4 t = coop_sum4(make_uint4(lane == 0 ? wr : 0u, lane == 0 ? wp : 0u,
                                         lane == 0 ? wv_cnt : 0u, 0u), sum_sm);
    if (tid == 0) a.seg_counts[c] = make_int4((int)t.x, (int)t.y, (int)t.z, 0);
  }
  grid_barrier(a.bar, a.w.ctl);
  stamp();
  int u_rows = 0, u_pairs = 0;   // unique rows and prefixes (every CTA has the totals)
  {
    uint4 mine_pre = make_uint4(0, 0, 0, 0), mine_tot = make_uint4(0, 0, 0, 0);
    for (int cc = tid; cc < G; cc += kCoopThreads) {
      const int4 v = __ldcg(a.seg_counts + cc);
      mine_tot.x += v.x;
      mine_tot.y += v.y;
      mine_tot.z += v.z;
      if (cc < c) {
        mine_pre.x += v.x;
        mine_pre.y += v.y;
      }
    }
    const uint4 pre = coop_sum4(mine_pre, sum_sm);
    const uint4 tot = coop_sum4(mine_tot, sum_sm);
    const int64_t nv = (int64_t)tot.z;     // valid lookups (they sort first)
    u_rows = (int)tot.x;
    u_pairs = (int)tot.y;
    if (c == 0 && tid == 0) {
      a.w.ctl->method = kGroupCoop;
      a.w.ctl->n_valid = (int32_t)nv;
      a.w.ctl->U_r = (int32_t)tot.x;
      a.w.ctl->U_12 = (int32_t)tot.y;
      a.w.row_start[tot.x] = (int32_t)nv;
      a.w.pair_row_start[tot.y] = (int32_t)tot.x;
    }
    int rr = (int)pre.x, pp = (int)pre.y;   // runs before this warp's first position
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
          } else {
            const uint32_t q = fdiv((uint32_t)key, a.s.fm3);
            if (pf) {
              const uint32_t q2 = fdiv(q, a.s.fm1);
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
          }
        }
      }
      rr += __popc(rbits[it]);
      pp += __popc(pbits[it]);
    }
  }
  grid_barrier(a.bar, a.w.ctl);
  stamp();

  // ------------------------------------------------------------------ chunks
  // Chunk starts, enumerated per unique prefix p (rows f0 .. f1-1 of the
  // prefix, nr = f1 - f0): its first row f0 starts a chunk when p is 0 or a
  // multiple of CP, its i2 differs from prefix p-1's, or p or p-1 holds more
  // than CR rows; rows f0 + k CR (k >= 1) start the CR-row pieces of a hot
  // prefix.  Each thread owns Pt consecutive prefixes of the CTA's range and
  // issues all their loads at once.  Counted as (head chunks) | (later pieces)
  // << 16 (at most 8192 heads and 2^16 - 1 pieces per CTA for the batches this
  // launch takes): the claim order puts every later piece after all heads.
  {
    const int U = u_rows, P = u_pairs;
    const int Lp = (P + G - 1) / G;
    const int y0 = c * Lp, y1 = min(y0 + Lp, P);
    const int Pt = (Lp + kCoopThreads - 1) / kCoopThreads;   // <= ITEMS (P <= nnz)
    const int yt = y0 + tid * Pt;
    int f0s[ITEMS], nrs[ITEMS];
    uint32_t firsts = 0, mine = 0;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      const int pp = yt + k;
      f0s[k] = 0;
      nrs[k] = 0;
      if (k < Pt && pp < y1) {
        const int32_t f0 = __ldcg(a.w.pair_row_start + pp);
        const int32_t f1 = __ldcg(a.w.pair_row_start + pp + 1);
        const int32_t pf = pp > 0 ? __ldcg(a.w.pair_row_start + pp - 1) : 0;
        const int32_t i2 = __ldcg(a.w.pair_i2 + pp);
        const int32_t i2p = pp > 0 ? __ldcg(a.w.pair_i2 + pp - 1) : -1;
        const int32_t nr = f1 - f0;
        const bool f = pp == 0 || (pp % a.CP) == 0 || i2 != i2p || nr > a.CR || (f0 - pf) > a.CR;
        f0s[k] = f0;
        nrs[k] = nr;
        firsts |= (f ? 1u : 0u) << k;
        mine += (f ? 1u : 0u) + ((uint32_t)((nr - 1) / a.CR) << 16);
      }
    }
    uint32_t tot;
    const uint32_t ex = coop_scan(mine, &tot, scan_sm);
    if (tid == 0) a.chunk_counts[c] = (int)tot;
    grid_barrier(a.bar, a.w.ctl);
    stamp();
    uint4 pr = make_uint4(0, 0, 0, 0);
    for (int cc = tid; cc < G; cc += kCoopThreads) {
      const uint32_t v = (uint32_t)__ldcg(a.chunk_counts + cc);
      pr.z += v & 0xffffu;
      pr.w += v >> 16;
      if (cc < c) {
        pr.x += v & 0xffffu;
        pr.y += v >> 16;
      }
    }
    const uint4 ps = coop_sum4(pr, sum_sm);
    const uint32_t H = ps.z;                          // head chunks of the whole batch
    uint32_t hr = ps.x + (ex & 0xffffu), tr = H + ps.y + (ex >> 16);
    int ci = (int)(hr + tr - H);                      // natural (row-order) chunk number
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      const int pp = yt + k;
      if (k < Pt && pp < y1) {
        if ((firsts >> k) & 1u) {
          a.w.chunk_start[ci] = f0s[k];
          a.w.chunk_desc[ci] = make_int2(f0s[k], pp | (int32_t)0x80000000);
          a.w.chunk_order[hr++] = ci;
          ++ci;
        }
        for (int x = f0s[k] + a.CR; x < f0s[k] + nrs[k]; x += a.CR) {
          a.w.chunk_start[ci] = x;
          a.w.chunk_desc[ci] = make_int2(x, pp);
          a.w.chunk_order[tr++] = ci;
          ++ci;
        }
      }
    }
    stamp();
    if (c == 0 && tid == 0) {
      const int n = (int)(ps.z + ps.w);
      a.w.ctl->n_chunks = n;
      a.w.chunk_start[n] = U;
      a.w.chunk_desc[n] = make_int2(U, P | (int32_t)0x80000000);
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
  return sizeof(uint32_t) * kMaxPasses * kCoopMaxGrid * (kRadix / 2) + sizeof(int4) * kCoopMaxGrid +
         sizeof(int) * kCoopMaxGrid + 16 * sizeof(unsigned long long);
}

// Runs the whole grouping as one cooperative launch if the batch fits the
// register-resident segments; returns TT_EMB_ERR_UNSUPPORTED otherwise (the
// caller then uses the multi-kernel path).
int launch_group_coop(const Shape& s, const Layout& L, const WS& w, void* scratch,
                      Idx indices, int64_t nnz, const int64_t* offsets,
                      int64_t num_bags, int pairs_per_chunk, int rows_per_chunk,
                      cudaStream_t st) {
  const int G = coop_grid();
  if (G < 4 || G > kCoopMaxGrid || nnz <= 0) return TT_EMB_ERR_UNSUPPORTED;
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
  // barrier words: the digit-histogram area, zeroed by the grouping's memset and
  // otherwise unused on this path (18 words 128 bytes apart = 2.3 KB)
  ca.bar = w.hist;
  ca.counts = reinterpret_cast<uint32_t*>(sc);
  ca.seg_counts = reinterpret_cast<int4*>(sc + sizeof(uint32_t) * kMaxPasses * kCoopMaxGrid * (kRadix / 2));
  ca.chunk_counts = reinterpret_cast<int*>(reinterpret_cast<char*>(ca.seg_counts) +
                                           sizeof(int4) * kCoopMaxGrid);
  ca.trace = reinterpret_cast<unsigned long long*>(ca.chunk_counts + kCoopMaxGrid);
  if (Lseg <= kCoopThreads * 4) return launch_coop_items<4>(ca, G, st);
  if (Lseg <= kCoopThreads * 8) return launch_coop_items<8>(ca, G, st);
  if (Lseg <= kCoopThreads * 12) return launch_coop_items<12>(ca, G, st);
  return launch_coop_items<16>(ca, G, st);
}

}  // namespace tt
