// Prefix grouping of a batch of TT lookups on the device.
//
// FlowTT (summary card, key innovations; abstract) groups the lookups that
// share high-order TT-core indices so that every shared partial product is
// formed once.  Here that grouping is:
//
//   1. k_prepare   index decomposition + range check, offsets check, digit
//                  histograms of the grouping key
//   2. k_scatter   one LSD radix pass per 8-bit digit (onesweep style:
//                  tiles ranked in shared memory, tile prefixes chained by
//                  decoupled look-back), sorting (key << 32 | position)
//   3. k_segment   run boundaries of rows and of (i1, i2) prefixes, their
//                  CSR arrays and the unique row of every lookup
//   4. k_chunks    work chunks for the persistent contraction kernels
//
// The key is (i2, i1, i3) with i3 least significant: runs of equal (i1, i2)
// are the shared prefixes, and prefixes that read the same G2 slice are
// adjacent, so a chunk of prefixes stages one G2 slice.
//
// Every inter-CTA wait is a capped poll of a look-back word published by a
// CTA that took its tile number earlier (tile numbers come from an atomic
// counter, so a waited-on tile is always already running); a poll that runs
// out sets the timeout bit and the kernel finishes.
#include "tt_internal.cuh"

namespace tt {

struct PrepArgs {
  Idx indices;
  int64_t nnz;
  const int64_t* offsets;
  int64_t B;
  Shape s;
  uint32_t sentinel;
  int passes;
  WS w;
  uint32_t* zero32;
  size_t zero32_words;
  unsigned long long* zero64;
  size_t zero64_words;
  uint32_t* zero32b;
  size_t zero32b_words;
};

__global__ void __launch_bounds__(256) k_prepare(PrepArgs a) {
  __shared__ uint32_t sh[kMaxPasses * kRadix];
  const int tid = threadIdx.x, lane = tid & 31;
  for (int i = tid; i < a.passes * kRadix; i += blockDim.x) sh[i] = 0;
  if (blockIdx.x == 0 && tid == 0) a.w.ctl->method = kGroupMulti;
  __syncthreads();

  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  bool bad_index = false;
  // warp-uniform loop so that the digit counts can be aggregated per warp
  for (int64_t l0 = (int64_t)blockIdx.x * blockDim.x + (tid & ~31); l0 < a.nnz; l0 += stride) {
    const int64_t l = l0 + lane;
    uint32_t key = a.sentinel;
    const bool live = l < a.nnz;
    if (live) {
      const int64_t r = a.indices.at(l);
      if (r >= 0 && r < a.s.M) key = group_key(r, a.s);
      else bad_index = true;
    }
    for (int p = 0; p < a.passes; ++p) {
      const uint32_t d = live ? ((key >> (kRadixBits * p)) & (kRadix - 1)) : 0xffffffffu;
      const uint32_t peers = __match_any_sync(0xffffffffu, d);
      if (live && lane == __ffs(peers) - 1) atomicAdd(&sh[p * kRadix + d], __popc(peers));
    }
  }
  if (bad_index) set_status(a.w.ctl, kStIndex);

  // offsets must be CSR: offsets[0] = 0, offsets[B] = nnz, non-decreasing
  bool bad_off = false;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + tid; b <= a.B; b += stride) {
    const int64_t v = a.offsets[b];
    if (v < 0 || v > a.nnz) bad_off = true;
    if (b == 0 && v != 0) bad_off = true;
    if (b == a.B && v != a.nnz) bad_off = true;
    if (b < a.B && a.offsets[b + 1] < v) bad_off = true;
  }
  if (bad_off) set_status(a.w.ctl, kStOffsets);

  // clear the look-back words of the passes that follow
  for (size_t i = (size_t)blockIdx.x * blockDim.x + tid; i < a.zero32_words; i += stride) a.zero32[i] = 0;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + tid; i < a.zero64_words; i += stride) a.zero64[i] = 0;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + tid; i < a.zero32b_words; i += stride) a.zero32b[i] = 0;

  __syncthreads();
  uint32_t* h = a.w.hist + (size_t)(blockIdx.x % kHistCopies) * kMaxPasses * kRadix;
  for (int i = tid; i < a.passes * kRadix; i += blockDim.x)
    if (sh[i]) atomicAdd(&h[i], sh[i]);
}

struct ScatterArgs {
  Idx indices;              // pass 0 reads the indices directly
  const uint64_t* in;
  uint64_t* out;
  int64_t nnz;
  Shape s;
  uint32_t sentinel;
  int pass;
  int n_tiles;
  WS w;
};

__global__ void __launch_bounds__(kSortThreads) k_scatter(ScatterArgs a) {
  __shared__ uint32_t whist[kSortThreads / 32][kRadix];
  __shared__ uint32_t digit_base[kRadix];
  __shared__ uint32_t scan8[8];
  __shared__ uint32_t tile_sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) tile_sh = atomicAdd(&a.w.ctl->sort_tile_ctr[a.pass], 1u);
  for (int i = tid; i < (kSortThreads / 32) * kRadix; i += kSortThreads) (&whist[0][0])[i] = 0;
  uint32_t total;
  uint32_t hsum = 0;
#pragma unroll
  for (int c = 0; c < kHistCopies; ++c) hsum += a.w.hist[(c * kMaxPasses + a.pass) * kRadix + tid];
  const uint32_t bucket = block_exclusive_scan_256(hsum, &total, scan8);
  __syncthreads();
  const uint32_t tile = tile_sh;
  const int64_t base = (int64_t)tile * kSortTile;
  const int shift = 32 + kRadixBits * a.pass;

  uint64_t word[kSortItems];
  uint32_t dig[kSortItems];
  uint32_t rank[kSortItems];
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const int64_t i = base + warp * (32 * kSortItems) + it * 32 + lane;
    uint64_t wv = ~0ull;
    if (i < a.nnz) {
      if (a.pass == 0) {
        const int64_t r = a.indices.at(i);
        const uint32_t key = (r >= 0 && r < a.s.M) ? group_key(r, a.s) : a.sentinel;
        wv = ((uint64_t)key << 32) | (uint64_t)(uint32_t)i;
      } else {
        wv = a.in[i];
      }
    }
    word[it] = wv;
    dig[it] = (uint32_t)(wv >> shift) & (kRadix - 1);
  }
  // stable rank of every item among the items of its warp with the same digit
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const uint32_t d = dig[it];
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const int leader = __ffs(peers) - 1;
    uint32_t prev = 0;
    if (lane == leader) {
      prev = whist[warp][d];
      whist[warp][d] = prev + __popc(peers);
    }
    prev = __shfl_sync(0xffffffffu, prev, leader);
    rank[it] = prev + __popc(peers & lanemask_lt());
    __syncwarp();
  }
  __syncthreads();
  // per digit: exclusive prefix over the warps, tile count, then the look-back
  {
    const int d = tid;
    uint32_t sum = 0;
#pragma unroll
    for (int w = 0; w < kSortThreads / 32; ++w) {
      const uint32_t c = whist[w][d];
      whist[w][d] = sum;
      sum += c;
    }
    uint32_t* st = a.w.sort_status + ((size_t)a.pass * a.n_tiles) * kRadix + d;
    uint32_t excl = 0;
    if (tile == 0) {
      st_relaxed_u32(st, kFlagIncl | sum);
    } else {
      st_relaxed_u32(st + (size_t)tile * kRadix, kFlagAgg | sum);
      // walk back 8 predecessor tiles per round trip
      int64_t j = (int64_t)tile - 1;
      long long spins = 0;
      while (j >= 0) {
        uint32_t v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          v[k] = (j - k >= 0) ? ld_relaxed_u32(st + (size_t)(j - k) * kRadix) : kFlagIncl;
        int k = 0;
        bool done = false;
        for (; k < 8; ++k) {
          const uint32_t f = v[k] & kFlagMask;
          if (f == 0) break;
          excl += v[k] & kValMask;
          if (f == kFlagIncl) {
            done = true;
            break;
          }
        }
        if (done) break;
        j -= k;
        if (k < 8 && ++spins > kSpinCap) {
          set_status(a.w.ctl, kStTimeout);
          break;
        }
      }
      st_relaxed_u32(st + (size_t)tile * kRadix, kFlagIncl | ((excl + sum) & kValMask));
    }
    digit_base[d] = bucket + excl;
  }
  __syncthreads();
#pragma unroll
  for (int it = 0; it < kSortItems; ++it) {
    const int64_t i = base + warp * (32 * kSortItems) + it * 32 + lane;
    if (i < a.nnz) {
      const uint32_t d = dig[it];
      const uint32_t pos = digit_base[d] + whist[warp][d] + rank[it];
      if (pos < (uint64_t)a.nnz) a.out[pos] = word[it];
    }
  }
}

struct SegArgs {
  const uint64_t* sorted;
  int64_t nnz;
  Shape s;
  WS w;
};

// Row and prefix runs of the sorted keys; 64-bit look-back word:
// flag (2 bits) | rows so far (31 bits) | prefixes so far (31 bits).
__global__ void __launch_bounds__(kScanThreads) k_segment(SegArgs a) {
  __shared__ uint32_t scan8[8];
  __shared__ uint32_t tile_sh;
  __shared__ unsigned long long prefix_sh;
  const int tid = threadIdx.x;
  if (tid == 0) tile_sh = atomicAdd(&a.w.ctl->seg_tile_ctr, 1u);
  __syncthreads();
  const uint32_t tile = tile_sh;
  const int64_t k0 = (int64_t)tile * kScanTile + (int64_t)tid * kScanItems;
  const uint64_t M = (uint64_t)a.s.M;
  const uint32_t m3 = (uint32_t)a.s.m3;

  uint64_t w[kScanItems];
  uint32_t rflag = 0, pflag = 0;
  uint64_t prev = (k0 > 0 && k0 - 1 < a.nnz) ? a.sorted[k0 - 1] : ~0ull;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t k = k0 + i;
    const uint64_t wv = k < a.nnz ? a.sorted[k] : ~0ull;
    w[i] = wv;
    const uint64_t key = wv >> 32;
    if (k < a.nnz && key < M) {
      const uint64_t pk = prev >> 32;
      const bool first = (k == 0);
      if (first || key != pk) rflag |= 1u << i;
      if (first || fdiv((uint32_t)key, a.s.fm3) != fdiv((uint32_t)pk, a.s.fm3)) pflag |= 1u << i;
    }
    prev = wv;
  }
  const uint32_t cnt = (uint32_t)__popc(rflag) | ((uint32_t)__popc(pflag) << 16);
  uint32_t tot;
  const uint32_t excl = block_exclusive_scan_256(cnt, &tot, scan8);
  if (tid < 32) {
    const unsigned long long agg = ((unsigned long long)(tot & 0xffffu) << 31) | (tot >> 16);
    const unsigned long long e = warp_lookback<unsigned long long>(a.w.seg_status, tile, agg, a.w.ctl);
    if (tid == 0) prefix_sh = e;
  }
  __syncthreads();
  int32_t rr = (int32_t)((prefix_sh >> 31) & ((1ull << 31) - 1)) + (int32_t)(excl & 0xffffu);
  int32_t pp = (int32_t)(prefix_sh & ((1ull << 31) - 1)) + (int32_t)(excl >> 16);
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t k = k0 + i;
    if (k >= a.nnz) break;
    const uint64_t key = w[i] >> 32;
    const int32_t l = (int32_t)(w[i] & 0xffffffffu);
    a.w.perm[k] = l;
    if ((uint64_t)(uint32_t)l >= (uint64_t)a.nnz) continue;   // only after a timed-out look-back
    if (key >= M) {
      a.w.uid[l] = -1;
      if (k == 0) {   // no valid lookup at all
        a.w.ctl->n_valid = 0;
        a.w.ctl->U_r = 0;
        a.w.ctl->U_12 = 0;
        a.w.row_start[0] = 0;
        a.w.pair_row_start[0] = 0;
      }
      continue;
    }
    const uint32_t q = fdiv((uint32_t)key, a.s.fm3);
    if (pflag & (1u << i)) {
      const uint32_t q2 = fdiv(q, a.s.fm1);
      a.w.pair_row_start[pp] = rr;
      a.w.pair_i1[pp] = (int32_t)(q - q2 * (uint32_t)a.s.m1);
      a.w.pair_i2[pp] = (int32_t)q2;
      ++pp;
    }
    if (rflag & (1u << i)) {
      a.w.row_start[rr] = (int32_t)k;
      a.w.row_i3[rr] = (int32_t)((uint32_t)key - q * m3);
      a.w.row_pair[rr] = pp - 1;
      ++rr;
    }
    a.w.uid[l] = rr - 1;
    const bool last = (k + 1 == a.nnz) || ((a.sorted[k + 1] >> 32) >= M);
    if (last) {
      a.w.ctl->n_valid = (int32_t)(k + 1);
      a.w.ctl->U_r = rr;
      a.w.ctl->U_12 = pp;
      a.w.row_start[rr] = (int32_t)(k + 1);
      a.w.pair_row_start[pp] = rr;
    }
  }
}

struct ChunkArgs {
  WS w;
  int pairs_per_chunk;   // small prefixes: at most this many per chunk
  int rows_per_chunk;    // a prefix with more unique rows is split into pieces of this many
};

__device__ __forceinline__ bool chunk_starts_at(const WS& w, int32_t x, int CP, int CR) {
  const int32_t p = w.row_pair[x];
  const int32_t f = w.pair_row_start[p];
  const int32_t nr = w.pair_row_start[p + 1] - f;
  if (x != f) return ((x - f) % CR) == 0;
  if (p == 0) return true;
  const int32_t pf = w.pair_row_start[p - 1];
  return (p % CP) == 0 || w.pair_i2[p] != w.pair_i2[p - 1] || nr > CR || (f - pf) > CR;
}

__global__ void __launch_bounds__(kScanThreads) k_chunks(ChunkArgs a) {
  __shared__ uint32_t scan8[8];
  __shared__ uint32_t tile_sh;
  __shared__ uint32_t prefix_sh;
  const int tid = threadIdx.x;
  if (tid == 0) tile_sh = atomicAdd(&a.w.ctl->chunk_tile_ctr, 1u);
  __syncthreads();
  const uint32_t tile = tile_sh;
  const int32_t U = a.w.ctl->U_r;
  const int64_t base = (int64_t)tile * kScanTile;
  if (base >= U) {
    if (tile == 0 && tid == 0) {   // no unique row: no chunk
      a.w.ctl->n_chunks = 0;
      a.w.chunk_start[0] = 0;
      a.w.chunk_desc[0] = make_int2(0, (int32_t)0x80000000);
    }
    return;
  }
  const int64_t x0 = base + (int64_t)tid * kScanItems;
  uint32_t flags = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t x = x0 + i;
    if (x < U && chunk_starts_at(a.w, (int32_t)x, a.pairs_per_chunk, a.rows_per_chunk))
      flags |= 1u << i;
  }
  uint32_t tot;
  const uint32_t excl = block_exclusive_scan_256((uint32_t)__popc(flags), &tot, scan8);
  if (tid < 32) {
    const uint32_t e = warp_lookback<uint32_t>(a.w.chunk_status, tile, tot, a.w.ctl);
    if (tid == 0) prefix_sh = e;
  }
  __syncthreads();
  int32_t c = (int32_t)(prefix_sh + excl);
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t x = x0 + i;
    if (x >= U) break;
    if (flags & (1u << i)) {
      const int32_t p = a.w.row_pair[x];
      const bool first = a.w.pair_row_start[p] == (int32_t)x;
      a.w.chunk_start[c] = (int32_t)x;
      a.w.chunk_desc[c] = make_int2((int32_t)x, p | (first ? (int32_t)0x80000000 : 0));
      a.w.chunk_order[c] = c;          // claimed in row order on this path
      ++c;
    }
    if (x == U - 1) {
      a.w.ctl->n_chunks = c;
      a.w.chunk_start[c] = U;
      a.w.chunk_desc[c] = make_int2(U, a.w.ctl->U_12 | (int32_t)0x80000000);
    }
  }
}

int launch_group(const Shape& s, const Layout& L, const WS& w, Idx indices,
                 int64_t nnz, const int64_t* offsets, int64_t num_bags, int pairs_per_chunk,
                 int rows_per_chunk, cudaStream_t st, int lists) {
  // control block + digit histograms start from zero
  if (cudaMemsetAsync(w.ctl, 0, L.zero_end - L.ctl, st) != cudaSuccess) return TT_EMB_ERR_CUDA;
  // the zero row after the unique rows (pooling points out-of-range lookups at it)
  if (cudaMemsetAsync(w.rowbuf + (size_t)L.rowbuf_rows * s.D, 0, sizeof(float) * (size_t)s.D, st) !=
      cudaSuccess)
    return TT_EMB_ERR_CUDA;
  if (nnz == 0) return TT_EMB_OK;   // counts stay zero; row_start etc. are never read
  if (!lists) {
    // a forward-only call on a batch dense in its table: bitmap of the keys, no sort
    const int rc = launch_group_bitmap(s, L, w, indices, nnz, offsets, num_bags, pairs_per_chunk,
                                       rows_per_chunk, st);
    if (rc != TT_EMB_ERR_UNSUPPORTED) return rc;
  }
  {
    const int rc = launch_group_coop(s, L, w, w.coop, indices, nnz, offsets, num_bags,
                                     pairs_per_chunk, rows_per_chunk, st);
    if (rc != TT_EMB_ERR_UNSUPPORTED) return rc;
  }
  const uint32_t sentinel = L.key_bits >= 32 ? 0xffffffffu : ((1u << L.key_bits) - 1u);

  PrepArgs pa;
  pa.indices = indices;
  pa.nnz = nnz;
  pa.offsets = offsets;
  pa.B = num_bags;
  pa.s = s;
  pa.sentinel = sentinel;
  pa.passes = L.passes;
  pa.w = w;
  pa.zero32 = w.sort_status;
  pa.zero32_words = (size_t)kMaxPasses * L.n_sort_tiles * kRadix;
  pa.zero64 = w.seg_status;
  pa.zero64_words = (size_t)L.n_scan_tiles;
  pa.zero32b = w.chunk_status;
  pa.zero32b_words = (size_t)L.n_scan_tiles;
  const int64_t work = nnz > num_bags + 1 ? nnz : num_bags + 1;
  int grid = (int)ceil_div(work, 256);
  const int cap = sm_count() * 2;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  TT_TIMED("k_prepare", st, (k_prepare<<<grid, 256, 0, st>>>(pa)));

  const uint64_t* in = nullptr;
  for (int p = 0; p < L.passes; ++p) {
    ScatterArgs sa;
    sa.indices = indices;
    sa.in = in;
    sa.out = (p & 1) ? w.keysB : w.keysA;
    sa.nnz = nnz;
    sa.s = s;
    sa.sentinel = sentinel;
    sa.pass = p;
    sa.n_tiles = L.n_sort_tiles;
    sa.w = w;
    TT_TIMED("k_scatter", st, (k_scatter<<<L.n_sort_tiles, kSortThreads, 0, st>>>(sa)));
    in = sa.out;
  }
  SegArgs ga;
  ga.sorted = in;
  ga.nnz = nnz;
  ga.s = s;
  ga.w = w;
  TT_TIMED("k_segment", st, (k_segment<<<L.n_scan_tiles, kScanThreads, 0, st>>>(ga)));

  ChunkArgs ca;
  ca.w = w;
  ca.pairs_per_chunk = pairs_per_chunk;
  ca.rows_per_chunk = rows_per_chunk;
  TT_TIMED("k_chunks", st, (k_chunks<<<L.n_scan_tiles, kScanThreads, 0, st>>>(ca)));
  return cudaGetLastError() == cudaSuccess ? TT_EMB_OK : TT_EMB_ERR_CUDA;
}

}  // namespace tt
