// Internal definitions shared by the CUDA translation units of the TT
// embedding-bag library: workspace layout, the control block, launch
// parameter structs and small device helpers.
#pragma once

#include <climits>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/tt_emb.h"

namespace tt {

// ---------------------------------------------------------------- constants

constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;
constexpr int kMaxPasses = 4;               // keys of up to 32 bits
constexpr int kHistCopies = 8;              // digit histograms are striped over 8 copies
constexpr int kSortThreads = 256;
constexpr int kSortItems = 8;               // per thread
constexpr int kSortTile = kSortThreads * kSortItems;
constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;
constexpr int kSSlice = 64;                 // sorted positions per warp in the grad gather
constexpr int kMaxSmemFloats = 53248;       // 208 KB of shared memory per CTA
constexpr int kMaxTables = 8;               // tables of one tt_emb_forward_tables call
constexpr int kMaxCores = 8;                // cores of one chain (tt_emb_*_d)
constexpr int kCkptSlots = 1024;            // L2 checkpoint slots of prefix partials
// Stage slot value of the forward chunk kernels: the stage buffer already holds
// the chunk's G2 slice (tested before the i2 and checkpoint-slot readings).
constexpr int kKeepG2 = INT_MIN;

// status word bits
constexpr uint32_t kStIndex = 1u;
constexpr uint32_t kStOffsets = 2u;
constexpr uint32_t kStTimeout = 4u;
constexpr uint32_t kStNoLists = 8u;         // a backward reused a forward-only grouping

// decoupled look-back flags (top two bits of a 32-bit status word)
constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagIncl = 2u << 30;
constexpr uint32_t kFlagMask = 3u << 30;
constexpr uint32_t kValMask = (1u << 30) - 1u;
constexpr long long kSpinCap = 1ll << 22;   // polls before a look-back gives up

// Grouping methods (Ctl::method).
constexpr int32_t kGroupBitmap = 1;   // key bitmap, one cooperative launch, no per-row
                                      // lookup lists (perm, row_start): forward-only calls
constexpr int32_t kGroupCoop = 2;     // radix sort, one cooperative launch
constexpr int32_t kGroupMulti = 3;    // radix sort, one launch per phase
constexpr int32_t kGroupDirect = 4;   // no grouping: a small forward-only batch whose rows
                                      // were formed per lookup (k_fwd_direct)

// A forward-only call takes the per-lookup kernel when the batch's arithmetic
// in that form (nnz * direct_macs_per_lookup) is at most this, D <= kDirectMaxD
// and one warp's shared memory (two lookups' core slices and the partial) fits
// kDirectMaxSmem.
constexpr int64_t kDirectMaxMacs = 1ll << 27;
constexpr int kDirectMaxD = 256;
constexpr int kDirectMaxSmem = 200 * 1024;

// The control block at the start of the workspace (256 bytes).
struct Ctl {
  int32_t n_valid;        // lookups with an in-range index
  int32_t U_r;            // unique rows
  int32_t U_12;           // unique (i1, i2) prefixes
  int32_t n_chunks;       // work chunks
  uint32_t status;        // kSt* bits
  int32_t method;         // grouping that ran: kGroupBitmap, kGroupCoop or kGroupMulti
  int32_t ckpt_reused;    // chunks of the last forward that reused a checkpointed P2
  uint32_t sort_tile_ctr[kMaxPasses];
  uint32_t seg_tile_ctr;
  uint32_t chunk_tile_ctr;
  uint32_t fwd_chunk_ctr;
  uint32_t bwd_chunk_ctr;
  uint32_t split_valid;   // the bf16 split planes hold the cores split_src (reset by every grouping)
  unsigned long long split_src[3];   // G1, G2, G3 addresses the planes were split from
  uint32_t pad[42];
};
static_assert(sizeof(Ctl) == 256, "control block is 256 bytes");

// Shape of one TT table as the kernels see it.
// Unsigned 32-bit division by a divisor fixed per shape (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994,
// section 4, for all 32-bit dividends): with l = ceil(log2 d) and
// mul = floor(2^32 (2^l - d) / d) + 1, n / d = (t + ((n - t) >> s1)) >> s2 where
// t = umulhi(mul, n), s1 = min(l, 1), s2 = max(l - 1, 0).
struct FastDiv {
  uint32_t mul, s1, s2, pad;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while (l < 32 && ((uint64_t)1 << l) < (uint64_t)d) ++l;
  FastDiv f;
  f.mul = (uint32_t)(((((uint64_t)1) << 32) * ((((uint64_t)1) << l) - d)) / d + 1);
  f.s1 = l < 1 ? l : 1;
  f.s2 = l > 0 ? l - 1 : 0;
  f.pad = 0;
  return f;
}
__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(f.mul, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

struct Shape {
  int64_t m1, m2, m3, M;
  int n1, n2, n3, R1, R2, D;
  FastDiv fm1, fm2, fm3;     // division by m1, m2, m3
};

// Workspace layout (byte offsets from the workspace base; 256-aligned).
struct Layout {
  size_t ctl, hist, ckpt, zero_end, sort_status, keysA, keysB, bag_of, uid, perm;
  size_t row_start, row_i3, row_pair, pair_row_start, pair_i1, pair_i2;
  size_t seg_status, chunk_start, chunk_desc, chunk_status, coop, rowbuf, total;
  size_t g1h, g1l, g2h, g2l;   // bf16 split planes of G1 and G2 (tensor-core shape only; their
                               // offsets depend on the shape alone, not on the batch)
  size_t g3h, g3l, g3th, g3tl; // bf16 split planes of G3 [m3][R2][n3] and of its transpose [m3][n3][R2]
  int key_bits, passes, n_sort_tiles, n_scan_tiles;
  int64_t rowbuf_rows;
};

// Device pointers into one workspace.
struct WS {
  Ctl* ctl;
  uint32_t* hist;          // [kHistCopies][kMaxPasses][kRadix]
  uint32_t* ckpt;          // [2][kCkptSlots] checkpoint slot owner / ready words (prefix + 1)
  int32_t* chunk_order;    // [chunks] claim order of the work chunks (aliases keysB)
  uint32_t* sort_status;   // [kMaxPasses][n_sort_tiles][kRadix]
  uint64_t* keysA;
  uint64_t* keysB;
  int32_t* bag_of;
  int32_t* uid;
  int32_t* perm;
  int32_t* row_start;
  int32_t* row_i3;
  int32_t* row_pair;
  int32_t* pair_row_start;
  int32_t* pair_i1;
  int32_t* pair_i2;
  unsigned long long* seg_status;   // [n_scan_tiles]
  int32_t* chunk_start;
  int2* chunk_desc;                 // [chunks+1] {first row, prefix | starts-a-prefix << 31}
  uint32_t* chunk_status;           // [n_scan_tiles]
  void* coop;                       // scratch of the cooperative grouping
  float* rowbuf;                    // [rowbuf_rows + 1][D]; the last row stays zero
  int64_t rowbuf_rows;
  uint16_t* g1h;                    // bf16 planes hi / lo of G1 [m1][n1][R1] and G2
  uint16_t* g1l;                    // [m2][R1][n2 R2] (x = hi + lo + O(2^-18 |x|)), written
  uint16_t* g2h;                    // per call by k_split_cores; null unless the shape
  uint16_t* g2l;                    // runs the tensor-core chunk kernels
  uint16_t* g3h;                    // G3 [m3][R2][n3] planes and the planes of its
  uint16_t* g3l;                    // per-i3 transpose [m3][n3][R2], likewise
  uint16_t* g3th;
  uint16_t* g3tl;
};

// Shapes served by the tensor-core chunk kernels of the forward and the
// backward (n1 = n3 = 4, n2 = 8, R1 = R2 = 32).
inline bool tc_shape(const Shape& s) {
  return s.n1 == 4 && s.n2 == 8 && s.n3 == 4 && s.R1 == 32 && s.R2 == 32;
}
// n1 = n3 = 4, n2 = 8, R1 = R2 = 64: forward rows on the tensor cores
// (k_fwd_mma64), backward on the generic kernel.
inline bool tc64_shape(const Shape& s) {
  return s.n1 == 4 && s.n2 == 8 && s.n3 == 4 && s.R1 == 64 && s.R2 == 64;
}
// Shapes whose workspace holds the bf16 split planes of the cores.
inline bool split_shape(const Shape& s) { return tc_shape(s) || tc64_shape(s); }

// ---------------------------------------------------------------- device helpers

__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ void set_status(Ctl* ctl, uint32_t bit) { atomicOr(&ctl->status, bit); }

__device__ __forceinline__ void f4add(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

// a += c * b, component-wise
__device__ __forceinline__ void f4fma(float4& a, float c, const float4& b) {
  a.x = fmaf(c, b.x, a.x);
  a.y = fmaf(c, b.y, a.y);
  a.z = fmaf(c, b.z, a.z);
  a.w = fmaf(c, b.w, a.w);
}

// Bag ids of the lookups of the 32 consecutive bags wb .. wb+31 (whole warp,
// warp-uniform wb; lane k holds bag wb+k's bounds o0 = offsets[wb+k],
// o1 = offsets[wb+k+1]): bag_of[l] = bag for every lookup l of each bag,
// consecutive lanes writing consecutive lookups.  Bounds are clamped to
// [0, nnz] so that bad offsets stay in bounds.
__device__ __forceinline__ void write_bag_ids(int32_t* bag_of, int64_t wb, int64_t B, int64_t nnz,
                                              int64_t o0, int64_t o1, int lane) {
  const int64_t l0 = o0 < 0 ? 0 : (o0 > nnz ? nnz : o0);
  const int64_t l1 = o1 < l0 ? l0 : (o1 > nnz ? nnz : o1);
  const int nb = B - wb < 32 ? (int)(B - wb) : 32;
  for (int k = 0; k < nb; ++k) {
    const int64_t t0 = __shfl_sync(0xffffffffu, l0, k), t1 = __shfl_sync(0xffffffffu, l1, k);
    for (int64_t l = t0 + lane; l < t1; l += 32) bag_of[l] = (int32_t)(wb + k);
  }
}

// Pooling rule of a bag: the plain sum of its rows, the sum with each row
// scaled by its lookup's per-sample weight, or the sum divided by the bag's
// number of lookups.
enum PoolMode { kPoolSum = 0, kPoolWeighted = 1, kPoolMean = 2 };
struct Pooling {
  int mode;            // PoolMode
  const float* psw;    // [nnz] per-sample weights (kPoolWeighted), else null
};

// Grouping key of an in-range row index (r < M <= 2^32 - 2, so 32-bit
// arithmetic is exact): (i2, i1, i3) with i3 least significant, so that unique
// (i1, i2) prefixes come out grouped by the G2 slice they read.
__device__ __forceinline__ uint32_t group_key(int64_t r, const Shape& s) {
  const uint32_t ru = (uint32_t)r, m1 = (uint32_t)s.m1, m2 = (uint32_t)s.m2, m3 = (uint32_t)s.m3;
  const uint32_t q = fdiv(ru, s.fm3), i3 = ru - q * m3;
  const uint32_t i1 = fdiv(q, s.fm2), i2 = q - i1 * m2;
  return (i2 * m1 + i1) * m3 + i3;
}

// Decoupled look-back over the tiles before `tile`, done by one whole warp:
// the lanes read 32 predecessor words at once, so the walk costs one round
// trip per 32 tiles.  Words hold a 2-bit flag in the top bits (1 = tile
// aggregate, 2 = inclusive prefix) and an additive value below; `agg` is this
// tile's own aggregate, published first.  Returns the exclusive prefix; after
// kSpinCap polls of a window with an unpublished tile it sets the timeout bit
// and returns what it has.  Called by all 32 lanes of one warp.
template <typename W>
__device__ __forceinline__ W warp_lookback(W* st, uint32_t tile, W agg, Ctl* ctl) {
  constexpr int kTop = sizeof(W) * 8 - 2;
  const W kAgg = (W)1 << kTop, kIncl = (W)2 << kTop, kVal = ((W)1 << kTop) - 1;
  const int lane = threadIdx.x & 31;
  if (tile == 0) {
    if (lane == 0) {
      if constexpr (sizeof(W) == 8) st_relaxed_u64((unsigned long long*)st, kIncl | agg);
      else st_relaxed_u32((uint32_t*)st, kIncl | agg);
    }
    return 0;
  }
  if (lane == 0) {
    if constexpr (sizeof(W) == 8) st_relaxed_u64((unsigned long long*)(st + tile), kAgg | agg);
    else st_relaxed_u32((uint32_t*)(st + tile), kAgg | agg);
  }
  W excl = 0;
  int64_t top = (int64_t)tile - 1;
  long long spins = 0;
  while (top >= 0) {
    const int64_t j = top - lane;
    W v = kIncl;                       // before tile 0: an inclusive prefix of 0
    if (j >= 0) {
      if constexpr (sizeof(W) == 8) v = (W)ld_relaxed_u64((const unsigned long long*)(st + j));
      else v = (W)ld_relaxed_u32((const uint32_t*)(st + j));
    }
    const W f = v >> kTop;
    const uint32_t incl = __ballot_sync(0xffffffffu, f == 2);
    const uint32_t none = __ballot_sync(0xffffffffu, f == 0);
    const int first = incl ? __ffs(incl) - 1 : 31;
    const uint32_t needed = first == 31 ? 0xffffffffu : ((2u << first) - 1u);
    if (none & needed) {
      if (++spins > kSpinCap) {
        if (lane == 0) set_status(ctl, kStTimeout);
        break;
      }
      continue;
    }
    W part = lane <= first ? (v & kVal) : (W)0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    excl += part;
    if (incl) break;
    top -= 32;
  }
  if (lane == 0) {
    if constexpr (sizeof(W) == 8)
      st_relaxed_u64((unsigned long long*)(st + tile), kIncl | ((excl + agg) & kVal));
    else
      st_relaxed_u32((uint32_t*)(st + tile), kIncl | ((excl + agg) & kVal));
  }
  return excl;
}

// Block-wide exclusive scan of one uint32 per thread (blockDim = 256).
__device__ __forceinline__ uint32_t block_exclusive_scan_256(uint32_t v, uint32_t* total,
                                                             uint32_t* smem8) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) smem8[warp] = x;
  __syncthreads();
  uint32_t wpre = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    uint32_t c = smem8[w];
    if (w < warp) wpre += c;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return wpre + x - v;
}

// ---------------------------------------------------------------- host side

// opt-in launch timing (tt_prof.cu)
extern bool g_prof_on;
void prof_begin(const char* name, cudaStream_t st);
void prof_end(cudaStream_t st);
#define TT_TIMED(name, st, launch) \
  do {                             \
    ::tt::prof_begin(name, st);    \
    launch;                        \
    ::tt::prof_end(st);            \
  } while (0)

int64_t ceil_div(int64_t a, int64_t b);
Layout make_layout(const Shape& s, int64_t nnz, int64_t num_bags);
WS make_ws(void* base, const Layout& L);
int shape_from_args(const int64_t m[3], const int32_t n[3], const int32_t R[4], Shape* s);
int sm_count();

// The lookups' row indices, int64 or (TT_EMB_INDICES_I32) int32 values; a
// negative int32 reads as the same negative int64, out of range either way.
struct Idx {
  const void* p;
  int i32;
  __device__ __forceinline__ int64_t at(int64_t i) const {
    return i32 ? (int64_t)__ldg(static_cast<const int32_t*>(p) + i) : __ldg(static_cast<const int64_t*>(p) + i);
  }
};

// grouping in one cooperative launch (tt_group_coop.cu)
size_t coop_scratch_bytes();
int launch_group_bitmap(const Shape& s, const Layout& L, const WS& w, Idx indices,
                        int64_t nnz, const int64_t* offsets, int64_t num_bags, int pairs_per_chunk,
                        int rows_per_chunk, cudaStream_t st);
bool bitmap_grouping_applies(const Shape& s, const Layout& L, int64_t nnz);
int launch_group_coop(const Shape& s, const Layout& L, const WS& w, void* scratch,
                      Idx indices, int64_t nnz, const int64_t* offsets,
                      int64_t num_bags, int pairs_per_chunk, int rows_per_chunk, cudaStream_t st);
// grouping (tt_group.cu)
// lists = 0: a forward-only call, whose grouping may leave out the per-row
// lookup lists (perm, row_start) that only a backward reads: the key-bitmap
// grouping then serves a batch dense in its table
int launch_group(const Shape& s, const Layout& L, const WS& w, Idx indices,
                 int64_t nnz, const int64_t* offsets, int64_t num_bags, int pairs_per_chunk,
                 int rows_per_chunk, cudaStream_t st, int lists = 1);
// chains of d > 3 cores (tt_chain.cu): the leading d - 2 cores merged into one
struct ChainShape {
  int d;
  int64_t m[kMaxCores];
  int n[kMaxCores];
  int R[kMaxCores + 1];
};
// merged[k] = C_k = C_{k-1} (x) G_k for k = 1 .. d-3 (C_0 = cores[0])
int launch_merge_chain(const ChainShape& c, const float* const* cores, float* const* merged,
                       cudaStream_t st);
// from dmerged[d-3] (gradient of the merged core) back into dmerged[k] (zeroed
// by the caller) and core_grads[0 .. d-3] (accumulated)
int launch_unmerge_chain(const ChainShape& c, const float* const* cores, const float* const* merged,
                         float* const* dmerged, float* const* core_grads, cudaStream_t st);
int launch_sgd_counts(float* const G[3], float* const dG[3], const int64_t counts[3], float lr,
                      int zero_grads, cudaStream_t st);
// bag of every lookup into the workspace (tt_bwd.cu); the forward's pooling
// writes it too
int launch_bag_ids(const WS& w, const int64_t* offsets, int64_t num_bags, int64_t nnz,
                   cudaStream_t st);
// forward (tt_fwd.cu): the unique rows into the row buffer, then the pooling
// presplit != 0: the workspace's split planes already hold these cores
int launch_rows(const Shape& s, const WS& w, const float* const cores[3], int presplit,
                cudaStream_t st);
int launch_forward(const Shape& s, const Layout& L, const WS& w, const float* const cores[3],
                   const int64_t* offsets, int64_t nnz, int64_t num_bags, const Pooling& pool,
                   int presplit, float* out, cudaStream_t st);
int forward_chunk_params(const Shape& s, int* pairs_per_chunk, int* rows_per_chunk);
// forward of T tables already grouped into their workspaces, sum pooling: one
// launch of the chunk kernel for all tables where the shape runs the tiled
// kernel, table by table otherwise
int launch_forward_tables(int T, const Shape* s, const Layout* L, const WS* w,
                          const float* const* const* cores, const int64_t* const* offsets,
                          const int64_t* nnz, const int64_t* num_bags, float* const* out,
                          int presplit, cudaStream_t st);
// R = 64 tensor-core rows of T tables in one launch (tt_fwd64.cu); the split
// planes of every table must hold its cores
int launch_fwd_mma64(int T, const WS* w, const float* const* const* cores, cudaStream_t st);
// backward (tt_bwd.cu)
int launch_backward(const Shape& s, const Layout& L, const WS& w, const float* grad_out, int reuse,
                    const float* const cores[3], const int64_t* offsets, int64_t nnz,
                    int64_t num_bags, const Pooling& pool, float* const core_grads[3],
                    float* grad_weights, cudaStream_t st);
int launch_split(const Shape& s, const WS& w, const float* const cores[3], int reuse, cudaStream_t st);
int64_t direct_macs_per_lookup(const Shape& s);
bool direct_eligible(const Shape& s, int64_t nnz);
int launch_forward_direct(const Shape& s, const WS& w, const float* const cores[3],
                          Idx indices, int64_t nnz, const int64_t* offsets,
                          int64_t num_bags, const Pooling& pool, float* out, cudaStream_t st);
// Called by one thread of a kernel that runs after k_split_cores in the same
// stream: the split planes now hold the cores at g1, g2, g3.
__device__ __forceinline__ void mark_split(Ctl* ctl, const float* g1, const float* g2, const float* g3) {
  ctl->split_src[0] = (unsigned long long)g1;
  ctl->split_src[1] = (unsigned long long)g2;
  ctl->split_src[2] = (unsigned long long)g3;
  ctl->split_valid = 1;
}
// ws non-null: the updated cores are also split into the planes of that workspace
int launch_sgd(float* const cores[3], float* const grads[3], const Shape& s, float lr,
               int zero_grads, const WS* ws, cudaStream_t st);

}  // namespace tt
