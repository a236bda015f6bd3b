// Internal definitions shared by the CUDA translation units of the TT
// embedding-bag library: workspace layout, the control block, launch
// parameter structs and small device helpers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/tt_emb.h"

namespace tt {

// ---------------------------------------------------------------- constants

constexpr int kRadixBits = 8;
constexpr int kRadix = 1 << kRadixBits;
constexpr int kMaxPasses = 4;               // keys of up to 32 bits
constexpr int kSortThreads = 256;
constexpr int kSortItems = 8;               // per thread
constexpr int kSortTile = kSortThreads * kSortItems;
constexpr int kScanThreads = 256;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;
constexpr int kSSlice = 64;                 // sorted positions per warp in the grad gather
constexpr int kMaxSmemFloats = 53248;       // 208 KB of shared memory per CTA

// status word bits
constexpr uint32_t kStIndex = 1u;
constexpr uint32_t kStOffsets = 2u;
constexpr uint32_t kStTimeout = 4u;

// decoupled look-back flags (top two bits of a 32-bit status word)
constexpr uint32_t kFlagAgg = 1u << 30;
constexpr uint32_t kFlagIncl = 2u << 30;
constexpr uint32_t kFlagMask = 3u << 30;
constexpr uint32_t kValMask = (1u << 30) - 1u;
constexpr long long kSpinCap = 1ll << 22;   // polls before a look-back gives up

// The control block at the start of the workspace (256 bytes).
struct Ctl {
  int32_t n_valid;        // lookups with an in-range index
  int32_t U_r;            // unique rows
  int32_t U_12;           // unique (i1, i2) prefixes
  int32_t n_chunks;       // work chunks
  uint32_t status;        // kSt* bits
  uint32_t sort_tile_ctr[kMaxPasses];
  uint32_t seg_tile_ctr;
  uint32_t chunk_tile_ctr;
  uint32_t fwd_chunk_ctr;
  uint32_t bwd_chunk_ctr;
  uint32_t pad[51];
};
static_assert(sizeof(Ctl) == 256, "control block is 256 bytes");

// Shape of one TT table as the kernels see it.
struct Shape {
  int64_t m1, m2, m3, M;
  int n1, n2, n3, R1, R2, D;
};

// Workspace layout (byte offsets from the workspace base; 256-aligned).
struct Layout {
  size_t ctl, hist, sort_status, keysA, keysB, bag_of, uid, perm;
  size_t row_start, row_i3, row_pair, pair_row_start, pair_i1, pair_i2;
  size_t seg_status, chunk_start, chunk_status, rowbuf, total;
  int key_bits, passes, n_sort_tiles, n_scan_tiles;
  int64_t rowbuf_rows;
};

// Device pointers into one workspace.
struct WS {
  Ctl* ctl;
  uint32_t* hist;          // [kMaxPasses][kRadix]
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
  uint32_t* chunk_status;           // [n_scan_tiles]
  float* rowbuf;                    // [rowbuf_rows][D]
};

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

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ void set_status(Ctl* ctl, uint32_t bit) { atomicOr(&ctl->status, bit); }

// Grouping key of a row index: (i2, i1, i3) with i3 least significant, so that
// unique (i1, i2) prefixes come out grouped by the G2 slice they read.
__device__ __forceinline__ uint32_t group_key(int64_t r, const Shape& s) {
  int64_t i3 = r % s.m3;
  int64_t q = r / s.m3;
  int64_t i2 = q % s.m2;
  int64_t i1 = q / s.m2;
  return (uint32_t)((i2 * s.m1 + i1) * s.m3 + i3);
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

// grouping (tt_group.cu)
int launch_group(const Shape& s, const Layout& L, const WS& w, const int64_t* indices,
                 int64_t nnz, const int64_t* offsets, int64_t num_bags, int pairs_per_chunk,
                 int rows_per_chunk, cudaStream_t st);
// forward (tt_fwd.cu)
int launch_forward(const Shape& s, const Layout& L, const WS& w, const float* const cores[3],
                   const int64_t* offsets, int64_t nnz, int64_t num_bags, float* out,
                   cudaStream_t st);
int forward_chunk_params(const Shape& s, int* pairs_per_chunk, int* rows_per_chunk);
// backward (tt_bwd.cu)
int launch_backward(const Shape& s, const Layout& L, const WS& w, const float* grad_out,
                    const float* const cores[3], const int64_t* offsets, int64_t nnz,
                    int64_t num_bags, float* const core_grads[3], cudaStream_t st);
int launch_sgd(float* const cores[3], const float* const grads[3], const Shape& s, float lr,
               cudaStream_t st);

}  // namespace tt
