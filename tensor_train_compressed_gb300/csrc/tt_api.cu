// C ABI of the TT embedding-bag library: argument checks, workspace layout and
// the order of launches.  The declarations and their contracts are in
// include/tt_emb.h.
#include <string.h>

#include "tt_internal.cuh"

namespace tt {

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (cached[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1)
      v = 152;
    cached[dev] = v;
  }
  return cached[dev];
}

int shape_from_args(const int64_t m[3], const int32_t n[3], const int32_t R[4], Shape* s) {
  if (!m || !n || !R || !s) return TT_EMB_ERR_ARG;
  if (R[0] != 1 || R[3] != 1 || R[1] < 1 || R[2] < 1) return TT_EMB_ERR_ARG;
  for (int k = 0; k < 3; ++k) {
    if (m[k] < 1 || m[k] >= (1ll << 31)) return TT_EMB_ERR_ARG;
    if (n[k] < 1) return TT_EMB_ERR_ARG;
  }
  const unsigned __int128 M = (unsigned __int128)m[0] * (unsigned __int128)m[1] * m[2];
  if (M > (unsigned __int128)0xfffffffeull) return TT_EMB_ERR_UNSUPPORTED;
  const int64_t D = (int64_t)n[0] * n[1] * n[2];
  if (D > (1 << 20)) return TT_EMB_ERR_UNSUPPORTED;
  s->m1 = m[0];
  s->m2 = m[1];
  s->fm1 = make_fastdiv((uint32_t)m[0]);
  s->fm2 = make_fastdiv((uint32_t)m[1]);
  s->fm3 = make_fastdiv((uint32_t)m[2]);
  s->m3 = m[2];
  s->M = (int64_t)M;
  s->n1 = n[0];
  s->n2 = n[1];
  s->n3 = n[2];
  s->R1 = R[1];
  s->R2 = R[2];
  s->D = (int)D;
  const int64_t g2n = (int64_t)s->R1 * s->n2 * s->R2;
  const int64_t p2n = (int64_t)s->n1 * s->n2 * s->R2;
  if (g2n + (int64_t)s->n1 * s->R1 + 2 * p2n > kMaxSmemFloats) return TT_EMB_ERR_UNSUPPORTED;
  return TT_EMB_OK;
}

Layout make_layout(const Shape& s, int64_t nnz, int64_t num_bags) {
  (void)num_bags;
  Layout L;
  memset(&L, 0, sizeof(L));
  int kb = 1;
  while (kb < 32 && (((uint64_t)1 << kb) - 1) < (uint64_t)s.M) ++kb;
  L.key_bits = kb;
  L.passes = (kb + kRadixBits - 1) / kRadixBits;
  const int64_t n = nnz > 0 ? nnz : 1;
  L.n_sort_tiles = (int)ceil_div(n, kSortTile);
  L.n_scan_tiles = (int)ceil_div(n, kScanTile);
  L.rowbuf_rows = nnz < s.M ? nnz : s.M;
  if (L.rowbuf_rows < 1) L.rowbuf_rows = 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.ctl = take(sizeof(Ctl));
  L.hist = take(sizeof(uint32_t) * kHistCopies * kMaxPasses * kRadix);
  L.ckpt = take(sizeof(uint32_t) * 2 * kCkptSlots);
  L.zero_end = off;   // every grouping zeroes [ctl, zero_end)
  // bf16 split planes of the cores, at offsets fixed by the shape: a split made
  // by tt_emb_split or tt_emb_sgd_ex outlives the groupings of later batches
  if (split_shape(s)) {
    const size_t n1 = (size_t)s.m1 * s.n1 * s.R1, n2 = (size_t)s.m2 * s.R1 * s.n2 * s.R2;
    const size_t n3 = (size_t)s.m3 * s.R2 * s.n3;
    L.g1h = take(2 * n1);
    L.g1l = take(2 * n1);
    L.g2h = take(2 * n2);
    L.g2l = take(2 * n2);
    L.g3h = take(2 * n3);
    L.g3l = take(2 * n3);
    L.g3th = take(2 * n3);
    L.g3tl = take(2 * n3);
  }
  L.sort_status = take(sizeof(uint32_t) * kMaxPasses * (size_t)L.n_sort_tiles * kRadix);
  L.keysA = take(sizeof(uint64_t) * (size_t)n);
  L.keysB = take(sizeof(uint64_t) * (size_t)n);
  L.bag_of = take(sizeof(int32_t) * (size_t)n);
  L.uid = take(sizeof(int32_t) * (size_t)n);
  L.perm = take(sizeof(int32_t) * (size_t)n);
  L.row_start = take(sizeof(int32_t) * ((size_t)n + 1));
  L.row_i3 = take(sizeof(int32_t) * (size_t)n);
  L.row_pair = take(sizeof(int32_t) * (size_t)n);
  L.pair_row_start = take(sizeof(int32_t) * ((size_t)n + 1));
  L.pair_i1 = take(sizeof(int32_t) * (size_t)n);
  L.pair_i2 = take(sizeof(int32_t) * (size_t)n);
  L.seg_status = take(sizeof(unsigned long long) * (size_t)L.n_scan_tiles);
  L.chunk_start = take(sizeof(int32_t) * ((size_t)n + 1));
  L.chunk_desc = take(sizeof(int2) * ((size_t)n + 1));
  L.chunk_status = take(sizeof(uint32_t) * (size_t)L.n_scan_tiles);
  L.coop = take(coop_scratch_bytes());
  // one extra row, kept at zero, that out-of-range lookups point at while pooling
  L.rowbuf = take(sizeof(float) * ((size_t)L.rowbuf_rows + 1) * (size_t)s.D);
  L.total = off;
  return L;
}

WS make_ws(void* base, const Layout& L) {
  char* b = static_cast<char*>(base);
  WS w;
  w.ctl = reinterpret_cast<Ctl*>(b + L.ctl);
  w.hist = reinterpret_cast<uint32_t*>(b + L.hist);
  w.ckpt = reinterpret_cast<uint32_t*>(b + L.ckpt);
  // the claim order of the chunks is written by the grouping's last phase, when
  // the sort keys are no longer needed
  w.chunk_order = reinterpret_cast<int32_t*>(b + L.keysB);
  w.sort_status = reinterpret_cast<uint32_t*>(b + L.sort_status);
  w.keysA = reinterpret_cast<uint64_t*>(b + L.keysA);
  w.keysB = reinterpret_cast<uint64_t*>(b + L.keysB);
  w.bag_of = reinterpret_cast<int32_t*>(b + L.bag_of);
  w.uid = reinterpret_cast<int32_t*>(b + L.uid);
  w.perm = reinterpret_cast<int32_t*>(b + L.perm);
  w.row_start = reinterpret_cast<int32_t*>(b + L.row_start);
  w.row_i3 = reinterpret_cast<int32_t*>(b + L.row_i3);
  w.row_pair = reinterpret_cast<int32_t*>(b + L.row_pair);
  w.pair_row_start = reinterpret_cast<int32_t*>(b + L.pair_row_start);
  w.pair_i1 = reinterpret_cast<int32_t*>(b + L.pair_i1);
  w.pair_i2 = reinterpret_cast<int32_t*>(b + L.pair_i2);
  w.seg_status = reinterpret_cast<unsigned long long*>(b + L.seg_status);
  w.chunk_start = reinterpret_cast<int32_t*>(b + L.chunk_start);
  w.chunk_desc = reinterpret_cast<int2*>(b + L.chunk_desc);
  w.chunk_status = reinterpret_cast<uint32_t*>(b + L.chunk_status);
  w.coop = b + L.coop;
  w.rowbuf = reinterpret_cast<float*>(b + L.rowbuf);
  w.rowbuf_rows = L.rowbuf_rows;
  const bool split = L.g2l != 0;
  w.g1h = split ? reinterpret_cast<uint16_t*>(b + L.g1h) : nullptr;
  w.g1l = split ? reinterpret_cast<uint16_t*>(b + L.g1l) : nullptr;
  w.g2h = split ? reinterpret_cast<uint16_t*>(b + L.g2h) : nullptr;
  w.g2l = split ? reinterpret_cast<uint16_t*>(b + L.g2l) : nullptr;
  w.g3h = split ? reinterpret_cast<uint16_t*>(b + L.g3h) : nullptr;
  w.g3l = split ? reinterpret_cast<uint16_t*>(b + L.g3l) : nullptr;
  w.g3th = split ? reinterpret_cast<uint16_t*>(b + L.g3th) : nullptr;
  w.g3tl = split ? reinterpret_cast<uint16_t*>(b + L.g3tl) : nullptr;
  return w;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Common checks of the batch arguments.
static int check_batch(const Shape& s, const int64_t* indices, int64_t nnz, const int64_t* offsets,
                       int64_t num_bags, const void* workspace, size_t ws_bytes, Layout* L,
                       size_t idx_align = 8) {
  (void)s;
  if (nnz < 0 || nnz >= (1ll << 30) || num_bags < 0 || num_bags >= (1ll << 31)) return TT_EMB_ERR_ARG;
  if (nnz > 0 && num_bags == 0) return TT_EMB_ERR_ARG;   // offsets[0] = 0 != offsets[B] = nnz
  // indices: aligned to the element size the call reads (1: not read)
  if (nnz > 0 && (!indices || !aligned(indices, idx_align))) return TT_EMB_ERR_ARG;
  if (!offsets || !workspace) return TT_EMB_ERR_ARG;
  if (!aligned(workspace, 256)) return TT_EMB_ERR_ARG;
  *L = make_layout(s, nnz, num_bags);
  if (ws_bytes < L->total) return TT_EMB_ERR_WORKSPACE;
  return TT_EMB_OK;
}

// Pooling rule and per-sample weights (float32 [nnz], 4-byte aligned; only
// with the sum).
static int check_pooling(const float* psw, int pooling, Pooling* p) {
  if (pooling != TT_EMB_POOL_SUM && pooling != TT_EMB_POOL_MEAN) return TT_EMB_ERR_ARG;
  if (psw && (pooling != TT_EMB_POOL_SUM || !aligned(psw, 4))) return TT_EMB_ERR_ARG;
  p->mode = psw ? kPoolWeighted : (pooling == TT_EMB_POOL_MEAN ? kPoolMean : kPoolSum);
  p->psw = psw;
  return TT_EMB_OK;
}

static int check_cores(const float* const cores[3]) {
  if (!cores) return TT_EMB_ERR_ARG;
  for (int k = 0; k < 3; ++k)
    if (!cores[k] || !aligned(cores[k], 16)) return TT_EMB_ERR_ARG;
  return TT_EMB_OK;
}


// A chain of 4 <= d <= 8 cores, its three-core view (the leading d - 2 cores
// merged: m' = m_0 .. m_{d-3}, n' likewise, rank R_{d-2}) and the byte offsets
// of its workspace parts: the three-core workspace first (its control block,
// and so the status word, at the workspace base), then the merged cores
// C_1 .. C_{d-3} and their gradients.
struct ChainPlan {
  ChainShape c;
  int64_t m3[3];
  int32_t n3[3], R3[4];
  size_t merged[kMaxCores], dmerged[kMaxCores], count[kMaxCores], ws3, total;
};

static int chain_plan(int d, const int64_t* m, const int32_t* n, const int32_t* R, int64_t nnz,
                      int64_t num_bags, ChainPlan* p) {
  if (d < 4 || d > kMaxCores || !m || !n || !R) return TT_EMB_ERR_ARG;
  if (R[0] != 1 || R[d] != 1) return TT_EMB_ERR_ARG;
  ChainShape& c = p->c;
  c.d = d;
  c.R[0] = 1;
  for (int k = 0; k < d; ++k) {
    if (m[k] < 1 || m[k] >= (1ll << 31) || n[k] < 1 || R[k + 1] < 1) return TT_EMB_ERR_ARG;
    c.m[k] = m[k];
    c.n[k] = n[k];
    c.R[k + 1] = R[k + 1];
  }
  // merged cores: C_k holds (m_0 .. m_k)(n_0 .. n_k) R_{k+1} floats, at most 2^28
  unsigned __int128 mm = (unsigned __int128)m[0];
  int64_t nn = n[0];
  for (int k = 1; k <= d - 3; ++k) {
    mm *= (unsigned __int128)m[k];
    nn *= n[k];
    if (mm >= ((unsigned __int128)1 << 31) || nn > (1 << 20)) return TT_EMB_ERR_UNSUPPORTED;
    const unsigned __int128 cnt = mm * (unsigned __int128)nn * (unsigned __int128)R[k + 1];
    if (cnt > ((unsigned __int128)1 << 28)) return TT_EMB_ERR_UNSUPPORTED;
    p->count[k] = (size_t)cnt;
  }
  p->m3[0] = (int64_t)mm;
  p->m3[1] = m[d - 2];
  p->m3[2] = m[d - 1];
  p->n3[0] = (int32_t)nn;
  p->n3[1] = n[d - 2];
  p->n3[2] = n[d - 1];
  p->R3[0] = 1;
  p->R3[1] = R[d - 2];
  p->R3[2] = R[d - 1];
  p->R3[3] = 1;
  size_t b3 = 0;
  const int rc = tt_emb_workspace_bytes(p->m3, p->n3, p->R3, nnz, num_bags, &b3);
  if (rc) return rc;
  p->ws3 = b3;
  size_t off = align_up(b3, 256);
  for (int k = 1; k <= d - 3; ++k) {
    p->merged[k] = off;
    off = align_up(off + 4 * p->count[k], 256);
  }
  for (int k = 1; k <= d - 3; ++k) {
    p->dmerged[k] = off;
    off = align_up(off + 4 * p->count[k], 256);
  }
  p->total = off;
  return TT_EMB_OK;
}

static int check_cores_d(int d, const float* const* cores) {
  if (!cores) return TT_EMB_ERR_ARG;
  for (int k = 0; k < d; ++k)
    if (!cores[k] || !aligned(cores[k], 16)) return TT_EMB_ERR_ARG;
  return TT_EMB_OK;
}

}  // namespace tt

using namespace tt;

extern "C" {

int tt_emb_version(void) { return 300; }

int tt_emb_workspace_bytes(const int64_t m[3], const int32_t n[3], const int32_t R[4], int64_t nnz,
                           int64_t num_bags, size_t* bytes) {
  Shape s;
  int rc = shape_from_args(m, n, R, &s);
  if (rc) return rc;
  if (!bytes || nnz < 0 || nnz >= (1ll << 30) || num_bags < 0) return TT_EMB_ERR_ARG;
  *bytes = make_layout(s, nnz, num_bags).total;
  return TT_EMB_OK;
}

int tt_emb_group(const int64_t m[3], const int32_t n[3], const int32_t R[4], const int64_t* indices,
                 int64_t nnz, const int64_t* offsets, int64_t num_bags, void* workspace,
                 size_t ws_bytes, void* stream) {
  Shape s;
  int rc = shape_from_args(m, n, R, &s);
  if (rc) return rc;
  Layout L;
  rc = check_batch(s, indices, nnz, offsets, num_bags, workspace, ws_bytes, &L);
  if (rc) return rc;
  int CP, CR;
  rc = forward_chunk_params(s, &CP, &CR);
  if (rc) return rc;
  const WS w = make_ws(workspace, L);
  rc = launch_group(s, L, w, Idx{indices, 0}, nnz, offsets, num_bags, CP, CR, (cudaStream_t)stream);
  if (rc) return rc;
  return launch_bag_ids(w, offsets, num_bags, nnz, (cudaStream_t)stream);
}

int tt_emb_forward_ex(const float* const cores[3], const int64_t m[3], const int32_t n[3],
                      const int32_t R[4], const int64_t* indices, int64_t nnz,
                      const int64_t* offsets, int64_t num_bags, const float* per_sample_weights,
                      int pooling, int flags, float* out, void* workspace, size_t ws_bytes,
                      void* stream) {
  Shape s;
  int rc = shape_from_args(m, n, R, &s);
  if (rc) return rc;
  rc = check_cores(cores);
  if (rc) return rc;
  if (flags & ~(TT_EMB_CORES_SPLIT | TT_EMB_FORWARD_ONLY | TT_EMB_INDICES_I32)) return TT_EMB_ERR_ARG;
  Pooling pool;
  rc = check_pooling(per_sample_weights, pooling, &pool);
  if (rc) return rc;
  const Idx idx{indices, (flags & TT_EMB_INDICES_I32) ? 1 : 0};
  Layout L;
  rc = check_batch(s, indices, nnz, offsets, num_bags, workspace, ws_bytes, &L, idx.i32 ? 4 : 8);
  if (rc) return rc;
  if (num_bags > 0 && (!out || !aligned(out, 16))) return TT_EMB_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const WS w = make_ws(workspace, L);
  if ((flags & TT_EMB_FORWARD_ONLY) && direct_eligible(s, nnz)) {
    // a small batch: each lookup's row formed on its own, no grouping
    if (!(flags & TT_EMB_CORES_SPLIT)) {
      // the split a forward leaves for later TT_EMB_CORES_SPLIT calls
      rc = launch_split(s, w, cores, 0, st);
      if (rc) return rc;
    }
    return launch_forward_direct(s, w, cores, idx, nnz, offsets, num_bags, pool, out, st);
  }
  int CP, CR;
  rc = forward_chunk_params(s, &CP, &CR);
  if (rc) return rc;
  rc = launch_group(s, L, w, idx, nnz, offsets, num_bags, CP, CR, st,
                    (flags & TT_EMB_FORWARD_ONLY) ? 0 : 1);
  if (rc) return rc;
  if (nnz == 0) {
    if (num_bags > 0 &&
        cudaMemsetAsync(out, 0, sizeof(float) * (size_t)num_bags * s.D, st) != cudaSuccess)
      return TT_EMB_ERR_CUDA;
    return TT_EMB_OK;
  }
  return launch_forward(s, L, w, cores, offsets, nnz, num_bags, pool,
                        (flags & TT_EMB_CORES_SPLIT) ? 1 : 0, out, st);
}

int tt_emb_forward(const float* const cores[3], const int64_t m[3], const int32_t n[3],
                   const int32_t R[4], const int64_t* indices, int64_t nnz,
                   const int64_t* offsets, int64_t num_bags, float* out, void* workspace,
                   size_t ws_bytes, void* stream) {
  return tt_emb_forward_ex(cores, m, n, R, indices, nnz, offsets, num_bags, nullptr,
                           TT_EMB_POOL_SUM, 0, out, workspace, ws_bytes, stream);
}

int tt_emb_forward_tables(int num_tables, const tt_emb_table* tables, void* stream) {
  return tt_emb_forward_tables_ex(num_tables, tables, 0, stream);
}

int tt_emb_forward_tables_ex(int num_tables, const tt_emb_table* tables, int flags, void* stream) {
  if (num_tables < 1 || num_tables > kMaxTables || !tables) return TT_EMB_ERR_ARG;
  if (flags & ~(TT_EMB_CORES_SPLIT | TT_EMB_INDICES_I32)) return TT_EMB_ERR_ARG;
  const int idx32 = (flags & TT_EMB_INDICES_I32) ? 1 : 0;
  Shape s[kMaxTables];
  Layout L[kMaxTables];
  WS w[kMaxTables];
  const float* const* cores[kMaxTables];
  const int64_t* offsets[kMaxTables];
  int64_t nnz[kMaxTables], bags[kMaxTables];
  float* out[kMaxTables];
  int64_t total_bags = 0;
  for (int t = 0; t < num_tables; ++t) {
    const tt_emb_table& tb = tables[t];
    int rc = shape_from_args(tb.m, tb.n, tb.R, &s[t]);
    if (rc) return rc;
    for (int k = 0; k < 3; ++k)
      if (tb.n[k] != tables[0].n[k]) return TT_EMB_ERR_ARG;
    for (int k = 0; k < 4; ++k)
      if (tb.R[k] != tables[0].R[k]) return TT_EMB_ERR_ARG;
    rc = check_cores(tb.cores);
    if (rc) return rc;
    rc = check_batch(s[t], tb.indices, tb.nnz, tb.offsets, tb.num_bags, tb.workspace, tb.ws_bytes,
                     &L[t], idx32 ? 4 : 8);
    if (rc) return rc;
    if (tb.num_bags > 0 && (!tb.out || !aligned(tb.out, 16))) return TT_EMB_ERR_ARG;
    // every table groups into its own workspace
    for (int u = 0; u < t; ++u) {
      const char* a0 = static_cast<const char*>(tb.workspace);
      const char* b0 = static_cast<const char*>(tables[u].workspace);
      if (a0 < b0 + tables[u].ws_bytes && b0 < a0 + tb.ws_bytes) return TT_EMB_ERR_ARG;
    }
    w[t] = make_ws(tb.workspace, L[t]);
    total_bags += tb.num_bags;
    if (total_bags >= (1ll << 31)) return TT_EMB_ERR_ARG;   // bags are numbered in 32 bits
    cores[t] = tb.cores;
    offsets[t] = tb.offsets;
    nnz[t] = tb.nnz;
    bags[t] = tb.num_bags;
    out[t] = tb.out;
  }
  cudaStream_t st = (cudaStream_t)stream;
  for (int t = 0; t < num_tables; ++t) {
    int CP, CR;
    int rc = forward_chunk_params(s[t], &CP, &CR);
    if (rc) return rc;
    // forward-only groupings: no backward reuses them
    rc = launch_group(s[t], L[t], w[t], Idx{tables[t].indices, idx32}, nnz[t], offsets[t], bags[t],
                      CP, CR, st, 0);
    if (rc) return rc;
    if (nnz[t] == 0 && bags[t] > 0 &&
        cudaMemsetAsync(out[t], 0, sizeof(float) * (size_t)bags[t] * s[t].D, st) != cudaSuccess)
      return TT_EMB_ERR_CUDA;
  }
  return launch_forward_tables(num_tables, s, L, w, cores, offsets, nnz, bags, out,
                               (flags & TT_EMB_CORES_SPLIT) ? 1 : 0, st);
}

int tt_emb_backward_ex(const float* grad_out, const float* const cores[3], const int64_t m[3],
                       const int32_t n[3], const int32_t R[4], const int64_t* indices,
                       int64_t nnz, const int64_t* offsets, int64_t num_bags,
                       const float* per_sample_weights, int pooling, float* const core_grads[3],
                       float* grad_weights, void* workspace, size_t ws_bytes, int reuse_grouping,
                       void* stream) {
  Shape s;
  int rc = shape_from_args(m, n, R, &s);
  if (rc) return rc;
  rc = check_cores(cores);
  if (rc) return rc;
  rc = check_cores(core_grads);
  if (rc) return rc;
  Pooling pool;
  rc = check_pooling(per_sample_weights, pooling, &pool);
  if (rc) return rc;
  if (grad_weights && (!per_sample_weights || !aligned(grad_weights, 4))) return TT_EMB_ERR_ARG;
  Layout L;
  rc = check_batch(s, indices, nnz, offsets, num_bags, workspace, ws_bytes, &L,
                   reuse_grouping ? 1 : 8);   // a reused grouping reads no index
  if (rc) return rc;
  if (num_bags > 0 && (!grad_out || !aligned(grad_out, 16))) return TT_EMB_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const WS w = make_ws(workspace, L);
  if (!reuse_grouping) {
    int CP, CR;
    rc = forward_chunk_params(s, &CP, &CR);
    if (rc) return rc;
    rc = launch_group(s, L, w, Idx{indices, 0}, nnz, offsets, num_bags, CP, CR, st);
    if (rc) return rc;
    rc = launch_bag_ids(w, offsets, num_bags, nnz, st);
    if (rc) return rc;
  }
  return launch_backward(s, L, w, grad_out, reuse_grouping ? 1 : 0, cores, offsets, nnz, num_bags,
                         pool, core_grads, grad_weights, st);
}

int tt_emb_backward(const float* grad_out, const float* const cores[3], const int64_t m[3],
                    const int32_t n[3], const int32_t R[4], const int64_t* indices, int64_t nnz,
                    const int64_t* offsets, int64_t num_bags, float* const core_grads[3],
                    void* workspace, size_t ws_bytes, int reuse_grouping, void* stream) {
  return tt_emb_backward_ex(grad_out, cores, m, n, R, indices, nnz, offsets, num_bags, nullptr,
                            TT_EMB_POOL_SUM, core_grads, nullptr, workspace, ws_bytes,
                            reuse_grouping, stream);
}

int tt_emb_sgd(float* const cores[3], float* const core_grads[3], const int64_t m[3],
               const int32_t n[3], const int32_t R[4], float lr, int zero_grads, void* stream) {
  Shape s;
  int rc = shape_from_args(m, n, R, &s);
  if (rc) return rc;
  rc = check_cores(cores);
  if (rc) return rc;
  rc = check_cores(core_grads);
  if (rc) return rc;
  return launch_sgd(cores, core_grads, s, lr, zero_grads, nullptr, (cudaStream_t)stream);
}

// The workspace part that holds the split planes (its offsets depend on the
// shape alone): a workspace sized for any batch of this shape holds it.
static int check_split_ws(const Shape& s, const void* workspace, size_t ws_bytes, Layout* L) {
  if (!workspace || !aligned(workspace, 256)) return TT_EMB_ERR_ARG;
  *L = make_layout(s, 0, 0);
  if (ws_bytes < L->sort_status) return TT_EMB_ERR_WORKSPACE;
  return TT_EMB_OK;
}

int tt_emb_split(const float* const cores[3], const int64_t m[3], const int32_t n[3],
                 const int32_t R[4], void* workspace, size_t ws_bytes, void* stream) {
  Shape s;
  int rc = shape_from_args(m, n, R, &s);
  if (rc) return rc;
  rc = check_cores(cores);
  if (rc) return rc;
  Layout L;
  rc = check_split_ws(s, workspace, ws_bytes, &L);
  if (rc) return rc;
  return launch_split(s, make_ws(workspace, L), cores, 0, (cudaStream_t)stream);
}

int tt_emb_sgd_ex(float* const cores[3], float* const core_grads[3], const int64_t m[3],
                  const int32_t n[3], const int32_t R[4], float lr, int zero_grads,
                  void* workspace, size_t ws_bytes, void* stream) {
  Shape s;
  int rc = shape_from_args(m, n, R, &s);
  if (rc) return rc;
  rc = check_cores(cores);
  if (rc) return rc;
  rc = check_cores(core_grads);
  if (rc) return rc;
  Layout L;
  rc = check_split_ws(s, workspace, ws_bytes, &L);
  if (rc) return rc;
  const WS w = make_ws(workspace, L);
  return launch_sgd(cores, core_grads, s, lr, zero_grads, &w, (cudaStream_t)stream);
}

int tt_emb_workspace_bytes_d(int d, const int64_t* m, const int32_t* n, const int32_t* R,
                             int64_t nnz, int64_t num_bags, size_t* bytes) {
  if (d == 3) return tt_emb_workspace_bytes(m, n, R, nnz, num_bags, bytes);
  if (!bytes) return TT_EMB_ERR_ARG;
  ChainPlan p;
  const int rc = chain_plan(d, m, n, R, nnz, num_bags, &p);
  if (rc) return rc;
  *bytes = p.total;
  return TT_EMB_OK;
}

int tt_emb_forward_d(int d, const float* const* cores, const int64_t* m, const int32_t* n,
                     const int32_t* R, const int64_t* indices, int64_t nnz, const int64_t* offsets,
                     int64_t num_bags, float* out, void* workspace, size_t ws_bytes, void* stream) {
  if (d == 3)
    return tt_emb_forward(cores, m, n, R, indices, nnz, offsets, num_bags, out, workspace, ws_bytes,
                          stream);
  if (nnz < 0 || nnz >= (1ll << 30) || num_bags < 0) return TT_EMB_ERR_ARG;
  ChainPlan p;
  int rc = chain_plan(d, m, n, R, nnz, num_bags, &p);
  if (rc) return rc;
  rc = check_cores_d(d, cores);
  if (rc) return rc;
  if (!workspace || !aligned(workspace, 256)) return TT_EMB_ERR_ARG;
  if (ws_bytes < p.total) return TT_EMB_ERR_WORKSPACE;
  char* b = static_cast<char*>(workspace);
  float* merged[kMaxCores] = {nullptr};
  for (int k = 1; k <= d - 3; ++k) merged[k] = reinterpret_cast<float*>(b + p.merged[k]);
  const float* cores3[3] = {merged[d - 3], cores[d - 2], cores[d - 1]};
  // argument checks of the three-core call first (nothing is enqueued on error)
  Shape s3;
  rc = shape_from_args(p.m3, p.n3, p.R3, &s3);
  if (rc) return rc;
  Layout L;
  rc = check_batch(s3, indices, nnz, offsets, num_bags, b, p.ws3, &L);
  if (rc) return rc;
  rc = launch_merge_chain(p.c, cores, merged, (cudaStream_t)stream);
  if (rc) return rc;
  return tt_emb_forward(cores3, p.m3, p.n3, p.R3, indices, nnz, offsets, num_bags, out, b, p.ws3,
                        stream);
}

int tt_emb_backward_d(int d, const float* grad_out, const float* const* cores, const int64_t* m,
                      const int32_t* n, const int32_t* R, const int64_t* indices, int64_t nnz,
                      const int64_t* offsets, int64_t num_bags, float* const* core_grads,
                      void* workspace, size_t ws_bytes, int reuse_grouping, void* stream) {
  if (d == 3)
    return tt_emb_backward(grad_out, cores, m, n, R, indices, nnz, offsets, num_bags, core_grads,
                           workspace, ws_bytes, reuse_grouping, stream);
  if (nnz < 0 || nnz >= (1ll << 30) || num_bags < 0) return TT_EMB_ERR_ARG;
  ChainPlan p;
  int rc = chain_plan(d, m, n, R, nnz, num_bags, &p);
  if (rc) return rc;
  rc = check_cores_d(d, cores);
  if (rc) return rc;
  rc = check_cores_d(d, core_grads);
  if (rc) return rc;
  if (!workspace || !aligned(workspace, 256)) return TT_EMB_ERR_ARG;
  if (ws_bytes < p.total) return TT_EMB_ERR_WORKSPACE;
  char* b = static_cast<char*>(workspace);
  float* merged[kMaxCores] = {nullptr};
  float* dmerged[kMaxCores] = {nullptr};
  for (int k = 1; k <= d - 3; ++k) {
    merged[k] = reinterpret_cast<float*>(b + p.merged[k]);
    dmerged[k] = reinterpret_cast<float*>(b + p.dmerged[k]);
  }
  Shape s3;
  rc = shape_from_args(p.m3, p.n3, p.R3, &s3);
  if (rc) return rc;
  Layout L;
  rc = check_batch(s3, indices, nnz, offsets, num_bags, b, p.ws3, &L);
  if (rc) return rc;
  if (num_bags > 0 && (!grad_out || !aligned(grad_out, 16))) return TT_EMB_ERR_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  // the merged cores of the forward stand when the grouping is reused (the
  // cores are unchanged under that contract); otherwise merge again
  if (!reuse_grouping) {
    rc = launch_merge_chain(p.c, cores, merged, st);
    if (rc) return rc;
  }
  for (int k = 1; k <= d - 3; ++k)
    if (cudaMemsetAsync(dmerged[k], 0, 4 * p.count[k], st) != cudaSuccess) return TT_EMB_ERR_CUDA;
  const float* cores3[3] = {merged[d - 3], cores[d - 2], cores[d - 1]};
  float* grads3[3] = {dmerged[d - 3], core_grads[d - 2], core_grads[d - 1]};
  rc = tt_emb_backward(grad_out, cores3, p.m3, p.n3, p.R3, indices, nnz, offsets, num_bags, grads3,
                       b, p.ws3, reuse_grouping, stream);
  if (rc) return rc;
  return launch_unmerge_chain(p.c, cores, merged, dmerged, core_grads, st);
}

int tt_emb_sgd_d(int d, float* const* cores, float* const* core_grads, const int64_t* m,
                 const int32_t* n, const int32_t* R, float lr, int zero_grads, void* stream) {
  if (d < 2 || d > kMaxCores || !m || !n || !R || !cores || !core_grads) return TT_EMB_ERR_ARG;
  if (R[0] != 1 || R[d] != 1) return TT_EMB_ERR_ARG;
  int rc = check_cores_d(d, cores);
  if (rc) return rc;
  rc = check_cores_d(d, core_grads);
  if (rc) return rc;
  for (int k = 0; k < d; ++k)
    if (m[k] < 1 || n[k] < 1 || R[k + 1] < 1) return TT_EMB_ERR_ARG;
  for (int k0 = 0; k0 < d; k0 += 3) {
    float* G[3];
    float* dG[3];
    int64_t cnt[3];
    for (int u = 0; u < 3; ++u) {
      const int k = k0 + u < d ? k0 + u : k0;
      G[u] = cores[k];
      dG[u] = core_grads[k];
      cnt[u] = k0 + u < d ? m[k] * (int64_t)R[k] * n[k] * R[k + 1] : 0;
    }
    rc = launch_sgd_counts(G, dG, cnt, lr, zero_grads, (cudaStream_t)stream);
    if (rc) return rc;
  }
  return TT_EMB_OK;
}

int tt_emb_get_error(const void* workspace, void* stream, int* device_status) {
  if (!workspace || !device_status) return TT_EMB_ERR_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return TT_EMB_ERR_CUDA;
  uint32_t st = 0;
  const Ctl* c = static_cast<const Ctl*>(workspace);
  if (cudaMemcpy(&st, &c->status, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
    return TT_EMB_ERR_CUDA;
  *device_status = (int)st;
  if (st & kStTimeout) return TT_EMB_ERR_TIMEOUT;
  if (st & kStNoLists) return TT_EMB_ERR_REUSE;
  if (st & kStOffsets) return TT_EMB_ERR_OFFSETS;
  if (st & kStIndex) return TT_EMB_ERR_INDEX;
  return TT_EMB_OK;
}

int tt_emb_grouping_view(const int64_t m[3], const int32_t n[3], const int32_t R[4], int64_t nnz,
                         int64_t num_bags, const void* workspace, tt_emb_grouping* view) {
  Shape s;
  int rc = shape_from_args(m, n, R, &s);
  if (rc) return rc;
  if (!workspace || !view || nnz < 0 || nnz >= (1ll << 30)) return TT_EMB_ERR_ARG;
  const Layout L = make_layout(s, nnz, num_bags);
  const WS w = make_ws(const_cast<void*>(workspace), L);
  view->counts = reinterpret_cast<const int32_t*>(w.ctl);
  view->perm = w.perm;
  view->row_start = w.row_start;
  view->row_i3 = w.row_i3;
  view->row_pair = w.row_pair;
  view->pair_row_start = w.pair_row_start;
  view->pair_i1 = w.pair_i1;
  view->pair_i2 = w.pair_i2;
  view->uid = w.uid;
  view->bag_of = w.bag_of;
  view->chunk_start = w.chunk_start;
  view->rowbuf = w.rowbuf;
  view->chunk_order = w.chunk_order;
  return TT_EMB_OK;
}

}  // extern "C"
