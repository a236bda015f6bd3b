/*
 * tt_emb.h -- C ABI of the GB300 Tensor-Train embedding bag.
 *
 * The operation (FlowTT: Exploiting Computation Flow Reuse in Irregular
 * Tensor-Train Embedding, summary card, problem statement; TT-Rec: Tensor
 * Train Compression for Deep Learning Recommendation Models, abstract):
 * a table of M = m1*m2*m3 rows of width D = n1*n2*n3 is held as three TT
 * cores; looking up row r contracts the chain of cores selected by the
 * mixed-radix digits of r, and the looked-up rows are sum-pooled per bag.
 *
 *   core k:   float32, contiguous [m_k][R_{k-1}][n_k][R_k], R_0 = R_3 = 1
 *   row r:    r = (i1*m2 + i2)*m3 + i3 (i1 most significant)
 *   row(r)[j] = sum_{a,b} G1[i1][0][j1][a] * G2[i2][a][j2][b] * G3[i3][b][j3][0],
 *             j = (j1*n2 + j2)*n3 + j3
 *   bags:     CSR; offsets has num_bags+1 int64 entries, offsets[0] = 0,
 *             offsets[num_bags] = nnz, non-decreasing; bag b holds lookups
 *             offsets[b] .. offsets[b+1]-1 of `indices` (int64 row numbers)
 *   out[b]    = sum over the bag's lookups of row(indices[l]); empty bag -> 0
 *
 * How it is computed (FlowTT, summary card, key innovations; FlowTT
 * abstract): lookups are grouped by their (i1, i2) prefix on the device (a
 * radix sort + run segmentation, or for a forward-only call on a batch dense in
 * its table a presence bitmap over the row keys), the prefix partial P2 = G1[i1].G2[i2] is
 * formed once per unique prefix and kept on chip, each unique row is formed
 * once from it, and rows are pooled per bag.  Persistent CTAs take work
 * chunks from an atomic queue so that Zipf-skewed prefixes do not stall the
 * grid.
 *
 * Conventions for every entry point:
 *  - All array arguments are DEVICE pointers owned by the caller (CUDA
 *    global memory of the current device), except the host arrays of
 *    tt_emb_step_host.  The library allocates no memory and keeps no state
 *    between calls beyond the caller's workspace, with three exceptions,
 *    each described at its declaration: the fixed device array of
 *    tt_emb_forward_static (shared by every call of that entry point), the
 *    per-thread, per-device CUDA events and CUDA graphs of tt_emb_step_host
 *    (created on a thread's first calls on a device, kept until the process
 *    exits), and the opt-in launch records of tt_emb_profile_start.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call only enqueues work on it and returns; none synchronises except
 *    tt_emb_get_error.
 *  - Shape arguments (m, n, R) are HOST arrays: m[3] int64, n[3] int32,
 *    R[4] int32.
 *  - Returns TT_EMB_OK (0) or a negative TT_EMB_ERR_* code.  Argument errors
 *    are detected on the host before anything is enqueued.  Errors found by
 *    the kernels (an index outside [0, M), bad offsets, a capped wait that
 *    gave up) never trap: they set a status word in the workspace, the
 *    offending lookups contribute nothing, and tt_emb_get_error reports them.
 *
 * Limits: M <= 2^32 - 2, nnz < 2^30, num_bags < 2^31, every m_k < 2^31,
 * and R1*n2*R2 + n1*R1 + 2*n1*n2*R2 <= 53248 (the G2 slice and one prefix
 * partial must fit in shared memory); larger shapes return
 * TT_EMB_ERR_UNSUPPORTED.  Cores, out, grad_out and workspace must be
 * 16-byte aligned (workspace: 256-byte).
 */
#ifndef TT_EMB_H
#define TT_EMB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TT_EMB_OK 0
#define TT_EMB_ERR_ARG (-1)          /* null pointer, bad dims, R[0] != 1, misalignment ...  */
#define TT_EMB_ERR_WORKSPACE (-2)    /* ws_bytes smaller than tt_emb_workspace_bytes         */
#define TT_EMB_ERR_CUDA (-3)         /* a launch or runtime call failed                      */
#define TT_EMB_ERR_INDEX (-4)        /* device: an index outside [0, M)                      */
#define TT_EMB_ERR_OFFSETS (-5)      /* device: offsets not CSR (see above)                  */
#define TT_EMB_ERR_TIMEOUT (-6)      /* device: a capped inter-CTA wait gave up              */
#define TT_EMB_ERR_UNSUPPORTED (-7)  /* shape beyond the limits above                        */
#define TT_EMB_ERR_REUSE (-8)        /* device: a backward reused the grouping of a forward
                                        called with TT_EMB_FORWARD_ONLY                      */

/* Bytes of workspace that forward/backward/group need for this shape and
 * batch.  The workspace holds the prefix grouping (sorted lookups, unique
 * rows, unique prefixes, work chunks), the unique-row buffer and a status
 * word.  Host-only; touches no device memory. */
int tt_emb_workspace_bytes(const int64_t m[3], const int32_t n[3], const int32_t R[4],
                           int64_t nnz, int64_t num_bags, size_t* bytes);

/* Prefix grouping only (index decomposition, grouping by the (i2, i1, i3)
 * key, unique rows / unique (i1,i2) prefixes, work chunks), written into the
 * workspace, by a radix sort.  (A forward called with TT_EMB_FORWARD_ONLY on a
 * batch dense in its table -- ceil(M / 32) <= 8 nnz, at most 8192 lookups per
 * SM -- groups by a presence bitmap over the M keys instead: the same unique
 * rows, prefixes, per-lookup unique rows and chunks, without perm and
 * row_start.)  FlowTT summary card, key innovations ("prefix-based index
 * grouping").  tt_emb_forward calls this itself. */
int tt_emb_group(const int64_t m[3], const int32_t n[3], const int32_t R[4],
                 const int64_t* indices, int64_t nnz, const int64_t* offsets,
                 int64_t num_bags, void* workspace, size_t ws_bytes, void* stream);

/* Forward TT embedding bag.  cores[k] as above; out is float32 [num_bags][D]
 * row-major and is overwritten (every bag, empty ones with zeros).  The
 * grouping it builds stays in the workspace for a later
 * tt_emb_backward(..., reuse_grouping = 1). */
int tt_emb_forward(const float* const cores[3], const int64_t m[3], const int32_t n[3],
                   const int32_t R[4], const int64_t* indices, int64_t nnz,
                   const int64_t* offsets, int64_t num_bags, float* out, void* workspace,
                   size_t ws_bytes, void* stream);

/* One table of tt_emb_forward_tables: the arguments of tt_emb_forward. */
typedef struct {
  const float* cores[3];
  int64_t m[3];
  int32_t n[3];
  int32_t R[4];
  const int64_t* indices;
  int64_t nnz;
  const int64_t* offsets;
  int64_t num_bags;
  float* out;
  void* workspace;          /* this table's own workspace (no two tables share one) */
  size_t ws_bytes;
} tt_emb_table;

/* Forward of up to 8 tables in one call (a recommendation model looks up
 * several embedding tables per batch; the pages have no counterpart of this
 * entry point).  Every table's `out` receives exactly what tt_emb_forward would
 * write for it
 * (sum pooling).  All tables share n and R (TT_EMB_ERR_ARG otherwise); their m,
 * batches and workspaces are their own, and workspaces must not overlap.
 * Each table is grouped into its own workspace as by a forward-only call
 * (TT_EMB_FORWARD_ONLY: a backward must not reuse these groupings); for
 * n = (4, 8, 4) with R1 = R2 = 64 (tensor-core chunk kernel) and n = (4, 4, 4)
 * with R1 = R2 = 16 (tiled FP32 chunk kernel) one persistent launch then works
 * through the chunks of all tables (one counter, chunks numbered across the
 * tables), so the tables share the grid instead of each draining it; other
 * shapes run table by table.  num_tables in [1, 8]; the tables' bags together
 * fewer than 2^31 (TT_EMB_ERR_ARG otherwise). */
int tt_emb_forward_tables(int num_tables, const tt_emb_table* tables, void* stream);

/* tt_emb_forward_tables with flags: 0 or a combination of TT_EMB_CORES_SPLIT,
 * which promises that every table's workspace already holds the split of that
 * table's cores (tt_emb_split or tt_emb_sgd_ex on that workspace, as for
 * tt_emb_forward_ex; the per-call split of the cores is then skipped), and
 * TT_EMB_INDICES_I32 (every table's indices are int32; defined below).  Other
 * flag bits: TT_EMB_ERR_ARG. */
int tt_emb_forward_tables_ex(int num_tables, const tt_emb_table* tables, int flags, void* stream);

/* Pooling rules of tt_emb_forward_ex / tt_emb_backward_ex. */
#define TT_EMB_POOL_SUM 0    /* out[b] = sum of the bag's rows (optionally weighted)   */
#define TT_EMB_POOL_MEAN 1   /* out[b] = that sum / number of the bag's lookups        */

/* Flags of tt_emb_forward_ex. */
#define TT_EMB_CORES_SPLIT 1 /* the workspace already holds the bf16 split of these
                                cores (see tt_emb_split): the forward skips the split */
#define TT_EMB_FORWARD_ONLY 2 /* no backward will reuse this call's grouping (inference):
                                the grouping may leave out the per-row lookup lists
                                that only the backward reads (perm and row_start of
                                tt_emb_grouping_view), and a small batch (D <= 256 and
                                nnz * (n1*n2*R2*R1 + D*R2) <= 2^27 multiply-adds) is
                                not grouped at all: each lookup's row is formed on its
                                own (TT-Rec's per-lookup chain) in one launch, and the
                                workspace then holds no grouping.  A tt_emb_backward
                                with reuse_grouping != 0 after such a call adds
                                nothing and tt_emb_get_error returns TT_EMB_ERR_REUSE */
#define TT_EMB_INDICES_I32 4  /* `indices` points at nnz int32 values (4-byte aligned)
                                instead of int64 ones (8-byte aligned); PyTorch's
                                EmbeddingBag takes either.  Values are read as
                                they are (a negative one is out of range).  Also a
                                flag of tt_emb_forward_tables_ex (every table's
                                indices) and tt_emb_step_host (h_indices and
                                d_indices).  A tt_emb_backward that reuses the
                                call's grouping does not read indices; one that
                                regroups reads int64 */

/* Forward with the other pooling rules of an embedding bag (the TT-Rec
 * abstract names its operator after the EmbeddingBag; the pages themselves
 * only sum).  Same arguments and contract as tt_emb_forward, plus:
 *  - per_sample_weights: NULL, or float32 [nnz] (device, 4-byte aligned):
 *    out[b] = sum over the bag's lookups l of per_sample_weights[l] * row(indices[l]).
 *    Only with pooling = TT_EMB_POOL_SUM (TT_EMB_ERR_ARG otherwise).
 *  - pooling: TT_EMB_POOL_SUM, or TT_EMB_POOL_MEAN: every non-empty bag's sum
 *    is divided by its number of lookups (out-of-range lookups included in
 *    the count); empty bags give zeros.
 *  - flags: 0, or a combination of TT_EMB_CORES_SPLIT, when the caller
 *    guarantees that the workspace holds the bf16 split of exactly these core
 *    values, made by the last tt_emb_split, tt_emb_sgd_ex or forward on this
 *    workspace with the cores unchanged since (a serving loop with fixed cores;
 *    a training loop that updates them with tt_emb_sgd_ex), TT_EMB_FORWARD_ONLY
 *    and TT_EMB_INDICES_I32 (above).  Other bits: TT_EMB_ERR_ARG.
 *  - indices must be aligned to its element size (TT_EMB_ERR_ARG otherwise).
 * tt_emb_forward is tt_emb_forward_ex(..., NULL, TT_EMB_POOL_SUM, 0, ...). */
int tt_emb_forward_ex(const float* const cores[3], const int64_t m[3], const int32_t n[3],
                      const int32_t R[4], const int64_t* indices, int64_t nnz,
                      const int64_t* offsets, int64_t num_bags, const float* per_sample_weights,
                      int pooling, int flags, float* out, void* workspace, size_t ws_bytes,
                      void* stream);

/* Backward into the cores: core_grads[k] (same layout as cores[k]) are
 * ACCUMULATED (+=) with d<grad_out, out>/dG_k; the caller zeroes them.
 * grad_out is float32 [num_bags][D].  With reuse_grouping != 0 the grouping
 * left in the workspace by the last tt_emb_forward / tt_emb_group on the SAME
 * indices, offsets and shape is reused (the caller guarantees that, and that
 * the cores' contents did not change since that call: the bf16 split of the
 * cores made by that forward is reused too when the core addresses match);
 * otherwise it is rebuilt.  The accumulation uses float atomics, so the
 * summation order (and the last bits) may differ from call to call. */
int tt_emb_backward(const float* grad_out, const float* const cores[3], const int64_t m[3],
                    const int32_t n[3], const int32_t R[4], const int64_t* indices, int64_t nnz,
                    const int64_t* offsets, int64_t num_bags, float* const core_grads[3],
                    void* workspace, size_t ws_bytes, int reuse_grouping, void* stream);

/* Backward of tt_emb_forward_ex: per_sample_weights and pooling as given to
 * that forward; core_grads accumulated as in tt_emb_backward.
 *  - grad_weights: NULL, or float32 [nnz] (device, 4-byte aligned; requires
 *    per_sample_weights): OVERWRITTEN with d<grad_out, out>/d per_sample_weights[l]
 *    = <grad_out[bag(l)], row(indices[l])>, 0 for out-of-range lookups.  The
 *    rows are recomputed inside this call (one extra pass of the row kernels).
 * tt_emb_backward is tt_emb_backward_ex(..., NULL, TT_EMB_POOL_SUM, core_grads, NULL, ...). */
int tt_emb_backward_ex(const float* grad_out, const float* const cores[3], const int64_t m[3],
                       const int32_t n[3], const int32_t R[4], const int64_t* indices,
                       int64_t nnz, const int64_t* offsets, int64_t num_bags,
                       const float* per_sample_weights, int pooling, float* const core_grads[3],
                       float* grad_weights, void* workspace, size_t ws_bytes, int reuse_grouping,
                       void* stream);

/* Plain SGD on the three cores, one launch: G_k <- G_k - lr * dG_k
 * (element-wise, fp32).  With zero_grads != 0 the same pass also resets every
 * dG_k to zero, ready for the next accumulating tt_emb_backward. */
int tt_emb_sgd(float* const cores[3], float* const core_grads[3], const int64_t m[3],
               const int32_t n[3], const int32_t R[4], float lr, int zero_grads, void* stream);

/* The bf16 split of the cores (hi = bf16(x), lo = bf16(x - hi), the operands
 * of the three-term tensor-core products) into the workspace, where it stays
 * until the cores are split again: later forwards on this workspace may pass
 * TT_EMB_CORES_SPLIT while the core values do not change.  The planes sit at
 * offsets that depend on the shape alone, so any workspace sized for this
 * shape (any batch) holds them; a smaller one returns TT_EMB_ERR_WORKSPACE.
 * Shapes without tensor-core kernels have no planes: the call does nothing.
 * (The pages have no counterpart: the split is this implementation's operand
 * format.) */
int tt_emb_split(const float* const cores[3], const int64_t m[3], const int32_t n[3],
                 const int32_t R[4], void* workspace, size_t ws_bytes, void* stream);

/* tt_emb_sgd, and in the same pass the split of the updated cores into the
 * workspace (as tt_emb_split would make it), so that the next forward may pass
 * TT_EMB_CORES_SPLIT.  Workspace requirements as for tt_emb_split. */
int tt_emb_sgd_ex(float* const cores[3], float* const core_grads[3], const int64_t m[3],
                  const int32_t n[3], const int32_t R[4], float lr, int zero_grads,
                  void* workspace, size_t ws_bytes, void* stream);

/* The host-side arrays of one batch for tt_emb_step_host (the one entry
 * point that takes HOST arrays) and the caller's device arrays they are
 * copied to and from.  Host arrays should be page-locked (cudaHostAlloc /
 * cudaHostRegister): copies from or to pageable memory are correct but block
 * the calling thread and do not overlap. */
typedef struct {
  const int64_t* h_indices;  /* host, nnz entries (int32 with TT_EMB_INDICES_I32)       */
  const int64_t* h_offsets;  /* host, num_bags + 1 entries (CSR, as above)             */
  const float* h_grad_out;   /* host, float32 [num_bags][D], or NULL: forward only      */
  float* h_out;              /* host, float32 [num_bags][D], or NULL: not copied back   */
  int64_t* d_indices;        /* device, nnz entries, aligned to their size (likewise)   */
  int64_t* d_offsets;        /* device, num_bags + 1 entries                            */
  float* d_grad_out;         /* device, [num_bags][D], 16-byte aligned (training only)  */
  float* d_out;              /* device, [num_bags][D], 16-byte aligned                  */
  int64_t nnz;
  int64_t num_bags;
} tt_emb_host_batch;

/* One step from host memory (a training step when batch->h_grad_out is not
 * NULL, else a forward): indices and offsets are copied in, the forward
 * (tt_emb_forward_ex with sum pooling and `flags`) runs into d_out, and for a
 * training step the output gradient is copied in, tt_emb_backward reuses the
 * forward's grouping and tt_emb_sgd_ex(lr, zero_grads = 1) updates the cores
 * (so the next step may pass TT_EMB_CORES_SPLIT); h_out receives the pooled
 * output.  Indices and offsets are copied in on `stream`, after the work
 * enqueued on it before the call, and the forward follows them there; the
 * output gradient is copied in on `copy_stream` once they are in, while the
 * forward runs, and the output is copied back on `copy_stream` while the
 * backward runs, all ordered by events.  Everything the call does is complete when `stream` reaches the end
 * of what it enqueued, h_out included.  copy_stream may equal stream (no
 * overlap).  `flags` as for tt_emb_forward_ex; TT_EMB_FORWARD_ONLY only for a
 * forward (TT_EMB_ERR_ARG with h_grad_out).  core_grads may be NULL for a forward; otherwise they are
 * overwritten with zeros after the SGD.  Argument errors return before
 * anything is enqueued; device-side conditions as for the calls named.  If a
 * call fails after its copies were enqueued (a CUDA error, or an error code
 * of one of the calls named), `stream` is still made to wait for every copy
 * the call enqueued, so the host buffers may be reused once `stream` drains.
 * Graphs: the second call of a thread whose arguments (every pointer, size,
 * lr, flags and both streams) equal an earlier call's captures the call's
 * work into a CUDA graph, and later such calls launch that graph on `stream`
 * (the same copies and kernels with the same dependencies, without their
 * launch costs), after the work enqueued on either stream before the call and
 * before the copy stream's later work.  A thread keeps the last four argument
 * sets per device.  Calls with pageable host buffers, on the legacy or
 * per-thread default stream, on a stream being captured, or with launch
 * records on (tt_emb_profile_start) always run eagerly.  The events and
 * graphs belong to the device's context: after cudaDeviceReset a thread's
 * calls return TT_EMB_ERR_CUDA. */
int tt_emb_step_host(float* const cores[3], float* const core_grads[3], const int64_t m[3],
                     const int32_t n[3], const int32_t R[4], const tt_emb_host_batch* batch,
                     float lr, int flags, void* workspace, size_t ws_bytes, void* stream,
                     void* copy_stream);

/* Chains of d cores, 3 <= d <= 8 (tt_emb_sgd_d: 2 <= d <= 8): core k is
 * float32 [m[k]][R[k]][n[k]][R[k+1]], R has d + 1 entries with R[0] = R[d] = 1,
 * the row index splits mixed-radix over m (m[0] most significant) and the
 * output position over n likewise; otherwise the contracts of tt_emb_forward,
 * tt_emb_backward and tt_emb_sgd (`cores` and `core_grads` point to d HOST
 * arrays of device pointers).  d = 3 is the three-core call.  For d >= 4 the
 * leading d - 2 cores are contracted once per call into one core over all
 * their index combinations (its (m[0]..m[d-3]) (n[0]..n[d-3]) R[d-2] floats
 * live in the workspace; more than 2^28 of them, or m[0]..m[d-3] >= 2^31,
 * return TT_EMB_ERR_UNSUPPORTED) and the three-core path runs on that core
 * and the last two; the backward carries the merged core's gradient back to
 * the leading cores.  With reuse_grouping != 0 the merged core of the last
 * tt_emb_forward_d on this workspace is reused too (the cores are unchanged
 * under that contract).  Size the workspace with tt_emb_workspace_bytes_d. */
int tt_emb_workspace_bytes_d(int d, const int64_t* m, const int32_t* n, const int32_t* R,
                             int64_t nnz, int64_t num_bags, size_t* bytes);
int tt_emb_forward_d(int d, const float* const* cores, const int64_t* m, const int32_t* n,
                     const int32_t* R, const int64_t* indices, int64_t nnz, const int64_t* offsets,
                     int64_t num_bags, float* out, void* workspace, size_t ws_bytes, void* stream);
int tt_emb_backward_d(int d, const float* grad_out, const float* const* cores, const int64_t* m,
                      const int32_t* n, const int32_t* R, const int64_t* indices, int64_t nnz,
                      const int64_t* offsets, int64_t num_bags, float* const* core_grads,
                      void* workspace, size_t ws_bytes, int reuse_grouping, void* stream);
int tt_emb_sgd_d(int d, float* const* cores, float* const* core_grads, const int64_t* m,
                 const int32_t* n, const int32_t* R, float lr, int zero_grads, void* stream);

/* Synchronises `stream`, then reads the workspace status word written by the
 * kernels of the calls enqueued so far.  *device_status receives the raw
 * bit set (1 = index out of range, 2 = bad offsets, 4 = timeout, 8 = a
 * backward reused a forward-only grouping).  Returns TT_EMB_OK or the code of
 * the most severe condition found (TIMEOUT > REUSE > OFFSETS > INDEX), or
 * TT_EMB_ERR_CUDA. */
int tt_emb_get_error(const void* workspace, void* stream, int* device_status);

/* Device pointers into a workspace holding a grouping (pure pointer
 * arithmetic; reads no device memory).  For inspection and tests. */
typedef struct {
  const int32_t* counts;          /* [0] valid lookups, [1] U_r unique rows, [2] U_12 unique
                                     (i1,i2) prefixes, [3] work chunks, [4] status bits,
                                     [5] grouping method: 1 key bitmap (a forward-only
                                     call: no perm, no row_start), 2 one-launch radix sort,
                                     3 multi-launch radix sort, [6] work chunks of the last
                                     forward that took their prefix partial from the L2
                                     checkpoint instead of forming it                      */
  const int32_t* perm;            /* [nnz]   lookup positions sorted by (i2,i1,i3, position);
                                              out-of-range lookups last                     */
  const int32_t* row_start;       /* [U_r+1] first sorted position of each unique row         */
  const int32_t* row_i3;          /* [U_r]   i3 digit of each unique row                       */
  const int32_t* row_pair;        /* [U_r]   unique prefix of each unique row                  */
  const int32_t* pair_row_start;  /* [U_12+1] first unique row of each unique prefix           */
  const int32_t* pair_i1;         /* [U_12]                                                     */
  const int32_t* pair_i2;         /* [U_12]                                                     */
  const int32_t* uid;             /* [nnz]   unique row of each lookup, -1 if out of range      */
  const int32_t* bag_of;          /* [nnz]   bag of each lookup (written by tt_emb_backward)   */
  const int32_t* chunk_start;     /* [chunks+1] first unique row of each work chunk             */
  const float* rowbuf;            /* [U_r][D] unique rows (after a forward)                    */
  const int32_t* chunk_order;     /* [chunks]   the chunk each forward claim takes (a hot
                                                prefix's later pieces after all other chunks)  */
} tt_emb_grouping;

int tt_emb_grouping_view(const int64_t m[3], const int32_t n[3], const int32_t R[4],
                         int64_t nnz, int64_t num_bags, const void* workspace,
                         tt_emb_grouping* view);

/* Opt-in launch timing (process-wide host state, off by default, not
 * thread-safe).  After tt_emb_profile_start, every kernel launch of the
 * library is bracketed by two CUDA events recorded on its stream (inside a
 * stream capture they become event nodes of the graph).
 * tt_emb_profile_stop ends recording and returns the number of launches
 * recorded.  tt_emb_profile_read(i, ...) synchronises the i-th record's end
 * event and returns the kernel's name and its device duration in ms. */
int tt_emb_profile_start(void);
int tt_emb_profile_stop(void);
int tt_emb_profile_read(int i, char* name, int name_len, float* ms);

/* Forward for callers that cannot allocate device memory.  (None of the TT embedding designs has a
 * counterpart of this entry point.)  Some callers cannot call cudaMalloc at
 * all -- an allocator-less runtime that only hands out input and output
 * buffers, a plugin whose host framework owns every device allocation, code
 * that must not allocate once it is in steady state -- and so cannot provide
 * the workspace tt_emb_forward needs.  This variant computes exactly what
 * tt_emb_forward computes, with the same arguments minus the workspace: its
 * scratch is one file-scope device array of TT_EMB_STATIC_WORKSPACE_BYTES
 * (16 MiB) that every GPU loading this library holds until the process exits.
 *  - Sizes whose tt_emb_workspace_bytes exceed that capacity return
 *    TT_EMB_ERR_WORKSPACE before anything is enqueued (for D = 128 with
 *    R1 = R2 = 32 about 21k lookups at m = (100, 60, 120) and 11k at
 *    m = (200, 240, 250): the bf16 split of the cores takes part of it).
 *  - The first call on a device looks up the array's device address with
 *    that device current; make that first call before any stream capture.
 *    The address is kept per device id for the life of the process: after a
 *    cudaDeviceReset the array is gone and so is its cached address, so this
 *    entry point must not be called again in that process.
 *  - Every call shares the one array, which keeps the last call's contents;
 *    the call clears what must start at zero itself.  Calls whose work
 *    overlaps on the GPU (other streams or threads) race on the array: the
 *    caller must serialise them.
 *  - It allocates nothing: no cudaMalloc, cudaFree or allocating library
 *    routine.  Argument errors are returned as usual; conditions found by
 *    the kernels (an index outside [0, M), bad offsets) are handled as in
 *    tt_emb_forward (the lookup contributes nothing) but their status word
 *    lives in the shared array and is not reported. */
#define TT_EMB_STATIC_WORKSPACE_BYTES (16u << 20)
int tt_emb_forward_static(const float* const cores[3], const int64_t m[3], const int32_t n[3],
                          const int32_t R[4], const int64_t* indices, int64_t nnz,
                          const int64_t* offsets, int64_t num_bags, float* out, void* stream);

/* Library version (major*10000 + minor*100 + patch). */
int tt_emb_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TT_EMB_H */
