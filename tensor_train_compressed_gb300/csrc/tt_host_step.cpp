// One step from host memory (tt_emb_step_host): the batch is copied in on a
// copy stream, the pooled output copied back, and the kernels of the step run
// on the caller's stream in between, ordered by events so that the copies of
// the output gradient and of the pooled output overlap with the forward and
// with the backward.  Host code only: every kernel is launched through the
// other entry points of the library.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <vector>

#include "../../include/tt_emb.h"

namespace tt {
extern bool g_prof_on;   // opt-in launch records (tt_prof.cu): calls then run eagerly
}

namespace {

enum { kEvIn, kEvGrad, kEvFwd, kEvDone, kNumEv };

// Events of this thread on the current device, created once and reused: a
// wait enqueued on a stream refers to the record that preceded it, so a later
// call may record the same events again.
int step_events(cudaEvent_t** ev) {
  thread_local std::vector<std::vector<cudaEvent_t>> per_device;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return TT_EMB_ERR_CUDA;
  if ((size_t)dev >= per_device.size()) per_device.resize(dev + 1);
  std::vector<cudaEvent_t>& e = per_device[dev];
  if (e.empty()) {
    e.assign(kNumEv, nullptr);
    for (int i = 0; i < kNumEv; ++i)
      if (cudaEventCreateWithFlags(&e[i], cudaEventDisableTiming) != cudaSuccess) {
        for (int j = 0; j < i; ++j) cudaEventDestroy(e[j]);
        e.clear();
        return TT_EMB_ERR_CUDA;
      }
  }
  *ev = e.data();
  return TT_EMB_OK;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// Every argument of one call, compared byte for byte (zero-filled, so that
// padding compares equal).
struct StepKey {
  const void* cores[3];
  const void* grads[3];
  int64_t m[3];
  int32_t n[3];
  int32_t R[4];
  tt_emb_host_batch b;
  uint32_t lr_bits;
  int flags;
  const void* ws;
  size_t ws_bytes;
  const void* st;
  const void* cs;
};

// One set of call arguments seen by this thread on a device: the graph of
// its work once the same arguments came a second time (then captured),
// no_graph if that capture failed.
struct StepGraph {
  bool valid = false, no_graph = false;
  StepKey key;
  cudaGraphExec_t exec = nullptr;
};
constexpr int kStepGraphs = 4;   // argument sets kept per thread and device

struct StepGraphs {
  StepGraph e[kStepGraphs];
  int next = 0;                  // the entry a new argument set replaces
};

StepGraphs* step_graphs() {
  thread_local std::vector<StepGraphs> per_device;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  if ((size_t)dev >= per_device.size()) per_device.resize(dev + 1);
  return &per_device[dev];
}

bool pinned_or_absent(const void* p, bool needed) {
  if (!needed || !p) return true;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// Whether the call's work may be captured into a graph: both streams are
// ordinary streams not already being captured, every host buffer is page-locked
// (a copy from pageable memory cannot be captured), and launch records are off.
bool graph_eligible(cudaStream_t st, cudaStream_t cs, const tt_emb_host_batch& b, bool train,
                    size_t out_bytes) {
  if (tt::g_prof_on) return false;
  for (cudaStream_t x : {st, cs}) {
    if (x == nullptr || x == cudaStreamLegacy || x == cudaStreamPerThread) return false;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(x, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone)
      return false;
  }
  return pinned_or_absent(b.h_indices, b.nnz > 0) && pinned_or_absent(b.h_offsets, true) &&
         pinned_or_absent(b.h_grad_out, train && out_bytes > 0) &&
         pinned_or_absent(b.h_out, out_bytes > 0);
}

bool cores_ok(const void* const* c) {
  if (!c) return false;
  for (int k = 0; k < 3; ++k)
    if (!c[k] || !aligned(c[k], 16)) return false;
  return true;
}

// The step's work, enqueued on `st` and `cs` (eagerly, or into a capture).
int enqueue_step(float* const cores[3], float* const core_grads[3], const int64_t m[3],
                 const int32_t n[3], const int32_t R[4], const tt_emb_host_batch& b, float lr,
                 int flags, void* workspace, size_t ws_bytes, cudaStream_t st, cudaStream_t cs,
                 size_t idx_bytes, size_t out_bytes, bool train) {
  void* stream = st;
  int rc = 0;
  cudaEvent_t* ev = nullptr;
  rc = step_events(&ev);
  if (rc) return rc;
  bool ok = true;
  auto cuda = [&ok](cudaError_t e) { ok = ok && e == cudaSuccess; };

  // Once a copy is enqueued, every return goes through `finish`: it still
  // records kEvDone on the copy stream and makes `stream` wait for it, so
  // that the caller's host buffers are free to reuse once `stream` drains,
  // whatever failed on the way.
  auto finish = [&](int code) {
    cudaError_t e1 = cudaEventRecord(ev[kEvDone], cs);
    cudaError_t e2 = cudaStreamWaitEvent(st, ev[kEvDone], 0);
    if (code) return code;
    return (ok && e1 == cudaSuccess && e2 == cudaSuccess) ? TT_EMB_OK : TT_EMB_ERR_CUDA;
  };

  // The lookups come in on `stream` itself, after the work the caller ordered
  // before this call, so the forward follows them with no wait across
  // streams; the output gradient comes in on the copy stream once they are in
  // (not competing with them for the copy bandwidth) while the forward runs.
  if (b.nnz > 0)
    cuda(cudaMemcpyAsync(b.d_indices, b.h_indices, idx_bytes * (size_t)b.nnz,
                         cudaMemcpyHostToDevice, st));
  cuda(cudaMemcpyAsync(b.d_offsets, b.h_offsets, sizeof(int64_t) * (size_t)(b.num_bags + 1),
                       cudaMemcpyHostToDevice, st));
  cuda(cudaEventRecord(ev[kEvIn], st));
  cuda(cudaStreamWaitEvent(cs, ev[kEvIn], 0));
  if (!ok) return TT_EMB_ERR_CUDA;            // nothing enqueued on the copy stream yet
  if (train && out_bytes > 0)
    cuda(cudaMemcpyAsync(b.d_grad_out, b.h_grad_out, out_bytes, cudaMemcpyHostToDevice, cs));
  cuda(cudaEventRecord(ev[kEvGrad], cs));
  if (!ok) return finish(TT_EMB_ERR_CUDA);
  const float* const* cc = (const float* const*)cores;
  rc = tt_emb_forward_ex(cc, m, n, R, b.d_indices, b.nnz, b.d_offsets, b.num_bags, nullptr,
                         TT_EMB_POOL_SUM, flags, b.d_out, workspace, ws_bytes, stream);
  if (rc) return finish(rc);
  cuda(cudaEventRecord(ev[kEvFwd], st));
  if (train) {
    // backward on the forward's grouping and split, then SGD that resets the
    // gradients and leaves the split of the updated cores
    cuda(cudaStreamWaitEvent(st, ev[kEvGrad], 0));
    if (!ok) return finish(TT_EMB_ERR_CUDA);
    rc = tt_emb_backward(b.d_grad_out, cc, m, n, R, b.d_indices, b.nnz, b.d_offsets, b.num_bags,
                         core_grads, workspace, ws_bytes, 1, stream);
    if (rc) return finish(rc);
    rc = tt_emb_sgd_ex(cores, core_grads, m, n, R, lr, 1, workspace, ws_bytes, stream);
    if (rc) return finish(rc);
  }
  // the pooled output goes back while the backward runs; enqueued after the
  // kernels, since a copy into pageable host memory blocks the host
  cuda(cudaStreamWaitEvent(cs, ev[kEvFwd], 0));
  if (b.h_out && out_bytes > 0 && ok)
    cuda(cudaMemcpyAsync(b.h_out, b.d_out, out_bytes, cudaMemcpyDeviceToHost, cs));
  return finish(TT_EMB_OK);
}

}  // namespace

extern "C" int tt_emb_step_host(float* const cores[3], float* const core_grads[3],
                                const int64_t m[3], const int32_t n[3], const int32_t R[4],
                                const tt_emb_host_batch* batch, float lr, int flags,
                                void* workspace, size_t ws_bytes, void* stream,
                                void* copy_stream) {
  // Every check of the calls below is made here first, so that an argument
  // error returns before any copy is enqueued.
  if (!batch) return TT_EMB_ERR_ARG;
  const tt_emb_host_batch& b = *batch;
  size_t need = 0;
  int rc = tt_emb_workspace_bytes(m, n, R, b.nnz, b.num_bags, &need);
  if (rc) return rc;
  const bool train = b.h_grad_out != nullptr;
  if (flags & ~(TT_EMB_CORES_SPLIT | TT_EMB_FORWARD_ONLY | TT_EMB_INDICES_I32)) return TT_EMB_ERR_ARG;
  const size_t idx_bytes = (flags & TT_EMB_INDICES_I32) ? sizeof(int32_t) : sizeof(int64_t);
  if (train && (flags & TT_EMB_FORWARD_ONLY)) return TT_EMB_ERR_ARG;   // the backward reuses it
  if (!cores_ok((const void* const*)cores) || (train && !cores_ok((const void* const*)core_grads)))
    return TT_EMB_ERR_ARG;
  if (b.nnz > 0 && (b.num_bags == 0 || !b.h_indices || !b.d_indices || !aligned(b.d_indices, idx_bytes)))
    return TT_EMB_ERR_ARG;
  if (b.num_bags >= (1ll << 31)) return TT_EMB_ERR_ARG;
  if (!b.h_offsets || !b.d_offsets) return TT_EMB_ERR_ARG;
  if (b.num_bags > 0 && (!b.d_out || !aligned(b.d_out, 16))) return TT_EMB_ERR_ARG;
  if (train && b.num_bags > 0 && (!b.d_grad_out || !aligned(b.d_grad_out, 16)))
    return TT_EMB_ERR_ARG;
  if (!workspace || !aligned(workspace, 256)) return TT_EMB_ERR_ARG;
  if (ws_bytes < need) return TT_EMB_ERR_WORKSPACE;

  const int64_t D = (int64_t)n[0] * n[1] * n[2];
  const size_t out_bytes = sizeof(float) * (size_t)b.num_bags * (size_t)D;
  cudaStream_t st = (cudaStream_t)stream, cs = (cudaStream_t)copy_stream;

  StepKey key;
  memset(&key, 0, sizeof key);
  for (int k = 0; k < 3; ++k) {
    key.cores[k] = cores[k];
    key.grads[k] = core_grads ? core_grads[k] : nullptr;
    key.m[k] = m[k];
    key.n[k] = n[k];
  }
  for (int k = 0; k < 4; ++k) key.R[k] = R[k];
  key.b = b;
  memcpy(&key.lr_bits, &lr, sizeof lr);
  key.flags = flags;
  key.ws = workspace;
  key.ws_bytes = ws_bytes;
  key.st = st;
  key.cs = cs;
  // A call with the same arguments as an earlier one of this thread replays
  // the CUDA graph of that work (captured the second time the arguments come):
  // the same copies and kernels in the same order, without their launch costs.
  StepGraphs* gs = step_graphs();
  if (gs && graph_eligible(st, cs, b, train, out_bytes)) {
    StepGraph* g = nullptr;
    for (StepGraph& e : gs->e)
      if (e.valid && memcmp(&e.key, &key, sizeof key) == 0) g = &e;
    if (!g) {                                   // a new argument set: run it eagerly
      g = &gs->e[gs->next];
      gs->next = (gs->next + 1) % kStepGraphs;
      if (g->exec) cudaGraphExecDestroy(g->exec);   // freed once a replay in flight ends
      g->exec = nullptr;
      g->valid = true;
      g->no_graph = false;
      g->key = key;
    } else if (!g->no_graph) {
      if (!g->exec) {                           // the second time: capture the work
        cudaGraph_t graph = nullptr;
        bool good = false;
        if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
          const int crc = enqueue_step(cores, core_grads, m, n, R, b, lr, flags, workspace,
                                       ws_bytes, st, cs, idx_bytes, out_bytes, train);
          const cudaError_t e = cudaStreamEndCapture(st, &graph);
          good = crc == TT_EMB_OK && e == cudaSuccess && graph != nullptr &&
                 cudaGraphInstantiate(&g->exec, graph, 0) == cudaSuccess;
          if (graph) cudaGraphDestroy(graph);
        }
        if (!good) {                            // nothing of it ran: run it eagerly
          cudaGetLastError();
          if (g->exec) cudaGraphExecDestroy(g->exec);
          g->exec = nullptr;
          g->no_graph = true;
        }
      }
      if (g->exec) {
        // ordered as the eager calls are: after the caller's earlier work on
        // both streams, and the copy stream's later work after this call's
        cudaEvent_t* ev = nullptr;
        rc = step_events(&ev);
        if (rc) return rc;
        bool ok = cudaEventRecord(ev[kEvIn], cs) == cudaSuccess &&
                  cudaStreamWaitEvent(st, ev[kEvIn], 0) == cudaSuccess &&
                  cudaGraphLaunch(g->exec, st) == cudaSuccess;
        ok = cudaEventRecord(ev[kEvDone], st) == cudaSuccess && ok;
        ok = cudaStreamWaitEvent(cs, ev[kEvDone], 0) == cudaSuccess && ok;
        return ok ? TT_EMB_OK : TT_EMB_ERR_CUDA;
      }
    }
  }
  return enqueue_step(cores, core_grads, m, n, R, b, lr, flags, workspace, ws_bytes, st, cs,
                      idx_bytes, out_bytes, train);
}
