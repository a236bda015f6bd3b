// Opt-in launch timing: when enabled, every kernel launch of the library is
// bracketed by two CUDA events recorded on its stream, so that per-kernel
// device durations can be read back afterwards (also inside a captured CUDA
// graph, where the records become event nodes).  Off by default; host state
// of the process, not thread-safe.
#include <string.h>

#include <vector>

#include "tt_internal.cuh"

namespace tt {

bool g_prof_on = false;

namespace {
struct Rec {
  const char* name;
  int a, b;   // indices into the event pool
};
std::vector<cudaEvent_t> g_pool;
std::vector<Rec> g_recs;
size_t g_next = 0;
int g_open = -1;

// Inside a stream capture a plain record only orders the graph; the external
// flag makes it an event node that takes a timestamp on every replay.
void record(cudaEvent_t e, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(e, st, cudaEventRecordExternal);
  else
    cudaEventRecord(e, st);
}

int take_event() {
  if (g_next == g_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return -1;
    g_pool.push_back(e);
  }
  return (int)g_next++;
}
}  // namespace

void prof_begin(const char* name, cudaStream_t st) {
  if (!g_prof_on) return;
  const int a = take_event();
  if (a < 0) return;
  record(g_pool[a], st);
  g_recs.push_back(Rec{name, a, -1});
  g_open = (int)g_recs.size() - 1;
}

void prof_end(cudaStream_t st) {
  if (!g_prof_on || g_open < 0) return;
  const int b = take_event();
  if (b >= 0) {
    record(g_pool[b], st);
    g_recs[g_open].b = b;
  }
  g_open = -1;
}

}  // namespace tt

using namespace tt;

extern "C" {

int tt_emb_profile_start(void) {
  g_recs.clear();
  g_next = 0;
  g_open = -1;
  g_prof_on = true;
  return TT_EMB_OK;
}

int tt_emb_profile_stop(void) {
  g_prof_on = false;
  return (int)g_recs.size();
}

int tt_emb_profile_read(int i, char* name, int name_len, float* ms) {
  if (i < 0 || i >= (int)g_recs.size() || !ms) return TT_EMB_ERR_ARG;
  const Rec& r = g_recs[(size_t)i];
  if (name && name_len > 0) {
    strncpy(name, r.name, (size_t)name_len - 1);
    name[name_len - 1] = 0;
  }
  if (r.b < 0) return TT_EMB_ERR_ARG;
  if (cudaEventSynchronize(g_pool[(size_t)r.b]) != cudaSuccess) return TT_EMB_ERR_CUDA;
  if (cudaEventElapsedTime(ms, g_pool[(size_t)r.a], g_pool[(size_t)r.b]) != cudaSuccess)
    return TT_EMB_ERR_CUDA;
  return TT_EMB_OK;
}

}  // extern "C"
