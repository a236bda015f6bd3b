// tt_emb_forward_static: the forward TT embedding bag for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a workspace: code that runs where
// cudaMalloc is forbidden or unavailable (an allocator-less runtime that only
// hands out input and output buffers, a plugin whose host framework owns all
// device allocations, or code that must not allocate between a warm-up and
// its steady state).  For them this entry point takes its scratch from one
// file-scope device array of fixed size instead of a caller-owned workspace.
//
// The array holds kStaticWorkspaceBytes (16 MiB) on every GPU that loads this
// library, until the process exits.  Its address is looked up once per device
// (cudaGetSymbolAddress, with that device current) on the first call that
// device sees; that first call should therefore come before any stream
// capture.  All calls share the one array and it keeps the last call's
// contents: calls whose kernels overlap on the GPU (two streams, or two
// threads) race on it and must be serialised by the caller.  Everything a
// call needs zeroed is cleared by the call itself.
#include <mutex>

#include "tt_internal.cuh"

namespace tt {

constexpr size_t kStaticWorkspaceBytes = TT_EMB_STATIC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

namespace {
constexpr int kMaxDevices = 64;
void* g_static_ptr[kMaxDevices] = {nullptr};
std::mutex g_static_mu;

// Device address of the array on the current device (looked up once).
int static_workspace(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TT_EMB_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TT_EMB_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return TT_EMB_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *ptr = g_static_ptr[dev];
  return TT_EMB_OK;
}
}  // namespace

}  // namespace tt

using namespace tt;

extern "C" {

int tt_emb_forward_static(const float* const cores[3], const int64_t m[3], const int32_t n[3],
                          const int32_t R[4], const int64_t* indices, int64_t nnz,
                          const int64_t* offsets, int64_t num_bags, float* out, void* stream) {
  size_t need = 0;
  int rc = tt_emb_workspace_bytes(m, n, R, nnz, num_bags, &need);
  if (rc) return rc;
  if (need > kStaticWorkspaceBytes) return TT_EMB_ERR_WORKSPACE;
  void* ws = nullptr;
  rc = static_workspace(&ws);
  if (rc) return rc;
  return tt_emb_forward(cores, m, n, R, indices, nnz, offsets, num_bags, out, ws,
                        kStaticWorkspaceBytes, stream);
}

}  // extern "C"
