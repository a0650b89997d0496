// oscar_decode_attention_static: decode attention with a library-owned,
// statically allocated workspace, for callers that cannot allocate device
// memory themselves.
//
// The workspace is one file-scope __device__ array of kStaticWorkspaceBytes.
// Host code never uses the array's name as a device address (on the host it
// names a host-side shadow); the device address is looked up with
// cudaGetSymbolAddress while the device is current, once per device and
// context: the lookup is repeated when the device's current context is not
// the one the cached address belongs to (after cudaDeviceReset the module
// is loaded again and the array may move).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "oscar.h"
#include "trace.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(OSCAR_STATIC_WORKSPACE_BYTES);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mutex;
void* g_ptr[kMaxDevices] = {nullptr};
CUcontext g_ctx[kMaxDevices] = {nullptr};

// The calling thread's current driver context (nullptr if none or if the
// driver entry point is unavailable).
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 get = nullptr;
  if (!get) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  }
  CUcontext c = nullptr;
  return get(&c) == CUDA_SUCCESS ? c : nullptr;
}

// Device address of g_static_workspace on the current device.  The first
// call on a device (and the first after its context changed) performs the
// lookup; later calls reuse it.
oscar_status static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return OSCAR_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  const CUcontext ctx = current_context();
  if (!g_ptr[dev] || !ctx || ctx != g_ctx[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) return OSCAR_ERR_CUDA;
    g_ptr[dev] = ptr;
    // (the runtime made its primary context current during the lookup)
    g_ctx[dev] = current_context();
  }
  *out = g_ptr[dev];
  return OSCAR_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

extern "C" oscar_status oscar_decode_attention_static(const oscar_layer_desc* desc, const uint16_t* q,
                                                      float* out, void* stream) {
  OSCAR_TRACE_CALL();
  if (!desc) return OSCAR_ERR_INVALID_ARG;
  size_t need = 0;
  oscar_status st = oscar_decode_attention(desc, q, out, nullptr, &need, stream);
  if (st != OSCAR_OK) return st;
  if (need > kStaticWorkspaceBytes) return OSCAR_ERR_WORKSPACE;   // beyond the static maximum
  void* ws = nullptr;
  st = static_workspace(&ws);
  if (st != OSCAR_OK) return st;
  // the merge tickets at the start of the workspace must be zero; the rest
  // is written before it is read
  const size_t tickets = align256(size_t(desc->batch) * size_t(desc->n_kv_heads) * 4);
  if (cudaMemsetAsync(ws, 0, tickets, static_cast<cudaStream_t>(stream)) != cudaSuccess) return OSCAR_ERR_CUDA;
  size_t have = kStaticWorkspaceBytes;
  return oscar_decode_attention(desc, q, out, ws, &have, stream);
}
