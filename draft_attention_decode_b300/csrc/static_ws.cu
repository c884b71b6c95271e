// draft_attn_run_static: draft_attn_run with a library-owned workspace.
//
// For callers that cannot allocate device memory at the point where they run
// the draft step: code running inside another framework's memory pool or
// allocator hooks, a captured or replayed sequence where an allocation would
// be illegal, or a runtime that only hands out the tensors it owns.  The
// scratch is a fixed array in the library's device image, so the call itself
// allocates nothing.
#include <mutex>

#include "internal.h"

// The shared scratch: every GPU that loads the library holds this array
// until the process exits.
static __device__ __align__(256) uint8_t g_da_static_ws[DA_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;

struct StaticWs {
  std::mutex mu;
  void* ptr[kMaxDevices] = {};
};

StaticWs& static_ws() {
  static StaticWs s;
  return s;
}

// Device address of the array on `device`, looked up with that device
// current.  In host code the array's name is only a host-side stand-in; this
// lookup is the address a kernel may be given.  Only a successful lookup is
// kept: after a failure (which also clears the runtime's last-error state)
// the next call tries again.
void* static_ws_ptr(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  StaticWs& s = static_ws();
  std::lock_guard<std::mutex> lock(s.mu);
  if (s.ptr[device]) return s.ptr[device];
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (prev != device && cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_da_static_ws) == cudaSuccess) {
    s.ptr[device] = p;
  } else {
    p = nullptr;
    cudaGetLastError();
  }
  if (prev != device) cudaSetDevice(prev);
  return p;
}

}  // namespace

extern "C" int draft_attn_run_static(da_plan_t plan, const void* q, const int32_t* q_pos,
                                     const int32_t* ctx_lens, const int32_t* block_table,
                                     const void* k_cache, const void* v_cache,
                                     const void* k_side, void* out, void* stream) {
  int device = -1;
  size_t counter_bytes = 0, workspace_bytes = 0;
  if (!da::plan_workspace_layout(plan, &device, &counter_bytes, &workspace_bytes))
    return DA_ERR_INVALID_ARG;
  if (workspace_bytes > (size_t)DA_STATIC_WORKSPACE_BYTES) return DA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = static_ws_ptr(device);
  if (!ws) return DA_ERR_CUDA;
  // The page counters at the head of the workspace must start at zero; the
  // array keeps whatever the previous call left, so clear them on the stream.
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return DA_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return DA_ERR_CUDA;
  const cudaError_t e = cudaMemsetAsync(ws, 0, counter_bytes, static_cast<cudaStream_t>(stream));
  if (prev != device) cudaSetDevice(prev);
  if (e != cudaSuccess) return DA_ERR_CUDA;
  return draft_attn_run(plan, q, q_pos, ctx_lens, block_table, k_cache, v_cache, k_side, out, ws,
                        (size_t)DA_STATIC_WORKSPACE_BYTES, stream);
}
