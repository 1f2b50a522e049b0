// vsa_forward_static_workspace: the VSA forward for callers that cannot
// allocate device memory.
//
// Some hosts of this library hand a kernel only its input and output buffers
// and give it no way to allocate: serving engines that budget every byte of
// device memory at start-up, plugin interfaces without an allocator callback,
// or latency-critical paths where a cudaMalloc (which can synchronise the
// device) is not acceptable. This entry point runs the regular forward with
// its scratch (pooled statistics, tile selections, coarse output, error
// words) placed in a fixed-size array that lives in the library itself.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds VSA_STATIC_WORKSPACE_BYTES of device memory until the process
// exits. Host code cannot use the array's name as a device address (it is a
// host-side stand-in); the device address is resolved with
// cudaGetSymbolAddress, once per device, with that device current, on the
// first call made for a plan on that device.
#include <mutex>

#include "kernels.cuh"
#include "plan.h"
#include "vsa.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[VSA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_workspace_ptr[kMaxDevices] = {};

// Device address of g_static_workspace on `device` (the current device),
// resolved on first use. Returns null if the runtime cannot resolve it.
void* static_workspace(int device) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_workspace_ptr[device] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess) {
      cudaGetLastError();  // do not leave the failed lookup as the sticky "last error"
      return nullptr;
    }
    g_workspace_ptr[device] = ptr;
  }
  return g_workspace_ptr[device];
}

// Runs fn(ws) with the plan's device current and ws the device address of the
// array on it; restores the caller's device afterwards.
template <typename Fn>
vsa_status_t with_static_workspace(vsa_plan_t plan, Fn&& fn) {
  const int device = plan->device;
  if (device < 0 || device >= kMaxDevices) return VSA_ERR_UNSUPPORTED;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return VSA_ERR_CUDA;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return VSA_ERR_CUDA;
  void* ws = static_workspace(device);
  const vsa_status_t s = ws != nullptr ? fn(ws) : VSA_ERR_CUDA;
  if (prev != device) cudaSetDevice(prev);
  return s;
}

}  // namespace

extern "C" vsa_status_t vsa_forward_static_workspace(vsa_plan_t plan, const void* q, const void* k,
                                                     const void* v, const void* gate, void* out,
                                                     void* stream) {
  if (!plan) return VSA_ERR_INVALID_ARG;
  if (plan->ws_bytes > VSA_STATIC_WORKSPACE_BYTES) return VSA_ERR_UNSUPPORTED;
  return with_static_workspace(plan, [&](void* ws) {
    return vsa_forward(plan, q, k, v, gate, out, ws, VSA_STATIC_WORKSPACE_BYTES, stream);
  });
}

extern "C" vsa_status_t vsa_check_static_workspace(vsa_plan_t plan, void* stream) {
  if (!plan) return VSA_ERR_INVALID_ARG;
  return with_static_workspace(plan, [&](void* ws) { return vsa_check(plan, ws, stream); });
}

extern "C" vsa_status_t vsa_diag_wait_timeout_static(vsa_plan_t plan, int n_ctas, void* stream) {
  if (!plan) return VSA_ERR_INVALID_ARG;
  return with_static_workspace(plan, [&](void* ws) { return vsa_diag_wait_timeout(plan, ws, n_ctas, stream); });
}
