// pa_static.cu - pa_run_static: the attention path without any device allocation.
//
// Some callers cannot call cudaMalloc: a plugin hosted by an inference server
// that owns every device allocation through its own pool, code running inside
// a real-time loop where an allocation may block or fail, or an embedding with
// a fixed device-memory budget.  For them the library carries one fixed
// scratch buffer, g_static_ws below, and pa_run_static uses it as the
// workspace (plan arrays, status word and split-KV partial states).  The
// caller still passes its own inputs and outputs in pa_args.
//
// Properties a caller must know:
//   - the buffer is kStaticWorkspaceBytes (32 MiB) per device; every GPU on
//     which the library's kernels are loaded holds it until the process exits;
//     plans whose workspace is larger are rejected with PA_ERR_INVALID_ARG;
//   - the device address of the buffer is looked up once per device
//     (cudaGetSymbolAddress, with that device current) by the first
//     pa_run_static call on that device, so make that first call before any
//     stream capture;
//   - all calls share the one buffer and it keeps the last call's contents:
//     calls whose work may overlap on the GPU (different streams, or several
//     host threads) race with each other; serialise them;
//   - the status word is cleared on every call; the partial states need no
//     clearing (the attention writes every slot the merge reads).
#include <mutex>
#include <string>

#include "pa_internal.h"

namespace pa {
namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_ws[kStaticWorkspaceBytes];

std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_ws on the current device (looked up once).
pa_status static_workspace(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error(std::string("pa_run_static: cudaGetDevice: ") + cudaGetErrorString(e));
    return PA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("pa_run_static: device index out of range");
    return PA_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_ws);
    if (e != cudaSuccess || ptr == nullptr) {
      set_error(std::string("pa_run_static: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      return PA_ERR_CUDA;
    }
    g_static_ptr[dev] = ptr;
  }
  *out = g_static_ptr[dev];
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_run_static(const pa_plan_t* plan, const pa_args* args, void* stream,
                                   int32_t check) {
  if (!plan || !args) {
    pa::set_error("pa_run_static: null plan or args");
    return PA_ERR_INVALID_ARG;
  }
  const size_t need = pa_workspace_size(plan);
  if (need > pa::kStaticWorkspaceBytes) {
    pa::set_error("pa_run_static: this plan needs a " + std::to_string(need) +
                  "-byte workspace but the built-in buffer holds " +
                  std::to_string(pa::kStaticWorkspaceBytes) +
                  " bytes; use pa_run with a caller-provided workspace");
    return PA_ERR_INVALID_ARG;
  }
  void* ws = nullptr;
  pa_status s = pa::static_workspace(&ws);
  if (s != PA_OK) return s;
  s = pa_plan_upload(plan, ws, stream);  // also clears the status word
  if (s != PA_OK) return s;
  s = pa_run(plan, args, ws, stream);
  if (s != PA_OK) return s;
  s = pa_merge(plan, args, ws, stream);
  if (s != PA_OK) return s;
  if (check) return pa_check(plan, ws, stream, nullptr);
  return PA_OK;
}
