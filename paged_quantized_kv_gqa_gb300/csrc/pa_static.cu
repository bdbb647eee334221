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
//     stream capture; the address is kept together with the id of the CUDA
//     context it belongs to, and looked up again when the current context is
//     a different one (after cudaDeviceReset the module is loaded anew);
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
struct StaticSlot {
  unsigned long long ctx_id;   // context the address belongs to (0: none yet)
  void* ptr;
};
StaticSlot g_static[kMaxDevices] = {};

// Driver entry points for the current context's id (the runtime exposes none).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

bool current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_static_ws on the current device and context (looked up
// once per device and context).
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
  // initialises the device's primary context if nothing is current yet
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) {
    set_error(std::string("pa_run_static: context: ") + cudaGetErrorString(e));
    return PA_ERR_CUDA;
  }
  unsigned long long ctx = 0;
  if (!current_context_id(&ctx)) {
    set_error("pa_run_static: cannot read the current CUDA context's id");
    return PA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static[dev].ptr == nullptr || g_static[dev].ctx_id != ctx) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_static_ws);
    if (e != cudaSuccess || ptr == nullptr) {
      set_error(std::string("pa_run_static: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
      return PA_ERR_CUDA;
    }
    g_static[dev].ptr = ptr;
    g_static[dev].ctx_id = ctx;
  }
  *out = g_static[dev].ptr;
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
