// pa_noalloc.cu - paged decode for callers that cannot allocate device memory.
//
// pa_decode needs a scratch buffer for the split-K partials and its work counters, and expects
// the caller to allocate it. Some callers cannot: code that runs where every allocation must be
// planned ahead (an inference runtime with a fixed memory arena, a plugin that only receives the
// tensors it works on, a real-time path that may not call the allocator). For them this file
// keeps one fixed scratch array in the library's own device memory. It is created when the
// library's device code is loaded on a GPU and lives until the process exits, on every GPU that
// loads the library.
#include <mutex>
#include <string>

#include "pa_internal.h"

namespace pa {
namespace {

// Scratch shared by every call of pa_decode_static_workspace on a device (16 MiB).
static __device__ __align__(256) unsigned char g_static_scratch[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
// Per device: the array's device address and the context it was looked up in. After a device
// reset (a new primary context) the module is loaded again and the array may sit elsewhere, so
// the address is looked up again whenever the current context differs.
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

pa_status current_context(CUcontext* ctx, std::string& msg) {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  });
  if (fn == nullptr) {
    msg = "cuCtxGetCurrent is not available from the driver";
    return PA_ECUDA;
  }
  *ctx = nullptr;
  if (fn(ctx) != CUDA_SUCCESS) {
    msg = "cuCtxGetCurrent failed";
    return PA_ECUDA;
  }
  return PA_OK;  // *ctx stays NULL while the thread has no current context yet
}

// Device address of g_static_scratch on the current device, looked up once per device and
// context. In host code the array's name only stands for the symbol, so the address must come
// from the runtime.
pa_status scratch_address(void** out, std::string& msg) {
  int dev = 0;
  pa_status st = cuda_status(cudaGetDevice(&dev), "cudaGetDevice", msg);
  if (st != PA_OK) return st;
  if (dev < 0 || dev >= kMaxDevices) {
    msg = "device ordinal beyond the static scratch table";
    return PA_EUNSUPPORTED;
  }
  CUcontext ctx = nullptr;
  st = current_context(&ctx, msg);
  if (st != PA_OK) return st;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr || ctx == nullptr || g_scratch_ctx[dev] != ctx) {
    void* ptr = nullptr;
    // (makes the device's primary context current first if the thread had none)
    st = cuda_status(cudaGetSymbolAddress(&ptr, g_static_scratch),
                     "cudaGetSymbolAddress of the static decode scratch", msg);
    if (st != PA_OK) return st;
    st = current_context(&ctx, msg);
    if (st != PA_OK) return st;
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_static_workspace(const pa_decode_args* args, pa_stream stream) {
  std::string msg;
  if (args == nullptr) return pa::record_error(PA_EINVAL, "args is NULL");
  pa::DecodePlan plan;
  pa_status st = pa::plan_decode(*args, pa::device_sm_count(), plan, msg);
  if (st != PA_OK) return pa::record_error(st, msg);
  if (plan.workspace > PA_STATIC_WORKSPACE_BYTES) {
    return pa::record_error(
        PA_EINVAL, "this decode needs " + std::to_string(plan.workspace) +
                       " bytes of scratch; the built-in buffer holds " +
                       std::to_string(static_cast<size_t>(PA_STATIC_WORKSPACE_BYTES)) +
                       " (raise split_tokens, or use pa_decode with a caller workspace)");
  }
  void* scratch = nullptr;
  st = pa::scratch_address(&scratch, msg);
  if (st != PA_OK) return pa::record_error(st, msg);
  pa_decode_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = PA_STATIC_WORKSPACE_BYTES;
  st = pa::run_decode(a, reinterpret_cast<cudaStream_t>(stream), msg);
  return st == PA_OK ? PA_OK : pa::record_error(st, msg);
}
