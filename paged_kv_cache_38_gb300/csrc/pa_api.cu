// pa_api.cu - the extern "C" entry points declared in include/pa.h.
//
// Each entry point validates its arguments on the host, enqueues its kernels on the caller's
// stream and returns; no call allocates, frees or synchronises.
#include <atomic>
#include <string>

#include "pa_internal.h"

namespace {

thread_local std::string g_last_error;

constexpr unsigned long long kDefaultWaitNs = 1000000000ull;  // one second
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_stall_cta{-1};

pa_status finish(pa_status st, const std::string& msg) {
  if (st != PA_OK) g_last_error = msg.empty() ? pa_status_string(st) : msg;
  return st;
}

}  // namespace

namespace pa {
pa_status record_error(pa_status st, const std::string& msg) { return finish(st, msg); }
unsigned long long launch_wait_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
int launch_stall_cta() { return g_stall_cta.load(std::memory_order_relaxed); }
}  // namespace pa

extern "C" {

const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK:
      return "PA_OK";
    case PA_EINVAL:
      return "PA_EINVAL: invalid argument";
    case PA_EUNSUPPORTED:
      return "PA_EUNSUPPORTED: combination not built";
    case PA_ECUDA:
      return "PA_ECUDA: CUDA runtime error";
    case PA_ENOSPACE:
      return "PA_ENOSPACE: host-side pool exhausted";
  }
  return "unknown pa_status";
}

const char* pa_last_error_message(void) { return g_last_error.c_str(); }

pa_status pa_testing_set_wait_limit(uint64_t wait_ns, int32_t stall_cta) {
  if (stall_cta < -1) return finish(PA_EINVAL, "stall_cta must be -1 or a CTA index");
  g_wait_ns.store(wait_ns == 0 ? kDefaultWaitNs : static_cast<unsigned long long>(wait_ns),
                  std::memory_order_relaxed);
  g_stall_cta.store(stall_cta, std::memory_order_relaxed);
  return PA_OK;
}

size_t pa_decode_workspace_size(const pa_decode_args* args) {
  std::string msg;
  if (args == nullptr) {
    finish(PA_EINVAL, "args is NULL");
    return 0;
  }
  pa::DecodePlan plan;
  pa_status st = pa::plan_decode(*args, pa::device_sm_count(), plan, msg);
  if (st != PA_OK) {
    finish(st, msg);
    return 0;
  }
  return plan.workspace;
}

pa_status pa_decode(const pa_decode_args* args, pa_stream stream) {
  std::string msg;
  if (args == nullptr) return finish(PA_EINVAL, "args is NULL");
  return finish(pa::run_decode(*args, reinterpret_cast<cudaStream_t>(stream), msg), msg);
}

pa_status pa_prefill(const pa_prefill_args* args, pa_stream stream) {
  std::string msg;
  if (args == nullptr) return finish(PA_EINVAL, "args is NULL");
  return finish(pa::run_prefill(*args, reinterpret_cast<cudaStream_t>(stream), msg), msg);
}

pa_status pa_write_kv(const void* k, const void* v, void* k_pool, void* v_pool,
                      const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int32_t num_blocks, pa_dtype kv_dtype,
                      int32_t* err_flag, pa_stream stream) {
  std::string msg;
  return finish(pa::run_write_kv(k, v, k_pool, v_pool, slot_mapping, num_tokens, num_kv_heads,
                                 head_dim, block_size, num_blocks, kv_dtype, err_flag,
                                 reinterpret_cast<cudaStream_t>(stream), msg),
                msg);
}

pa_status pa_write_kv_fp8(const void* k, const void* v, pa_dtype src_dtype, void* k_pool,
                          void* v_pool, const int64_t* slot_mapping, int32_t num_tokens,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, float k_scale, float v_scale, int32_t* err_flag,
                          pa_stream stream) {
  std::string msg;
  return finish(pa::run_write_kv_fp8(k, v, src_dtype, k_pool, v_pool, slot_mapping, num_tokens,
                                     num_kv_heads, head_dim, block_size, num_blocks, k_scale,
                                     v_scale, err_flag, reinterpret_cast<cudaStream_t>(stream),
                                     msg),
                msg);
}

pa_status pa_copy_blocks(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                         const int32_t* pairs, int32_t num_pairs, int32_t num_blocks,
                         size_t block_bytes, int32_t* err_flag, pa_stream stream) {
  std::string msg;
  return finish(pa::run_copy_blocks(k_pools, v_pools, num_layers, pairs, num_pairs, num_blocks,
                                    block_bytes, err_flag, reinterpret_cast<cudaStream_t>(stream),
                                    msg),
                msg);
}

pa_status pa_swap_blocks(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                         void* host_buf, const int32_t* block_ids, int32_t n, int32_t num_blocks,
                         size_t block_bytes, pa_swap_dir dir, void* staging, size_t staging_bytes,
                         pa_stream stream) {
  std::string msg;
  return finish(pa::run_swap_blocks(k_pools, v_pools, num_layers, host_buf, block_ids, n,
                                    num_blocks, block_bytes, dir, staging, staging_bytes,
                                    reinterpret_cast<cudaStream_t>(stream), msg),
                msg);
}

}  // extern "C"
