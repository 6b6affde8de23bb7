// pa_internal.h - host-side interfaces shared by the translation units of libpa.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <string>

#include "../../include/pa.h"

namespace pa {

struct DecodeParams;

// Sizes of one pa_decode launch, derived only from the arguments and the SM count.
struct DecodePlan {
  int elt = 2;             // bytes per KV element
  int regions = 1;         // 128-byte column regions per token row
  int stage_tokens = 16;   // tokens per pipeline stage (16, or 32 for 1-byte KV; <= 4 blocks)
  int stage_rows = 16;     // rows of one copy: min(block_size, stage_tokens)
  int region_stride = 0;   // bytes of one region of one copy inside a stage
  int stage_bytes = 0;     // bytes of K (or V) per stage
  int stages = 0;          // ring depth
  int split_tokens = 0;    // tokens per work item
  int max_splits = 1;
  int seqs_per_launch = 0; // sequences handled by one kernel launch
  int off_merge = 0, off_q = 0, off_bar = 0, off_meta = 0, off_items = 0, off_tbl = 0, off_scan = 0;
  int tbl_stride = 0;      // block-table entries per queued work item
  size_t smem_bytes = 0;   // dynamic shared memory per CTA
  size_t workspace = 0;    // bytes: 256 of work counters, then the split partials
  size_t partial_o_bytes = 0;
};

// Validate decode arguments (no device access; pointers only when check_pointers). On failure
// returns PA_EINVAL or PA_EUNSUPPORTED and fills msg.
pa_status check_decode_args(const pa_decode_args& a, bool check_pointers, std::string& msg);
pa_status plan_decode(const pa_decode_args& a, int sm_count, DecodePlan& plan, std::string& msg);
int device_sm_count();

// Kernel launchers per KV dtype (one translation unit each).
cudaError_t launch_decode_f16(int head_dim, int group, const CUtensorMap& kmap,
                              const CUtensorMap& vmap, const DecodeParams& p, dim3 grid,
                              size_t smem, cudaStream_t stream);
cudaError_t launch_decode_bf16(int head_dim, int group, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, const DecodeParams& p, dim3 grid,
                               size_t smem, cudaStream_t stream);
cudaError_t launch_decode_e4m3(int head_dim, int group, const CUtensorMap& kmap,
                               const CUtensorMap& vmap, const DecodeParams& p, dim3 grid,
                               size_t smem, cudaStream_t stream);

pa_status run_decode(const pa_decode_args& a, cudaStream_t stream, std::string& msg);

// Block movers.
pa_status run_write_kv(const void* k, const void* v, void* k_pool, void* v_pool,
                       const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t num_blocks, pa_dtype kv_dtype,
                       int32_t* err_flag, cudaStream_t stream, std::string& msg);
pa_status run_write_kv_fp8(const void* k, const void* v, pa_dtype src_dtype, void* k_pool,
                           void* v_pool, const int64_t* slot_mapping, int32_t num_tokens,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           int32_t num_blocks, float k_scale, float v_scale, int32_t* err_flag,
                           cudaStream_t stream, std::string& msg);
pa_status run_copy_blocks(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                          const int32_t* pairs, int32_t num_pairs, int32_t num_blocks,
                          size_t block_bytes, int32_t* err_flag, cudaStream_t stream,
                          std::string& msg);
pa_status run_swap_blocks(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                          void* host_buf, const int32_t* block_ids, int32_t n, int32_t num_blocks,
                          size_t block_bytes, pa_swap_dir dir, void* staging, size_t staging_bytes,
                          cudaStream_t stream, std::string& msg);

// A scheduler plan's moves: swap-outs ((GPU block, CPU slot) pairs), swap-ins ((CPU slot, GPU
// block) pairs), copy-on-write (src, dst) pairs, all in host memory, into launches in that order.
pa_status run_plan_moves(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                         int32_t num_blocks, size_t block_bytes, void* cpu_pool,
                         int32_t num_cpu_blocks, const int32_t* swap_out, int32_t num_swap_out,
                         const int32_t* swap_in, int32_t num_swap_in, const int32_t* copies,
                         int32_t num_copies, int32_t* err_flag, cudaStream_t stream,
                         std::string& msg);

// Records msg as the calling thread's last-error message and returns st.
pa_status run_prefill(const pa_prefill_args& a, cudaStream_t stream, std::string& msg);
pa_status encode_pool_rows_map(CUtensorMap* map, const void* pool, long long rows, int head_dim,
                               int elt, int box_rows, std::string& msg);
pa_status encode_query_tile_map(CUtensorMap* map, const void* q, int num_tokens, int num_q_heads,
                                int head_dim, int group, int tokens, std::string& msg);
pa_status record_error(pa_status st, const std::string& msg);

// Wait limit (ns) and stalled CTA (-1: none) for the next launches; see pa_testing_set_wait_limit.
unsigned long long launch_wait_ns();
int launch_stall_cta();

// Sets msg from a CUDA error and returns PA_ECUDA (or PA_OK for cudaSuccess).
pa_status cuda_status(cudaError_t e, const char* what, std::string& msg);

}  // namespace pa
