// pa_decode_host.cu - validation, launch planning and tensor maps for pa_decode.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

int log2i(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// The pool as a 2-D tensor [num_blocks*num_kv_heads*block_size rows][head_dim] with a box of
// one copy: `rows` token rows of one (block, kv head) tile x 128 bytes, 128-byte swizzle.
pa_status encode_pool_map(CUtensorMap* map, const void* pool, const pa_decode_args& a, int elt,
                          int box_rows, std::string& msg) {
  return encode_pool_rows_map(map, pool, static_cast<long long>(a.num_blocks) * a.num_kv_heads *
                                             a.block_size,
                              a.head_dim, elt, box_rows, msg);
}

}  // namespace

// The pool as a 2-D tensor [rows][head_dim] of elt-byte elements with a box of box_rows rows x
// 128 bytes, 128-byte swizzle (the shared-memory operand layout of the decode and prefill
// kernels).
pa_status encode_pool_rows_map(CUtensorMap* map, const void* pool, long long rows, int head_dim,
                               int elt, int box_rows, std::string& msg) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) {
    msg = "cuTensorMapEncodeTiled is not available from the driver";
    return PA_ECUDA;
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * elt};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elt), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, elt == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                   2, const_cast<void*>(pool), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    msg = "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(static_cast<int>(r));
    return PA_ECUDA;
  }
  return PA_OK;
}

// Queries [num_tokens][num_q_heads][head_dim] (16-bit) as a 3-D tensor {head_dim, num_q_heads,
// num_tokens} with a box of {64, group, tokens} and 128-byte swizzle: one box lands as
// tokens * group rows of 128 bytes, row t * group + h holding head h of token t, the layout of a
// 2-D box of as many rows (tokens past num_tokens read as zero).
pa_status encode_query_tile_map(CUtensorMap* map, const void* q, int num_tokens, int num_q_heads,
                                int head_dim, int group, int tokens, std::string& msg) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) {
    msg = "cuTensorMapEncodeTiled is not available from the driver";
    return PA_ECUDA;
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_q_heads),
                        static_cast<cuuint64_t>(num_tokens)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                           static_cast<cuuint64_t>(num_q_heads) * head_dim * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tokens)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    msg = "cuTensorMapEncodeTiled (queries) failed with CUresult " +
          std::to_string(static_cast<int>(r));
    return PA_ECUDA;
  }
  return PA_OK;
}

pa_status cuda_status(cudaError_t e, const char* what, std::string& msg) {
  if (e == cudaSuccess) return PA_OK;
  msg = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return PA_ECUDA;
}

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev] = n;
  return n;
}

pa_status check_decode_args(const pa_decode_args& a, bool check_pointers, std::string& msg) {
  if (a.num_seqs < 0 || a.num_q_heads <= 0 || a.num_kv_heads <= 0 || a.num_blocks <= 0 ||
      a.max_blocks_per_seq <= 0 || a.max_ctx_len < 0) {
    msg = "sizes must be positive (num_seqs and max_ctx_len may be 0)";
    return PA_EINVAL;
  }
  if (a.num_q_heads % a.num_kv_heads != 0) {
    msg = "num_q_heads must be a multiple of num_kv_heads";
    return PA_EINVAL;
  }
  const int group = a.num_q_heads / a.num_kv_heads;
  if (a.block_size != 4 && a.block_size != 8 && a.block_size != 16 && a.block_size != 32 &&
      a.block_size != 64) {
    msg = "block_size must be 4, 8, 16, 32 or 64";
    return PA_EINVAL;
  }
  if (a.head_dim != 64 && a.head_dim != 128) {
    msg = "head_dim must be 64 or 128";
    return PA_EINVAL;
  }
  if (a.q_dtype != PA_F16 && a.q_dtype != PA_BF16) {
    msg = "q_dtype must be PA_F16 or PA_BF16";
    return PA_EINVAL;
  }
  if (a.kv_dtype != PA_F16 && a.kv_dtype != PA_BF16 && a.kv_dtype != PA_FP8_E4M3) {
    msg = "unknown kv_dtype";
    return PA_EINVAL;
  }
  if (a.kv_dtype != PA_FP8_E4M3 && a.kv_dtype != a.q_dtype) {
    msg = "for 16-bit KV the query dtype must equal the KV dtype";
    return PA_EUNSUPPORTED;
  }
  if (a.kv_dtype == PA_FP8_E4M3 && a.head_dim != 128) {
    msg = "E4M3 KV is built for head_dim 128";
    return PA_EUNSUPPORTED;
  }
  if (!(group == 1 || group == 2 || group == 4 || group == 8 || group == 16)) {
    msg = "num_q_heads / num_kv_heads must be 1, 2, 4, 8 or 16";
    return PA_EUNSUPPORTED;
  }
  if (a.max_ctx_len > a.max_blocks_per_seq * a.block_size) {
    msg = "max_ctx_len exceeds max_blocks_per_seq * block_size";
    return PA_EINVAL;
  }
  const long long rows = static_cast<long long>(a.num_blocks) * a.num_kv_heads * a.block_size;
  if (rows >= (1ll << 31)) {
    msg = "pool has more than 2^31 token rows per kv head layout";
    return PA_EUNSUPPORTED;
  }
  if (a.num_seqs > 65535) {
    msg = "num_seqs must be <= 65535";
    return PA_EUNSUPPORTED;
  }
  if (check_pointers && a.num_seqs > 0) {
    if (!a.q || !a.k_pool || !a.v_pool || !a.block_tables || !a.ctx_lens || !a.out) {
      msg = "null pointer argument";
      return PA_EINVAL;
    }
    if (!aligned(a.q, 16) || !aligned(a.k_pool, 16) || !aligned(a.v_pool, 16) ||
        !aligned(a.out, 4) || !aligned(a.block_tables, 4) || !aligned(a.ctx_lens, 4)) {
      msg = "q, k_pool, v_pool must be 16-byte aligned; out, tables, ctx_lens 4-byte aligned";
      return PA_EINVAL;
    }
  }
  if (!(a.scale == a.scale) || !(a.k_scale == a.k_scale) || !(a.v_scale == a.v_scale)) {
    msg = "scale, k_scale and v_scale must not be NaN";
    return PA_EINVAL;
  }
  if (a.split_tokens < 0) {
    msg = "split_tokens must be >= 0";
    return PA_EINVAL;
  }
  return PA_OK;
}

pa_status plan_decode(const pa_decode_args& a, int sm_count, DecodePlan& pl, std::string& msg) {
  pa_status st = check_decode_args(a, false, msg);
  if (st != PA_OK) return st;
  const int B = a.block_size, D = a.head_dim;
  const int group = a.num_q_heads / a.num_kv_heads;
  pl.elt = a.kv_dtype == PA_FP8_E4M3 ? 1 : 2;
  pl.regions = D * pl.elt / 128;
  // 16 tokens per stage (32 for 1-byte KV, so a stage still moves 8 KiB per head pair of
  // K and V and the per-stage costs are paid half as often): up to 4 whole blocks when blocks
  // are smaller, one part of one block when they are larger. Each copy brings srows rows.
  pl.stage_tokens = std::min(pl.elt == 1 ? 32 : 16, 4 * B);
  pl.stage_rows = std::min(B, pl.stage_tokens);
  pl.region_stride = std::max(pl.stage_rows * 128, 1024);
  pl.stage_bytes = (pl.stage_tokens / pl.stage_rows) * pl.regions * pl.region_stride;

  const int stok = std::max(16, B);  // split granularity of the API
  if (a.split_tokens > 0) {
    if (a.split_tokens % stok != 0) {
      msg = "split_tokens must be a multiple of max(16, block_size)";
      return PA_EINVAL;
    }
    pl.split_tokens = a.split_tokens;
  } else {
    // 512-token work items for 16-bit KV, 2048 for 1-byte KV (its 32-token stages amortise the
    // per-item merge over more stages); fewer tokens when there would be too few items
    int tokens = pl.elt == 1 ? 2048 : 512;
    const long long units = static_cast<long long>(a.num_seqs) * a.num_kv_heads;
    const int sms = sm_count > 0 ? sm_count : 148;
    while (tokens > 4 * stok && units * ((a.max_ctx_len + tokens - 1) / tokens) < 8LL * sms)
      tokens /= 2;
    // a work item's table slice holds at most kMaxItemUnits copy units (small blocks of a
    // 1-byte cache would exceed it at 2048 tokens)
    while (tokens > stok && tokens / pl.stage_rows + 1 > kMaxItemUnits) tokens /= 2;
    pl.split_tokens = std::max(stok, (tokens / stok) * stok);
  }
  pl.max_splits = std::max(1, (a.max_ctx_len + pl.split_tokens - 1) / pl.split_tokens);
  pl.seqs_per_launch = std::max(1, std::min(a.num_seqs, kMaxSeqsPerLaunch));

  // shared memory: [ring][merge][queries][barriers][stage meta][items + flag][tables][scan]
  const int tbl_entries = pl.split_tokens / pl.stage_rows + 1;  // copy units of one work item
  if (tbl_entries > kMaxItemUnits) {
    msg = "split_tokens / min(block_size, stage tokens) must be below 256";
    return PA_EINVAL;
  }
  auto up = [](size_t x, size_t al) { return (x + al - 1) / al * al; };
  const size_t merge = static_cast<size_t>(kConsumerWarps) * group * D * 4 +
                       static_cast<size_t>(kConsumerWarps) * group * 8;
  const size_t qbytes = static_cast<size_t>(kItemSlots) * group * D * 2;
  const size_t bars = (2 * kMaxStages + 3 * kItemSlots + 1) * 8;
  const size_t meta = kMaxStages * 4;
  const size_t items = kItemSlots * sizeof(ItemDesc) + 16;
  pl.tbl_stride = ((tbl_entries + 3) / 4) * 4;
  const size_t tbls = static_cast<size_t>(kItemSlots) * pl.tbl_stride * 4;
  const size_t scan = scan_ints(static_cast<size_t>(pl.seqs_per_launch)) * 4;
  const size_t fixed = up(merge, 16) + up(qbytes, 128) + bars + meta + items + tbls + up(scan, 16);
  const size_t limit = 227 * 1024 - 1024;  // opt-in maximum per CTA, minus alignment slack
  if (fixed + 2 * static_cast<size_t>(pl.stage_bytes) * 8 > limit) {
    msg = "shared-memory budget exceeded (too many sequences per launch for this group size)";
    return PA_EUNSUPPORTED;
  }
  // The ring depth must be a multiple of the consumer and producer warp counts: two tiles that
  // share a stage then always belong to the same consumer warp and the same producer warp, which
  // handle them in order, so no mbarrier parity wait can see an older phase of the stage.
  static_assert(kConsumerWarps % kProducerWarps == 0, "ring depth rule");
  size_t depth = std::min<size_t>(kMaxStages, (limit - fixed) / (2 * pl.stage_bytes));
  depth = (depth / kConsumerWarps) * kConsumerWarps;
  pl.stages = static_cast<int>(depth);
  size_t off = static_cast<size_t>(pl.stages) * 2 * pl.stage_bytes;
  pl.off_merge = static_cast<int>(off);
  off = up(off + merge, 128);
  pl.off_q = static_cast<int>(off);
  off = up(off + qbytes, 16);
  pl.off_bar = static_cast<int>(off);
  off += bars;
  pl.off_meta = static_cast<int>(off);
  off += meta;
  pl.off_items = static_cast<int>(off);
  off += items;
  pl.off_tbl = static_cast<int>(off);
  off += tbls;
  pl.off_scan = static_cast<int>(off);
  off += scan;
  pl.smem_bytes = 1024 + off;

  const size_t slots = static_cast<size_t>(pl.seqs_per_launch) * a.num_q_heads * pl.max_splits;
  pl.partial_o_bytes = pl.max_splits > 1 ? up(slots * D * 4, 256) : 0;
  pl.workspace = 256 + (pl.max_splits > 1 ? pl.partial_o_bytes + slots * 8 : 0);
  return PA_OK;
}

pa_status run_decode(const pa_decode_args& a, cudaStream_t stream, std::string& msg) {
  static std::atomic<uint32_t> launch_counter{1};
  DecodePlan pl;
  pa_status st = check_decode_args(a, true, msg);
  if (st != PA_OK) return st;
  const int sms = device_sm_count();
  st = plan_decode(a, sms, pl, msg);
  if (st != PA_OK) return st;
  if (a.workspace == nullptr || a.workspace_bytes < pl.workspace) {
    msg = "workspace smaller than pa_decode_workspace_size()";
    return PA_EINVAL;
  }
  if (!aligned(a.workspace, 256)) {
    msg = "workspace must be 256-byte aligned";
    return PA_EINVAL;
  }
  if (a.num_seqs == 0) return PA_OK;

  CUtensorMap kmap, vmap;
  st = encode_pool_map(&kmap, a.k_pool, a, pl.elt, pl.stage_rows, msg);
  if (st != PA_OK) return st;
  st = encode_pool_map(&vmap, a.v_pool, a, pl.elt, pl.stage_rows, msg);
  if (st != PA_OK) return st;

  DecodeParams p{};
  char* ws = static_cast<char*>(a.workspace);
  p.counters = reinterpret_cast<unsigned long long*>(ws);
  char* parts = ws + 256;
  p.part_o = pl.max_splits > 1 ? reinterpret_cast<float*>(parts) : nullptr;
  p.part_ml = pl.max_splits > 1 ? reinterpret_cast<float2*>(parts + pl.partial_o_bytes) : nullptr;
  p.err = a.err_flag;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.block_size = a.block_size;
  p.log2_block = log2i(a.block_size);
  p.log2_srows = log2i(pl.stage_rows);
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks_per_seq;
  p.max_ctx = a.max_ctx_len;
  p.split_tokens = pl.split_tokens;
  p.max_splits = pl.max_splits;
  p.stages = pl.stages;
  p.region_stride = pl.region_stride;
  p.stage_bytes = pl.stage_bytes;
  p.stage_tokens = pl.stage_tokens;
  p.off_merge = pl.off_merge;
  p.off_q = pl.off_q;
  p.off_bar = pl.off_bar;
  p.off_meta = pl.off_meta;
  p.off_items = pl.off_items;
  p.off_tbl = pl.off_tbl;
  p.tbl_stride = pl.tbl_stride;
  p.off_scan = pl.off_scan;
  p.score_scale = a.scale * a.k_scale * kLog2e;
  p.v_scale = a.v_scale;
  p.q_bf16 = a.q_dtype == PA_BF16 ? 1 : 0;
  p.wait_ns = launch_wait_ns();
  p.stall_cta = launch_stall_cta();

  const int group = a.num_q_heads / a.num_kv_heads;
  const int elt_q = 2;
  const dim3 grid(std::max(1, sms));
  for (int s0 = 0; s0 < a.num_seqs; s0 += pl.seqs_per_launch) {
    const int n = std::min(pl.seqs_per_launch, a.num_seqs - s0);
    const size_t row = static_cast<size_t>(s0) * a.num_q_heads * a.head_dim * elt_q;
    p.q = static_cast<const char*>(a.q) + row;
    p.out = static_cast<char*>(a.out) + row;
    p.block_tables = a.block_tables + static_cast<size_t>(s0) * a.max_blocks_per_seq;
    p.ctx_lens = a.ctx_lens + s0;
    p.num_seqs = n;
    p.launch_id = launch_counter.fetch_add(1);
    if (p.launch_id == 0) p.launch_id = launch_counter.fetch_add(1);
    cudaError_t e;
    switch (a.kv_dtype) {
      case PA_F16:
        e = launch_decode_f16(a.head_dim, group, kmap, vmap, p, grid, pl.smem_bytes, stream);
        break;
      case PA_BF16:
        e = launch_decode_bf16(a.head_dim, group, kmap, vmap, p, grid, pl.smem_bytes, stream);
        break;
      default:
        e = launch_decode_e4m3(a.head_dim, group, kmap, vmap, p, grid, pl.smem_bytes, stream);
        break;
    }
    st = cuda_status(e, "pa_decode kernel launch", msg);
    if (st != PA_OK) return st;
  }
  return PA_OK;
}

}  // namespace pa
