/*
 * pa.h - C ABI of the paged KV-cache hot path for NVIDIA GB300 (sm_103a).
 *
 * The operations follow the PagedAttention serving scheme:
 *   - "Efficient Memory Management for Large Language Model Serving with PagedAttention"
 *     (paper summary page), paragraphs on the PagedAttention kernel, the block table,
 *     copy-on-write sharing and all-or-nothing preemption;
 *   - "When KV Capacity Runs Out: Pausing and Resuming Requests", Figures 1, 2 and 4;
 *   - "KV Cache Preemption in vLLM", section "Swap versus recompute";
 *   - "41 · Preemption, Recomputation & KV Pressure", section 3 (swap).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * Memory.    Every buffer is owned by the caller. Pointers documented as "device" must be
 *            device memory of the current CUDA device; "host" pointers are ordinary host
 *            memory read synchronously during the call; "pinned host" pointers must come
 *            from cudaHostAlloc / cudaHostRegister (e.g. torch pin_memory()). The library
 *            allocates and frees nothing.
 * Ordering.  Every call only enqueues work on `stream` (a cudaStream_t; NULL = legacy
 *            default stream) and returns; nothing blocks on the device. Results are
 *            visible to later work on the same stream.
 * Errors.    Host-side validation failures return PA_EINVAL (bad pointer, size, alignment,
 *            layout) or PA_EUNSUPPORTED (a valid combination this build has no kernel for)
 *            and enqueue nothing. A failed launch returns PA_ECUDA. pa_last_error_message()
 *            describes the latest non-OK status of the calling thread.
 *            Indices that live in device memory (block tables, slot mappings, copy pairs,
 *            context lengths) are checked on the device: a bad index is skipped and the
 *            matching PA_ERR_* bit is OR-ed into *err_flag (a device int32, may be NULL).
 *            No kernel traps. Every bounded wait inside a kernel gives up after about one
 *            second and sets PA_ERR_TIMEOUT.
 *
 * KV pool layout (one pool per layer, one for K and one for V):
 *     pool[num_blocks][num_kv_heads][block_size][head_dim]   elements of kv_dtype
 * so the keys of one (physical block, kv head) pair are one contiguous run of
 * block_size * head_dim * elt bytes. Logical position t of a sequence lives in logical
 * block t / block_size at slot t % block_size (0-indexed), i.e. physical block
 * block_tables[seq][t / block_size].
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* pa_stream; /* identical to cudaStream_t */

typedef enum {
  PA_OK = 0,
  PA_EINVAL = 1,        /* invalid argument; nothing was enqueued */
  PA_EUNSUPPORTED = 2,  /* valid but not built: dtype / head_dim / group combination */
  PA_ECUDA = 3,         /* a CUDA runtime call or launch failed */
  PA_ENOSPACE = 4       /* a host-side pool ran out (a scheduler's CPU swap slots) */
} pa_status;

typedef enum {
  PA_F16 = 0,       /* IEEE binary16 */
  PA_BF16 = 1,      /* bfloat16 */
  PA_FP8_E4M3 = 2   /* OCP FP8 E4M3 (raw bytes), dequantised with a per-tensor fp32 scale */
} pa_dtype;

typedef enum {
  PA_SWAP_OUT = 0,  /* device pool blocks -> pinned host buffer */
  PA_SWAP_IN = 1    /* pinned host buffer -> device pool blocks */
} pa_swap_dir;

/* Bits OR-ed into the optional device error flag. */
#define PA_ERR_BLOCK_ID 1 /* block table entry, slot or pair outside [0, num_blocks) */
#define PA_ERR_CTX_LEN 2  /* ctx_len < 0, > max_ctx_len or > max_blocks_per_seq*block_size;
                              prefill: a chunk longer than its ctx_len or than max_q_len
                              (rounded up to whole query tiles) */
#define PA_ERR_TIMEOUT 4  /* a bounded wait inside a kernel expired */

/*
 * pa_decode - single-token decode attention over a paged KV pool.
 *
 * Source: PagedAttention summary page, paragraph on the PagedAttention kernel (block K_j holds
 * the keys of tokens (j-1)B+1..jB, the kernel fetches each block wherever it is stored and the
 * result is identical to ordinary attention) and paragraph on the block table (logical blocks
 * filled left to right, a filled-slot count per sequence).
 *
 * For sequence s with L = ctx_lens[s] and query head h (group g = h / (num_q_heads/num_kv_heads)):
 *     K^[t] = k_pool[block_tables[s][t / B]][g][t % B][:] * k_scale      (t < L)
 *     V^[t] = v_pool[...same...] * v_scale
 *     s_t   = scale * <q[s][h], K^[t]>
 *     out[s][h] = sum_t softmax(s)_t * V^[t]
 * L includes the token written by pa_write_kv in the same step. L == 0 gives a zero row.
 * Slots at positions >= L and block-table entries beyond ceil(L/B) are never read, so freed
 * or unwritten slots may hold any bytes (including NaN patterns).
 *
 * Layouts (all device, contiguous, row-major):
 *   q            [num_seqs][num_q_heads][head_dim]          q_dtype (PA_F16 or PA_BF16)
 *   k_pool/v_pool [num_blocks][num_kv_heads][block_size][head_dim]   kv_dtype, 16-byte aligned
 *   block_tables [num_seqs][max_blocks_per_seq]              int32 physical block ids
 *   ctx_lens     [num_seqs]                                  int32
 *   out          [num_seqs][num_q_heads][head_dim]           q_dtype
 *   workspace    >= pa_decode_workspace_size(args) bytes, 256-byte aligned, contents ignored
 * Supported: head_dim in {64, 128}; block_size in {4, 8, 16, 32, 64}; group size
 * num_q_heads/num_kv_heads in {1, 2, 4, 8, 16}; (q, kv) dtype pairs (F16, F16), (BF16, BF16),
 * (F16, FP8_E4M3), (BF16, FP8_E4M3), the E4M3 pairs at head_dim 128 only (PA_EUNSUPPORTED
 * otherwise). k_scale / v_scale multiply the stored values (use 1.0
 * for 16-bit KV). Work is split along the context ("split-K") when that improves occupancy;
 * split_tokens = 0 lets the library choose, otherwise it must be a multiple of max(16, B) and
 * split_tokens / min(B, 16) (min(B, 32) for an E4M3 cache) must be below 256 (PA_EINVAL
 * otherwise).
 */
typedef struct pa_decode_args {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  const int32_t* ctx_lens;
  void* out;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t max_ctx_len;   /* host-known upper bound of ctx_lens; plans the split-K grid */
  int32_t split_tokens;  /* 0 = automatic */
  pa_dtype q_dtype;
  pa_dtype kv_dtype;
  float scale;           /* softmax scale, usually 1/sqrt(head_dim) */
  float k_scale;         /* per-tensor dequantisation scale of K (1.0 for 16-bit KV) */
  float v_scale;         /* per-tensor dequantisation scale of V (1.0 for 16-bit KV) */
  void* workspace;       /* device scratch for split-K partials; may be NULL if size is 0 */
  size_t workspace_bytes;
  int32_t* err_flag;     /* device int32 or NULL */
} pa_decode_args;

/* Bytes of device workspace pa_decode needs for these arguments (0 when no split is used).
 * Depends only on the sizes in args and on the current device's SM count. Returns 0 and sets
 * the last-error message if the arguments are invalid. */
size_t pa_decode_workspace_size(const pa_decode_args* args);

/* Enqueue the decode described by args on stream. */
pa_status pa_decode(const pa_decode_args* args, pa_stream stream);

/*
 * pa_prefill - causal attention of chunks of new tokens over the paged KV pool (prompt
 * processing, recomputation of a preempted request, chunked prefill).
 *
 * Source: PagedAttention summary page, paragraph on the two phases (the prompt phase processes
 * all prompt tokens at once, matrix-matrix work that builds their KV cache); "When KV Capacity
 * Runs Out", Figure 3 (a recomputed request feeds all its retained tokens together); the block
 * table as in pa_decode. Sequence s holds L = ctx_lens[s] positions, including its chunk's own
 * K/V (written first with pa_write_kv); its chunk is the n = q_starts[s + 1] - q_starts[s] query
 * rows q_starts[s] .. q_starts[s + 1] - 1, query i standing at position L - n + i. For query
 * head h (group g = h / (num_q_heads / num_kv_heads)):
 *     out[q_starts[s] + i][h] = sum_{t <= L - n + i} softmax_t(scale * <q, K^[t]>) V^[t]
 * computed on the tensor cores (tcgen05.mma, fp32 accumulation in tensor memory).
 *   q, out        device [num_tokens][num_q_heads][head_dim], dtype, 16-byte aligned
 *   q_starts      device int32 [num_seqs + 1], non-decreasing, q_starts[num_seqs] = num_tokens
 *   max_q_len     host upper bound of the chunk lengths (sizes the work: query tiles of
 *                 128 / G tokens per (sequence, kv head))
 * A sequence with n > L, L > max_blocks_per_seq * block_size or n above max_q_len rounded up to
 * whole query tiles sets PA_ERR_CTX_LEN and its rows are zero (past that bound they are not
 * written); an out-of-pool block id sets PA_ERR_BLOCK_ID (those rows are then unspecified).
 * Supported: dtype PA_F16 or PA_BF16 (q and out); kv_dtype equal to dtype, or PA_FP8_E4M3
 * for an FP8 cache ("KV Cache Preemption in vLLM", section "How much KV cache a token costs":
 * one byte per element), read as K^ = k_scale * value, V^ = v_scale * value (k_scale, v_scale
 * finite and > 0; head_dim 128), so that a recomputed request of an FP8 cache is prefilled over
 * the bytes its decode steps read; head_dim 64 or 128; block_size 8, 16, 32 or 64; group size
 * 1, 2, 4, 8 or 16. A caller that zero-initialises the struct must set kv_dtype.
 * The kernel is persistent (two CTAs per SM). With work_counter set, the call zeroes that int32
 * on the stream and the CTAs take work items from it: the 4 longest query tiles of every
 * (sequence, kv head), then the next 4, and so on; NULL assigns the same items round-robin.
 * The counter must not be shared by calls that can run at the same time.
 */
typedef struct {
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  const int32_t* ctx_lens;
  const int32_t* q_starts;
  void* out;
  int32_t num_seqs;
  int32_t num_tokens;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t max_q_len;
  pa_dtype dtype;
  float scale;
  int32_t* err_flag;     /* device int32 or NULL */
  int32_t* work_counter; /* device int32 or NULL, see above */
  pa_dtype kv_dtype;     /* the pools' element type: dtype, or PA_FP8_E4M3 (see above) */
  float k_scale;         /* E4M3 cache: K^ = k_scale * stored value (ignored otherwise) */
  float v_scale;         /* E4M3 cache: V^ = v_scale * stored value (ignored otherwise) */
} pa_prefill_args;

pa_status pa_prefill(const pa_prefill_args* args, pa_stream stream);

/*
 * pa_write_kv - store each new token's key and value in its slot.
 *
 * Source: "When KV Capacity Runs Out", section "Pause requests and release KV blocks"
 * (Figure 2: the KV of position 8 is written into the first slot of the block just linked
 * into A's block table) and section "Running out of KV space during generation" (each processed
 * input adds KV). For every token t with sigma = slot_mapping[t] >= 0 and every kv head h:
 *     k_pool[sigma / block_size][h][sigma % block_size][:] = k[t][h][:]     (same for v)
 * as a raw element copy in kv_dtype (fp8 bytes are copied, not re-quantised). sigma < 0 marks
 * a padding token and is skipped; sigma >= num_blocks*block_size sets PA_ERR_BLOCK_ID.
 * Two tokens with the same slot leave either token's data.
 *   k, v          device [num_tokens][num_kv_heads][head_dim], kv_dtype, 16-byte aligned
 *   k_pool,v_pool device pool layout above
 *   slot_mapping  device int64 [num_tokens]
 */
pa_status pa_write_kv(const void* k, const void* v, void* k_pool, void* v_pool,
                      const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int32_t num_blocks, pa_dtype kv_dtype,
                      int32_t* err_flag, pa_stream stream);

/*
 * pa_write_kv_fp8 - store each new token's key and value, given in f16 or bf16, in an E4M3
 * pool (quantise on write).
 *
 * Source: "KV Cache Preemption in vLLM: Swap, Recompute and Behavior Under Memory Pressure",
 * section "How much KV cache a token costs" (an FP8 cache stores one byte per element, half of
 * FP16) and section "What to do next" (switch the cache to FP8); slots as in pa_write_kv. For
 * every token t with sigma = slot_mapping[t] >= 0, kv head h and element d:
 *     k_pool[sigma / block_size][h][sigma % block_size][d] = E4M3(k[t][h][d] * (1 / k_scale))
 * (same for v with v_scale), where 1 / k_scale and the product are rounded to nearest binary32
 * (the pages give no rounding for this step; this is the usual form) and E4M3(x) is the nearest
 * OCP E4M3 code, ties to the even code, magnitudes at or beyond 448 (infinities included)
 * saturating to +-448, NaN giving a NaN code. pa_decode with the same k_scale / v_scale
 * dequantises code * scale. Bad or padding slots as in pa_write_kv.
 *   k, v          device [num_tokens][num_kv_heads][head_dim], src_dtype (PA_F16 or PA_BF16),
 *                 16-byte aligned
 *   k_pool,v_pool device E4M3 pools, layout above, 16-byte aligned
 *   k_scale,v_scale  finite and > 0 (PA_EINVAL otherwise); head_dim a multiple of 16
 */
pa_status pa_write_kv_fp8(const void* k, const void* v, pa_dtype src_dtype, void* k_pool,
                          void* v_pool, const int64_t* slot_mapping, int32_t num_tokens,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_blocks, float k_scale, float v_scale, int32_t* err_flag,
                          pa_stream stream);

/*
 * pa_copy_blocks - copy-on-write duplication of whole physical blocks.
 *
 * Source: PagedAttention summary page, paragraph on sharing (a sample that must write into a
 * shared block receives its own copy, as when a process forks) and paragraph on shared
 * prefixes (the last prefix block is copy-on-write). For every pair p, every layer l and both
 * pools:  pool_l[pairs[p][1]] = pool_l[pairs[p][0]]  (block_bytes bytes; source unchanged).
 * All pairs form one parallel step: no destination may equal a source or another destination
 * of the same call (results are unspecified otherwise).
 *   k_pools, v_pools  HOST arrays of num_layers device pointers (one pool per layer),
 *                     each 16-byte aligned; num_layers <= 256
 *   pairs             device int32 [num_pairs][2] = (src, dst) physical block ids
 *   block_bytes       num_kv_heads * block_size * head_dim * elt; a multiple of 16
 * Ids outside [0, num_blocks) set PA_ERR_BLOCK_ID and that pair is skipped.
 */
pa_status pa_copy_blocks(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                         const int32_t* pairs, int32_t num_pairs, int32_t num_blocks,
                         size_t block_bytes, int32_t* err_flag, pa_stream stream);

/*
 * pa_swap_blocks - move a preempted sequence's whole block set to pinned host memory and back.
 *
 * Source: "When KV Capacity Runs Out", section "Restore KV stored outside the GPU" (Figure 4:
 * the KV is copied to CPU memory, the GPU blocks are released only after the copy finished,
 * and it is later restored into blocks that may sit elsewhere); PagedAttention summary page,
 * paragraph on all-or-nothing eviction; "KV Cache Preemption in vLLM", section "Swap versus
 * recompute" (pinned memory; a block's data is spread over every layer).
 *   PA_SWAP_OUT:  host_buf[i][l][0][:] = k_pools[l][block_ids[i]][...]
 *                 host_buf[i][l][1][:] = v_pools[l][block_ids[i]][...]
 *   PA_SWAP_IN:   the reverse assignment.
 *   host_buf   pinned host, [n][num_layers][2][block_bytes] bytes, 16-byte aligned
 *   block_ids  HOST int32 [n], each in [0, num_blocks) (checked on the host), no duplicates
 *              for PA_SWAP_IN
 *   staging    optional device buffer of >= n*num_layers*2*block_bytes bytes. NULL: the kernel
 *              reads/writes the pinned buffer directly through its mapped device address.
 *              Non-NULL: a gather/scatter kernel packs blocks into staging and one bulk
 *              cudaMemcpyAsync crosses the host link.
 * The caller must not reuse the blocks (swap-out) or the host buffer (swap-in) until the
 * stream has passed this call.
 */
pa_status pa_swap_blocks(void* const* k_pools, void* const* v_pools, int32_t num_layers,
                         void* host_buf, const int32_t* block_ids, int32_t n, int32_t num_blocks,
                         size_t block_bytes, pa_swap_dir dir, void* staging, size_t staging_bytes,
                         pa_stream stream);

/*
 * pa_decode_static_workspace - pa_decode for callers that cannot allocate device memory.
 *
 * The pages have no counterpart: this is a convenience of this library. Some callers cannot call
 * cudaMalloc or any allocator -- an inference runtime whose device memory is one arena planned
 * ahead of time, a plugin that is handed only the tensors it works on, a latency-critical path
 * where an allocation could block. This call takes the same arguments as pa_decode but ignores
 * args->workspace and args->workspace_bytes: the split-K partials and work counters live in a
 * scratch array of PA_STATIC_WORKSPACE_BYTES inside the library's own device memory. That array
 * exists on every GPU that loads the library, from load until the process exits.
 *   - It allocates nothing. A decode whose pa_decode_workspace_size() exceeds
 *     PA_STATIC_WORKSPACE_BYTES is rejected with PA_EINVAL (raise split_tokens, or use
 *     pa_decode with a workspace of your own).
 *   - The first call on a device looks up the array's device address (once per device and
 *     CUDA context: again after a device reset); make that first call before any stream
 *     capture.
 *   - Every call on a device shares the one array, which keeps whatever the last call left in
 *     it (the kernel needs no zeroed scratch). Calls that may overlap on the GPU -- on different
 *     streams, or from different host threads -- race on it and must be serialised by the caller.
 */
#define PA_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)
pa_status pa_decode_static_workspace(const pa_decode_args* args, pa_stream stream);

/*
 * pa_testing_set_wait_limit - make the kernels' bounded waits run out (tests only).
 *
 * Not an operation of the pages: it exists so that tests can show that a kernel gives up
 * cleanly. Every wait of one warp, role or CTA on another inside pa_decode and pa_prefill is
 * bounded; when it expires the kernel sets PA_ERR_TIMEOUT, waits for its own copies and tensor
 * core operations still in flight, frees its tensor memory, leaves pa_decode's work counters
 * cleared for the next launch and returns (the outputs of that call are unspecified).
 *   wait_ns    limit of those waits in nanoseconds for launches enqueued from now on;
 *              0 restores the default of one second. Waits for a kernel's own copies keep
 *              their one-second limit.
 *   stall_cta  -1: no effect. Otherwise the CTA with this index withholds its part, so that
 *              the others' waits on it must run out: in pa_decode it does not arrive at the
 *              grid-wide barrier before the split-K combine (only launches with more than one
 *              split reach that barrier); in pa_prefill its MMA issuer stops after its first
 *              S = Q K^T group.
 * The setting is process-wide, is read when a call is enqueued (a captured CUDA graph keeps
 * the setting it was captured with) and is not thread-safe with respect to concurrent calls.
 */
pa_status pa_testing_set_wait_limit(uint64_t wait_ns, int32_t stall_cta);

/* Static description of a status code. */
const char* pa_status_string(pa_status status);

/* Detail for the latest non-OK status returned on the calling thread ("" if none). */
const char* pa_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
