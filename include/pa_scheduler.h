/*
 * pa_scheduler.h - host-side scheduler and KV block manager for the paged KV cache.
 *
 * It plans, step by step, what the kernels of pa.h do: which sequences run, their block
 * tables and context lengths, the slot of every KV position written, the copy-on-write pairs
 * and the blocks swapped to and from CPU memory. Planning uses host memory only and makes no
 * CUDA call; pa_scheduler_execute_moves enqueues a plan's block moves on the GPU.
 *
 * Sources:
 *   "When KV Capacity Runs Out: Pausing and Resuming Requests", Figures 1-5: a block is linked
 *   only when the last one is full; when none is free a running request is paused and its
 *   blocks released (not zeroed) for the request that needs one; a paused request resumes by
 *   recomputing its KV from its retained tokens (Figure 3) or by restoring KV kept in CPU
 *   memory into possibly different blocks and then processing its pending token (Figure 4).
 *   PagedAttention summary page: block tables fill logical blocks left to right and count
 *   filled slots; samples of one prompt share its blocks through a reference count; a write
 *   into a shared block first gets its own copy (copy-on-write); blocks whose count drops to
 *   zero are freed; with first-come-first-served scheduling the latest requests are preempted,
 *   all blocks of a sequence group at once.
 *   "Continuous Batching and PagedAttention", section "The scheduler loop, written out":
 *   retire, admit while memory permits, evict the newest while a running sequence cannot grow
 *   (back to the front of the waiting queue), then one step for every running sequence.
 *
 * Policy of one pa_scheduler_step (the readings where the sources leave a choice):
 *   1. retire groups whose samples have each produced max_new_tokens; free their blocks;
 *   2. while the blocks the running sequences need to grow by one token exceed the free ones,
 *      preempt the running group that arrived last. A sequence needs a block when its last
 *      block is full or shared (reference count > 1). A single-sequence group in
 *      PA_PREEMPT_RECOMPUTE mode releases its blocks; any other group is swapped: its distinct
 *      blocks are assigned CPU slots (in order of first appearance) and released;
 *   3. only if nothing was preempted: admit waiting groups in queue order (preempted groups
 *      go back to the front) while the group fits in max_running_seqs and its blocks fit
 *      beside the running sequences' growth; the first that does not fit stops admission.
 *      A new group writes its prompt once into ceil(prompt / B) blocks shared by its samples;
 *      a recomputed sequence rewrites positions [0, L + 1) into fresh blocks; a swapped group
 *      gets fresh GPU blocks for its CPU slots, in the same order;
 *   4. every running sequence that was not just prefilled or recomputed appends one token:
 *      a fresh block if its last block is full, a copy-on-write if it is shared.
 * Free lists are FIFO: blocks start free in id order, freed blocks join the back, allocation
 * takes the front. The batch lists running groups in arrival order, samples in order; a
 * sequence id is request_id * 256 + sample. Each step's decode attends over ctx_lens and
 * yields one token for every sequence in the batch.
 *
 * The caller executes a plan in this order: swap-outs (GPU block -> CPU slot), swap-ins
 * (CPU slot -> GPU block), copy-on-write copies (the three by pa_scheduler_execute_moves), KV
 * writes (slot_mapping), decode.
 *
 * Ownership: a scheduler owns the arrays of the plan it last returned; they stay valid until
 * its next step or its destruction. Calls on one scheduler must not overlap.
 */
#ifndef PA_SCHEDULER_H
#define PA_SCHEDULER_H

#include <stddef.h>
#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_scheduler pa_scheduler; /* opaque */

typedef enum {
  PA_PREEMPT_RECOMPUTE = 0, /* release; resume by rewriting the history (one-sample groups) */
  PA_PREEMPT_SWAP = 1       /* copy to CPU slots, release; resume by copying back */
} pa_preempt_mode;

typedef struct {
  int32_t num_seqs;
  const int64_t* seq_ids;       /* [num_seqs] request_id * 256 + sample */
  const int32_t* block_tables;  /* [num_seqs][max_blocks_per_seq], -1 after the last block */
  const int32_t* ctx_lens;      /* [num_seqs] KV positions after this step's writes */
  int32_t num_writes;
  const int32_t* write_seq;     /* [num_writes] batch index of the sequence written */
  const int32_t* write_pos;     /* [num_writes] position within that sequence */
  const int64_t* slot_mapping;  /* [num_writes] block * block_size + slot (pa_write_kv) */
  int32_t num_copies;
  const int32_t* copies;        /* [num_copies][2] (src, dst) GPU blocks (pa_copy_blocks) */
  int32_t num_swap_out;
  const int32_t* swap_out;      /* [num_swap_out][2] (GPU block, CPU slot) */
  int32_t num_swap_in;
  const int32_t* swap_in;       /* [num_swap_in][2] (CPU slot, GPU block) */
  int32_t num_finished;
  const int64_t* finished;      /* request ids retired at the start of the step */
  int32_t num_preempted;
  const int64_t* preempted;     /* request ids preempted in the step */
  int32_t num_free_blocks;      /* free GPU blocks after the step */
} pa_step_plan;

/* A scheduler over num_blocks GPU blocks of block_size slots and num_cpu_blocks CPU slots.
 * Returns NULL (and sets pa_last_error_message) if a size is not positive (num_cpu_blocks may
 * be 0). */
pa_scheduler* pa_scheduler_create(int32_t num_blocks, int32_t block_size,
                                  int32_t max_blocks_per_seq, int32_t max_running_seqs,
                                  pa_preempt_mode mode, int32_t num_cpu_blocks);
void pa_scheduler_destroy(pa_scheduler* s);

/* Queue a request of prompt_len tokens that produces max_new_tokens tokens in each of
 * num_samples samples (1..256) sharing the prompt. PA_EINVAL for a repeated id, sizes < 1, or
 * a request that could never fit (ceil((prompt_len + max_new_tokens) / block_size) above
 * max_blocks_per_seq, that many blocks per sample above the pool, or more samples than
 * max_running_seqs: admission stops at the first waiting group that does not fit, so such a
 * group would hold every request behind it). */
pa_status pa_scheduler_add_request(pa_scheduler* s, int64_t request_id, int32_t prompt_len,
                                   int32_t max_new_tokens, int32_t num_samples);

/* Plan one step (policy above) into *plan. PA_ENOSPACE if a swap needs more CPU slots than
 * are free (the scheduler is then left unusable). */
pa_status pa_scheduler_step(pa_scheduler* s, pa_step_plan* plan);

/* Free GPU blocks now; their ids in free-list order into out[0..cap) (out may be NULL). */
int32_t pa_scheduler_free_blocks(const pa_scheduler* s, int32_t* out, int32_t cap);

/* 1 while some request is waiting or running, else 0. */
int32_t pa_scheduler_has_unfinished(const pa_scheduler* s);

/*
 * pa_scheduler_execute_moves - enqueue a plan's block moves, in the order the plan requires.
 *
 * Sources: "When KV Capacity Runs Out", Figure 4 (a preempted request's KV goes to CPU memory
 * before its blocks are reused, and comes back into possibly different blocks); PagedAttention
 * summary page, copy-on-write paragraph. Enqueues on `stream`, in this order:
 *   1. swap-outs:  for each (GPU block b, CPU slot c) of plan->swap_out, every layer l:
 *                  cpu_pool[c][l][0][:] = k_pools[l][b][...], cpu_pool[c][l][1][:] = v_pools[l][b]
 *   2. swap-ins:   for each (CPU slot c, GPU block b) of plan->swap_in: the reverse assignment;
 *   3. copies:     for each (src, dst) of plan->copies: every layer's K and V block dst
 *                  becomes a copy of block src (pa_copy_blocks semantics).
 * The plan's lists are read on the host during the call (nothing is uploaded: the ids travel
 * as kernel parameters), so the plan may be released or re-planned as soon as this returns.
 * The KV writes (pa_write_kv with plan->slot_mapping) and the decode are the caller's: they
 * need this step's new K/V and queries.
 *   k_pools, v_pools  host arrays of num_layers device pool pointers, each
 *                     [num_blocks][block_bytes] (16-byte aligned)
 *   cpu_pool          pinned host memory [num_cpu_blocks][num_layers][2][block_bytes]
 *                     (16-byte aligned; may be NULL when the plan has no swaps)
 *   err_flag          optional device int32 (as in pa.h; host-checked ids cannot set it)
 * Errors: PA_EINVAL, with nothing enqueued, if a block id lies outside [0, num_blocks), a CPU
 * slot outside [0, num_cpu_blocks), or cpu_pool is not pinned; PA_ECUDA if a launch fails. The
 * caller must not reuse swapped-out GPU blocks, or overwrite swapped-in CPU slots, until the
 * stream has passed this call.
 */
pa_status pa_scheduler_execute_moves(const pa_step_plan* plan, void* const* k_pools,
                                     void* const* v_pools, int32_t num_layers, int32_t num_blocks,
                                     size_t block_bytes, void* cpu_pool, int32_t num_cpu_blocks,
                                     int32_t* err_flag, pa_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_SCHEDULER_H */
