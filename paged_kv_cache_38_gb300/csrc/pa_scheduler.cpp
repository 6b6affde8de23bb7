// pa_scheduler.cpp - host scheduler and KV block manager (include/pa_scheduler.h).
//
// Plans the block tables, slots, copy-on-write pairs and swaps of each decode step; the
// policy and its sources are stated in the header. Plain host C++; only the last entry point,
// which enqueues a plan's block moves, reaches the mover kernels (pa_movers.cu).
#include <algorithm>
#include <deque>
#include <memory>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/pa_scheduler.h"
#include "pa_internal.h"

namespace {

enum GroupState { kNew, kRunning, kWaitRecompute, kSwapped, kFinished };

struct Seq {
  int32_t sample = 0;
  std::vector<int32_t> table;  // GPU blocks (CPU slots while swapped)
  int32_t length = 0;          // KV positions stored
  int32_t generated = 0;       // tokens produced
  int32_t row = -1;            // batch row in the last plan
};

struct Group {
  int64_t id = 0;
  int64_t arrival = 0;
  int32_t prompt = 0;
  int32_t max_new = 0;
  GroupState state = kNew;
  std::vector<Seq> seqs;
};

struct Write {
  const Seq* seq;
  int32_t pos;
  int64_t slot;
};

int32_t ceil_div(int64_t a, int64_t b) { return static_cast<int32_t>((a + b - 1) / b); }

}  // namespace

struct pa_scheduler {
  int32_t num_blocks, block_size, max_blocks, max_running;
  pa_preempt_mode mode;
  std::deque<int32_t> free_gpu, free_cpu;  // FIFO: allocate from the front, release to the back
  std::vector<int32_t> ref_gpu, ref_cpu;
  std::unordered_map<int64_t, std::unique_ptr<Group>> groups;
  std::deque<Group*> waiting;
  std::vector<Group*> running;  // ascending arrival
  int64_t arrivals = 0;
  bool broken = false;

  // the last plan's storage
  std::vector<int64_t> seq_ids, finished, preempted, slots;
  std::vector<int32_t> ctx_lens, write_seq, write_pos, copies, swap_out, swap_in;
  // The plan's block tables persist across steps: row i holds row_len[i] entries and -1 after
  // them, so a step rewrites each row's entries and clears only what its old length covered
  // beyond the new one, instead of all max_blocks entries of every row.
  std::vector<int32_t> tables, row_len;

  int32_t alloc_gpu() {
    const int32_t b = free_gpu.front();
    free_gpu.pop_front();
    ref_gpu[b] = 1;
    return b;
  }
  void release_gpu(int32_t b) {
    if (--ref_gpu[b] == 0) free_gpu.push_back(b);
  }
  void free_group(Group* g) {
    for (Seq& s : g->seqs) {
      for (int32_t b : s.table) release_gpu(b);
      s.table.clear();
    }
  }
  int64_t need(const Seq& s) const {
    if (s.length % block_size == 0) return 1;
    return ref_gpu[s.table.back()] > 1 ? 1 : 0;
  }
  int64_t growth() const {
    int64_t n = 0;
    for (const Group* g : running)
      for (const Seq& s : g->seqs) n += need(s);
    return n;
  }
  int64_t running_seqs() const {
    int64_t n = 0;
    for (const Group* g : running) n += static_cast<int64_t>(g->seqs.size());
    return n;
  }
  static std::vector<int32_t> distinct(const Group* g) {
    std::vector<int32_t> out;
    for (const Seq& s : g->seqs)
      for (int32_t b : s.table)
        if (std::find(out.begin(), out.end(), b) == out.end()) out.push_back(b);
    return out;
  }
  int64_t admission_cost(const Group* g) const {
    if (g->state == kNew) return ceil_div(g->prompt, block_size);
    if (g->state == kWaitRecompute) return ceil_div(g->seqs[0].length + 1, block_size);
    int64_t cost = static_cast<int64_t>(distinct(g).size());
    for (const Seq& s : g->seqs)
      if (s.length % block_size == 0 || ref_cpu[s.table.back()] > 1) ++cost;
    return cost;
  }
  void insert_running(Group* g) {
    auto it = std::upper_bound(running.begin(), running.end(), g,
                               [](const Group* a, const Group* b) { return a->arrival < b->arrival; });
    running.insert(it, g);
  }

  pa_status step(pa_step_plan* plan, std::string& msg) {
    seq_ids.clear();
    finished.clear();
    preempted.clear();
    slots.clear();
    ctx_lens.clear();
    write_seq.clear();
    write_pos.clear();
    copies.clear();
    swap_out.clear();
    swap_in.clear();
    std::vector<Write> writes;

    // 1. retire groups whose samples have produced every token
    for (auto it = running.begin(); it != running.end();) {
      Group* g = *it;
      const bool done = std::all_of(g->seqs.begin(), g->seqs.end(),
                                    [&](const Seq& s) { return s.generated >= g->max_new; });
      if (done) {
        free_group(g);
        g->state = kFinished;
        finished.push_back(g->id);
        it = running.erase(it);
      } else {
        ++it;
      }
    }

    // 2. every running sequence must be able to grow: preempt the group that arrived last
    while (!running.empty() && growth() > static_cast<int64_t>(free_gpu.size())) {
      Group* v = running.back();
      running.pop_back();
      if (mode == PA_PREEMPT_RECOMPUTE && v->seqs.size() == 1) {
        free_group(v);
        v->state = kWaitRecompute;
      } else {
        const std::vector<int32_t> blocks = distinct(v);
        if (blocks.size() > free_cpu.size()) {
          broken = true;
          msg = "CPU swap space exhausted";
          return PA_ENOSPACE;
        }
        std::unordered_map<int32_t, int32_t> to_cpu;
        for (int32_t b : blocks) {
          const int32_t c = free_cpu.front();
          free_cpu.pop_front();
          to_cpu[b] = c;
          swap_out.push_back(b);
          swap_out.push_back(c);
        }
        for (Seq& s : v->seqs)
          for (int32_t& e : s.table) {
            e = to_cpu[e];
            ++ref_cpu[e];
          }
        for (int32_t b : blocks)
          for (int32_t r = ref_gpu[b]; r > 0; --r) release_gpu(b);
        v->state = kSwapped;
      }
      waiting.push_front(v);
      preempted.push_back(v->id);
    }

    // 3. admissions, only in a step without preemption
    std::vector<const Group*> prefilled;
    if (preempted.empty()) {
      while (!waiting.empty()) {
        Group* g = waiting.front();
        if (running_seqs() + static_cast<int64_t>(g->seqs.size()) > max_running) break;
        if (admission_cost(g) > static_cast<int64_t>(free_gpu.size()) - growth()) break;
        waiting.pop_front();
        if (g->state == kNew) {
          const int32_t n = ceil_div(g->prompt, block_size);
          std::vector<int32_t> blocks;
          for (int32_t i = 0; i < n; ++i) blocks.push_back(alloc_gpu());
          for (int32_t b : blocks) ref_gpu[b] = static_cast<int32_t>(g->seqs.size());
          for (Seq& s : g->seqs) {
            s.table = blocks;
            s.length = g->prompt;
            s.generated = 1;
          }
          for (int32_t pos = 0; pos < g->prompt; ++pos)
            writes.push_back({&g->seqs[0], pos,
                              static_cast<int64_t>(blocks[pos / block_size]) * block_size +
                                  pos % block_size});
          prefilled.push_back(g);
        } else if (g->state == kWaitRecompute) {
          Seq& s = g->seqs[0];
          const int32_t total = s.length + 1;
          s.table.clear();
          for (int32_t i = 0; i < ceil_div(total, block_size); ++i) s.table.push_back(alloc_gpu());
          for (int32_t pos = 0; pos < total; ++pos)
            writes.push_back({&s, pos,
                              static_cast<int64_t>(s.table[pos / block_size]) * block_size +
                                  pos % block_size});
          s.length = total;
          s.generated += 1;
          prefilled.push_back(g);
        } else {  // swapped: CPU slots back into fresh GPU blocks, same order
          const std::vector<int32_t> cslots = distinct(g);
          std::unordered_map<int32_t, int32_t> to_gpu;
          for (int32_t c : cslots) {
            const int32_t b = free_gpu.front();
            free_gpu.pop_front();
            ref_gpu[b] = 0;
            to_gpu[c] = b;
            swap_in.push_back(c);
            swap_in.push_back(b);
          }
          for (Seq& s : g->seqs)
            for (int32_t& e : s.table) {
              e = to_gpu[e];
              ++ref_gpu[e];
            }
          for (int32_t c : cslots) {
            ref_cpu[c] = 0;
            free_cpu.push_back(c);
          }
        }
        g->state = kRunning;
        insert_running(g);
      }
    }

    // 4. one new token for every running sequence that was not just prefilled
    for (Group* g : running) {
      if (std::find(prefilled.begin(), prefilled.end(), g) != prefilled.end()) continue;
      for (Seq& s : g->seqs) {
        int32_t b;
        if (s.length % block_size == 0) {
          b = alloc_gpu();
          s.table.push_back(b);
        } else {
          const int32_t last = s.table.back();
          if (ref_gpu[last] > 1) {
            b = alloc_gpu();
            copies.push_back(last);
            copies.push_back(b);
            --ref_gpu[last];
            s.table.back() = b;
          }
          b = s.table.back();
        }
        writes.push_back({&s, s.length,
                          static_cast<int64_t>(b) * block_size + s.length % block_size});
        s.length += 1;
        s.generated += 1;
      }
    }

    // 5. the batch
    const int64_t n = running_seqs();
    if (static_cast<int64_t>(row_len.size()) < n) {
      tables.resize(static_cast<size_t>(n) * max_blocks, -1);
      row_len.resize(static_cast<size_t>(n), 0);
    }
    for (Group* g : running)
      for (Seq& s : g->seqs) {
        const int32_t i = static_cast<int32_t>(seq_ids.size());
        s.row = i;
        seq_ids.push_back(g->id * 256 + s.sample);
        int32_t* row = tables.data() + static_cast<size_t>(i) * max_blocks;
        const int32_t len = static_cast<int32_t>(s.table.size());
        std::copy(s.table.begin(), s.table.end(), row);
        if (len < row_len[i]) std::fill(row + len, row + row_len[i], -1);
        row_len[i] = len;
        ctx_lens.push_back(s.length);
      }
    for (const Write& w : writes) {
      write_seq.push_back(w.seq->row);
      write_pos.push_back(w.pos);
      slots.push_back(w.slot);
    }
    plan->num_seqs = static_cast<int32_t>(seq_ids.size());
    plan->seq_ids = seq_ids.data();
    plan->block_tables = tables.data();
    plan->ctx_lens = ctx_lens.data();
    plan->num_writes = static_cast<int32_t>(slots.size());
    plan->write_seq = write_seq.data();
    plan->write_pos = write_pos.data();
    plan->slot_mapping = slots.data();
    plan->num_copies = static_cast<int32_t>(copies.size() / 2);
    plan->copies = copies.data();
    plan->num_swap_out = static_cast<int32_t>(swap_out.size() / 2);
    plan->swap_out = swap_out.data();
    plan->num_swap_in = static_cast<int32_t>(swap_in.size() / 2);
    plan->swap_in = swap_in.data();
    plan->num_finished = static_cast<int32_t>(finished.size());
    plan->finished = finished.data();
    plan->num_preempted = static_cast<int32_t>(preempted.size());
    plan->preempted = preempted.data();
    plan->num_free_blocks = static_cast<int32_t>(free_gpu.size());
    return PA_OK;
  }
};

extern "C" {

pa_scheduler* pa_scheduler_create(int32_t num_blocks, int32_t block_size,
                                  int32_t max_blocks_per_seq, int32_t max_running_seqs,
                                  pa_preempt_mode mode, int32_t num_cpu_blocks) {
  if (num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 || max_running_seqs <= 0 ||
      num_cpu_blocks < 0 || (mode != PA_PREEMPT_RECOMPUTE && mode != PA_PREEMPT_SWAP)) {
    pa::record_error(PA_EINVAL, "pa_scheduler_create: sizes must be positive, mode valid");
    return nullptr;
  }
  auto* s = new pa_scheduler();
  s->num_blocks = num_blocks;
  s->block_size = block_size;
  s->max_blocks = max_blocks_per_seq;
  s->max_running = max_running_seqs;
  s->mode = mode;
  for (int32_t b = 0; b < num_blocks; ++b) s->free_gpu.push_back(b);
  for (int32_t c = 0; c < num_cpu_blocks; ++c) s->free_cpu.push_back(c);
  s->ref_gpu.assign(num_blocks, 0);
  s->ref_cpu.assign(num_cpu_blocks, 0);
  return s;
}

void pa_scheduler_destroy(pa_scheduler* s) { delete s; }

pa_status pa_scheduler_add_request(pa_scheduler* s, int64_t request_id, int32_t prompt_len,
                                   int32_t max_new_tokens, int32_t num_samples) {
  if (s == nullptr) return pa::record_error(PA_EINVAL, "scheduler is NULL");
  if (s->groups.count(request_id) || prompt_len < 1 || max_new_tokens < 1 || num_samples < 1 ||
      num_samples > 256)
    return pa::record_error(PA_EINVAL, "repeated request id, or a size out of range");
  // admission takes whole groups within max_running_seqs: a larger group could never run, and
  // would hold every request queued behind it
  if (num_samples > s->max_running)
    return pa::record_error(PA_EINVAL, "more samples than max_running_seqs");
  const int64_t longest = ceil_div(static_cast<int64_t>(prompt_len) + max_new_tokens, s->block_size);
  if (longest > s->max_blocks || longest * num_samples > s->num_blocks)
    return pa::record_error(PA_EINVAL, "the request can never fit the pool or a block table");
  auto g = std::make_unique<Group>();
  g->id = request_id;
  g->arrival = s->arrivals++;
  g->prompt = prompt_len;
  g->max_new = max_new_tokens;
  g->seqs.resize(num_samples);
  for (int32_t i = 0; i < num_samples; ++i) g->seqs[i].sample = i;
  s->waiting.push_back(g.get());
  s->groups[request_id] = std::move(g);
  return PA_OK;
}

pa_status pa_scheduler_step(pa_scheduler* s, pa_step_plan* plan) {
  if (s == nullptr || plan == nullptr) return pa::record_error(PA_EINVAL, "NULL argument");
  if (s->broken) return pa::record_error(PA_ENOSPACE, "scheduler stopped: CPU swap space exhausted");
  std::string msg;
  const pa_status st = s->step(plan, msg);
  return st == PA_OK ? st : pa::record_error(st, msg);
}

int32_t pa_scheduler_free_blocks(const pa_scheduler* s, int32_t* out, int32_t cap) {
  if (s == nullptr) return 0;
  int32_t i = 0;
  for (int32_t b : s->free_gpu) {
    if (out != nullptr && i < cap) out[i] = b;
    ++i;
  }
  return i;
}

int32_t pa_scheduler_has_unfinished(const pa_scheduler* s) {
  return s != nullptr && (!s->waiting.empty() || !s->running.empty()) ? 1 : 0;
}

pa_status pa_scheduler_execute_moves(const pa_step_plan* plan, void* const* k_pools,
                                     void* const* v_pools, int32_t num_layers, int32_t num_blocks,
                                     size_t block_bytes, void* cpu_pool, int32_t num_cpu_blocks,
                                     int32_t* err_flag, pa_stream stream) {
  if (plan == nullptr) return pa::record_error(PA_EINVAL, "plan is NULL");
  std::string msg;
  const pa_status st = pa::run_plan_moves(
      k_pools, v_pools, num_layers, num_blocks, block_bytes, cpu_pool, num_cpu_blocks,
      plan->swap_out, plan->num_swap_out, plan->swap_in, plan->num_swap_in, plan->copies,
      plan->num_copies, err_flag, reinterpret_cast<cudaStream_t>(stream), msg);
  return st == PA_OK ? PA_OK : pa::record_error(st, msg);
}

}  // extern "C"
