"""Plain Python scheduler and KV block manager (test infrastructure: the oracle of the C++ one).

Only the tests may use this module. It shares no code with the library. It restates, step by
step and without any optimisation, the bookkeeping the sources describe:

 [P1] "When KV Capacity Runs Out: Pausing and Resuming Requests", Figures 1-5: blocks are linked
      only when the last one is full; when none is free a running request is paused and its
      blocks released (not zeroed); the freed block goes to the request that needs it; a
      paused request keeps its token history and later resumes either by recomputing its KV
      (all retained tokens processed together, Figure 3) or by restoring KV stored in CPU
      memory into possibly different blocks and then processing its pending token (Figure 4).
 [PA] "Efficient Memory Management for Large Language Model Serving with PagedAttention"
      (summary page): a block table per request maps logical blocks, filled left to right, to
      physical blocks and counts filled slots; samples of one prompt share its blocks through a
      reference count; a write into a shared block gets its own copy (copy-on-write); blocks
      whose count drops to zero are freed; with first-come-first-served scheduling the latest
      requests are preempted, all blocks of a sequence group at once.
 [CB] "Continuous Batching and PagedAttention", section "The scheduler loop, written out":
      retire finished sequences, fill vacancies from the waiting queue while memory permits,
      evict the newest running sequence while a running one cannot grow (it goes back to the
      front of the waiting queue), then one step for every running sequence.

Readings where the sources leave a choice open (the C++ scheduler follows the same ones):
  * Free lists are FIFO: physical blocks start free in id order, freed blocks join the back in
    the order they are released (sample order, then logical order), allocation takes the front.
    [P1] Figure 2 then holds: B's P2 and P3 are released and A receives P2.
  * A step first retires groups whose samples reached max_new_tokens, then makes every running
    group able to grow by one token (preempting the latest-arrived running group while the
    blocks needed exceed the free ones), then -- only if nothing was preempted in this step --
    admits waiting groups in queue order while their blocks fit beside the growth of the running
    ones (head-of-line: the first that does not fit stops admission), then appends one token to
    every running sequence that was not just admitted by prefill or recompute.
  * Growth need of a sequence = 1 if its last block is full or shared (reference count > 1),
    else 0; a group's need is the sum over its samples (an upper bound: the last sharer writes
    in place).
  * A new group's prompt (P tokens) is written once into ceil(P / B) blocks shared by all its
    samples; the step's decode then yields each sample's first token. A single-sequence group
    in recompute mode is released on preemption and resumes by rewriting positions
    [0, L + 1) (its L stored positions and the pending token) into fresh blocks. Groups of
    several samples are always swapped (their sharing is kept): their distinct blocks go to CPU
    slots (FIFO) and come back, on resumption, into fresh GPU blocks in the same order, after
    which the group grows by one token like any running group.
  * The batch lists running groups in arrival order, samples in order. Sequence id =
    request_id * 256 + sample.
  * Per step the caller executes, in this order: swap-outs (GPU block -> CPU slot), swap-ins
    (CPU slot -> GPU block), copy-on-write copies (src -> dst), KV writes (slot mapping), decode.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field
from typing import Deque, Dict, List, Optional, Tuple

RECOMPUTE, SWAP = 0, 1
_NEW, _RUNNING, _WAITING_RECOMPUTE, _SWAPPED, _FINISHED = range(5)


@dataclass
class Sequence:
    sample: int
    table: List[int] = field(default_factory=list)   # GPU block ids (or CPU slots when swapped)
    length: int = 0                                  # KV positions stored
    generated: int = 0                               # tokens produced so far


@dataclass
class Group:
    request_id: int
    arrival: int
    prompt_len: int
    max_new_tokens: int
    seqs: List[Sequence]
    state: int = _NEW


@dataclass
class Plan:
    seq_ids: List[int]
    block_tables: List[List[int]]     # padded with -1 to max_blocks_per_seq
    ctx_lens: List[int]
    writes: List[Tuple[int, int, int]]  # (batch index, position, slot)
    copies: List[Tuple[int, int]]       # (src, dst) GPU blocks
    swap_out: List[Tuple[int, int]]     # (GPU block, CPU slot)
    swap_in: List[Tuple[int, int]]      # (CPU slot, GPU block)
    finished: List[int]                 # request ids retired at the start of the step
    preempted: List[int]                # request ids preempted in the step
    num_free_blocks: int


class Scheduler:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int,
                 max_running_seqs: int, mode: int, num_cpu_blocks: int):
        self.B = block_size
        self.num_blocks = num_blocks
        self.max_blocks = max_blocks_per_seq
        self.max_running = max_running_seqs
        self.mode = mode
        self.free: Deque[int] = deque(range(num_blocks))
        self.ref = [0] * num_blocks
        self.cpu_free: Deque[int] = deque(range(num_cpu_blocks))
        self.cpu_ref = [0] * num_cpu_blocks
        self.waiting: Deque[Group] = deque()
        self.running: List[Group] = []
        self.arrivals = 0
        self.requests: Dict[int, Group] = {}

    # -------------------------------------------------------------- requests
    def add_request(self, request_id: int, prompt_len: int, max_new_tokens: int,
                    num_samples: int) -> bool:
        if request_id in self.requests or prompt_len < 1 or max_new_tokens < 1:
            return False
        if not 1 <= num_samples <= min(256, self.max_running):
            return False  # a group larger than max_running_seqs could never be admitted
        longest = prompt_len + max_new_tokens
        if -(-longest // self.B) > self.max_blocks:
            return False
        if -(-longest // self.B) * num_samples > self.num_blocks:
            return False
        g = Group(request_id, self.arrivals, prompt_len, max_new_tokens,
                  [Sequence(i) for i in range(num_samples)])
        self.arrivals += 1
        self.requests[request_id] = g
        self.waiting.append(g)
        return True

    # -------------------------------------------------------------- block helpers
    def _alloc(self) -> int:
        b = self.free.popleft()
        self.ref[b] = 1
        return b

    def _release(self, b: int) -> None:
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def _free_group(self, g: Group) -> None:
        for s in g.seqs:
            for b in s.table:
                self._release(b)
            s.table = []

    def _need(self, s: Sequence) -> int:
        if s.length % self.B == 0:
            return 1
        return 1 if self.ref[s.table[-1]] > 1 else 0

    def _growth(self) -> int:
        return sum(self._need(s) for g in self.running for s in g.seqs)

    def _distinct(self, g: Group) -> List[int]:
        seen: List[int] = []
        for s in g.seqs:
            for b in s.table:
                if b not in seen:
                    seen.append(b)
        return seen

    def _admission_cost(self, g: Group) -> int:
        if g.state == _NEW:
            return -(-g.prompt_len // self.B)
        if g.state == _WAITING_RECOMPUTE:
            return -(-(g.seqs[0].length + 1) // self.B)
        # swapped: its distinct blocks, plus its own growth after coming back
        cost = len(self._distinct(g))
        for s in g.seqs:
            if s.length % self.B == 0 or self.cpu_ref[s.table[-1]] > 1:
                cost += 1
        return cost

    # -------------------------------------------------------------- one step
    def step(self) -> Plan:
        finished: List[int] = []
        preempted: List[int] = []
        writes: List[Tuple[Sequence, int, int]] = []
        copies: List[Tuple[int, int]] = []
        swap_out: List[Tuple[int, int]] = []
        swap_in: List[Tuple[int, int]] = []

        # 1. retire groups whose samples have produced every token
        for g in list(self.running):
            if all(s.generated >= g.max_new_tokens for s in g.seqs):
                self._free_group(g)
                g.state = _FINISHED
                self.running.remove(g)
                finished.append(g.request_id)

        # 2. every running group must be able to grow by one token: preempt the latest
        while self.running and self._growth() > len(self.free):
            victim = max(self.running, key=lambda x: x.arrival)
            self.running.remove(victim)
            if self.mode == RECOMPUTE and len(victim.seqs) == 1:
                self._free_group(victim)
                victim.state = _WAITING_RECOMPUTE
            else:
                blocks = self._distinct(victim)
                if len(blocks) > len(self.cpu_free):
                    raise RuntimeError("CPU swap space exhausted")
                to_cpu = {}
                for b in blocks:
                    c = self.cpu_free.popleft()
                    to_cpu[b] = c
                    swap_out.append((b, c))
                for s in victim.seqs:
                    for b in s.table:
                        self.cpu_ref[to_cpu[b]] += 1
                    s.table = [to_cpu[b] for b in s.table]
                for b in blocks:
                    refs = self.ref[b]
                    for _ in range(refs):
                        self._release(b)
                victim.state = _SWAPPED
            self.waiting.appendleft(victim)
            preempted.append(victim.request_id)

        # 3. admissions, only in a step without preemption
        prefilled: List[Group] = []
        if not preempted:
            while self.waiting:
                g = self.waiting[0]
                if sum(len(x.seqs) for x in self.running) + len(g.seqs) > self.max_running:
                    break
                if self._admission_cost(g) > len(self.free) - self._growth():
                    break
                self.waiting.popleft()
                if g.state == _NEW:
                    n = -(-g.prompt_len // self.B)
                    blocks = [self._alloc() for _ in range(n)]
                    for b in blocks:
                        self.ref[b] = len(g.seqs)
                    for s in g.seqs:
                        s.table = list(blocks)
                        s.length = g.prompt_len
                        s.generated = 1
                    for pos in range(g.prompt_len):
                        writes.append((g.seqs[0], pos, blocks[pos // self.B] * self.B + pos % self.B))
                    prefilled.append(g)
                elif g.state == _WAITING_RECOMPUTE:
                    s = g.seqs[0]
                    total = s.length + 1
                    s.table = [self._alloc() for _ in range(-(-total // self.B))]
                    for pos in range(total):
                        writes.append((s, pos, s.table[pos // self.B] * self.B + pos % self.B))
                    s.length = total
                    s.generated += 1
                    prefilled.append(g)
                else:  # swapped: CPU slots back into fresh GPU blocks, same order
                    slots: List[int] = []
                    for s in g.seqs:
                        for c in s.table:
                            if c not in slots:
                                slots.append(c)
                    to_gpu = {}
                    for c in slots:
                        b = self.free.popleft()
                        self.ref[b] = 0
                        to_gpu[c] = b
                        swap_in.append((c, b))
                    for s in g.seqs:
                        for c in s.table:
                            self.ref[to_gpu[c]] += 1
                        s.table = [to_gpu[c] for c in s.table]
                    for c in slots:
                        self.cpu_ref[c] = 0
                        self.cpu_free.append(c)
                g.state = _RUNNING
                self.running.append(g)
                self.running.sort(key=lambda x: x.arrival)

        # 4. one new token for every running sequence that was not just prefilled
        for g in self.running:
            if g in prefilled:
                continue
            for s in g.seqs:
                if s.length % self.B == 0:
                    b = self._alloc()
                    s.table.append(b)
                else:
                    last = s.table[-1]
                    if self.ref[last] > 1:
                        b = self._alloc()
                        copies.append((last, b))
                        self.ref[last] -= 1
                        s.table[-1] = b
                    b = s.table[-1]
                writes.append((s, s.length, b * self.B + s.length % self.B))
                s.length += 1
                s.generated += 1

        # 5. the batch
        seq_ids: List[int] = []
        tables: List[List[int]] = []
        lens: List[int] = []
        index: Dict[int, int] = {}
        for g in self.running:
            for s in g.seqs:
                index[id(s)] = len(seq_ids)
                seq_ids.append(g.request_id * 256 + s.sample)
                tables.append(s.table + [-1] * (self.max_blocks - len(s.table)))
                lens.append(s.length)
        return Plan(seq_ids, tables, lens, [(index[id(s)], pos, slot) for s, pos, slot in writes],
                    copies, swap_out, swap_in, finished, preempted, len(self.free))

    # -------------------------------------------------------------- inspection
    def num_free_blocks(self) -> int:
        return len(self.free)

    def has_unfinished(self) -> bool:
        return bool(self.waiting or self.running)
