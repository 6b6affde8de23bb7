"""Pins of the scheduler / block-manager oracle: checks against something other than itself.

Each ``pin_*`` takes a module exposing the oracle's interface (``Scheduler``, ``RECOMPUTE``,
``SWAP``) and raises AssertionError when it disagrees with
  * the worked example of "When KV Capacity Runs Out", Figures 1-5 (tests/golden), run through
    both resumption methods;
  * a data-level replay of every plan: a pool of token identities to which the plan's swaps,
    copies and writes are applied in the documented order, after which every running sequence,
    gathered through its block table, must read back its own history -- the property the
    PagedAttention summary page states (logical blocks anywhere, shared blocks copied before a
    write, swapped blocks restored, possibly elsewhere);
  * the bookkeeping invariants of the sources: at most one partly filled block per sequence,
    blocks shared only within a sequence group, every used block referenced, first-come-first-
    served admission, the newest running group preempted, all of a group's blocks evicted at
    once, every sample delivering exactly its max_new_tokens.
The same replay and invariants check the C++ scheduler's plans in ``tests/test_scheduler.py``.
"""
from __future__ import annotations

import os
import random

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ worked example

def _parse_golden(path):
    pool, requests, runs = None, [], []
    for raw in open(path):
        line = raw.split("#")[0].strip()
        if not line:
            continue
        w = line.split()
        if w[0] == "pool":
            pool = (int(w[1]), int(w[2]))
        elif w[0] == "request":
            requests.append((w[1], int(w[2]), int(w[3]), int(w[4])))
        elif w[0] == "mode":
            runs.append((w[1], []))
        elif w[0] == "step":
            runs[-1][1].append([])
        elif w[0] == "expect":
            runs[-1][1][-1].append(w[1:])
    return pool, requests, runs


def _block(name: str) -> int:
    assert name.startswith("P"), name
    return int(name[1:])


def pin_figures_1_5(bm):
    pool, requests, runs = _parse_golden(os.path.join(GOLDEN, "scheduler_figures_1_5.txt"))
    for mode_name, steps in runs:
        mode = bm.RECOMPUTE if mode_name == "recompute" else bm.SWAP
        s = bm.Scheduler(pool[0], pool[1], 8, 16, mode, 8)
        ids = {}
        for i, (name, prompt, max_new, samples) in enumerate(requests):
            ids[name] = i
            assert s.add_request(i, prompt, max_new, samples)
        name_of = {v: k for k, v in ids.items()}
        for n, expects in enumerate(steps):
            plan = s.step()
            where = f"{mode_name} step {n + 1}"
            batch = {name_of[sid // 256]: j for j, sid in enumerate(plan.seq_ids)}
            for e in expects:
                if e[0] == "free":
                    assert plan.num_free_blocks == int(e[1]), where
                elif e[0] == "free_blocks":
                    assert sorted(s.free) == sorted(_block(x) for x in e[1:]), where
                elif e[0] == "preempted":
                    assert [name_of[r] for r in plan.preempted] == e[1:], where
                elif e[0] == "finished":
                    assert [name_of[r] for r in plan.finished] == e[1:], where
                elif e[0] == "idle":
                    assert e[1] not in batch, where
                elif e[0] == "write":
                    j = batch[e[1]]
                    want = (j, int(e[2]), _block(e[3]) * pool[1] + int(e[4]))
                    assert want in plan.writes, (where, want, plan.writes)
                elif e[0] in ("swap_out", "swap_in"):
                    assert len(getattr(plan, e[0])) == int(e[1]), where
                else:
                    j = batch[e[0]]
                    assert plan.ctx_lens[j] == int(e[1]), where
                    table = [b for b in plan.block_tables[j] if b >= 0]
                    if len(e) == 3 and not e[2].startswith("P"):
                        assert len(table) == int(e[2]), where
                    else:
                        assert table == [_block(x) for x in e[2:]], (where, table)


# ------------------------------------------------------------------ replay of plans

class Replay:
    """Token identities in GPU blocks and CPU slots; applies plans and checks every gather."""

    def __init__(self, num_blocks: int, block_size: int, prompts: dict, arrival: dict):
        self.B = block_size
        self.num_blocks = num_blocks
        self.gpu = {b: [None] * block_size for b in range(num_blocks)}
        self.cpu = {}
        self.prompts = prompts          # request id -> prompt length
        self.delivered = {}             # sequence id -> tokens delivered
        self.arrival = arrival          # request id -> rank of its add_request call
        self.admitted = []              # request ids in order of first admission
        self.running = []               # request ids running after the previous step
        self.finished = set()

    def identity(self, seq_id: int, pos: int):
        req, sample = divmod(seq_id, 256)
        return ("p", req, pos) if pos < self.prompts[req] else ("g", req, sample, pos)

    def apply(self, plan, max_new: dict):
        B = self.B
        # preemption: the newest running group goes, with all of its blocks (the step retires
        # finished groups first, so they no longer count as running)
        before = [r for r in self.running if r not in plan.finished]
        for r in plan.preempted:
            assert r in before, "only running groups are preempted"
            assert all(self.arrival[r] >= self.arrival[x] for x in before if x != r), \
                "the preempted group must be the newest running one"
            before.remove(r)
        self.finished.update(plan.finished)
        for r in plan.finished:
            for sid, n in self.delivered.items():
                if sid // 256 == r:
                    assert n == max_new[r], "a sample must deliver exactly max_new_tokens"
        for b, c in plan.swap_out:
            self.cpu[c] = list(self.gpu[b])
        for c, b in plan.swap_in:
            self.gpu[b] = list(self.cpu[c])
        srcs = [s for s, _ in plan.copies]
        for s, d in plan.copies:
            assert d not in srcs, "a copy destination is never a source of the same step"
            self.gpu[d] = list(self.gpu[s])
        for j, pos, slot in plan.writes:
            self.gpu[slot // B][slot % B] = self.identity(plan.seq_ids[j], pos)
        owners = {}
        for j, sid in enumerate(plan.seq_ids):
            L = plan.ctx_lens[j]
            table = plan.block_tables[j]
            nb = -(-L // B)
            assert all(b >= 0 for b in table[:nb]) and all(b < 0 for b in table[nb:]), \
                "a sequence holds ceil(L / B) blocks: at most one partly filled"
            for pos in range(L):
                got = self.gpu[table[pos // B]][pos % B]
                assert got == self.identity(sid, pos), (sid, pos, got)
            for b in table[:nb]:
                owners.setdefault(b, set()).add(sid // 256)
            self.delivered[sid] = self.delivered.get(sid, 0) + 1
        assert all(len(o) == 1 for o in owners.values()), "blocks are shared only within a group"
        assert len(owners) + plan.num_free_blocks == self.num_blocks, \
            "every block is free or referenced by a running sequence"
        now = []
        for sid in plan.seq_ids:
            if sid // 256 not in now:
                now.append(sid // 256)
        for r in now:
            if r not in self.admitted:
                assert all(self.arrival[x] < self.arrival[r] for x in self.admitted), \
                    "requests are admitted in arrival order"
                self.admitted.append(r)
        assert [self.arrival[r] for r in now] == sorted(self.arrival[r] for r in now), \
            "the batch lists running groups in arrival order"
        for r in now:
            if r not in self.running:  # admitted or resumed in this step
                older = [x for x in self.arrival
                         if self.arrival[x] < self.arrival[r] and x not in self.finished]
                assert all(x in now for x in older), \
                    "first come, first served: no older unfinished request is left waiting"
        self.running = now


def random_script(seed: int):
    """Seeded workload: pool size, block size, requests (prompt, max_new, samples, arrival step)."""
    rng = random.Random(seed)
    B = rng.choice([4, 8, 16])
    num_blocks = rng.randint(12, 60)
    reqs = []
    for r in range(rng.randint(4, 14)):
        samples = rng.choice([1, 1, 1, 2, 3, 4])
        prompt = rng.randint(1, 5 * B)
        max_new = rng.randint(1, 4 * B)
        while -(-(prompt + max_new) // B) * samples > num_blocks:
            max_new = max(1, max_new // 2)
            prompt = max(1, prompt // 2)
        reqs.append((r, prompt, max_new, samples, rng.randint(0, 30)))
    return num_blocks, B, reqs


def drive(bm, seed: int, mode: int, max_steps: int = 600, check=True):
    """Run a random script on scheduler module ``bm``; returns the list of plans."""
    num_blocks, B, reqs = random_script(seed)
    s = bm.Scheduler(num_blocks, B, 64, 32, mode, 4 * num_blocks)
    order = sorted(reqs, key=lambda x: (x[4], x[0]))
    rep = Replay(num_blocks, B, {r: p for r, p, _, _, _ in reqs},
                 {x[0]: i for i, x in enumerate(order)})
    max_new = {r: m for r, _, m, _, _ in reqs}
    plans = []
    for step in range(max_steps):
        for r, p, m, n, at in order:
            if at == step:
                assert s.add_request(r, p, m, n)
        plan = s.step()
        if check:
            rep.apply(plan, max_new)
        plans.append(plan)
        if step > max(a for *_, a in reqs) and not s.has_unfinished():
            break
    else:
        raise AssertionError("the script did not finish")
    return plans


def pin_replay_recompute(bm):
    for seed in range(40):
        drive(bm, seed, bm.RECOMPUTE)


def pin_replay_swap(bm):
    for seed in range(40):
        drive(bm, 100 + seed, bm.SWAP)


def pin_preemption_happens(bm):
    """The random scripts do exercise preemption, copy-on-write and swapping."""
    seen = {"pre": 0, "cow": 0, "out": 0, "in": 0}
    for seed in range(40):
        for mode in (bm.RECOMPUTE, bm.SWAP):
            for p in drive(bm, 200 + seed, mode, check=False):
                seen["pre"] += len(p.preempted)
                seen["cow"] += len(p.copies)
                seen["out"] += len(p.swap_out)
                seen["in"] += len(p.swap_in)
    assert all(v > 0 for v in seen.values()), seen


def pin_oversized_group_refused(bm):
    """Admission takes whole groups, in queue order, within max_running_seqs ("Continuous
    Batching and PagedAttention", the scheduler loop: admit while memory permits; the summary
    page: all sequences of a group are scheduled together). A group with more samples than that
    could never run and, first in the queue, would hold every request behind it: it is refused
    when added, and the requests after it all finish."""
    for mode in (bm.RECOMPUTE, bm.SWAP):
        s = bm.Scheduler(64, 4, 16, 3, mode, 64)
        assert s.add_request(0, 5, 3, 1)
        assert not s.add_request(1, 5, 3, 4), "a group larger than max_running_seqs"
        assert s.add_request(2, 5, 3, 3), "a group of exactly max_running_seqs"
        assert s.add_request(3, 6, 2, 1)
        for _ in range(100):
            s.step()
            if not s.has_unfinished():
                break
        assert not s.has_unfinished(), "every admitted request finishes"


ALL_PINS = [pin_figures_1_5, pin_replay_recompute, pin_replay_swap, pin_preemption_happens,
            pin_oversized_group_refused]
