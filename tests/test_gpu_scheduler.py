"""The C++ scheduler driving the kernels over many decode steps (needs a GB300).

Every step's plan is executed as documented -- swap-outs, swap-ins, copy-on-write copies, KV
writes, decode -- on a small pool under memory pressure (preemption by recompute and by swap,
prompts shared by sample groups). The K and V of every token are a fixed function of its
identity (the prompt position of its request, or the position of its sample's own output), so
after each step every running sequence, gathered through its block table from the GPU pool,
must read back exactly its history, and the decode must match the oracle on that pool.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import TOL

import paged_kv_cache_38_gb300 as pa  # noqa: E402
from paged_kv_cache_38_gb300 import scheduler as sch

pytestmark = pytest.mark.gpu

HKV, HQ, D, B = 2, 4, 64, 16
ROWS = 4096


def _identity_rows(seq_ids, positions, prompts):
    """Row of the fixed K/V tables for each (sequence, position): a mix of the token identity."""
    req = seq_ids // 256
    sample = seq_ids % 256
    prompt = np.array([prompts[int(r)] for r in req], dtype=np.int64)
    gen = positions >= prompt
    key = req * 1000003 + positions * 7919 + np.where(gen, (sample + 1) * 104729, 0)
    return (key % ROWS).astype(np.int64)


@pytest.mark.parametrize("mode", [sch.RECOMPUTE, sch.SWAP], ids=["recompute", "swap"])
def test_scheduler_drives_the_kernels(mode):
    rng = np.random.default_rng(11 + mode)
    dev = torch.device("cuda")
    nblk, ncpu = 40, 160
    s = sch.Scheduler(nblk, B, 24, 12, mode, ncpu)
    reqs = []
    for r in range(16):
        n = int(rng.choice([1, 1, 2, 3])) if mode == sch.SWAP else 1
        p = int(rng.integers(1, 70))
        m = int(rng.integers(1, 90))
        while -(-(p + m) // B) * n > nblk:
            m //= 2
        reqs.append((r, p, max(m, 1), n, int(rng.integers(0, 40))))
    prompts = {r: p for r, p, *_ in reqs}
    g = torch.Generator().manual_seed(5)
    k_rows = torch.randn(ROWS, HKV, D, generator=g).to(torch.float16)
    v_rows = torch.randn(ROWS, HKV, D, generator=g).to(torch.float16)
    k_rows_d, v_rows_d = k_rows.to(dev), v_rows.to(dev)
    nan = torch.tensor(0x7E00, dtype=torch.int16).view(torch.float16)
    kp = torch.full((nblk, HKV, B, D), float(nan), dtype=torch.float16, device=dev)
    vp = kp.clone()
    cpu_pool = torch.zeros(ncpu, 1, 2, HKV * B * D * 2, dtype=torch.uint8).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    orc = oracle.load()
    seen = {"preempted": 0, "copies": 0, "swap": 0, "prefills": 0, "recomputes": 0}
    preempted_ids = set()
    step = 0
    while step < 400:
        for r, p, m, n, at in reqs:
            if at == step:
                assert s.add_request(r, p, m, n)
        plan = s.step()
        seen["preempted"] += len(plan.preempted)
        preempted_ids.update(int(x) for x in plan.preempted)
        seen["copies"] += len(plan.copies)
        seen["swap"] += len(plan.swap_out) + len(plan.swap_in)
        sch.execute_moves(plan, [kp], [vp], cpu_pool, err_flag=err)
        ids = plan.seq_ids_np
        if len(plan.slots_np):
            wseq = ids[plan.write_seq_np]
            rows = torch.from_numpy(_identity_rows(wseq, plan.write_pos_np.astype(np.int64), prompts))
            pa.pa_write_kv(k_rows_d[rows.to(dev)].contiguous(), v_rows_d[rows.to(dev)].contiguous(),
                           kp, vp, torch.from_numpy(plan.slots_np).to(dev), err_flag=err)
        # sequences whose whole context is written this step (an admitted prompt, or a recomputed
        # victim's prompt and generated tokens) are prefilled: causal attention of all their
        # positions over the pool, through pa_prefill, against the oracle
        full = []
        if len(plan.slots_np):
            for j in np.unique(plan.write_seq_np):
                pos = plan.write_pos_np[plan.write_seq_np == j]
                if pos.min() == 0 and len(pos) == int(plan.ctx_np[j]):
                    full.append(int(j))
        if full:
            lens = [int(plan.ctx_np[j]) for j in full]
            qs = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32))
            qq = torch.randn(int(qs[-1]), HQ, D, generator=g).to(torch.float16)
            bt = torch.from_numpy(np.ascontiguousarray(plan.tables_np[full]))
            cl = torch.from_numpy(np.ascontiguousarray(plan.ctx_np[full]))
            pout = pa.pa_prefill(qq.to(dev), kp, vp, bt.to(dev), cl.to(dev), qs.to(dev), 0.125,
                                 err_flag=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0, step
            ref = orc.prefill(qq, kp.cpu(), vp.cpu(), bt, cl, qs, dtype="f16", num_q_heads=HQ,
                              num_kv_heads=HKV, head_dim=D, block_size=B, scale=0.125)
            e = float(np.abs(pout.double().cpu().numpy() - ref).max())
            assert e <= TOL["f16"], (step, e)
            seen["prefills"] += len(full)
            # preempted lists request ids; a sequence id is request * 256 + sample
            seen["recomputes"] += sum(int(ids[j]) // 256 in preempted_ids for j in full)
        if len(ids):
            q = torch.randn(len(ids), HQ, D, generator=g).to(torch.float16)
            bt = torch.from_numpy(plan.tables_np).to(dev)
            cl = torch.from_numpy(plan.ctx_np).to(dev)
            out = pa.pa_decode(q.to(dev), kp, vp, bt, cl, 0.125, max_ctx_len=int(plan.ctx_np.max()),
                               err_flag=err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0, step
            # every running sequence reads back its own history through its table
            kh, vh = kp.cpu(), vp.cpu()
            for j, sid in enumerate(ids):
                L = int(plan.ctx_np[j])
                pos = np.arange(L)
                want = torch.from_numpy(_identity_rows(np.full(L, sid), pos, prompts))
                tb = torch.from_numpy(plan.tables_np[j][pos // B].astype(np.int64))
                slot = torch.from_numpy(pos % B)
                got_k = kh[tb, :, slot].view(torch.int16)
                got_v = vh[tb, :, slot].view(torch.int16)
                assert torch.equal(got_k, k_rows[want].view(torch.int16)), (step, int(sid))
                assert torch.equal(got_v, v_rows[want].view(torch.int16)), (step, int(sid))
            if step % 5 == 0:
                ref = orc.decode(q, kh, vh, plan.tables_np, plan.ctx_np, q_dtype="f16",
                                 kv_dtype="f16", num_q_heads=HQ, num_kv_heads=HKV, head_dim=D,
                                 block_size=B, scale=0.125)
                e = float(np.abs(out.double().cpu().numpy() - ref).max())
                assert e <= TOL["f16"], (step, e)
        step += 1
        if step > 40 and not s.has_unfinished():
            break
    assert not s.has_unfinished(), "the run did not finish"
    assert seen["preempted"] > 0 and seen["prefills"] > 0, seen
    if mode == sch.RECOMPUTE:
        assert seen["recomputes"] > 0, seen  # a preempted victim came back through pa_prefill
    if mode == sch.SWAP:
        assert seen["copies"] > 0 and seen["swap"] > 0, seen
