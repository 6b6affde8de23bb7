"""pa_write_kv, pa_write_kv_fp8, pa_copy_blocks and pa_swap_blocks on the GPU: bit-exact against
the oracle."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import pins
import synth
from helpers import TOL, gpu_decode, max_abs_err, oracle_decode

pytestmark = pytest.mark.gpu

import paged_kv_cache_38_gb300 as pa  # noqa: E402


def _u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().copy()


@pytest.mark.parametrize("spec", pins.small_specs(), ids=[s.name for s in pins.small_specs()])
def test_write_kv_bit_exact(spec):
    case = synth.make_case(spec, seed=400)
    orc = oracle.load()
    # poison the slots being written, plus padding tokens (-1) and one repeated token
    kp, vp = case.k_pool.clone(), case.v_pool.clone()
    B = spec.block_size
    raw_k = kp.view(torch.uint8).view(case.num_blocks, spec.num_kv_heads, B, -1)
    raw_v = vp.view(torch.uint8).view(case.num_blocks, spec.num_kv_heads, B, -1)
    for s in range(spec.num_seqs):
        sig = int(case.slot_mapping[s])
        if sig >= 0:
            raw_k[sig // B, :, sig % B] = 0xFF
            raw_v[sig // B, :, sig % B] = 0xFF
    sm = torch.cat([case.slot_mapping, torch.tensor([-1, -7], dtype=torch.int64)])
    knew = torch.cat([case.k_new, case.k_new[:2]])
    vnew = torch.cat([case.v_new, case.v_new[:2]])
    exp_k, exp_v = _u8(kp), _u8(vp)
    assert orc.write_kv(knew, vnew, exp_k, exp_v, sm, num_kv_heads=spec.num_kv_heads,
                        head_dim=spec.head_dim, block_size=B, kv_dtype=spec.kv_dtype) == 0
    gk, gv = kp.cuda(), vp.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_write_kv(knew.cuda(), vnew.cuda(), gk, gv, sm.cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(_u8(gk), exp_k) and np.array_equal(_u8(gv), exp_v)


def test_write_kv_generic_geometry():
    """bf16 rows of 6 chunks (head_dim 48), 12-token blocks, 3 kv heads (the kernel's division
    path), padding tokens, and enough tokens that threads make more than one pass: the pools
    equal the oracle's byte for byte."""
    orc = oracle.load()
    D, B, H, ntok = 48, 12, 3, 40001
    g = torch.Generator().manual_seed(12)
    k = torch.randn(ntok, H, D, generator=g).to(torch.bfloat16)
    v = torch.randn(ntok, H, D, generator=g).to(torch.bfloat16)
    nblk = ntok // B + 5
    slots = torch.randperm(nblk * B, generator=g)[:ntok].to(torch.int64)
    slots[::13] = -1
    kp = torch.full((nblk, H, B, D), 7.0, dtype=torch.bfloat16)
    vp = torch.full((nblk, H, B, D), -3.0, dtype=torch.bfloat16)
    exp_k, exp_v = _u8(kp), _u8(vp)
    assert orc.write_kv(k, v, exp_k, exp_v, slots, num_kv_heads=H, head_dim=D, block_size=B,
                        kv_dtype="bf16") == 0
    gk, gv = kp.cuda(), vp.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_write_kv(k.cuda(), v.cuda(), gk, gv, slots.cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(_u8(gk), exp_k) and np.array_equal(_u8(gv), exp_v)


def test_write_kv_out_of_pool_flagged():
    spec = synth.SPECS["toy"]
    case = synth.make_case(spec, seed=1).to("cuda")
    before = case.k_pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = torch.tensor([case.num_blocks * spec.block_size + 3], dtype=torch.int64, device="cuda")
    pa.pa_write_kv(case.k_new[:1], case.v_new[:1], case.k_pool, case.v_pool, bad, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_ERR_BLOCK_ID
    assert torch.equal(before.view(torch.uint8), case.k_pool.view(torch.uint8))


def _nan_codes_agree(got: np.ndarray, exp: np.ndarray) -> bool:
    """Equal codes, except that where the oracle wrote its NaN code the kernel may write the
    NaN code of either sign (the sign of a NaN carries nothing)."""
    nan = exp == 0x7F
    return np.array_equal(got[~nan], exp[~nan]) and bool(np.all((got[nan] & 0x7F) == 0x7F))


@pytest.mark.parametrize("src", ["bf16", "f16"])
def test_write_kv_fp8_every_bit_pattern(src):
    """All 65,536 source bit patterns, over several scales, quantised on write: the pools equal
    the oracle's, code for code."""
    orc = oracle.load()
    dt = torch.bfloat16 if src == "bf16" else torch.float16
    D, B = 128, 16
    ntok = 65536 // D
    vals = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(dt).reshape(ntok, 1, D)
    perm = torch.randperm(65536, generator=torch.Generator().manual_seed(3))
    vvals = vals.reshape(-1)[perm].reshape(ntok, 1, D).contiguous()
    nblk = ntok // B + 2
    slots = (torch.randperm(nblk * B, generator=torch.Generator().manual_seed(4))[:ntok]
             .to(torch.int64))
    for ks, vs in ((1.0, 1.0), (0.05, 0.37), (3.3e-3, 170.0)):
        kp = torch.full((nblk, 1, B, D), 0xAB, dtype=torch.uint8)
        vp = torch.full((nblk, 1, B, D), 0xCD, dtype=torch.uint8)
        exp_k, exp_v = _u8(kp), _u8(vp)
        assert orc.write_kv_fp8(vals, vvals, exp_k, exp_v, slots, src_dtype=src, num_kv_heads=1,
                                head_dim=D, block_size=B, k_scale=ks, v_scale=vs) == 0
        gk, gv = kp.cuda(), vp.cuda()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_write_kv_fp8(vals.cuda(), vvals.cuda(), gk, gv, slots.cuda(), ks, vs, err_flag=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert _nan_codes_agree(_u8(gk), exp_k), (src, ks)
        assert _nan_codes_agree(_u8(gv), exp_v), (src, vs)


def test_write_kv_fp8_generic_geometry():
    """A row of 3 chunks (head_dim 48), 12-token blocks and 3 kv heads (the kernel's division
    path, not its power-of-two shifts), padding tokens, and enough tokens that threads make
    more than one pass: the pools equal the oracle's byte for byte."""
    orc = oracle.load()
    D, B, H, ntok = 48, 12, 3, 70001
    g = torch.Generator().manual_seed(11)
    k = (torch.randn(ntok, H, D, generator=g) * 3).to(torch.bfloat16)
    v = torch.randn(ntok, H, D, generator=g).to(torch.bfloat16)
    nblk = ntok // B + 5
    slots = torch.randperm(nblk * B, generator=g)[:ntok].to(torch.int64)
    slots[::17] = -1
    ks, vs = float(k.float().abs().max()) / 448.0, float(v.float().abs().max()) / 448.0
    kp = torch.full((nblk, H, B, D), 0xAB, dtype=torch.uint8)
    vp = torch.full((nblk, H, B, D), 0xCD, dtype=torch.uint8)
    exp_k, exp_v = _u8(kp), _u8(vp)
    assert orc.write_kv_fp8(k, v, exp_k, exp_v, slots, src_dtype="bf16", num_kv_heads=H,
                            head_dim=D, block_size=B, k_scale=ks, v_scale=vs) == 0
    gk, gv = kp.cuda(), vp.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_write_kv_fp8(k.cuda(), v.cuda(), gk, gv, slots.cuda(), ks, vs, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(_u8(gk), exp_k) and np.array_equal(_u8(gv), exp_v)


def test_write_kv_fp8_then_decode():
    """A step on an E4M3 cache written by quantise-on-write: bit-exact pools (padding and an
    out-of-pool slot included), then the decode of the written cache matches the oracle."""
    orc = oracle.load()
    spec = synth.SPECS["fp8_long"].scaled(num_seqs=8, ctx_range=(40, 600))
    case = synth.make_case(spec, seed=77)
    g = torch.Generator().manual_seed(9)
    shape = (spec.num_seqs, spec.num_kv_heads, spec.head_dim)
    k_new = (torch.randn(shape, generator=g) * 2).to(torch.bfloat16)
    v_new = torch.randn(shape, generator=g).to(torch.bfloat16)
    ks = float(k_new.float().abs().max()) / 448.0
    vs = float(v_new.float().abs().max()) / 448.0
    sm = torch.cat([case.slot_mapping, torch.tensor([-1], dtype=torch.int64)])
    kn = torch.cat([k_new, k_new[:1]])
    vn = torch.cat([v_new, v_new[:1]])
    exp_k, exp_v = _u8(case.k_pool), _u8(case.v_pool)
    assert orc.write_kv_fp8(kn, vn, exp_k, exp_v, sm, src_dtype="bf16",
                            num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                            block_size=spec.block_size, k_scale=ks, v_scale=vs) == 0
    gcase = case.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_write_kv_fp8(kn.cuda(), vn.cuda(), gcase.k_pool, gcase.v_pool, sm.cuda(), ks, vs,
                       err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(_u8(gcase.k_pool), exp_k) and np.array_equal(_u8(gcase.v_pool), exp_v)
    # the newest tokens now hold codes of value / (ks, vs); decode the whole cache with those
    # per-tensor scales on both sides
    scaled = dataclasses.replace(gcase, k_scale=ks, v_scale=vs)
    out = gpu_decode(scaled)
    ref = oracle_decode(scaled)
    assert max_abs_err(out, ref) <= TOL["e4m3"]
    bad = torch.tensor([case.num_blocks * spec.block_size], dtype=torch.int64, device="cuda")
    before = _u8(gcase.k_pool)
    pa.pa_write_kv_fp8(kn[:1].cuda(), vn[:1].cuda(), gcase.k_pool, gcase.v_pool, bad, ks, vs,
                       err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_ERR_BLOCK_ID
    assert np.array_equal(_u8(gcase.k_pool), before)


def test_write_kv_fp8_host_validation():
    k = torch.zeros(2, 1, 128, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(4, 1, 16, 128, dtype=torch.uint8, device="cuda")
    sm = torch.zeros(2, dtype=torch.int64, device="cuda")
    for ks in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(pa.PaError) as e:
            pa.pa_write_kv_fp8(k, k, pool, pool, sm, ks, 1.0)
        assert e.value.status == pa.PA_EINVAL
    with pytest.raises(pa.PaError):
        pa.pa_write_kv_fp8(k.float(), k.float(), pool, pool, sm, 1.0, 1.0)


@pytest.mark.parametrize("layers,block_bytes_kib", [(1, 32), (3, 2), (4, 64)])
def test_copy_blocks_bit_exact(layers, block_bytes_kib):
    """Copy-on-write: destinations become source copies, sources and the rest stay unchanged."""
    orc = oracle.load()
    rng = np.random.default_rng(layers)
    nblk = 64
    bb = block_bytes_kib * 1024
    kps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(layers)]
    vps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(layers)]
    perm = rng.permutation(nblk)
    pairs = np.stack([perm[:20], perm[20:40]], axis=1).astype(np.int32)
    gk = [torch.from_numpy(p.copy()).cuda().view(nblk, -1) for p in kps]
    gv = [torch.from_numpy(p.copy()).cuda().view(nblk, -1) for p in vps]
    assert orc.copy_blocks(kps, vps, pairs, block_bytes=bb) == 0
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(gk, gv, torch.from_numpy(pairs).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in range(layers):
        assert np.array_equal(gk[l].cpu().numpy().reshape(-1), kps[l])
        assert np.array_equal(gv[l].cpu().numpy().reshape(-1), vps[l])
    bad = torch.tensor([[0, nblk]], dtype=torch.int32, device="cuda")
    pa.pa_copy_blocks(gk, gv, bad, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_ERR_BLOCK_ID
    assert np.array_equal(gk[0].cpu().numpy().reshape(-1), kps[0])


def test_copy_blocks_cow_step_matches_decode():
    """The per-group copy-on-write of the shared-prompt workload: poison the private copies,
    copy, and the members that read them get the oracle's attention again."""
    spec = synth.SPECS["gqa_pressure"].scaled(num_seqs=16, ctx_range=(100, 600), shared_prompt=64)
    case = synth.make_case(spec, seed=41)
    ref = oracle_decode(case)
    g = case.to("cuda")
    raw_k, raw_v = g.k_pool.view(torch.int16), g.v_pool.view(torch.int16)
    dst = g.cow_pairs[:, 1].long()
    raw_k[dst] = synth.NAN_BITS["bf16"]
    raw_v[dst] = synth.NAN_BITS["bf16"]
    pa.pa_copy_blocks([g.k_pool], [g.v_pool], g.cow_pairs)
    assert max_abs_err(gpu_decode(g), ref) <= TOL["bf16"]


@pytest.mark.parametrize("staged", [False, True])
def test_swap_round_trip(staged):
    """Swap a sequence's whole block set out to pinned memory and back into other blocks:
    the host image matches the oracle's byte for byte and decode output is unchanged."""
    spec = synth.SPECS["preemption"].scaled(num_seqs=12, ctx_range=(100, 900), shared_prompt=64,
                                            num_layers=3, victim_len=400, occupancy=0.6)
    case = synth.make_case(spec, seed=52, device="cuda", logical=False, poison=False)
    victim = spec.num_seqs - 1
    out_ids, in_ids = synth.swap_plan(case, victim, seed=3)
    bb = case.block_bytes
    n, L = len(out_ids), spec.num_layers
    before = gpu_decode(case)
    host = torch.zeros(n * L * 2 * bb, dtype=torch.uint8).pin_memory()
    staging = torch.empty(n * L * 2 * bb, dtype=torch.uint8, device="cuda") if staged else None
    pa.pa_swap_blocks(case.k_pools, case.v_pools, host, out_ids, pa.PA_SWAP_OUT, staging=staging)
    torch.cuda.synchronize()
    # oracle swap-out on host copies of the pools
    kps = [_u8(p) for p in case.k_pools]
    vps = [_u8(p) for p in case.v_pools]
    exp = np.zeros(n * L * 2 * bb, np.uint8)
    assert oracle.load().swap_blocks(kps, vps, exp, out_ids, block_bytes=bb, direction="out") == 0
    assert np.array_equal(host.numpy(), exp)
    # the released blocks are reused by someone else (the same bytes land in the GPU pools and
    # in the oracle's copies), then the victim comes back elsewhere
    for p in case.k_pools + case.v_pools:
        p.view(torch.uint8).view(case.num_blocks, -1)[torch.from_numpy(out_ids).long().cuda()] = 0x7F
    for p in kps + vps:
        p.reshape(case.num_blocks, -1)[out_ids] = 0x7F
    pa.pa_swap_blocks(case.k_pools, case.v_pools, host, in_ids, pa.PA_SWAP_IN, staging=staging)
    torch.cuda.synchronize()
    assert oracle.load().swap_blocks(kps, vps, exp, in_ids, block_bytes=bb, direction="in") == 0
    # whole pools, every layer: the restored blocks and every block the swap-in must not touch
    for l in range(L):
        np.testing.assert_array_equal(_u8(case.k_pools[l]), kps[l])
        np.testing.assert_array_equal(_u8(case.v_pools[l]), vps[l])
    bt = case.block_tables.clone()
    bt[victim, :n] = torch.from_numpy(in_ids).cuda()
    after = gpu_decode(case, block_tables=bt)
    assert torch.equal(after[victim], before[victim]), "resumed decode must be bit-identical"


def test_swap_rejects_pageable_and_bad_ids():
    spec = synth.SPECS["toy"]
    case = synth.make_case(spec, seed=2).to("cuda")
    bb = case.block_bytes
    pageable = torch.zeros(2 * 2 * bb, dtype=torch.uint8)
    with pytest.raises(pa.PaError) as e:
        pa.pa_swap_blocks([case.k_pool], [case.v_pool], pageable, [0, 1], pa.PA_SWAP_OUT)
    assert e.value.status == pa.PA_EINVAL
    pinned = pageable.pin_memory()
    with pytest.raises(pa.PaError) as e:
        pa.pa_swap_blocks([case.k_pool], [case.v_pool], pinned, [0, 9], pa.PA_SWAP_OUT)
    assert e.value.status == pa.PA_EINVAL


def test_execute_moves_matches_oracle_on_whole_pools():
    """pa_scheduler_execute_moves on a plan with scattered CPU slots: swap-outs, then swap-ins,
    then copy-on-write copies, over 3 layers. The GPU pools and the pinned CPU pool equal the
    oracle's (the same moves applied one pair at a time by its literal swap and copy formulas)
    byte for byte, untouched blocks and slots included."""
    from paged_kv_cache_38_gb300 import scheduler as sch

    orc = oracle.load()
    rng = np.random.default_rng(90)
    L, nblk, ncpu, bb = 3, 48, 20, 8 * 1024
    kps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(L)]
    vps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(L)]
    cpu = rng.integers(0, 256, ncpu * L * 2 * bb, dtype=np.uint8)
    perm = rng.permutation(nblk)
    slots = rng.permutation(ncpu)
    swap_out = np.stack([perm[:5], slots[:5]], 1).astype(np.int32)       # (block, slot)
    swap_in = np.stack([slots[5:9], perm[5:9]], 1).astype(np.int32)      # (slot, block)
    copies = np.stack([perm[9:12], perm[12:15]], 1).astype(np.int32)     # (src, dst)
    gk = [torch.from_numpy(p.copy()).cuda().view(nblk, -1) for p in kps]
    gv = [torch.from_numpy(p.copy()).cuda().view(nblk, -1) for p in vps]
    gcpu = torch.from_numpy(cpu.copy()).view(ncpu, L, 2, bb).pin_memory()
    plan = sch.Plan(*([np.zeros(0, np.int64)] + [np.zeros((0, 1), np.int32)]
                      + [np.zeros(0, np.int32)] * 3 + [np.zeros(0, np.int64)]
                      + [copies, swap_out, swap_in, [], [], 0]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    sch.execute_moves(plan, gk, gv, gcpu, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    per_slot = L * 2 * bb
    for b, c in swap_out:
        view = cpu[c * per_slot:(c + 1) * per_slot]
        assert orc.swap_blocks(kps, vps, view, [b], block_bytes=bb, direction="out") == 0
    for c, b in swap_in:
        view = cpu[c * per_slot:(c + 1) * per_slot]
        assert orc.swap_blocks(kps, vps, view, [b], block_bytes=bb, direction="in") == 0
    assert orc.copy_blocks(kps, vps, copies, block_bytes=bb) == 0
    for l in range(L):
        assert np.array_equal(gk[l].cpu().numpy().reshape(-1), kps[l])
        assert np.array_equal(gv[l].cpu().numpy().reshape(-1), vps[l])
    assert np.array_equal(gcpu.numpy().reshape(-1), cpu)


def test_execute_moves_many_pairs_across_launches():
    """More swap and copy pairs than one launch carries (1,024 per launch): 1,500 copies and
    1,100 swap-outs then 1,100 swap-ins over 2 layers equal the oracle's pools byte for byte."""
    from paged_kv_cache_38_gb300 import scheduler as sch

    orc = oracle.load()
    rng = np.random.default_rng(91)
    L, nblk, ncpu, bb = 2, 6000, 1200, 1024
    kps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(L)]
    vps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(L)]
    cpu = rng.integers(0, 256, ncpu * L * 2 * bb, dtype=np.uint8)
    perm = rng.permutation(nblk)
    slots = rng.permutation(ncpu)
    swap_out = np.stack([perm[:1100], slots[:1100]], 1).astype(np.int32)
    back = rng.permutation(1100)
    swap_in = np.stack([slots[:1100][back], perm[1100:2200]], 1).astype(np.int32)
    copies = np.stack([perm[2200:3700], perm[3700:5200]], 1).astype(np.int32)
    gk = [torch.from_numpy(p.copy()).cuda().view(nblk, -1) for p in kps]
    gv = [torch.from_numpy(p.copy()).cuda().view(nblk, -1) for p in vps]
    gcpu = torch.from_numpy(cpu.copy()).view(ncpu, L, 2, bb).pin_memory()
    plan = sch.Plan(*([np.zeros(0, np.int64)] + [np.zeros((0, 1), np.int32)]
                      + [np.zeros(0, np.int32)] * 3 + [np.zeros(0, np.int64)]
                      + [copies, swap_out, swap_in, [], [], 0]))
    sch.execute_moves(plan, gk, gv, gcpu)
    torch.cuda.synchronize()
    per_slot = L * 2 * bb
    for b, c in swap_out:
        assert orc.swap_blocks(kps, vps, cpu[c * per_slot:(c + 1) * per_slot], [b], block_bytes=bb,
                               direction="out") == 0
    for c, b in swap_in:
        assert orc.swap_blocks(kps, vps, cpu[c * per_slot:(c + 1) * per_slot], [b], block_bytes=bb,
                               direction="in") == 0
    assert orc.copy_blocks(kps, vps, copies, block_bytes=bb) == 0
    for l in range(L):
        assert np.array_equal(gk[l].cpu().numpy().reshape(-1), kps[l])
        assert np.array_equal(gv[l].cpu().numpy().reshape(-1), vps[l])
    assert np.array_equal(gcpu.numpy().reshape(-1), cpu)
