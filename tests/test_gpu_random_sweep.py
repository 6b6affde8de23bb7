"""Seeded random sweeps of pa_decode, pa_prefill and the block movers against the oracle.

Beside the hand-picked geometries of test_gpu_decode.py and test_gpu_prefill.py, each sweep
draws every supported shape parameter at random (group size, kv heads, head_dim, block size,
KV and query dtype, number of sequences, context lengths, decode split, prefill chunk mix), so
that combinations nobody listed are checked too. The draws are seeded: a failure names a case
that reproduces.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL, gpu_decode, max_abs_err, oracle_decode

import paged_kv_cache_38_gb300 as pa  # noqa: E402

pytestmark = pytest.mark.gpu


def _draw(rng, *, prefill: bool):
    g = int(rng.choice([1, 2, 4, 8, 16]))
    hkv = int(rng.choice([h for h in (1, 2, 4, 8) if g * h <= 32]))
    d = int(rng.choice([64, 128]))
    blocks = [8, 16, 32, 64] if prefill else [4, 8, 16, 32, 64]
    b = int(rng.choice(blocks))
    kv_choices = ["f16", "bf16", "e4m3"] if d == 128 else ["f16", "bf16"]  # E4M3: head_dim 128
    kv = str(rng.choice(kv_choices))
    qd = (("bf16" if rng.random() < 0.5 else "f16") if kv == "e4m3" else kv)
    nseq = int(rng.integers(1, 13 if prefill else 41))
    maxctx = int(rng.choice([40, 130, 300, 500] if prefill else [20, 200, 900, 2000]))
    return g, hkv, d, b, kv, qd, nseq, maxctx


@pytest.mark.parametrize("i", range(40))
def test_decode_random_geometry(i):
    rng = np.random.default_rng(5000 + i)
    g, hkv, d, b, kv, qd, nseq, maxctx = _draw(rng, prefill=False)
    spec = synth.DecodeSpec(f"sweep{i}", nseq, g * hkv, hkv, d, b, kv, qd, ctx_range=(0, maxctx))
    unit = max(16, b)
    split = 0 if rng.random() < 0.5 else unit * int(rng.integers(1, 9))
    case = synth.make_case(spec, seed=6000 + i).to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(case, split_tokens=split, err_flag=err)
    torch.cuda.synchronize()
    e = max_abs_err(out, oracle_decode(case))
    assert int(err.item()) == 0
    assert e <= TOL[kv], f"G={g} Hkv={hkv} D={d} B={b} kv={kv} q={qd} seqs={nseq} split={split}: {e}"


@pytest.mark.parametrize("i", range(40))
def test_prefill_random_geometry(i):
    rng = np.random.default_rng(7000 + i)
    g, hkv, d, b, kv, qd, nseq, maxctx = _draw(rng, prefill=True)
    spec = synth.DecodeSpec(f"sweep{i}", nseq, g * hkv, hkv, d, b, kv, qd, ctx_range=(1, maxctx))
    case = synth.make_case(spec, seed=8000 + i)
    mode = int(rng.integers(0, 3))  # whole prompts, one-token chunks, or random chunks
    qs, q = synth.prefill_queries(case, seed=i, whole=mode == 0,
                                  max_chunk=1 if mode == 1 else None)
    ref = oracle.load().prefill(q, case.k_pool, case.v_pool, case.block_tables, case.ctx_lens, qs,
                                dtype=kv, q_dtype=qd, num_q_heads=spec.num_q_heads,
                                num_kv_heads=hkv, head_dim=d, block_size=b, scale=case.scale,
                                k_scale=case.k_scale, v_scale=case.v_scale)
    gc = case.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pa.pa_prefill(q.cuda(), gc.k_pool, gc.v_pool, gc.block_tables, gc.ctx_lens, qs.cuda(),
                        case.scale, err_flag=err, k_scale=case.k_scale, v_scale=case.v_scale)
    torch.cuda.synchronize()
    e = max_abs_err(out, ref)
    assert int(err.item()) == 0
    assert e <= TOL[kv], f"G={g} Hkv={hkv} D={d} B={b} kv={kv} q={qd} seqs={nseq} mode={mode}: {e}"


def _u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.uint8).cpu().numpy().copy()


_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def _fp8_codes_agree(got: np.ndarray, exp: np.ndarray) -> bool:
    """Equal codes, except that where the oracle wrote its NaN code either NaN code is fine."""
    nan = exp == 0x7F
    return np.array_equal(got[~nan], exp[~nan]) and bool(np.all((got[nan] & 0x7F) == 0x7F))


@pytest.mark.parametrize("i", range(10))
def test_movers_random_geometry(i):
    """pa_write_kv, pa_write_kv_fp8 (with saturating, infinite, NaN and subnormal inputs),
    pa_copy_blocks and pa_swap_blocks (out, blocks reused, back into other blocks; direct or
    staged) at random geometries: whole pools and the host image equal the oracle's byte for
    byte."""
    orc = oracle.load()
    rng = np.random.default_rng(9000 + i)
    g = torch.Generator().manual_seed(9000 + i)
    # write_kv: any head_dim with 16-byte rows, any block size, padding slots
    dt = str(rng.choice(["f16", "bf16"]))
    D, H = 8 * int(rng.integers(1, 33)), int(rng.integers(1, 17))
    B, ntok = int(rng.choice([1, 3, 4, 8, 12, 16, 32, 64])), int(rng.integers(1, 6001))
    nblk = ntok // B + int(rng.integers(1, 21))
    k = torch.randn(ntok, H, D, generator=g).to(_DT[dt])
    v = torch.randn(ntok, H, D, generator=g).to(_DT[dt])
    slots = torch.from_numpy(rng.permutation(nblk * B)[:ntok].astype(np.int64))
    slots[torch.from_numpy(rng.random(ntok) < 0.05)] = -1
    raw = lambda: torch.from_numpy(rng.integers(0, 256, nblk * H * B * D * 2, dtype=np.uint8))
    kp, vp = raw().view(_DT[dt]).view(nblk, H, B, D), raw().view(_DT[dt]).view(nblk, H, B, D)
    ek, ev = _u8(kp), _u8(vp)
    assert orc.write_kv(k, v, ek, ev, slots, num_kv_heads=H, head_dim=D, block_size=B,
                        kv_dtype=dt) == 0
    gk, gv = kp.cuda(), vp.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_write_kv(k.cuda(), v.cuda(), gk, gv, slots.cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(_u8(gk), ek) and np.array_equal(_u8(gv), ev), ("write_kv", dt, D, H, B)
    # write_kv_fp8: magnitudes from 1e-3 to 1e3 against scales from 1e-4 to 1e3
    src = str(rng.choice(["f16", "bf16"]))
    D, H = 16 * int(rng.integers(1, 17)), int(rng.integers(1, 17))
    B, ntok = int(rng.choice([1, 3, 4, 8, 12, 16, 32, 64])), int(rng.integers(1, 4001))
    nblk = ntok // B + int(rng.integers(1, 21))
    mag = float(10 ** rng.uniform(-3, 3))
    kf = torch.randn(ntok, H, D, generator=g) * mag
    vf = torch.randn(ntok, H, D, generator=g) * mag
    for val in (float("inf"), float("-inf"), float("nan"), 1e-30, -1e-30, 0.0, -0.0):
        kf.view(-1)[int(rng.integers(0, kf.numel()))] = val
    k, v = kf.to(_DT[src]), vf.to(_DT[src])
    ks, vs = float(10 ** rng.uniform(-4, 3)), float(10 ** rng.uniform(-4, 3))
    slots = torch.from_numpy(rng.permutation(nblk * B)[:ntok].astype(np.int64))
    slots[torch.from_numpy(rng.random(ntok) < 0.05)] = -1
    kp = torch.from_numpy(rng.integers(0, 256, (nblk, H, B, D), dtype=np.uint8))
    vp = torch.from_numpy(rng.integers(0, 256, (nblk, H, B, D), dtype=np.uint8))
    ek, ev = _u8(kp), _u8(vp)
    assert orc.write_kv_fp8(k, v, ek, ev, slots, src_dtype=src, num_kv_heads=H, head_dim=D,
                            block_size=B, k_scale=ks, v_scale=vs) == 0
    gk, gv = kp.cuda(), vp.cuda()
    pa.pa_write_kv_fp8(k.cuda(), v.cuda(), gk, gv, slots.cuda(), ks, vs, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _fp8_codes_agree(_u8(gk), ek) and _fp8_codes_agree(_u8(gv), ev), ("fp8", src, D, H, B)
    # copy_blocks: up to 6 layers, disjoint pairs (sometimes more than one launch's worth)
    L, bb, nblk = int(rng.integers(1, 7)), 16 * int(rng.integers(1, 4097)), int(rng.integers(2, 301))
    P = int(rng.integers(1, nblk // 2 + 1))
    if rng.random() < 0.3:
        nblk, bb = int(rng.integers(2100, 6001)), 16 * int(rng.integers(1, 65))
        P = int(rng.integers(1025, nblk // 2 + 1))
    kps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(L)]
    vps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(L)]
    perm = rng.permutation(nblk)
    pairs = np.stack([perm[:P], perm[P:2 * P]], axis=1).astype(np.int32)
    gk = [torch.from_numpy(p.copy()).cuda().view(nblk, -1) for p in kps]
    gv = [torch.from_numpy(p.copy()).cuda().view(nblk, -1) for p in vps]
    assert orc.copy_blocks(kps, vps, pairs, block_bytes=bb) == 0
    pa.pa_copy_blocks(gk, gv, torch.from_numpy(pairs).cuda(), err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in range(L):
        assert np.array_equal(gk[l].cpu().numpy().reshape(-1), kps[l]), ("copy", L, bb, P)
        assert np.array_equal(gv[l].cpu().numpy().reshape(-1), vps[l]), ("copy", L, bb, P)
    # swap_blocks: out, the blocks reused, back in elsewhere
    L, bb, nblk = int(rng.integers(1, 5)), 16 * int(rng.integers(1, 2049)), int(rng.integers(4, 401))
    n = int(rng.integers(1, nblk // 2 + 1))
    perm = rng.permutation(nblk)
    out_ids, in_ids = perm[:n].astype(np.int32), perm[n:2 * n].astype(np.int32)
    kps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(L)]
    vps = [rng.integers(0, 256, nblk * bb, dtype=np.uint8) for _ in range(L)]
    gk = [torch.from_numpy(p.copy()).cuda().view(nblk, bb) for p in kps]
    gv = [torch.from_numpy(p.copy()).cuda().view(nblk, bb) for p in vps]
    host = torch.zeros(n * L * 2 * bb, dtype=torch.uint8).pin_memory()
    staging = (torch.empty(n * L * 2 * bb, dtype=torch.uint8, device="cuda")
               if rng.random() < 0.5 else None)
    pa.pa_swap_blocks(gk, gv, host, out_ids, pa.PA_SWAP_OUT, staging=staging)
    torch.cuda.synchronize()
    exp = np.zeros(n * L * 2 * bb, np.uint8)
    assert orc.swap_blocks(kps, vps, exp, out_ids, block_bytes=bb, direction="out") == 0
    assert np.array_equal(host.numpy(), exp), ("swap out", L, bb, n, staging is not None)
    for p in gk + gv:
        p[torch.from_numpy(out_ids).long().cuda()] = 0x5A
    for p in kps + vps:
        p.reshape(nblk, -1)[out_ids] = 0x5A
    pa.pa_swap_blocks(gk, gv, host, in_ids, pa.PA_SWAP_IN, staging=staging)
    torch.cuda.synchronize()
    assert orc.swap_blocks(kps, vps, exp, in_ids, block_bytes=bb, direction="in") == 0
    for l in range(L):
        assert np.array_equal(gk[l].cpu().numpy().reshape(-1), kps[l]), ("swap in", L, bb, n)
        assert np.array_equal(gv[l].cpu().numpy().reshape(-1), vps[l]), ("swap in", L, bb, n)
