"""Seeded random sweeps of pa_decode and pa_prefill geometries against the fp64 oracle.

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
