"""Calls on separate streams at the same time: two decodes (each with its own workspace) and a
prefill give the same bits as the same calls made one after another. The library keeps no state
that concurrent calls on different streams could share, beyond what pa.h documents."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import synth

import paged_kv_cache_38_gb300 as pa  # noqa: E402

pytestmark = pytest.mark.gpu


def _decode(c, stream, ws):
    with torch.cuda.stream(stream):
        return pa.pa_decode(c.q, c.k_pool, c.v_pool, c.block_tables, c.ctx_lens, c.scale,
                            k_scale=c.k_scale, v_scale=c.v_scale, workspace=ws, stream=stream)


def _prefill(c, qs, q, stream):
    with torch.cuda.stream(stream):
        return pa.pa_prefill(q, c.k_pool, c.v_pool, c.block_tables, c.ctx_lens, qs, c.scale,
                             stream=stream)


@pytest.mark.parametrize("i", range(5))
def test_concurrent_streams_bit_identical(i):
    rng = np.random.default_rng(31000 + i)
    cases = []
    for j in range(2):
        g, hkv = int(rng.choice([1, 4, 8])), int(rng.choice([2, 4, 8]))
        kv = str(rng.choice(["bf16", "e4m3"]))
        spec = synth.DecodeSpec(f"st{i}_{j}", int(rng.integers(20, 200)), g * hkv, hkv, 128,
                                int(rng.choice([8, 16, 32])), kv, "bf16",
                                ctx_range=(1, int(rng.choice([500, 3000]))))
        cases.append(synth.make_case(spec, seed=31500 + 2 * i + j, device="cuda", logical=False))
    spec = synth.DecodeSpec(f"stp{i}", int(rng.integers(2, 8)), 32, 8, 128, 16, "bf16", "bf16",
                            ctx_range=(200, 1500))
    pc = synth.make_case(spec, seed=31900 + i, device="cuda", logical=False)
    qs, q = synth.prefill_queries(pc, seed=i)
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ws1 = torch.empty(1 << 27, dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(1 << 27, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    # references one call at a time (each finished before its result is copied)
    refs = []
    for call in (lambda: _decode(cases[0], s1, ws1), lambda: _decode(cases[1], s1, ws2),
                 lambda: _prefill(pc, qs, q, s1)):
        r = call()
        torch.cuda.synchronize()
        refs.append(r.clone())
    a1, a2, ap = refs
    for _ in range(3):
        b1 = _decode(cases[0], s1, ws1)
        b2 = _decode(cases[1], s2, ws2)
        bp = _prefill(pc, qs, q, s3)
        torch.cuda.synchronize()
        assert torch.equal(a1, b1) and torch.equal(a2, b2) and torch.equal(ap, bp)
