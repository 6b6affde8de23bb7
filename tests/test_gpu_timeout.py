"""Bounded waits that run out: the kernels give up cleanly and the next call is correct.

Every wait of one warp, role or CTA on another inside pa_decode and pa_prefill is bounded
("When KV Capacity Runs Out", Figure 4: a transfer must be known complete before its blocks are
reused, so no kernel may leave copies in flight). pa_testing_set_wait_limit shortens those waits
and makes one CTA withhold its part, so that the others' waits expire for certain. Each test
then checks that the call returns, PA_ERR_TIMEOUT is set, the CUDA context is still usable, the
decode work counters were left cleared, and a normal call straight after (eager and from a CUDA
graph captured before the failure) matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL, max_abs_err, oracle_decode

import paged_kv_cache_38_gb300 as pa  # noqa: E402

pytestmark = pytest.mark.gpu

SHORT_NS = 200_000  # 200 us: far longer than any wait of these small cases, far below 1 s
# A launch that gave up under the shortened limit returns well before the one-second default
# could have expired once (the kernel is loaded and warm before any timed call).
FAST_S = 0.9


@pytest.fixture(autouse=True)
def default_wait_limit():
    pa.pa_testing_set_wait_limit(0, -1)
    yield
    pa.pa_testing_set_wait_limit(0, -1)


def _decode(case, ws, out, err):
    return pa.pa_decode(case.q, case.k_pool, case.v_pool, case.block_tables, case.ctx_lens,
                        case.scale, out=out, k_scale=case.k_scale, v_scale=case.v_scale,
                        workspace=ws, err_flag=err, split_tokens=64)


@pytest.mark.parametrize("name", ["gqa_pressure", "mha7b"])
def test_decode_grid_barrier_wait_expires(name):
    spec = synth.SPECS[name].scaled(num_seqs=12, ctx_range=(40, 700),
                                    shared_prompt=64 if synth.SPECS[name].shared_prompt else 0)
    case = synth.make_case(spec, seed=81).to("cuda")
    ref = oracle_decode(case)
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(case.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")

    # a graph of a normal call, captured before the failing call
    _decode(case, ws, out, err)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _decode(case, ws, out, err)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _decode(case, ws, out, err)
    torch.cuda.synchronize()

    # CTA 0 withholds its grid-barrier arrival: every CTA's barrier wait must run out
    pa.pa_testing_set_wait_limit(SHORT_NS, 0)
    for _ in range(2):
        err.zero_()
        out.fill_(float("nan"))
        t0 = time.perf_counter()
        _decode(case, ws, out, err)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
        assert int(err.item()) & pa.PA_ERR_TIMEOUT
        assert elapsed < FAST_S, f"the shortened limit was not applied ({elapsed:.3f} s)"
        # the last CTA to finish cleared the three work counters even though the launch gave up
        assert int(ws[:24].count_nonzero().item()) == 0

    pa.pa_testing_set_wait_limit(0, -1)
    err.zero_()
    res = _decode(case, ws, out, err).clone()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert max_abs_err(res, ref) <= TOL[spec.kv_dtype]
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(out, res)


def _prefill_case():
    spec = synth.DecodeSpec("pf_timeout", 6, 32, 8, 128, 16, "bf16", "bf16", ctx_range=(200, 900))
    case = synth.make_case(spec, seed=83)
    qs, q = synth.prefill_queries(case, seed=9, whole=True)
    ref = oracle.load().prefill(q, case.k_pool, case.v_pool, case.block_tables, case.ctx_lens,
                                qs, dtype="bf16", num_q_heads=32, num_kv_heads=8, head_dim=128,
                                block_size=16, scale=case.scale)
    return case.to("cuda"), qs.cuda(), q.cuda(), ref


def _prefill(g, qs, q, err):
    return pa.pa_prefill(q, g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qs, g.scale,
                         err_flag=err)


def _prefill_err(out, ref):
    o = out.double().cpu().numpy()
    return float(np.abs(o - ref).max()) if np.all(np.isfinite(o)) else float("inf")


def test_prefill_waits_expire_when_mma_issuer_stalls():
    """CTA 0's MMA issuer stops after its first S group: its softmax warps, K/V producers and
    query loader wait in vain and give up; the issuer's MMAs drain through a last commit and the
    CTA frees its tensor memory before returning."""
    g, qs, q, ref = _prefill_case()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    _prefill(g, qs, q, err)  # load and warm the kernel before anything is timed
    torch.cuda.synchronize()
    pa.pa_testing_set_wait_limit(SHORT_NS, 0)
    for _ in range(2):
        err.zero_()
        t0 = time.perf_counter()
        _prefill(g, qs, q, err)
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < FAST_S
        assert int(err.item()) & pa.PA_ERR_TIMEOUT
    pa.pa_testing_set_wait_limit(0, -1)
    err.zero_()
    out = _prefill(g, qs, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _prefill_err(out, ref) <= TOL["bf16"]
