"""Stream semantics: CUDA-graph capture/replay and inputs produced by copies just before the call."""
import pytest
import torch

import synth
from helpers import TOL, max_abs_err, oracle_decode

pytestmark = pytest.mark.gpu

import paged_kv_cache_38_gb300 as pa  # noqa: E402


def _step(case, ws, out):
    pa.pa_write_kv(case.k_new, case.v_new, case.k_pool, case.v_pool, case.slot_mapping)
    pa.pa_copy_blocks([case.k_pool], [case.v_pool], case.cow_pairs)
    return pa.pa_decode(case.q, case.k_pool, case.v_pool, case.block_tables, case.ctx_lens,
                        case.scale, out=out, workspace=ws, split_tokens=64)


def test_graph_replay_matches_eager_bitwise():
    spec = synth.SPECS["gqa_pressure"].scaled(num_seqs=12, ctx_range=(40, 600), shared_prompt=64)
    case = synth.make_case(spec, seed=61).to("cuda")
    ws = torch.empty(1 << 24, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(case.q)
    eager = _step(case, ws, out).clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _step(case, ws, out)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _step(case, ws, out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)
    assert max_abs_err(eager, oracle_decode(case)) <= TOL["bf16"]


def test_inputs_copied_from_host_right_before_the_call():
    spec = synth.SPECS["fp8_long"].scaled(num_seqs=8, ctx_range=(100, 3000))
    host = synth.make_case(spec, seed=62)
    dev = host.to("cuda")
    q_pinned = host.q.pin_memory()
    bt_pinned = host.block_tables.pin_memory()
    cl_pinned = host.ctx_lens.pin_memory()
    q = torch.empty_like(dev.q)
    bt = torch.empty_like(dev.block_tables)
    cl = torch.empty_like(dev.ctx_lens)
    ref = oracle_decode(host)
    for _ in range(3):
        q.zero_(); bt.fill_(-1); cl.zero_()
        q.copy_(q_pinned, non_blocking=True)
        bt.copy_(bt_pinned, non_blocking=True)
        cl.copy_(cl_pinned, non_blocking=True)
        out = pa.pa_decode(q, dev.k_pool, dev.v_pool, bt, cl, dev.scale, k_scale=dev.k_scale,
                           v_scale=dev.v_scale, split_tokens=256)
        res = out.cpu()
        assert max_abs_err(res, ref) <= TOL["e4m3"]
