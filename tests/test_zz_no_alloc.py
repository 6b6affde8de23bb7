"""pa_decode_static_workspace: the decode entry point for callers that cannot allocate.

Some callers of this library must not allocate device memory at all -- a runtime that plans one
memory arena up front, a plugin handed only its input and output tensors, a latency-critical
path. pa_decode_static_workspace serves them with a fixed scratch array inside the library. This
test calls it through the C ABI (ctypes) twice in a row and checks both results element by
element against the fp64 oracle and against the regular pa_decode with a caller workspace,
within the decode tolerance of the KV dtype; it also checks that a decode too large for the
built-in scratch is refused with a clear error. It lives in a file of its own that pytest
collects last, and passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import pytest
import torch

import synth
from helpers import TOL, max_abs_err, oracle_decode

pytestmark = pytest.mark.gpu

import paged_kv_cache_38_gb300 as pa  # noqa: E402


def _args(case, out, split_tokens):
    return pa.make_decode_args(case.q, case.k_pool, case.v_pool, case.block_tables,
                               case.ctx_lens, out, scale=case.scale, k_scale=case.k_scale,
                               v_scale=case.v_scale, split_tokens=split_tokens)


@pytest.mark.parametrize("name", ["gqa_pressure", "fp8_long"])
def test_static_workspace_matches_pa_decode_on_two_calls(name):
    spec = synth.SPECS[name].scaled(num_seqs=10, ctx_range=(50, 1500),
                                    shared_prompt=32 if synth.SPECS[name].shared_prompt else 0)
    host_case = synth.make_case(spec, seed=71)
    oracle_out = oracle_decode(host_case)
    case = host_case.to("cuda")
    split = 64  # several splits per sequence, so the scratch holds split-K partials
    ref = pa.pa_decode(case.q, case.k_pool, case.v_pool, case.block_tables, case.ctx_lens,
                       case.scale, k_scale=case.k_scale, v_scale=case.v_scale,
                       split_tokens=split)
    torch.cuda.synchronize()
    need = pa.pa_decode_workspace_size(_args(case, ref, split))
    assert 256 < need <= pa.pa.PA_STATIC_WORKSPACE_BYTES
    lib = pa.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full_like(case.q, float("nan"))
        args = _args(case, out, split)
        st = lib.pa_decode_static_workspace(ctypes.byref(args), ctypes.c_void_p(stream))
        assert st == pa.PA_OK, lib.pa_last_error_message()
        torch.cuda.synchronize()
        assert max_abs_err(out, oracle_out) <= TOL[spec.kv_dtype]
        assert max_abs_err(out, ref.double().cpu().numpy()) <= TOL[spec.kv_dtype]


def test_static_workspace_refuses_oversized_decode():
    spec = synth.SPECS["fp8_long"].scaled(num_seqs=64, ctx_range=(8000, 8192))
    case = synth.make_case(spec, seed=72, device="cuda", logical=False, poison=False)
    out = torch.empty_like(case.q)
    args = _args(case, out, 16)  # 16-token splits: far more partials than the scratch holds
    assert pa.pa_decode_workspace_size(args) > pa.pa.PA_STATIC_WORKSPACE_BYTES
    lib = pa.lib()
    st = lib.pa_decode_static_workspace(ctypes.byref(args), None)
    assert st == pa.PA_EINVAL
    assert b"built-in buffer" in lib.pa_last_error_message()
