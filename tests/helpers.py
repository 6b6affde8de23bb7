"""Shared helpers for the GPU parity tests: run the CUDA path and the oracle on the same inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

# Maximum absolute error allowed against the fp64 oracle, per KV storage dtype.
TOL = {"f16": 2e-3, "bf16": 1e-2, "e4m3": 3e-2}


def gpu_available() -> bool:
    return torch.cuda.is_available()


def oracle_decode(case: synth.PagedCase, seqs=None, *, k_pool=None, v_pool=None,
                  block_tables=None, ctx_lens=None) -> np.ndarray:
    """fp64 oracle output for all (or the listed) sequences of ``case`` (inputs read on host)."""
    spec = case.spec
    q = case.q.cpu()
    bt = (case.block_tables if block_tables is None else block_tables).cpu()
    cl = (case.ctx_lens if ctx_lens is None else ctx_lens).cpu()
    if seqs is not None:
        idx = torch.as_tensor(seqs, dtype=torch.long)
        q, bt, cl = q[idx], bt[idx], cl[idx]
    kp = (case.k_pool if k_pool is None else k_pool).cpu()
    vp = (case.v_pool if v_pool is None else v_pool).cpu()
    return oracle.load().decode(q, kp, vp, bt, cl, q_dtype=spec.q_dtype, kv_dtype=spec.kv_dtype,
                                num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                                head_dim=spec.head_dim, block_size=spec.block_size,
                                scale=case.scale, k_scale=case.k_scale, v_scale=case.v_scale)


def gpu_decode(case: synth.PagedCase, *, split_tokens: int = 0, err_flag=None,
               block_tables=None, ctx_lens=None, k_pool=None, v_pool=None, max_ctx_len=None):
    import paged_kv_cache_38_gb300 as pa

    bt = case.block_tables if block_tables is None else block_tables
    return pa.pa_decode(case.q, case.k_pool if k_pool is None else k_pool,
                        case.v_pool if v_pool is None else v_pool, bt,
                        case.ctx_lens if ctx_lens is None else ctx_lens, case.scale,
                        k_scale=case.k_scale, v_scale=case.v_scale, split_tokens=split_tokens,
                        err_flag=err_flag, max_ctx_len=max_ctx_len)


def max_abs_err(gpu_out: torch.Tensor, ref: np.ndarray) -> float:
    g = gpu_out.detach().double().cpu().numpy()
    if not np.all(np.isfinite(g)):
        return float("inf")
    return float(np.abs(g - ref).max()) if g.size else 0.0
