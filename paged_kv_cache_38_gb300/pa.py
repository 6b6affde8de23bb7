"""Python binding of libpa (include/pa.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does nothing but turn torch
tensors (device memory, pinned host memory) and Python numbers into the C arguments; all work
runs in the library's CUDA kernels on the caller's current stream. A missing or unloadable
library raises -- there is no other code path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

PA_OK, PA_EINVAL, PA_EUNSUPPORTED, PA_ECUDA, PA_ENOSPACE = 0, 1, 2, 3, 4
PA_F16, PA_BF16, PA_FP8_E4M3 = 0, 1, 2
PA_SWAP_OUT, PA_SWAP_IN = 0, 1
PA_ERR_BLOCK_ID, PA_ERR_CTX_LEN, PA_ERR_TIMEOUT = 1, 2, 4
PA_STATIC_WORKSPACE_BYTES = 16 * 1024 * 1024

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32


class pa_decode_args(ctypes.Structure):
    """Mirror of ``struct pa_decode_args`` (field order and types as in include/pa.h)."""

    _fields_ = [
        ("q", _vp), ("k_pool", _vp), ("v_pool", _vp), ("block_tables", _vp), ("ctx_lens", _vp),
        ("out", _vp),
        ("num_seqs", _i32), ("num_q_heads", _i32), ("num_kv_heads", _i32), ("head_dim", _i32),
        ("block_size", _i32), ("num_blocks", _i32), ("max_blocks_per_seq", _i32),
        ("max_ctx_len", _i32), ("split_tokens", _i32),
        ("q_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int),
        ("scale", ctypes.c_float), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("err_flag", _vp),
    ]


class PaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{message} (status {status})")
        self.status = status


_LIB: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIBRARY


def lib() -> ctypes.CDLL:
    """The loaded libpa (built in-tree first if a source is newer than it)."""
    global _LIB
    if _LIB is None:
        path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"libpa.so not found at {path}")
        L = ctypes.CDLL(path)
        L.pa_decode_workspace_size.restype = ctypes.c_size_t
        L.pa_decode_workspace_size.argtypes = [ctypes.POINTER(pa_decode_args)]
        L.pa_decode.restype = ctypes.c_int
        L.pa_decode.argtypes = [ctypes.POINTER(pa_decode_args), _vp]
        L.pa_write_kv.restype = ctypes.c_int
        L.pa_write_kv.argtypes = [_vp] * 5 + [_i32] * 5 + [ctypes.c_int, _vp, _vp]
        L.pa_prefill.restype = ctypes.c_int
        L.pa_prefill.argtypes = [ctypes.POINTER(pa_prefill_args), _vp]
        L.pa_write_kv_fp8.restype = ctypes.c_int
        L.pa_write_kv_fp8.argtypes = [_vp, _vp, ctypes.c_int, _vp, _vp, _vp] + [_i32] * 5 + [
            ctypes.c_float, ctypes.c_float, _vp, _vp]
        L.pa_copy_blocks.restype = ctypes.c_int
        L.pa_copy_blocks.argtypes = [_vp, _vp, _i32, _vp, _i32, _i32, ctypes.c_size_t, _vp, _vp]
        L.pa_swap_blocks.restype = ctypes.c_int
        L.pa_swap_blocks.argtypes = [_vp, _vp, _i32, _vp, _vp, _i32, _i32, ctypes.c_size_t,
                                     ctypes.c_int, _vp, ctypes.c_size_t, _vp]
        L.pa_decode_static_workspace.restype = ctypes.c_int
        L.pa_decode_static_workspace.argtypes = [ctypes.POINTER(pa_decode_args), _vp]
        L.pa_testing_set_wait_limit.restype = ctypes.c_int
        L.pa_testing_set_wait_limit.argtypes = [ctypes.c_uint64, _i32]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_status_string.argtypes = [ctypes.c_int]
        L.pa_last_error_message.restype = ctypes.c_char_p
        L.pa_last_error_message.argtypes = []
        _LIB = L
    return _LIB


def _check(status: int) -> None:
    if status != PA_OK:
        msg = lib().pa_last_error_message().decode() or lib().pa_status_string(status).decode()
        raise PaError(status, msg)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def kv_dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return PA_FP8_E4M3
    raise ValueError(f"unsupported KV dtype {t.dtype}")


def q_dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise ValueError(f"unsupported query dtype {t.dtype}")


def make_decode_args(q, k_pool, v_pool, block_tables, ctx_lens, out, *, scale: float,
                     k_scale: float = 1.0, v_scale: float = 1.0, max_ctx_len: Optional[int] = None,
                     split_tokens: int = 0, workspace: Optional[torch.Tensor] = None,
                     err_flag: Optional[torch.Tensor] = None) -> pa_decode_args:
    """Fill a ``pa_decode_args`` from tensors (shapes as in include/pa.h)."""
    n, hq, d = q.shape
    nblk, hkv, bsz, d2 = k_pool.shape
    if max_ctx_len is None:
        max_ctx_len = block_tables.shape[1] * bsz
    a = pa_decode_args()
    a.q, a.k_pool, a.v_pool = _ptr(q), _ptr(k_pool), _ptr(v_pool)
    a.block_tables, a.ctx_lens, a.out = _ptr(block_tables), _ptr(ctx_lens), _ptr(out)
    a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim = n, hq, hkv, d
    a.block_size, a.num_blocks = bsz, nblk
    a.max_blocks_per_seq = block_tables.shape[1] if block_tables.dim() == 2 else 0
    a.max_ctx_len, a.split_tokens = int(max_ctx_len), int(split_tokens)
    a.q_dtype, a.kv_dtype = q_dtype_code(q), kv_dtype_code(k_pool)
    a.scale, a.k_scale, a.v_scale = float(scale), float(k_scale), float(v_scale)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.err_flag = _ptr(err_flag)
    return a


def pa_decode_workspace_size(args: pa_decode_args) -> int:
    """Bytes of split-K workspace the call described by ``args`` needs (0: none)."""
    return int(lib().pa_decode_workspace_size(ctypes.byref(args)))


def pa_decode(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
              block_tables: torch.Tensor, ctx_lens: torch.Tensor, scale: float, *,
              out: Optional[torch.Tensor] = None, k_scale: float = 1.0, v_scale: float = 1.0,
              max_ctx_len: Optional[int] = None, split_tokens: int = 0,
              workspace: Optional[torch.Tensor] = None, err_flag: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    """Paged decode attention; returns ``out`` [num_seqs][num_q_heads][head_dim] (q dtype)."""
    if out is None:
        out = torch.empty_like(q)
    args = make_decode_args(q, k_pool, v_pool, block_tables, ctx_lens, out, scale=scale,
                            k_scale=k_scale, v_scale=v_scale, max_ctx_len=max_ctx_len,
                            split_tokens=split_tokens, workspace=workspace, err_flag=err_flag)
    if workspace is None:
        need = pa_decode_workspace_size(args)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            args.workspace, args.workspace_bytes = workspace.data_ptr(), need
    _check(lib().pa_decode(ctypes.byref(args), _stream(stream)))
    return out


def pa_decode_static_workspace(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                               block_tables: torch.Tensor, ctx_lens: torch.Tensor, scale: float,
                               *, out: Optional[torch.Tensor] = None, k_scale: float = 1.0,
                               v_scale: float = 1.0, max_ctx_len: Optional[int] = None,
                               split_tokens: int = 0, err_flag: Optional[torch.Tensor] = None,
                               stream=None) -> torch.Tensor:
    """pa_decode using the library's built-in scratch instead of a caller workspace, for callers
    that must not allocate device memory. ``out`` should be passed in by such callers; it is
    created here only for convenience when omitted."""
    if out is None:
        out = torch.empty_like(q)
    args = make_decode_args(q, k_pool, v_pool, block_tables, ctx_lens, out, scale=scale,
                            k_scale=k_scale, v_scale=v_scale, max_ctx_len=max_ctx_len,
                            split_tokens=split_tokens, err_flag=err_flag)
    _check(lib().pa_decode_static_workspace(ctypes.byref(args), _stream(stream)))
    return out


class pa_prefill_args(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p), ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("block_tables", ctypes.c_void_p), ("ctx_lens", ctypes.c_void_p),
        ("q_starts", ctypes.c_void_p), ("out", ctypes.c_void_p), ("num_seqs", ctypes.c_int32),
        ("num_tokens", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32), ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32), ("max_q_len", ctypes.c_int32),
        ("dtype", ctypes.c_int), ("scale", ctypes.c_float), ("err_flag", ctypes.c_void_p),
        ("work_counter", ctypes.c_void_p), ("kv_dtype", ctypes.c_int),
        ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
    ]


def pa_prefill(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
               block_tables: torch.Tensor, ctx_lens: torch.Tensor, q_starts: torch.Tensor,
               scale: float, *, out: Optional[torch.Tensor] = None,
               max_q_len: Optional[int] = None, err_flag: Optional[torch.Tensor] = None,
               work_counter: Optional[torch.Tensor] = None, dynamic: bool = True,
               k_scale: float = 1.0, v_scale: float = 1.0, stream=None) -> torch.Tensor:
    """Causal attention of each sequence's chunk of query tokens (rows q_starts[s] ..
    q_starts[s + 1] - 1 of q [num_tokens][num_q_heads][head_dim]) over its paged cache.

    Pools of uint8 (or float8_e4m3fn) are an E4M3 cache read as value x k_scale / v_scale;
    otherwise they have the query dtype. dynamic: the persistent CTAs take work items from an
    int32 counter (work_counter, or one allocated for the call); False assigns them
    round-robin."""
    if out is None:
        out = torch.empty_like(q)
    dt = {torch.float16: PA_F16, torch.bfloat16: PA_BF16}.get(q.dtype)
    if dt is None:
        raise PaError(PA_EINVAL, "q must be float16 or bfloat16")
    if max_q_len is None:
        max_q_len = int((q_starts[1:] - q_starts[:-1]).max().item()) if q_starts.numel() > 1 else 0
    a = pa_prefill_args()
    a.q, a.k_pool, a.v_pool = q.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr()
    a.block_tables, a.ctx_lens = block_tables.data_ptr(), ctx_lens.data_ptr()
    a.q_starts, a.out = q_starts.data_ptr(), out.data_ptr()
    a.num_seqs = ctx_lens.numel()
    a.num_tokens, a.num_q_heads, a.head_dim = q.shape[0], q.shape[1], q.shape[2]
    a.num_kv_heads, a.block_size, a.num_blocks = k_pool.shape[1], k_pool.shape[2], k_pool.shape[0]
    a.max_blocks_per_seq = block_tables.shape[1] if block_tables.dim() == 2 else 0
    a.max_q_len, a.dtype, a.scale = int(max_q_len), dt, float(scale)
    a.kv_dtype = kv_dtype_code(k_pool)
    a.k_scale, a.v_scale = float(k_scale), float(v_scale)
    a.err_flag = _ptr(err_flag)
    if dynamic and work_counter is None:
        work_counter = torch.empty(1, dtype=torch.int32, device=q.device)
        if stream is not None and hasattr(stream, "cuda_stream"):
            work_counter.record_stream(stream)
    a.work_counter = _ptr(work_counter) if dynamic else None
    _check(lib().pa_prefill(ctypes.byref(a), _stream(stream)))
    return out


def pa_write_kv(k: torch.Tensor, v: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                slot_mapping: torch.Tensor, *, err_flag: Optional[torch.Tensor] = None,
                stream=None) -> None:
    """k, v [num_tokens][num_kv_heads][head_dim] into their slots of the pools."""
    t, hkv, d = k.shape
    nblk, _, bsz, _ = k_pool.shape
    _check(lib().pa_write_kv(_ptr(k), _ptr(v), _ptr(k_pool), _ptr(v_pool), _ptr(slot_mapping),
                             t, hkv, d, bsz, nblk, kv_dtype_code(k_pool), _ptr(err_flag),
                             _stream(stream)))


def pa_write_kv_fp8(k: torch.Tensor, v: torch.Tensor, k_pool: torch.Tensor,
                    v_pool: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                    v_scale: float, *, err_flag: Optional[torch.Tensor] = None,
                    stream=None) -> None:
    """f16/bf16 k, v [num_tokens][num_kv_heads][head_dim] quantised into uint8 E4M3 pools."""
    t, hkv, d = k.shape
    nblk, _, bsz, _ = k_pool.shape
    src = {torch.float16: PA_F16, torch.bfloat16: PA_BF16}.get(k.dtype)
    if src is None or v.dtype != k.dtype:
        raise PaError(PA_EINVAL, "k and v must both be float16 or both bfloat16")
    _check(lib().pa_write_kv_fp8(_ptr(k), _ptr(v), src, _ptr(k_pool), _ptr(v_pool),
                                 _ptr(slot_mapping), t, hkv, d, bsz, nblk, float(k_scale),
                                 float(v_scale), _ptr(err_flag), _stream(stream)))


def _ptr_array(ts: Sequence[torch.Tensor]):
    return (ctypes.c_void_p * len(ts))(*[x.data_ptr() for x in ts])


def pa_copy_blocks(k_pools: Sequence[torch.Tensor], v_pools: Sequence[torch.Tensor],
                   pairs: torch.Tensor, *, err_flag: Optional[torch.Tensor] = None,
                   stream=None) -> None:
    """pairs: device int32 [num_pairs][2] (src, dst); copies every layer's K and V block."""
    p0 = k_pools[0]
    block_bytes = p0[0].numel() * p0.element_size()
    kp, vp = _ptr_array(k_pools), _ptr_array(v_pools)
    _check(lib().pa_copy_blocks(kp, vp, len(k_pools), _ptr(pairs), pairs.shape[0], p0.shape[0],
                                block_bytes, _ptr(err_flag), _stream(stream)))


def pa_swap_blocks(k_pools: Sequence[torch.Tensor], v_pools: Sequence[torch.Tensor],
                   host_buf: torch.Tensor, block_ids, direction: int, *,
                   staging: Optional[torch.Tensor] = None, stream=None) -> None:
    """direction PA_SWAP_OUT: pools -> pinned host_buf [n][layers][2][block]; PA_SWAP_IN: back."""
    p0 = k_pools[0]
    block_bytes = p0[0].numel() * p0.element_size()
    ids = torch.as_tensor(block_ids, dtype=torch.int32).contiguous()
    kp, vp = _ptr_array(k_pools), _ptr_array(v_pools)
    st_bytes = 0 if staging is None else staging.numel() * staging.element_size()
    _check(lib().pa_swap_blocks(kp, vp, len(k_pools), _ptr(host_buf), ids.data_ptr(), ids.numel(),
                                p0.shape[0], block_bytes, direction, _ptr(staging), st_bytes,
                                _stream(stream)))


def pa_testing_set_wait_limit(wait_ns: int, stall_cta: int = -1) -> None:
    """Shorten the kernels' waits on one another (0 restores one second) and, with stall_cta
    >= 0, make that CTA withhold its part so the others' waits run out. For tests only."""
    _check(lib().pa_testing_set_wait_limit(int(wait_ns), int(stall_cta)))
