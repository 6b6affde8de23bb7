"""ctypes binding of ``include/pa_scheduler.h`` (argument marshalling only).

``Scheduler`` wraps one ``pa_scheduler``; ``step()`` copies the C plan into a ``Plan`` holding
Python lists (for checks) and numpy arrays (for the kernels: block tables, context lengths,
slot mapping, copy pairs, swap lists).
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import List, Tuple

import numpy as np

from .pa import PaError, lib

RECOMPUTE, SWAP = 0, 1

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)


class pa_step_plan(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32), ("seq_ids", _i64p), ("block_tables", _i32p),
        ("ctx_lens", _i32p), ("num_writes", ctypes.c_int32), ("write_seq", _i32p),
        ("write_pos", _i32p), ("slot_mapping", _i64p), ("num_copies", ctypes.c_int32),
        ("copies", _i32p), ("num_swap_out", ctypes.c_int32), ("swap_out", _i32p),
        ("num_swap_in", ctypes.c_int32), ("swap_in", _i32p), ("num_finished", ctypes.c_int32),
        ("finished", _i64p), ("num_preempted", ctypes.c_int32), ("preempted", _i64p),
        ("num_free_blocks", ctypes.c_int32),
    ]


def _bind(L) -> None:
    if getattr(L, "_scheduler_bound", False):
        return
    L.pa_scheduler_create.restype = ctypes.c_void_p
    L.pa_scheduler_create.argtypes = [ctypes.c_int32] * 4 + [ctypes.c_int, ctypes.c_int32]
    L.pa_scheduler_destroy.restype = None
    L.pa_scheduler_destroy.argtypes = [ctypes.c_void_p]
    L.pa_scheduler_add_request.restype = ctypes.c_int
    L.pa_scheduler_add_request.argtypes = [ctypes.c_void_p, ctypes.c_int64] + [ctypes.c_int32] * 3
    L.pa_scheduler_step.restype = ctypes.c_int
    L.pa_scheduler_step.argtypes = [ctypes.c_void_p, ctypes.POINTER(pa_step_plan)]
    L.pa_scheduler_free_blocks.restype = ctypes.c_int32
    L.pa_scheduler_free_blocks.argtypes = [ctypes.c_void_p, _i32p, ctypes.c_int32]
    L.pa_scheduler_has_unfinished.restype = ctypes.c_int32
    L.pa_scheduler_has_unfinished.argtypes = [ctypes.c_void_p]
    L._scheduler_bound = True


def _arr(ptr, n, dtype) -> np.ndarray:
    if n == 0:
        return np.zeros(0, dtype=dtype)
    return np.ctypeslib.as_array(ptr, shape=(n,)).astype(dtype, copy=True)


@dataclass
class Plan:
    seq_ids: List[int]
    block_tables: List[List[int]]
    ctx_lens: List[int]
    writes: List[Tuple[int, int, int]]
    copies: List[Tuple[int, int]]
    swap_out: List[Tuple[int, int]]
    swap_in: List[Tuple[int, int]]
    finished: List[int]
    preempted: List[int]
    num_free_blocks: int
    # the same data as arrays
    tables_np: np.ndarray     # int32 [num_seqs][max_blocks_per_seq]
    ctx_np: np.ndarray        # int32 [num_seqs]
    write_seq_np: np.ndarray  # int32 [num_writes]
    write_pos_np: np.ndarray  # int32 [num_writes]
    slots_np: np.ndarray      # int64 [num_writes]
    copies_np: np.ndarray     # int32 [num_copies][2]
    swap_out_np: np.ndarray   # int32 [n][2] (GPU block, CPU slot)
    swap_in_np: np.ndarray    # int32 [n][2] (CPU slot, GPU block)


class Scheduler:
    def __init__(self, num_blocks: int, block_size: int, max_blocks_per_seq: int,
                 max_running_seqs: int, mode: int, num_cpu_blocks: int):
        self._lib = lib()
        _bind(self._lib)
        self.max_blocks = max_blocks_per_seq
        self._h = self._lib.pa_scheduler_create(num_blocks, block_size, max_blocks_per_seq,
                                                max_running_seqs, mode, num_cpu_blocks)
        if not self._h:
            raise PaError(1, self._lib.pa_last_error_message().decode())

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pa_scheduler_destroy(h)
            self._h = None

    def add_request(self, request_id: int, prompt_len: int, max_new_tokens: int,
                    num_samples: int) -> bool:
        return self._lib.pa_scheduler_add_request(self._h, request_id, prompt_len,
                                                  max_new_tokens, num_samples) == 0

    def step(self) -> Plan:
        p = pa_step_plan()
        st = self._lib.pa_scheduler_step(self._h, ctypes.byref(p))
        if st != 0:
            raise PaError(st, self._lib.pa_last_error_message().decode())
        n, mb = p.num_seqs, self.max_blocks
        tables = _arr(p.block_tables, n * mb, np.int32).reshape(n, mb)
        ctx = _arr(p.ctx_lens, n, np.int32)
        ws, wp = _arr(p.write_seq, p.num_writes, np.int32), _arr(p.write_pos, p.num_writes, np.int32)
        slots = _arr(p.slot_mapping, p.num_writes, np.int64)
        copies = _arr(p.copies, 2 * p.num_copies, np.int32).reshape(-1, 2)
        sout = _arr(p.swap_out, 2 * p.num_swap_out, np.int32).reshape(-1, 2)
        sin = _arr(p.swap_in, 2 * p.num_swap_in, np.int32).reshape(-1, 2)
        pairs = lambda a: [tuple(int(v) for v in r) for r in a]  # noqa: E731
        return Plan(
            seq_ids=_arr(p.seq_ids, n, np.int64).tolist(), block_tables=tables.tolist(),
            ctx_lens=ctx.tolist(),
            writes=[(int(a), int(b), int(c)) for a, b, c in zip(ws, wp, slots)],
            copies=pairs(copies), swap_out=pairs(sout), swap_in=pairs(sin),
            finished=_arr(p.finished, p.num_finished, np.int64).tolist(),
            preempted=_arr(p.preempted, p.num_preempted, np.int64).tolist(),
            num_free_blocks=int(p.num_free_blocks), tables_np=tables, ctx_np=ctx,
            write_seq_np=ws, write_pos_np=wp, slots_np=slots, copies_np=copies,
            swap_out_np=sout, swap_in_np=sin)

    @property
    def free(self) -> List[int]:
        n = self._lib.pa_scheduler_free_blocks(self._h, None, 0)
        out = (ctypes.c_int32 * max(1, n))()
        self._lib.pa_scheduler_free_blocks(self._h, out, n)
        return list(out[:n])

    def num_free_blocks(self) -> int:
        return int(self._lib.pa_scheduler_free_blocks(self._h, None, 0))

    def has_unfinished(self) -> bool:
        return bool(self._lib.pa_scheduler_has_unfinished(self._h))
