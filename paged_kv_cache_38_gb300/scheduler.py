"""ctypes binding of ``include/pa_scheduler.h`` (argument marshalling only).

``Scheduler`` wraps one ``pa_scheduler``; ``step()`` copies the C plan into a ``Plan`` of numpy
arrays (for the kernels: block tables, context lengths, slot mapping, copy pairs, swap lists),
with list views of the same data for checks.
"""
from __future__ import annotations

import ctypes
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
    L.pa_scheduler_execute_moves.restype = ctypes.c_int
    L.pa_scheduler_execute_moves.argtypes = [ctypes.POINTER(pa_step_plan), ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                             ctypes.c_size_t, ctypes.c_void_p, ctypes.c_int32,
                                             ctypes.c_void_p, ctypes.c_void_p]
    L._scheduler_bound = True


def _arr(ptr, n, dtype) -> np.ndarray:
    """A copy of n elements at ptr (one memmove into a new array)."""
    out = np.empty(n, dtype=dtype)
    if n:
        ctypes.memmove(out.ctypes.data, ptr, out.nbytes)
    return out


class Plan:
    """One step's plan as arrays (copies of the scheduler's, so they outlive its next step);
    the list views of the same data are built on first use."""

    def __init__(self, seq_ids, tables, ctx, write_seq, write_pos, slots, copies, swap_out,
                 swap_in, finished, preempted, num_free_blocks):
        self.seq_ids_np = seq_ids     # int64 [num_seqs]
        self.tables_np = tables       # int32 [num_seqs][max_blocks_per_seq]
        self.ctx_np = ctx             # int32 [num_seqs]
        self.write_seq_np = write_seq  # int32 [num_writes]
        self.write_pos_np = write_pos  # int32 [num_writes]
        self.slots_np = slots         # int64 [num_writes]
        self.copies_np = copies       # int32 [num_copies][2] (src, dst)
        self.swap_out_np = swap_out   # int32 [n][2] (GPU block, CPU slot)
        self.swap_in_np = swap_in     # int32 [n][2] (CPU slot, GPU block)
        self.finished: List[int] = finished
        self.preempted: List[int] = preempted
        self.num_free_blocks = num_free_blocks

    @staticmethod
    def _pairs(a: np.ndarray) -> List[Tuple[int, int]]:
        return [(int(x), int(y)) for x, y in a]

    @property
    def seq_ids(self) -> List[int]:
        return self.seq_ids_np.tolist()

    @property
    def block_tables(self) -> List[List[int]]:
        return self.tables_np.tolist()

    @property
    def ctx_lens(self) -> List[int]:
        return self.ctx_np.tolist()

    @property
    def writes(self) -> List[Tuple[int, int, int]]:
        return list(zip(self.write_seq_np.tolist(), self.write_pos_np.tolist(),
                        self.slots_np.tolist()))

    @property
    def copies(self) -> List[Tuple[int, int]]:
        return self._pairs(self.copies_np)

    @property
    def swap_out(self) -> List[Tuple[int, int]]:
        return self._pairs(self.swap_out_np)

    @property
    def swap_in(self) -> List[Tuple[int, int]]:
        return self._pairs(self.swap_in_np)


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
        return Plan(
            _arr(p.seq_ids, n, np.int64), _arr(p.block_tables, n * mb, np.int32).reshape(n, mb),
            _arr(p.ctx_lens, n, np.int32), _arr(p.write_seq, p.num_writes, np.int32),
            _arr(p.write_pos, p.num_writes, np.int32), _arr(p.slot_mapping, p.num_writes, np.int64),
            _arr(p.copies, 2 * p.num_copies, np.int32).reshape(-1, 2),
            _arr(p.swap_out, 2 * p.num_swap_out, np.int32).reshape(-1, 2),
            _arr(p.swap_in, 2 * p.num_swap_in, np.int32).reshape(-1, 2),
            _arr(p.finished, p.num_finished, np.int64).tolist(),
            _arr(p.preempted, p.num_preempted, np.int64).tolist(), int(p.num_free_blocks))

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


def execute_moves(plan: Plan, k_pools, v_pools, cpu_pool, *, err_flag=None, stream=None) -> None:
    """pa_scheduler_execute_moves on a plan's move lists: swap-outs (GPU block -> CPU slot),
    swap-ins (CPU slot -> GPU block), then copy-on-write copies, enqueued by the library in that
    order. ``cpu_pool`` is a pinned uint8 tensor [num_cpu_blocks][layers][2][block_bytes] (or
    None when the plan has no swaps). The KV writes and the decode are the caller's (they need
    the new K/V)."""
    from .pa import _check, _ptr, _ptr_array, _stream

    L = lib()
    _bind(L)
    p = pa_step_plan()
    lists = {}
    for name, arr in (("copies", plan.copies_np), ("swap_out", plan.swap_out_np),
                      ("swap_in", plan.swap_in_np)):
        a = np.ascontiguousarray(arr, dtype=np.int32)
        lists[name] = a  # kept alive for the call
        setattr(p, "num_" + name, a.shape[0] if a.size else 0)
        setattr(p, name, a.ctypes.data_as(_i32p) if a.size else None)
    k0 = k_pools[0]
    block_bytes = k0[0].numel() * k0.element_size()
    ncpu = 0 if cpu_pool is None else cpu_pool.shape[0]
    _check(L.pa_scheduler_execute_moves(ctypes.byref(p), _ptr_array(k_pools),
                                        _ptr_array(v_pools), len(k_pools), k0.shape[0],
                                        block_bytes, _ptr(cpu_pool), ncpu, _ptr(err_flag),
                                        _stream(stream)))
