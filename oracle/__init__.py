"""Plain CPU oracle for the paged KV-cache hot path -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package. It never imports the CUDA library and the CUDA library never imports it; the two
share nothing but the seeded input generators in ``synth``.

The arithmetic lives in ``pa_oracle.c`` (fp64, straight loops); this module compiles it with gcc
and marshals numpy / torch CPU buffers into it as raw bytes.

Every function is pinned by the ``-m "not gpu"`` tests (``tests/test_oracle_pins.py``) against
library decoders, a library attention routine run on the unpaged data, closed forms, and the
worked example of "When KV Capacity Runs Out: Pausing and Resuming Requests" (Figures 1-2);
``tests/test_oracle_mutants.py`` plants mistakes in copies of the C source and checks that a
pin catches each one.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import tempfile
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "pa_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

# Oracle dtype codes (private to the oracle; the CUDA library has its own enum).
DTYPES = {"f16": 0, "bf16": 1, "e4m3": 2}
ELT_BYTES = {"f16": 2, "bf16": 2, "e4m3": 1}

_c_int = ctypes.c_int
_c_dbl = ctypes.c_double
_ptr = ctypes.c_void_p


def build(source: str = SOURCE, output: str = LIBRARY, openmp: bool = True) -> str:
    """Compile ``source`` into the shared library ``output`` with gcc; returns ``output``."""
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", source, "-o", output, "-lm"]
    if openmp:
        try:
            subprocess.run(base[:5] + ["-fopenmp"] + base[5:], check=True,
                           capture_output=True, text=True)
            return output
        except subprocess.CalledProcessError:
            pass  # no OpenMP runtime: fall through to a single-threaded build
    subprocess.run(base, check=True, capture_output=True, text=True)
    return output


def _raw(a) -> np.ndarray:
    """Contiguous uint8 view of a numpy array or torch CPU tensor (no value conversion)."""
    if hasattr(a, "detach"):  # torch tensor
        import torch

        t = a.detach()
        if t.device.type != "cpu":
            t = t.cpu()
        t = t.contiguous()
        return t.view(torch.uint8).numpy() if t.numel() else np.zeros(0, np.uint8)
    return np.ascontiguousarray(a).view(np.uint8)


def _int_array(a, dtype) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray) -> int:
    return a.ctypes.data if a.size else 0


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.pao_f16_value.restype = _c_dbl
        lib.pao_f16_value.argtypes = [ctypes.c_uint16]
        lib.pao_bf16_value.restype = _c_dbl
        lib.pao_bf16_value.argtypes = [ctypes.c_uint16]
        lib.pao_e4m3_value.restype = _c_dbl
        lib.pao_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.pao_decode.restype = _c_int
        lib.pao_decode.argtypes = [_ptr, _c_int, _ptr, _ptr, _c_int, _ptr, _ptr] + [_c_int] * 7 + [
            _c_dbl, _c_dbl, _c_dbl, _ptr, _c_int]
        lib.pao_write_kv.restype = _c_int
        lib.pao_write_kv.argtypes = [_ptr] * 5 + [_c_int] * 6
        lib.pao_copy_blocks.restype = _c_int
        lib.pao_copy_blocks.argtypes = [_ptr, _ptr, _c_int, _ptr, _c_int, _c_int, ctypes.c_size_t]
        lib.pao_swap_blocks.restype = _c_int
        lib.pao_swap_blocks.argtypes = [_ptr, _ptr, _c_int, _ptr, _ptr, _c_int, _c_int,
                                        ctypes.c_size_t, _c_int]
        lib.pao_max_threads.restype = _c_int
        lib.pao_prefill.restype = _c_int
        lib.pao_prefill.argtypes = [_ptr, _c_int, _ptr, _ptr, _c_int, _ptr, _ptr, _ptr] + [
            _c_int] * 7 + [_c_dbl, _c_dbl, _c_dbl, _ptr, _c_int]
        lib.pao_e4m3_encode_array.restype = None
        lib.pao_e4m3_encode_array.argtypes = [_ptr, _ptr, ctypes.c_size_t]
        lib.pao_write_kv_fp8.restype = _c_int
        lib.pao_write_kv_fp8.argtypes = [_ptr, _ptr, _c_int, _ptr, _ptr, _ptr] + [_c_int] * 5 + [
            ctypes.c_float, ctypes.c_float]
        self.lib = lib

    # -------------------------------------------------------------- number formats
    def value(self, bits, dtype: str) -> np.ndarray:
        """fp64 values of raw element bit patterns (uint16 for f16/bf16, uint8 for e4m3)."""
        fn = {"f16": self.lib.pao_f16_value, "bf16": self.lib.pao_bf16_value,
              "e4m3": self.lib.pao_e4m3_value}[dtype]
        flat = np.asarray(bits).reshape(-1)
        return np.array([fn(int(b)) for b in flat], dtype=np.float64).reshape(np.shape(bits))

    def e4m3_encode(self, x) -> np.ndarray:
        """E4M3 codes (uint8) of float32 values: nearest, ties to even, saturating, NaN -> 0x7F."""
        xf = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
        out = np.empty(xf.shape, dtype=np.uint8)
        self.lib.pao_e4m3_encode_array(_p(xf), _p(out), xf.size)
        return out

    def max_threads(self) -> int:
        return int(self.lib.pao_max_threads())

    # -------------------------------------------------------------- decode attention
    def decode(self, q, k_pool, v_pool, block_tables, ctx_lens, *, q_dtype: str, kv_dtype: str,
               num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
               scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
               num_threads: int = 0, return_status: bool = False):
        """fp64 attention output [num_seqs][num_q_heads][head_dim] of a paged decode step."""
        qb, kb, vb = _raw(q), _raw(k_pool), _raw(v_pool)
        bt = _int_array(block_tables, np.int32)
        cl = _int_array(ctx_lens, np.int32).reshape(-1)
        n = cl.shape[0]
        bt = bt.reshape(n, -1) if n else bt.reshape(0, 0)
        max_blocks = bt.shape[1] if n else 0
        elt = ELT_BYTES[kv_dtype]
        per_block = num_kv_heads * block_size * head_dim * elt
        num_blocks = kb.size // per_block
        assert qb.size == n * num_q_heads * head_dim * ELT_BYTES[q_dtype], "q size"
        out = np.zeros((n, num_q_heads, head_dim), dtype=np.float64)
        rc = self.lib.pao_decode(_p(qb), DTYPES[q_dtype], _p(kb), _p(vb), DTYPES[kv_dtype],
                                 _p(bt), _p(cl), n, num_q_heads, num_kv_heads, head_dim,
                                 block_size, num_blocks, max_blocks, float(scale),
                                 float(k_scale), float(v_scale), _p(out), int(num_threads))
        return (out, rc) if return_status else out

    def prefill(self, q, k_pool, v_pool, block_tables, ctx_lens, q_starts, *, dtype: str,
                num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                scale: float, q_dtype: Optional[str] = None, k_scale: float = 1.0,
                v_scale: float = 1.0, num_threads: int = 0, return_status: bool = False):
        """fp64 causal attention of each sequence's chunk of query tokens over its paged cache:
        [num_tokens][num_q_heads][head_dim]. ``dtype`` is the KV dtype; the queries have
        ``q_dtype`` (default: the KV dtype); an E4M3 cache is read as stored value x scale."""
        qb, kb, vb = _raw(q), _raw(k_pool), _raw(v_pool)
        cl = _int_array(ctx_lens, np.int32).reshape(-1)
        qs = _int_array(q_starts, np.int32).reshape(-1)
        n = cl.shape[0]
        bt = _int_array(block_tables, np.int32).reshape(n, -1)
        per_block = num_kv_heads * block_size * head_dim * ELT_BYTES[dtype]
        ntok = int(qs[-1]) if qs.size else 0
        out = np.zeros((ntok, num_q_heads, head_dim), dtype=np.float64)
        rc = self.lib.pao_prefill(_p(qb), DTYPES[q_dtype or dtype], _p(kb), _p(vb), DTYPES[dtype],
                                  _p(bt), _p(cl), _p(qs), n, num_q_heads, num_kv_heads, head_dim,
                                  block_size, kb.size // per_block, bt.shape[1], float(scale),
                                  float(k_scale), float(v_scale), _p(out), int(num_threads))
        return (out, rc) if return_status else out

    # -------------------------------------------------------------- block movers
    def write_kv(self, k, v, k_pool: np.ndarray, v_pool: np.ndarray, slot_mapping, *,
                 num_kv_heads: int, head_dim: int, block_size: int, kv_dtype: str) -> int:
        """In-place on the uint8 numpy pools; returns 0 or -1 (a slot outside the pool)."""
        kb, vb = _raw(k), _raw(v)
        sm = _int_array(slot_mapping, np.int64).reshape(-1)
        assert k_pool.dtype == np.uint8 and k_pool.flags.c_contiguous
        assert v_pool.dtype == np.uint8 and v_pool.flags.c_contiguous
        per_block = num_kv_heads * block_size * head_dim * ELT_BYTES[kv_dtype]
        return int(self.lib.pao_write_kv(_p(kb), _p(vb), _p(k_pool), _p(v_pool), _p(sm),
                                         sm.shape[0], num_kv_heads, head_dim, block_size,
                                         k_pool.size // per_block, DTYPES[kv_dtype]))

    def write_kv_fp8(self, k, v, k_pool: np.ndarray, v_pool: np.ndarray, slot_mapping, *,
                     src_dtype: str, num_kv_heads: int, head_dim: int, block_size: int,
                     k_scale: float, v_scale: float) -> int:
        """Quantise-on-write into uint8 E4M3 pools, in place; returns 0 or -1 (a bad slot)."""
        kb, vb = _raw(k), _raw(v)
        sm = _int_array(slot_mapping, np.int64).reshape(-1)
        assert k_pool.dtype == np.uint8 and k_pool.flags.c_contiguous
        assert v_pool.dtype == np.uint8 and v_pool.flags.c_contiguous
        per_block = num_kv_heads * block_size * head_dim
        return int(self.lib.pao_write_kv_fp8(_p(kb), _p(vb), DTYPES[src_dtype], _p(k_pool),
                                             _p(v_pool), _p(sm), sm.shape[0], num_kv_heads,
                                             head_dim, block_size, k_pool.size // per_block,
                                             float(k_scale), float(v_scale)))

    def copy_blocks(self, k_pools: Sequence[np.ndarray], v_pools: Sequence[np.ndarray], pairs,
                    *, block_bytes: int) -> int:
        """In-place on lists of uint8 numpy pools (one per layer)."""
        pr = _int_array(pairs, np.int32).reshape(-1, 2)
        kp = (ctypes.c_void_p * len(k_pools))(*[p.ctypes.data for p in k_pools])
        vp = (ctypes.c_void_p * len(v_pools))(*[p.ctypes.data for p in v_pools])
        num_blocks = k_pools[0].size // block_bytes
        return int(self.lib.pao_copy_blocks(kp, vp, len(k_pools), _p(pr), pr.shape[0],
                                            num_blocks, block_bytes))

    def swap_blocks(self, k_pools: Sequence[np.ndarray], v_pools: Sequence[np.ndarray],
                    host_buf: np.ndarray, block_ids, *, block_bytes: int, direction: str) -> int:
        """direction 'out': pools -> host_buf; 'in': host_buf -> pools (uint8 arrays)."""
        ids = _int_array(block_ids, np.int32).reshape(-1)
        kp = (ctypes.c_void_p * len(k_pools))(*[p.ctypes.data for p in k_pools])
        vp = (ctypes.c_void_p * len(v_pools))(*[p.ctypes.data for p in v_pools])
        num_blocks = k_pools[0].size // block_bytes
        assert host_buf.dtype == np.uint8 and host_buf.size >= ids.size * len(k_pools) * 2 * block_bytes
        return int(self.lib.pao_swap_blocks(kp, vp, len(k_pools), _p(host_buf), _p(ids),
                                            ids.shape[0], num_blocks, block_bytes,
                                            {"out": 0, "in": 1}[direction]))


_default: Optional[Oracle] = None


def load(path: Optional[str] = None) -> Oracle:
    """The oracle compiled from ``pa_oracle.c`` (built on first use), or the library at ``path``."""
    global _default
    if path is not None:
        return Oracle(path)
    if _default is None:
        stale = (not os.path.exists(LIBRARY)
                 or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE))
        if stale:
            # build into a temp file and rename: concurrent test workers never see half a file
            fd, tmp = tempfile.mkstemp(suffix=".so", dir=HERE)
            os.close(fd)
            build(SOURCE, tmp)
            shutil.move(tmp, LIBRARY)
        _default = Oracle(LIBRARY)
    return _default
