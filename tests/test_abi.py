"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every entry point the
header declares, matches the binding's struct layout and validates arguments on the host."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import paged_kv_cache_38_gb300 as pa
from paged_kv_cache_38_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))


def declared_functions(header=None):
    names = set()
    for path in [header] if header else HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names.update(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_boundary():
    assert declared_functions(HEADER) == sorted([
        "pa_copy_blocks", "pa_decode", "pa_decode_static_workspace", "pa_decode_workspace_size",
        "pa_last_error_message", "pa_prefill", "pa_status_string", "pa_swap_blocks",
        "pa_testing_set_wait_limit", "pa_write_kv", "pa_write_kv_fp8"])
    assert declared_functions(os.path.join(os.path.dirname(HEADER), "pa_scheduler.h")) == sorted([
        "pa_scheduler_add_request", "pa_scheduler_create", "pa_scheduler_destroy",
        "pa_scheduler_execute_moves", "pa_scheduler_free_blocks", "pa_scheduler_has_unfinished",
        "pa_scheduler_step"])


def test_library_exports_every_declared_symbol():
    lib = pa.lib()
    out = subprocess.run(["nm", "-D", "--defined-only", pa_build.LIBRARY], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s+(pa_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


@pytest.mark.parametrize("name,header,cls", [
    ("pa_decode_args", "pa.h", lambda: pa.pa.pa_decode_args),
    ("pa_prefill_args", "pa.h", lambda: pa.pa.pa_prefill_args),
    ("pa_step_plan", "pa_scheduler.h", lambda: __import__(
        "paged_kv_cache_38_gb300.scheduler", fromlist=["x"]).pa_step_plan)])
def test_struct_layout_matches_header(tmp_path, name, header, cls):
    struct = cls()
    fields = [f for f, _ in struct._fields_]
    src = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{header}"', 'int main(void){',
             f'printf("%zu\\n", sizeof({name}));']
    lines += [f'printf("%zu\\n", offsetof({name}, {f}));' for f in fields]
    lines += ["return 0;}"]
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(struct)
    for f, off in zip(fields, vals[1:]):
        assert getattr(struct, f).offset == off, f


def test_status_strings():
    lib = pa.lib()
    for code in (pa.PA_OK, pa.PA_EINVAL, pa.PA_EUNSUPPORTED, pa.PA_ECUDA, pa.pa.PA_ENOSPACE):
        assert lib.pa_status_string(code).startswith(b"PA_")


def _args(**kw):
    a = pa.pa.pa_decode_args()
    base = dict(num_seqs=100, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                num_blocks=12000, max_blocks_per_seq=256, max_ctx_len=4096, q_dtype=pa.PA_BF16,
                kv_dtype=pa.PA_BF16, scale=0.0884, k_scale=1.0, v_scale=1.0)
    base.update(kw)
    for k, v in base.items():
        setattr(a, k, v)
    return a


def test_workspace_size_and_validation_on_host():
    lib = pa.lib()
    assert pa.pa_decode_workspace_size(_args()) > 0
    # the work counters only, no split partials
    assert pa.pa_decode_workspace_size(_args(max_ctx_len=16, split_tokens=16)) == 256
    for bad in (dict(head_dim=96), dict(block_size=12), dict(num_q_heads=30),
                dict(max_ctx_len=5000), dict(split_tokens=24)):
        assert pa.pa_decode_workspace_size(_args(**bad)) == 0
        assert lib.pa_last_error_message()
    st = lib.pa_decode(ctypes.byref(_args(head_dim=96)), None)
    assert st == pa.PA_EINVAL
    st = lib.pa_decode(ctypes.byref(_args(num_q_heads=24)), None)  # group 3
    assert st == pa.PA_EUNSUPPORTED
    st = lib.pa_decode(ctypes.byref(_args()), None)  # null pointers
    assert st == pa.PA_EINVAL
    assert lib.pa_write_kv(None, None, None, None, None, 0, 8, 128, 16, 10, pa.PA_BF16, None,
                           None) == pa.PA_OK
    assert lib.pa_write_kv(None, None, None, None, None, 4, 8, 128, 16, 10, pa.PA_BF16, None,
                           None) == pa.PA_EINVAL
    arr = (ctypes.c_void_p * 1)(None)
    assert lib.pa_copy_blocks(arr, arr, 0, None, 1, 10, 4096, None, None) == pa.PA_EINVAL
    assert lib.pa_copy_blocks(arr, arr, 1, None, 1, 10, 4096, None, None) == pa.PA_EINVAL
    ids = (ctypes.c_int32 * 1)(20)
    assert lib.pa_swap_blocks(arr, arr, 1, None, ids, 1, 10, 4096, pa.PA_SWAP_OUT, None, 0,
                              None) == pa.PA_EINVAL


def test_wait_limit_hook_validates_on_the_host():
    """The testing hook of the bounded waits: a CTA index below -1 is refused; a valid setting
    and the reset to the default are accepted (nothing is launched)."""
    with pytest.raises(pa.PaError) as e:
        pa.pa_testing_set_wait_limit(1000, -2)
    assert e.value.status == pa.PA_EINVAL
    pa.pa_testing_set_wait_limit(1000, 3)
    pa.pa_testing_set_wait_limit(0, -1)


def test_execute_moves_validates_ids_on_the_host():
    """pa_scheduler_execute_moves checks every block id and CPU slot of the plan before it
    enqueues anything (the pool pointers are never dereferenced on this path)."""
    from paged_kv_cache_38_gb300 import scheduler as sch

    L = pa.lib()
    sch._bind(L)
    fake = (ctypes.c_void_p * 1)(1 << 20)
    for field, pairs in (("copies", [3, 64]), ("swap_out", [2, 8]), ("swap_in", [-1, 0])):
        plan = sch.pa_step_plan()
        arr = (ctypes.c_int32 * 2)(*pairs)
        setattr(plan, "num_" + field, 1)
        setattr(plan, field, ctypes.cast(arr, sch._i32p))
        st = L.pa_scheduler_execute_moves(ctypes.byref(plan), fake, fake, 1, 64, 4096, None, 8,
                                          None, None)
        assert st == pa.PA_EINVAL, field
        assert b"outside" in L.pa_last_error_message(), field
