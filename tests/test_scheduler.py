"""The C++ scheduler (include/pa_scheduler.h) on the CPU: the oracle's pins, and plan-for-plan
equality with the oracle on seeded scripts (integer bookkeeping: bit-exact)."""
import types

import pytest

import pins_blocks
from oracle import block_manager as oracle_bm

import paged_kv_cache_38_gb300 as pa  # noqa: E402
from paged_kv_cache_38_gb300 import scheduler as cxx

CXX = types.SimpleNamespace(Scheduler=cxx.Scheduler, RECOMPUTE=cxx.RECOMPUTE, SWAP=cxx.SWAP)
FIELDS = ["seq_ids", "block_tables", "ctx_lens", "writes", "copies", "swap_out", "swap_in",
          "finished", "preempted", "num_free_blocks"]


@pytest.mark.parametrize("pin", pins_blocks.ALL_PINS, ids=[p.__name__ for p in pins_blocks.ALL_PINS])
def test_cxx_scheduler_meets_the_pins(pin):
    pin(CXX)


@pytest.mark.parametrize("mode", [0, 1], ids=["recompute", "swap"])
def test_plans_equal_the_oracle(mode):
    for seed in range(60):
        a = pins_blocks.drive(CXX, 500 + seed, mode, check=False)
        b = pins_blocks.drive(oracle_bm, 500 + seed, mode, check=False)
        assert len(a) == len(b), seed
        for step, (pa_, pb) in enumerate(zip(a, b)):
            for f in FIELDS:
                assert getattr(pa_, f) == getattr(pb, f), (seed, step, f)


def test_large_batch_equals_the_oracle():
    """The GQA workload's shape: 25 groups of 4 samples sharing a 512-token prompt, plus
    single-sequence requests, through growth, copy-on-write and swapping."""
    def run(mod):
        s = mod.Scheduler(3000, 16, 512, 256, mod.SWAP, 6000)
        for r in range(25):
            assert s.add_request(r, 512 + 7 * r, 200, 4)
        for r in range(25, 60):
            assert s.add_request(r, 100 + 37 * r, 300, 1)
        plans = []
        while s.has_unfinished():
            plans.append(s.step())
        return plans
    a, b = run(CXX), run(oracle_bm)
    assert len(a) == len(b)
    for pa_, pb in zip(a, b):
        for f in FIELDS:
            assert getattr(pa_, f) == getattr(pb, f), f
    assert any(p.copies for p in a) and any(p.swap_out for p in a)


def test_errors():
    with pytest.raises(pa.PaError):
        cxx.Scheduler(0, 16, 8, 4, cxx.SWAP, 4)
    s = cxx.Scheduler(8, 4, 4, 4, cxx.SWAP, 0)
    assert s.add_request(1, 5, 3, 1)
    assert not s.add_request(1, 5, 3, 1)          # repeated id
    assert not s.add_request(2, 0, 3, 1)          # empty prompt
    assert not s.add_request(3, 15, 3, 1)         # more than 4 blocks per sequence
    assert not s.add_request(4, 5, 3, 257)        # too many samples
    # two running requests that cannot both grow, and no CPU slot to swap into
    s = cxx.Scheduler(4, 4, 4, 4, cxx.SWAP, 0)
    assert s.add_request(1, 3, 10, 1) and s.add_request(2, 3, 10, 1)
    with pytest.raises(pa.PaError) as e:
        for _ in range(20):
            s.step()
    assert e.value.status == pa.pa.PA_ENOSPACE
