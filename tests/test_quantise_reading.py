"""How much the quantise-on-write reading matters: E4M3 codes of x * RN32(1 / scale) against
codes of the IEEE binary32 quotient RN32(x / scale).

"KV Cache Preemption in vLLM", section "How much KV cache a token costs", gives an FP8 cache
(one byte per element) but no rounding rule for quantising into it. The oracle and the kernel
multiply by the binary32 reciprocal of the scale (one multiply per element instead of a
division). This test counts, over every finite bf16 and f16 input, how many stored codes would
differ had the exact quotient been taken instead: none at the scales the parity tests use, and
the count over 2,000 seeded log-uniform scales in [1e-4, 1e3] is pinned, so the size of the
difference between the two readings is stated, not assumed. (No GPU.)
"""
import numpy as np
import torch

import oracle

TEST_SCALES = (1.0, 0.0078125, 0.05, 0.37, 3.3e-3, 170.0)
# (inputs, codes differing) over the 2,000 seeded scales, per source type
SURVEY = {"bf16": (2000 * 65280, 0), "f16": (2000 * 63488, 28)}


def _finite_inputs(src):
    bits = np.arange(65536, dtype=np.uint16)
    if src == "bf16":
        vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    else:
        vals = bits.view(np.float16).astype(np.float32)
    return vals[np.isfinite(vals)].astype(np.float64)


def _differing(orc, v, scale):
    s32 = np.float32(scale)
    inv = np.float32(1.0 / np.float64(s32))
    with np.errstate(over="ignore", invalid="ignore"):
        by_reciprocal = (v * np.float64(inv)).astype(np.float32)
        by_quotient = (v / np.float64(s32)).astype(np.float32)
    return int((orc.e4m3_encode(by_reciprocal) != orc.e4m3_encode(by_quotient)).sum())


def test_readings_agree_at_the_tested_scales():
    orc = oracle.load()
    for src in ("bf16", "f16"):
        v = _finite_inputs(src)
        for sc in TEST_SCALES:
            assert _differing(orc, v, sc) == 0, (src, sc)


def test_readings_differ_rarely_over_many_scales():
    orc = oracle.load()
    scales = np.float32(10.0) ** np.random.default_rng(38).uniform(-4, 3, 2000).astype(np.float32)
    for src in ("bf16", "f16"):
        v = _finite_inputs(src)
        diff = sum(_differing(orc, v, sc) for sc in scales)
        assert (v.size * len(scales), diff) == SURVEY[src], (src, diff)
