"""Pins of the CPU oracle: checks against something other than the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError when the oracle
disagrees with
  * a library decoder or encoder (numpy float16, torch bfloat16 / float8_e4m3fn) or the OCP
    E4M3 table,
  * a library attention routine (torch scaled_dot_product_attention in fp64, with its own GQA
    grouping) run on the unpaged keys and values the generator kept,
  * closed forms (one token, equal keys, zero scale, one dominant key, empty context),
  * invariants the pages state (physical placement is irrelevant; copy-on-write leaves the
    source alone; swapped blocks come back bit-exact, possibly elsewhere),
  * the worked example of "When KV Capacity Runs Out", Figures 1-2 (tests/golden).
``tests/test_oracle_pins.py`` runs them on the real oracle; ``tests/test_oracle_mutants.py``
runs them on copies of the oracle with planted mistakes and expects at least one to fail.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------ helpers

def logical_values(case: synth.PagedCase, s: int):
    """fp64 unpaged K, V of sequence s as [Hkv][L][D] using library casts."""
    spec = case.spec

    def conv(t, sc):
        if spec.kv_dtype == "e4m3":
            return t.view(torch.float8_e4m3fn).to(torch.float64) * sc
        return t.to(torch.float64)

    return (conv(case.k_logical[s], case.k_scale).permute(1, 0, 2),
            conv(case.v_logical[s], case.v_scale).permute(1, 0, 2))


def library_attention(case: synth.PagedCase) -> np.ndarray:
    """torch SDPA in fp64 on the unpaged data (enable_gqa groups query heads contiguously)."""
    spec = case.spec
    out = np.zeros((spec.num_seqs, spec.num_q_heads, spec.head_dim))
    for s in range(spec.num_seqs):
        if int(case.ctx_lens[s]) == 0:
            continue
        K, V = logical_values(case, s)
        q = case.q[s].to(torch.float64)[None, :, None, :]
        r = F.scaled_dot_product_attention(q, K[None], V[None], scale=case.scale,
                                           enable_gqa=True)
        out[s] = r[0, :, 0, :].numpy()
    return out


def run_decode(orc, case: synth.PagedCase, **over):
    spec = case.spec
    kw = dict(q_dtype=spec.q_dtype, kv_dtype=spec.kv_dtype, num_q_heads=spec.num_q_heads,
              num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
              block_size=spec.block_size, scale=case.scale, k_scale=case.k_scale,
              v_scale=case.v_scale)
    kw.update(over)
    args = dict(q=case.q, k_pool=case.k_pool, v_pool=case.v_pool,
                block_tables=case.block_tables, ctx_lens=case.ctx_lens)
    for key in list(kw):
        if key in args:
            args[key] = kw.pop(key)
    return orc.decode(args["q"], args["k_pool"], args["v_pool"], args["block_tables"],
                      args["ctx_lens"], **kw)


def small_specs():
    """Small workloads covering every dtype pair, group size, head_dim and block size."""
    S = synth.SPECS
    return [
        S["toy"],
        S["mha7b"].scaled(num_seqs=3, ctx_range=(17, 61), num_blocks=None),
        S["gqa_pressure"].scaled(num_seqs=8, ctx_range=(20, 90), shared_prompt=32),
        S["fp8_long"].scaled(num_seqs=4, ctx_range=(30, 100)),
        S["fp8_long"].scaled(name="fp8_f16q", q_dtype="f16", num_seqs=2, ctx_range=(5, 40)),
        synth.DecodeSpec("g2_b8", 3, 8, 4, 64, 8, "bf16", "bf16", ctx_range=(1, 40)),
        synth.DecodeSpec("g16_b32", 2, 16, 1, 128, 32, "f16", "f16", ctx_range=(30, 70)),
    ]


def _raw_u8(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.uint8).numpy().copy()


# ------------------------------------------------------------------ number formats

def pin_f16_decoder(orc):
    bits = np.arange(65536, dtype=np.uint16)
    got = orc.value(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "binary16 decoding differs from numpy"
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def pin_bf16_decoder(orc):
    bits = np.arange(65536, dtype=np.uint16)
    got = orc.value(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "bfloat16 decoding differs from torch"


def pin_e4m3_decoder(orc):
    bits = np.arange(256, dtype=np.uint8)
    got = orc.value(bits, "e4m3")
    ref = torch.from_numpy(bits).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "E4M3 decoding differs from torch"
    with open(os.path.join(GOLDEN, "e4m3_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            b, v = line.split()
            val = orc.value(np.array([int(b, 16)], np.uint8), "e4m3")[0]
            if v == "nan":
                assert math.isnan(val), b
            else:
                assert val == float(v) and math.copysign(1, val) == math.copysign(1, float(v)), b


def _e4m3_library(q: np.ndarray) -> np.ndarray:
    """E4M3 codes by the library cast. torch rounds to nearest-even but turns magnitudes beyond
    the largest finite value into NaN, so values are clamped to +-448 first: the saturating
    reading of the FP8 cache. NaN inputs give a NaN code of either sign."""
    t = torch.from_numpy(np.ascontiguousarray(q, dtype=np.float32))
    return t.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_e4m3_encoder(orc):
    """Every bf16 and f16 value, divided by several scales in binary32, encodes as the library
    cast does; decoding then encoding every code gives the code back; the midpoint of two
    neighbouring codes goes to the one with the even fraction field."""
    bits = np.arange(65536, dtype=np.uint16)
    bf = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    hf = bits.view(np.float16).astype(np.float32)
    for vals in (bf, hf):
        for sc in (1.0, 0.0078125, 0.37, 3.3e-3, 170.0):
            q = (vals / np.float32(sc)).astype(np.float32)
            got = orc.e4m3_encode(q)
            ref = _e4m3_library(q)
            nan = np.isnan(q)
            assert np.all(got[nan] == 0x7F), "NaN must give the NaN code"
            assert np.array_equal(got[~nan], ref[~nan]), f"E4M3 encoding differs, scale {sc}"
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.value(codes, "e4m3")
    ok = ~np.isnan(vals)
    assert np.array_equal(orc.e4m3_encode(vals[ok].astype(np.float32)), codes[ok])
    pos = vals[:0x7F]                       # codes 0x00..0x7E, increasing
    mid = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)  # exact in binary32
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(orc.e4m3_encode(mid), want), "ties must go to the even code"
    assert np.array_equal(orc.e4m3_encode(-mid), want | 0x80)


# ------------------------------------------------------------------ attention

def pin_paged_equals_library_attention(orc):
    """Paged attention reproduces ordinary attention on the unpaged data (PagedAttention
    summary page, kernel paragraph: the result is identical to ordinary attention)."""
    for i, spec in enumerate(small_specs()):
        case = synth.make_case(spec, seed=100 + i)
        got = run_decode(orc, case)
        ref = library_attention(case)
        err = np.abs(got - ref).max()
        assert err < 1e-12, f"{spec.name}: max |oracle - sdpa| = {err}"


def pin_closed_forms(orc):
    spec = synth.DecodeSpec("cf", 4, 4, 2, 64, 4, "bf16", "bf16", ctx_lens=(1, 9, 9, 9))
    case = synth.make_case(spec, seed=7)
    # (a) one token: softmax of one score is 1, the output is that token's value row
    got = run_decode(orc, case)
    K0, V0 = logical_values(case, 0)
    for h in range(4):
        assert np.array_equal(got[0, h], V0[h // 2, 0].numpy()), "L=1 must return V[0]"
    # (b) zero scale: uniform weights, the output is the mean of the value rows
    got0 = run_decode(orc, case, scale=0.0)
    for s in (1, 2, 3):
        _, V = logical_values(case, s)
        for h in range(4):
            assert np.abs(got0[s, h] - V[h // 2].mean(0).numpy()).max() < 1e-14
    # (c) every key equal: again the mean of the values, for any scale
    eq = synth.make_case(spec, seed=8)
    B = spec.block_size
    for s in range(spec.num_seqs):
        L = int(eq.ctx_lens[s])
        for t in range(L):
            phys = int(eq.block_tables[s, t // B])
            eq.k_pool[phys, :, t % B, :] = eq.k_pool[int(eq.block_tables[0, 0]), :, 0, :]
    gq = run_decode(orc, eq)
    for s in (1, 2, 3):
        _, V = logical_values(eq, s)
        for h in range(4):
            assert np.abs(gq[s, h] - V[h // 2].mean(0).numpy()).max() < 1e-14
    # (d) one dominant key (scores of order 1e4 overflow exp without the max shift)
    dom = synth.make_case(spec, seed=9)
    s, hot = 2, 5
    phys = int(dom.block_tables[s, hot // B])
    qrow = dom.q[s, 0].clone()
    dom.k_pool[phys, 0, hot % B, :] = (qrow * 64).to(torch.bfloat16)
    dom.k_logical = None
    gd = run_decode(orc, dom, scale=1.0)
    V = dom.v_pool[phys, 0, hot % B, :].to(torch.float64).numpy()
    assert np.all(np.isfinite(gd[s, 0])), "dominant score overflowed"
    assert np.abs(gd[s, 0] - V).max() < 1e-12, "dominant key must select its value row"
    # (e) empty context: zero row
    empty = synth.make_case(spec.scaled(ctx_lens=(0, 3, 0, 1)), seed=10)
    ge = run_decode(orc, empty)
    assert np.array_equal(ge[0], np.zeros_like(ge[0])) and np.array_equal(ge[2], ge[0])


def pin_scales(orc):
    """Per-tensor scales: k_scale multiplies every score, v_scale every output."""
    spec = synth.SPECS["fp8_long"].scaled(num_seqs=3, ctx_range=(10, 50))
    case = synth.make_case(spec, seed=11)
    base = run_decode(orc, case, k_scale=1.0, v_scale=1.0)
    a = run_decode(orc, case, k_scale=0.5, v_scale=1.0, scale=case.scale * 2.0)
    assert np.abs(a - base).max() < 1e-13, "k_scale must scale the scores"
    b = run_decode(orc, case, k_scale=1.0, v_scale=3.0)
    assert np.abs(b - 3.0 * base).max() < 1e-12, "v_scale must scale the output"


def pin_group_equals_replicated_heads(orc):
    """A GQA group reads its KV head exactly like multi-head attention on KV heads replicated
    G times (contiguous query-head groups)."""
    spec = synth.DecodeSpec("g4", 3, 8, 2, 64, 8, "f16", "f16", ctx_range=(5, 40))
    case = synth.make_case(spec, seed=12)
    got = run_decode(orc, case)
    rep = dict(k_pool=case.k_pool.repeat_interleave(4, dim=1),
               v_pool=case.v_pool.repeat_interleave(4, dim=1))
    mha = run_decode(orc, case, num_kv_heads=8, **rep)
    assert np.array_equal(got, mha)


def pin_permutation_invariance(orc):
    """Any physical placement gives the same output (summary page, block table paragraph;
    "When KV Capacity Runs Out", Figure 4: restored blocks may sit elsewhere)."""
    spec = synth.SPECS["gqa_pressure"].scaled(num_seqs=8, ctx_range=(20, 80), shared_prompt=32)
    case = synth.make_case(spec, seed=13)
    ref = run_decode(orc, case)
    for seed in (1, 2, 3):
        p = synth.permuted(case, seed)
        assert not torch.equal(p.block_tables, case.block_tables)
        assert np.array_equal(run_decode(orc, p), ref)


def pin_bounds(orc):
    """Out-of-pool block ids and over-long contexts are reported (status -1)."""
    spec = synth.DecodeSpec("b", 2, 4, 4, 64, 4, "f16", "f16", ctx_lens=(6, 5))
    case = synth.make_case(spec, seed=14)
    bt = case.block_tables.clone()
    bt[1, 1] = case.num_blocks
    _, rc = run_decode(orc, case, block_tables=bt, return_status=True)
    assert rc == -1
    _, rc = run_decode(orc, case, ctx_lens=torch.tensor([6, 9], dtype=torch.int32),
                       return_status=True)
    assert rc == -1
    out, rc = run_decode(orc, case, return_status=True)
    assert rc == 0 and np.all(np.isfinite(out))


# ------------------------------------------------------------------ movers

def pin_write_kv(orc):
    """Writing each sequence's newest token restores it exactly: poison the slots, write,
    and the paged attention equals the library attention again; stale slots stay unread."""
    for i, spec in enumerate(small_specs()):
        case = synth.make_case(spec, seed=200 + i)
        kp, vp = _raw_u8(case.k_pool), _raw_u8(case.v_pool)
        ref_k, ref_v = kp.copy(), vp.copy()
        # poison each sequence's newest slot, then write it back with write_kv
        B, elt = spec.block_size, synth.ELT_BYTES[spec.kv_dtype]
        row = spec.head_dim * elt
        kv = kp.reshape(case.num_blocks, spec.num_kv_heads, B, row)
        vv = vp.reshape(case.num_blocks, spec.num_kv_heads, B, row)
        for s in range(spec.num_seqs):
            sigma = int(case.slot_mapping[s])
            kv[sigma // B, :, sigma % B, :] = 0xFF
            vv[sigma // B, :, sigma % B, :] = 0xFF
        sm = case.slot_mapping.clone()
        sm_pad = torch.cat([sm, torch.tensor([-1, -5], dtype=torch.int64)])
        knew = torch.cat([case.k_new, case.k_new[:2]])
        vnew = torch.cat([case.v_new, case.v_new[:2]])
        rc = orc.write_kv(knew, vnew, kp, vp, sm_pad, num_kv_heads=spec.num_kv_heads,
                          head_dim=spec.head_dim, block_size=B, kv_dtype=spec.kv_dtype)
        assert rc == 0
        assert np.array_equal(kp, ref_k) and np.array_equal(vp, ref_v), spec.name
        # a slot beyond the pool is reported and skipped
        bad = torch.tensor([case.num_blocks * B], dtype=torch.int64)
        rc = orc.write_kv(case.k_new[:1], case.v_new[:1], kp, vp, bad,
                          num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                          block_size=B, kv_dtype=spec.kv_dtype)
        assert rc == -1 and np.array_equal(kp, ref_k)


def pin_write_kv_fp8(orc):
    """Quantise-on-write stores in each new token's slot the library-cast E4M3 code of
    value * (1 / scale) (reciprocal and product in binary32): the same pools as quantising first
    and then writing the bytes with the pinned raw write_kv. Specials included: signed zeros,
    infinities, values beyond 448, f16 subnormals, NaN."""
    specials = [0.0, -0.0, math.inf, -math.inf, 1.0e4, -1.0e4, 3.0e-6, math.nan]
    for i, src in enumerate(("bf16", "f16")):
        spec = synth.DecodeSpec(f"q8_{src}", 6, 8, 2, 64, 8, "e4m3", src, ctx_range=(1, 40))
        case = synth.make_case(spec, seed=71 + i)
        dt = torch.bfloat16 if src == "bf16" else torch.float16
        g = torch.Generator().manual_seed(5 + i)
        shape = (spec.num_seqs, spec.num_kv_heads, spec.head_dim)
        kn = (torch.randn(shape, generator=g) * 3).to(dt)
        vn = (torch.randn(shape, generator=g) * 0.2).to(dt)
        kn.view(-1)[: len(specials)] = torch.tensor(specials).to(dt)
        vn.view(-1)[-len(specials):] = torch.tensor(specials).to(dt)
        ks, vs = 0.05, 0.3
        kp, vp = _raw_u8(case.k_pool), _raw_u8(case.v_pool)
        kp2, vp2 = kp.copy(), vp.copy()
        sm = torch.cat([case.slot_mapping, torch.tensor([-1], dtype=torch.int64)])
        kn_p = torch.cat([kn, kn[:1]])
        vn_p = torch.cat([vn, vn[:1]])
        rc = orc.write_kv_fp8(kn_p, vn_p, kp, vp, sm, src_dtype=src,
                              num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                              block_size=spec.block_size, k_scale=ks, v_scale=vs)
        assert rc == 0

        def quant(t, sc):
            q = t.to(torch.float32).numpy() * (np.float32(1.0) / np.float32(sc))
            codes = _e4m3_library(q)
            codes[np.isnan(q)] = 0x7F
            return codes

        rc = orc.write_kv(quant(kn_p, ks), quant(vn_p, vs), kp2, vp2, sm,
                          num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                          block_size=spec.block_size, kv_dtype="e4m3")
        assert rc == 0
        assert np.array_equal(kp, kp2) and np.array_equal(vp, vp2), src
        bad = torch.tensor([case.num_blocks * spec.block_size], dtype=torch.int64)
        rc = orc.write_kv_fp8(kn[:1], vn[:1], kp, vp, bad, src_dtype=src,
                              num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                              block_size=spec.block_size, k_scale=ks, v_scale=vs)
        assert rc == -1 and np.array_equal(kp, kp2)


def _prefill_specs():
    S = synth.SPECS
    return [
        S["mha7b"].scaled(num_seqs=3, ctx_range=(17, 61), num_blocks=None),
        S["gqa_pressure"].scaled(num_seqs=5, ctx_range=(20, 90), shared_prompt=32),
        synth.DecodeSpec("g2_b8", 3, 8, 4, 64, 8, "bf16", "bf16", ctx_range=(1, 40)),
        synth.DecodeSpec("g16_b32", 2, 16, 1, 128, 32, "f16", "f16", ctx_range=(30, 70)),
        # an FP8 cache (bf16 queries, E4M3 K/V with per-tensor scales), as a recomputed
        # request of the FP8 workload is prefilled
        S["fp8_long"].scaled(num_seqs=4, ctx_range=(15, 80)),
    ]


def _run_prefill(orc, case, qs, q):
    spec = case.spec
    return orc.prefill(q, case.k_pool, case.v_pool, case.block_tables, case.ctx_lens, qs,
                       dtype=spec.kv_dtype, q_dtype=spec.q_dtype, num_q_heads=spec.num_q_heads,
                       num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim,
                       block_size=spec.block_size, scale=case.scale, k_scale=case.k_scale,
                       v_scale=case.v_scale)


def pin_prefill_equals_library_attention(orc):
    """A chunk of n new tokens over a cache of L positions: query i, at position L - n + i,
    attends to positions 0 .. L - n + i. torch SDPA in fp64 on the unpaged data with that
    boolean mask (enable_gqa groups query heads contiguously) must agree, for whole prompts
    (n = L, the prompt phase) and partial chunks (recompute, chunked prefill)."""
    for i, spec in enumerate(_prefill_specs()):
        case = synth.make_case(spec, seed=500 + i)
        for whole in (False, True):
            qs, q = synth.prefill_queries(case, seed=40 + i, whole=whole)
            got = _run_prefill(orc, case, qs, q)
            for s in range(spec.num_seqs):
                L, a, b = int(case.ctx_lens[s]), int(qs[s]), int(qs[s + 1])
                n = b - a
                if n == 0:
                    continue
                K, V = logical_values(case, s)
                qq = q[a:b].to(torch.float64).permute(1, 0, 2)[None]
                mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
                ref = F.scaled_dot_product_attention(qq, K[None], V[None], attn_mask=mask,
                                                     scale=case.scale, enable_gqa=True)
                err = np.abs(got[a:b] - ref[0].permute(1, 0, 2).numpy()).max()
                assert err < 1e-12, (spec.name, whole, s, err)


def pin_prefill_one_token_is_decode(orc):
    """A chunk of one token is a decode step: the pinned decode oracle, fed that token as its
    query, gives the same output."""
    for i, spec in enumerate(_prefill_specs()):
        case = synth.make_case(spec, seed=520 + i)
        qs, q = synth.prefill_queries(case, seed=60 + i, max_chunk=1)
        got = _run_prefill(orc, case, qs, q)
        ok = (qs[1:] - qs[:-1]) == 1
        dq = case.q.clone()
        dq[ok] = q
        ref = run_decode(orc, case, q=dq)
        assert np.abs(got - ref[ok.numpy()]).max() < 1e-12, spec.name


def pin_prefill_closed_forms(orc):
    """One cached position attended by itself gives its value row; a query of zeros weighs all
    visible positions equally (mean of the values it may see)."""
    spec = synth.DecodeSpec("pf_one", 3, 4, 2, 64, 4, "f16", "f16", ctx_lens=(1, 9, 13))
    case = synth.make_case(spec, seed=3)
    qs = torch.tensor([0, 1, 4, 9], dtype=torch.int32)
    q = torch.randn(9, 4, 64, generator=torch.Generator().manual_seed(1)).to(torch.float16)
    q[1:4] = 0
    got = _run_prefill(orc, case, qs, q)
    K, V = logical_values(case, 0)
    for h in range(4):
        assert np.array_equal(got[0, h], V[h // 2, 0].numpy())
    K, V = logical_values(case, 1)
    for i in range(3):  # positions 6, 7, 8 of a 9-position cache
        for h in range(4):
            want = V[h // 2, : 6 + i + 1].mean(0).numpy()
            assert np.abs(got[1 + i, h] - want).max() < 1e-12


def _toy_script():
    with open(os.path.join(GOLDEN, "toy_figures_1_2.txt")) as f:
        return [ln.split() for ln in (l.split("#")[0].strip() for l in f) if ln]


def pin_toy_figures(orc, rename=None):
    """Replay Figures 1-2 of "When KV Capacity Runs Out" with write_kv and decode.

    ``rename`` maps the page's block names P0..P3 to physical ids (default: identity); the
    config uses a seeded permutation, and the outcome must not depend on it."""
    rename = rename or {f"P{i}": i for i in range(4)}
    script = _toy_script()
    nblk, B = int(script[0][1]), int(script[0][2])
    Hkv, D, elt = 4, 64, 2
    rng = torch.Generator().manual_seed(38)
    logical = {r: (torch.randn((12, Hkv, D), generator=rng).half(),
                   torch.randn((12, Hkv, D), generator=rng).half()) for r in "AB"}
    q = torch.randn((1, Hkv, D), generator=rng).half()
    kp = np.full(nblk * Hkv * B * D * elt, 0xFF, np.uint8)  # NaN everywhere until written
    vp = kp.copy()
    tables, npos, free = {}, {}, set(rename.values())

    def write(r, pos, phys):
        sigma = torch.tensor([phys * B + pos % B], dtype=torch.int64)
        rc = orc.write_kv(logical[r][0][pos:pos + 1], logical[r][1][pos:pos + 1], kp, vp, sigma,
                          num_kv_heads=Hkv, head_dim=D, block_size=B, kv_dtype="f16")
        assert rc == 0

    for cmd in script[1:]:
        if cmd[0] == "own":
            r, ids = cmd[1], [rename[p] for p in cmd[2:]]
            tables[r] = ids
            free -= set(ids)
            npos[r] = 7
            for pos in range(7):  # the 7 positions already processed
                write(r, pos, ids[pos // B])
        elif cmd[0] == "write":
            r, pos, blk, slot = cmd[1], int(cmd[2]), rename[cmd[3]], int(cmd[4])
            # the 0-indexed reading: position -> (logical block pos // B, slot pos % B)
            assert tables[r][pos // B] == blk and pos % B == slot, cmd
            write(r, pos, blk)
            npos[r] = pos + 1
        elif cmd[0] == "release":
            free |= set(tables.pop(cmd[1]))
            npos.pop(cmd[1])
        elif cmd[0] == "link":
            blk = rename[cmd[2]]
            assert blk in free
            free.discard(blk)
            tables[cmd[1]].append(blk)
        elif cmd[0] == "expect":
            if cmd[1] == "free":
                assert len(free) == int(cmd[2]), cmd
            elif cmd[1] == "free_block":
                assert free == {rename[cmd[2]]}, cmd
            else:
                r = cmd[1]
                assert npos[r] == int(cmd[3]) and len(tables[r]) == int(cmd[5]), cmd
                # at most one partially filled block, the last one (summary page, block table)
                assert (len(tables[r]) - 1) * B < npos[r] <= len(tables[r]) * B
                # decode over the filled positions equals attention on the unpaged rows;
                # stale slots (never written, or B's old data in P2) must not be read
                L = npos[r]
                out = orc.decode(q, kp, vp, torch.tensor([tables[r]], dtype=torch.int32),
                                 torch.tensor([L], dtype=torch.int32), q_dtype="f16",
                                 kv_dtype="f16", num_q_heads=Hkv, num_kv_heads=Hkv, head_dim=D,
                                 block_size=B, scale=1 / 8)
                K = logical[r][0][:L].to(torch.float64).permute(1, 0, 2)
                V = logical[r][1][:L].to(torch.float64).permute(1, 0, 2)
                ref = F.scaled_dot_product_attention(q.to(torch.float64)[:, :, None, :],
                                                     K[None], V[None], scale=1 / 8)
                assert np.abs(out[0] - ref[0, :, 0, :].numpy()).max() < 1e-12, cmd
    # B's released block P2 keeps B's stale positions 1..3 (release does not zero a block)
    row = D * elt
    kv = kp.reshape(nblk, Hkv, B, row)
    stale = logical["B"][0][1:4].contiguous().view(torch.uint8).numpy()
    assert np.array_equal(kv[rename["P2"], :, 1:4, :].transpose(1, 0, 2), stale)


def pin_toy_permuted(orc):
    perm = np.random.default_rng(38).permutation(4)
    pin_toy_figures(orc, {f"P{i}": int(perm[i]) for i in range(4)})


def pin_copy_on_write(orc):
    """Copy-on-write (summary page, sharing paragraph): each destination becomes a byte copy
    of its source in every layer; sources and all other blocks stay unchanged; the member that
    now owns the copy reads the same attention output."""
    spec = synth.SPECS["gqa_pressure"].scaled(num_seqs=8, ctx_range=(40, 90), shared_prompt=32)
    case = synth.make_case(spec, seed=15)
    bb = case.block_bytes
    layers = 3
    gen = np.random.default_rng(3)
    kps = [_raw_u8(case.k_pool)] + [gen.integers(0, 256, case.num_blocks * bb, dtype=np.uint8)
                                    for _ in range(layers - 1)]
    vps = [_raw_u8(case.v_pool)] + [gen.integers(0, 256, case.num_blocks * bb, dtype=np.uint8)
                                    for _ in range(layers - 1)]
    pairs = case.cow_pairs.numpy()
    for p in kps + vps:  # poison the destinations first
        p.reshape(case.num_blocks, bb)[pairs[:, 1]] = 0xFF
    before_k = [p.copy() for p in kps]
    before_v = [p.copy() for p in vps]
    assert orc.copy_blocks(kps, vps, pairs, block_bytes=bb) == 0
    for l in range(layers):
        for pools, before in ((kps, before_k), (vps, before_v)):
            a = pools[l].reshape(case.num_blocks, bb)
            b = before[l].reshape(case.num_blocks, bb)
            for src, dst in pairs:
                assert np.array_equal(a[dst], b[src]), "destination must equal source"
                assert np.array_equal(a[src], b[src]), "source must stay untouched"
            others = np.setdiff1d(np.arange(case.num_blocks), pairs[:, 1])
            assert np.array_equal(a[others], b[others]), "other blocks must stay untouched"
    got = run_decode(orc, case, k_pool=kps[0], v_pool=vps[0])
    assert np.abs(got - library_attention(case)).max() < 1e-12
    bad = np.array([[0, case.num_blocks]], np.int32)
    assert orc.copy_blocks(kps, vps, bad, block_bytes=bb) == -1


def pin_swap_round_trip(orc):
    """Swap-out then swap-in into other blocks ("When KV Capacity Runs Out", Figure 4) is
    bit-exact, lays the host buffer out as [block][layer][K,V], and after repointing the block
    table the attention output is unchanged bit for bit."""
    spec = synth.SPECS["gqa_pressure"].scaled(num_seqs=8, ctx_range=(40, 90), shared_prompt=32,
                                              victim_len=70, occupancy=0.5)
    case = synth.make_case(spec, seed=16)
    bb, layers = case.block_bytes, 2
    victim = spec.num_seqs - 1
    out_ids, in_ids = synth.swap_plan(case, victim, seed=5)
    gen = np.random.default_rng(4)
    kps = [_raw_u8(case.k_pool), gen.integers(0, 256, case.num_blocks * bb, dtype=np.uint8)]
    vps = [_raw_u8(case.v_pool), gen.integers(0, 256, case.num_blocks * bb, dtype=np.uint8)]
    ref = run_decode(orc, case)
    host = np.zeros(len(out_ids) * layers * 2 * bb, np.uint8)
    assert orc.swap_blocks(kps, vps, host, out_ids, block_bytes=bb, direction="out") == 0
    hv = host.reshape(len(out_ids), layers, 2, bb)
    for i, b in enumerate(out_ids):
        for l in range(layers):
            assert np.array_equal(hv[i, l, 0], kps[l].reshape(-1, bb)[b])
            assert np.array_equal(hv[i, l, 1], vps[l].reshape(-1, bb)[b])
    saved = [p.copy() for p in kps + vps]
    for p in kps + vps:  # the released blocks get reused by someone else
        p.reshape(-1, bb)[out_ids] = 0xFF
    assert orc.swap_blocks(kps, vps, host, in_ids, block_bytes=bb, direction="in") == 0
    for p, s in zip(kps + vps, saved):
        assert np.array_equal(p.reshape(-1, bb)[in_ids], s.reshape(-1, bb)[out_ids])
    bt = case.block_tables.clone()
    bt[victim, :len(in_ids)] = torch.from_numpy(in_ids)
    got = run_decode(orc, case, k_pool=kps[0], v_pool=vps[0], block_tables=bt)
    assert np.array_equal(got[victim], ref[victim])
    assert orc.swap_blocks(kps, vps, host, np.array([case.num_blocks], np.int32), block_bytes=bb,
                           direction="out") == -1


ALL_PINS = [
    pin_f16_decoder, pin_bf16_decoder, pin_e4m3_decoder, pin_paged_equals_library_attention,
    pin_closed_forms, pin_scales, pin_group_equals_replicated_heads, pin_permutation_invariance,
    pin_bounds, pin_write_kv, pin_toy_figures, pin_toy_permuted, pin_copy_on_write,
    pin_swap_round_trip, pin_e4m3_encoder, pin_write_kv_fp8,
    pin_prefill_equals_library_attention, pin_prefill_one_token_is_decode,
    pin_prefill_closed_forms,
]
