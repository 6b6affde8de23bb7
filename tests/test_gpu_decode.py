"""pa_decode on the GPU against the fp64 oracle, through the C ABI (needs a GB300)."""
import numpy as np
import pytest
import torch

import pins
import synth
from helpers import TOL, gpu_decode, max_abs_err, oracle_decode

pytestmark = pytest.mark.gpu

import paged_kv_cache_38_gb300 as pa  # noqa: E402


def _specs():
    S = synth.SPECS
    extra = [
        synth.DecodeSpec("bf16_g8_b16", 5, 64, 8, 128, 16, "bf16", "bf16", ctx_range=(1, 300)),
        synth.DecodeSpec("f16_g4_d64_b8", 6, 16, 4, 64, 8, "f16", "f16", ctx_range=(1, 120)),
        synth.DecodeSpec("bf16_g1_b4", 4, 4, 4, 128, 4, "bf16", "bf16", ctx_range=(1, 70)),
        synth.DecodeSpec("e4m3_g2", 3, 8, 4, 128, 16, "e4m3", "bf16", ctx_range=(1, 200)),
        synth.DecodeSpec("e4m3_g16_b32", 3, 32, 2, 128, 32, "e4m3", "f16", ctx_range=(40, 260)),
        S["gqa_pressure"].scaled(name="gqa_small", num_seqs=12, ctx_range=(40, 700),
                                 shared_prompt=64),
        # blocks larger than a pipeline stage: each copy brings part of one block
        synth.DecodeSpec("bf16_g4_b64", 5, 16, 4, 128, 64, "bf16", "bf16", ctx_range=(1, 700)),
        synth.DecodeSpec("f16_g8_d64_b64", 4, 16, 2, 64, 64, "f16", "f16", ctx_range=(1, 400)),
        synth.DecodeSpec("e4m3_g4_b64", 4, 16, 4, 128, 64, "e4m3", "bf16", ctx_range=(1, 600)),
        synth.DecodeSpec("bf16_g2_b32", 4, 8, 4, 128, 32, "bf16", "bf16", ctx_range=(1, 300)),
        synth.DecodeSpec("f16_g1_b64", 3, 4, 4, 128, 64, "f16", "f16", ctx_range=(1, 300)),
    ]
    return pins.small_specs() + extra


SPECS = _specs()


def _splits(spec):
    st = max(16, spec.block_size)
    return [0, st, 3 * st]


CASES = [(s, sp) for s in SPECS for sp in _splits(s)]


@pytest.mark.parametrize("spec,split", CASES, ids=[f"{s.name}-split{sp}" for s, sp in CASES])
def test_decode_matches_oracle(spec, split):
    case = synth.make_case(spec, seed=300).to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(case, split_tokens=split, err_flag=err)
    torch.cuda.synchronize()
    ref = oracle_decode(case)
    e = max_abs_err(out, ref)
    assert e <= TOL[spec.kv_dtype], f"{spec.name} split={split}: max abs err {e}"
    assert int(err.item()) == 0


@pytest.mark.parametrize("B,nseq", [(4, 100), (8, 160)])
def test_decode_e4m3_small_blocks_automatic_split(B, nseq):
    """An E4M3 cache of 4- or 8-token blocks with the automatic split: enough work that the
    planner would keep 2048 (or 1024) tokens per work item, more copy units than one item's
    table slice holds; it halves the split instead of refusing its own plan. An explicit split
    past that bound is refused (PA_EINVAL), as pa.h states."""
    spec = synth.DecodeSpec(f"e4m3_b{B}_auto", nseq, 8, 8, 128, B, "e4m3", "bf16",
                            ctx_range=(1000, 2000))
    case = synth.make_case(spec, seed=B).to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(case, split_tokens=0, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert max_abs_err(out, oracle_decode(case)) <= TOL["e4m3"]
    with pytest.raises(pa.PaError) as e:
        gpu_decode(case, split_tokens=256 * B)
    assert e.value.status == pa.PA_EINVAL


def test_decode_edge_lengths():
    """Empty, single-token, block-boundary and full-capacity contexts, NaN in stale slots."""
    for B in (4, 8, 16, 32, 64):
        lens = [0, 1, B - 1, B, B + 1, 2 * B - 1, 2 * B, 2 * B + 1, 10 * B, 10 * B - 3]
        spec = synth.DecodeSpec(f"edge_b{B}", len(lens), 8, 2, 128, B, "bf16", "bf16",
                                ctx_lens=tuple(lens))
        case = synth.make_case(spec, seed=B).to("cuda")
        for split in (0, max(16, B)):
            out = gpu_decode(case, split_tokens=split)
            ref = oracle_decode(case)
            assert max_abs_err(out, ref) <= TOL["bf16"], (B, split)
            assert torch.count_nonzero(out[0]).item() == 0, "empty context must give zeros"


@pytest.mark.parametrize("head_dim", [64, 128])
def test_decode_split_counts(head_dim):
    """Split counts on both sides of each combine batch boundary (8, 16, 32 partials per head)."""
    lens = (16 * 8, 16 * 8 + 1, 16 * 16, 16 * 16 + 3, 16 * 17, 16 * 32, 16 * 32 + 1, 16 * 40 - 5)
    spec = synth.DecodeSpec(f"splits_d{head_dim}", len(lens), 16, 4, head_dim, 16, "f16", "f16",
                            ctx_lens=lens)
    case = synth.make_case(spec, seed=head_dim).to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(case, split_tokens=16, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert max_abs_err(out, oracle_decode(case)) <= TOL["f16"]


def test_decode_many_sequences():
    """More sequences than one launch takes (4096) and than one scan chunk (416 threads), with
    every remainder size class of the last split present."""
    spec = synth.DecodeSpec("many", 4500, 4, 2, 64, 4, "f16", "f16", ctx_range=(0, 90))
    case = synth.make_case(spec, seed=17).to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(case, split_tokens=32, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert max_abs_err(out, oracle_decode(case)) <= TOL["f16"]


def test_decode_permutation_invariant_bitwise():
    """Moving blocks around the pool changes nothing, bit for bit (summary page, block table)."""
    spec = synth.SPECS["gqa_pressure"].scaled(num_seqs=16, ctx_range=(40, 500), shared_prompt=32)
    case = synth.make_case(spec, seed=31)
    ref = gpu_decode(case.to("cuda"))
    for seed in (1, 2, 3):
        p = synth.permuted(case, seed).to("cuda")
        assert torch.equal(gpu_decode(p), ref)


def test_decode_deterministic():
    case = synth.make_case(synth.SPECS["fp8_long"].scaled(num_seqs=6, ctx_range=(100, 900)),
                           seed=5).to("cuda")
    a = gpu_decode(case, split_tokens=64)
    b = gpu_decode(case, split_tokens=64)
    assert torch.equal(a, b)


def test_decode_bad_block_and_length_flags():
    spec = synth.DecodeSpec("flags", 4, 8, 2, 128, 16, "bf16", "bf16", ctx_lens=(40, 40, 40, 40))
    case = synth.make_case(spec, seed=9).to("cuda")
    bt = case.block_tables.clone()
    bt[1, 1] = case.num_blocks + 5  # outside the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(case, block_tables=bt, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_ERR_BLOCK_ID
    ref = oracle_decode(case)
    for s in (0, 2, 3):
        assert max_abs_err(out[s], ref[s]) <= TOL["bf16"]
    assert torch.isfinite(out[1].float()).all(), "a skipped block must not poison the row"

    err.zero_()
    cl = case.ctx_lens.clone()
    cl[2] = 9999  # beyond max_ctx_len and the table capacity
    out = gpu_decode(case, ctx_lens=cl, err_flag=err, max_ctx_len=48)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_ERR_CTX_LEN
    assert torch.count_nonzero(out[2]).item() == 0


def test_decode_host_validation():
    case = synth.make_case(synth.SPECS["toy"], seed=1).to("cuda")
    with pytest.raises(pa.PaError) as e:
        gpu_decode(case, split_tokens=10)  # not a multiple of 16
    assert e.value.status == pa.PA_EINVAL
    bad = synth.DecodeSpec("g3", 1, 6, 2, 64, 4, "f16", "f16", ctx_lens=(4,), num_blocks=4)
    c3 = synth.make_case(bad, seed=1).to("cuda")
    with pytest.raises(pa.PaError) as e:
        gpu_decode(c3)
    assert e.value.status == pa.PA_EUNSUPPORTED


# Full-size workloads in the launch configuration the benchmark times: every sequence of the
# step is decoded, a seeded sample of sequences is checked against the oracle.
FULL = ["mha7b", "gqa_pressure", "fp8_long"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled(name):
    spec = synth.SPECS[name]
    case = synth.make_case(spec, seed=38, device="cuda", logical=False, poison=True)
    pa.pa_write_kv(case.k_new, case.v_new, case.k_pool, case.v_pool, case.slot_mapping)
    if case.cow_pairs.numel():
        pa.pa_copy_blocks([case.k_pool], [case.v_pool], case.cow_pairs)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    import bench

    out = gpu_decode(case, err_flag=err, max_ctx_len=int(case.ctx_lens.max()),
                     split_tokens=bench.split_tokens_for(spec))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rng = np.random.default_rng(7)
    seqs = sorted(rng.choice(spec.num_seqs, size=min(6, spec.num_seqs), replace=False).tolist())
    seqs.append(int(torch.argmax(case.ctx_lens).item()))
    ref = oracle_decode(case, seqs)
    e = max_abs_err(out[torch.as_tensor(seqs, device="cuda")], ref)
    assert e <= TOL[spec.kv_dtype], f"{name}: max abs err {e}"
    assert torch.isfinite(out.float()).all()
