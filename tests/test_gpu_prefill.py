"""pa_prefill (tcgen05 tensor cores) against the fp64 oracle, through the C ABI (needs a GB300).

Each sequence's chunk of n new tokens stands at its last n cache positions and attends
causally; whole prompts (n = L), partial chunks and one-token chunks; stale slots and free
blocks hold NaN, so any read past a sequence's context shows."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import TOL

import paged_kv_cache_38_gb300 as pa  # noqa: E402

pytestmark = pytest.mark.gpu

SPECS = [
    synth.DecodeSpec("pf_bf16_g4_b16", 6, 16, 4, 128, 16, "bf16", "bf16", ctx_range=(1, 300)),
    synth.DecodeSpec("pf_f16_g1_b16", 4, 4, 4, 128, 16, "f16", "f16", ctx_range=(1, 260)),
    synth.DecodeSpec("pf_bf16_g8_d64_b32", 5, 16, 2, 64, 32, "bf16", "bf16", ctx_range=(1, 200)),
    synth.DecodeSpec("pf_f16_g16_b64", 3, 32, 2, 128, 64, "f16", "f16", ctx_range=(1, 330)),
    synth.DecodeSpec("pf_bf16_g2_d64_b8", 5, 8, 4, 64, 8, "bf16", "bf16", ctx_range=(1, 150)),
    # an E4M3 cache (per-tensor k_scale / v_scale) with bf16 and with f16 queries
    synth.DecodeSpec("pf_e4m3_g4_b16", 6, 32, 8, 128, 16, "e4m3", "bf16", ctx_range=(1, 300)),
    synth.DecodeSpec("pf_e4m3_g1_b32_f16q", 4, 4, 4, 128, 32, "e4m3", "f16", ctx_range=(1, 260)),
    synth.DecodeSpec("pf_e4m3_g16_b8", 3, 32, 2, 128, 8, "e4m3", "bf16", ctx_range=(1, 200)),
]
CHUNKS = ["whole", "partial", "one"]


def _oracle(case, qs, q):
    spec = case.spec
    return oracle.load().prefill(q.cpu(), case.k_pool.cpu(), case.v_pool.cpu(),
                                 case.block_tables.cpu(), case.ctx_lens.cpu(), qs.cpu(),
                                 dtype=spec.kv_dtype, q_dtype=spec.q_dtype,
                                 num_q_heads=spec.num_q_heads, num_kv_heads=spec.num_kv_heads,
                                 head_dim=spec.head_dim, block_size=spec.block_size,
                                 scale=case.scale, k_scale=case.k_scale, v_scale=case.v_scale)


def _err(out, ref):
    g = out.double().cpu().numpy()
    return float(np.abs(g - ref).max()) if np.all(np.isfinite(g)) else float("inf")


@pytest.mark.parametrize("spec,chunk", [(s, c) for s in SPECS for c in CHUNKS],
                         ids=[f"{s.name}-{c}" for s in SPECS for c in CHUNKS])
def test_prefill_matches_oracle(spec, chunk):
    case = synth.make_case(spec, seed=700)
    qs, q = synth.prefill_queries(case, seed=7, whole=chunk == "whole",
                                  max_chunk=1 if chunk == "one" else None)
    ref = _oracle(case, qs, q)
    g = case.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pa.pa_prefill(q.cuda(), g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qs.cuda(),
                        case.scale, err_flag=err, k_scale=case.k_scale, v_scale=case.v_scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    e = _err(out, ref)
    assert e <= TOL[spec.kv_dtype], f"{spec.name} {chunk}: max abs err {e}"


def test_prefill_long_chunks():
    """Long prompts and chunks (several query tiles and many key tiles per sequence)."""
    spec = synth.DecodeSpec("pf_long", 3, 32, 8, 128, 16, "bf16", "bf16", ctx_lens=(1500, 777, 2048))
    case = synth.make_case(spec, seed=71)
    qs = torch.tensor([0, 1500, 1500 + 300, 1500 + 300 + 1024], dtype=torch.int32)
    q = torch.randn(int(qs[-1]), 32, 128, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    ref = _oracle(case, qs, q)
    g = case.to("cuda")
    out = pa.pa_prefill(q.cuda(), g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qs.cuda(),
                        case.scale)
    torch.cuda.synchronize()
    assert _err(out, ref) <= TOL["bf16"]


def test_prefill_growing_scores_rescale():
    """Scores that grow along the context (each key row scaled by 1 + position / 100): every
    row's running maximum passes the lazy-rescaling threshold several times, so O is rescaled
    in tensor memory, and the result still matches the oracle (V scaled down so that outputs
    stay below 1 and bf16 output rounding stays far inside the tolerance)."""
    spec = synth.DecodeSpec("pf_grow", 3, 16, 4, 128, 16, "bf16", "bf16", ctx_lens=(700, 400, 1000))
    case = synth.make_case(spec, seed=72)
    bt, lens = case.block_tables.numpy(), case.ctx_lens.numpy()
    kp, vp = case.k_pool, case.v_pool
    done = set()
    for si in range(spec.num_seqs):
        for t in range(int(lens[si])):
            blk, off = int(bt[si, t // spec.block_size]), t % spec.block_size
            if (blk, off) in done:
                continue
            done.add((blk, off))
            kp[blk, :, off] = (kp[blk, :, off].float() * (1.0 + t / 100.0)).to(kp.dtype)
            vp[blk, :, off] = (vp[blk, :, off].float() * 0.25).to(vp.dtype)
    qs, q = synth.prefill_queries(case, seed=8, whole=True)
    ref = _oracle(case, qs, q)
    g = case.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pa.pa_prefill(q.cuda(), g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qs.cuda(),
                        case.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _err(out, ref) <= TOL["bf16"]


def test_prefill_bad_lengths_flagged():
    spec = synth.DecodeSpec("pf_bad", 3, 8, 2, 128, 16, "bf16", "bf16", ctx_lens=(40, 40, 40))
    case = synth.make_case(spec, seed=5).to("cuda")
    qs = torch.tensor([0, 10, 60, 70], dtype=torch.int32, device="cuda")  # 50 > 40 for seq 1
    q = torch.randn(70, 8, 128, device="cuda").to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pa.pa_prefill(q, case.k_pool, case.v_pool, case.block_tables, case.ctx_lens, qs,
                        case.scale, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_ERR_CTX_LEN
    assert torch.count_nonzero(out[10:60]).item() == 0
    ref = _oracle(case, qs.cpu(), q.cpu())
    assert _err(out[:10], ref[:10]) <= TOL["bf16"] and _err(out[60:], ref[60:]) <= TOL["bf16"]


def test_prefill_host_validation():
    case = synth.make_case(synth.SPECS["toy"], seed=1).to("cuda")  # block_size 4: not built
    qs = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    q = torch.randn(2, 4, 64, device="cuda").to(torch.float16)
    with pytest.raises(pa.PaError) as e:
        pa.pa_prefill(q, case.k_pool, case.v_pool, case.block_tables, case.ctx_lens, qs, 0.125)
    assert e.value.status == pa.PA_EUNSUPPORTED


@pytest.mark.parametrize("group,n", [(4, 20), (4, 33), (1, 129), (16, 9), (8, 17)])
def test_prefill_tile_edges(group, n):
    """Chunks that end just inside or just past a 128-row query tile (128 / G tokens)."""
    hkv = 2
    spec = synth.DecodeSpec(f"pf_edge_g{group}", 2, hkv * group, hkv, 128, 16, "bf16", "bf16",
                            ctx_lens=(n + 37, n))
    case = synth.make_case(spec, seed=90 + group)
    qs = torch.tensor([0, n, 2 * n], dtype=torch.int32)
    q = torch.randn(2 * n, hkv * group, 128, generator=torch.Generator().manual_seed(n)).to(torch.bfloat16)
    ref = _oracle(case, qs, q)
    g = case.to("cuda")
    out = pa.pa_prefill(q.cuda(), g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qs.cuda(),
                        case.scale)
    torch.cuda.synchronize()
    assert _err(out, ref) <= TOL["bf16"]


def test_prefill_permutation_invariant_bitwise():
    """Moving blocks around the pool changes nothing, bit for bit (summary page, block table):
    the key tiles are gathered in logical order whatever their physical place."""
    spec = synth.DecodeSpec("pf_perm", 5, 32, 8, 128, 16, "bf16", "bf16", ctx_range=(100, 700))
    case = synth.make_case(spec, seed=123)
    qs, q = synth.prefill_queries(case, seed=4)
    qd, qsd = q.cuda(), qs.cuda()

    def run(c):
        g = c.to("cuda")
        return pa.pa_prefill(qd, g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qsd, c.scale)

    ref = run(case)
    for seed in (1, 2, 3):
        assert torch.equal(run(synth.permuted(case, seed)), ref)


def test_prefill_chunk_longer_than_max_q_len_flagged():
    """A chunk longer than the max_q_len the grid was sized with is an error, not a silently
    half-written output: the flag is set and the rows the grid covers are zero."""
    spec = synth.DecodeSpec("pf_maxq", 2, 8, 2, 128, 16, "bf16", "bf16", ctx_lens=(300, 90))
    case = synth.make_case(spec, seed=6).to("cuda")
    qs = torch.tensor([0, 300, 390], dtype=torch.int32, device="cuda")
    q = torch.randn(390, 8, 128, device="cuda").to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    pa.pa_prefill(q, case.k_pool, case.v_pool, case.block_tables, case.ctx_lens, qs, case.scale,
                  out=out, max_q_len=100, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_ERR_CTX_LEN
    covered = 128 // 4 * ((100 + 31) // 32)  # tokens per 128-row tile (G = 4) x tiles
    assert torch.count_nonzero(out[:covered]).item() == 0
    ref = _oracle(case, qs.cpu(), q.cpu())
    assert _err(out[300:], ref[300:]) <= TOL["bf16"]  # the other sequence is unaffected


def test_prefill_work_distribution():
    """More work items (query tiles x kv heads x sequences) than the persistent CTAs: the
    dynamic work counter and the round-robin assignment give the same bits, both matching the
    oracle; an explicit counter left dirty by a previous call is reset by the call itself."""
    spec = synth.DecodeSpec("pf_many", 40, 32, 8, 128, 16, "bf16", "bf16", ctx_range=(1, 700))
    case = synth.make_case(spec, seed=77)
    qs, q = synth.prefill_queries(case, seed=8)
    ref = _oracle(case, qs, q)
    g = case.to("cuda")
    qd, qsd = q.cuda(), qs.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for kw in (dict(dynamic=False),
               dict(work_counter=torch.full((1,), 12345, dtype=torch.int32, device="cuda")),
               dict()):
        outs.append(pa.pa_prefill(qd, g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qsd,
                                  case.scale, err_flag=err, **kw))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _err(outs[0], ref) <= TOL["bf16"]
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


def test_prefill_in_cuda_graph_bitwise():
    """pa_prefill captured in a CUDA graph (the work counter's reset and the persistent kernel
    both in the graph) and replayed gives the eager call's bits, replay after replay."""
    spec = synth.DecodeSpec("pf_graph", 6, 32, 8, 128, 16, "bf16", "bf16", ctx_range=(50, 900))
    case = synth.make_case(spec, seed=31)
    qs, q = synth.prefill_queries(case, seed=12)
    g = case.to("cuda")
    qd, qsd = q.cuda(), qs.cuda()
    max_q = int((qs[1:] - qs[:-1]).max())
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(qd)

    def call():
        pa.pa_prefill(qd, g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qsd, case.scale,
                      out=out, max_q_len=max_q, work_counter=counter)

    call()
    torch.cuda.synchronize()
    eager = out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for _ in range(2):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager)


def test_prefill_out_of_pool_block_flagged():
    """A block-table entry outside the pool sets PA_ERR_BLOCK_ID; the other sequences of the
    launch are unaffected (their rows still match the oracle)."""
    spec = synth.DecodeSpec("pf_badblk", 4, 16, 4, 128, 16, "bf16", "bf16", ctx_lens=(200, 120, 300, 90))
    case = synth.make_case(spec, seed=21)
    qs, q = synth.prefill_queries(case, seed=3, whole=True)
    ref = _oracle(case, qs, q)
    g = case.to("cuda")
    bt = g.block_tables.clone()
    bt[1, 2] = g.k_pool.shape[0] + 5  # sequence 1 reads a block past the pool
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pa.pa_prefill(q.cuda(), g.k_pool, g.v_pool, bt, g.ctx_lens, qs.cuda(), case.scale,
                        err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pa.PA_ERR_BLOCK_ID
    lo, hi = int(qs[1]), int(qs[2])
    keep = torch.cat([out[:lo], out[hi:]])
    want = np.concatenate([ref[:lo], ref[hi:]])
    assert _err(keep, want) <= TOL["bf16"]


@pytest.mark.parametrize("log2_mag", [16, -20])
def test_prefill_e4m3_queries_beyond_f16_range(log2_mag):
    """bf16 queries scaled by 2^16 (above f16's largest value) or 2^-20 (below its normal range),
    with the softmax scale divided by the same power of two: the scores are those of the
    unscaled queries, exactly. The kernel moves each query row to f16 with its own power-of-two
    scale, so both match the oracle (which reads the bf16 values exactly); a plain conversion
    would overflow or lose the small values."""
    spec = synth.DecodeSpec("pf_e4m3_mag", 4, 32, 8, 128, 16, "e4m3", "bf16", ctx_range=(40, 400))
    case = synth.make_case(spec, seed=77)
    qs, q = synth.prefill_queries(case, seed=5, whole=True)
    q = (q.float() * 2.0 ** log2_mag).to(torch.bfloat16)  # exact: a power of two
    case = dataclasses.replace(case, scale=case.scale * 2.0 ** -log2_mag)
    ref = _oracle(case, qs, q)
    g = case.to("cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pa.pa_prefill(q.cuda(), g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qs.cuda(),
                        case.scale, err_flag=err, k_scale=case.k_scale, v_scale=case.v_scale)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert _err(out, ref) <= TOL["e4m3"]


def test_prefill_e4m3_recompute_matches_decode():
    """A recomputed request of the FP8 workload: its whole history is prefilled over the E4M3
    cache, and the last row of the chunk equals what pa_decode computes for that position."""
    spec = synth.SPECS["fp8_long"].scaled(num_seqs=6, ctx_range=(300, 1500))
    case = synth.make_case(spec, seed=78)
    qs, q = synth.prefill_queries(case, seed=6, whole=True)
    ref = _oracle(case, qs, q)
    g = case.to("cuda")
    out = pa.pa_prefill(q.cuda(), g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, qs.cuda(),
                        case.scale, k_scale=case.k_scale, v_scale=case.v_scale)
    last = (qs[1:] - 1).long()
    dec = pa.pa_decode(q[last].cuda(), g.k_pool, g.v_pool, g.block_tables, g.ctx_lens, case.scale,
                       k_scale=case.k_scale, v_scale=case.v_scale)
    torch.cuda.synchronize()
    assert _err(out, ref) <= TOL["e4m3"]
    assert _err(dec, ref[last.numpy()]) <= TOL["e4m3"]
    assert float((out[last.cuda()].float() - dec.float()).abs().max()) <= 2 * TOL["e4m3"]


def test_prefill_fp8_recompute_after_quantise_on_write():
    """The FP8 workload's recompute path end to end: a victim's retained history (bf16 K/V) is
    quantised into an E4M3 cache by pa_write_kv_fp8 at fresh, scattered slots, prefilled over
    that cache by pa_prefill, and its next step decoded by pa_decode; both equal the oracle
    run on the bytes the kernel wrote (and the write equals the oracle's quantise-on-write)."""
    g = torch.Generator().manual_seed(12)
    hq, hkv, d, B, L = 32, 8, 128, 16, 700
    nblk = 200
    k = torch.randn(L, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(L, hkv, d, generator=g).to(torch.bfloat16)
    ks, vs = float(k.float().abs().max()) / 448.0, float(v.float().abs().max()) / 448.0
    table = torch.randperm(nblk, generator=g)[: (L + B - 1) // B].to(torch.int32)
    pos = torch.arange(L)
    slots = (table[pos // B].long() * B + pos % B).to(torch.int64)
    kp = torch.full((nblk, hkv, B, d), 0x7F, dtype=torch.uint8)  # stale bytes: E4M3 NaN
    vp = kp.clone()
    exp_k, exp_v = kp.numpy().copy(), vp.numpy().copy()
    orc = oracle.load()
    assert orc.write_kv_fp8(k, v, exp_k, exp_v, slots, src_dtype="bf16", num_kv_heads=hkv,
                            head_dim=d, block_size=B, k_scale=ks, v_scale=vs) == 0
    gk, gv = kp.cuda(), vp.cuda()
    pa.pa_write_kv_fp8(k.cuda(), v.cuda(), gk, gv, slots.cuda(), ks, vs)
    torch.cuda.synchronize()
    assert np.array_equal(gk.cpu().numpy(), exp_k) and np.array_equal(gv.cpu().numpy(), exp_v)
    bt = torch.full((1, 64), -1, dtype=torch.int32)
    bt[0, : table.numel()] = table
    cl = torch.tensor([L], dtype=torch.int32)
    qs = torch.tensor([0, L], dtype=torch.int32)
    q = torch.randn(L, hq, d, generator=g).to(torch.bfloat16)
    scale = 1.0 / math.sqrt(d)
    ref = orc.prefill(q, torch.from_numpy(exp_k), torch.from_numpy(exp_v), bt, cl, qs,
                      dtype="e4m3", q_dtype="bf16", num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                      block_size=B, scale=scale, k_scale=ks, v_scale=vs)
    out = pa.pa_prefill(q.cuda(), gk, gv, bt.cuda(), cl.cuda(), qs.cuda(), scale, k_scale=ks,
                        v_scale=vs)
    qd = torch.randn(1, hq, d, generator=g).to(torch.bfloat16)
    dec_ref = orc.decode(qd, torch.from_numpy(exp_k), torch.from_numpy(exp_v), bt, cl,
                         q_dtype="bf16", kv_dtype="e4m3", num_q_heads=hq, num_kv_heads=hkv,
                         head_dim=d, block_size=B, scale=scale, k_scale=ks, v_scale=vs)
    dec = pa.pa_decode(qd.cuda(), gk, gv, bt.cuda(), cl.cuda(), scale, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert _err(out, ref) <= TOL["e4m3"]
    assert _err(dec, dec_ref) <= TOL["e4m3"]
