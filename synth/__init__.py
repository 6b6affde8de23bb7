"""Seeded synthetic inputs for the paged KV-cache hot path.

This module is shared by the tests, the benchmark, the oracle side and the CUDA side. It only
builds inputs -- block pools, block tables, context lengths, slot mappings, copy-on-write pairs
and swap lists -- with seeded random numbers. It holds none of the attention arithmetic and
imports neither the oracle nor the CUDA library.

Workload shapes come from the pages:
  * ``toy``          -- "When KV Capacity Runs Out", Figures 1-2: 4 physical blocks of 4 slots,
                        requests A and B with 2 blocks each (7 positions, then position 7 is written).
  * ``mha7b``        -- "KV Cache Preemption in vLLM", worked example (7B model, 48 GB GPU,
                        ~1,700 blocks, ~24 requests of 850-token prompts): 32 heads x 128, fp16.
  * ``gqa_pressure`` -- "41 · Preemption, Recomputation & KV Pressure", section 1 (100 requests
                        decoding, 16-token blocks) with 8 KV heads x 128 (GQA, 128 KiB/token over
                        32 layers), bf16; 25 groups of 4 samples share a 512-token prompt
                        (PagedAttention summary page, paragraph on sharing) and each step makes
                        one copy-on-write copy per group.
  * ``fp8_long``     -- FP8 KV cache ("switch the KV cache to FP8 ... roughly doubles capacity"),
                        256 sequences of 1,024-8,192 tokens, pool at 95% occupancy.
  * ``preemption``   -- ``gqa_pressure`` over 32 layers plus a 1,500-token victim
                        (section 3 of the note: 94 blocks x 2 MiB = 188 MiB swapped each way).

Readings (the pages leave these open): positions are 0-indexed (position t -> logical block t//B,
slot t%B); a context length counts the token written this step; when a drawn length is shorter
than the shared prompt it is raised to prompt + 1; unused slots and free blocks hold stale bytes,
which the tests model with NaN patterns so that any read of them shows up.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

TORCH_DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.uint8}
ELT_BYTES = {"f16": 2, "bf16": 2, "e4m3": 1}
# Bit patterns of a quiet NaN in each storage format (poison for stale slots).
NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F}
E4M3_MAX = 448.0


@dataclass
class DecodeSpec:
    """Shape of one decode workload."""

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str
    q_dtype: str
    ctx_range: Tuple[int, int] = (1, 1)        # inclusive uniform range of context lengths
    ctx_lens: Optional[Sequence[int]] = None   # explicit lengths (overrides ctx_range)
    num_blocks: Optional[int] = None           # pool size; None -> from occupancy
    occupancy: float = 0.95                    # used / pool when num_blocks is None
    group_size: int = 1                        # sequences sharing a prompt
    shared_prompt: int = 0                     # shared prompt tokens per group (multiple of B)
    cow_per_group: bool = False                # one copy-on-write destination per group
    num_layers: int = 1
    victim_len: Optional[int] = None           # context of the last sequence (preemption)

    def scaled(self, **kw) -> "DecodeSpec":
        return dataclasses.replace(self, **kw)


SPECS: Dict[str, DecodeSpec] = {
    "toy": DecodeSpec("toy", 2, 4, 4, 64, 4, "f16", "f16", ctx_lens=(8, 8), num_blocks=4),
    "mha7b": DecodeSpec("mha7b", 24, 32, 32, 128, 16, "f16", "f16", ctx_range=(850, 1100),
                        num_blocks=1700),
    "gqa_pressure": DecodeSpec("gqa_pressure", 100, 32, 8, 128, 16, "bf16", "bf16",
                               ctx_range=(256, 4096), group_size=4, shared_prompt=512,
                               cow_per_group=True),
    "fp8_long": DecodeSpec("fp8_long", 256, 32, 8, 128, 16, "e4m3", "bf16",
                           ctx_range=(1024, 8192)),
    "preemption": DecodeSpec("preemption", 100, 32, 8, 128, 16, "bf16", "bf16",
                             ctx_range=(256, 4096), group_size=4, shared_prompt=512,
                             cow_per_group=True, num_layers=32, victim_len=1500),
}


@dataclass
class PagedCase:
    """One seeded decode workload (all tensors on ``device``)."""

    spec: DecodeSpec
    seed: int
    q: torch.Tensor                  # [N][Hq][D] q dtype
    k_pools: List[torch.Tensor]      # per layer [num_blocks][Hkv][B][D] (uint8 for e4m3)
    v_pools: List[torch.Tensor]
    block_tables: torch.Tensor       # int32 [N][max_blocks_per_seq], -1 beyond the last block
    ctx_lens: torch.Tensor           # int32 [N]
    scale: float
    k_scale: float
    v_scale: float
    slot_mapping: torch.Tensor       # int64 [N]: slot of position ctx_len-1 (this step's token)
    k_new: torch.Tensor              # [N][Hkv][D] pool dtype: this step's K (layer 0)
    v_new: torch.Tensor
    cow_pairs: torch.Tensor          # int32 [P][2] (src, dst)
    free_blocks: List[int]           # physical blocks referenced by no table
    k_logical: Optional[List[torch.Tensor]] = None  # per seq [L][Hkv][D] pool dtype (layer 0)
    v_logical: Optional[List[torch.Tensor]] = None

    # convenience
    @property
    def num_blocks(self) -> int:
        return self.k_pools[0].shape[0]

    @property
    def max_blocks_per_seq(self) -> int:
        return self.block_tables.shape[1]

    @property
    def k_pool(self) -> torch.Tensor:
        return self.k_pools[0]

    @property
    def v_pool(self) -> torch.Tensor:
        return self.v_pools[0]

    @property
    def block_bytes(self) -> int:
        s = self.spec
        return s.num_kv_heads * s.block_size * s.head_dim * ELT_BYTES[s.kv_dtype]

    def to(self, device) -> "PagedCase":
        mv = lambda t: t.to(device) if isinstance(t, torch.Tensor) else t
        return dataclasses.replace(
            self, q=mv(self.q), k_pools=[mv(p) for p in self.k_pools],
            v_pools=[mv(p) for p in self.v_pools], block_tables=mv(self.block_tables),
            ctx_lens=mv(self.ctx_lens), slot_mapping=mv(self.slot_mapping),
            k_new=mv(self.k_new), v_new=mv(self.v_new), cow_pairs=mv(self.cow_pairs),
            k_logical=None if self.k_logical is None else [mv(t) for t in self.k_logical],
            v_logical=None if self.v_logical is None else [mv(t) for t in self.v_logical])


# ------------------------------------------------------------------ block assignment

@dataclass
class Assignment:
    ctx_lens: np.ndarray            # int32 [N]
    tables: np.ndarray              # int32 [N][max_blocks] (-1 padded)
    num_blocks: int
    cow_pairs: np.ndarray           # int32 [P][2]
    free_blocks: List[int]


def _draw_lengths(spec: DecodeSpec, rng: np.random.Generator) -> np.ndarray:
    if spec.ctx_lens is not None:
        lens = np.asarray(spec.ctx_lens, dtype=np.int64)
    else:
        lo, hi = spec.ctx_range
        lens = rng.integers(lo, hi + 1, size=spec.num_seqs)
    if spec.shared_prompt:
        lens = np.maximum(lens, spec.shared_prompt + 1)
    if spec.victim_len is not None:
        lens[-1] = spec.victim_len
    return lens.astype(np.int32)


def assign_blocks(spec: DecodeSpec, rng: np.random.Generator) -> Assignment:
    """Host block manager in miniature: allocate each sequence's blocks on demand from a
    seeded random permutation of the pool (so tables point all over it), sharing the prompt
    blocks inside each group and reserving one copy-on-write destination per group."""
    B = spec.block_size
    lens = _draw_lengths(spec, rng)
    n = len(lens)
    nb = [(int(L) + B - 1) // B for L in lens]
    shared = spec.shared_prompt // B if spec.shared_prompt else 0
    assert spec.shared_prompt % B == 0
    groups = (n + spec.group_size - 1) // spec.group_size
    used = sum(nb) - (shared * (n - groups) if shared else 0)
    cow = groups if spec.cow_per_group and shared else 0
    num_blocks = spec.num_blocks or int(math.ceil((used + cow) / spec.occupancy))
    assert num_blocks >= used + cow, "pool too small for the drawn lengths"
    order = rng.permutation(num_blocks)
    cursor = 0
    max_blocks = max(nb) if nb else 1
    tables = np.full((n, max_blocks), -1, dtype=np.int32)
    pairs = []
    for gidx in range(groups):
        members = range(gidx * spec.group_size, min(n, (gidx + 1) * spec.group_size))
        prompt_ids = order[cursor:cursor + shared]
        cursor += shared
        for s in members:
            tables[s, :shared] = prompt_ids
            own = nb[s] - shared
            tables[s, shared:nb[s]] = order[cursor:cursor + own]
            cursor += own
        if cow:
            dst = int(order[cursor])
            cursor += 1
            src = int(prompt_ids[-1])
            pairs.append((src, dst))
            first = members[0]
            tables[first, shared - 1] = dst  # the writer now owns a private copy
    free = [int(b) for b in order[cursor:]]
    return Assignment(lens, tables, num_blocks,
                      np.asarray(pairs, dtype=np.int32).reshape(-1, 2), free)


# ------------------------------------------------------------------ values

def _poison_fill(shape, kv_dtype: str, device) -> torch.Tensor:
    bits = NAN_BITS[kv_dtype]
    if kv_dtype == "e4m3":
        return torch.full(shape, bits, dtype=torch.uint8, device=device)
    return torch.full(shape, bits, dtype=torch.int16, device=device).view(TORCH_DTYPES[kv_dtype])


def quantize_e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    """Store x / scale as E4M3 bytes with the library cast (round to nearest even)."""
    y = (x / scale).clamp(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn).view(torch.uint8)


def _cast(x: torch.Tensor, kv_dtype: str, scale: float) -> torch.Tensor:
    if kv_dtype == "e4m3":
        return quantize_e4m3(x, scale)
    return x.to(TORCH_DTYPES[kv_dtype])


def make_case(spec: DecodeSpec, seed: int, *, device="cpu", logical: bool = True,
              poison: bool = True) -> PagedCase:
    """Build a seeded workload.

    logical=True generates each sequence's keys/values as contiguous tensors first and places
    them into the pool (the unpaged data stays available for checks); unused slots get NaN
    patterns when ``poison``. logical=False fills the whole pool with random values directly on
    ``device`` (large configurations) and, when ``poison``, overwrites unused slots with NaN.
    """
    rng = np.random.default_rng(seed)
    asg = assign_blocks(spec, rng)
    n, Hq, Hkv, D, B = spec.num_seqs, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.block_size
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    lens = asg.ctx_lens
    tables_t = torch.from_numpy(asg.tables)

    q32 = torch.randn((n, Hq, D), generator=gen, device=device)
    q = q32.to(TORCH_DTYPES[spec.q_dtype])

    k_pools, v_pools = [], []
    k_log = v_log = None
    k_scale = v_scale = 1.0
    shape = (asg.num_blocks, Hkv, B, D)
    if logical:
        assert spec.num_layers == 1, "logical mode builds one layer"
        # per-sequence logical keys/values; members of a group share the prompt part
        k32, v32 = [], []
        prompt = spec.shared_prompt
        group_prompt: Dict[int, Tuple[torch.Tensor, torch.Tensor]] = {}
        for s in range(n):
            L = int(lens[s])
            g = s // spec.group_size
            if prompt and g not in group_prompt:
                group_prompt[g] = (torch.randn((prompt, Hkv, D), generator=gen, device=device),
                                   torch.randn((prompt, Hkv, D), generator=gen, device=device))
            own = L - (prompt if prompt else 0)
            ks = torch.randn((own, Hkv, D), generator=gen, device=device)
            vs = torch.randn((own, Hkv, D), generator=gen, device=device)
            if prompt:
                ks = torch.cat([group_prompt[g][0], ks])
                vs = torch.cat([group_prompt[g][1], vs])
            k32.append(ks)
            v32.append(vs)
        if spec.kv_dtype == "e4m3":  # empty contexts hold no values: scale 1 if all are empty
            k_scale = max((float(t.abs().max()) for t in k32 if t.numel()),
                          default=E4M3_MAX) / E4M3_MAX
            v_scale = max((float(t.abs().max()) for t in v32 if t.numel()),
                          default=E4M3_MAX) / E4M3_MAX
        k_log = [_cast(t, spec.kv_dtype, k_scale) for t in k32]
        v_log = [_cast(t, spec.kv_dtype, v_scale) for t in v32]
        kp = _poison_fill(shape, spec.kv_dtype, device) if poison else \
            _cast(torch.randn(shape, generator=gen, device=device), spec.kv_dtype, 1.0)
        vp = _poison_fill(shape, spec.kv_dtype, device) if poison else \
            _cast(torch.randn(shape, generator=gen, device=device), spec.kv_dtype, 1.0)
        for s in range(n):
            L = int(lens[s])
            t = torch.arange(L, device=device)
            phys = tables_t.to(device)[s, (t // B)].long()
            slot = t % B
            kp[phys, :, slot, :] = k_log[s]
            vp[phys, :, slot, :] = v_log[s]
        k_pools, v_pools = [kp], [vp]
    else:
        for layer in range(spec.num_layers):
            kp, ks = _bulk_pool(shape, spec.kv_dtype, gen, device)
            vp, vs = _bulk_pool(shape, spec.kv_dtype, gen, device)
            if layer == 0:
                k_scale, v_scale = ks, vs
            if poison:
                _poison_unused(kp, asg, spec)
                _poison_unused(vp, asg, spec)
            k_pools.append(kp)
            v_pools.append(vp)

    # this step's token: position ctx_len - 1 of every sequence
    last = lens.astype(np.int64) - 1
    slots = np.array([int(asg.tables[s, last[s] // B]) * B + int(last[s] % B) if last[s] >= 0
                      else -1 for s in range(n)], dtype=np.int64)  # -1: padding (empty sequence)
    if k_log is not None:
        blank = torch.zeros((Hkv, D), dtype=TORCH_DTYPES[spec.kv_dtype], device=device)
        k_new = torch.stack([k_log[s][int(last[s])] if last[s] >= 0 else blank for s in range(n)])
        v_new = torch.stack([v_log[s][int(last[s])] if last[s] >= 0 else blank for s in range(n)])
    else:
        k_new = _cast(torch.randn((n, Hkv, D), generator=gen, device=device), spec.kv_dtype,
                      k_scale)
        v_new = _cast(torch.randn((n, Hkv, D), generator=gen, device=device), spec.kv_dtype,
                      v_scale)

    return PagedCase(
        spec=spec, seed=seed, q=q, k_pools=k_pools, v_pools=v_pools,
        block_tables=tables_t.to(device), ctx_lens=torch.from_numpy(lens).to(device),
        scale=1.0 / math.sqrt(D), k_scale=k_scale, v_scale=v_scale,
        slot_mapping=torch.from_numpy(slots).to(device), k_new=k_new, v_new=v_new,
        cow_pairs=torch.from_numpy(asg.cow_pairs).to(device), free_blocks=asg.free_blocks,
        k_logical=k_log, v_logical=v_log)


def _bulk_pool(shape, kv_dtype: str, gen: torch.Generator, device, chunk_rows: int = 4096):
    """Random pool filled chunk by chunk on ``device``; for E4M3 a first pass finds amax so
    that scale = amax / 448 (then the same chunks are regenerated and quantised)."""
    out = torch.empty(shape, dtype=TORCH_DTYPES[kv_dtype], device=device)
    rows = shape[0]
    inner = shape[1:]
    state = gen.get_state()
    scale = 1.0
    if kv_dtype == "e4m3":
        amax = 0.0
        for r0 in range(0, rows, chunk_rows):
            r1 = min(rows, r0 + chunk_rows)
            x = torch.randn((r1 - r0,) + tuple(inner), generator=gen, device=device)
            amax = max(amax, float(x.abs().max()))
        scale = amax / E4M3_MAX
        gen.set_state(state)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(inner), generator=gen, device=device)
        out[r0:r1] = _cast(x, kv_dtype, scale)
    return out, scale


def _poison_unused(pool: torch.Tensor, asg: Assignment, spec: DecodeSpec) -> None:
    """NaN-fill free blocks and the unwritten tail slots of each sequence's last block."""
    B = spec.block_size
    bits = NAN_BITS[spec.kv_dtype]
    raw = pool.view(torch.uint8) if spec.kv_dtype == "e4m3" else pool.view(torch.int16)
    if asg.free_blocks:
        raw[torch.tensor(asg.free_blocks, device=pool.device)] = bits
    for s, L in enumerate(asg.ctx_lens):
        L = int(L)
        if L % B:
            phys = int(asg.tables[s, (L - 1) // B])
            raw[phys, :, L % B:, :] = bits


def prefill_queries(case: PagedCase, seed: int, *, max_chunk: Optional[int] = None,
                    whole: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """A chunk of new query tokens per sequence for a prefill over ``case``'s cache: each
    sequence gets n in [1, L] tokens (all L when ``whole``; at most ``max_chunk``), standing at
    its last n positions. Returns (q_starts int32 [N + 1], q [total][Hq][D] in the q dtype), on
    the case's device."""
    spec = case.spec
    rng = np.random.default_rng(seed)
    lens = case.ctx_lens.cpu().numpy()
    n = np.zeros(len(lens), dtype=np.int64)
    for s, L in enumerate(lens):
        if L <= 0:
            continue
        hi = int(L) if max_chunk is None else min(int(L), max_chunk)
        n[s] = hi if whole else int(rng.integers(1, hi + 1))
    starts = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    dev = case.q.device
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    q = torch.randn((int(starts[-1]), spec.num_q_heads, spec.head_dim), generator=gen, device=dev)
    return torch.from_numpy(starts).to(dev), q.to(TORCH_DTYPES[spec.q_dtype])


def swap_plan(case: PagedCase, seq: int, seed: int) -> Tuple[np.ndarray, np.ndarray]:
    """Blocks of ``seq`` to swap out and a seeded choice of free blocks to swap them into
    ("When KV Capacity Runs Out", Figure 4: restored blocks may sit elsewhere)."""
    B = case.spec.block_size
    L = int(case.ctx_lens[seq])
    nb = (L + B - 1) // B
    out_ids = case.block_tables[seq, :nb].cpu().numpy().astype(np.int32)
    rng = np.random.default_rng(seed)
    assert len(case.free_blocks) >= nb, "not enough free blocks to swap back in"
    in_ids = rng.choice(np.asarray(case.free_blocks, dtype=np.int32), size=nb, replace=False)
    return out_ids, in_ids.astype(np.int32)


def permuted(case: PagedCase, seed: int) -> PagedCase:
    """The same logical workload with every physical block moved to a new seeded location
    (block tables, copy pairs and free list renamed accordingly)."""
    perm = torch.from_numpy(np.random.default_rng(seed).permutation(case.num_blocks)).long()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    dev = case.k_pool.device
    new_k = [torch.empty_like(p) for p in case.k_pools]
    new_v = [torch.empty_like(p) for p in case.v_pools]
    for a, b in zip(new_k, case.k_pools):
        a[perm.to(dev)] = b
    for a, b in zip(new_v, case.v_pools):
        a[perm.to(dev)] = b
    bt = case.block_tables.cpu().long()
    bt = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).to(torch.int32)
    pairs = perm[case.cow_pairs.cpu().long()].to(torch.int32) if case.cow_pairs.numel() else \
        case.cow_pairs.cpu()
    B = case.spec.block_size
    sm = case.slot_mapping.cpu()
    sm = perm[sm // B] * B + sm % B
    return dataclasses.replace(
        case, k_pools=new_k, v_pools=new_v, block_tables=bt.to(case.block_tables.device),
        cow_pairs=pairs.to(case.cow_pairs.device), slot_mapping=sm.to(case.slot_mapping.device),
        free_blocks=[int(perm[b]) for b in case.free_blocks])
