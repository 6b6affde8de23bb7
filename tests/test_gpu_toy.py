"""The 4-block worked example ("When KV Capacity Runs Out", Figures 1-2) replayed with the GPU
kernels next to the oracle: pools bit-exact after every write, attention within tolerance."""
import numpy as np
import pytest
import torch

import oracle
import pins

pytestmark = pytest.mark.gpu

import paged_kv_cache_38_gb300 as pa  # noqa: E402


@pytest.mark.parametrize("seed", [None, 38, 39])
def test_toy_figures_on_gpu(seed):
    if seed is None:
        rename = {f"P{i}": i for i in range(4)}
    else:
        perm = np.random.default_rng(seed).permutation(4)
        rename = {f"P{i}": int(perm[i]) for i in range(4)}
    orc = oracle.load()
    script = pins._toy_script()
    nblk, B = int(script[0][1]), int(script[0][2])
    Hkv, D = 4, 64
    gen = torch.Generator().manual_seed(38)
    logical = {r: (torch.randn((12, Hkv, D), generator=gen).half(),
                   torch.randn((12, Hkv, D), generator=gen).half()) for r in "AB"}
    q = torch.randn((1, Hkv, D), generator=gen).half()
    host_k = np.full(nblk * Hkv * B * D * 2, 0xFF, np.uint8)
    host_v = host_k.copy()
    dev_k = torch.full((nblk, Hkv, B, D), float("nan"), dtype=torch.float16, device="cuda")
    dev_k.view(torch.uint8).fill_(0xFF)
    dev_v = dev_k.clone()
    tables, npos = {}, {}

    def write(r, pos, phys):
        sigma = torch.tensor([phys * B + pos % B], dtype=torch.int64)
        k, v = logical[r][0][pos:pos + 1], logical[r][1][pos:pos + 1]
        assert orc.write_kv(k, v, host_k, host_v, sigma, num_kv_heads=Hkv, head_dim=D,
                            block_size=B, kv_dtype="f16") == 0
        pa.pa_write_kv(k.cuda(), v.cuda(), dev_k, dev_v, sigma.cuda())
        torch.cuda.synchronize()
        assert np.array_equal(dev_k.view(torch.uint8).cpu().numpy().reshape(-1), host_k)
        assert np.array_equal(dev_v.view(torch.uint8).cpu().numpy().reshape(-1), host_v)

    for cmd in script[1:]:
        if cmd[0] == "own":
            tables[cmd[1]] = [rename[p] for p in cmd[2:]]
            npos[cmd[1]] = 7
            for pos in range(7):
                write(cmd[1], pos, tables[cmd[1]][pos // B])
        elif cmd[0] == "write":
            r, pos, blk = cmd[1], int(cmd[2]), rename[cmd[3]]
            write(r, pos, blk)
            npos[r] = pos + 1
        elif cmd[0] == "release":
            tables.pop(cmd[1])
            npos.pop(cmd[1])
        elif cmd[0] == "link":
            tables[cmd[1]].append(rename[cmd[2]])
        elif cmd[0] == "expect" and cmd[1] in tables:
            r = cmd[1]
            bt = torch.tensor([tables[r]], dtype=torch.int32)
            cl = torch.tensor([npos[r]], dtype=torch.int32)
            ref = orc.decode(q, host_k, host_v, bt, cl, q_dtype="f16", kv_dtype="f16",
                             num_q_heads=Hkv, num_kv_heads=Hkv, head_dim=D, block_size=B,
                             scale=1 / 8)
            out = pa.pa_decode(q.cuda(), dev_k, dev_v, bt.cuda(), cl.cuda(), 1 / 8)
            g = out.double().cpu().numpy()
            assert np.isfinite(g).all() and np.abs(g - ref).max() <= 2e-3, cmd
