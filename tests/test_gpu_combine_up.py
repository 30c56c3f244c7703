"""GPU parity of the fused split-KV merge + up-projection (mla_combine_up_project).

The decode's partials are merged and projected in one launch.  Expected
values come from the fp64 oracle (latent attention of the pages' absorbed
score, then o = W^UV o_lat); the same workspace is also run through the
two-call path (mla_splitkv_combine, mla_up_project) for comparison.  Cases
cover S = 2 with two row blocks, H not a power of two, query-row counts
that are not a multiple of the 32-row tile, and single long sequences split
into more than 32 and more than 64 segments (the weights of segments 32..95
are held in a row's second and third register of the lanes).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, bits, f64
from mla_latent_kv_68_b300 import binding as mb

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192.0)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_68_b300 import build
    build.build()
    mb.lib()
    yield
    assert mb.read_status() == mb.MLA_OK


def _case(B, S, H, seqlens, seed):
    g = torch.Generator().manual_seed(seed)
    Lmax = max(seqlens)
    c = torch.zeros(B, Lmax, 512)
    k = torch.zeros(B, Lmax, 64)
    for b, L in enumerate(seqlens):
        c[b, :L] = torch.randn(L, 512, generator=g)
        k[b, :L] = torch.randn(L, 64, generator=g)
    q = torch.cat([0.5 * torch.randn(B, S, H, 512, generator=g),
                   torch.randn(B, S, H, 64, generator=g)], dim=-1)
    W = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    return (q.to(torch.bfloat16), c.to(torch.bfloat16), k.to(torch.bfloat16),
            torch.tensor(seqlens, dtype=torch.int32), W)


CASES = [
    (1, 1, 16, [256], 1),
    (3, 1, 128, [1, 64, 65], 2),
    (2, 2, 128, [2, 130], 3),
    (4, 1, 96, [17, 300, 1000, 4096], 4),
    (2, 2, 96, [77, 2048], 5),
    (33, 1, 128, [4096] * 33, 6),        # 33 query rows: a second, partly filled row tile
    (1, 1, 128, [6144], 7),              # 48 tiles over more groups: empty groups' slots skipped
    (1, 2, 64, [40000], 8),              # one sequence over every group (more than 64 segments)
]


@pytest.mark.parametrize("B,S,H,seqlens,seed", CASES)
def test_combine_up_matches_oracle_and_two_call_path(B, S, H, seqlens, seed):
    q, c, k, sl, W = _case(B, S, H, seqlens, seed)
    ws = mb.new_workspace(B, S, H)
    qd, cd, kd, sld, Wd = q.cuda(), c.cuda(), k.cuda(), sl.cuda(), W.cuda()
    mb.decode(qd, cd, kd, sld, ws)
    fused = torch.full((B, S, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.combine_up_project(ws, Wd, fused)
    o = torch.empty(B, S, H, 512, dtype=torch.bfloat16, device="cuda")
    mb.splitkv_combine(ws, o)
    two = torch.empty(B, S, H, 128, dtype=torch.bfloat16, device="cuda")
    mb.up_project(o, Wd, two)
    assert mb.read_status(ws) == mb.MLA_OK
    lat = oracle.latent_attention(bits(q), bits(c), bits(k), sl.numpy(), d_r=64, softmax_scale=SCALE)
    # o = W^UV o_lat per head, in fp64 on the oracle's latent result
    ref = np.einsum("bshk,hvk->bshv", lat, W.double().numpy())
    got = f64(fused)
    assert_close(got, ref, what=f"fused out B{B} S{S} H{H}")
    # the two paths round o_lat to bf16 alike and differ only in summation order
    assert_close(got, f64(two), max_abs=1e-2, rel=2e-3, what=f"fused vs two-call B{B} S{S} H{H}")


def test_combine_up_step_runs_twice_alike():
    B, S, H, seqlens = 5, 1, 128, [4999, 1, 3000, 129, 8191]
    q, c, k, sl, W = _case(B, S, H, seqlens, 9)
    ws = mb.new_workspace(B, S, H)
    qd, cd, kd, sld, Wd = q.cuda(), c.cuda(), k.cuda(), sl.cuda(), W.cuda()
    outs = []
    for _ in range(2):
        mb.decode(qd, cd, kd, sld, ws)
        out = torch.empty(B, S, H, 128, dtype=torch.bfloat16, device="cuda")
        mb.combine_up_project(ws, Wd, out)
        outs.append(out)
    assert mb.read_status(ws) == mb.MLA_OK
    assert torch.equal(outs[0], outs[1])


def test_combine_up_with_cache_values_beyond_fp16_range():
    # cache rows near 1e5 (see the decode test of the same name): the split
    # partials carry a power-of-two exponent per half row, which the fused
    # merge applies before the up-projection
    g = torch.Generator().manual_seed(41)
    B, S, H, seqlens = 2, 1, 128, [7000, 2500]
    Lmax = max(seqlens)
    c = torch.zeros(B, Lmax, 512)
    k = torch.zeros(B, Lmax, 64)
    for b, L in enumerate(seqlens):
        c[b, :L] = 1e5 * (1.0 + 0.01 * torch.randn(L, 512, generator=g))
        k[b, :L] = torch.randn(L, 64, generator=g)
    q = torch.cat([5e-4 * torch.randn(B, S, H, 512, generator=g),
                   torch.randn(B, S, H, 64, generator=g)], dim=-1).to(torch.bfloat16)
    c, k = c.to(torch.bfloat16), k.to(torch.bfloat16)
    W = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    ws = mb.new_workspace(B, S, H)
    mb.decode(q.cuda(), c.cuda(), k.cuda(), sl.cuda(), ws)
    fused = torch.full((B, S, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.combine_up_project(ws, W.cuda(), fused)
    assert mb.read_status(ws) == mb.MLA_OK
    lat = oracle.latent_attention(bits(q), bits(c), bits(k), sl.numpy(), d_r=64, softmax_scale=SCALE)
    ref = np.einsum("bshk,hvk->bshv", lat, W.double().numpy())
    assert np.abs(lat).max() > 65504.0
    assert_close(f64(fused) / 1e5, ref / 1e5, what="fused merge, cache values near 1e5")
