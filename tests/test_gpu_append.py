"""GPU parity of the cache-append step (mla_cache_append) against the oracle.

"DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention / KeyValue":
c_t = W^DKV h_t and k^R_t = RoPE_t(W^KR h_t) land in the cache rows of the
new tokens, t = seqlens[b] - S + s.  Cases span d = 64 (one slice), a d
whose last 256-column slice is partly empty, the 7168 of the model at
positions up to 131071, S = 2, token counts that are not a multiple of the
token tile and more than one token tile, YaRN frequencies, and a position
past the cache (reported, other tokens still written).  Every other cache
row must keep its bytes.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import bits, f64
from mla_latent_kv_68_b300 import binding as mb

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_68_b300 import build
    build.build()
    mb.lib()
    yield
    assert mb.read_status() == mb.MLA_OK


def _case(B, S, d, seed):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn(B, S, d, generator=g).to(torch.bfloat16)
    wd = (torch.randn(512, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    wr = (torch.randn(64, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    return h, wd, wr


def _run(h, wd, wr, seqlens, Lmax, theta=None):
    B, S, d = h.shape
    c = torch.full((B, Lmax, 512), SENTINEL, dtype=torch.bfloat16, device="cuda")
    k = torch.full((B, Lmax, 64), SENTINEL, dtype=torch.bfloat16, device="cuda")
    ws = mb.cache_append_workspace(B, S, d)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    mb.cache_append(h.cuda(), wd.cuda(), wr.cuda(), sl.cuda(), c, k, ws, theta=theta)
    return c, k, ws


def _check(c, k, h, wd, wr, seqlens, theta=None, skip=()):
    B, S, d = h.shape
    pos = np.array([[L - S + s for s in range(S)] for L in seqlens]).reshape(-1)
    ref_c, ref_k = oracle.cache_append(bits(h).reshape(B * S, d), bits(wd), bits(wr), np.maximum(pos, 0),
                                       theta=theta)
    cg, kg = f64(c), f64(k)
    written = np.zeros(cg.shape[:2], bool)
    for n in range(B * S):
        b = n // S
        if b in skip:
            continue
        t = pos[n]
        written[b, t] = True
        for got, ref in ((cg[b, t], ref_c[n]), (kg[b, t], ref_k[n])):
            err = np.abs(got - ref)
            assert (err <= 2.0 ** -8 * np.abs(ref) + 1e-3).all(), (b, t, float(err.max()))
    assert (cg[~written] == SENTINEL).all() and (kg[~written] == SENTINEL).all()


@pytest.mark.parametrize("B,S,d,seqlens,Lmax", [
    (1, 1, 64, [1], 4),
    (3, 2, 448, [2, 50, 4097], 5000),
    (4, 1, 7168, [1, 100, 131072, 65536], 131072),
    (33, 1, 1024, list(range(1, 34)), 40),
    (150, 2, 512, [2 + (i * 37) % 900 for i in range(150)], 1000),
    # 600 tokens at d = 7168: 5 x 28 x 3 CTAs, more than can be resident at
    # once, so the GEMM and the finalize run as two launches
    (300, 2, 7168, [2 + (i * 53) % 500 for i in range(300)], 600),
])
def test_cache_append_matches_oracle(B, S, d, seqlens, Lmax):
    h, wd, wr = _case(B, S, d, seed=B * 7 + S * 3 + d)
    c, k, ws = _run(h, wd, wr, seqlens, Lmax)
    assert mb.read_status(ws) == mb.MLA_OK
    _check(c, k, h, wd, wr, seqlens)


def test_cache_append_with_yarn_frequencies():
    B, S, d, seqlens, Lmax = 2, 1, 7168, [4096, 131072], 131072
    h, wd, wr = _case(B, S, d, seed=11)
    th = oracle.yarn_theta(64)          # the expected value takes the oracle's frequencies
    c, k, ws = _run(h, wd, wr, seqlens, Lmax, theta=mb.yarn_frequencies())
    assert mb.read_status(ws) == mb.MLA_OK
    _check(c, k, h, wd, wr, seqlens, theta=th)


def test_cache_append_reports_a_position_past_the_cache():
    B, S, d, Lmax = 3, 1, 256, 64
    seqlens = [10, 65, 64]   # sequence 1 would write row 64 of a 64-row cache
    h, wd, wr = _case(B, S, d, seed=12)
    c, k, ws = _run(h, wd, wr, seqlens, Lmax)
    assert mb.read_status(ws) == mb.MLA_ERR_BAD_SEQLEN
    assert mb.read_status(ws) == mb.MLA_OK   # reading clears it
    _check(c, k, h, wd, wr, [10, 1, 64], skip=(1,))


def test_cache_append_twice_with_one_workspace():
    # a workspace serves call after call: nothing of the first call's partial
    # products leaks into the second's result
    B, S, d, seqlens, Lmax = 4, 2, 1024, [2, 50, 300, 9], 320
    ws = mb.cache_append_workspace(B, S, d)
    for seed in (21, 22):
        h, wd, wr = _case(B, S, d, seed=seed)
        c = torch.full((B, Lmax, 512), SENTINEL, dtype=torch.bfloat16, device="cuda")
        k = torch.full((B, Lmax, 64), SENTINEL, dtype=torch.bfloat16, device="cuda")
        mb.cache_append(h.cuda(), wd.cuda(), wr.cuda(), torch.tensor(seqlens, dtype=torch.int32).cuda(), c, k, ws)
        assert mb.read_status(ws) == mb.MLA_OK
        _check(c, k, h, wd, wr, seqlens)
