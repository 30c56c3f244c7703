"""The allocation-free decode entry point (mla_decode_noalloc) against the
regular one (mla_decode + mla_splitkv_combine with a caller workspace).

mla_decode_noalloc serves callers that cannot allocate device memory on their
decode path (a serving process that has reserved all of HBM for its own pool,
or a real-time loop that must not call cudaMalloc because it can synchronise
the device): its split-KV scratch is a fixed array inside the library.  Two
calls in a row, with different shapes and lengths, must each match the
regular path; the second call also shows that what the first left in the
shared scratch does not leak into its result.  This file is collected last so
that a failure here cannot hide another test's result.
"""
import ctypes
import math

import pytest
import torch

import oracle
from gpu_util import assert_close, bits, f64
from mla_latent_kv_68_b300 import binding as mb

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_68_b300 import build
    build.build()
    mb.lib()


def _case(B, S, H, seqlens, seed, Lmax=None):
    g = torch.Generator().manual_seed(seed)
    Lmax = Lmax or max(seqlens)
    c = torch.zeros(B, Lmax, 512)
    k = torch.zeros(B, Lmax, 64)
    for b, L in enumerate(seqlens):
        c[b, :L] = torch.randn(L, 512, generator=g)
        k[b, :L] = torch.randn(L, 64, generator=g)
    q = torch.cat([0.5 * torch.randn(B, S, H, 512, generator=g),
                   torch.randn(B, S, H, 64, generator=g)], dim=-1)
    dev = "cuda"
    return (q.to(torch.bfloat16).to(dev), c.to(torch.bfloat16).to(dev),
            k.to(torch.bfloat16).to(dev), torch.tensor(seqlens, dtype=torch.int32, device=dev))


def _regular(q, c, k, sl):
    B, S, H, _ = q.shape
    ws = mb.new_workspace(B, S, H)
    o = torch.empty(B, S, H, 512, dtype=torch.bfloat16, device="cuda")
    mb.decode(q, c, k, sl, ws)
    mb.splitkv_combine(ws, o)
    assert mb.read_status(ws) == mb.MLA_OK
    return o


def _noalloc(q, c, k, sl):
    B, S, H, _ = q.shape
    o = torch.full((B, S, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.decode_noalloc(q, c, k, sl, o)
    assert mb.read_status() == mb.MLA_OK
    return o


def test_noalloc_matches_regular_decode_on_two_calls_in_a_row():
    cases = [
        (5, 1, 128, [4999, 1, 3000, 129, 8191], 101),   # ragged lengths, one row block
        (3, 2, 96, [2, 700, 2500], 202),                # S = 2, 192 rows: two row blocks
    ]
    for B, S, H, seqlens, seed in cases:
        q, c, k, sl = _case(B, S, H, seqlens, seed)
        want = f64(_regular(q, c, k, sl))
        got = f64(_noalloc(q, c, k, sl))
        assert_close(got, want, what=f"noalloc vs regular B{B} S{S} H{H}")
        # and against the fp64 oracle of the absorbed latent attention
        ref = oracle.latent_attention(bits(q.cpu()), bits(c.cpu()), bits(k.cpu()), sl.cpu().numpy(),
                                      d_r=64, softmax_scale=1.0 / math.sqrt(192.0))
        assert_close(got, ref, what=f"noalloc vs oracle B{B} S{S} H{H}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    B = 1
    while mb.decode_workspace_size(B, 1, 128) <= mb.STATIC_SCRATCH_BYTES:
        B *= 2
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check comes first
    rc = mb.lib().mla_decode_noalloc(fake, fake, fake, fake, B, 1, 128, 16, 0.07, fake, None)
    assert rc == 3                     # MLA_ERR_WORKSPACE, nothing launched
