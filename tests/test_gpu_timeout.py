"""A bounded wait inside the decode kernel that runs out is reported as
MLA_ERR_TIMEOUT, and the device stays usable.

The test hook mla_debug_decode_stall leaves the next decode's split-plan
barrier incomplete (nothing the kernels wait on is faulted or broken: one
barrier simply never completes), with a 20 ms wait limit.  Every warp gives
up before issuing any copy or MMA, the status word records the timeout, and
the very next call is clean and matches the oracle.
"""
import math

import numpy as np
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


def test_wait_that_runs_out_is_reported_and_the_next_call_is_clean():
    g = torch.Generator().manual_seed(77)
    B, S, H, seqlens = 3, 1, 128, [300, 70, 1500]
    Lmax = max(seqlens)
    c = torch.zeros(B, Lmax, 512)
    k = torch.zeros(B, Lmax, 64)
    for b, L in enumerate(seqlens):
        c[b, :L] = torch.randn(L, 512, generator=g)
        k[b, :L] = torch.randn(L, 64, generator=g)
    q = torch.cat([0.5 * torch.randn(B, S, H, 512, generator=g), torch.randn(B, S, H, 64, generator=g)], -1)
    q, c, k = q.to(torch.bfloat16), c.to(torch.bfloat16), k.to(torch.bfloat16)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    qd, cd, kd, sld = q.cuda(), c.cuda(), k.cuda(), sl.cuda()
    ws = mb.new_workspace(B, S, H)
    o = torch.full((B, S, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")

    mb.debug_decode_stall(20_000_000)       # 20 ms instead of 1 s
    mb.decode(qd, cd, kd, sld, ws)
    assert mb.read_status(ws) == mb.MLA_ERR_TIMEOUT
    assert mb.read_status(ws) == mb.MLA_OK  # reading clears the status

    mb.decode(qd, cd, kd, sld, ws)          # the hook was one-shot
    mb.splitkv_combine(ws, o)
    assert mb.read_status(ws) == mb.MLA_OK
    ref = oracle.latent_attention(bits(q), bits(c), bits(k), sl.numpy(), d_r=64,
                                  softmax_scale=1.0 / math.sqrt(192.0))
    assert_close(f64(o), ref, what="after a timeout")
