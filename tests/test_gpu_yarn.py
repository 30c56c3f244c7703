"""GPU parity of the YaRN path (frequencies of "YaRN 扩展", setting of "Long
Context Extension": s = 40, alpha = 1, beta = 32, score scale 0.1 ln s + 1)
against the fp64 oracle with the same frequencies."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, bits, f64, to_dev
from mla_latent_kv_68_b300 import binding as mb
from mla_latent_kv_68_b300.inputs import make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_68_b300 import build
    build.build()
    mb.lib()


def _yarn():
    return oracle.yarn_theta(64)   # the expected frequencies come from the oracle


def test_rope_with_yarn_frequencies_matches_oracle():
    th = _yarn()
    g = torch.Generator().manual_seed(21)
    N, nh = 41, 2
    x = torch.randn(N, nh, 64, generator=g).to(torch.bfloat16)
    pos = torch.randint(0, 131072, (N,), generator=g, dtype=torch.int32)
    pos[0], pos[1] = 0, 131071
    out = torch.full((N, nh, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.rope_apply(x.cuda(), nh * 64, 64, out, nh * 64, 64, N, nh, mb.POS_EXPLICIT, pos.cuda(),
                  theta=list(th))
    ref = oracle.rope_theta(bits(x).reshape(N * nh, 64), np.repeat(pos.numpy().astype(np.int64), nh), th)
    got = f64(out).reshape(N * nh, 64)
    assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5).all(), float(np.abs(got - ref).max())


def test_absorb_rope_with_yarn_frequencies_matches_oracle():
    th = _yarn()
    B, S, H = 3, 2, 16
    g = torch.Generator().manual_seed(22)
    q = torch.randn(B, S, H, 128, generator=g).to(torch.bfloat16)
    qr = torch.randn(B, S, H, 64, generator=g).to(torch.bfloat16)
    W = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    seqlens = torch.tensor([2, 70000, 131072], dtype=torch.int32)
    q_cat = torch.empty(B, S, H, 576, dtype=torch.bfloat16, device="cuda")
    mb.absorb_rope_q(q.cuda(), qr.cuda(), W.cuda(), seqlens.cuda(), q_cat, theta=list(th))
    got = f64(q_cat)
    pos = np.array([[L - S + s for s in range(S)] for L in seqlens.tolist()]).reshape(-1)
    rref = oracle.rope_theta(bits(qr).reshape(-1, 64), np.repeat(pos, H), th).reshape(B, S, H, 64)
    assert (np.abs(got[..., 512:] - rref) <= 2.0 ** -8 * np.abs(rref) + 1e-5).all()


def _yarn_step(x, th, scale):
    d = to_dev(x)
    mb.rope_cache(d["k_r"], d["seqlens"], theta=list(th))
    step = mb.DecodeStep(x["B"], x["S"], x["H"], rope_theta=list(th))
    out = step(d["q_nope"], d["q_rope"], d["c_kv"], d["k_r"], d["seqlens"], d["W_UK"], d["W_UV"],
               softmax_scale=scale)
    assert mb.read_status(step.workspace) == mb.MLA_OK
    return f64(out)


def _oracle_rows(x, th, scale, rows=None):
    b = {k: bits(x[k]) for k in ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV")}
    return oracle.decode(b["q_nope"], b["q_rope"], b["c_kv"], b["k_r"], b["W_UK"], b["W_UV"],
                         x["seqlens"].numpy(), softmax_scale=scale, rope_theta=th, rows=rows)


def test_whole_step_with_yarn_matches_unabsorbed_oracle():
    # the GPU step takes the library's frequencies and scale, the oracle its own
    x = make_inputs(3, 2, 8, [2, 300, 5000], seed=23)
    got = _yarn_step(x, mb.yarn_frequencies(), mb.yarn_softmax_scale(40.0))
    assert_close(got, _oracle_rows(x, oracle.yarn_theta(64), oracle.yarn_softmax_scale(40.0)),
                 what="yarn step")


def test_long_workload_with_yarn_sampled_rows():
    x = workload_inputs("long_b4_s1_h128_l131072")
    got = _yarn_step(x, mb.yarn_frequencies(), mb.yarn_softmax_scale(40.0)).reshape(-1, 128)
    rows = np.array([0, 127, 128 + 5, 2 * 128 + 64, 3 * 128 + 127], np.int64)
    ref = _oracle_rows(x, oracle.yarn_theta(64), oracle.yarn_softmax_scale(40.0), rows=rows)
    assert_close(got[rows], ref, what="yarn 128K")
    torch.cuda.empty_cache()
