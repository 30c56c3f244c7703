"""Pins of the oracle's YaRN frequencies and of its decode with explicit RoPE
frequencies.

"DeepSeek-V3" (ekkoxiao.github.io), section "YaRN 扩展": theta'_j =
(1 - g_j) theta_j / s + g_j theta_j, with g_j = 1 in the high-frequency band
(kept) and 0 in the low-frequency band (divided by s), a smooth transition in
between; "DeepSeek-V3 Technical Report" (process-cxr.github.io), "Long Context
Extension": s = 40, alpha = 1, beta = 32, applied to the decoupled RoPE key,
original context 4K.  The band edges are read as turn counts over the original
context, r_j = L_orig theta_j / (2 pi) (alpha = 1 turn, beta = 32 turns), with
g linear in r between them.  Each test checks a property the pages or the
reading fix, so that swapping alpha and beta, dividing the wrong band by s,
or a ramp in the wrong variable fails one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle

D_R = 64
BASE = 10000.0
L_ORIG = 4096.0


def _theta():
    return BASE ** (-2.0 * np.arange(D_R // 2) / D_R)


def _turns(theta):
    return L_ORIG * theta / (2.0 * math.pi)


def test_yarn_with_s_one_is_plain_rope():
    rng = np.random.default_rng(10)
    x = rng.standard_normal((5, D_R))
    pos = np.array([0, 1, 4095, 65536, 131071])
    np.testing.assert_allclose(oracle.yarn_theta(D_R, s=1.0), _theta(), rtol=1e-15)
    np.testing.assert_allclose(oracle.rope_theta(x, pos, oracle.yarn_theta(D_R, s=1.0)),
                               oracle.rope(x, pos), rtol=0, atol=1e-10)


def test_yarn_keeps_high_and_divides_low_frequencies():
    th, yt = _theta(), oracle.yarn_theta(D_R, s=40.0, alpha=1.0, beta=32.0, orig_len=L_ORIG)
    r = _turns(th)
    high, low = r >= 32.0, r <= 1.0
    assert high.sum() >= 5 and low.sum() >= 5            # both bands exist at these settings
    np.testing.assert_allclose(yt[high], th[high], rtol=1e-15)
    np.testing.assert_allclose(yt[low], th[low] / 40.0, rtol=1e-15)
    assert yt[0] == th[0] == 1.0                         # pair 0 turns every position: kept


def test_yarn_frequencies_lie_between_the_bands_and_fall_with_j():
    th, yt = _theta(), oracle.yarn_theta(D_R)
    assert np.all(yt <= th * (1 + 1e-15)) and np.all(yt >= th / 40.0 * (1 - 1e-15))
    assert np.all(np.diff(yt) < 0)


def test_yarn_ramp_is_affine_in_turns_between_alpha_and_beta():
    th, yt = _theta(), oracle.yarn_theta(D_R, s=40.0, alpha=1.0, beta=32.0)
    r = _turns(th)
    mid = (r > 1.0) & (r < 32.0)
    assert mid.sum() >= 5
    g = (yt[mid] - th[mid] / 40.0) / (th[mid] - th[mid] / 40.0)  # recovered blend weight
    slope, icpt = np.polyfit(r[mid], g, 1)
    np.testing.assert_allclose(g, slope * r[mid] + icpt, atol=1e-12)
    assert slope == pytest.approx(1.0 / 31.0, rel=1e-9)
    assert -icpt / slope == pytest.approx(1.0, rel=1e-9)         # g = 0 at alpha = 1 turn
    assert (1.0 - icpt) / slope == pytest.approx(32.0, rel=1e-9)  # g = 1 at beta = 32 turns


def test_yarn_rope_keeps_norms_and_relative_positions():
    yt = oracle.yarn_theta(D_R)
    rng = np.random.default_rng(11)
    q, k = rng.standard_normal((1, D_R)), rng.standard_normal((1, D_R))
    for m in (0, 5, 131071):
        np.testing.assert_allclose(np.linalg.norm(oracle.rope_theta(q, [m], yt)),
                                   np.linalg.norm(q), rtol=1e-13)
    ref = float(np.sum(oracle.rope_theta(q, [900], yt) * oracle.rope_theta(k, [300], yt)))
    for delta in (1, 4096, 100000):
        got = float(np.sum(oracle.rope_theta(q, [900 + delta], yt) *
                           oracle.rope_theta(k, [300 + delta], yt)))
        assert got == pytest.approx(ref, abs=1e-9)


def test_rope_theta_with_plain_frequencies_equals_rope():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((7, D_R))
    pos = np.array([0, 1, 2, 1000, 4095, 70000, 131071])
    np.testing.assert_allclose(oracle.rope_theta(x, pos, _theta()), oracle.rope(x, pos),
                               rtol=0, atol=1e-10)  # the two pow() differ in the last bit


def _complex_rope_theta(x, pos, theta):
    """RoPE as multiplication of x_{2j} + i x_{2j+1} by exp(i pos theta_j)."""
    z = x[..., 0::2] + 1j * x[..., 1::2]
    z = z * np.exp(1j * np.asarray(pos, np.float64)[..., None] * theta)
    out = np.empty_like(x)
    out[..., 0::2], out[..., 1::2] = z.real, z.imag
    return out


def test_decode_with_yarn_matches_sdpa_on_expanded_kv():
    """The decode with explicit YaRN frequencies and the YaRN score scale
    (0.1 ln s + 1) / sqrt(d_h + d_h^R) against torch's scaled_dot_product_attention
    in float64 on explicitly expanded, YaRN-rotated keys."""
    rng = np.random.default_rng(13)
    B, S, H, d_c, d_h, d_r, d_v = 2, 2, 3, 12, 5, 8, 7
    seqlens = [3, 9]
    Lmax = 9
    yt = oracle.yarn_theta(d_r, orig_len=8.0)
    q_nope = rng.standard_normal((B, S, H, d_h))
    q_rope = rng.standard_normal((B, S, H, d_r))
    c_kv = rng.standard_normal((B, Lmax, d_c))
    k_r = rng.standard_normal((B, Lmax, d_r))
    W_UK = rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c)
    W_UV = rng.standard_normal((H, d_v, d_c)) / math.sqrt(d_c)
    scale = oracle.yarn_softmax_scale(40.0, d_h, d_r)
    got = oracle.decode(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, np.array(seqlens, np.int32),
                        softmax_scale=scale, rope_theta=yt)
    for b in range(B):
        L = seqlens[b]
        c = c_kv[b, :L]
        kc = np.einsum("hdk,jk->hjd", W_UK, c)
        kr = _complex_rope_theta(k_r[b, :L], np.arange(L) * 1.0, yt)
        K = np.concatenate([kc, np.broadcast_to(kr, (H, L, d_r))], axis=-1)
        V = np.einsum("hdk,jk->hjd", W_UV, c)
        pos_q = L - S + np.arange(S)
        qr = _complex_rope_theta(q_rope[b], pos_q[:, None] * 1.0, yt)
        Q = np.concatenate([q_nope[b], qr], axis=-1).transpose(1, 0, 2)
        mask = np.arange(L)[None, :] <= pos_q[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(np.ascontiguousarray(Q)), torch.from_numpy(np.ascontiguousarray(K)),
            torch.from_numpy(np.ascontiguousarray(V)), attn_mask=torch.from_numpy(mask),
            scale=scale).numpy()
        np.testing.assert_allclose(got[b], ref.transpose(1, 0, 2), rtol=1e-11, atol=1e-12)


def test_yarn_score_factor_closed_forms():
    # "Long Context Extension": the scores are scaled by 0.1 ln s + 1 on top of
    # 1/sqrt(d_h + d_r).  s = 1 is plain attention; s = e^10 doubles the scale;
    # the factor grows with s; d_h + d_r = 192 for the pages' model.
    assert oracle.yarn_softmax_scale(1.0, 128, 64) == 1.0 / math.sqrt(192.0)
    assert oracle.yarn_softmax_scale(math.exp(10.0), 128, 64) == pytest.approx(2.0 / math.sqrt(192.0),
                                                                              rel=1e-15)
    assert oracle.yarn_softmax_scale(40.0, 128, 64) == pytest.approx(1.3688879454113936 / math.sqrt(192.0),
                                                                     rel=1e-15)
    assert oracle.yarn_softmax_scale(40.0, 3, 1) == pytest.approx(1.3688879454113936 / 2.0, rel=1e-15)
    with pytest.raises(ValueError):
        oracle.yarn_softmax_scale(0.5)
