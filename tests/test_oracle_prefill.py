"""Pins of the oracle's prefill steps: the per-head expansion of keys and
values, and causal attention over the expanded keys.

"DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention / KeyValue":
k^C_{t,i} = W_i^UK c_t and v^C_{t,i} = W_i^UV c_t with W_i a row block of
d_h x d_c; "注意力计算": query t sees keys 1..t (here 0..t), scores scaled by
1/sqrt(d_h + d_h^R), one softmax, o = sum a v^C.  The checks below are fixed by
those statements, not by the oracle's formulas: one-hot weight rows pick
latent coordinates, the first query of a prompt returns the first value
exactly, the prefill chain equals the unabsorbed decode oracle (pinned on its
own against SDPA and closed forms) for every query position, future keys and
padding never matter, and uniform scores average the visible values.  A
transposed W, an off-by-one causal window, a dropped RoPE term or keys read
from the wrong head each fail one of them.
"""
import math

import numpy as np

import oracle


def bits(t):
    from mla_latent_kv_68_b300.inputs import bf16_bits
    return bf16_bits(t)


def f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_one_hot_weight_rows_pick_latent_coordinates():
    rng = np.random.default_rng(1)
    c = rng.standard_normal((2, 5, 16))
    W = np.zeros((3, 4, 16))
    W[2, 1, 7] = 1.0            # head 2, output 1 <- latent 7
    W[0, 3, 0] = -0.5
    e = oracle.expand_kv(c, W)
    assert e.shape == (2, 5, 3, 4)
    np.testing.assert_array_equal(e[..., 2, 1], c[..., 7])
    np.testing.assert_array_equal(e[..., 0, 3], -0.5 * c[..., 0])
    assert np.count_nonzero(e[..., 1, :]) == 0


def test_expansion_is_linear_in_the_cache():
    rng = np.random.default_rng(2)
    c1, c2 = rng.standard_normal((2, 4, 8))
    W = rng.standard_normal((2, 3, 8))
    np.testing.assert_allclose(oracle.expand_kv(3.0 * c1 - c2, W),
                               3.0 * oracle.expand_kv(c1, W) - oracle.expand_kv(c2, W), rtol=1e-12, atol=1e-12)


def _rotated(x):
    """Rotated q^R and k^R of a make_inputs problem, and the expanded keys/values."""
    L = x["seqlens"].numpy()
    B, S, H = x["B"], x["S"], x["H"]
    qr = np.zeros((B, S, H, 64))
    kr = np.zeros((B, x["Lmax"], 64))
    qb, kb = bits(x["q_rope"]), bits(x["k_r"])
    for b in range(B):
        pos = np.repeat(L[b] - S + np.arange(S), H)
        qr[b] = oracle.rope(qb[b].reshape(-1, 64), pos).reshape(S, H, 64)
        kr[b, :L[b]] = oracle.rope(kb[b, :L[b]], np.arange(L[b]))
    kc = oracle.expand_kv(bits(x["c_kv"]), bits(x["W_UK"]))
    vc = oracle.expand_kv(bits(x["c_kv"]), bits(x["W_UV"]))
    return qr, kr, kc, vc


def test_prefill_chain_equals_the_unabsorbed_decode_oracle():
    from mla_latent_kv_68_b300.inputs import make_inputs
    x = make_inputs(2, 9, 3, [9, 14], Lmax=16, seed=7, pad=float("nan"))
    qr, kr, kc, vc = _rotated(x)
    L = x["seqlens"].numpy()
    out = oracle.prefill_attention(bits(x["q_nope"]), qr, kc, kr, vc, L, softmax_scale=1.0 / math.sqrt(192.0))
    ref = oracle.decode(bits(x["q_nope"]), bits(x["q_rope"]), bits(x["c_kv"]), bits(x["k_r"]),
                        bits(x["W_UK"]), bits(x["W_UV"]), L)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_first_query_of_a_prompt_returns_the_first_value():
    rng = np.random.default_rng(3)
    B, S, H, L = 1, 6, 2, 6
    q_nope, q_rot = rng.standard_normal((B, S, H, 8)), rng.standard_normal((B, S, H, 4))
    kc, kr, vc = rng.standard_normal((B, L, H, 8)), rng.standard_normal((B, L, 4)), rng.standard_normal((B, L, H, 5))
    out = oracle.prefill_attention(q_nope, q_rot, kc, kr, vc, [L], softmax_scale=0.3)
    np.testing.assert_array_equal(out[0, 0], vc[0, 0])      # position 0 sees key 0 only


def test_future_keys_and_padding_do_not_matter():
    rng = np.random.default_rng(4)
    B, S, H, L, Lmax = 1, 4, 2, 7, 9
    q_nope, q_rot = rng.standard_normal((B, S, H, 8)), rng.standard_normal((B, S, H, 4))
    kc, kr, vc = rng.standard_normal((B, Lmax, H, 8)), rng.standard_normal((B, Lmax, 4)), rng.standard_normal((B, Lmax, H, 5))
    out = oracle.prefill_attention(q_nope, q_rot, kc, kr, vc, [L], softmax_scale=0.5)
    # query s sits at L - S + s: keys after it, and rows past L, change nothing
    kc2, kr2, vc2 = kc.copy(), kr.copy(), vc.copy()
    kc2[0, L - 1] += 100.0
    vc2[0, L - 1] -= 50.0
    kr2[0, L:] = np.nan
    kc2[0, L:] = np.nan
    vc2[0, L:] = np.nan
    out2 = oracle.prefill_attention(q_nope, q_rot, kc2, kr2, vc2, [L], softmax_scale=0.5)
    np.testing.assert_array_equal(out2[0, :S - 1], out[0, :S - 1])
    assert not np.allclose(out2[0, S - 1], out[0, S - 1])   # the last query does see key L - 1


def test_uniform_scores_average_the_visible_values():
    rng = np.random.default_rng(5)
    B, S, H, L = 1, 3, 1, 5
    q_nope = np.zeros((B, S, H, 8))
    q_rot = np.zeros((B, S, H, 4))
    kc, kr, vc = rng.standard_normal((B, L, H, 8)), rng.standard_normal((B, L, 4)), rng.standard_normal((B, L, H, 5))
    out = oracle.prefill_attention(q_nope, q_rot, kc, kr, vc, [L], softmax_scale=1.0)
    for s in range(S):
        t = L - S + s
        np.testing.assert_allclose(out[0, s, 0], vc[0, :t + 1, 0].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_heads_use_their_own_keys():
    # two heads with identical queries but different keys give different
    # weights; the rope key is shared
    rng = np.random.default_rng(6)
    B, S, H, L = 1, 2, 2, 4
    q_nope = np.repeat(rng.standard_normal((B, S, 1, 8)), 2, axis=2)
    q_rot = np.repeat(rng.standard_normal((B, S, 1, 4)), 2, axis=2)
    kc = rng.standard_normal((B, L, H, 8)) * 3.0
    kr = rng.standard_normal((B, L, 4))
    vc = np.repeat(rng.standard_normal((B, L, 1, 5)), 2, axis=2)
    out = oracle.prefill_attention(q_nope, q_rot, kc, kr, vc, [L], softmax_scale=1.0)
    assert not np.allclose(out[0, 1, 0], out[0, 1, 1])
    kc[0, :, 1] = kc[0, :, 0]
    out = oracle.prefill_attention(q_nope, q_rot, kc, kr, vc, [L], softmax_scale=1.0)
    np.testing.assert_array_equal(out[0, :, 0], out[0, :, 1])
