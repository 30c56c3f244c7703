"""Pins of the oracle's cache-append step (oracle.cache_append).

"DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention / KeyValue":
c_t^KV = W^DKV h_t with W^DKV in R^{d_c x d}, and k_t^R = RoPE_t(W^KR h_t)
with W^KR in R^{d_h^R x d}.  Each test checks the oracle against something
other than itself: unit inputs that pick a weight column, an explicit
triple loop, the rotation written as complex multiplication, and invariants
(no rotation at position 0, norms kept, linearity), with d_c != d_r != d so
that a transposed weight or a swapped index fails.
"""
import numpy as np
import pytest

import oracle

D, D_C, D_R = 96, 24, 8


def _w(seed):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((D_C, D)), rng.standard_normal((D_R, D)), rng


def _complex_rope(x, pos, base=10000.0):
    z = x[..., 0::2] + 1j * x[..., 1::2]
    theta = base ** (-2.0 * np.arange(x.shape[-1] // 2) / x.shape[-1])
    z = z * np.exp(1j * np.asarray(pos, np.float64)[:, None] * theta)
    out = np.empty_like(x)
    out[..., 0::2], out[..., 1::2] = z.real, z.imag
    return out


def test_unit_input_picks_weight_columns():
    wd, wr, _ = _w(1)
    for i in (0, 7, D - 1):
        h = np.zeros((1, D))
        h[0, i] = 1.0
        c, k = oracle.cache_append(h, wd, wr, [0])
        np.testing.assert_array_equal(c[0], wd[:, i])
        np.testing.assert_array_equal(k[0], wr[:, i])   # position 0: no rotation


def test_down_projection_matches_explicit_loops():
    wd, wr, rng = _w(2)
    h = rng.standard_normal((3, D))
    c, k = oracle.cache_append(h, wd, wr, [0, 0, 0])
    for n in range(3):
        for r in range(D_C):
            assert c[n, r] == pytest.approx(sum(wd[r, j] * h[n, j] for j in range(D)), rel=1e-12, abs=1e-12)
        for r in range(D_R):
            assert k[n, r] == pytest.approx(sum(wr[r, j] * h[n, j] for j in range(D)), rel=1e-12, abs=1e-12)


def test_key_rotation_is_complex_multiplication_at_each_position():
    wd, wr, rng = _w(3)
    h = rng.standard_normal((5, D))
    pos = np.array([0, 1, 4095, 65536, 131071])
    _, k = oracle.cache_append(h, wd, wr, pos)
    np.testing.assert_allclose(k, _complex_rope(h @ wr.T, pos), rtol=0, atol=1e-9)
    np.testing.assert_allclose(np.linalg.norm(k, axis=1), np.linalg.norm(h @ wr.T, axis=1), rtol=1e-12)


def test_append_is_linear_in_the_hidden_state():
    wd, wr, rng = _w(4)
    h1, h2 = rng.standard_normal((2, D)), rng.standard_normal((2, D))
    pos = [3, 900]
    c1, k1 = oracle.cache_append(h1, wd, wr, pos)
    c2, k2 = oracle.cache_append(h2, wd, wr, pos)
    c, k = oracle.cache_append(2.0 * h1 - 0.5 * h2, wd, wr, pos)
    np.testing.assert_allclose(c, 2.0 * c1 - 0.5 * c2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(k, 2.0 * k1 - 0.5 * k2, rtol=1e-12, atol=1e-11)


def test_yarn_frequencies_change_only_the_key():
    wd, wr, rng = _w(5)
    h = rng.standard_normal((2, D))
    pos = [10, 5000]
    c0, k0 = oracle.cache_append(h, wd, wr, pos)
    th = oracle.yarn_theta(D_R, orig_len=64.0)
    c1, k1 = oracle.cache_append(h, wd, wr, pos, theta=th)
    np.testing.assert_array_equal(c0, c1)
    np.testing.assert_allclose(k1, oracle.rope_theta(h @ wr.T, pos, th), rtol=0, atol=1e-12)
    assert not np.allclose(k0, k1)


def test_bf16_bit_inputs_read_as_their_values():
    wd, wr, rng = _w(6)
    h = rng.standard_normal((2, D))
    to_bits = lambda a: (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    from_bits = lambda b: (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    hb, wdb, wrb = to_bits(h), to_bits(wd), to_bits(wr)   # truncated to bf16 patterns
    c_b, k_b = oracle.cache_append(hb, wdb, wrb, [7, 8])
    c_f, k_f = oracle.cache_append(from_bits(hb), from_bits(wdb), from_bits(wrb), [7, 8])
    np.testing.assert_array_equal(c_b, c_f)
    np.testing.assert_array_equal(k_b, k_f)
    assert abs(c_b[0, 0] - (from_bits(wdb)[0] @ from_bits(hb)[0])) < 1e-12
