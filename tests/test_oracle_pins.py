"""Pins of the fp64 CPU oracle to facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a closed
form, an invariant, a special case that reduces to a plain matrix product, or
torch's scaled_dot_product_attention run in float64 on explicitly expanded
keys and values.  Shapes are deliberately non-square (d_c != d_h != d_v,
H > 1, S = 2) so that a transposed operand, a swapped index or an
off-by-one in the causal window fails at least one test.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _complex_rope(x, pos, base=10000.0):
    """RoPE written as multiplication of complex numbers x_{2j} + i x_{2j+1} by
    exp(i * pos * theta_j): an independent formulation of the same rotation."""
    x = np.asarray(x, np.float64)
    d_r = x.shape[-1]
    z = x[..., 0::2] + 1j * x[..., 1::2]
    theta = base ** (-2.0 * np.arange(d_r // 2) / d_r)
    pos = np.asarray(pos, np.float64)
    z = z * np.exp(1j * pos[..., None] * theta)
    out = np.empty_like(x)
    out[..., 0::2] = z.real
    out[..., 1::2] = z.imag
    return out


def _rand_problem(rng, B, S, H, seqlens, d_c, d_h, d_r, d_v, Lmax=None):
    Lmax = Lmax or max(seqlens)
    return dict(
        q_nope=rng.standard_normal((B, S, H, d_h)),
        q_rope=rng.standard_normal((B, S, H, d_r)),
        c_kv=rng.standard_normal((B, Lmax, d_c)),
        k_r=rng.standard_normal((B, Lmax, d_r)),
        W_UK=rng.standard_normal((H, d_h, d_c)) / math.sqrt(d_c),
        W_UV=rng.standard_normal((H, d_v, d_c)) / math.sqrt(d_c),
        seqlens=np.asarray(seqlens, np.int32),
    )


# ---------------------------------------------------------------- RoPE pins
def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((5, 64))
    np.testing.assert_array_equal(oracle.rope(x, np.zeros(5, np.int64)), x)


def test_rope_closed_form_angles():
    # pair 0 has theta_0 = 1: e_0 at position 1 turns by exactly 1 rad.
    # pair 16 of 32 has theta = 10000^(-1/2) = 1/100: at position 100 it also turns by 1 rad.
    # pair 31 has theta = 10000^(-62/64); at position 0 nothing turns.
    x = np.zeros((3, 64))
    x[0, 0] = 1.0
    x[1, 32] = 1.0
    x[2, 63] = 2.0
    y = oracle.rope(x, np.array([1, 100, 0], np.int64))
    assert y[0, 0] == pytest.approx(math.cos(1.0), abs=1e-15)
    assert y[0, 1] == pytest.approx(math.sin(1.0), abs=1e-15)  # counter-clockwise
    assert y[1, 32] == pytest.approx(math.cos(1.0), abs=1e-13)
    assert y[1, 33] == pytest.approx(math.sin(1.0), abs=1e-13)
    assert np.count_nonzero(y[0, 2:]) == 0 and np.count_nonzero(y[1, :32]) == 0
    assert y[2, 63] == 2.0 and y[2, 62] == 0.0
    # the second element of a pair rotates towards minus the first one
    z = np.zeros((1, 64))
    z[0, 1] = 1.0
    w = oracle.rope(z, np.array([1], np.int64))
    assert w[0, 0] == pytest.approx(-math.sin(1.0), abs=1e-15)
    assert w[0, 1] == pytest.approx(math.cos(1.0), abs=1e-15)


def test_rope_matches_complex_formulation():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((40, 64))
    pos = rng.integers(0, 131072, 40)
    np.testing.assert_allclose(oracle.rope(x, pos), _complex_rope(x, pos), rtol=0, atol=1e-9)


def test_rope_preserves_norm_and_composes():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((10, 64))
    a = rng.integers(0, 5000, 10)
    b = rng.integers(0, 5000, 10)
    ya = oracle.rope(x, a)
    np.testing.assert_allclose(np.linalg.norm(ya, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    np.testing.assert_allclose(oracle.rope(ya, b), oracle.rope(x, a + b), atol=1e-10)


def test_rope_relative_position_invariance():
    # "RoPE 数据流": the dot product of a rotated query and key depends on m - n only.
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 64))
    k = rng.standard_normal((1, 64))
    m, n = 777, 123
    base = float(np.sum(oracle.rope(q, [m]) * oracle.rope(k, [n])))
    for delta in (1, 50, 4096, 100000):
        shifted = float(np.sum(oracle.rope(q, [m + delta]) * oracle.rope(k, [n + delta])))
        assert shifted == pytest.approx(base, abs=1e-9)


# ---------------------------------------------------------------- decode pins
@pytest.mark.parametrize("S,seqlens", [(2, [2, 6, 9]), (5, [5, 6, 10])])
def test_decode_matches_sdpa_on_expanded_kv(S, seqlens):
    """Library cross-check: keys k = [W^UK c ; RoPE(k_R)] and values v = W^UV c
    expanded explicitly, then torch's scaled_dot_product_attention (float64)
    with a causal mask whose query s sits at position L_b - S + s (S = 5: a
    prefill chunk, including a sequence exactly as long as its chunk)."""
    rng = np.random.default_rng(5 + S)
    B, H, d_c, d_h, d_r, d_v = 3, 3, 12, 5, 4, 7
    p = _rand_problem(rng, B, S, H, seqlens, d_c, d_h, d_r, d_v, Lmax=10)
    scale = 1.0 / math.sqrt(d_h + d_r)
    got = oracle.decode(p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"], p["W_UV"],
                        p["seqlens"], softmax_scale=scale)
    for b in range(B):
        L = seqlens[b]
        c = p["c_kv"][b, :L]                                   # [L, d_c]
        kc = np.einsum("hdk,jk->hjd", p["W_UK"], c)           # [H, L, d_h]
        kr = _complex_rope(p["k_r"][b, :L], np.arange(L))      # [L, d_r]
        K = np.concatenate([kc, np.broadcast_to(kr, (H, L, d_r))], axis=-1)
        V = np.einsum("hdk,jk->hjd", p["W_UV"], c)            # [H, L, d_v]
        pos_q = L - S + np.arange(S)
        qr = _complex_rope(p["q_rope"][b], pos_q[:, None])     # [S, H, d_r]
        Q = np.concatenate([p["q_nope"][b], qr], axis=-1).transpose(1, 0, 2)  # [H, S, d]
        mask = np.arange(L)[None, :] <= pos_q[:, None]         # [S, L]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(np.ascontiguousarray(Q)), torch.from_numpy(np.ascontiguousarray(K)),
            torch.from_numpy(np.ascontiguousarray(V)), attn_mask=torch.from_numpy(mask),
            scale=scale).numpy()                               # [H, S, d_v]
        np.testing.assert_allclose(got[b], ref.transpose(1, 0, 2), rtol=1e-11, atol=1e-12)


def test_decode_default_scale_is_inverse_sqrt_192():
    rng = np.random.default_rng(6)
    p = _rand_problem(rng, 1, 1, 2, [5], 512, 128, 64, 128)
    a = oracle.decode(p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"], p["W_UV"],
                      p["seqlens"])
    b = oracle.decode(p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"], p["W_UV"],
                      p["seqlens"], softmax_scale=1.0 / math.sqrt(192.0))
    np.testing.assert_array_equal(a, b)


def test_softmax_weights_sum_to_one():
    rng = np.random.default_rng(7)
    p = _rand_problem(rng, 2, 2, 3, [3, 40], 16, 8, 4, 8)
    _, wsum = oracle.decode(p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"],
                            p["W_UV"], p["seqlens"], return_wsum=True)
    np.testing.assert_allclose(wsum, 1.0, rtol=0, atol=1e-14)


def test_one_token_context_returns_value_of_that_token():
    # L = 1, S = 1: the only weight is 1, so o = W^UV c_0 for every head.
    rng = np.random.default_rng(8)
    p = _rand_problem(rng, 2, 1, 4, [1, 1], 512, 128, 64, 128)
    got = oracle.decode(p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"], p["W_UV"],
                        p["seqlens"])
    want = np.einsum("hdk,bk->bhd", p["W_UV"], p["c_kv"][:, 0])
    np.testing.assert_allclose(got[:, 0], want, rtol=1e-12, atol=1e-13)  # 512-term sums


def test_zero_query_gives_uniform_attention():
    # q = 0 makes every score 0, so a_j = 1/(pos+1) and o = W^UV mean_j c_j.
    rng = np.random.default_rng(9)
    p = _rand_problem(rng, 2, 2, 3, [4, 11], 20, 6, 4, 9)
    p["q_nope"][:] = 0.0
    p["q_rope"][:] = 0.0
    got = oracle.decode(p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"], p["W_UV"],
                        p["seqlens"])
    for b, L in enumerate([4, 11]):
        for s in range(2):
            mean_c = p["c_kv"][b, :L - 2 + s + 1].mean(axis=0)
            np.testing.assert_allclose(got[b, s], np.einsum("hdk,k->hd", p["W_UV"], mean_c),
                                       rtol=1e-13, atol=1e-14)


def test_two_token_closed_form():
    # d_c = d_h = d_v = 1, no RoPE part, W^UK = W^UV = 1, scale 1:
    # keys c_0 = 0, c_1 = 1 and query q = ln 3 give scores 0 and ln 3,
    # so a = (1/4, 3/4) and o = 1/4 * 0 + 3/4 * 1 = 0.75.
    one = np.ones((1, 1, 1))
    got = oracle.decode(np.full((1, 1, 1, 1), math.log(3.0)), np.zeros((1, 1, 1, 0)),
                        np.array([[[0.0], [1.0]]]), np.zeros((1, 2, 0)), one, one,
                        np.array([2], np.int32), softmax_scale=1.0)
    assert got[0, 0, 0, 0] == pytest.approx(0.75, abs=1e-15)


def test_dominant_key_selects_its_value():
    # A score gap of 60 puts all but e^-60 of the weight on one key.
    rng = np.random.default_rng(10)
    d_c, d_h, d_r, d_v, L = 8, 8, 2, 3, 6
    p = _rand_problem(rng, 1, 1, 1, [L], d_c, d_h, d_r, d_v)
    p["W_UK"][0] = np.eye(d_h, d_c)
    p["c_kv"][0] = 0.0
    p["c_kv"][0, 3, 0] = 1.0
    p["q_nope"][0, 0, 0] = 0.0
    p["q_nope"][0, 0, 0, 0] = 60.0
    p["q_rope"][:] = 0.0
    got = oracle.decode(p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"], p["W_UV"],
                        p["seqlens"], softmax_scale=1.0)
    np.testing.assert_allclose(got[0, 0, 0], p["W_UV"][0] @ p["c_kv"][0, 3], atol=1e-20)


def test_causality_future_token_invisible_to_earlier_query():
    rng = np.random.default_rng(11)
    p = _rand_problem(rng, 1, 2, 2, [7], 10, 4, 4, 5)
    args = lambda q: (q["q_nope"], q["q_rope"], q["c_kv"], q["k_r"], q["W_UK"], q["W_UV"],
                      q["seqlens"])
    base = oracle.decode(*args(p))
    p2 = {k: v.copy() for k, v in p.items()}
    p2["c_kv"][0, 6] += 5.0
    p2["k_r"][0, 6] -= 3.0
    pert = oracle.decode(*args(p2))
    np.testing.assert_array_equal(pert[0, 0], base[0, 0])   # query 0 sits at position 5
    assert np.abs(pert[0, 1] - base[0, 1]).max() > 1e-3      # query 1 sees position 6
    # the padding rows beyond L_b are never read
    p3 = {k: v.copy() for k, v in p.items()}
    p3["c_kv"] = np.concatenate([p["c_kv"], np.full((1, 3, 10), np.nan)], axis=1)
    p3["k_r"] = np.concatenate([p["k_r"], np.full((1, 3, 4), np.nan)], axis=1)
    np.testing.assert_array_equal(oracle.decode(*args(p3)), base)


def test_rows_subset_matches_full():
    rng = np.random.default_rng(12)
    p = _rand_problem(rng, 2, 2, 3, [5, 9], 16, 8, 4, 8)
    args = (p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"], p["W_UV"], p["seqlens"])
    full = oracle.decode(*args).reshape(-1, 8)
    rows = np.array([11, 0, 7, 3])
    np.testing.assert_array_equal(oracle.decode(*args, rows=rows), full[rows])


def test_bf16_input_widening_is_exact():
    from mla_latent_kv_68_b300.inputs import bf16_bits, make_inputs
    x = make_inputs(1, 2, 2, [6], seed=3)
    bits = {k: bf16_bits(x[k]) for k in ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV")}
    f64 = {k: x[k].double().numpy() for k in bits}
    order = ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV")
    a = oracle.decode(*[bits[k] for k in order], x["seqlens"].numpy())
    b = oracle.decode(*[f64[k] for k in order], x["seqlens"].numpy())
    np.testing.assert_array_equal(a, b)


def test_invalid_arguments_are_rejected():
    rng = np.random.default_rng(13)
    p = _rand_problem(rng, 1, 2, 1, [3], 4, 2, 2, 2)
    p["seqlens"][:] = 1  # shorter than S = 2
    with pytest.raises(ValueError):
        oracle.decode(p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"], p["W_UV"],
                      p["seqlens"])


# ------------------------------------------------------ step oracles chain up
def test_absorbed_steps_reproduce_unabsorbed_decode():
    """"潜在向量的作用": (q^C)^T W^UK c = ((W^UK)^T q^C)^T c and
    o = W^UV (sum_j a_j c_j).  Chaining the step oracles (absorb -> RoPE ->
    latent attention -> up-projection) must give the unabsorbed decode."""
    rng = np.random.default_rng(14)
    B, S, H, d_c, d_h, d_r, d_v = 2, 2, 3, 24, 6, 4, 5
    seqlens = [3, 13]
    p = _rand_problem(rng, B, S, H, seqlens, d_c, d_h, d_r, d_v, Lmax=14)
    scale = 1.0 / math.sqrt(d_h + d_r)
    want = oracle.decode(p["q_nope"], p["q_rope"], p["c_kv"], p["k_r"], p["W_UK"], p["W_UV"],
                         p["seqlens"], softmax_scale=scale)
    qt = oracle.absorb(p["q_nope"].reshape(B * S, H, d_h), p["W_UK"]).reshape(B, S, H, d_c)
    pos_q = np.array([[L - S + s for s in range(S)] for L in seqlens])
    qr = oracle.rope(p["q_rope"].reshape(-1, d_r), np.repeat(pos_q.reshape(-1), H))
    q_cat = np.concatenate([qt, qr.reshape(B, S, H, d_r)], axis=-1)
    k_rot = oracle.rope(p["k_r"].reshape(-1, d_r), np.tile(np.arange(14), B)).reshape(B, 14, d_r)
    o_lat = oracle.latent_attention(q_cat, p["c_kv"], k_rot, p["seqlens"], d_r=d_r,
                                    softmax_scale=scale)
    got = oracle.up_project(o_lat.reshape(B * S, H, d_c), p["W_UV"]).reshape(B, S, H, d_v)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-13)


def test_absorb_and_up_project_against_matrix_products():
    rng = np.random.default_rng(15)
    q = rng.standard_normal((3, 2, 5))
    W = rng.standard_normal((2, 5, 7))
    np.testing.assert_allclose(oracle.absorb(q, W), np.einsum("hdk,nhd->nhk", W, q), rtol=1e-13)
    o = rng.standard_normal((3, 2, 7))
    np.testing.assert_allclose(oracle.up_project(o, W), np.einsum("hdk,nhk->nhd", W, o),
                               rtol=1e-13)


# ------------------------------------------------------------ golden fixture
def test_cache_size_arithmetic_from_the_pages():
    """Per-token cache size printed on the pages (fixture cites them)."""
    with open(os.path.join(GOLDEN, "cache_size.json")) as f:
        g = json.load(f)
    from mla_latent_kv_68_b300.inputs import D_C, D_H, D_R, D_V
    assert D_C + D_R == g["mla_elements_per_token_per_layer"]
    assert (D_C, D_R, D_H, D_V) == (g["kv_lora_rank"], g["qk_rope_head_dim"],
                                    g["qk_nope_head_dim"], g["v_head_dim"])
    per_token_all_layers = (D_C + D_R) * 2 * g["num_layers"]
    assert abs(per_token_all_layers - g["mla_bytes_per_token_all_layers_approx"]) < 1000
    assert g["mha_elements_per_token_per_layer"] / g["mla_elements_per_token_per_layer"] == \
        pytest.approx(g["ratio_approx"], rel=0.01)
