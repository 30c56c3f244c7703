"""Pins of the oracle's output projection and of its folded weights.

"DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention / 注意力计算":
u_t = W^O [o_{t,1}; ...; o_{t,H}], the heads' outputs concatenated in head
order; "DeepSeek-V3 技术报告精读" (oopvo.github.io), "MLA": W^UV can be absorbed
into W^O.  Each check is fixed by those statements, not by the oracle's
formula: an identity W^O returns the concatenation, a one-hot row picks one
head's coordinate, the folded weights applied to o_lat equal W^O applied to
the up-projected heads of the unabsorbed decode, and the projection is linear.
A transposed weight, heads concatenated in the wrong order or a folding that
mixes heads each fail one of them.
"""
import numpy as np

import oracle


def test_identity_weight_returns_the_concatenated_heads():
    rng = np.random.default_rng(1)
    N, H, dv = 3, 4, 8
    heads = rng.standard_normal((N, H, dv))
    u = oracle.output_project(heads.reshape(N, H * dv), np.eye(H * dv))
    np.testing.assert_array_equal(u, heads.reshape(N, H * dv))
    assert u[1, 2 * dv + 5] == heads[1, 2, 5]          # head 2 sits after heads 0 and 1


def test_one_hot_row_picks_one_head_coordinate():
    rng = np.random.default_rng(2)
    N, H, dv, d = 4, 3, 5, 7
    x = rng.standard_normal((N, H * dv))
    W = np.zeros((d, H * dv))
    W[6, 1 * dv + 3] = 1.0                              # output 6 <- head 1, coordinate 3
    W[0, 0] = -2.0
    u = oracle.output_project(x, W)
    np.testing.assert_array_equal(u[:, 6], x[:, dv + 3])
    np.testing.assert_array_equal(u[:, 0], -2.0 * x[:, 0])
    assert np.count_nonzero(u[:, 1:6]) == 0


def test_folded_weights_equal_the_unfolded_chain():
    rng = np.random.default_rng(3)
    N, H, dv, dc, d = 5, 3, 4, 6, 9
    o_lat = rng.standard_normal((N, H, dc))
    W_UV = rng.standard_normal((H, dv, dc))
    W_O = rng.standard_normal((d, H * dv))
    heads = oracle.up_project(o_lat, W_UV)              # o_i = W_i^UV o_lat_i
    u_chain = oracle.output_project(heads.reshape(N, H * dv), W_O)
    u_fold = oracle.output_project(o_lat.reshape(N, H * dc), oracle.fold_output_weights(W_O, W_UV))
    np.testing.assert_allclose(u_fold, u_chain, rtol=1e-12, atol=1e-12)


def test_folded_projection_of_the_unabsorbed_decode():
    # the whole layer: the unabsorbed decode's per-head outputs through W^O
    # equal the absorbed latent result through the folded weights
    from mla_latent_kv_68_b300.inputs import make_inputs
    import math
    x = make_inputs(2, 1, 3, [7, 3], seed=5)
    b = {k: oracle_bits(x[k]) for k in ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV")}
    out = oracle.decode(b["q_nope"], b["q_rope"], b["c_kv"], b["k_r"], b["W_UK"], b["W_UV"],
                        x["seqlens"].numpy())                               # [B,S,H,128]
    rng = np.random.default_rng(6)
    W_O = rng.standard_normal((16, 3 * 128))
    u_heads = oracle.output_project(out.reshape(2, 3 * 128), W_O)
    # latent result from the absorbed steps, then the folded weights
    qt = oracle.absorb(b["q_nope"].reshape(2, 3, 128), b["W_UK"])
    L = x["seqlens"].numpy()
    qr = oracle.rope(b["q_rope"].reshape(-1, 64), np.repeat(L - 1, 3)).reshape(2, 1, 3, 64)
    q_cat = np.concatenate([qt.reshape(2, 1, 3, 512), qr], axis=-1)
    k_rot = np.zeros((2, x["Lmax"], 64))
    for i in range(2):
        k_rot[i, :L[i]] = oracle.rope(b["k_r"][i, :L[i]], np.arange(L[i]))
    lat = oracle.latent_attention(q_cat, oracle_f64(b["c_kv"]), k_rot, L, d_r=64,
                                  softmax_scale=1.0 / math.sqrt(192.0))
    u_fold = oracle.output_project(lat.reshape(2, 3 * 512), oracle.fold_output_weights(W_O, b["W_UV"]))
    np.testing.assert_allclose(u_fold, u_heads, rtol=1e-10, atol=1e-12)


def test_output_projection_is_linear():
    rng = np.random.default_rng(4)
    x, y = rng.standard_normal((2, 3, 12))
    W = rng.standard_normal((5, 12))
    np.testing.assert_allclose(oracle.output_project(2.5 * x - y, W),
                               2.5 * oracle.output_project(x, W) - oracle.output_project(y, W), rtol=1e-12)


def oracle_bits(t):
    from mla_latent_kv_68_b300.inputs import bf16_bits
    return bf16_bits(t)


def oracle_f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
