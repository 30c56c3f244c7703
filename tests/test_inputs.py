"""Host-side checks of the seeded input generator (no GPU)."""
import numpy as np
import torch

from mla_latent_kv_68_b300.inputs import WORKLOADS, make_inputs


def test_deterministic_and_seed_sensitive():
    a = make_inputs(2, 1, 4, [5, 9], seed=11)
    b = make_inputs(2, 1, 4, [5, 9], seed=11)
    c = make_inputs(2, 1, 4, [5, 9], seed=12)
    for k in ("c_kv", "k_r", "q_nope", "q_rope", "W_UK", "W_UV"):
        assert torch.equal(a[k], b[k])
        assert not torch.equal(a[k], c[k])


def test_shapes_dtypes_and_padding():
    x = make_inputs(3, 2, 8, [2, 7, 4], Lmax=8, seed=1, pad=float("nan"))
    assert x["c_kv"].shape == (3, 8, 512) and x["k_r"].shape == (3, 8, 64)
    assert x["q_nope"].shape == (3, 2, 8, 128) and x["q_rope"].shape == (3, 2, 8, 64)
    assert x["W_UK"].shape == (8, 128, 512) and x["W_UV"].shape == (8, 128, 512)
    assert all(x[k].dtype == torch.bfloat16 for k in ("c_kv", "k_r", "q_nope", "W_UK"))
    assert x["seqlens"].dtype == torch.int32
    assert torch.isnan(x["c_kv"][1, 7:]).all() and not torch.isnan(x["c_kv"][1, :7]).any()
    assert torch.isnan(x["k_r"][0, 2:]).all() and not torch.isnan(x["k_r"][0, :2]).any()


def test_drawn_lengths_in_range_and_distributions():
    x = make_inputs(64, 1, 2, None, Lmax=512, L_range=(1, 512), seed=5)
    L = x["seqlens"].numpy()
    assert L.min() >= 1 and L.max() <= 512 and len(np.unique(L)) > 30
    w = x["W_UK"].float()
    assert abs(w.std().item() - 1 / np.sqrt(512)) < 2e-3
    q = x["q_nope"].float()
    assert abs(q.std().item() - 1.0) < 0.05


def test_workload_table():
    assert [(w.B, w.S, w.H) for w in WORKLOADS.values()] == [
        (1, 1, 16), (32, 1, 128), (64, 1, 128), (16, 2, 128), (4, 1, 128)]
    assert WORKLOADS["long_b4_s1_h128_l131072"].c_scale == 0.5
    assert WORKLOADS["varlen_b64_s1_h128_l1to32768"].L_range == (1, 32768)
