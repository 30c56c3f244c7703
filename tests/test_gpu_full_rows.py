"""Every latent output row of the decode kernel at full size, against the fp64
oracle's absorbed latent attention ("DeepSeek-V3" (ekkoxiao.github.io),
"Multi-Head Latent Attention / 注意力计算": one softmax over all visible
positions; "潜在向量的作用": o_lat = sum_j a_j c_j).

The GPU runs mla_decode + mla_splitkv_combine in the launch configuration the
benchmark times, on the workloads' own cache.  Its absorbed, rotated queries
and rotated keys are computed by the oracle (absorb and RoPE) and rounded to
bf16, so both sides see the same bf16 inputs and no expected value depends on
the CUDA path.  Checked: all 4096 rows of the 4096-token workload, all rows
of one sequence of the 128K workload, and all rows of the longest and the
shortest sequence of the variable-length workload.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, bits, f64
from mla_latent_kv_68_b300 import binding as mb
from mla_latent_kv_68_b300.inputs import workload_inputs

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192.0)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_68_b300 import build
    build.build()
    mb.lib()


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16)


def _oracle_inputs(x):
    """q_cat = [(W_UK)^T q_nope ; RoPE(q_rope)] and RoPE(k_r), from the oracle, in bf16."""
    B, S, H, Lmax = x["B"], x["S"], x["H"], x["Lmax"]
    L = x["seqlens"].numpy().astype(np.int64)
    qt = oracle.absorb(bits(x["q_nope"]).reshape(B * S, H, 128), bits(x["W_UK"]))
    pos = np.repeat(np.array([[l - S + s for s in range(S)] for l in L]).reshape(-1), H)
    qr = oracle.rope(bits(x["q_rope"]).reshape(-1, 64), pos)
    q_cat = _bf16(np.concatenate([qt.reshape(B, S, H, 512), qr.reshape(B, S, H, 64)], axis=-1))
    k_rot = torch.zeros(B, Lmax, 64, dtype=torch.bfloat16)
    for b in range(B):
        k_rot[b, :L[b]] = _bf16(oracle.rope(bits(x["k_r"][b, :L[b]]), np.arange(L[b])))
    return q_cat, k_rot


def _gpu_latent(x, q_cat, k_rot):
    B, S, H = x["B"], x["S"], x["H"]
    ws = mb.new_workspace(B, S, H)
    o = torch.full((B, S, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.decode(q_cat.cuda(), x["c_kv"].cuda(), k_rot.cuda(), x["seqlens"].cuda(), ws)
    mb.splitkv_combine(ws, o)
    assert mb.read_status(ws) == mb.MLA_OK
    return f64(o).reshape(-1, 512)


@pytest.mark.parametrize("name,pick", [
    ("uniform_b32_s1_h128_l4096", "all"),
    ("long_b4_s1_h128_l131072", "seq1"),
    ("varlen_b64_s1_h128_l1to32768", "extremes"),
])
def test_full_size_every_row_of_the_chosen_sequences(name, pick):
    x = workload_inputs(name)
    q_cat, k_rot = _oracle_inputs(x)
    got = _gpu_latent(x, q_cat, k_rot)
    B, S, H = x["B"], x["S"], x["H"]
    L = x["seqlens"].numpy()
    if pick == "all":
        seqs = list(range(B))
    elif pick == "seq1":
        seqs = [1]
    else:
        seqs = sorted({int(np.argmax(L)), int(np.argmin(L))})
    rows = np.concatenate([np.arange(b * S * H, (b + 1) * S * H) for b in seqs]).astype(np.int64)
    ref = oracle.latent_attention(bits(q_cat), bits(x["c_kv"]), bits(k_rot), L, d_r=64,
                                  softmax_scale=SCALE, rows=rows)
    assert np.isfinite(got).all()
    assert_close(got[rows], ref, what=f"{name} rows of sequences {seqs}")
    torch.cuda.empty_cache()
