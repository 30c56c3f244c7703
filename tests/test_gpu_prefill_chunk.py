"""Chunked prefill through the decode path: S new queries per sequence.

"DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention / 注意力计算":
query s of a chunk sits at position L_b - S + s and sees the cache rows
0 .. L_b - S + s.  The decode kernel takes S * H <= 2048 query rows per
sequence (up to 16 row blocks of 128); this checks chunks of S = 4, 8 and 16
against the fp64 oracle of the unabsorbed definition, through the whole step
(absorb + RoPE, decode, combine, up-projection), with ragged lengths, a
sequence exactly as long as its chunk, and row blocks that mix queries.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, bits, f64, to_dev
from mla_latent_kv_68_b300 import binding as mb
from mla_latent_kv_68_b300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_68_b300 import build
    build.build()
    mb.lib()
    yield
    assert mb.read_status() == mb.MLA_OK


@pytest.mark.parametrize("B,S,H,seqlens,seed", [
    (2, 4, 32, [4, 300], 41),          # one sequence exactly as long as its chunk
    (3, 8, 16, [8, 129, 1000], 42),    # 128 rows: one row block per sequence
    (2, 8, 48, [520, 77], 43),         # 384 rows: row blocks that mix queries
    (1, 16, 128, [1100], 44),          # 2048 rows: sixteen row blocks
])
def test_chunked_prefill_matches_oracle(B, S, H, seqlens, seed):
    x = make_inputs(B, S, H, seqlens, seed=seed)
    d = to_dev(x)
    mb.rope_cache(d["k_r"], d["seqlens"])
    step = mb.DecodeStep(B, S, H)
    out = step(d["q_nope"], d["q_rope"], d["c_kv"], d["k_r"], d["seqlens"], d["W_UK"], d["W_UV"])
    assert mb.read_status(step.workspace) == mb.MLA_OK
    b = {k: bits(x[k]) for k in ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV")}
    n = B * S * H
    # every row when few; otherwise a seeded sample plus every head of the first and last query
    rows = np.arange(n) if n <= 1024 else np.unique(np.concatenate([
        np.random.default_rng(seed).choice(n, 384, replace=False), np.arange(H), np.arange(n - H, n)]))
    ref = oracle.decode(b["q_nope"], b["q_rope"], b["c_kv"], b["k_r"], b["W_UK"], b["W_UV"],
                        x["seqlens"].numpy(), rows=rows)
    assert_close(f64(out).reshape(n, -1)[rows], ref, what=f"prefill chunk B{B} S{S} H{H}")
