"""Prefill: the per-head expansion of keys and values and causal attention
over them, against the fp64 oracle.

"DeepSeek-V3" (ekkoxiao.github.io), "Multi-Head Latent Attention":
"KeyValue" (k^C = W^UK c, v^C = W^UV c), "Query" and "注意力计算" (query t sees
keys 0..t; one softmax over them).  The attention kernel is checked alone on
the same bf16 inputs as the oracle's step (expanded keys and values, rotated
q^R and k^R all rounded to bf16 once, by the oracle's values), and the whole
chain (RoPE of the queries, expansion, attention) against the unabsorbed
decode oracle.  Cases: a single query and a single key; prompts of exactly
128 positions; partial query blocks; chunks after cached context; padding
rows that hold NaN; a sequence whose length is out of range.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, bits, f64, to_dev
from mla_latent_kv_68_b300 import binding as mb
from mla_latent_kv_68_b300.inputs import make_inputs

pytestmark = pytest.mark.gpu

SCALE = 1.0 / math.sqrt(192.0)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_latent_kv_68_b300 import build
    build.build()
    mb.lib()
    yield
    assert mb.read_status() == mb.MLA_OK


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("B,Lmax,H,seed", [(1, 1, 1, 1), (2, 300, 3, 2), (3, 129, 128, 3)])
def test_expand_matches_oracle(B, Lmax, H, seed):
    x = make_inputs(B, 1, H, [Lmax] * B, seed=seed)
    d = to_dev(x)
    k_c = torch.empty(B, Lmax, H, 128, dtype=torch.bfloat16, device="cuda")
    v_c = torch.empty_like(k_c)
    mb.prefill_expand(d["c_kv"], d["W_UK"], d["W_UV"], k_c, v_c)
    assert mb.read_status() == mb.MLA_OK
    cb = bits(x["c_kv"])
    assert_close(f64(k_c), oracle.expand_kv(cb, bits(x["W_UK"])), what="k^C")
    assert_close(f64(v_c), oracle.expand_kv(cb, bits(x["W_UV"])), what="v^C")


def _attention_inputs(B, S, H, seqlens, Lmax, seed):
    """bf16 inputs of the attention step, formed by the oracle and rounded once."""
    x = make_inputs(B, S, H, seqlens, Lmax=Lmax, seed=seed)
    L = x["seqlens"].numpy()
    qb, kb = bits(x["q_rope"]), bits(x["k_r"])
    q_rot = np.zeros((B, S, H, 64))
    k_rot = np.full((B, Lmax, 64), np.nan)
    for b in range(B):
        pos = np.repeat(L[b] - S + np.arange(S), H)
        q_rot[b] = oracle.rope(qb[b].reshape(-1, 64), pos).reshape(S, H, 64)
        k_rot[b, :L[b]] = oracle.rope(kb[b, :L[b]], np.arange(L[b]))
    k_c = oracle.expand_kv(bits(x["c_kv"]), bits(x["W_UK"]))
    v_c = oracle.expand_kv(bits(x["c_kv"]), bits(x["W_UV"]))
    for b in range(B):                       # padding rows hold NaN: never read
        k_c[b, L[b]:] = np.nan
        v_c[b, L[b]:] = np.nan
    t = dict(q_nope=x["q_nope"], q_rot=_bf16(q_rot), k_c=_bf16(k_c), k_r=_bf16(k_rot), v_c=_bf16(v_c),
             seqlens=x["seqlens"])
    return t, L


@pytest.mark.parametrize("B,S,H,seqlens,Lmax,seed", [
    (1, 1, 1, [1], 1, 11),               # one query, one key
    (1, 128, 2, [128], 128, 12),         # one whole query block, a whole prompt
    (2, 77, 3, [77, 200], 256, 13),      # partial block; a chunk after 123 cached tokens
    (2, 300, 2, [300, 555], 600, 14),    # three blocks, the last partial; ragged context
    (1, 513, 1, [1000], 1024, 15),       # five blocks after 487 cached tokens
])
def test_attention_matches_oracle(B, S, H, seqlens, Lmax, seed):
    t, L = _attention_inputs(B, S, H, seqlens, Lmax, seed)
    d = to_dev(t)
    out = torch.full((B, S, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.prefill_attention(d["q_nope"], d["q_rot"], d["k_c"], d["k_r"], d["v_c"], d["seqlens"], out, SCALE)
    assert mb.read_status() == mb.MLA_OK
    ref = oracle.prefill_attention(bits(t["q_nope"]), bits(t["q_rot"]), bits(t["k_c"]), bits(t["k_r"]),
                                   bits(t["v_c"]), L, softmax_scale=SCALE)
    assert_close(f64(out), ref, what=f"prefill attention B{B} S{S} H{H}")


@pytest.mark.parametrize("B,S,H,seqlens,seed", [
    (2, 200, 4, [200, 333], 21),
    (1, 384, 16, [384], 22),
])
def test_prefill_chain_matches_unabsorbed_oracle(B, S, H, seqlens, seed):
    x = make_inputs(B, S, H, seqlens, seed=seed, pad=float("nan"))
    d = to_dev(x)
    mb.rope_cache(d["k_r"], d["seqlens"])
    step = mb.PrefillStep(B, S, H, x["Lmax"])
    out = step(d["q_nope"], d["q_rope"], d["c_kv"], d["k_r"], d["seqlens"], d["W_UK"], d["W_UV"])
    assert mb.read_status() == mb.MLA_OK
    n = B * S * H
    rows = np.unique(np.concatenate([np.random.default_rng(seed).choice(n, 600, replace=False),
                                     np.arange(H), np.arange(n - H, n)]))
    b = {k: bits(x[k]) for k in ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV")}
    ref = oracle.decode(b["q_nope"], b["q_rope"], b["c_kv"], b["k_r"], b["W_UK"], b["W_UV"],
                        x["seqlens"].numpy(), rows=rows)
    assert_close(f64(out).reshape(n, -1)[rows], ref, what=f"prefill chain B{B} S{S} H{H}")


def test_prefill_with_yarn_matches_oracle():
    B, S, H = 1, 256, 2
    x = make_inputs(B, S, H, [700], seed=31)
    d = to_dev(x)
    theta = oracle.yarn_theta()
    scale = oracle.yarn_softmax_scale()
    mb.rope_cache(d["k_r"], d["seqlens"], theta=theta)
    step = mb.PrefillStep(B, S, H, x["Lmax"])
    out = step(d["q_nope"], d["q_rope"], d["c_kv"], d["k_r"], d["seqlens"], d["W_UK"], d["W_UV"],
               softmax_scale=scale, theta=theta)
    assert mb.read_status() == mb.MLA_OK
    b = {k: bits(x[k]) for k in ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV")}
    ref = oracle.decode(b["q_nope"], b["q_rope"], b["c_kv"], b["k_r"], b["W_UK"], b["W_UV"],
                        x["seqlens"].numpy(), softmax_scale=scale, rope_theta=theta)
    assert_close(f64(out), ref, what="prefill with YaRN")


def test_out_of_range_length_is_reported_and_skipped():
    t, L = _attention_inputs(2, 100, 2, [100, 180], 200, 41)
    d = to_dev(t)
    d["seqlens"] = torch.tensor([100, 50], dtype=torch.int32, device="cuda")   # 50 < S
    out = torch.zeros(2, 100, 2, 128, dtype=torch.bfloat16, device="cuda")
    mb.prefill_attention(d["q_nope"], d["q_rot"], d["k_c"], d["k_r"], d["v_c"], d["seqlens"], out, SCALE)
    assert mb.read_status() == mb.MLA_ERR_BAD_SEQLEN
    assert not out[1].any()                                                     # its rows untouched
    ref = oracle.prefill_attention(bits(t["q_nope"])[:1], bits(t["q_rot"])[:1], bits(t["k_c"])[:1],
                                   bits(t["k_r"])[:1], bits(t["v_c"])[:1], L[:1], softmax_scale=SCALE)
    assert_close(f64(out[:1]), ref, what="the valid sequence")


def test_prefill_bench_workload_heads_match_oracle():
    """The benchmark's prefill (4 prompts of 4096 tokens, 128 heads, the same
    seeded inputs): every query row of three (sequence, head) pairs, against the
    oracle's own expansion, RoPE and causal attention for those heads."""
    B, S, H = 4, 4096, 128
    x = make_inputs(B, S, H, [S] * B, seed=68005)
    d = to_dev(x)
    mb.rope_cache(d["k_r"], d["seqlens"])
    step = mb.PrefillStep(B, S, H, S)
    out = step(d["q_nope"], d["q_rope"], d["c_kv"], d["k_r"], d["seqlens"], d["W_UK"], d["W_UV"])
    assert mb.read_status() == mb.MLA_OK
    qn, qr, ck, kr = (bits(x[k]) for k in ("q_nope", "q_rope", "c_kv", "k_r"))
    wk, wv = bits(x["W_UK"]), bits(x["W_UV"])
    for b, h in [(0, 0), (3, 127), (1, 77)]:
        kc = oracle.expand_kv(ck[b:b + 1], wk[h:h + 1])                     # [1, S, 1, 128]
        vc = oracle.expand_kv(ck[b:b + 1], wv[h:h + 1])
        q_rot = oracle.rope(qr[b, :, h], np.arange(S)).reshape(1, S, 1, 64)  # query s at position s
        k_rot = oracle.rope(kr[b], np.arange(S)).reshape(1, S, 64)
        ref = oracle.prefill_attention(qn[b:b + 1, :, h:h + 1], q_rot, kc, k_rot, vc, [S], softmax_scale=SCALE)
        assert_close(f64(out[b, :, h]), ref[0, :, 0], what=f"prefill 4x4096 sequence {b} head {h}")
