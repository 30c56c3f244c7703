"""GPU parity of every kernel of the decode step against the fp64 CPU oracle.

All calls go through the C ABI (ctypes binding).  Inputs are seeded and drawn
on the CPU; expected values come only from ``oracle/``.  Shapes span several
64-row cache tiles, ragged tails, L = 1, S = 2 at L = 2, H that is not a
power of two, more query rows than one 128-row block, and batches larger than
one MMA tile.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, bits, f64, rel_l2, to_dev
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


def _bf16(a, shape=None):
    t = torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)
    return t.reshape(shape) if shape is not None else t


# ------------------------------------------------------------------ RoPE
def test_rope_explicit_positions_match_oracle():
    g = torch.Generator().manual_seed(1)
    N, nh = 37, 3
    x = torch.randn(N, nh, 64, generator=g).to(torch.bfloat16)
    pos = torch.randint(0, 131072, (N,), generator=g, dtype=torch.int32)
    pos[0], pos[1], pos[2] = 0, 1, 131071
    xd, pd = x.cuda(), pos.cuda()
    out = torch.full((N, nh, 64), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.rope_apply(xd, nh * 64, 64, out, nh * 64, 64, N, nh, mb.POS_EXPLICIT, pd)
    ref = oracle.rope(bits(x).reshape(N * nh, 64), np.repeat(pos.numpy().astype(np.int64), nh))
    got = f64(out).reshape(N * nh, 64)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5   # half a bf16 ulp of the result, plus fp32 slack
    assert (np.abs(got - ref) <= bound).all(), float(np.abs(got - ref).max())


def test_rope_query_mode_writes_only_the_rope_columns():
    B, S, H = 3, 2, 5
    g = torch.Generator().manual_seed(2)
    q_rope = torch.randn(B, S, H, 64, generator=g).to(torch.bfloat16)
    seqlens = torch.tensor([2, 9, 4000], dtype=torch.int32)
    q_cat = torch.randn(B, S, H, 576, generator=g).to(torch.bfloat16)
    before = q_cat.clone()
    qd = q_cat.cuda()
    mb.rope_queries(q_rope.cuda(), qd, seqlens.cuda())
    got = qd.cpu()
    assert torch.equal(got[..., :512], before[..., :512])
    pos = np.array([[L - S + s for s in range(S)] for L in seqlens.tolist()]).reshape(-1)
    ref = oracle.rope(bits(q_rope).reshape(-1, 64), np.repeat(pos, H))
    g64 = got[..., 512:].double().numpy().reshape(-1, 64)
    assert (np.abs(g64 - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5).all()


def test_rope_cache_mode_in_place_leaves_padding():
    B, Lmax = 3, 70
    g = torch.Generator().manual_seed(3)
    k = torch.randn(B, Lmax, 64, generator=g).to(torch.bfloat16)
    seqlens = torch.tensor([1, 70, 33], dtype=torch.int32)
    kd = k.cuda()
    mb.rope_cache(kd, seqlens.cuda())
    got = kd.cpu()
    for b, L in enumerate(seqlens.tolist()):
        assert torch.equal(got[b, L:], k[b, L:])
        ref = oracle.rope(bits(k[b, :L]), np.arange(L))
        assert (np.abs(got[b, :L].double().numpy() - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5).all()


# ------------------------------------------------------------------ absorb / up-projection
@pytest.mark.parametrize("B,S,H", [(1, 1, 16), (32, 1, 128), (16, 2, 128), (3, 1, 5),
                                   (300, 1, 2), (64, 1, 128)])
def test_absorb_matches_oracle(B, S, H):
    g = torch.Generator().manual_seed(B * 1000 + S * 100 + H)
    q = torch.randn(B, S, H, 128, generator=g).to(torch.bfloat16)
    W = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    q_cat = torch.randn(B, S, H, 576, generator=g).to(torch.bfloat16)
    tail = q_cat[..., 512:].clone()
    qd = q_cat.cuda()
    mb.absorb_q(q.cuda(), W.cuda(), qd)
    got = qd.cpu()
    assert torch.equal(got[..., 512:], tail)
    ref = oracle.absorb(bits(q).reshape(B * S, H, 128), bits(W)).reshape(B, S, H, 512)
    g64 = got[..., :512].double().numpy()
    # fp32 accumulation of 128 products, then one bf16 rounding
    assert (np.abs(g64 - ref) <= 2.0 ** -8 * np.abs(ref) + 2e-4).all(), float(np.abs(g64 - ref).max())
    assert rel_l2(g64, ref) < 3e-3


@pytest.mark.parametrize("B,S,H", [(1, 1, 16), (32, 1, 128), (16, 2, 128), (3, 2, 5), (300, 1, 2)])
def test_absorb_rope_matches_oracle(B, S, H):
    g = torch.Generator().manual_seed(B * 977 + S * 31 + H)
    q = torch.randn(B, S, H, 128, generator=g).to(torch.bfloat16)
    qr = torch.randn(B, S, H, 64, generator=g).to(torch.bfloat16)
    W = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    seqlens = torch.randint(S, 140000, (B,), generator=g, dtype=torch.int32)
    seqlens[0] = S                                   # the query at position 0 .. S-1
    q_cat = torch.full((B, S, H, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.absorb_rope_q(q.cuda(), qr.cuda(), W.cuda(), seqlens.cuda(), q_cat)
    got = q_cat.cpu().double().numpy()
    ref = oracle.absorb(bits(q).reshape(B * S, H, 128), bits(W)).reshape(B, S, H, 512)
    assert (np.abs(got[..., :512] - ref) <= 2.0 ** -8 * np.abs(ref) + 2e-4).all()
    pos = np.array([[L - S + s for s in range(S)] for L in seqlens.tolist()]).reshape(-1)
    rref = oracle.rope(bits(qr).reshape(-1, 64), np.repeat(pos, H)).reshape(B, S, H, 64)
    assert (np.abs(got[..., 512:] - rref) <= 2.0 ** -8 * np.abs(rref) + 1e-5).all()


@pytest.mark.parametrize("B,S,H", [(1, 1, 16), (32, 1, 128), (64, 1, 128), (100, 1, 3),
                                   (16, 2, 128)])
def test_up_project_matches_oracle(B, S, H):
    g = torch.Generator().manual_seed(7 + B * 1000 + S * 100 + H)
    o = torch.randn(B, S, H, 512, generator=g).to(torch.bfloat16)
    W = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    out = torch.empty(B, S, H, 128, dtype=torch.bfloat16, device="cuda")
    mb.up_project(o.cuda(), W.cuda(), out)
    ref = oracle.up_project(bits(o).reshape(B * S, H, 512), bits(W)).reshape(B, S, H, 128)
    got = f64(out)
    assert (np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2e-4).all(), float(np.abs(got - ref).max())
    assert rel_l2(got, ref) < 3e-3


# ------------------------------------------------------------------ decode + combine
def _latent_case(B, S, H, seqlens, seed, Lmax=None, pad=0.0, c_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    Lmax = Lmax or max(seqlens)
    c = torch.full((B, Lmax, 512), pad)
    k = torch.full((B, Lmax, 64), pad)
    for b, L in enumerate(seqlens):
        c[b, :L] = torch.randn(L, 512, generator=g) * c_scale
        k[b, :L] = torch.randn(L, 64, generator=g)
    q = torch.cat([0.5 * torch.randn(B, S, H, 512, generator=g),
                   torch.randn(B, S, H, 64, generator=g)], dim=-1)
    return (q.to(torch.bfloat16), c.to(torch.bfloat16), k.to(torch.bfloat16),
            torch.tensor(seqlens, dtype=torch.int32))


def _run_latent(q, c, k, sl):
    B, S, H, _ = q.shape
    ws = mb.new_workspace(B, S, H)
    o = torch.empty(B, S, H, 512, dtype=torch.bfloat16, device="cuda")
    sld = sl.cuda()
    mb.decode(q.cuda(), c.cuda(), k.cuda(), sld, ws)
    mb.splitkv_combine(ws, o)
    assert mb.read_status(ws) == mb.MLA_OK
    return f64(o)


LATENT_CASES = [
    (1, 1, 16, [256]),                 # the tiny workload's shape
    (3, 1, 128, [1, 64, 65]),          # one row, one full tile, one tile plus one row
    (2, 2, 128, [2, 130]),             # S = 2 at the minimum length; two row blocks
    (4, 1, 96, [17, 300, 1000, 4096]), # H not a power of two, ragged tails
    (2, 2, 96, [77, 2048]),            # 192 rows: a row block mixing both queries
    (5, 1, 128, [4999, 1, 3000, 129, 8191]),
]


@pytest.mark.parametrize("B,S,H,seqlens", LATENT_CASES)
def test_decode_combine_matches_latent_oracle(B, S, H, seqlens):
    q, c, k, sl = _latent_case(B, S, H, seqlens, seed=B * 31 + S * 7 + H)
    got = _run_latent(q, c, k, sl)
    ref = oracle.latent_attention(bits(q), bits(c), bits(k), sl.numpy(), d_r=64,
                                  softmax_scale=1.0 / math.sqrt(192.0))
    assert_close(got, ref, what=f"o_lat B{B} S{S} H{H}")


def test_decode_one_token_returns_that_latent():
    q, c, k, sl = _latent_case(2, 1, 128, [1, 1], seed=5)
    got = _run_latent(q, c, k, sl)
    want = c[:, 0].double().numpy()[:, None, None, :]
    assert np.abs(got - want).max() <= 2.0 ** -8 * np.abs(want).max()


def test_decode_ignores_nan_padding():
    q, c, k, sl = _latent_case(3, 2, 128, [2, 70, 333], seed=9, Lmax=400, pad=float("nan"))
    got = _run_latent(q, c, k, sl)
    ref = oracle.latent_attention(bits(q), bits(c), bits(k), sl.numpy(), d_r=64,
                                  softmax_scale=1.0 / math.sqrt(192.0))
    assert_close(got, ref, what="nan padding")


def test_large_cache_values_keep_the_split_partials_in_range():
    # Cache rows near 1e5 (a common offset plus 1% noise): every latent mix
    # U = O / l of a split is near 1e5, beyond fp16's 65504, so the stored
    # partials need their per-half-row power-of-two exponent.  The queries are
    # scaled down so the scores stay ordinary; compare relative to 1e5.
    g = torch.Generator().manual_seed(31)
    B, S, H, seqlens = 3, 1, 128, [5000, 300, 9000]
    Lmax = max(seqlens)
    c = torch.zeros(B, Lmax, 512)
    k = torch.zeros(B, Lmax, 64)
    for b, L in enumerate(seqlens):
        c[b, :L] = 1e5 * (1.0 + 0.01 * torch.randn(L, 512, generator=g))
        k[b, :L] = torch.randn(L, 64, generator=g)
    q = torch.cat([5e-4 * torch.randn(B, S, H, 512, generator=g),
                   torch.randn(B, S, H, 64, generator=g)], dim=-1)
    q, c, k = q.to(torch.bfloat16), c.to(torch.bfloat16), k.to(torch.bfloat16)
    sl = torch.tensor(seqlens, dtype=torch.int32)
    got = _run_latent(q, c, k, sl)
    ref = oracle.latent_attention(bits(q), bits(c), bits(k), sl.numpy(), d_r=64,
                                  softmax_scale=1.0 / math.sqrt(192.0))
    assert np.abs(ref).max() > 65504.0
    assert_close(got / 1e5, ref / 1e5, what="cache values near 1e5")


def test_huge_scores_select_the_top_key():
    # Queries scaled by 1e4: scores reach tens of thousands in log2 units,
    # far from each other, so the softmax is one-hot on each row's top key;
    # the row maximum is carried as a float (no clamp on its range).
    B, S, H, seqlens = 2, 2, 64, [1000, 777]
    q, c, k, sl = _latent_case(B, S, H, seqlens, seed=33)
    q = (q.float() * torch.cat([torch.full((512,), 1e4), torch.ones(64)])).to(torch.bfloat16)
    got = _run_latent(q, c, k, sl)
    ref = oracle.latent_attention(bits(q), bits(c), bits(k), sl.numpy(), d_r=64,
                                  softmax_scale=1.0 / math.sqrt(192.0))
    s2 = (q[..., :512].double() @ c.double().transpose(1, 2).unsqueeze(1)) / math.sqrt(192.0) / math.log(2.0)
    assert s2.abs().max() > 32000.0
    assert_close(got, ref, what="one-hot rows")


def test_bad_seqlen_is_reported_and_recovers():
    q, c, k, sl = _latent_case(2, 2, 16, [5, 9], seed=11)
    ws = mb.new_workspace(2, 2, 16)
    o = torch.empty(2, 2, 16, 512, dtype=torch.bfloat16, device="cuda")
    bad = torch.tensor([1, 9], dtype=torch.int32, device="cuda")   # 1 < S
    mb.decode(q.cuda(), c.cuda(), k.cuda(), bad, ws)
    mb.splitkv_combine(ws, o)
    assert mb.read_status(ws) == 5                                  # MLA_ERR_BAD_SEQLEN
    too_long = torch.tensor([5, 10], dtype=torch.int32, device="cuda")  # > Lmax = 9
    mb.decode(q.cuda(), c.cuda(), k.cuda(), too_long, ws)
    assert mb.read_status(ws) == 5
    got = _run_latent(q, c, k, sl)                                  # clean afterwards
    ref = oracle.latent_attention(bits(q), bits(c), bits(k), sl.numpy(), d_r=64,
                                  softmax_scale=1.0 / math.sqrt(192.0))
    assert_close(got, ref, what="after error")


def test_decode_never_reads_unwritten_workspace():
    # Few tiles and two row blocks: fewer tiles than split groups, so some
    # groups own no tile.  The workspace (beyond its status word) is filled
    # with finite garbage that a stray read would fold into the result.
    q, c, k, sl = _latent_case(3, 2, 96, [2, 700, 2500], seed=202)
    B, S, H = 3, 2, 96
    ws = mb.new_workspace(B, S, H)
    ws[256:] = 0x3F                     # every (m, l) reads as 0.747, every fp16 partial as 1.81
    o = torch.empty(B, S, H, 512, dtype=torch.bfloat16, device="cuda")
    for _ in range(2):
        mb.decode(q.cuda(), c.cuda(), k.cuda(), sl.cuda(), ws)
        mb.splitkv_combine(ws, o)
        assert mb.read_status(ws) == mb.MLA_OK
        ref = oracle.latent_attention(bits(q), bits(c), bits(k), sl.numpy(), d_r=64,
                                      softmax_scale=1.0 / math.sqrt(192.0))
        assert_close(f64(o), ref, what="garbage workspace")


def test_workspace_too_small_is_rejected():
    q, c, k, sl = _latent_case(1, 1, 16, [10], seed=12)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(mb.MLAError) as e:
        mb.decode(q.cuda(), c.cuda(), k.cuda(), sl.cuda(), ws)
    assert e.value.status == 3


# ------------------------------------------------------------------ whole step vs unabsorbed oracle
def _step(x):
    d = to_dev(x)
    mb.rope_cache(d["k_r"], d["seqlens"])
    step = mb.DecodeStep(x["B"], x["S"], x["H"])
    out = step(d["q_nope"], d["q_rope"], d["c_kv"], d["k_r"], d["seqlens"], d["W_UK"], d["W_UV"])
    assert mb.read_status(step.workspace) == mb.MLA_OK
    return f64(out)


def _oracle_rows(x, rows=None):
    b = {kk: bits(x[kk]) for kk in ("q_nope", "q_rope", "c_kv", "k_r", "W_UK", "W_UV")}
    return oracle.decode(b["q_nope"], b["q_rope"], b["c_kv"], b["k_r"], b["W_UK"], b["W_UV"],
                         x["seqlens"].numpy(), rows=rows)


@pytest.mark.parametrize("B,S,H,seqlens,seed", [
    (1, 1, 16, [256], 68000),
    (3, 2, 8, [2, 100, 333], 3),
    (2, 1, 128, [64, 1500], 4),
])
def test_whole_step_matches_unabsorbed_oracle(B, S, H, seqlens, seed):
    x = make_inputs(B, S, H, seqlens, seed=seed)
    got = _step(x)
    ref = _oracle_rows(x)
    assert_close(got, ref, what=f"out B{B} S{S} H{H}")
