"""ctypes wrapper of the fp64 C oracle (``mla_oracle.c``).

TEST INFRASTRUCTURE ONLY.  Inputs are numpy arrays of float64, or of uint16
holding raw bf16 bit patterns (widened exactly inside the C code).  Outputs
are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

F64 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with gcc + OpenMP (plain C, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
             "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _LIB)
    return _LIB


def load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        vp, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.mla_oracle_num_threads.restype = i32
        lib.mla_oracle_rope.argtypes = [vp, i32, vp, i32, i32, f64, vp]
        lib.mla_oracle_rope_theta.argtypes = [vp, i32, vp, i32, i32, vp, vp]
        lib.mla_oracle_yarn_theta.argtypes = [f64, i32, f64, f64, f64, f64, vp]
        lib.mla_oracle_yarn_softmax_scale.argtypes = [f64, i32, i32, vp]
        lib.mla_oracle_decode_theta.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32,
                                                i32, i32, i32, i32, i32, f64, vp, vp, i64, vp, vp]
        lib.mla_oracle_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                          i32, i32, i32, i32, f64, f64, vp, i64, vp, vp]
        lib.mla_oracle_absorb.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp]
        lib.mla_oracle_up_project.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp]
        lib.mla_oracle_latent_attention.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, i32,
                                                    i32, i32, f64, vp, i64, vp]
        for name in ("mla_oracle_rope", "mla_oracle_decode", "mla_oracle_absorb",
                     "mla_oracle_up_project", "mla_oracle_latent_attention",
                     "mla_oracle_rope_theta", "mla_oracle_yarn_theta", "mla_oracle_decode_theta",
                     "mla_oracle_yarn_softmax_scale"):
            getattr(lib, name).restype = i32
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(load().mla_oracle_num_threads())


def _arr(x, dtype_code=None):
    """Return (contiguous array, dtype code).  uint16 means raw bf16 bits."""
    a = np.ascontiguousarray(x)
    if a.dtype == np.uint16:
        code = BF16
    elif a.dtype == np.float64:
        code = F64
    else:
        raise TypeError(f"oracle inputs must be float64 or uint16 (bf16 bits), got {a.dtype}")
    if dtype_code is not None and code != dtype_code:
        raise TypeError("all oracle inputs of one call must share one dtype")
    return a, code


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _f64(x):
    """Inputs as fp64: uint16 arrays are raw bf16 bits (widened exactly), as
    for every other entry of this oracle."""
    a, code = _arr(x)
    if code == BF16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def rope(x, pos, base: float = 10000.0):
    """RoPE of x[n, d_r] at integer positions pos[n] (interleaved pairs)."""
    a, code = _arr(x)
    n, d_r = a.shape
    p = np.ascontiguousarray(pos, dtype=np.int64)
    assert p.shape == (n,)
    out = np.empty((n, d_r), np.float64)
    _check(load().mla_oracle_rope(_ptr(a), code, _ptr(p), n, d_r, base, _ptr(out)), "rope")
    return out


def yarn_theta(d_r: int = 64, *, base: float = 10000.0, s: float = 40.0, alpha: float = 1.0,
               beta: float = 32.0, orig_len: float = 4096.0):
    """YaRN RoPE frequencies theta'_j (section "YaRN 扩展"), fp64 [d_r/2]."""
    out = np.empty(d_r // 2, np.float64)
    _check(load().mla_oracle_yarn_theta(float(base), d_r, float(s), float(alpha), float(beta),
                                        float(orig_len), _ptr(out)), "yarn_theta")
    return out


def yarn_softmax_scale(s: float = 40.0, d_h: int = 128, d_r: int = 64) -> float:
    """Softmax scale with YaRN's score factor, (0.1 ln s + 1) / sqrt(d_h + d_r)
    ("Long Context Extension"; "YaRN 扩展" scales the scores before the softmax)."""
    out = ctypes.c_double()
    _check(load().mla_oracle_yarn_softmax_scale(float(s), int(d_h), int(d_r), ctypes.byref(out)),
           "yarn_softmax_scale")
    return float(out.value)


def rope_theta(x, pos, theta):
    """RoPE of x[n, d_r] at positions pos[n] with explicit frequencies theta[d_r/2]."""
    a, code = _arr(x)
    n, d_r = a.shape
    p = np.ascontiguousarray(pos, dtype=np.int64)
    th = np.ascontiguousarray(theta, dtype=np.float64)
    assert p.shape == (n,) and th.shape == (d_r // 2,)
    out = np.empty((n, d_r), np.float64)
    _check(load().mla_oracle_rope_theta(_ptr(a), code, _ptr(p), n, d_r, _ptr(th), _ptr(out)),
           "rope_theta")
    return out


def decode(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, seqlens, *, softmax_scale=None,
           rope_base: float = 10000.0, rope_theta=None, rows=None, return_wsum: bool = False):
    """Unabsorbed MLA decode.  Shapes: q_nope [B,S,H,d_h], q_rope [B,S,H,d_r],
    c_kv [B,Lmax,d_c], k_r [B,Lmax,d_r] (pre-RoPE), W_UK [H,d_h,d_c],
    W_UV [H,d_v,d_c], seqlens [B].  Returns out [n_rows, d_v] for the flat rows
    (b*S+s)*H+h (all rows, shaped [B,S,H,d_v], when rows is None)."""
    qn, code = _arr(q_nope)
    qr, _ = _arr(q_rope, code)
    ck, _ = _arr(c_kv, code)
    kr, _ = _arr(k_r, code)
    wk, _ = _arr(W_UK, code)
    wv, _ = _arr(W_UV, code)
    B, S, H, d_h = qn.shape
    d_r = qr.shape[3]
    Lmax, d_c = ck.shape[1], ck.shape[2]
    d_v = wv.shape[1]
    assert qr.shape == (B, S, H, d_r) and ck.shape == (B, Lmax, d_c)
    assert kr.shape == (B, Lmax, d_r) and wk.shape == (H, d_h, d_c) and wv.shape == (H, d_v, d_c)
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    assert sl.shape == (B,)
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(d_h + d_r)
    if rows is None:
        n_rows, rp = B * S * H, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows, rp = rows.shape[0], _ptr(rows)
    out = np.empty((n_rows, d_v), np.float64)
    wsum = np.empty((n_rows,), np.float64)
    if rope_theta is None:
        rc = load().mla_oracle_decode(_ptr(qn), _ptr(qr), _ptr(ck), _ptr(kr), _ptr(wk), _ptr(wv),
                                      code, _ptr(sl), B, S, H, Lmax, d_c, d_h, d_r, d_v,
                                      float(softmax_scale), float(rope_base), rp, n_rows,
                                      _ptr(out), _ptr(wsum))
    else:
        th = np.ascontiguousarray(rope_theta, dtype=np.float64)
        assert th.shape == (d_r // 2,)
        rc = load().mla_oracle_decode_theta(_ptr(qn), _ptr(qr), _ptr(ck), _ptr(kr), _ptr(wk),
                                            _ptr(wv), code, _ptr(sl), B, S, H, Lmax, d_c, d_h,
                                            d_r, d_v, float(softmax_scale), _ptr(th), rp, n_rows,
                                            _ptr(out), _ptr(wsum))
    _check(rc, "decode")
    if rows is None:
        out = out.reshape(B, S, H, d_v)
        wsum = wsum.reshape(B, S, H)
    return (out, wsum) if return_wsum else out


def cache_append(h, W_DKV, W_KR, pos, *, rope_base: float = 10000.0, theta=None):
    """The cache entry of new tokens ("DeepSeek-V3" (ekkoxiao.github.io),
    "Multi-Head Latent Attention / KeyValue"):
        c_t^KV = W^DKV h_t,        k_t^R = RoPE_t(W^KR h_t),
    h [N, d], W_DKV [d_c, d], W_KR [d_r, d] (fp64, or uint16 bf16 bits),
    pos [N] (the position t of each token).  Returns (c [N, d_c], k_r [N, d_r]) in fp64.  The down-projections
    are plain matrix products (numpy, fp64); the rotation is this oracle's
    RoPE (base 10000, or explicit frequencies theta)."""
    hh, wd, wr = _f64(h), _f64(W_DKV), _f64(W_KR)
    N, d = hh.shape
    assert wd.shape[1] == d and wr.shape[1] == d
    c = hh @ wd.T
    k_pre = hh @ wr.T
    k_r = rope(k_pre, pos, rope_base) if theta is None else rope_theta(k_pre, pos, theta)
    return c, k_r


def absorb(q_nope, W_UK):
    """q~[n,h,:] = W_UK[h]^T q_nope[n,h,:].  q_nope [N,H,d_h], W_UK [H,d_h,d_c]."""
    qn, code = _arr(q_nope)
    wk, _ = _arr(W_UK, code)
    N, H, d_h = qn.shape
    d_c = wk.shape[2]
    assert wk.shape == (H, d_h, d_c)
    out = np.empty((N, H, d_c), np.float64)
    _check(load().mla_oracle_absorb(_ptr(qn), _ptr(wk), code, N, H, d_h, d_c, _ptr(out)), "absorb")
    return out


def up_project(o_lat, W_UV):
    """out[n,h,:] = W_UV[h] o_lat[n,h,:].  o_lat [N,H,d_c], W_UV [H,d_v,d_c]."""
    ol, code = _arr(o_lat)
    wv, _ = _arr(W_UV, code)
    N, H, d_c = ol.shape
    d_v = wv.shape[1]
    assert wv.shape == (H, d_v, d_c)
    out = np.empty((N, H, d_v), np.float64)
    _check(load().mla_oracle_up_project(_ptr(ol), _ptr(wv), code, N, H, d_v, d_c, _ptr(out)),
           "up_project")
    return out


def latent_attention(q_cat, c_kv, k_rot, seqlens, *, d_r: int, softmax_scale, rows=None):
    """Absorbed latent attention o_lat for already rotated inputs.
    q_cat [B,S,H,d_c+d_r], c_kv [B,Lmax,d_c], k_rot [B,Lmax,d_r]."""
    qc, code = _arr(q_cat)
    ck, _ = _arr(c_kv, code)
    kr, _ = _arr(k_rot, code)
    B, S, H, dq = qc.shape
    Lmax, d_c = ck.shape[1], ck.shape[2]
    assert dq == d_c + d_r and kr.shape == (B, Lmax, d_r)
    sl = np.ascontiguousarray(seqlens, dtype=np.int32)
    if rows is None:
        n_rows, rp = B * S * H, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows, rp = rows.shape[0], _ptr(rows)
    out = np.empty((n_rows, d_c), np.float64)
    rc = load().mla_oracle_latent_attention(_ptr(qc), _ptr(ck), _ptr(kr), code, _ptr(sl), B, S,
                                            H, Lmax, d_c, d_r, float(softmax_scale), rp, n_rows,
                                            _ptr(out))
    _check(rc, "latent_attention")
    if rows is None:
        out = out.reshape(B, S, H, d_c)
    return out


def output_project(x, W):
    """The layer's output projection ("DeepSeek-V3" (ekkoxiao.github.io),
    "Multi-Head Latent Attention / 注意力计算"): u_t = W^O [o_{t,1}; ...; o_{t,H}].
    x [N, K] (the heads' outputs of each token, concatenated), W [d, K]
    (fp64, or uint16 bf16 bits).  Returns u [N, d] in fp64: a plain matrix
    product (numpy)."""
    xx, ww = _f64(x), _f64(W)
    assert xx.ndim == 2 and ww.ndim == 2 and xx.shape[1] == ww.shape[1]
    return xx @ ww.T


def fold_output_weights(W_O, W_UV):
    """W^O with the value up-projection absorbed ("DeepSeek-V3 技术报告精读"
    (oopvo.github.io), "MLA": W^UV is absorbed into W^O): since
    o_i = W_i^UV o_lat_i, W^O [o_1; ...; o_H] = W~ [o_lat_1; ...; o_lat_H] with
    W~[:, i d_c:(i+1) d_c] = W^O[:, i d_v:(i+1) d_v] W_i^UV.
    W_O [d, H d_v], W_UV [H, d_v, d_c].  Returns W~ [d, H d_c] in fp64."""
    wo, wv = _f64(W_O), _f64(W_UV)
    H, d_v, d_c = wv.shape
    assert wo.shape[1] == H * d_v
    return np.concatenate([wo[:, i * d_v:(i + 1) * d_v] @ wv[i] for i in range(H)], axis=1)


def expand_kv(c_kv, W):
    """Keys or values expanded per head ("DeepSeek-V3" (ekkoxiao.github.io),
    "Multi-Head Latent Attention / KeyValue": k^C_{t,i} = W_i^UK c_t and
    v^C_{t,i} = W_i^UV c_t).  c_kv [..., d_c], W [H, d, d_c] (fp64, or uint16
    bf16 bits).  Returns [..., H, d] in fp64: a plain matrix product (numpy)."""
    cc, ww = _f64(c_kv), _f64(W)
    H, d, d_c = ww.shape
    assert cc.shape[-1] == d_c
    out = cc.reshape(-1, d_c) @ ww.reshape(H * d, d_c).T
    return out.reshape(*cc.shape[:-1], H, d)


def prefill_attention(q_nope, q_rot, k_c, k_rot, v_c, seqlens, *, softmax_scale):
    """Causal attention over expanded keys and values ("DeepSeek-V3"
    (ekkoxiao.github.io), "Multi-Head Latent Attention / 注意力计算"): query s of
    sequence b sits at position t = seqlens[b] - S + s and sees keys 0..t;
    score_j = (q^C . k^C_j + q^R . k^R_j) * softmax_scale; a = softmax over
    j <= t (shifted by the row maximum); o = sum_j a_j v^C_j.  q^R and k^R are
    taken as already rotated.
      q_nope [B,S,H,d_h], q_rot [B,S,H,d_r], k_c [B,Lmax,H,d_h],
      k_rot [B,Lmax,d_r], v_c [B,Lmax,H,d_v]  ->  out [B,S,H,d_v] (fp64).
    Plain numpy products per (sequence, head); cache rows at or past seqlens[b]
    are never read."""
    qn, qr, kc, kr, vc = (_f64(a) for a in (q_nope, q_rot, k_c, k_rot, v_c))
    B, S, H, _ = qn.shape
    d_v = vc.shape[-1]
    out = np.empty((B, S, H, d_v), np.float64)
    for b in range(B):
        L = int(seqlens[b])
        assert S <= L <= kc.shape[1]
        pos = L - S + np.arange(S)
        visible = np.arange(L)[None, :] <= pos[:, None]          # [S, L]
        for h in range(H):
            q = np.concatenate([qn[b, :, h], qr[b, :, h]], axis=1)  # [S, d_h + d_r]
            k = np.concatenate([kc[b, :L, h], kr[b, :L]], axis=1)   # [L, d_h + d_r]
            s = (q @ k.T) * softmax_scale
            s = np.where(visible, s, -np.inf)
            a = np.exp(s - s.max(axis=1, keepdims=True))
            a /= a.sum(axis=1, keepdims=True)
            out[b, :, h] = a @ vc[b, :L, h]
    return out
