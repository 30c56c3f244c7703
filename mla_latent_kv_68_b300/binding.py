"""ctypes binding of ``libmla.so`` (the C ABI of include/mla.h).

Argument marshalling only: every function checks tensor dtypes, devices and
contiguity, passes raw device pointers and the current CUDA stream, and raises
``MLAError`` for any status other than MLA_OK.  There is no CPU fallback: if
the CUDA library is missing or no GPU is present, the calls fail.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "mla.h")

MLA_OK = 0
MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED, MLA_ERR_WORKSPACE, MLA_ERR_CUDA = 1, 2, 3, 4
MLA_ERR_BAD_SEQLEN, MLA_ERR_TIMEOUT = 5, 6
STATUS_NAMES = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED",
                3: "MLA_ERR_WORKSPACE", 4: "MLA_ERR_CUDA", 5: "MLA_ERR_BAD_SEQLEN",
                6: "MLA_ERR_TIMEOUT"}
POS_EXPLICIT, POS_QUERY, POS_CACHE = 0, 1, 2
D_C, D_R, D_QK, D_H, D_V = 512, 64, 576, 128, 128
SOFTMAX_SCALE = 1.0 / math.sqrt(D_H + D_R)
STATIC_SCRATCH_BYTES = 32 << 20   # MLA_STATIC_SCRATCH_BYTES of include/mla.h
ROPE_BASE = 10000.0


class MLAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")


_lib = None


def lib():
    """Load libmla.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m mla_latent_kv_68_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        L.mla_status_string.restype = ctypes.c_char_p
        L.mla_status_string.argtypes = [i32]
        L.mla_version.restype = i32
        L.mla_absorb_q.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.mla_absorb_rope_q.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, f32, vp]
        L.mla_absorb_rope_q_freq.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp, vp]
        L.mla_rope_apply_freq.argtypes = [vp, i64, i64, vp, i64, i64, i64, i32, i32, vp, i32, vp, vp]
        f64 = ctypes.c_double
        L.mla_rope_yarn_frequencies.argtypes = [f64, f64, f64, f64, f64, vp]
        L.mla_rope_yarn_softmax_scale.argtypes = [f64, vp]
        L.mla_rope_apply.argtypes = [vp, i64, i64, vp, i64, i64, i64, i32, i32, vp, i32, f32, vp]
        L.mla_decode_workspace_size.restype = sz
        L.mla_decode_workspace_size.argtypes = [i32, i32, i32]
        L.mla_decode.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, vp, sz, vp]
        L.mla_splitkv_combine.argtypes = [vp, sz, vp, i32, i32, i32, vp]
        L.mla_up_project.argtypes = [vp, vp, vp, i32, i32, i32, vp]
        L.mla_combine_up_project.argtypes = [vp, sz, vp, vp, i32, i32, i32, vp]
        L.mla_cache_append_workspace_size.restype = sz
        L.mla_cache_append_workspace_size.argtypes = [i32, i32, i32]
        L.mla_cache_append.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, sz, vp]
        L.mla_read_status.argtypes = [vp, vp]
        L.mla_debug_decode_stall.argtypes = [ctypes.c_uint64]
        L.mla_output_project_workspace_size.restype = sz
        L.mla_output_project_workspace_size.argtypes = [i32, i32, i32]
        L.mla_output_project.argtypes = [vp, vp, vp, i32, i32, i32, vp, sz, vp]
        L.mla_decode_noalloc.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, vp, vp]
        L.mla_prefill_expand.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, vp]
        L.mla_prefill_attention.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, vp, vp]
        for n in ("mla_absorb_q", "mla_absorb_rope_q", "mla_absorb_rope_q_freq", "mla_rope_apply",
                  "mla_rope_apply_freq", "mla_rope_yarn_frequencies", "mla_rope_yarn_softmax_scale",
                  "mla_decode",
                  "mla_splitkv_combine", "mla_up_project", "mla_combine_up_project", "mla_read_status",
                  "mla_cache_append", "mla_debug_decode_stall", "mla_output_project",
                  "mla_decode_noalloc", "mla_prefill_expand", "mla_prefill_attention"):
            getattr(L, n).restype = i32
        _lib = L
    return _lib


def header_symbols() -> list[str]:
    """Every function the public header declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", text)))


def _ptr(t: torch.Tensor):
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, what: str):
    if rc != MLA_OK:
        raise MLAError(rc, what)


def _need(t: torch.Tensor, name: str, dtype=torch.bfloat16, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def absorb_q(q_nope, W_UK, q_cat, stream=None):
    """q_cat[..., :512] = W_UK[h]^T q_nope[b,s,h]   (q_nope [B,S,H,128])."""
    B, S, H, _ = q_nope.shape
    _need(q_nope, "q_nope", shape=(B, S, H, D_H))
    _need(W_UK, "W_UK", shape=(H, D_H, D_C))
    _need(q_cat, "q_cat", shape=(B, S, H, D_QK))
    _check(lib().mla_absorb_q(_ptr(q_nope), _ptr(W_UK), _ptr(q_cat), B, S, H, _stream(stream)),
           "mla_absorb_q")


def yarn_frequencies(s=40.0, alpha=1.0, beta=32.0, orig_len=4096.0, base=ROPE_BASE):
    """YaRN RoPE frequencies (32 pairs, float64) from mla_rope_yarn_frequencies;
    the defaults are the pages' long-context setting."""
    out = (ctypes.c_double * 32)()
    _check(lib().mla_rope_yarn_frequencies(base, s, alpha, beta, orig_len, out),
           "mla_rope_yarn_frequencies")
    return [float(v) for v in out]


def yarn_softmax_scale(s=40.0):
    """Softmax scale of the YaRN setting, from mla_rope_yarn_softmax_scale."""
    out = ctypes.c_double()
    _check(lib().mla_rope_yarn_softmax_scale(float(s), ctypes.byref(out)),
           "mla_rope_yarn_softmax_scale")
    return float(out.value)


def _theta_arg(theta):
    if len(theta) != 32:
        raise ValueError("theta must hold 32 frequencies")
    return (ctypes.c_double * 32)(*[float(v) for v in theta])


def absorb_rope_q(q_nope, q_rope, W_UK, seqlens, q_cat, base=ROPE_BASE, theta=None, stream=None):
    """q_cat[..., :512] = W_UK[h]^T q_nope and q_cat[..., 512:] = RoPE(q_rope) at
    positions seqlens[b] - S + s, in one launch (frequencies from `base`, or
    the 32 given in `theta`)."""
    B, S, H, _ = q_nope.shape
    _need(q_nope, "q_nope", shape=(B, S, H, D_H))
    _need(q_rope, "q_rope", shape=(B, S, H, D_R))
    _need(W_UK, "W_UK", shape=(H, D_H, D_C))
    _need(seqlens, "seqlens", dtype=torch.int32, shape=(B,))
    _need(q_cat, "q_cat", shape=(B, S, H, D_QK))
    if theta is None:
        _check(lib().mla_absorb_rope_q(_ptr(q_nope), _ptr(q_rope), _ptr(W_UK), _ptr(seqlens),
                                       _ptr(q_cat), B, S, H, base, _stream(stream)),
               "mla_absorb_rope_q")
    else:
        _check(lib().mla_absorb_rope_q_freq(_ptr(q_nope), _ptr(q_rope), _ptr(W_UK), _ptr(seqlens),
                                            _ptr(q_cat), B, S, H, _theta_arg(theta),
                                            _stream(stream)), "mla_absorb_rope_q_freq")


def rope_apply(x_in, in_stride_n, in_stride_h, x_out, out_stride_n, out_stride_h, N, nh,
               pos_mode, pos_src, group=1, base=ROPE_BASE, stream=None, theta=None):
    """Raw mla_rope_apply (strides in elements); mla_rope_apply_freq when the
    32 frequencies `theta` are given."""
    if x_in.dtype != torch.bfloat16 or x_out.dtype != torch.bfloat16:
        raise TypeError("rope tensors must be bf16")
    _need(pos_src, "pos_src", dtype=torch.int32)
    if theta is None:
        _check(lib().mla_rope_apply(_ptr(x_in), in_stride_n, in_stride_h, _ptr(x_out),
                                    out_stride_n, out_stride_h, N, nh, pos_mode, _ptr(pos_src),
                                    group, base, _stream(stream)), "mla_rope_apply")
    else:
        _check(lib().mla_rope_apply_freq(_ptr(x_in), in_stride_n, in_stride_h, _ptr(x_out),
                                         out_stride_n, out_stride_h, N, nh, pos_mode,
                                         _ptr(pos_src), group, _theta_arg(theta),
                                         _stream(stream)), "mla_rope_apply_freq")


def rope_queries(q_rope, q_cat, seqlens, base=ROPE_BASE, stream=None, theta=None):
    """q_cat[..., 512:] = RoPE(q_rope) at positions seqlens[b] - S + s."""
    B, S, H, _ = q_rope.shape
    _need(q_rope, "q_rope", shape=(B, S, H, D_R))
    _need(q_cat, "q_cat", shape=(B, S, H, D_QK))
    _need(seqlens, "seqlens", dtype=torch.int32, shape=(B,))
    out = q_cat.view(-1)[D_C:]
    rope_apply(q_rope, H * D_R, D_R, out, H * D_QK, D_QK, B * S, H, POS_QUERY, seqlens, S, base,
               stream, theta)


def rope_cache(k_r, seqlens, base=ROPE_BASE, stream=None, theta=None):
    """Rotate the cached k_R [B,Lmax,64] in place at positions 0..seqlens[b]-1."""
    B, Lmax, _ = k_r.shape
    _need(k_r, "k_r", shape=(B, Lmax, D_R))
    _need(seqlens, "seqlens", dtype=torch.int32, shape=(B,))
    rope_apply(k_r, D_R, 0, k_r, D_R, 0, B * Lmax, 1, POS_CACHE, seqlens, Lmax, base, stream,
               theta)


def decode_workspace_size(B: int, S: int, H: int) -> int:
    n = int(lib().mla_decode_workspace_size(B, S, H))
    if n == 0:
        raise MLAError(2, "mla_decode_workspace_size")
    return n


def new_workspace(B: int, S: int, H: int, device=None) -> torch.Tensor:
    """Zero-filled byte workspace for mla_decode / mla_splitkv_combine."""
    return torch.zeros(decode_workspace_size(B, S, H), dtype=torch.uint8, device=device or "cuda")


def cache_append_workspace(B: int, S: int, d: int, device=None) -> torch.Tensor:
    """Zero-filled byte workspace for mla_cache_append."""
    n = lib().mla_cache_append_workspace_size(B, S, d)
    if n == 0:
        raise ValueError(f"unsupported cache-append shape B={B} S={S} d={d}")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def cache_append(h, W_DKV, W_KR, seqlens, c_kv, k_r, workspace, theta=None, stream=None):
    """c_kv[b, t] = W_DKV h[b, s] and k_r[b, t] = RoPE_t(W_KR h[b, s]) at
    t = seqlens[b] - S + s (frequencies base 10000, or the 32 in `theta`)."""
    B, S, d = h.shape
    Lmax = c_kv.shape[1]
    _need(h, "h", shape=(B, S, d))
    _need(W_DKV, "W_DKV", shape=(D_C, d))
    _need(W_KR, "W_KR", shape=(D_R, d))
    _need(seqlens, "seqlens", dtype=torch.int32, shape=(B,))
    _need(c_kv, "c_kv", shape=(B, Lmax, D_C))
    _need(k_r, "k_r", shape=(B, Lmax, D_R))
    _need(workspace, "workspace", dtype=torch.uint8)
    th = None if theta is None else _theta_arg(theta)
    _check(lib().mla_cache_append(_ptr(h), _ptr(W_DKV), _ptr(W_KR), _ptr(seqlens), _ptr(c_kv), _ptr(k_r),
                                  B, S, d, Lmax, th, _ptr(workspace), workspace.numel(), _stream(stream)),
           "mla_cache_append")


def decode(q_cat, c_kv, k_r, seqlens, workspace, softmax_scale=SOFTMAX_SCALE, stream=None):
    B, S, H, _ = q_cat.shape
    Lmax = c_kv.shape[1]
    _need(q_cat, "q_cat", shape=(B, S, H, D_QK))
    _need(c_kv, "c_kv", shape=(B, Lmax, D_C))
    _need(k_r, "k_r", shape=(B, Lmax, D_R))
    _need(seqlens, "seqlens", dtype=torch.int32, shape=(B,))
    _need(workspace, "workspace", dtype=torch.uint8)
    _check(lib().mla_decode(_ptr(q_cat), _ptr(c_kv), _ptr(k_r), _ptr(seqlens), B, S, H, Lmax,
                            softmax_scale, _ptr(workspace), workspace.numel(), _stream(stream)),
           "mla_decode")


def splitkv_combine(workspace, o_lat, stream=None):
    B, S, H, _ = o_lat.shape
    _need(o_lat, "o_lat", shape=(B, S, H, D_C))
    _need(workspace, "workspace", dtype=torch.uint8)
    _check(lib().mla_splitkv_combine(_ptr(workspace), workspace.numel(), _ptr(o_lat), B, S, H,
                                     _stream(stream)), "mla_splitkv_combine")


def up_project(o_lat, W_UV, out, stream=None):
    B, S, H, _ = o_lat.shape
    _need(o_lat, "o_lat", shape=(B, S, H, D_C))
    _need(W_UV, "W_UV", shape=(H, D_V, D_C))
    _need(out, "out", shape=(B, S, H, D_V))
    _check(lib().mla_up_project(_ptr(o_lat), _ptr(W_UV), _ptr(out), B, S, H, _stream(stream)),
           "mla_up_project")


def combine_up_project(workspace, W_UV, out, stream=None):
    """mla_splitkv_combine + mla_up_project in one launch: the merged latent
    rows go straight into the up-projection, o_lat is not stored."""
    B, S, H, _ = out.shape
    _need(out, "out", shape=(B, S, H, D_V))
    _need(W_UV, "W_UV", shape=(H, D_V, D_C))
    _need(workspace, "workspace", dtype=torch.uint8)
    _check(lib().mla_combine_up_project(_ptr(workspace), workspace.numel(), _ptr(W_UV), _ptr(out), B, S, H,
                                        _stream(stream)), "mla_combine_up_project")


def decode_noalloc(q_cat, c_kv, k_r, seqlens, o_lat, softmax_scale=SOFTMAX_SCALE, stream=None):
    """mla_decode + mla_splitkv_combine with the library's own fixed scratch
    array instead of a caller workspace, for callers that cannot allocate
    device memory on their decode path.  Device errors are read with
    ``read_status()`` (no workspace argument)."""
    B, S, H, _ = q_cat.shape
    Lmax = c_kv.shape[1]
    _need(q_cat, "q_cat", shape=(B, S, H, D_QK))
    _need(c_kv, "c_kv", shape=(B, Lmax, D_C))
    _need(k_r, "k_r", shape=(B, Lmax, D_R))
    _need(seqlens, "seqlens", dtype=torch.int32, shape=(B,))
    _need(o_lat, "o_lat", shape=(B, S, H, D_C))
    _check(lib().mla_decode_noalloc(_ptr(q_cat), _ptr(c_kv), _ptr(k_r), _ptr(seqlens), B, S, H,
                                    Lmax, softmax_scale, _ptr(o_lat), _stream(stream)),
           "mla_decode_noalloc")


def debug_decode_stall(wait_limit_ns: int):
    """Test hook: the next decode() call's plan barrier is never completed, so
    its bounded waits run out after wait_limit_ns and it reports
    MLA_ERR_TIMEOUT (see mla_debug_decode_stall)."""
    _check(lib().mla_debug_decode_stall(int(wait_limit_ns)), "mla_debug_decode_stall")


def output_project_workspace(BS: int, K: int, d: int, device=None):
    """Workspace for output_project (None when the shape needs none)."""
    n = int(lib().mla_output_project_workspace_size(BS, K, d))
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda") if n else None


def output_project(x, W, u, workspace=None, stream=None):
    """u[n] = W x[n]: x [BS, K], W [d, K], u [BS, d] (bf16).  With x = out
    [B,S,H,128] viewed as [B*S, H*128] and W = W^O this is the layer's output
    projection; with x = o_lat viewed as [B*S, H*512] and W = W^O blockdiag(W^UV)
    the same projection with the value up-projection folded into W^O."""
    BS, K = x.shape
    d = W.shape[0]
    _need(x, "x", shape=(BS, K))
    _need(W, "W", shape=(d, K))
    _need(u, "u", shape=(BS, d))
    ws, n = ctypes.c_void_p(0), 0
    if workspace is not None:
        _need(workspace, "workspace", dtype=torch.uint8)
        ws, n = _ptr(workspace), workspace.numel()
    _check(lib().mla_output_project(_ptr(x), _ptr(W), _ptr(u), BS, K, d, ws, n, _stream(stream)),
           "mla_output_project")


def rope_prefill_queries(q_rope, q_rot, seqlens, base=ROPE_BASE, stream=None, theta=None):
    """q_rot [B,S,H,64] = RoPE(q_rope) at positions seqlens[b] - S + s."""
    B, S, H, _ = q_rope.shape
    _need(q_rope, "q_rope", shape=(B, S, H, D_R))
    _need(q_rot, "q_rot", shape=(B, S, H, D_R))
    _need(seqlens, "seqlens", dtype=torch.int32, shape=(B,))
    rope_apply(q_rope, H * D_R, D_R, q_rot, H * D_R, D_R, B * S, H, POS_QUERY, seqlens, S, base,
               stream, theta)


def prefill_expand(c_kv, W_UK, W_UV, k_c, v_c, stream=None):
    """k_c / v_c [B,Lmax,H,128] = W_UK[h] c_t / W_UV[h] c_t for every cache row."""
    B, Lmax, _ = c_kv.shape
    H = W_UK.shape[0]
    _need(c_kv, "c_kv", shape=(B, Lmax, D_C))
    _need(W_UK, "W_UK", shape=(H, D_H, D_C))
    _need(W_UV, "W_UV", shape=(H, D_V, D_C))
    _need(k_c, "k_c", shape=(B, Lmax, H, D_H))
    _need(v_c, "v_c", shape=(B, Lmax, H, D_V))
    _check(lib().mla_prefill_expand(_ptr(c_kv), _ptr(W_UK), _ptr(W_UV), _ptr(k_c), _ptr(v_c), B, Lmax, H,
                                    _stream(stream)), "mla_prefill_expand")


def prefill_attention(q_nope, q_rot, k_c, k_r, v_c, seqlens, out, softmax_scale=SOFTMAX_SCALE, stream=None):
    """Causal attention of the S queries per sequence over the expanded keys
    and values: out [B,S,H,128].  q_rot is the rotated q^R (rope_prefill_queries)."""
    B, S, H, _ = q_nope.shape
    Lmax = k_r.shape[1]
    _need(q_nope, "q_nope", shape=(B, S, H, D_H))
    _need(q_rot, "q_rot", shape=(B, S, H, D_R))
    _need(k_c, "k_c", shape=(B, Lmax, H, D_H))
    _need(k_r, "k_r", shape=(B, Lmax, D_R))
    _need(v_c, "v_c", shape=(B, Lmax, H, D_V))
    _need(seqlens, "seqlens", dtype=torch.int32, shape=(B,))
    _need(out, "out", shape=(B, S, H, D_V))
    _check(lib().mla_prefill_attention(_ptr(q_nope), _ptr(q_rot), _ptr(k_c), _ptr(k_r), _ptr(v_c), _ptr(seqlens),
                                       B, S, H, Lmax, softmax_scale, _ptr(out), _stream(stream)),
           "mla_prefill_attention")


class PrefillStep:
    """Buffers and calls of one prefill shape: RoPE of the queries, expansion
    of the cached keys and values per head, causal attention."""

    def __init__(self, B: int, S: int, H: int, Lmax: int, device="cuda"):
        self.B, self.S, self.H, self.Lmax = B, S, H, Lmax
        bf = torch.bfloat16
        self.q_rot = torch.empty(B, S, H, D_R, dtype=bf, device=device)
        self.k_c = torch.empty(B, Lmax, H, D_H, dtype=bf, device=device)
        self.v_c = torch.empty(B, Lmax, H, D_V, dtype=bf, device=device)
        self.out = torch.empty(B, S, H, D_V, dtype=bf, device=device)

    def __call__(self, q_nope, q_rope, c_kv, k_r, seqlens, W_UK, W_UV, softmax_scale=SOFTMAX_SCALE,
                 theta=None, stream=None):
        rope_prefill_queries(q_rope, self.q_rot, seqlens, stream=stream, theta=theta)
        prefill_expand(c_kv, W_UK, W_UV, self.k_c, self.v_c, stream=stream)
        prefill_attention(q_nope, self.q_rot, self.k_c, k_r, self.v_c, seqlens, self.out, softmax_scale, stream)
        return self.out


def read_status(workspace=None, stream=None) -> int:
    """Synchronise and return (and clear) the device-side status."""
    ws = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    return int(lib().mla_read_status(ws, _stream(stream)))


class DecodeStep:
    """Owns the per-step device buffers of one decode shape and issues the
    four library calls of a step on one stream:
    absorb + RoPE(queries) -> decode -> combine -> up-project."""

    def __init__(self, B: int, S: int, H: int, device="cuda", rope_theta=None,
                 softmax_scale=SOFTMAX_SCALE):
        """rope_theta: 32 RoPE frequencies for the queries (e.g. yarn_frequencies());
        None for base 10000.  The cache's k_R must be rotated with the same ones.
        softmax_scale: the score scale used when a call passes none."""
        self.B, self.S, self.H = B, S, H
        self.rope_theta = rope_theta
        self.softmax_scale = softmax_scale
        self.q_cat = torch.empty(B, S, H, D_QK, dtype=torch.bfloat16, device=device)
        self.o_lat = torch.empty(B, S, H, D_C, dtype=torch.bfloat16, device=device)
        self.out = torch.empty(B, S, H, D_V, dtype=torch.bfloat16, device=device)
        self.workspace = new_workspace(B, S, H, device)

    def __call__(self, q_nope, q_rope, c_kv, k_r, seqlens, W_UK, W_UV,
                 softmax_scale=None, stream=None):
        self.queries(q_nope, q_rope, seqlens, W_UK, stream)
        self.attend(c_kv, k_r, seqlens, softmax_scale, stream)
        self.project(W_UV, stream)
        return self.out

    # The three phases of a step, separately callable for per-phase timing.
    def queries(self, q_nope, q_rope, seqlens, W_UK, stream=None):
        absorb_rope_q(q_nope, q_rope, W_UK, seqlens, self.q_cat, theta=self.rope_theta,
                      stream=stream)

    def attend(self, c_kv, k_r, seqlens, softmax_scale=None, stream=None):
        scale = self.softmax_scale if softmax_scale is None else softmax_scale
        decode(self.q_cat, c_kv, k_r, seqlens, self.workspace, scale, stream)

    def project(self, W_UV, stream=None):
        # two launches: measured faster inside the pipelined step than the
        # fused combine_up_project (the small combine CTAs start beside the
        # decode's last clusters)
        splitkv_combine(self.workspace, self.o_lat, stream)
        up_project(self.o_lat, W_UV, self.out, stream)

    def capture(self, fn, *args, **kwargs):
        """Record ``fn(*args)`` (library calls only) into a CUDA graph and
        return it; ``graph.replay()`` re-issues the same launches on the
        current stream with no host work per kernel.  The graph reads the
        same device buffers on every replay, so new query or length values
        copied into them take effect."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(*args, **kwargs)
        return g

    LAUNCHES_PER_STEP = 4  # absorb + rope, decode (plans its own split), combine, up-projection
