"""Seeded synthetic inputs for MLA decode.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no RoPE, no projection, no softmax), so both the CUDA
path and the CPU oracle can take their inputs from it.

Recipe (all draws on the CPU with one ``torch.Generator``, in this order, each
drawn in fp32 and rounded to bf16 with round-to-nearest-even):
  1. seqlens (only when drawn: uniform integers in [lo, hi])
  2. c_KV  ~ N(0, 1) * c_scale, per sequence, rows 0..L_b-1
  3. k_R   ~ N(0, 1), pre-RoPE, per sequence, rows 0..L_b-1
  4. q_nope ~ N(0, 1)          [B,S,H,128]
  5. q_rope ~ N(0, 1)          [B,S,H,64], pre-RoPE
  6. W_UK  ~ N(0, 1/512)       [H,128,512]
  7. W_UV  ~ N(0, 1/512)       [H,128,512]
Cache rows L_b..Lmax-1 of each sequence are padding, filled with ``pad``
(0 by default; tests also use NaN to prove the padding is never read into a
result).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch

D_C = 512   # kv_lora_rank (latent width)
D_R = 64    # qk_rope_head_dim
D_H = 128   # qk_nope_head_dim
D_V = 128   # v_head_dim


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    S: int
    H: int
    L: int | None          # fixed length, or None when drawn
    L_range: tuple | None  # (lo, hi) inclusive, when drawn
    c_scale: float
    seed: int

    @property
    def Lmax(self) -> int:
        return self.L if self.L is not None else self.L_range[1]


# The five decode workloads, keyed by a descriptive name.
WORKLOADS = {
    "tiny_b1_s1_h16_l256": Workload("tiny_b1_s1_h16_l256", 1, 1, 16, 256, None, 1.0, 68000),
    "uniform_b32_s1_h128_l4096": Workload("uniform_b32_s1_h128_l4096", 32, 1, 128, 4096, None,
                                          1.0, 68001),
    "varlen_b64_s1_h128_l1to32768": Workload("varlen_b64_s1_h128_l1to32768", 64, 1, 128, None,
                                             (1, 32768), 1.0, 68002),
    "mtp_b16_s2_h128_l16384": Workload("mtp_b16_s2_h128_l16384", 16, 2, 128, 16384, None, 1.0,
                                       68003),
    "long_b4_s1_h128_l131072": Workload("long_b4_s1_h128_l131072", 4, 1, 128, 131072, None, 0.5,
                                        68004),
}
WORKLOAD_ORDER = list(WORKLOADS)


def _randn_bf16(gen, shape, scale=1.0):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x.to(torch.bfloat16)


def make_inputs(B: int, S: int, H: int, seqlens=None, *, Lmax: int | None = None,
                L_range: tuple | None = None, seed: int = 0, c_scale: float = 1.0,
                pad: float = 0.0, w_std: float | None = None) -> dict:
    """Draw one decode problem.  Returns CPU tensors:
    seqlens int32[B]; c_kv, k_r [B,Lmax,512|64] bf16 (k_r pre-RoPE);
    q_nope [B,S,H,128], q_rope [B,S,H,64] (pre-RoPE), W_UK, W_UV [H,128,512] bf16."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    if seqlens is None:
        lo, hi = L_range
        seqlens = torch.randint(lo, hi + 1, (B,), generator=gen, dtype=torch.int64)
    seqlens = torch.as_tensor(seqlens, dtype=torch.int64).reshape(B)
    if Lmax is None:
        Lmax = int(seqlens.max())
    c_kv = torch.full((B, Lmax, D_C), pad, dtype=torch.bfloat16)
    k_r = torch.full((B, Lmax, D_R), pad, dtype=torch.bfloat16)
    for b in range(B):
        L = int(seqlens[b])
        c_kv[b, :L] = _randn_bf16(gen, (L, D_C), c_scale)
    for b in range(B):
        L = int(seqlens[b])
        k_r[b, :L] = _randn_bf16(gen, (L, D_R))
    q_nope = _randn_bf16(gen, (B, S, H, D_H))
    q_rope = _randn_bf16(gen, (B, S, H, D_R))
    std = (1.0 / math.sqrt(D_C)) if w_std is None else w_std
    W_UK = _randn_bf16(gen, (H, D_H, D_C), std)
    W_UV = _randn_bf16(gen, (H, D_V, D_C), std)
    return dict(seqlens=seqlens.to(torch.int32), c_kv=c_kv, k_r=k_r, q_nope=q_nope,
                q_rope=q_rope, W_UK=W_UK, W_UV=W_UV, B=B, S=S, H=H, Lmax=Lmax)


def workload_inputs(name: str, pad: float = 0.0) -> dict:
    w = WORKLOADS[name]
    if w.L is not None:
        return make_inputs(w.B, w.S, w.H, [w.L] * w.B, Lmax=w.L, seed=w.seed,
                           c_scale=w.c_scale, pad=pad)
    return make_inputs(w.B, w.S, w.H, None, Lmax=w.Lmax, L_range=w.L_range, seed=w.seed,
                       c_scale=w.c_scale, pad=pad)


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a CPU bf16 tensor as a uint16 numpy array."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view("uint16")
