"""Shared helpers of the GPU parity tests (no method arithmetic here)."""
import numpy as np
import torch

from mla_latent_kv_68_b300.inputs import bf16_bits

# Tolerances fixed for the end-to-end output (bf16 inputs, fp32 accumulation):
MAX_ABS = 2e-2
REL_L2 = 5e-3


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.linalg.norm(ref))
    return float(np.linalg.norm(got - ref)) / (den if den > 0 else 1.0)


def assert_close(got, ref, max_abs=MAX_ABS, rel=REL_L2, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    r = rel_l2(got, ref)
    assert err <= max_abs and r <= rel, f"{what}: max-abs {err:.3e} rel-L2 {r:.3e}"
    return err, r


def bits(t: torch.Tensor):
    return bf16_bits(t.detach().cpu())


def to_dev(x: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()
