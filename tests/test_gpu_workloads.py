"""Parity at the five full-size decode workloads, in the launch configuration
the benchmark times.  The whole step runs on the GPU; the fp64 unabsorbed
oracle recomputes a sample of output rows one by one (first/last sequence,
first/last head, both query positions, the longest and shortest sequences)."""
import numpy as np
import pytest
import torch

from gpu_util import assert_close
from mla_latent_kv_68_b300.inputs import WORKLOADS, workload_inputs

from test_gpu_parity import _oracle_rows, _step

pytestmark = pytest.mark.gpu

SAMPLES = {
    "tiny_b1_s1_h16_l256": None,                # every row
    "uniform_b32_s1_h128_l4096": 32,
    "varlen_b64_s1_h128_l1to32768": 24,
    "mtp_b16_s2_h128_l16384": 16,
    "long_b4_s1_h128_l131072": 8,
}


def _sample_rows(x, n, seed):
    B, S, H = x["B"], x["S"], x["H"]
    L = x["seqlens"].numpy()
    rng = np.random.default_rng(seed)
    bs = {0, B - 1, int(np.argmax(L)), int(np.argmin(L))}
    while len(bs) < min(B, max(2, n // (2 * S))):
        bs.add(int(rng.integers(0, B)))
    rows = set()
    for b in sorted(bs):
        for s in range(S):
            for h in (0, H - 1, int(rng.integers(0, H))):
                rows.add((b * S + s) * H + h)
    rows = sorted(rows)
    if len(rows) > n:
        keep = set(rng.choice(len(rows), n, replace=False).tolist())
        rows = [r for i, r in enumerate(rows) if i in keep]
    return np.array(rows, np.int64)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_sampled_rows_match_oracle(name):
    x = workload_inputs(name)
    got = _step(x).reshape(-1, 128)
    n = SAMPLES[name]
    if n is None:
        rows = np.arange(x["B"] * x["S"] * x["H"])
    else:
        rows = _sample_rows(x, n, seed=WORKLOADS[name].seed)
    ref = _oracle_rows(x, rows=rows)
    assert_close(got[rows], ref, what=name)
    assert np.isfinite(got).all()
    torch.cuda.empty_cache()
