"""The library's YaRN frequencies (host arithmetic in the C ABI, no GPU) against
the oracle's, and their argument checks."""
import ctypes
import math

import numpy as np
import pytest

import oracle
from mla_latent_kv_68_b300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


@pytest.mark.parametrize("s,alpha,beta,L", [(40.0, 1.0, 32.0, 4096.0), (1.0, 1.0, 32.0, 4096.0),
                                            (8.0, 2.0, 16.0, 32768.0)])
def test_library_yarn_frequencies_match_oracle(lib, s, alpha, beta, L):
    got = np.array(binding.yarn_frequencies(s, alpha, beta, L))
    ref = oracle.yarn_theta(64, s=s, alpha=alpha, beta=beta, orig_len=L)
    np.testing.assert_allclose(got, ref, rtol=1e-14)


def test_yarn_frequencies_reject_bad_arguments(lib):
    out = (ctypes.c_double * 32)()
    assert lib.mla_rope_yarn_frequencies(10000.0, 0.5, 1.0, 32.0, 4096.0, out) == 1  # s < 1
    assert lib.mla_rope_yarn_frequencies(10000.0, 40.0, 32.0, 1.0, 4096.0, out) == 1  # beta <= alpha
    assert lib.mla_rope_yarn_frequencies(10000.0, 40.0, 1.0, 32.0, 0.0, out) == 1
    assert lib.mla_rope_yarn_frequencies(10000.0, 40.0, 1.0, 32.0, 4096.0, None) == 1


@pytest.mark.parametrize("s", [1.0, 2.0, 40.0, 1e6])
def test_library_yarn_softmax_scale_matches_oracle(lib, s):
    assert binding.yarn_softmax_scale(s) == pytest.approx(oracle.yarn_softmax_scale(s), rel=1e-15)


def test_yarn_softmax_scale_rejects_bad_arguments(lib):
    out = ctypes.c_double(-1.0)
    for s in (0.5, float("nan"), float("inf")):
        assert lib.mla_rope_yarn_softmax_scale(s, ctypes.byref(out)) == 1
    assert out.value == -1.0
    assert lib.mla_rope_yarn_softmax_scale(40.0, None) == 1


def test_freq_entries_reject_bad_frequencies(lib):
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: validation fails first
    bad = (ctypes.c_double * 32)(*([1.0] * 31 + [float("nan")]))
    assert lib.mla_rope_apply_freq(fake, 64, 0, fake, 64, 0, 1, 1, 0, fake, 1, bad, None) == 1
    assert lib.mla_absorb_rope_q_freq(fake, fake, fake, fake, fake, 1, 1, 1, bad, None) == 1
    assert lib.mla_rope_apply_freq(fake, 64, 0, fake, 64, 0, 1, 1, 0, fake, 1, None, None) == 1
