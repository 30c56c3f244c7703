"""The C-ABI library loads and exports every symbol the header declares, and
host-side validation rejects bad arguments before any launch (no GPU needed)."""
import ctypes
import shutil

import pytest

from mla_latent_kv_68_b300 import binding, build


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") or __import__("os").path.exists("/usr/local/cuda/bin/nvcc"):
        build.build()
    return binding.lib()


def test_header_declares_the_five_steps():
    syms = binding.header_symbols()
    for name in ("mla_absorb_q", "mla_rope_apply", "mla_decode", "mla_splitkv_combine",
                 "mla_up_project"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    for name in binding.header_symbols():
        assert hasattr(lib, name), f"{name} not exported by libmla.so"


def test_status_strings_and_version(lib):
    for code, name in binding.STATUS_NAMES.items():
        assert lib.mla_status_string(code).decode() == name
    assert lib.mla_status_string(99).decode() == "MLA_ERR_UNKNOWN"
    assert lib.mla_version() >= 100


def test_null_pointers_rejected_on_host(lib):
    nul = ctypes.c_void_p(0)
    assert lib.mla_absorb_q(nul, nul, nul, 1, 1, 1, nul) == 1
    assert lib.mla_up_project(nul, nul, nul, 1, 1, 1, nul) == 1
    assert lib.mla_decode(nul, nul, nul, nul, 1, 1, 1, 1, 0.1, nul, 0, nul) == 1
    assert lib.mla_splitkv_combine(nul, 0, nul, 1, 1, 1, nul) == 1
    assert lib.mla_rope_apply(nul, 64, 0, nul, 64, 0, 1, 1, 0, nul, 1, 10000.0, nul) == 1


def test_bad_sizes_rejected_on_host(lib):
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: validation fails first
    assert lib.mla_absorb_q(fake, fake, fake, 0, 1, 1, None) == 1
    assert lib.mla_absorb_q(fake, fake, fake, 1, 1, 129, None) == 2
    assert lib.mla_up_project(fake, fake, fake, 1, 1, 200, None) == 2
    assert lib.mla_rope_apply(fake, 63, 0, fake, 64, 0, 1, 1, 0, fake, 1, 10000.0, None) == 1
    assert lib.mla_rope_apply(fake, 64, 0, fake, 64, 0, 1, 1, 7, fake, 1, 10000.0, None) == 1
    assert lib.mla_decode(fake, fake, fake, fake, 1, 1, 1, 1, -1.0, fake, 0, None) == 1
    misaligned = ctypes.c_void_p((1 << 20) + 8)
    assert lib.mla_absorb_q(misaligned, fake, fake, 1, 1, 1, None) == 1


def test_static_scratch_limit_matches_the_header():
    import re
    with open(binding.HEADER_PATH) as f:
        m = re.search(r"MLA_STATIC_SCRATCH_BYTES\s*=\s*(\d+)\s*<<\s*(\d+)", f.read())
    assert m and int(m.group(1)) << int(m.group(2)) == binding.STATIC_SCRATCH_BYTES


def test_cache_append_host_validation(lib):
    nul, fake = ctypes.c_void_p(0), ctypes.c_void_p(1 << 20)  # fake: aligned, never dereferenced
    big = 1 << 30
    assert lib.mla_cache_append(nul, fake, fake, fake, fake, fake, 1, 1, 64, 4, None, fake, big, None) == 1
    assert lib.mla_cache_append(fake, fake, fake, fake, fake, fake, 0, 1, 64, 4, None, fake, big, None) == 1
    assert lib.mla_cache_append(fake, fake, fake, fake, fake, fake, 1, 2, 64, 1, None, fake, big, None) == 1
    assert lib.mla_cache_append(fake, fake, fake, fake, fake, fake, 1, 1, 100, 4, None, fake, big, None) == 2
    assert lib.mla_cache_append(fake, fake, fake, fake, fake, fake, 1, 1, 64, 4, None, fake, 16, None) == 3
    assert lib.mla_cache_append(fake, fake, fake, fake, fake, fake, 1, 1, 64, 4, None,
                                ctypes.c_void_p((1 << 20) + 64), big, None) == 3   # not 256-byte aligned
    misaligned = ctypes.c_void_p((1 << 20) + 8)
    assert lib.mla_cache_append(misaligned, fake, fake, fake, fake, fake, 1, 1, 64, 4, None, fake, big,
                                None) == 1


def test_cache_append_workspace_size(lib):
    assert lib.mla_cache_append_workspace_size(1, 1, 100) == 0     # d not a multiple of 64
    assert lib.mla_cache_append_workspace_size(0, 1, 64) == 0
    # status word, then fp32 partial products [ceil(d / 256)][B * S][576], 256-byte rounded
    n = 4 * 28 * 32 * 576
    assert lib.mla_cache_append_workspace_size(32, 1, 7168) == 256 + (n + 255) // 256 * 256
    assert lib.mla_cache_append_workspace_size(3, 2, 448) == 256 + (4 * 2 * 6 * 576 + 255) // 256 * 256


def test_combine_up_project_host_validation(lib):
    nul, fake = ctypes.c_void_p(0), ctypes.c_void_p(1 << 20)
    assert lib.mla_combine_up_project(fake, 1 << 30, nul, fake, 1, 1, 1, None) == 1
    assert lib.mla_combine_up_project(fake, 1 << 30, fake, fake, 0, 1, 1, None) == 1
    assert lib.mla_combine_up_project(fake, 1 << 30, fake, fake, 1, 1, 200, None) == 2
    assert lib.mla_combine_up_project(fake, 1 << 30, fake, fake, 1, 17, 128, None) == 2  # S*H > 2048
    assert lib.mla_combine_up_project(nul, 1 << 30, fake, fake, 1, 1, 16, None) == 3


def test_decode_stall_hook_rejects_bad_limits(lib):
    assert lib.mla_debug_decode_stall(ctypes.c_uint64(0)) == 1            # MLA_ERR_INVALID_ARG
    assert lib.mla_debug_decode_stall(ctypes.c_uint64(2_000_000_000)) == 1


def test_prefill_host_validation(lib):
    nul, fake, odd = ctypes.c_void_p(0), ctypes.c_void_p(1 << 20), ctypes.c_void_p((1 << 20) + 2)
    # expansion: null / misaligned pointers, bad sizes, more than 128 heads
    assert lib.mla_prefill_expand(nul, fake, fake, fake, fake, 1, 1, 1, None) == 1
    assert lib.mla_prefill_expand(fake, fake, odd, fake, fake, 1, 1, 1, None) == 1
    assert lib.mla_prefill_expand(fake, fake, fake, fake, fake, 1, 0, 1, None) == 1
    assert lib.mla_prefill_expand(fake, fake, fake, fake, fake, 1, 1, 129, None) == 2
    # attention: nulls, S > Lmax, a non-positive scale, more than 128 heads
    args = [fake] * 6
    assert lib.mla_prefill_attention(nul, *args[1:], 1, 1, 1, 1, 0.1, fake, None) == 1
    assert lib.mla_prefill_attention(*args, 1, 5, 1, 4, 0.1, fake, None) == 1
    assert lib.mla_prefill_attention(*args, 1, 1, 1, 1, 0.0, fake, None) == 1
    assert lib.mla_prefill_attention(*args, 1, 1, 1, 1, 0.1, odd, None) == 1
    assert lib.mla_prefill_attention(*args, 1, 1, 129, 1, 0.1, fake, None) == 2
