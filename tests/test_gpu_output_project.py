"""GPU parity of the output projection (mla_output_project) against the oracle.

u_t = W^O [o_{t,1}; ...; o_{t,H}] ("DeepSeek-V3" (ekkoxiao.github.io),
"注意力计算"), and the same projection with W^UV folded into W^O
("DeepSeek-V3 技术报告精读" (oopvo.github.io), "MLA").  The expected values come
from the oracle on the same bf16 inputs (the folded weight is formed by the
oracle in fp64 and rounded to bf16 for both sides).  Shapes cover one slice
and many, token counts that are not a multiple of the 16-row MMA step or of
the 64-token tile, and the full-size layer (32 tokens, 128 heads, d = 7168).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close, bits, f64
from mla_latent_kv_68_b300 import binding as mb

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


def _run(x, W):
    BS, K = x.shape
    d = W.shape[0]
    u = torch.full((BS, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    mb.output_project(x.cuda(), W.cuda(), u, mb.output_project_workspace(BS, K, d))
    assert mb.read_status() == mb.MLA_OK
    return f64(u)


@pytest.mark.parametrize("BS,K,d", [(1, 128, 128), (5, 384, 256), (33, 1024, 640), (64, 2048, 384),
                                    (100, 512, 128), (32, 128 * 128, 7168)])
def test_output_project_matches_oracle(BS, K, d):
    g = torch.Generator().manual_seed(BS * 7 + K + d)
    x = torch.randn(BS, K, generator=g).to(torch.bfloat16)
    W = (torch.randn(d, K, generator=g) / math.sqrt(K)).to(torch.bfloat16)
    got = _run(x, W)
    ref = oracle.output_project(bits(x), bits(W))
    assert_close(got, ref, what=f"u BS{BS} K{K} d{d}")


def test_folded_output_projection_matches_the_unfolded_chain():
    # x = o_lat of 8 tokens and 16 heads, W = W^O blockdiag(W^UV) (from the
    # oracle, rounded to bf16): the GPU result against the oracle's chain
    # W^O [W_1^UV o_lat_1; ...] on the same bf16 o_lat
    g = torch.Generator().manual_seed(99)
    N, H, d = 8, 16, 1024
    o_lat = (0.05 * torch.randn(N, H, 512, generator=g)).to(torch.bfloat16)
    W_UV = (torch.randn(H, 128, 512, generator=g) / math.sqrt(512)).to(torch.bfloat16)
    W_O = (torch.randn(d, H * 128, generator=g) / math.sqrt(H * 128)).to(torch.bfloat16)
    W_fold = torch.from_numpy(oracle.fold_output_weights(bits(W_O), bits(W_UV)).astype(np.float32)).to(torch.bfloat16)
    got = _run(o_lat.reshape(N, H * 512), W_fold)
    heads = oracle.up_project(bits(o_lat), bits(W_UV))
    ref = oracle.output_project(heads.reshape(N, H * 128), bits(W_O))
    scale = float(np.abs(ref).max())
    # the folded weight itself is rounded to bf16 once: compare relative to the output scale
    assert_close(got / scale, ref / scale, what="folded output projection")
