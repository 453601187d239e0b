"""GPU parity of attention_forward against the oracle's Algorithm 0.

Shapes cover T = 1, T below, at and past one 64-row tile, ragged tails,
the GPT-2 width (12 heads of 64) at T = 1024, and head sizes 16, 32 and 64.
Tolerances: fp32 CUDA cores 1e-5 absolute (outputs are convex combinations
of O(1) values); bf16 tensor cores 2e-2 absolute."""
import numpy as np
import pytest
import torch

import oracle
from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs

from gpu_helpers import assert_close, dev, host, need_gpu, no_device_error

pytestmark = pytest.mark.gpu
TOL = {ab.GPT2_BF16: 2e-2, ab.GPT2_TF32: 2e-2, ab.GPT2_FP32: 1e-5}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def run_attention(B, T, C, NH, precision, seed=0, qk_std=1.0):
    qkv = inputs.make_normal(400 + seed, (B, T, 3 * C), 1.0)
    qkv[..., :2 * C] *= qk_std
    out = torch.full((B, T, C), float("nan"), device="cuda")
    wsz = ab.attention_workspace_size(B, T, C, precision)
    ws = torch.empty(max(wsz, 1), dtype=torch.uint8, device="cuda")
    ab.attention_forward(out, dev(qkv), B, T, C, NH, precision, ws, wsz)
    no_device_error()
    return host(out), oracle.attention(qkv, NH)


SHAPES = [(1, 1, 64, 4), (2, 32, 64, 4), (1, 64, 128, 2), (2, 65, 128, 4), (1, 200, 768, 12),
          (1, 130, 256, 8), (2, 1024, 768, 12), (3, 97, 192, 12)]


@pytest.mark.parametrize("precision", [ab.GPT2_BF16, ab.GPT2_FP32])
@pytest.mark.parametrize("B,T,C,NH", SHAPES)
def test_attention(B, T, C, NH, precision):
    got, ref = run_attention(B, T, C, NH, precision)
    assert_close(got, ref, atol=TOL[precision], what=f"attention {B}x{T}x{C}/{NH} p{precision}")


@pytest.mark.parametrize("precision", [ab.GPT2_BF16, ab.GPT2_FP32])
def test_attention_peaked_scores(precision):
    # large scores: a few keys dominate each row, exercising the running max
    got, ref = run_attention(1, 300, 768, 12, precision, seed=3, qk_std=3.0)
    assert_close(got, ref, atol=TOL[precision], what="peaked")


def test_attention_causal_bitwise():
    B, T, C, NH = 1, 150, 768, 12
    qkv = inputs.make_normal(9, (B, T, 3 * C))
    ws = torch.empty(ab.attention_workspace_size(B, T, C, ab.GPT2_BF16), dtype=torch.uint8, device="cuda")
    outs = []
    for q in (qkv, np.concatenate([qkv[:, :100], inputs.make_normal(10, (B, T - 100, 3 * C))], axis=1)):
        o = torch.empty(B, T, C, device="cuda")
        ab.attention_forward(o, dev(q), B, T, C, NH, ab.GPT2_BF16, ws, ws.numel())
        outs.append(host(o))
    np.testing.assert_array_equal(outs[0][:, :100], outs[1][:, :100])
