"""GPU parity of attention_backward (fp32, CUDA cores) against the oracle's
backward of Algorithm 0 (itself pinned by finite differences).

The forward output `out` handed to the backward is the oracle's, rounded to
fp32, so that the comparison isolates the backward.  Shapes cover T = 1,
ragged tails of the 64-row tiles, head sizes 16, 32 and 64, and the GPT-2
width at T = 1024; inputs at the workload's scale and with peaked scores.
Tolerance: fp32 arithmetic with sums of at most T products per element:
|err| <= 1e-5 x max(1, max |ref|) (about 2^-17 relative to the largest
gradient)."""
import numpy as np
import pytest
import torch

import oracle
from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs

from gpu_helpers import assert_close, dev, host, need_gpu, no_device_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def run_backward(B, T, C, NH, seed, qk_std=1.0, std=0.55):
    qkv = inputs.make_normal(500 + seed, (B, T, 3 * C), std)
    qkv[..., :2 * C] *= qk_std
    qkv = qkv.astype(np.float32).astype(np.float64)
    dout = inputs.make_normal(600 + seed, (B, T, C), 1.0).astype(np.float32).astype(np.float64)
    out = oracle.attention(qkv, NH).astype(np.float32)
    dq = torch.full((B, T, 3 * C), float("nan"), dtype=torch.float32, device="cuda")
    wsz = ab.attention_backward_workspace_size(B, T, C, NH, ab.GPT2_FP32)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    ab.attention_backward(dq, dev(dout, torch.float32), dev(qkv, torch.float32), dev(out), B, T, C, NH, ab.GPT2_FP32, ws, wsz)
    no_device_error()
    return host(dq), oracle.attention_backward(qkv, dout, NH)


SHAPES = [(1, 1, 128, 2), (2, 64, 128, 2), (1, 65, 128, 2), (2, 129, 64, 4), (1, 130, 256, 8), (3, 97, 192, 12),
          (2, 200, 768, 12), (1, 1024, 768, 12)]


@pytest.mark.parametrize("B,T,C,NH", SHAPES)
def test_attention_backward(B, T, C, NH):
    got, ref = run_backward(B, T, C, NH, seed=B * 1000 + T)
    assert_close(got, ref, atol=1e-5 * max(1.0, np.abs(ref).max()), what=f"dqkv {B}x{T}x{C}/{NH}")


def test_attention_backward_peaked_scores():
    got, ref = run_backward(1, 300, 768, 12, seed=7, qk_std=3.0, std=1.0)
    assert_close(got, ref, atol=1e-5 * max(1.0, np.abs(ref).max()), what="peaked dqkv")


def test_attention_backward_after_the_gpu_forward():
    # the chain a training step runs: GPU forward (fp32), then backward
    B, T, C, NH = 2, 150, 256, 4
    qkv = inputs.make_normal(701, (B, T, 3 * C), 0.55).astype(np.float32)
    dout = inputs.make_normal(702, (B, T, C), 1.0).astype(np.float32)
    out = torch.empty((B, T, C), dtype=torch.float32, device="cuda")
    ab.attention_forward(out, dev(qkv), B, T, C, NH, ab.GPT2_FP32, None, 0)
    dq = torch.empty((B, T, 3 * C), dtype=torch.float32, device="cuda")
    wsz = ab.attention_backward_workspace_size(B, T, C, NH, ab.GPT2_FP32)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    ab.attention_backward(dq, dev(dout), dev(qkv), out, B, T, C, NH, ab.GPT2_FP32, ws, wsz)
    no_device_error()
    ref = oracle.attention_backward(qkv, dout, NH)
    assert_close(host(dq), ref, atol=1e-5 * max(1.0, np.abs(ref).max()), what="forward then backward")


def test_attention_backward_is_deterministic():
    B, T, C, NH = 2, 333, 768, 12
    qkv = dev(inputs.make_normal(703, (B, T, 3 * C), 0.55), torch.float32)
    dout = dev(inputs.make_normal(704, (B, T, C), 1.0), torch.float32)
    out = torch.empty((B, T, C), dtype=torch.float32, device="cuda")
    ab.attention_forward(out, qkv, B, T, C, NH, ab.GPT2_FP32, None, 0)
    wsz = ab.attention_backward_workspace_size(B, T, C, NH, ab.GPT2_FP32)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    res = []
    for _ in range(2):
        dq = torch.empty((B, T, 3 * C), dtype=torch.float32, device="cuda")
        ab.attention_backward(dq, dout, qkv, out, B, T, C, NH, ab.GPT2_FP32, ws, wsz)
        res.append(host(dq))
    np.testing.assert_array_equal(res[0], res[1])
