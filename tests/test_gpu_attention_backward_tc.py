"""GPU parity of attention_backward's tensor-core path (GPT2_BF16 and
GPT2_TF32: tcgen05, head size 64, bf16 operands, fp32 accumulation)
against the oracle's backward of Algorithm 0 (pinned by finite
differences).

Shapes cover T below, at and just past the 128-row tiles, ragged
tails, the GPT-2 width at T = 1024, and the full B=16 T=1024 launch (two
sequences compared).  Tolerance, from the arithmetic: Q, K, V, dout, P and
dS are each rounded once to bf16 (unit roundoff u = 2^-8); every product is
accumulated in fp32.  The rounding of Q and K moves each score by a few u
times |q||k| / 8, P by that relative amount, and dS = P (dP - D) inherits
the relative errors of P and of dP (dout and V rounded); each gradient
element is a sum of such terms.  The bound is per column block (dq, dk,
dv): |err| <= TOL x the block's largest |ref|, TOL = 2e-2 (about 5u).
T = 1 (dq = dk = 0 exactly) has its own bound from the same rounding."""
import numpy as np
import pytest
import torch

import oracle
from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs

from gpu_helpers import dev, host, need_gpu, no_device_error

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def make_inputs(B, T, C, seed, qk_std=1.0, std=0.55):
    qkv = inputs.make_normal(800 + seed, (B, T, 3 * C), std)
    qkv[..., :2 * C] *= qk_std
    qkv = qkv.astype(np.float32).astype(np.float64)
    dout = inputs.make_normal(900 + seed, (B, T, C), 1.0).astype(np.float32).astype(np.float64)
    return qkv, dout


def gpu_backward(qkv, dout, out, NH, precision=ab.GPT2_BF16):
    B, T, C3 = qkv.shape
    C = C3 // 3
    dq = torch.full((B, T, 3 * C), float("nan"), dtype=torch.float32, device="cuda")
    wsz = ab.attention_backward_workspace_size(B, T, C, NH, precision)
    assert wsz > 0
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    ab.attention_backward(dq, dev(dout, torch.float32), dev(qkv, torch.float32), dev(out, torch.float32), B, T, C, NH,
                          precision, ws, wsz)
    no_device_error()
    return host(dq)


def check_blocks(got, ref, C, what):
    assert np.isfinite(got).all(), what
    for name, k in (("dq", 0), ("dk", 1), ("dv", 2)):
        g, r = got[..., k * C:(k + 1) * C], ref[..., k * C:(k + 1) * C]
        scale = max(np.abs(r).max(), 1e-30)
        err = np.abs(g - r).max()
        assert err <= TOL * scale, f"{what} {name}: max err {err:.3e} = {err / scale:.2e} x max|ref| {scale:.3e}"


SHAPES = [(2, 64, 128, 2), (1, 127, 128, 2), (1, 128, 64, 1), (2, 129, 128, 2), (1, 257, 256, 4),
          (3, 97, 768, 12), (2, 300, 768, 12), (1, 1024, 768, 12)]


@pytest.mark.parametrize("B,T,C,NH", SHAPES)
def test_tensor_core_backward(B, T, C, NH):
    qkv, dout = make_inputs(B, T, C, seed=B * 1000 + T)
    out = oracle.attention(qkv, NH)
    got = gpu_backward(qkv, dout, out, NH)
    check_blocks(got, oracle.attention_backward(qkv, dout, NH), C, f"{B}x{T}x{C}/{NH}")


def test_single_position():
    # T = 1: P = 1, so dv = dout exactly and dq = dk = 0.  dv carries the
    # one rounding of dout to bf16.  dq, dk: dS = dP - D with dP = dout . v
    # from bf16-rounded dout and v (fp32 sum) and D = dout . out from the fp32
    # values, so |dS| <= (2u + u^2) sum_d |dout_d v_d| (u = 2^-8), and dq =
    # dS k / 8 (dS and k rounded once more): |dq_d| <= 3u sum_d |dout_d
    # v_d| |k_d| / 8, and the same with q for dk.
    B, T, C, NH = 3, 1, 256, 4
    qkv, dout = make_inputs(B, T, C, seed=1)
    out = oracle.attention(qkv, NH)
    got = gpu_backward(qkv, dout, out, NH)
    u = 2.0 ** -8
    np.testing.assert_allclose(got[..., 2 * C:], dout, rtol=u, atol=0)
    hs = C // NH
    q, k, v = (qkv[..., i * C:(i + 1) * C].reshape(B, T, NH, hs) for i in range(3))
    m = np.abs(dout.reshape(B, T, NH, hs) * v).sum(axis=-1, keepdims=True)  # sum_d |dout_d v_d| per head
    for name, blk, other in (("dq", 0, k), ("dk", 1, q)):
        bound = (3 * u * m * np.abs(other) / 8).reshape(B, T, C)
        g = got[..., blk * C:(blk + 1) * C]
        assert np.all(np.abs(g) <= bound), (name, np.abs(g).max(), bound.max())


def test_tf32_and_bf16_run_the_same_kernels():
    qkv, dout = make_inputs(2, 200, 256, seed=3)
    out = oracle.attention(qkv, 4)
    a = gpu_backward(qkv, dout, out, 4, ab.GPT2_BF16)
    b = gpu_backward(qkv, dout, out, 4, ab.GPT2_TF32)
    np.testing.assert_array_equal(a, b)


def test_tensor_core_backward_is_deterministic():
    qkv, dout = make_inputs(2, 333, 768, seed=4)
    out = oracle.attention(qkv, 12)
    a = gpu_backward(qkv, dout, out, 12)
    b = gpu_backward(qkv, dout, out, 12)
    np.testing.assert_array_equal(a, b)


def test_ragged_launch_with_several_items_per_cta():
    # B=8, T=1100, 12 heads: 9 tiles per (sequence, head), 864 items per
    # kernel on 152 CTAs, the shortest items (the last key tile's dK/dV, the
    # first query tile's dQ) one tile long and the last tile ragged
    B, T, C, NH = 8, 1100, 768, 12
    qkv, dout = make_inputs(B, T, C, seed=6)
    qkv_d = dev(qkv, torch.float32)
    out_d = torch.empty((B, T, C), dtype=torch.float32, device="cuda")
    ab.attention_forward(out_d, qkv_d, B, T, C, NH, ab.GPT2_FP32, None, 0)
    got = gpu_backward(qkv, dout, host(out_d), NH)
    for b in (0, B - 1):
        ref = oracle.attention_backward(qkv[b:b + 1], dout[b:b + 1], NH)
        check_blocks(got[b:b + 1], ref, C, f"sequence {b}")


def test_full_batch_launch_sampled():
    # the B=16 T=1024 launch the training step makes; sequences 0 and 15
    # against the oracle
    B, T, C, NH = 16, 1024, 768, 12
    qkv, dout = make_inputs(B, T, C, seed=5)
    qkv_d = dev(qkv, torch.float32)
    out_d = torch.empty((B, T, C), dtype=torch.float32, device="cuda")
    ab.attention_forward(out_d, qkv_d, B, T, C, NH, ab.GPT2_FP32, None, 0)
    got = gpu_backward(qkv, dout, host(out_d), NH)
    for b in (0, B - 1):
        ref = oracle.attention_backward(qkv[b:b + 1], dout[b:b + 1], NH)
        check_blocks(got[b:b + 1], ref, C, f"sequence {b}")

