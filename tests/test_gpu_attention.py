"""GPU parity of attention_forward against the oracle's Algorithm 0.

Shapes cover T = 1, T below, at and past one 64-row tile, ragged tails,
the GPT-2 width (12 heads of 64) at T = 1024, and head sizes 16, 32 and 64.
Q, K and V are drawn at the workload's scale (std 0.55: a LayerNorm output
times 0.02-scale weights over 768 channels).  Tolerances: tensor cores 2e-2
absolute (the bar for tensor-core results); fp32 CUDA cores 1e-5 absolute.
Inputs drawn on the 16-bit grid at std 1 (and with peaked scores) isolate
the kernel's own rounding, that of the probabilities P to the 16-bit type:
|err| <= u * max|v| with unit roundoff u = 2^-8 (bf16) or 2^-11 (fp16)."""
import numpy as np
import pytest
import torch

import oracle
from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs

from gpu_helpers import assert_close, dev, host, need_gpu, no_device_error

pytestmark = pytest.mark.gpu
TOL = {ab.GPT2_BF16: 2e-2, ab.GPT2_FP16: 2e-2, ab.GPT2_TF32: 2e-2, ab.GPT2_FP32: 1e-5}
UNIT = {ab.GPT2_BF16: 2.0 ** -8, ab.GPT2_FP16: 2.0 ** -11}
GRID = {ab.GPT2_BF16: "bf16", ab.GPT2_FP16: "fp16"}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def run_attention(B, T, C, NH, precision, seed=0, std=0.55, qk_std=1.0, grid=None):
    qkv = inputs.make_normal(400 + seed, (B, T, 3 * C), std)
    qkv[..., :2 * C] *= qk_std
    if grid is not None:
        qkv = inputs.on_grid(qkv, grid)
    out = torch.full((B, T, C), float("nan"), dtype=torch.float32, device="cuda")
    wsz = ab.attention_workspace_size(B, T, C, precision)
    ws = torch.empty(max(wsz, 1), dtype=torch.uint8, device="cuda")
    ab.attention_forward(out, dev(qkv), B, T, C, NH, precision, ws, wsz)
    no_device_error()
    return host(out), oracle.attention(qkv, NH), qkv


# head size 64 (the tcgen05 kernel): T = 1, within, at and past a 128-row
# tile, past 512 rows (a CTA whose second query tile is empty: 129, 513;
# or runs on alone: 200, 700), the GPT-2 width; head sizes 16 and 32 (the
# mma.sync kernel)
SHAPES = [(1, 1, 128, 2), (2, 64, 128, 2), (1, 128, 128, 2), (2, 129, 128, 2), (1, 200, 768, 12),
          (1, 513, 128, 2), (2, 700, 256, 4), (2, 1024, 768, 12), (1, 1000, 1024, 16),
          (1, 1, 64, 4), (2, 32, 64, 4), (2, 65, 128, 4), (1, 130, 256, 8), (3, 97, 192, 12)]


@pytest.mark.parametrize("precision", [ab.GPT2_BF16, ab.GPT2_FP16, ab.GPT2_TF32, ab.GPT2_FP32])
@pytest.mark.parametrize("B,T,C,NH", SHAPES)
def test_attention(B, T, C, NH, precision):
    got, ref, _ = run_attention(B, T, C, NH, precision)
    assert_close(got, ref, atol=TOL[precision], what=f"attention {B}x{T}x{C}/{NH} p{precision}")


@pytest.mark.parametrize("precision", [ab.GPT2_BF16, ab.GPT2_FP16])
@pytest.mark.parametrize("qk_std", [1.0, 3.0])
@pytest.mark.parametrize("B,T,C,NH", [(2, 65, 128, 4), (1, 300, 768, 12), (1, 1024, 768, 12), (2, 40, 64, 4),
                                      (2, 257, 128, 2)])
def test_attention_on_grid(B, T, C, NH, precision, qk_std):
    # qk_std 3: a few keys dominate each row, exercising the running max
    got, ref, qkv = run_attention(B, T, C, NH, precision, seed=3, std=1.0, qk_std=qk_std, grid=GRID[precision])
    vmax = np.abs(qkv[..., 2 * C:]).max()
    assert_close(got, ref, atol=UNIT[precision] * vmax, what=f"on-grid attention qk_std {qk_std}")


def test_attention_fp32_peaked():
    # scores of magnitude up to ~40: their fp32 rounding (ulp 3.8e-6) moves
    # each probability by a few 1e-6 relative, times |v| <= ~4
    got, ref, _ = run_attention(1, 300, 768, 12, ab.GPT2_FP32, seed=3, std=1.0, qk_std=3.0)
    assert_close(got, ref, atol=5e-5, what="peaked fp32")


@pytest.mark.parametrize("precision", [ab.GPT2_BF16, ab.GPT2_FP16])
@pytest.mark.parametrize("late", [40, 70, 100, 127, 250])
def test_attention_late_dominant_key(precision, late):
    # Every query is u and every key small except key `late`, which scores
    # about 17 log2 units above the others.  Rows t >= late meet it after
    # the 32-key chunks before it have been exponentiated against a lower
    # maximum: the kernel raises the maximum inside the tile and rescales the
    # probabilities already written (the key in the second, third or fourth
    # chunk of the first key tile, or in the second key tile, where O is
    # rescaled as well).  On the 16-bit grid; the probabilities rescaled a
    # second time are below 2^-17 of the largest, so the bound is that of
    # one rounding, u * max|v|, to within a factor 1 + 2^-6.
    B, T, C, NH = 1, 256, 128, 2
    hs = C // NH
    qkv = inputs.make_normal(410, (B, T, 3 * C), 0.3)
    u = np.full(hs, 0.5)
    for h in range(NH):
        qkv[0, :, h * hs:(h + 1) * hs] = u
        qkv[0, late, C + h * hs:C + (h + 1) * hs] = 6 * u
    qkv = inputs.on_grid(qkv, GRID[precision])
    out = torch.full((B, T, C), float("nan"), dtype=torch.float32, device="cuda")
    wsz = ab.attention_workspace_size(B, T, C, precision)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    ab.attention_forward(out, dev(qkv), B, T, C, NH, precision, ws, wsz)
    no_device_error()
    ref = oracle.attention(qkv, NH)
    vmax = np.abs(qkv[..., 2 * C:]).max()
    assert_close(host(out), ref, atol=UNIT[precision] * vmax * (1 + 2.0 ** -6), what=f"dominant key at {late}")


@pytest.mark.parametrize("precision", [ab.GPT2_BF16, ab.GPT2_FP16])
def test_attention_ragged_launch_with_several_units_per_cta(precision):
    # B=8, T=1100, 12 heads of 64: 9 query tiles, so 5 units per (sequence,
    # head), the last without a second query tile; 480 units on 152 CTAs, so
    # CTAs run several units in a row and write each unit's output during
    # the next one.  Sequences 0 and 7 against the oracle.
    B, T, C, NH = 8, 1100, 768, 12
    qkv = inputs.make_normal(420, (B, T, 3 * C), 0.55)
    out = torch.full((B, T, C), float("nan"), dtype=torch.float32, device="cuda")
    wsz = ab.attention_workspace_size(B, T, C, precision)
    ws = torch.empty(max(wsz, 1), dtype=torch.uint8, device="cuda")
    ab.attention_forward(out, dev(qkv), B, T, C, NH, precision, ws, wsz)
    no_device_error()
    got = host(out)
    assert np.isfinite(got).all()
    for b in (0, B - 1):
        assert_close(got[b:b + 1], oracle.attention(qkv[b:b + 1], NH), atol=TOL[precision], what=f"sequence {b}")


def test_attention_launch_past_the_unit_table():
    # B=136, T=250, 12 heads of 64: one unit per (sequence, head), the
    # second query tile ragged (122 rows); 1632 units, more than the
    # host-made table holds (1600), so the CTAs take units round-robin,
    # alternate rounds backwards.  Sequences 0, 67 and 135 against the
    # oracle.
    B, T, C, NH = 136, 250, 768, 12
    qkv = inputs.make_normal(421, (B, T, 3 * C), 0.55)
    out = torch.full((B, T, C), float("nan"), dtype=torch.float32, device="cuda")
    wsz = ab.attention_workspace_size(B, T, C, ab.GPT2_FP16)
    ws = torch.empty(max(wsz, 1), dtype=torch.uint8, device="cuda")
    ab.attention_forward(out, dev(qkv), B, T, C, NH, ab.GPT2_FP16, ws, wsz)
    no_device_error()
    got = host(out)
    assert np.isfinite(got).all()
    for b in (0, 67, B - 1):
        assert_close(got[b:b + 1], oracle.attention(qkv[b:b + 1], NH), atol=TOL[ab.GPT2_FP16], what=f"sequence {b}")


def test_attention_causal_bitwise():
    B, T, C, NH = 1, 150, 768, 12
    qkv = inputs.make_normal(9, (B, T, 3 * C), 0.55)
    ws = torch.empty(ab.attention_workspace_size(B, T, C, ab.GPT2_BF16), dtype=torch.uint8, device="cuda")
    outs = []
    for q in (qkv, np.concatenate([qkv[:, :100], inputs.make_normal(10, (B, T - 100, 3 * C))], axis=1)):
        o = torch.empty(B, T, C, dtype=torch.float32, device="cuda")
        ab.attention_forward(o, dev(q), B, T, C, NH, ab.GPT2_BF16, ws, ws.numel())
        outs.append(host(o))
    np.testing.assert_array_equal(outs[0][:, :100], outs[1][:, :100])
