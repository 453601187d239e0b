"""GPU parity of matmul_forward (every GEMM site's arithmetic) against the
oracle, in each precision mode, on GPT-2-scale values: activations N(0, 1)
as a LayerNorm produces them, weights N(0, 0.02), biases N(0, 0.02).

Tolerances: bf16 operands 2e-2 absolute (the bar for tensor-core results);
fp16 operands (unit roundoff 2^-11) and tf32 operands (10 stored bits,
truncated) 5e-3 absolute; fp32 CUDA cores 1e-5 * max(1, |ref|) (fp32
accumulation over K <= 3072 terms).  Inputs drawn on the 16-bit
grid are converted exactly, so there the tensor-core result must equal the
oracle to fp32-accumulation accuracy (1e-4): any fault in the TMA, swizzle,
descriptor or TMEM path shows up as an O(1) error."""
import numpy as np
import pytest
import torch

import oracle
from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs

from gpu_helpers import assert_close, dev, host, need_gpu, no_device_error

pytestmark = pytest.mark.gpu
TOL = {ab.GPT2_BF16: 2e-2, ab.GPT2_FP16: 5e-3, ab.GPT2_TF32: 5e-3, ab.GPT2_FP32: 1e-5}
ALL = [ab.GPT2_BF16, ab.GPT2_FP16, ab.GPT2_TF32, ab.GPT2_FP32]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def run_matmul(N, C, OC, precision, bias=True, seed=0, grid=None):
    x = inputs.make_normal(100 + seed, (N, C), 1.0)
    W = inputs.make_normal(200 + seed, (OC, C), 0.02)
    b = inputs.make_normal(300 + seed, (OC,), 0.02) if bias else None
    if grid is not None:
        x, W = inputs.on_grid(x, grid), inputs.on_grid(W, grid)
    out = torch.full((N, OC), float("nan"), dtype=torch.float32, device="cuda")
    wsz = ab.matmul_workspace_size(N, C, OC, precision)
    ws = torch.empty(max(wsz, 1), dtype=torch.uint8, device="cuda")
    ab.matmul_forward(out, dev(x), dev(W), dev(b) if bias else None, N, C, OC, precision, ws, wsz)
    no_device_error()
    return host(out), oracle.matmul(x, W, b)


# shapes: the GEMM sites at GPT-2 widths, ragged M and N tails, tiny cases
SHAPES = [
    (128, 64, 256),      # one tile
    (256, 768, 2304),    # QKV
    (300, 768, 768),     # attn-proj, ragged M
    (129, 768, 3072),    # FC, one row past a tile
    (200, 3072, 768),    # FC-proj, K = 3072
    (64, 768, 50304),    # LM head width, half-empty last N tile
    (5, 64, 40),         # tiny, ragged N inside one tile
    (32, 768, 2304),     # decode-sized M
    (1, 8, 4),           # smallest legal shape
    # M <= 64 (the small-M kernel: K split over a cluster, reduced in
    # distributed shared memory): padded activation rows 16/32/48/64, 16-way
    # splits at K = 3072, a ragged K (200 = 3 blocks + 8) and N tail
    (33, 768, 2304),
    (64, 3072, 768),
    (17, 768, 3072),
    (2, 3072, 768),
    (48, 200, 200),
]


@pytest.mark.parametrize("precision", ALL)
@pytest.mark.parametrize("N,C,OC", SHAPES)
def test_matmul(N, C, OC, precision):
    got, ref = run_matmul(N, C, OC, precision)
    if precision == ab.GPT2_FP32:  # fp32 rounding: relative to max(1, |ref|)
        assert_close(got, ref, rtol=TOL[precision], floor=1.0, what=f"matmul {N}x{C}x{OC} fp32")
    else:
        assert_close(got, ref, atol=TOL[precision], what=f"matmul {N}x{C}x{OC} p{precision}")


@pytest.mark.parametrize("precision,grid", [(ab.GPT2_BF16, "bf16"), (ab.GPT2_FP16, "fp16"),
                                            (ab.GPT2_TF32, "tf32")])
@pytest.mark.parametrize("N,C,OC", [(300, 768, 2304), (128 * 20, 256, 256 * 20), (64, 3072, 50304), (7, 64, 40),
                                    (32, 3072, 768), (3, 768, 2304)])
def test_matmul_on_grid_is_exact_to_fp32_accumulation(N, C, OC, precision, grid):
    got, ref = run_matmul(N, C, OC, precision, seed=9, grid=grid)
    assert_close(got, ref, atol=1e-4, what=f"on-grid matmul {N}x{C}x{OC} {grid}")


@pytest.mark.parametrize("precision", [ab.GPT2_BF16, ab.GPT2_FP16, ab.GPT2_TF32])
def test_matmul_no_bias_and_persistent_tiles(precision):
    # 2 * 148 + tiles: every CTA walks several tiles through both TMEM buffers
    got, ref = run_matmul(128 * 20, 256, 256 * 20, precision, bias=False, seed=5)
    assert_close(got, ref, atol=TOL[precision], what="persistent")


@pytest.mark.parametrize("precision", [ab.GPT2_BF16, ab.GPT2_FP16, ab.GPT2_TF32])
def test_small_m_split_sum_is_run_to_run_identical(precision):
    # the K-split partials are summed in a fixed order: repeated calls agree bit for bit
    a, ref = run_matmul(32, 3072, 768, precision, seed=11)
    b, _ = run_matmul(32, 3072, 768, precision, seed=11)
    np.testing.assert_array_equal(a, b)
    assert_close(a, ref, atol=TOL[precision], what="split-K small M")


def test_matmul_bf16_is_bf16_rounded():
    # with operands exactly representable in bf16 the tensor-core result is
    # the fp32-accumulated exact product (small K keeps fp32 sums exact)
    N, C, OC = 128, 16, 256
    x = np.round(inputs.make_normal(7, (N, C), 4.0)).astype(np.float32)
    W = np.round(inputs.make_normal(8, (OC, C), 4.0)).astype(np.float32)
    out = torch.empty(N, OC, dtype=torch.float32, device="cuda")
    wsz = ab.matmul_workspace_size(N, C, OC, ab.GPT2_BF16)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    ab.matmul_forward(out, dev(x), dev(W), None, N, C, OC, ab.GPT2_BF16, ws, wsz)
    np.testing.assert_array_equal(host(out), oracle.matmul(x, W, None))


def test_matmul_rejects_small_workspace():
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    out = torch.empty(8, 8, dtype=torch.float32, device="cuda")
    x = torch.zeros(8, 8, device="cuda")
    with pytest.raises(ab.GPT2Error) as e:
        ab.matmul_forward(out, x, x, None, 8, 8, 8, ab.GPT2_BF16, ws, 16)
    assert e.value.code == -4
