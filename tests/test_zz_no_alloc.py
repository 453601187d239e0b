"""matmul_forward_noalloc: the matmul entry point for callers that cannot
allocate device memory (its scratch is a fixed array inside the library).

Its results must equal matmul_forward's, given a workspace, on the same
inputs, on two calls in a row with different inputs (so stale scratch from
the first call would show), within the GEMM tolerances of the other tests.
This file is collected last; it passes alone in a fresh process too."""
import numpy as np
import pytest
import torch

from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs

from gpu_helpers import assert_close, dev, host, need_gpu, no_device_error

pytestmark = pytest.mark.gpu
TOL = {ab.GPT2_BF16: 2e-2, ab.GPT2_FP16: 5e-3}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def with_workspace(x, W, b, N, C, OC, precision):
    out = torch.empty(N, OC, dtype=torch.float32, device="cuda")
    wsz = ab.matmul_workspace_size(N, C, OC, precision)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    ab.matmul_forward(out, x, W, b, N, C, OC, precision, ws, wsz)
    return host(out)


@pytest.mark.parametrize("precision", [ab.GPT2_FP16, ab.GPT2_BF16])
@pytest.mark.parametrize("N,C,OC", [(300, 768, 2304), (64, 3072, 768), (5, 64, 40)])
def test_noalloc_matches_workspace_entry_point(N, C, OC, precision):
    for call, seed in enumerate((1, 2)):  # two calls in a row, different inputs
        x = dev(inputs.make_normal(500 + seed, (N, C), 1.0))
        W = dev(inputs.make_normal(600 + seed, (OC, C), 0.02))
        b = dev(inputs.make_normal(700 + seed, (OC,), 0.02))
        ref = with_workspace(x, W, b, N, C, OC, precision)
        out = torch.full((N, OC), float("nan"), dtype=torch.float32, device="cuda")
        ab.matmul_forward_noalloc(out, x, W, b, N, C, OC, precision)
        no_device_error()
        assert_close(host(out), ref, atol=TOL[precision], what=f"no-alloc call {call}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    N, C, OC = 8192, 1024, 1024  # 2 * (N*C + OC*C) bytes = 18 MiB > 16 MiB
    assert ab.matmul_workspace_size(N, C, OC, ab.GPT2_FP16) > 16 << 20
    x = torch.zeros(8, 8, device="cuda")
    with pytest.raises(ab.GPT2Error) as e:
        ab.matmul_forward_noalloc(x, x, x, None, N, C, OC, ab.GPT2_FP16)
    assert e.value.code == -4
