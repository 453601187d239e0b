"""Helpers shared by the GPU parity tests: device transfer and the
tolerance checks, which report the worst element when they fail."""
import numpy as np
import pytest
import torch

from gpt_transformer_forward_gb300 import binding as ab


def need_gpu():
    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA GPU"
    # output buffers are made with explicit dtypes, and no test may change
    # torch's default dtype for the others
    assert torch.get_default_dtype() == torch.float32
    ab.load()


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t) -> np.ndarray:
    torch.cuda.synchronize()
    return t.detach().float().cpu().numpy() if t.dtype != torch.int32 else t.cpu().numpy()


def assert_close(got, ref, atol=0.0, rtol=0.0, floor=None, what=""):
    """|got - ref| <= atol + rtol * max(floor, |ref|) elementwise (floor None: |ref|)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    scale = np.abs(ref) if floor is None else np.maximum(floor, np.abs(ref))
    err = np.abs(got - ref)
    bound = atol + rtol * scale
    bad = ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err - bound, -np.inf)), err.shape)
        pytest.fail(f"{what}: {int(bad.sum())} of {err.size} outside tolerance; worst at {i}: got {got[i]!r} "
                    f"ref {ref[i]!r} err {err[i]:.3e} bound {bound[i]:.3e}; max err {err.max():.3e}")
    return float(err.max()) if err.size else 0.0


def no_device_error():
    w = ab.gpt2_get_error()
    assert w == 0, f"device error word {w:#x}"
