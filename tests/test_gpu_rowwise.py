"""GPU parity of the HBM-bound steps against the oracle, element by element:
encoder and residual bit-exact (an fp32 add of two fp32 values is the
correctly rounded double sum), LayerNorm, GELU and softmax within 1e-5
relative, argmax exact.  Sizes span several blocks and ragged tails."""
import numpy as np
import pytest
import torch

import oracle
from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs

from gpu_helpers import assert_close, dev, host, need_gpu, no_device_error

pytestmark = pytest.mark.gpu
REL = 1e-5  # single-step fp32 kernels: |err| <= 1e-5 * max(1, |ref|)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("B,T,C,V", [(2, 32, 64, 512), (3, 77, 768, 50257), (1, 1, 8, 3), (4, 1024, 1024, 1000)])
def test_encoder_bit_exact(B, T, C, V):
    wte = inputs.make_normal(1, (V + 3, C), 0.02)
    wpe = inputs.make_normal(2, (T + 5, C), 0.02)
    tok = inputs.make_tokens(3, B, T, V)
    out = torch.empty(B, T, C, dtype=torch.float32, device="cuda")
    ab.encoder_forward(out, dev(tok), dev(wte), dev(wpe), B, T, C, V)
    ref = oracle.encoder(tok, wte, wpe).astype(np.float32)  # correctly rounded fp32 sums
    np.testing.assert_array_equal(host(out), ref)
    no_device_error()


def test_encoder_flags_bad_token():
    B, T, C, V = 1, 4, 16, 10
    wte = inputs.make_normal(4, (V, C))
    wpe = inputs.make_normal(5, (T, C))
    tok = np.array([[1, 10, -3, 2]], dtype=np.int32)
    out = torch.empty(B, T, C, dtype=torch.float32, device="cuda")
    ab.encoder_forward(out, dev(tok), dev(wte), dev(wpe), B, T, C, V)
    assert ab.gpt2_get_error() == ab.DEVERR_TOKEN
    assert ab.gpt2_get_error() == 0  # reading clears the word
    # the bad rows read token 0
    got = host(out)
    np.testing.assert_array_equal(got[0, 1], (wte[0] + wpe[1]).astype(np.float32))


@pytest.mark.parametrize("N,C", [(1, 768), (37, 768), (1000, 1024), (64, 64), (5, 200), (300, 1536)])
def test_layernorm(N, C):
    x = inputs.make_normal(6, (N, C), 1.3) + 0.25
    w = inputs.make_normal(7, (C,), 0.3) + 1.0
    b = inputs.make_normal(8, (C,), 0.1)
    out = torch.empty(N, C, dtype=torch.float32, device="cuda")
    mean = torch.empty(N, dtype=torch.float32, device="cuda")
    rstd = torch.empty(N, dtype=torch.float32, device="cuda")
    ab.layernorm_forward(out, mean, rstd, dev(x), dev(w), dev(b), N, C)
    ref, rm, rr = oracle.layernorm(x, w, b)
    assert_close(host(out), ref, rtol=REL, floor=1.0, what="layernorm out")
    assert_close(host(mean), rm, rtol=REL, floor=1.0, what="layernorm mean")
    assert_close(host(rstd), rr, rtol=REL, what="layernorm rstd")


def test_layernorm_in_place():
    N, C = 17, 768
    x = inputs.make_normal(9, (N, C))
    w, b = np.ones(C, np.float32), np.zeros(C, np.float32)
    t = dev(x)
    ab.layernorm_forward(t, None, None, t, dev(w), dev(b), N, C)
    assert_close(host(t), oracle.layernorm(x, w, b)[0], rtol=REL, floor=1.0, what="in place")


@pytest.mark.parametrize("n", [1, 3, 4, 1001, 16384 * 3 + 2])
def test_gelu(n):
    x = inputs.make_normal(10, (n,), 3.0)
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    ab.gelu_forward(out, dev(x), n)
    assert_close(host(out), oracle.gelu(x), rtol=REL, floor=1.0, what="gelu")


@pytest.mark.parametrize("n", [1, 7, 4096, 1 << 20 | 3])
def test_residual_bit_exact(n):
    a = inputs.make_normal(11, (n,))
    b = inputs.make_normal(12, (n,))
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    ab.residual_forward(out, dev(a), dev(b), n)
    np.testing.assert_array_equal(host(out), oracle.residual(a, b).astype(np.float32))
    ta = dev(a)
    ab.residual_forward(ta, ta, dev(b), n)  # out aliases a
    np.testing.assert_array_equal(host(ta), oracle.residual(a, b).astype(np.float32))


@pytest.mark.parametrize("N,V,Vp,std", [(3, 512, 512, 1.0), (5, 50257, 50304, 0.55), (2, 50257, 50304, 8.0),
                                        (7, 5, 8, 2.0), (1, 1000, 1024, 30.0)])
def test_softmax(N, V, Vp, std):
    lg = inputs.make_normal(13, (N, Vp), std)
    out = torch.empty(N, Vp, dtype=torch.float32, device="cuda")
    ab.softmax_forward(out, dev(lg), N, V, Vp)
    ref = oracle.softmax(lg, V)
    got = host(out)
    # relative to each probability itself (probabilities are far below 1)
    assert_close(got[:, :V], ref[:, :V], rtol=REL, atol=1e-37, what="softmax")
    assert (got[:, V:] == 0).all()


@pytest.mark.parametrize("ptype,dtype", [(ab.GPT2_PROBS_F16, torch.float16), (ab.GPT2_PROBS_BF16, torch.bfloat16)])
@pytest.mark.parametrize("N,V,Vp,std", [(5, 50257, 50304, 0.55), (7, 5, 8, 2.0), (1, 1000, 1024, 30.0)])
def test_softmax_16bit_probabilities(N, V, Vp, std, ptype, dtype):
    # each 16-bit probability is the fp32 one rounded to nearest once
    # (exactly what a round-to-nearest-even conversion of softmax_forward's
    # output gives), so within the fp32 bound plus half a 16-bit unit of the
    # oracle's value
    lg = inputs.make_normal(13, (N, Vp), std)
    out32 = torch.empty(N, Vp, dtype=torch.float32, device="cuda")
    out16 = torch.full((N, Vp), float("nan"), dtype=dtype, device="cuda")
    ab.softmax_forward(out32, dev(lg), N, V, Vp)
    ab.softmax_forward_ex(out16, ptype, dev(lg), N, V, Vp)
    no_device_error()
    assert torch.equal(out16, out32.to(dtype))
    u = 2.0 ** -11 if dtype == torch.float16 else 2.0 ** -8
    ref = oracle.softmax(lg, V)
    got = out16.float().cpu().numpy().astype(np.float64)
    # fp16 values below 2^-14 are subnormal: an absolute floor of half the
    # smallest fp16 step there
    floor = 2.0 ** -25 if dtype == torch.float16 else 1e-37
    assert_close(got[:, :V], ref[:, :V], rtol=REL + u, atol=floor, what="16-bit softmax")
    assert (got[:, V:] == 0).all()


# (Vp a multiple of 4: 16-byte loads with a scalar tail; 15: scalar loads)
@pytest.mark.parametrize("B,V,Vp", [(32, 50257, 50304), (3, 10, 12), (2, 13, 15)])
def test_argmax(B, V, Vp):
    lg = inputs.make_normal(14, (B, Vp))
    lg[0, V:] = 100.0          # padding never wins
    lg[1, 3] = lg[1, 7] = 50.0  # tie: the lower index
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    ab.gpt2_argmax(nxt, dev(lg), B, V, Vp)
    np.testing.assert_array_equal(host(nxt), oracle.argmax(lg, V))
