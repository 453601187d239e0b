"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test ties one oracle function to a closed form, an invariant, a brute
force on tiny inputs, or an independent library routine (PyTorch float64 CPU
operators and SciPy, which share no code with the oracle's C source).  The
cases are chosen so that a dropped term, a wrong sign, a wrong index or a
transposed operand anywhere in the oracle fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import ndtr

import oracle
from gpt_transformer_forward_gb300 import inputs


def rnd(seed, shape, std=1.0):
    return inputs.make_normal(seed, shape, std=std, dtype=np.float64)


# ------------------------------------------------------------------ matmul
def brute_matmul(x, W, b):
    N, C = x.shape
    OC = W.shape[0]
    out = [[0.0] * OC for _ in range(N)]
    for n in range(N):
        for o in range(OC):
            s = 0.0 if b is None else float(b[o])
            for k in range(C):
                s += float(x[n, k]) * float(W[o, k])
            out[n][o] = s
    return np.array(out)


@pytest.mark.parametrize("N,C,OC", [(7, 5, 3), (1, 1, 1), (9, 16, 33)])
def test_matmul_brute_force(N, C, OC):
    x, W, b = rnd(1, (N, C)), rnd(2, (OC, C)), rnd(3, (OC,))
    np.testing.assert_allclose(oracle.matmul(x, W, b), brute_matmul(x, W, b), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.matmul(x, W, None), brute_matmul(x, W, None), rtol=1e-13, atol=1e-13)


def test_matmul_identity_weight_gives_input_plus_bias():
    x, b = rnd(4, (11, 24)), rnd(5, (24,))
    np.testing.assert_array_equal(oracle.matmul(x, np.eye(24), b), x + b)


def test_matmul_not_transposed():
    # a non-square weight distinguishes x W^T from x W; torch is the library check
    x, W, b = rnd(6, (33, 96)), rnd(7, (40, 96)), rnd(8, (40,))
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(W), torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(oracle.matmul(x, W, b), ref, rtol=1e-12, atol=1e-12)


def test_matmul_param_buffer_matches_f64_route():
    # the forward pass reads weights as fp32 from the parameter buffer
    cfg = inputs.TINY
    p = inputs.make_params(cfg, 11, "perturbed")
    v = inputs.param_views(cfg, p)
    h = rnd(12, (5, cfg.channels))
    ours = oracle.lm_head(cfg, p, h)
    ref = h @ v["wte"].astype(np.float64).T
    np.testing.assert_allclose(ours, ref, rtol=1e-12, atol=1e-12)


# -------------------------------------------------------------------- GELU
def test_gelu_closed_form_points():
    x = np.array([0.0, 10.0, -10.0, 30.0])
    g = oracle.gelu(x)
    assert g[0] == 0.0
    assert abs(g[1] - 10.0) < 1e-12 and abs(g[2]) < 1e-12 and g[3] == 30.0


def test_gelu_odd_part_identity():
    # tanh is odd, so GELU(x) - GELU(-x) = x exactly in exact arithmetic
    x = np.linspace(-7, 7, 1001)
    np.testing.assert_allclose(oracle.gelu(x) - oracle.gelu(-x), x, rtol=0, atol=1e-14)


def test_gelu_is_the_tanh_approximation_of_exact_gelu():
    # |tanh-form - x*Phi(x)| stays below 5e-4 (the approximation's known error);
    # the erf form itself, a missing cubic term (3.4e-2) or a wrong constant
    # (1e-1) would fail one side of the check.
    x = np.linspace(-8, 8, 20001)
    dev = np.abs(oracle.gelu(x) - x * ndtr(x))
    assert dev.max() < 5e-4
    assert dev.max() > 1e-4


def test_gelu_matches_torch_tanh_gelu():
    x = rnd(13, (4096,), std=3.0)
    ref = F.gelu(torch.from_numpy(x), approximate="tanh").numpy()
    np.testing.assert_allclose(oracle.gelu(x), ref, rtol=1e-14, atol=1e-15)


# --------------------------------------------------------------- LayerNorm
def test_layernorm_pre_affine_moments():
    C = 768
    x = rnd(14, (64, C), std=0.3) + 0.7
    y, mean, rstd = oracle.layernorm(x, np.ones(C, np.float32), np.zeros(C, np.float32))
    var = x.var(axis=1)
    assert np.abs(y.mean(axis=1)).max() < 1e-12
    np.testing.assert_allclose(y.var(axis=1), var / (var + 1e-5), rtol=1e-12)
    np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-13)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(var + 1e-5), rtol=1e-12)


def test_layernorm_eps_is_present():
    # small-variance rows: with eps = 1e-5 the output variance is well below 1
    C = 64
    x = rnd(15, (8, C), std=1e-3)
    y, _, _ = oracle.layernorm(x, np.ones(C, np.float32), np.zeros(C, np.float32))
    assert (y.var(axis=1) < 0.2).all()


def test_layernorm_constant_row_gives_beta():
    C = 32
    x = np.full((3, C), 2.5)
    beta = inputs.make_normal(16, (C,))
    y, _, _ = oracle.layernorm(x, inputs.make_normal(17, (C,)), beta)
    np.testing.assert_array_equal(y, np.broadcast_to(beta.astype(np.float64), y.shape))


def test_layernorm_matches_torch_and_affine():
    C = 768
    x = rnd(18, (40, C), std=2.0)
    w = inputs.make_normal(19, (C,)) + 1
    b = inputs.make_normal(20, (C,))
    y, _, _ = oracle.layernorm(x, w, b)
    ref = F.layer_norm(torch.from_numpy(x), (C,), torch.from_numpy(w.astype(np.float64)),
                       torch.from_numpy(b.astype(np.float64)), eps=1e-5).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-12)
    # invariance to a positive scale and a shift of the input row (up to eps)
    y2, _, _ = oracle.layernorm(3.0 * x + 1.0, w, b)
    np.testing.assert_allclose(y2, y, rtol=1e-5, atol=1e-5)


# ----------------------------------------------------------------- softmax
def test_softmax_rows_padding_constant_and_shift():
    V, Vp = 500, 512
    logits = rnd(21, (6, Vp), std=2.0)
    p = oracle.softmax(logits, V)
    np.testing.assert_allclose(p[:, :V].sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert (p[:, V:] == 0).all()
    np.testing.assert_allclose(oracle.softmax(logits + 123.0, V), p, rtol=1e-12, atol=1e-16)
    const = oracle.softmax(np.full((2, Vp), -4.0), V)
    np.testing.assert_allclose(const[:, :V], 1.0 / V, rtol=1e-14)
    ref = torch.softmax(torch.from_numpy(logits[:, :V]), dim=-1).numpy()
    np.testing.assert_allclose(p[:, :V], ref, rtol=1e-13, atol=1e-18)


def test_softmax_large_logits_no_overflow():
    logits = np.array([[1000.0, 999.0, -1000.0, 7.0]])
    p = oracle.softmax(logits, 3)
    e = math.exp(-1.0)
    np.testing.assert_allclose(p[0], [1 / (1 + e), e / (1 + e), 0.0, 0.0], rtol=1e-14, atol=1e-300)


# --------------------------------------------------------------- attention
def test_attention_algorithm0_vs_algorithm1_tiles():
    B, T, C, NH = 2, 37, 48, 3
    qkv = rnd(22, (B, T, 3 * C))
    a0 = oracle.attention(qkv, NH)
    for Br, Bc in [(1, 1), (7, 7), (16, 16), (T, T), (5, 16), (16, 3)]:
        a1 = oracle.attention_online(qkv, NH, Br, Bc)
        np.testing.assert_allclose(a1, a0, rtol=1e-12, atol=1e-13)


def test_attention_matches_torch_sdpa():
    B, T, C, NH = 2, 29, 64, 4
    hs = C // NH
    qkv = rnd(23, (B, T, 3 * C))
    q, k, v = (torch.from_numpy(qkv[:, :, i * C:(i + 1) * C]).reshape(B, T, NH, hs).transpose(1, 2)
               for i in range(3))
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(1, 2).reshape(B, T, C)
    np.testing.assert_allclose(oracle.attention(qkv, NH), ref.numpy(), rtol=1e-12, atol=1e-13)


def test_attention_closed_forms():
    B, T, C, NH = 1, 20, 32, 2
    qkv = rnd(24, (B, T, 3 * C))
    # T = 1: the only visible key is itself, so the output is v_0
    one = oracle.attention(qkv[:, :1], NH)
    np.testing.assert_array_equal(one[0, 0], qkv[0, 0, 2 * C:])
    # q = 0: uniform weights over j <= t, the causal running mean of v
    z = qkv.copy()
    z[:, :, :C] = 0.0
    out = oracle.attention(z, NH)
    v = qkv[0, :, 2 * C:]
    runmean = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    np.testing.assert_allclose(out[0], runmean, rtol=1e-12, atol=1e-13)
    # one key aligned with q and much larger than the rest: output is that key's value
    d = qkv.copy()
    d[0, :, :2 * C] *= 1e-3
    d[0, 5, C:2 * C] = 50.0 * d[0, 12, :C] / np.linalg.norm(d[0, 12, :C])
    d[0, 12, :C] *= 50.0 / np.linalg.norm(d[0, 12, :C])
    out = oracle.attention(d, 1)
    np.testing.assert_allclose(out[0, 12], d[0, 5, 2 * C:], rtol=0, atol=1e-6)


def test_attention_is_causal():
    B, T, C, NH = 1, 16, 32, 4
    qkv = rnd(25, (B, T, 3 * C))
    a = oracle.attention(qkv, NH)
    pert = qkv.copy()
    pert[0, 9:] += rnd(26, (T - 9, 3 * C))
    b = oracle.attention(pert, NH)
    np.testing.assert_array_equal(a[0, :9], b[0, :9])
    assert np.abs(a[0, 9:] - b[0, 9:]).max() > 1e-3


def test_attention_head_columns():
    # head h reads only columns [h*hs, (h+1)*hs) of q, k, v
    B, T, C, NH = 1, 8, 32, 4
    hs = C // NH
    qkv = rnd(27, (B, T, 3 * C))
    a = oracle.attention(qkv, NH)
    pert = qkv.copy()
    for blk in range(3):
        pert[..., blk * C + 2 * hs: blk * C + 3 * hs] += 1.0
    b = oracle.attention(pert, NH)
    changed = np.abs(a - b).max(axis=(0, 1)).reshape(NH, hs).max(axis=1)
    assert changed[2] > 1e-3 and changed[0] == 0 and changed[1] == 0 and changed[3] == 0


# -------------------------------------------------- encoder, residual, argmax
def test_encoder_is_the_gather_add():
    cfg = inputs.TINY
    p = inputs.make_params(cfg, 28)
    v = inputs.param_views(cfg, p)
    tok = inputs.make_tokens(29, 3, 17, cfg.vocab_size)
    out = oracle.encoder(tok, v["wte"], v["wpe"])
    for b in range(3):
        for t in range(17):
            np.testing.assert_array_equal(
                out[b, t], v["wte"][tok[b, t]].astype(np.float64) + v["wpe"][t].astype(np.float64))


def test_residual_and_argmax():
    a, b = rnd(30, (100,)), rnd(31, (100,))
    np.testing.assert_array_equal(oracle.residual(a, b), a + b)
    lg = rnd(32, (4, 64))
    lg[1, 10] = lg[1, 20] = 9.0        # tie: lowest index wins
    lg[2, 60] = 99.0                   # beyond V: ignored
    nxt = oracle.argmax(lg, 50)
    assert nxt[1] == 10
    np.testing.assert_array_equal(nxt, np.argmax(lg[:, :50], axis=1))
