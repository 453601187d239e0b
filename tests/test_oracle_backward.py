"""Pins of the oracle's attention backward (FlashAttention (II): the
backward algorithms of Algorithms 0 and 1), independent of the oracle's
own formulas:

- central finite differences of L = sum(dO * attention(qkv)) on tiny shapes,
  every element of dqkv;
- the chain-rule form (Algorithm 0's backward) against the tiled form that
  recomputes the attention matrix from row statistics (Algorithm 1's
  backward) for several tile shapes;
- closed forms: T = 1 (dQ = dK = 0, dV = dO); Q = 0 (uniform causal
  weights: dV_j = sum_{t >= j} dO_t / (t + 1), dK = 0);
- invariants: the keys' gradients of a head sum to zero (adding one vector
  to every key moves each score row by a constant, which the softmax
  ignores); causality (dQ at t does not depend on dO after t, and dK, dV at
  j do not depend on dO before j);
- a float64 torch autograd cross-check."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def rand(seed, *shape, scale=1.0):
    return np.random.default_rng(seed).normal(size=shape) * scale


def loss(qkv, dout, NH):
    return float((oracle.attention(qkv, NH) * dout).sum())


@pytest.mark.parametrize("B,T,C,NH", [(1, 7, 8, 2), (2, 5, 12, 3), (1, 9, 4, 1)])
def test_matches_finite_differences(B, T, C, NH):
    qkv = rand(1, B, T, 3 * C)
    dout = rand(2, B, T, C)
    g = oracle.attention_backward(qkv, dout, NH)
    h = 1e-6
    fd = np.zeros_like(qkv)
    for idx in np.ndindex(qkv.shape):
        a, b = qkv.copy(), qkv.copy()
        a[idx] += h
        b[idx] -= h
        fd[idx] = (loss(a, dout, NH) - loss(b, dout, NH)) / (2 * h)
    np.testing.assert_allclose(g, fd, atol=1e-7 * max(1.0, np.abs(g).max()), rtol=0)
    assert np.abs(g[..., :C]).max() > 1e-3 and np.abs(g[..., C:2 * C]).max() > 1e-3  # dQ, dK are not trivially 0


@pytest.mark.parametrize("Br,Bc", [(1, 1), (3, 2), (5, 3), (16, 16), (40, 40), (7, 16)])
def test_algorithm0_and_tiled_backward_agree(Br, Bc):
    B, T, C, NH = 2, 40, 32, 4
    qkv = rand(3, B, T, 3 * C, scale=0.8)
    dout = rand(4, B, T, C)
    g0 = oracle.attention_backward(qkv, dout, NH)
    g1 = oracle.attention_backward_online(qkv, dout, oracle.attention(qkv, NH), NH, Br, Bc)
    np.testing.assert_allclose(g1, g0, atol=1e-12 * np.abs(g0).max(), rtol=0)


def test_single_position():
    B, T, C, NH = 3, 1, 16, 2
    qkv, dout = rand(5, B, T, 3 * C), rand(6, B, T, C)
    g = oracle.attention_backward(qkv, dout, NH)
    assert np.all(g[..., :2 * C] == 0.0)
    np.testing.assert_array_equal(g[..., 2 * C:], dout)


def test_zero_queries_give_uniform_causal_weights():
    B, T, C, NH = 1, 6, 8, 2
    qkv = rand(7, B, T, 3 * C)
    qkv[..., :C] = 0.0
    dout = rand(8, B, T, C)
    g = oracle.attention_backward(qkv, dout, NH)
    expect_dv = np.zeros((B, T, C))
    for j in range(T):
        for t in range(j, T):
            expect_dv[:, j] += dout[:, t] / (t + 1)
    np.testing.assert_allclose(g[..., 2 * C:], expect_dv, atol=1e-14)
    np.testing.assert_allclose(g[..., C:2 * C], 0.0, atol=1e-14)


def test_key_gradients_of_a_head_sum_to_zero():
    B, T, C, NH = 2, 11, 12, 3
    g = oracle.attention_backward(rand(9, B, T, 3 * C), rand(10, B, T, C), NH)
    np.testing.assert_allclose(g[..., C:2 * C].sum(axis=1), 0.0, atol=1e-12)


def test_causality_of_the_gradients():
    B, T, C, NH, cut = 1, 12, 8, 2, 6
    qkv, dout = rand(11, B, T, 3 * C), rand(12, B, T, C)
    g = oracle.attention_backward(qkv, dout, NH)
    late = dout.copy()
    late[:, cut:] += rand(13, B, T - cut, C)
    g_late = oracle.attention_backward(qkv, late, NH)
    np.testing.assert_array_equal(g_late[:, :cut, :C], g[:, :cut, :C])  # dQ before the cut
    early = dout.copy()
    early[:, :cut] += rand(14, B, cut, C)
    g_early = oracle.attention_backward(qkv, early, NH)
    np.testing.assert_array_equal(g_early[:, cut:, C:], g[:, cut:, C:])  # dK, dV from the cut on


def test_torch_autograd_float64():
    B, T, C, NH = 2, 13, 16, 4
    hs = C // NH
    qkv, dout = rand(15, B, T, 3 * C), rand(16, B, T, C)
    x = torch.tensor(qkv, dtype=torch.float64, requires_grad=True)
    q, k, v = (x[..., i * C:(i + 1) * C].reshape(B, T, NH, hs).transpose(1, 2) for i in range(3))
    s = (q @ k.transpose(-1, -2)) / hs ** 0.5
    s = s.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    o = (torch.softmax(s, -1) @ v).transpose(1, 2).reshape(B, T, C)
    (o * torch.tensor(dout)).sum().backward()
    np.testing.assert_allclose(oracle.attention_backward(qkv, dout, NH), x.grad.numpy(), atol=1e-12)
