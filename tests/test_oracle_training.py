"""Pins of the oracle's training step (the loss gradient of every parameter
and AdamW), independent of its own formulas:

- central finite differences of the loss on the tiny model, for parameters
  drawn from every tensor of the buffer;
- a float64 PyTorch autograd composite of the same model and loss;
- per step: LayerNorm's, GELU's and the matmul's backward against finite
  differences, GELU's derivative at closed-form points;
- structure: the padded vocabulary rows and the position rows past T get no
  gradient; the gradient of the mean loss is the mean of the per-sequence
  gradients;
- AdamW's first step in closed form, and a second step by hand."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gpt_transformer_forward_gb300 import inputs

CFG = inputs.TINY


@pytest.fixture(scope="module")
def problem():
    params = inputs.make_params(CFG, 11, "perturbed")
    tok = inputs.make_tokens(12, 2, 20, CFG.vocab_size)
    tgt = inputs.make_tokens(13, 2, 20, CFG.vocab_size)
    loss, g = oracle.forward_backward(CFG, params, tok, tgt)
    return params, tok, tgt, loss, g


def test_loss_gradient_matches_finite_differences(problem):
    params, tok, tgt, loss, g = problem
    rng = np.random.default_rng(14)
    offsets = np.cumsum([0] + [int(np.prod(s)) for _, s in inputs.param_shapes(CFG)])
    for (name, shape), lo, hi in zip(inputs.param_shapes(CFG), offsets[:-1], offsets[1:]):
        if name == "wpe":
            lo, hi = lo, lo + 20 * CFG.channels  # the positions in use
        for i in rng.integers(lo, hi, size=6):
            pa, pb = params.copy(), params.copy()
            pa[i] += np.float32(1e-3)
            pb[i] -= np.float32(1e-3)
            la, _ = oracle.forward_backward(CFG, pa, tok, tgt)
            lb, _ = oracle.forward_backward(CFG, pb, tok, tgt)
            fd = (la - lb) / (float(pa[i]) - float(pb[i]))
            assert abs(fd - g[i]) <= 1e-7 + 1e-5 * abs(g[i]), (name, int(i - lo), fd, g[i])


def test_matches_torch_autograd(problem):
    params, tok, tgt, loss, g = problem
    views = inputs.param_views(CFG, params)
    v = {k: torch.tensor(a.astype(np.float64), requires_grad=True) for k, a in views.items()}
    C, NH = CFG.channels, CFG.num_heads
    hs = C // NH
    B, T = tok.shape
    x = F.embedding(torch.from_numpy(tok.astype(np.int64)), v["wte"]) + v["wpe"][:T]
    for l in range(CFG.num_layers):
        h = F.layer_norm(x, (C,), v["ln1w"][l], v["ln1b"][l], eps=1e-5)
        q, k, vv = F.linear(h, v["qkvw"][l], v["qkvb"][l]).split(C, dim=-1)
        q, k, vv = (z.reshape(B, T, NH, hs).transpose(1, 2) for z in (q, k, vv))
        a = F.scaled_dot_product_attention(q, k, vv, is_causal=True).transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(a, v["attprojw"][l], v["attprojb"][l])
        u = F.gelu(F.linear(F.layer_norm(x, (C,), v["ln2w"][l], v["ln2b"][l], eps=1e-5), v["fcw"][l], v["fcb"][l]),
                   approximate="tanh")
        x = x + F.linear(u, v["fcprojw"][l], v["fcprojb"][l])
    logits = F.layer_norm(x, (C,), v["lnfw"], v["lnfb"], eps=1e-5) @ v["wte"].T
    tl = F.cross_entropy(logits[..., :CFG.vocab_size].reshape(B * T, -1), torch.from_numpy(tgt.astype(np.int64)).reshape(-1))
    tl.backward()
    assert abs(tl.item() - loss) < 1e-12
    ref = np.concatenate([v[name].grad.numpy().reshape(-1) for name, _ in inputs.param_shapes(CFG)])
    np.testing.assert_allclose(g, ref, atol=1e-12, rtol=0)


def test_padded_vocabulary_and_unused_positions_get_no_gradient():
    cfg = inputs.GPT2Config(max_seq_len=32, vocab_size=100, padded_vocab_size=104, num_layers=1, num_heads=2,
                            channels=16)
    params = inputs.make_params(cfg, 15, "perturbed")
    tok = inputs.make_tokens(16, 2, 9, cfg.vocab_size)
    _, g = oracle.forward_backward(cfg, params, tok, inputs.make_tokens(17, 2, 9, cfg.vocab_size))
    views = dict(zip([n for n, _ in inputs.param_shapes(cfg)],
                     np.split(g, np.cumsum([int(np.prod(s)) for _, s in inputs.param_shapes(cfg)])[:-1])))
    wte = views["wte"].reshape(cfg.padded_vocab_size, cfg.channels)
    wpe = views["wpe"].reshape(cfg.max_seq_len, cfg.channels)
    assert np.all(wte[cfg.vocab_size:] == 0.0) and np.abs(wte[:cfg.vocab_size]).max() > 0
    assert np.all(wpe[9:] == 0.0) and np.abs(wpe[:9]).max() > 0


def test_mean_loss_gradient_is_the_mean_over_sequences(problem):
    params, tok, tgt, loss, g = problem
    parts = [oracle.forward_backward(CFG, params, tok[b:b + 1], tgt[b:b + 1]) for b in range(2)]
    np.testing.assert_allclose(g, (parts[0][1] + parts[1][1]) / 2, atol=1e-14)
    assert abs(loss - (parts[0][0] + parts[1][0]) / 2) < 1e-13


def fd_vec(f, x, h=1e-6):
    out = np.zeros_like(x)
    for i in np.ndindex(x.shape):
        a, b = x.copy(), x.copy()
        a[i] += h
        b[i] -= h
        out[i] = (f(a) - f(b)) / (2 * h)
    return out


def test_layernorm_backward():
    rng = np.random.default_rng(18)
    x = rng.normal(size=(3, 8))
    w = rng.normal(size=8).astype(np.float32)
    b = rng.normal(size=8).astype(np.float32)
    dy = rng.normal(size=(3, 8))
    _, mean, rstd = oracle.layernorm(x, w, b)
    dx, dw, db = oracle.layernorm_backward(dy, x, w, mean, rstd)
    np.testing.assert_allclose(dx, fd_vec(lambda z: (oracle.layernorm(z, w, b)[0] * dy).sum(), x), atol=1e-8)
    xhat = (x - mean[:, None]) * rstd[:, None]
    np.testing.assert_allclose(dw, (dy * xhat).sum(0), atol=1e-13)
    np.testing.assert_allclose(db, dy.sum(0), atol=1e-13)


def test_gelu_backward():
    x = np.array([-3.0, -1.0, 0.0, 0.5, 1.0, 2.0, 10.0])
    d = oracle.gelu_backward(x, np.ones_like(x))
    assert d[2] == 0.5  # GELU'(0) = 1/2
    assert abs(d[-1] - 1.0) < 1e-12  # GELU(x) ~ x for large x
    np.testing.assert_allclose(d, fd_vec(lambda z: oracle.gelu(z).sum(), x), atol=1e-8)


def test_matmul_backward_brute_force():
    rng = np.random.default_rng(19)
    x = rng.normal(size=(5, 3))
    W = rng.normal(size=(4, 3)).astype(np.float32)
    dy = rng.normal(size=(5, 4))
    dx, dW, db = oracle.matmul_backward(dy, x, W)
    Wd = W.astype(np.float64)
    for n in range(5):
        for c in range(3):
            assert abs(dx[n, c] - sum(dy[n, o] * Wd[o, c] for o in range(4))) < 1e-13
    for o in range(4):
        for c in range(3):
            assert abs(dW[o, c] - sum(dy[n, o] * x[n, c] for n in range(5))) < 1e-13
        assert abs(db[o] - dy[:, o].sum()) < 1e-13


def test_adamw_steps():
    rng = np.random.default_rng(20)
    p, g = rng.normal(size=50), rng.normal(size=50)
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.95, 1e-8, 0.1
    p1, m1, v1 = oracle.adamw(p, g, np.zeros(50), np.zeros(50), lr, b1, b2, eps, wd, 1)
    # first step: mhat = g, vhat = g^2
    np.testing.assert_allclose(p1, p - lr * (g / (np.abs(g) + eps) + wd * p), atol=1e-15)
    g2 = rng.normal(size=50)
    p2, m2, v2 = oracle.adamw(p1, g2, m1, v1, lr, b1, b2, eps, wd, 2)
    m = b1 * (1 - b1) * g + (1 - b1) * g2
    v = b2 * (1 - b2) * g * g + (1 - b2) * g2 * g2
    np.testing.assert_allclose(m2, m, atol=1e-15)
    np.testing.assert_allclose(p2, p1 - lr * ((m / (1 - b1 ** 2)) / (np.sqrt(v / (1 - b2 ** 2)) + eps) + wd * p1),
                               atol=1e-15)
