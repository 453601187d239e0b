"""Pins of the oracle's whole forward pass and decode step (no GPU needed).

Invariants that hold for any correct GPT-2 forward pass (causality, batch
independence, a closed form when every block is the identity, KV-cached
decode equal to recomputation), plus an independent composite written with
PyTorch float64 library operators (layer_norm, linear, scaled_dot_product
attention with its own causal mask, tanh-GELU, softmax).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gpt_transformer_forward_gb300 import inputs

CFG = inputs.TINY


@pytest.fixture(scope="module")
def tiny():
    p = inputs.make_params(CFG, 101, "perturbed")
    tok = inputs.make_tokens(102, 3, 40, CFG.vocab_size)
    return p, tok


def torch_gpt2(cfg, params, tok):
    """A composite of PyTorch float64 operators, independent of the C oracle."""
    v = {k: torch.from_numpy(a.astype(np.float64)) for k, a in inputs.param_views(cfg, params).items()}
    C, NH = cfg.channels, cfg.num_heads
    hs = C // NH
    B, T = tok.shape
    t = torch.from_numpy(tok.astype(np.int64))
    x = F.embedding(t, v["wte"]) + v["wpe"][:T]
    for l in range(cfg.num_layers):
        h = F.layer_norm(x, (C,), v["ln1w"][l], v["ln1b"][l], eps=1e-5)
        qkv = F.linear(h, v["qkvw"][l], v["qkvb"][l])
        q, k, vv = qkv.split(C, dim=-1)
        q, k, vv = (z.view(B, T, NH, hs).transpose(1, 2) for z in (q, k, vv))
        a = F.scaled_dot_product_attention(q, k, vv, is_causal=True)
        a = a.transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(a, v["attprojw"][l], v["attprojb"][l])
        h = F.layer_norm(x, (C,), v["ln2w"][l], v["ln2b"][l], eps=1e-5)
        u = F.gelu(F.linear(h, v["fcw"][l], v["fcb"][l]), approximate="tanh")
        x = x + F.linear(u, v["fcprojw"][l], v["fcprojb"][l])
    h = F.layer_norm(x, (C,), v["lnfw"], v["lnfb"], eps=1e-5)
    logits = h @ v["wte"].T
    probs = torch.zeros_like(logits)
    probs[..., :cfg.vocab_size] = torch.softmax(logits[..., :cfg.vocab_size], dim=-1)
    return logits.numpy(), probs.numpy()


def test_forward_matches_torch_composite(tiny):
    p, tok = tiny
    lg, pr = oracle.forward(CFG, p, tok)
    rl, rp = torch_gpt2(CFG, p, tok)
    np.testing.assert_allclose(lg, rl, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(pr, rp, rtol=1e-10, atol=1e-14)


def test_forward_probs_rows(tiny):
    p, tok = tiny
    lg, pr = oracle.forward(CFG, p, tok)
    np.testing.assert_allclose(pr.sum(-1), 1.0, atol=1e-13)
    assert (pr >= 0).all()


def test_forward_padded_vocab():
    cfg = inputs.GPT2Config(max_seq_len=16, vocab_size=100, padded_vocab_size=128,
                            num_layers=1, num_heads=2, channels=32)
    p = inputs.make_params(cfg, 103, "perturbed")
    tok = inputs.make_tokens(104, 2, 9, cfg.vocab_size)
    lg, pr = oracle.forward(cfg, p, tok)
    assert (lg[..., 100:] == 0).all()   # zero embedding rows give zero logits
    assert (pr[..., 100:] == 0).all()
    np.testing.assert_allclose(pr.sum(-1), 1.0, atol=1e-13)


def test_forward_is_causal(tiny):
    p, tok = tiny
    lg, _ = oracle.forward(CFG, p, tok, want_probs=False)
    t0 = 17
    pert = tok.copy()
    pert[:, t0 + 1:] = (pert[:, t0 + 1:] + 7) % CFG.vocab_size
    lg2, _ = oracle.forward(CFG, p, pert, want_probs=False)
    np.testing.assert_array_equal(lg[:, :t0 + 1], lg2[:, :t0 + 1])
    assert np.abs(lg[:, t0 + 1:] - lg2[:, t0 + 1:]).max() > 1e-3


def test_forward_batch_independence(tiny):
    p, tok = tiny
    lg, _ = oracle.forward(CFG, p, tok, want_probs=False)
    perm = [2, 0, 1]
    lg2, _ = oracle.forward(CFG, p, tok[perm], want_probs=False)
    np.testing.assert_array_equal(lg2, lg[perm])
    one, _ = oracle.forward(CFG, p, tok[1:2], want_probs=False)
    np.testing.assert_array_equal(one[0], lg[1])


def test_forward_identity_blocks_closed_form():
    # all block matrices and biases zero: every sublayer adds exactly zero
    p = inputs.make_params(CFG, 105, "perturbed")
    v = inputs.param_views(CFG, p)
    for name in ("qkvw", "qkvb", "attprojw", "attprojb", "fcw", "fcb", "fcprojw", "fcprojb"):
        v[name][...] = 0.0
    tok = inputs.make_tokens(106, 2, 13, CFG.vocab_size)
    lg, _ = oracle.forward(CFG, p, tok, want_probs=False)
    wte = torch.from_numpy(v["wte"].astype(np.float64))
    x = wte[torch.from_numpy(tok.astype(np.int64))] + torch.from_numpy(v["wpe"][:13].astype(np.float64))
    mu = x.mean(-1, keepdim=True)
    var = ((x - mu) ** 2).mean(-1, keepdim=True)
    h = (x - mu) / torch.sqrt(var + 1e-5) * torch.from_numpy(v["lnfw"].astype(np.float64)) \
        + torch.from_numpy(v["lnfb"].astype(np.float64))
    np.testing.assert_allclose(lg, (h @ wte.T).numpy(), rtol=1e-11, atol=1e-12)


def test_decode_equals_full_recompute(tiny):
    p, tok = tiny
    B, T = tok.shape
    P = 23
    full, _ = oracle.forward(CFG, p, tok, want_probs=False)
    _, _, cache = oracle.forward(CFG, p, tok[:, :P], want_probs=False, with_cache=True)
    for pos in range(P, T):
        step = oracle.decode_step(CFG, p, cache, tok[:, pos], pos)
        np.testing.assert_allclose(step, full[:, pos], rtol=1e-11, atol=1e-12)


def test_decode_from_empty_cache(tiny):
    p, tok = tiny
    B = tok.shape[0]
    shape = (CFG.num_layers, B, CFG.num_heads, CFG.max_seq_len, CFG.channels // CFG.num_heads)
    cache = (np.zeros(shape), np.zeros(shape))
    full, _ = oracle.forward(CFG, p, tok[:, :6], want_probs=False)
    for pos in range(6):
        step = oracle.decode_step(CFG, p, cache, tok[:, pos], pos)
        np.testing.assert_allclose(step, full[:, pos], rtol=1e-11, atol=1e-12)


def test_forward_cache_contents(tiny):
    # the cached keys/values are the QKV projection's key and value columns
    p, tok = tiny
    _, _, (kc, vc) = oracle.forward(CFG, p, tok[:, :5], want_probs=False, with_cache=True)
    v = inputs.param_views(CFG, p)
    x = oracle.encoder(tok[:, :5], v["wte"], v["wpe"])
    h, _, _ = oracle.layernorm(x, v["ln1w"][0], v["ln1b"][0])
    qkv = oracle.matmul(h, v["qkvw"][0], v["qkvb"][0])
    C, NH = CFG.channels, CFG.num_heads
    hs = C // NH
    k = qkv[..., C:2 * C].reshape(3, 5, NH, hs).transpose(0, 2, 1, 3)
    vv = qkv[..., 2 * C:].reshape(3, 5, NH, hs).transpose(0, 2, 1, 3)
    np.testing.assert_allclose(kc[0, :, :, :5], k, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(vc[0, :, :, :5], vv, rtol=1e-12, atol=1e-13)
    assert (kc[:, :, :, 5:] == 0).all()
