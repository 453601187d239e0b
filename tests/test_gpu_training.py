"""GPU parity of the training step (gpt2_forward_backward, gpt2_adamw)
against the oracle's loss gradient (pinned by finite differences and an
autograd composite) and AdamW.

Tolerances, from the arithmetic: fp32 throughout (GPT2_FP32): loss within
1e-5 relative, every gradient element within 1e-4 x the largest gradient
(sums of up to B*T products, each rounded at 2^-24, through the layers);
tf32 operands (GPT2_TF32, 10 stored mantissa bits: 2^-11 per operand):
loss within 1e-3 relative, gradients within 2e-2 x the largest gradient.
AdamW: fp32 against double, 1e-6 relative."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs

from gpu_helpers import assert_close, dev, host, need_gpu, no_device_error

pytestmark = pytest.mark.gpu
TOL = {ab.GPT2_FP32: (1e-5, 1e-4), ab.GPT2_TF32: (1e-3, 2e-2)}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def gpu_step(cfg, params, tok, tgt, precision):
    B, T = tok.shape
    wsz = ab.gpt2_train_workspace_size(cfg, B, T, precision)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    grads = torch.full((params.size,), float("nan"), dtype=torch.float32, device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    ab.gpt2_forward_backward(cfg, dev(params), grads, dev(tok), dev(tgt), B, T, loss, ws, wsz, precision)
    no_device_error()
    return float(host(loss)[0]), host(grads)


def check(cfg, params, tok, tgt, precision, what):
    loss, g = gpu_step(cfg, params, tok, tgt, precision)
    rl, rg = oracle.forward_backward(cfg, params, tok, tgt)
    lt, gt = TOL[precision]
    assert abs(loss - rl) <= lt * abs(rl), (what, loss, rl)
    assert np.isfinite(g).all()
    assert_close(g, rg, atol=gt * np.abs(rg).max(), what=f"{what} gradient")


@pytest.mark.parametrize("precision", [ab.GPT2_FP32, ab.GPT2_TF32])
@pytest.mark.parametrize("init", ["gpt2", "perturbed"])
def test_tiny_training_step(precision, init):
    cfg = inputs.TINY
    params = inputs.make_params(cfg, 21, init)
    tok = inputs.make_tokens(22, 2, 32, cfg.vocab_size)
    tgt = inputs.make_tokens(23, 2, 32, cfg.vocab_size)
    check(cfg, params, tok, tgt, precision, "tiny")


@pytest.mark.parametrize("precision", [ab.GPT2_FP32, ab.GPT2_TF32])
def test_ragged_sequence_length(precision):
    cfg = inputs.TINY
    params = inputs.make_params(cfg, 24, "perturbed")
    tok = inputs.make_tokens(25, 4, 37, cfg.vocab_size)  # 148 rows: ragged 64-row and 128-row tiles
    tgt = inputs.make_tokens(26, 4, 37, cfg.vocab_size)
    check(cfg, params, tok, tgt, precision, "ragged")


@pytest.mark.parametrize("precision", [ab.GPT2_FP32, ab.GPT2_TF32])
@pytest.mark.parametrize("T", [100, 150])
def test_head_size_64_ragged_tiles(precision, T):
    # head size 64: in tf32 mode attention forward and backward run on the
    # tensor cores (128-row tiles: T = 100 one ragged tile, 150 two)
    cfg = inputs.GPT2Config(max_seq_len=160, vocab_size=512, padded_vocab_size=512, num_layers=2, num_heads=2,
                            channels=128)
    params = inputs.make_params(cfg, 33, "perturbed")
    tok = inputs.make_tokens(34, 2, T, cfg.vocab_size)
    tgt = inputs.make_tokens(35, 2, T, cfg.vocab_size)
    check(cfg, params, tok, tgt, precision, f"hs64 T={T}")


def test_several_attention_units_per_cta_ragged():
    # head size 64 in tf32 mode, B=16 sequences of T=600: 3 attention units
    # per (sequence, head), the last with one query tile, 192 units on 152
    # CTAs (several per CTA), the backward's items likewise; 9600 rows, not
    # a multiple of the GEMM tiles (the residual and GELU epilogues)
    cfg = inputs.GPT2Config(max_seq_len=640, vocab_size=512, padded_vocab_size=512, num_layers=2, num_heads=4,
                            channels=256)
    params = inputs.make_params(cfg, 39, "perturbed")
    tok = inputs.make_tokens(40, 16, 600, cfg.vocab_size)
    tgt = inputs.make_tokens(41, 16, 600, cfg.vocab_size)
    check(cfg, params, tok, tgt, ab.GPT2_TF32, "B=16 T=600")


@pytest.mark.parametrize("precision", [ab.GPT2_FP32, ab.GPT2_TF32])
def test_124m_width_one_layer(precision):
    cfg = dataclasses.replace(inputs.GPT2_124M, num_layers=1)
    params = inputs.make_params(cfg, 27)
    tok = inputs.make_tokens(28, 1, 64, cfg.vocab_size)
    tgt = inputs.make_tokens(29, 1, 64, cfg.vocab_size)
    check(cfg, params, tok, tgt, precision, "124M width")


def test_adamw_matches_the_oracle():
    rng = np.random.default_rng(30)
    n = 100_003
    p, g1, g2 = rng.normal(size=n), rng.normal(size=n), rng.normal(size=n)
    p = p.astype(np.float32)
    P, M, Vv = dev(p), torch.zeros(n, dtype=torch.float32, device="cuda"), torch.zeros(n, dtype=torch.float32, device="cuda")
    hp = (3e-4, 0.9, 0.95, 1e-8, 0.1)
    ref_p, ref_m, ref_v = p.astype(np.float64), np.zeros(n), np.zeros(n)
    for t, g in ((1, g1), (2, g2)):
        g = g.astype(np.float32)
        ab.gpt2_adamw(P, dev(g), M, Vv, n, *hp, t)
        ref_p, ref_m, ref_v = oracle.adamw(ref_p, g, ref_m, ref_v, *hp, t)
    assert_close(host(P), ref_p, atol=1e-6 * np.abs(ref_p).max(), what="params after two steps")
    assert_close(host(M), ref_m, atol=1e-6, rtol=1e-6, what="m")
    assert_close(host(Vv), ref_v, atol=1e-7, rtol=1e-6, what="v")


def test_training_lowers_the_loss_and_is_repeatable():
    cfg = inputs.TINY
    params = inputs.make_params(cfg, 31)
    tok = inputs.make_tokens(32, 2, 32, cfg.vocab_size)
    tgt = np.roll(tok, -1, axis=1)  # next-token targets
    B, T = tok.shape
    wsz = ab.gpt2_train_workspace_size(cfg, B, T, ab.GPT2_FP32)
    ws = torch.empty(wsz, dtype=torch.uint8, device="cuda")
    P = dev(params)
    G = torch.empty_like(P)
    M, V2 = torch.zeros_like(P), torch.zeros_like(P)
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    tk, tg = dev(tok), dev(tgt)
    losses = []
    for t in range(1, 9):
        ab.gpt2_forward_backward(cfg, P, G, tk, tg, B, T, loss, ws, wsz, ab.GPT2_FP32)
        losses.append(float(host(loss)[0]))
        ab.gpt2_adamw(P, G, M, V2, P.numel(), 1e-3, 0.9, 0.95, 1e-8, 0.0, t)
    no_device_error()
    assert losses[-1] < losses[0] - 0.05, losses
    # every gradient element but the token embedding's (atomics) is bitwise
    # repeatable at the same parameters
    ab.gpt2_forward_backward(cfg, P, G, tk, tg, B, T, loss, ws, wsz, ab.GPT2_FP32)
    g1 = host(G).copy()
    ab.gpt2_forward_backward(cfg, P, G, tk, tg, B, T, loss, ws, wsz, ab.GPT2_FP32)
    g2 = host(G)
    n_wte = cfg.padded_vocab_size * cfg.channels
    np.testing.assert_array_equal(g1[n_wte:], g2[n_wte:])
    np.testing.assert_allclose(g1[:n_wte], g2[:n_wte], atol=1e-6 * np.abs(g1).max())


def test_split_k_weight_gradients():
    # 1024 tokens: the tf32 weight-gradient products (K = the tokens, 32
    # k-blocks) run with their K range split over four units each, partial
    # products summed in a fixed order; against the oracle, and bitwise
    # repeatable
    cfg = inputs.GPT2Config(max_seq_len=256, vocab_size=512, padded_vocab_size=512, num_layers=2, num_heads=4,
                            channels=256)
    params = inputs.make_params(cfg, 36, "perturbed")
    tok = inputs.make_tokens(37, 4, 256, cfg.vocab_size)
    tgt = inputs.make_tokens(38, 4, 256, cfg.vocab_size)
    check(cfg, params, tok, tgt, ab.GPT2_TF32, "split K")
    _, g1 = gpu_step(cfg, params, tok, tgt, ab.GPT2_TF32)
    _, g2 = gpu_step(cfg, params, tok, tgt, ab.GPT2_TF32)
    n_wte = cfg.padded_vocab_size * cfg.channels
    np.testing.assert_array_equal(g1[n_wte:], g2[n_wte:])
