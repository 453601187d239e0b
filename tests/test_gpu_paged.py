"""KV-cached decoding through a paged cache [NTU "KV Caching"]: blocks of a
shared pool found through a per-sequence block table, each sequence at its
own position.

- With a shuffled block table, paged decoding gives bitwise the logits of
  the dense cache (the arithmetic is the same; only where rows live
  differs), at 80 and 256 sequences: more than 64 rows, so the decode GEMMs
  run on the tensor-core tile kernel (one CTA, and CTA pairs past 128
  rows), not the small-M one.
- Ragged batches: 128 and 256 sequences with prompts of 1..40 tokens
  prefilled together (padded to 40), then decoded each at its own position,
  against the oracle's full forward pass of each sequence (teacher-forced).
- GPT-2 124M width, 128 sequences (fp16): sampled sequences against the
  oracle.
- Block-table entries and positions outside the cache are flagged on the
  device, not faulted."""
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


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def shuffled_table(B, max_blocks, num_blocks, seed):
    """Each sequence its own max_blocks distinct blocks, in shuffled order."""
    perm = np.random.default_rng(seed).permutation(num_blocks)[:B * max_blocks]
    return perm.reshape(B, max_blocks).astype(np.int32)


def paged(m, B, block_size, extra_blocks, seed):
    cfg = m.cfg
    max_blocks = -(-cfg.max_seq_len // block_size)
    num_blocks = B * max_blocks + extra_blocks
    pool = m.new_paged_kvcache(num_blocks, block_size)
    table = dev(shuffled_table(B, max_blocks, num_blocks, seed))
    return ab.paged_kv(pool, table, num_blocks, block_size, max_blocks), (pool, table)


@pytest.mark.parametrize("precision,B", [(ab.GPT2_FP16, 80), (ab.GPT2_FP32, 80), (ab.GPT2_FP16, 256)])
def test_paged_decode_equals_dense_bitwise(precision, B):
    # 80 rows: the tile GEMM's one-CTA form; 256 rows: its paired-CTA form
    cfg = inputs.TINY
    P, steps = 24, 8
    params = inputs.make_params(cfg, 120, "perturbed")
    tok = inputs.make_tokens(121, B, P + steps, cfg.vocab_size)
    m = GPT2Model(cfg, params, B, P, precision)
    dense = m.new_kvcache(B)
    kv, keep = paged(m, B, 16, 5, 122)
    lg_d, _ = m.new_outputs(B, P, probs=False)
    lg_p, _ = m.new_outputs(B, P, probs=False)
    m.forward(dev(tok[:, :P]), lg_d, kvcache=dense)
    m.prefill_paged(dev(tok[:, :P]), lg_p, kv)
    np.testing.assert_array_equal(host(lg_p), host(lg_d))
    for i in range(steps):
        a, pa = m.new_outputs(B, None)
        b, pb = m.new_outputs(B, None)
        m.decode_step(dense, dev(tok[:, P + i]), P + i, a, pa)
        pos = torch.full((B,), P + i, dtype=torch.int32, device="cuda")
        m.decode_step_paged(kv, dev(tok[:, P + i]), pos, b, pb)
        np.testing.assert_array_equal(host(b), host(a))
        np.testing.assert_array_equal(host(pb), host(pa))
    no_device_error()


@pytest.mark.parametrize("precision,block_size,B", [(ab.GPT2_FP16, 16, 128), (ab.GPT2_BF16, 16, 128),
                                                    (ab.GPT2_FP32, 16, 128), (ab.GPT2_FP16, 32, 128),
                                                    (ab.GPT2_FP32, 32, 128), (ab.GPT2_FP16, 16, 256)])
def test_paged_ragged_decode_matches_oracle(precision, block_size, B):
    cfg = inputs.TINY
    P, steps = 40, 16
    rng = np.random.default_rng(123)
    params = inputs.make_params(cfg, 124, "perturbed")
    tok = inputs.make_tokens(125, B, P + steps, cfg.vocab_size)
    lens = rng.integers(1, P + 1, size=B).astype(np.int32)
    m = GPT2Model(cfg, params, B, P, precision)
    kv, keep = paged(m, B, block_size, 3, 126)
    lg, _ = m.new_outputs(B, P, probs=False)
    m.prefill_paged(dev(tok[:, :P]), lg, kv)  # padded prompts: each sequence's later steps overwrite its padding
    got = np.zeros((B, steps, cfg.padded_vocab_size))
    for i in range(steps):
        pos = lens + i
        step_tok = tok[np.arange(B), pos]
        out, _ = m.new_outputs(B, None, probs=False)
        m.decode_step_paged(kv, dev(step_tok), dev(pos), out)
        got[:, i] = host(out)
    no_device_error()
    for b in range(B):
        n = int(lens[b]) + steps
        ref, _ = oracle.forward(cfg, params, tok[b:b + 1, :n], want_probs=False)
        assert_close(got[b], ref[0, lens[b]:n], atol=LOGIT_TOL[precision], what=f"sequence {b} (prompt {lens[b]})")


def test_paged_124m_width_128_sequences():
    w = inputs.WORKLOADS["gpt2-124m-decode"]
    cfg = w.cfg
    B, P, steps = 128, 32, 3
    params = inputs.make_params(cfg, w.weight_seed)
    tok = inputs.make_tokens(w.token_seed, B, P + steps, cfg.vocab_size)
    lens = np.random.default_rng(127).integers(8, P + 1, size=B).astype(np.int32)
    m = GPT2Model(cfg, params, B, P, ab.GPT2_FP16)
    kv, keep = paged(m, B, 64, 9, 128)
    lg, _ = m.new_outputs(B, P, probs=False)
    m.prefill_paged(dev(tok[:, :P]), lg, kv)
    got = np.zeros((B, steps, cfg.padded_vocab_size))
    for i in range(steps):
        pos = lens + i
        out, pr = m.new_outputs(B, None)
        m.decode_step_paged(kv, dev(tok[np.arange(B), pos]), dev(pos), out, pr)
        got[:, i] = host(out)
        np.testing.assert_allclose(host(pr)[:, :cfg.vocab_size].sum(-1), 1.0, atol=1e-4)
    no_device_error()
    for b in (0, 77, 127):
        n = int(lens[b]) + steps
        ref, _ = oracle.forward(cfg, params, tok[b:b + 1, :n], want_probs=False)
        assert_close(got[b], ref[0, lens[b]:n], atol=2e-2, what=f"sequence {b} (prompt {lens[b]})")


def test_paged_flags_bad_table_entries_and_positions():
    cfg = inputs.TINY
    B = 4
    m = GPT2Model(cfg, inputs.make_params(cfg, 130), B, 8, ab.GPT2_FP16)
    kv, (pool, table) = paged(m, B, 16, 0, 131)
    lg, _ = m.new_outputs(B, 8, probs=False)
    m.prefill_paged(dev(inputs.make_tokens(132, B, 8, cfg.vocab_size)), lg, kv)
    assert ab.gpt2_get_error() == 0
    out, _ = m.new_outputs(B, None, probs=False)
    table[2, 0] = kv.num_blocks  # outside the pool
    m.decode_step_paged(kv, dev(np.zeros(B, np.int32)), dev(np.full(B, 8, np.int32)), out)
    assert ab.gpt2_get_error() & ab.DEVERR_BLOCK
    pos = np.full(B, 8, np.int32)
    pos[1] = cfg.max_seq_len  # past every sequence's capacity
    table[2, 0] = 0
    m.decode_step_paged(kv, dev(np.zeros(B, np.int32)), dev(pos), out)
    assert ab.gpt2_get_error() & ab.DEVERR_POSITION
    assert ab.gpt2_get_error() == 0  # read and cleared; the device stays usable
