"""The algorithmic cost model bench.py reports rooflines with, checked
against figures fixed independently of it: the whole-model FLOP count of a
forward pass (every weight matrix times every token, plus the causal
attention products), the parameter layout of the model, and the KV-cache
layout (one cached position = keys and values of every layer, head and
sequence)."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gpt_transformer_forward_gb300 import inputs  # noqa: E402


@pytest.mark.parametrize("B,tflop", [(4, 1.090), (16, 4.359)])
def test_forward_flops_match_whole_model_count(B, tflop):
    cfg, T = inputs.GPT2_124M, 1024
    C, L, NH, Vp = cfg.channels, cfg.num_layers, cfg.num_heads, cfg.padded_vocab_size
    N = B * T
    # every token through every weight matrix (4 C^2 + 8 C^2 per layer, the
    # tied head), 2 FLOPs per multiply-add; attention: QK^T and PV over the
    # T (T + 1) / 2 causal pairs per head
    matmul = 2 * N * (L * 12 * C * C + C * Vp)
    attention = L * B * NH * 2 * 2 * (C // NH) * T * (T + 1) // 2
    total = sum(f for f, _ in bench.stage_costs(cfg, B, T).values())
    assert total == matmul + attention
    assert abs(total / 1e12 - tflop) < 1e-3  # the published-sized figure for this shape


def test_decode_step_bytes_follow_the_cache_and_parameter_layouts():
    cfg = inputs.GPT2_124M
    C, L, maxT = cfg.channels, cfg.num_layers, cfg.max_seq_len
    B = 32
    # one more cached position: keys and values of every layer and sequence
    for act in (2, 4):
        step = bench.decode_step_bytes(cfg, B, 101, act) - bench.decode_step_bytes(cfg, B, 100, act)
        assert step == 2 * L * B * C * act
    # at position 0 (one cache row written, none read): the matrices of the
    # parameter layout (everything but the position table, biases and
    # LayerNorm parameters) in 16 bits, those small vectors in fp32, and the
    # token, embedding, logits and probability rows
    n_params = inputs.num_params(cfg)
    matrices = n_params - maxT * C - (L * 13 * C + 2 * C)
    small = (L * 13 * C + 2 * C) * 4
    rows = B * 4 + (B + 1) * C * 4 + 3 * B * cfg.padded_vocab_size * 4
    assert bench.decode_step_bytes(cfg, B, 0, 2) == 2 * matrices + small + 2 * L * B * C * 2 + rows
