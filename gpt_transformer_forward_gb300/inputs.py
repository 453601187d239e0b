"""Seeded synthetic inputs for the GPT-2 forward pass.

This module holds no arithmetic of the forward pass itself.  It only produces
the bytes that both the CUDA library and the CPU oracle consume: a flat fp32
parameter buffer in the GPT-2 tensor order, and int32 token ids.

Random numbers come from SplitMix64 (Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used as a counter-based
generator: draw i of a stream with seed s is the SplitMix64 output function
applied to ``s + (i + 1) * 0x9E3779B97F4A7C15``.  Normals use the Box-Muller
transform on two uniforms.  Every value is produced on the host, so the GPU
and the oracle read identical bytes and no device-side generator is needed.

Workloads follow the synthetic configurations the method is measured on:
GPT-2 weights drawn N(0, 0.02), the two residual projections scaled by
1/sqrt(2L), LayerNorm gamma=1 and beta=0, biases 0, and token ids uniform in
[0, V).  The padded vocabulary rows [V, Vp) of the token embedding are zero.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)


@dataclasses.dataclass(frozen=True)
class GPT2Config:
    """Model hyper-parameters: maxT, V, Vp, L, NH, C (GPT-2 naming)."""

    max_seq_len: int
    vocab_size: int
    padded_vocab_size: int
    num_layers: int
    num_heads: int
    channels: int

    @property
    def head_size(self) -> int:
        return self.channels // self.num_heads


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    cfg: GPT2Config
    B: int
    T: int
    # decode-only fields: prompt length and number of single-token steps
    decode_steps: int = 0
    index: int = 0  # selects the weight / token seeds

    @property
    def weight_seed(self) -> int:
        return 1000 + self.index

    @property
    def token_seed(self) -> int:
        return 2000 + self.index


TINY = GPT2Config(max_seq_len=64, vocab_size=512, padded_vocab_size=512,
                  num_layers=2, num_heads=4, channels=64)
GPT2_124M = GPT2Config(max_seq_len=1024, vocab_size=50257, padded_vocab_size=50304,
                       num_layers=12, num_heads=12, channels=768)
GPT2_MEDIUM = GPT2Config(max_seq_len=1024, vocab_size=50257, padded_vocab_size=50304,
                         num_layers=24, num_heads=16, channels=1024)

WORKLOADS = {
    "tiny": Workload("tiny", TINY, B=2, T=32, index=0),
    "gpt2-124m-b4": Workload("gpt2-124m-b4", GPT2_124M, B=4, T=1024, index=1),
    "gpt2-124m-b16": Workload("gpt2-124m-b16", GPT2_124M, B=16, T=1024, index=2),
    "gpt2-124m-decode": Workload("gpt2-124m-decode", GPT2_124M, B=32, T=512,
                                 decode_steps=128, index=3),
    "gpt2-medium-b8": Workload("gpt2-medium-b8", GPT2_MEDIUM, B=8, T=1024, index=4),
}


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Draws [start, start+count) of the SplitMix64 stream with this seed."""
    i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + i * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _MIX1
        z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def normal_stream(seed: int, count: int, chunk: int = 1 << 24) -> np.ndarray:
    """`count` standard normals (float64), Box-Muller on draws (2i, 2i+1)."""
    out = np.empty(count, dtype=np.float64)
    scale = 1.0 / float(1 << 53)
    for s in range(0, count, chunk):
        n = min(chunk, count - s)
        z = splitmix64(seed, 2 * s, 2 * n)
        u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * scale  # (0, 1]
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * scale          # [0, 1)
        out[s:s + n] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
    return out


def param_shapes(cfg: GPT2Config):
    """The flat parameter buffer's tensors, in order, as (name, shape)."""
    C, L, Vp, maxT = cfg.channels, cfg.num_layers, cfg.padded_vocab_size, cfg.max_seq_len
    return [
        ("wte", (Vp, C)), ("wpe", (maxT, C)),
        ("ln1w", (L, C)), ("ln1b", (L, C)),
        ("qkvw", (L, 3 * C, C)), ("qkvb", (L, 3 * C)),
        ("attprojw", (L, C, C)), ("attprojb", (L, C)),
        ("ln2w", (L, C)), ("ln2b", (L, C)),
        ("fcw", (L, 4 * C, C)), ("fcb", (L, 4 * C)),
        ("fcprojw", (L, C, 4 * C)), ("fcprojb", (L, C)),
        ("lnfw", (C,)), ("lnfb", (C,)),
    ]


def num_params(cfg: GPT2Config) -> int:
    return sum(int(np.prod(s)) for _, s in param_shapes(cfg))


def param_views(cfg: GPT2Config, flat: np.ndarray) -> dict:
    """Named views into a flat parameter buffer (no copy)."""
    views, off = {}, 0
    for name, shape in param_shapes(cfg):
        n = int(np.prod(shape))
        views[name] = flat[off:off + n].reshape(shape)
        off += n
    assert off == flat.size
    return views


def make_params(cfg: GPT2Config, seed: int, init: str = "gpt2") -> np.ndarray:
    """Flat fp32 parameter buffer.

    init="gpt2": N(0, 0.02) matrices and embeddings, residual projections
    N(0, 0.02/sqrt(2L)), gamma=1, beta=0, biases 0.
    init="perturbed": as above but biases N(0, 0.02), gamma 1 + N(0, 0.1) and
    beta N(0, 0.02), so that every parameter tensor changes the output.
    """
    total = num_params(cfg)
    z = normal_stream(seed, total)
    flat = np.empty(total, dtype=np.float32)
    off = 0
    proj_std = 0.02 / math.sqrt(2 * cfg.num_layers)
    for name, shape in param_shapes(cfg):
        n = int(np.prod(shape))
        src = z[off:off + n]
        if name in ("attprojw", "fcprojw"):
            val = proj_std * src
        elif name in ("wte", "wpe", "qkvw", "fcw"):
            val = 0.02 * src
        elif name in ("ln1w", "ln2w", "lnfw"):
            val = 1.0 + (0.1 * src if init == "perturbed" else 0.0 * src)
        else:  # biases and LayerNorm betas
            val = 0.02 * src if init == "perturbed" else 0.0 * src
        flat[off:off + n] = val.astype(np.float32)
        off += n
    v = param_views(cfg, flat)
    v["wte"][cfg.vocab_size:, :] = 0.0
    return flat


def make_tokens(seed: int, B: int, T: int, V: int) -> np.ndarray:
    """int32 token ids, uniform in [0, V)."""
    z = splitmix64(seed, 0, B * T)
    return (z % np.uint64(V)).astype(np.int32).reshape(B, T)


def make_normal(seed: int, shape, std: float = 1.0, dtype=np.float32) -> np.ndarray:
    """A seeded normal array, for the single-kernel tests."""
    n = int(np.prod(shape))
    return (std * normal_stream(seed, n)).astype(dtype).reshape(shape)


def on_grid(a: np.ndarray, fmt: str) -> np.ndarray:
    """float32 copy of `a` with every value rounded (to nearest, ties to even)
    onto the grid of a narrower format, "bf16", "fp16" or "tf32", so that a
    conversion to that format is exact.  Test-input preparation only."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    if fmt == "fp16":
        return a.astype(np.float16).astype(np.float32)
    drop = {"bf16": 16, "tf32": 13}[fmt]  # low mantissa bits removed
    u = a.view(np.uint32).astype(np.uint64)
    half = np.uint64(1 << (drop - 1))
    lsb = (u >> np.uint64(drop)) & np.uint64(1)
    u = ((u + half - np.uint64(1) + lsb) >> np.uint64(drop)) << np.uint64(drop)
    return u.astype(np.uint32).view(np.float32)


def workload_inputs(w: Workload, init: str = "gpt2"):
    """(params, tokens) for a named workload."""
    params = make_params(w.cfg, w.weight_seed, init)
    tokens = make_tokens(w.token_seed, w.B, w.T, w.cfg.vocab_size)
    return params, tokens
