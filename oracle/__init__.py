"""Python access to the double-precision CPU oracle of the GPT-2 forward pass.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never reaches it, and it imports nothing from the CUDA library: the two share
only the seeded input generator, which holds none of the method's arithmetic.

The arithmetic lives in ``gpt2_oracle.c`` (plain C, double precision); this
module compiles it with gcc on first use and marshals numpy arrays through
ctypes.  All outputs are float64 numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gpt2_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


class OracleConfig(ctypes.Structure):
    _fields_ = [("max_seq_len", ctypes.c_int), ("vocab_size", ctypes.c_int),
                ("padded_vocab_size", ctypes.c_int), ("num_layers", ctypes.c_int),
                ("num_heads", ctypes.c_int), ("channels", ctypes.c_int)]


def build(force: bool = False) -> str:
    """Compiles the oracle with gcc (OpenMP on) into oracle/_build."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            _lib.oracle_num_params.restype = ctypes.c_size_t
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def config(cfg) -> OracleConfig:
    return OracleConfig(cfg.max_seq_len, cfg.vocab_size, cfg.padded_vocab_size,
                        cfg.num_layers, cfg.num_heads, cfg.channels)


def num_params(cfg) -> int:
    c = config(cfg)
    return int(lib().oracle_num_params(ctypes.byref(c)))


# ----------------------------------------------------------- single steps
def encoder(tok, wte, wpe) -> np.ndarray:
    tok, wte, wpe = _i32(tok), _f32(wte), _f32(wpe)
    B, T = tok.shape
    C = wte.shape[1]
    out = np.empty((B, T, C), dtype=np.float64)
    lib().oracle_encoder(_p(out), _p(tok), _p(wte), _p(wpe), B, T, C)
    return out


def layernorm(x, w, b):
    x = _f64(x)
    C = x.shape[-1]
    N = x.size // C
    w, b = _f32(w), _f32(b)
    out = np.empty_like(x)
    mean = np.empty(N, dtype=np.float64)
    rstd = np.empty(N, dtype=np.float64)
    lib().oracle_layernorm(_p(out), _p(mean), _p(rstd), _p(x), _p(w), _p(b), N, C)
    return out, mean.reshape(x.shape[:-1]), rstd.reshape(x.shape[:-1])


def matmul(x, W, bias=None) -> np.ndarray:
    """out = x W^T + bias with W [OC, C]; W and bias are taken in double."""
    x = _f64(x)
    W = _f64(W)
    OC, C = W.shape
    N = x.size // C
    out = np.empty(x.shape[:-1] + (OC,), dtype=np.float64)
    bias64 = _f64(bias) if bias is not None else None
    lib().oracle_matmul_f64w(_p(out), _p(x), _p(W), _p(bias64) if bias64 is not None else None,
                             N, C, OC)
    return out


def attention(qkv, NH: int) -> np.ndarray:
    """Algorithm 0 causal attention; qkv [B, T, 3C] -> [B, T, C]."""
    qkv = _f64(qkv)
    B, T, C3 = qkv.shape
    C = C3 // 3
    out = np.empty((B, T, C), dtype=np.float64)
    lib().oracle_attention(_p(out), _p(qkv), B, T, C, NH)
    return out


def attention_online(qkv, NH: int, Br: int, Bc: int) -> np.ndarray:
    """Algorithm 1 (tiled, online softmax) recompute of the same attention."""
    qkv = _f64(qkv)
    B, T, C3 = qkv.shape
    C = C3 // 3
    out = np.empty((B, T, C), dtype=np.float64)
    lib().oracle_attention_online(_p(out), _p(qkv), B, T, C, NH, Br, Bc)
    return out


def attention_backward(qkv, dout, NH: int) -> np.ndarray:
    """Backward of Algorithm 0 causal attention: dqkv [B, T, 3C] (dQ, dK,
    dV in the Q, K, V column blocks) for dL/dO = dout [B, T, C]."""
    qkv, dout = _f64(qkv), _f64(dout)
    B, T, C3 = qkv.shape
    C = C3 // 3
    dqkv = np.empty_like(qkv)
    lib().oracle_attention_backward(_p(dqkv), _p(dout), _p(qkv), B, T, C, NH)
    return dqkv


def attention_backward_online(qkv, dout, out, NH: int, Br: int, Bc: int) -> np.ndarray:
    """The tiled (Algorithm 1) backward, recomputing the attention matrix
    block by block from row statistics; out = the forward's output."""
    qkv, dout, out = _f64(qkv), _f64(dout), _f64(out)
    B, T, C3 = qkv.shape
    C = C3 // 3
    dqkv = np.empty_like(qkv)
    lib().oracle_attention_backward_online(_p(dqkv), _p(dout), _p(qkv), _p(out), B, T, C, NH, Br, Bc)
    return dqkv


def gelu(x) -> np.ndarray:
    x = _f64(x)
    out = np.empty_like(x)
    lib().oracle_gelu(_p(out), _p(x), x.size)
    return out


def residual(a, b) -> np.ndarray:
    a, b = _f64(a), _f64(b)
    out = np.empty_like(a)
    lib().oracle_residual(_p(out), _p(a), _p(b), a.size)
    return out


def softmax(logits, V: int) -> np.ndarray:
    logits = _f64(logits)
    Vp = logits.shape[-1]
    N = logits.size // Vp
    out = np.empty_like(logits)
    lib().oracle_softmax(_p(out), _p(logits), N, V, Vp)
    return out


def argmax(logits, V: int) -> np.ndarray:
    logits = _f64(logits)
    Vp = logits.shape[-1]
    B = logits.size // Vp
    out = np.empty(B, dtype=np.int32)
    lib().oracle_argmax(_p(out), _p(logits), B, V, Vp)
    return out


# ------------------------------------------------------- the forward pass
def hidden(cfg, params, tok, with_cache: bool = False):
    """Final LayerNorm output [B, T, C] (and, optionally, the KV cache)."""
    params, tok = _f32(params), _i32(tok)
    assert params.size == num_params(cfg)
    B, T = tok.shape
    C = cfg.channels
    c = config(cfg)
    h = np.empty((B, T, C), dtype=np.float64)
    kc = vc = None
    if with_cache:
        shape = (cfg.num_layers, B, cfg.num_heads, cfg.max_seq_len, C // cfg.num_heads)
        kc = np.zeros(shape, dtype=np.float64)
        vc = np.zeros(shape, dtype=np.float64)
    lib().oracle_gpt2_hidden(ctypes.byref(c), _p(params), _p(tok), B, T, _p(h),
                             _p(kc) if kc is not None else None,
                             _p(vc) if vc is not None else None)
    return (h, kc, vc) if with_cache else h


def lm_head(cfg, params, h) -> np.ndarray:
    params, h = _f32(params), _f64(h)
    N = h.size // cfg.channels
    c = config(cfg)
    out = np.empty(h.shape[:-1] + (cfg.padded_vocab_size,), dtype=np.float64)
    lib().oracle_lm_head(ctypes.byref(c), _p(params), _p(h), N, _p(out))
    return out


def forward(cfg, params, tok, want_probs: bool = True, with_cache: bool = False):
    """logits [B, T, Vp], probs (or None) and, optionally, (kcache, vcache)."""
    params, tok = _f32(params), _i32(tok)
    assert params.size == num_params(cfg)
    B, T = tok.shape
    c = config(cfg)
    logits = np.empty((B, T, cfg.padded_vocab_size), dtype=np.float64)
    probs = np.empty_like(logits) if want_probs else None
    kc = vc = None
    if with_cache:
        shape = (cfg.num_layers, B, cfg.num_heads, cfg.max_seq_len, cfg.channels // cfg.num_heads)
        kc = np.zeros(shape, dtype=np.float64)
        vc = np.zeros(shape, dtype=np.float64)
    lib().oracle_gpt2_forward(ctypes.byref(c), _p(params), _p(tok), B, T, _p(logits),
                              _p(probs) if probs is not None else None,
                              _p(kc) if kc is not None else None,
                              _p(vc) if vc is not None else None)
    if with_cache:
        return logits, probs, (kc, vc)
    return logits, probs


def decode_step(cfg, params, cache, tok, pos: int, want_probs: bool = False):
    """One KV-cached step; cache = (kcache, vcache) is updated in place."""
    params, tok = _f32(params), _i32(tok)
    kc, vc = cache
    assert kc.flags.c_contiguous and kc.dtype == np.float64
    B = tok.size
    c = config(cfg)
    logits = np.empty((B, cfg.padded_vocab_size), dtype=np.float64)
    probs = np.empty_like(logits) if want_probs else None
    lib().oracle_gpt2_decode_step(ctypes.byref(c), _p(params), _p(kc), _p(vc), _p(tok), B, pos,
                                  _p(logits), _p(probs) if probs is not None else None)
    return (logits, probs) if want_probs else logits


# ----------------------------------------------------------- training step
def matmul_backward(dout, inp, W):
    """y = x W^T + b: (dx, dW, db)."""
    dout, inp, W = _f64(dout), _f64(inp), _f32(W)
    OC, C = W.shape
    N = inp.size // C
    dinp = np.empty(inp.shape, dtype=np.float64)
    dW = np.zeros((OC, C), dtype=np.float64)
    db = np.zeros(OC, dtype=np.float64)
    lib().oracle_matmul_backward(_p(dinp), _p(dW), _p(db), _p(dout), _p(inp), _p(W), N, C, OC)
    return dinp, dW, db


def layernorm_backward(dout, x, w, mean, rstd):
    """(dx, dw, db) of LayerNorm, with the forward's mean and rstd."""
    dout, x, w, mean, rstd = _f64(dout), _f64(x), _f32(w), _f64(mean), _f64(rstd)
    C = x.shape[-1]
    N = x.size // C
    dx = np.empty_like(x)
    dw = np.zeros(C, dtype=np.float64)
    db = np.zeros(C, dtype=np.float64)
    lib().oracle_layernorm_backward(_p(dx), _p(dw), _p(db), _p(dout), _p(x), _p(w), _p(mean), _p(rstd), N, C)
    return dx, dw, db


def gelu_backward(x, dout) -> np.ndarray:
    x, dout = _f64(x), _f64(dout)
    out = np.empty_like(x)
    lib().oracle_gelu_backward(_p(out), _p(x), _p(dout), x.size)
    return out


def forward_backward(cfg, params, tok, targets):
    """(mean cross-entropy loss, gradient [num_params] float64)."""
    params, tok, targets = _f32(params), _i32(tok), _i32(targets)
    B, T = tok.shape
    c = config(cfg)
    grads = np.empty(num_params(cfg), dtype=np.float64)
    loss = ctypes.c_double()
    lib().oracle_gpt2_forward_backward(ctypes.byref(c), _p(params), _p(tok), _p(targets), B, T, _p(grads),
                                       ctypes.byref(loss))
    return loss.value, grads


def adamw(p, g, m, v, lr, b1, b2, eps, wd, t):
    """One AdamW step on float64 copies; returns (p, m, v)."""
    p, g, m, v = _f64(p).copy(), _f64(g), _f64(m).copy(), _f64(v).copy()
    lib().oracle_adamw(_p(p), _p(g), _p(m), _p(v), ctypes.c_size_t(p.size), ctypes.c_double(lr),
                       ctypes.c_double(b1), ctypes.c_double(b2), ctypes.c_double(eps), ctypes.c_double(wd), t)
    return p, m, v
