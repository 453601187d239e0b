"""Thin Python binding of libgpt2fwd.so: the C ABI, name for name.

Argument marshalling only.  Pointer arguments accept a torch tensor (its
data_ptr), a raw integer address or None; `stream` accepts a torch.cuda.Stream,
a raw cudaStream_t integer or None (torch's current stream).  A negative
return code raises GPT2Error.  Every step of the forward pass runs in the
CUDA library; there is no Python or CPU fallback, and importing this module
fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re

from . import build as _build

GPT2_FP32, GPT2_TF32, GPT2_BF16, GPT2_FP16 = 0, 1, 2, 3
GPT2_PROBS_F32, GPT2_PROBS_F16, GPT2_PROBS_BF16 = 0, 1, 2
PRECISIONS = {"fp32": GPT2_FP32, "tf32": GPT2_TF32, "bf16": GPT2_BF16, "fp16": GPT2_FP16}

GPT2_OK = 0
ERRORS = {-1: "GPT2_ERR_ARG", -2: "GPT2_ERR_SHAPE", -3: "GPT2_ERR_ALIGN", -4: "GPT2_ERR_WORKSPACE",
          -5: "GPT2_ERR_CUDA", -6: "GPT2_ERR_DEVICE", -7: "GPT2_ERR_UNSUPPORTED"}
DEVERR_TOKEN, DEVERR_TIMEOUT, DEVERR_POSITION, DEVERR_BLOCK = 1, 2, 4, 8


class GPT2Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        detail = ""
        if code == -5:
            detail = ": " + _lib().gpt2_last_cuda_error().decode()
        super().__init__(f"{fn} returned {ERRORS.get(code, code)}{detail}")


class GPT2Config(ctypes.Structure):
    _fields_ = [("max_seq_len", ctypes.c_int), ("vocab_size", ctypes.c_int),
                ("padded_vocab_size", ctypes.c_int), ("num_layers", ctypes.c_int),
                ("num_heads", ctypes.c_int), ("channels", ctypes.c_int)]

    @classmethod
    def of(cls, cfg) -> "GPT2Config":
        if isinstance(cfg, cls):
            return cfg
        return cls(cfg.max_seq_len, cfg.vocab_size, cfg.padded_vocab_size, cfg.num_layers,
                   cfg.num_heads, cfg.channels)


class GPT2PagedKVCache(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("num_blocks", ctypes.c_int),
                ("block_size", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_CFG = ctypes.POINTER(GPT2Config)
_PKV = ctypes.POINTER(GPT2PagedKVCache)

# name -> (restype, argtypes), in the order of include/gpt2fwd.h
_SIGNATURES = {
    "encoder_forward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "layernorm_forward": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P]),
    "matmul_workspace_size": (_Z, [_I, _I, _I, _I]),
    "matmul_forward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _Z, _P]),
    "matmul_forward_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "attention_workspace_size": (_Z, [_I, _I, _I, _I]),
    "attention_forward": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "attention_backward_workspace_size": (_Z, [_I, _I, _I, _I, _I]),
    "attention_backward": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _Z, _P]),
    "gelu_forward": (_I, [_P, _P, _I, _P]),
    "residual_forward": (_I, [_P, _P, _P, _I, _P]),
    "softmax_forward": (_I, [_P, _P, _I, _I, _I, _P]),
    "softmax_forward_ex": (_I, [_P, _I, _P, _I, _I, _I, _P]),
    "gpt2_argmax": (_I, [_P, _P, _I, _I, _I, _P]),
    "gpt2_num_parameters": (_Z, [_CFG]),
    "gpt2_packed_weights_size": (_Z, [_CFG, _I]),
    "gpt2_prepare_weights": (_I, [_CFG, _P, _P, _Z, _I, _P]),
    "gpt2_workspace_size": (_Z, [_CFG, _I, _I, _I]),
    "gpt2_kvcache_size": (_Z, [_CFG, _I, _I]),
    "gpt2_forward": (_I, [_CFG, _P, _P, _P, _I, _I, _P, _P, _P, _P, _Z, _I, _P]),
    "gpt2_forward_ex": (_I, [_CFG, _P, _P, _P, _I, _I, _P, _P, _I, _P, _P, _Z, _I, _P]),
    "gpt2_decode_step": (_I, [_CFG, _P, _P, _P, _P, _I, _I, _P, _P, _P, _Z, _I, _P]),
    "gpt2_train_workspace_size": (_Z, [_CFG, _I, _I, _I]),
    "gpt2_forward_backward": (_I, [_CFG, _P, _P, _P, _P, _I, _I, _P, _P, _Z, _I, _P]),
    "gpt2_adamw": (_I, [_P, _P, _P, _P, _Z, ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                        ctypes.c_float, _I, _P]),
    "gpt2_paged_kvcache_size": (_Z, [_CFG, _I, _I, _I]),
    "gpt2_prefill_paged": (_I, [_CFG, _P, _P, _P, _I, _I, _P, _P, _PKV, _P, _Z, _I, _P]),
    "gpt2_decode_step_paged": (_I, [_CFG, _P, _P, _PKV, _P, _P, _I, _P, _P, _P, _Z, _I, _P]),
    "gpt2_forward_profile": (_I, [_CFG, _P, _P, _P, _I, _I, _P, _P, _I, _P, _Z, _I, _P, _P, _I]),
    "gpt2_get_error": (_I, [_P]),
    "gpt2_strerror": (ctypes.c_char_p, [_I]),
    "gpt2_last_cuda_error": (ctypes.c_char_p, []),
    "gpt2_diag_wait_timeout": (_I, [ctypes.c_longlong, _P, _P]),
}

_handle = None


def library_path() -> str:
    return _build.LIB


def _lib():
    global _handle
    if _handle is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"libgpt2fwd.so is not built ({path}); run "
                              "`python -m gpt_transformer_forward_gb300.build`")
        h = ctypes.CDLL(path)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _handle = h
    return _handle


def load(build_if_missing: bool = True):
    """Loads the library (building it first when asked and needed)."""
    if build_if_missing:
        _build.build()
    return _lib()


def header_functions() -> list:
    """Function names declared in include/gpt2fwd.h."""
    path = os.path.join(_build.INCLUDE, "gpt2fwd.h")
    with open(path) as f:
        return re.findall(r"^GPT2_API [^(]*?\b([a-z_0-9]+)\(", f.read(), flags=re.M)


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(fn: str, rc: int):
    if rc < 0:
        raise GPT2Error(fn, rc)
    return rc


def _cfg(cfg):
    return ctypes.byref(GPT2Config.of(cfg))


# --------------------------------------------------------------- the ABI
def encoder_forward(out, tok, wte, wpe, B, T, C, V, stream=None):
    _check("encoder_forward", _lib().encoder_forward(_ptr(out), _ptr(tok), _ptr(wte), _ptr(wpe), B, T, C, V,
                                                     _stream(stream)))


def layernorm_forward(out, mean, rstd, inp, w, b, N, C, stream=None):
    _check("layernorm_forward", _lib().layernorm_forward(_ptr(out), _ptr(mean), _ptr(rstd), _ptr(inp), _ptr(w),
                                                         _ptr(b), N, C, _stream(stream)))


def matmul_workspace_size(N, C, OC, precision) -> int:
    return _lib().matmul_workspace_size(N, C, OC, precision)


def matmul_forward(out, inp, W, bias, N, C, OC, precision, workspace=None, ws_bytes=0, stream=None):
    _check("matmul_forward", _lib().matmul_forward(_ptr(out), _ptr(inp), _ptr(W), _ptr(bias), N, C, OC, precision,
                                                   _ptr(workspace), ws_bytes, _stream(stream)))


def matmul_forward_noalloc(out, inp, W, bias, N, C, OC, precision, stream=None):
    """matmul_forward with its scratch in the library's fixed 16 MiB device
    array instead of a caller workspace (for callers that cannot allocate)."""
    _check("matmul_forward_noalloc", _lib().matmul_forward_noalloc(_ptr(out), _ptr(inp), _ptr(W), _ptr(bias), N, C,
                                                                   OC, precision, _stream(stream)))


def attention_workspace_size(B, T, C, precision) -> int:
    return _lib().attention_workspace_size(B, T, C, precision)


def attention_forward(out, qkv, B, T, C, NH, precision, workspace=None, ws_bytes=0, stream=None):
    _check("attention_forward", _lib().attention_forward(_ptr(out), _ptr(qkv), B, T, C, NH, precision,
                                                         _ptr(workspace), ws_bytes, _stream(stream)))


def attention_backward_workspace_size(B, T, C, NH, precision) -> int:
    return _lib().attention_backward_workspace_size(B, T, C, NH, precision)


def attention_backward(dqkv, dout, qkv, out, B, T, C, NH, precision, workspace=None, ws_bytes=0, stream=None):
    _check("attention_backward", _lib().attention_backward(_ptr(dqkv), _ptr(dout), _ptr(qkv), _ptr(out), B, T, C, NH,
                                                           precision, _ptr(workspace), ws_bytes, _stream(stream)))


def gelu_forward(out, inp, n, stream=None):
    _check("gelu_forward", _lib().gelu_forward(_ptr(out), _ptr(inp), n, _stream(stream)))


def residual_forward(out, a, b, n, stream=None):
    _check("residual_forward", _lib().residual_forward(_ptr(out), _ptr(a), _ptr(b), n, _stream(stream)))


def softmax_forward(probs, logits, N, V, Vp, stream=None):
    _check("softmax_forward", _lib().softmax_forward(_ptr(probs), _ptr(logits), N, V, Vp, _stream(stream)))


def softmax_forward_ex(probs, probs_type, logits, N, V, Vp, stream=None):
    _check("softmax_forward_ex", _lib().softmax_forward_ex(_ptr(probs), probs_type, _ptr(logits), N, V, Vp,
                                                           _stream(stream)))


def gpt2_argmax(next_tok, logits, B, V, Vp, stream=None):
    _check("gpt2_argmax", _lib().gpt2_argmax(_ptr(next_tok), _ptr(logits), B, V, Vp, _stream(stream)))


def gpt2_num_parameters(cfg) -> int:
    return _lib().gpt2_num_parameters(_cfg(cfg))


def gpt2_packed_weights_size(cfg, precision) -> int:
    return _lib().gpt2_packed_weights_size(_cfg(cfg), precision)


def gpt2_prepare_weights(cfg, params, packed, nbytes, precision, stream=None):
    _check("gpt2_prepare_weights", _lib().gpt2_prepare_weights(_cfg(cfg), _ptr(params), _ptr(packed), nbytes,
                                                               precision, _stream(stream)))


def gpt2_workspace_size(cfg, B, T, precision) -> int:
    return _lib().gpt2_workspace_size(_cfg(cfg), B, T, precision)


def gpt2_kvcache_size(cfg, B, precision) -> int:
    return _lib().gpt2_kvcache_size(_cfg(cfg), B, precision)


def gpt2_forward(cfg, params, packed, tok, B, T, logits, probs, kvcache, workspace, ws_bytes, precision,
                 stream=None):
    _check("gpt2_forward", _lib().gpt2_forward(_cfg(cfg), _ptr(params), _ptr(packed), _ptr(tok), B, T, _ptr(logits),
                                               _ptr(probs), _ptr(kvcache), _ptr(workspace), ws_bytes, precision,
                                               _stream(stream)))


def gpt2_forward_ex(cfg, params, packed, tok, B, T, logits, probs, probs_type, kvcache, workspace, ws_bytes,
                    precision, stream=None):
    _check("gpt2_forward_ex", _lib().gpt2_forward_ex(_cfg(cfg), _ptr(params), _ptr(packed), _ptr(tok), B, T,
                                                     _ptr(logits), _ptr(probs), probs_type, _ptr(kvcache),
                                                     _ptr(workspace), ws_bytes, precision, _stream(stream)))


def gpt2_decode_step(cfg, params, packed, kvcache, tok, B, pos, logits, probs, workspace, ws_bytes, precision,
                     stream=None):
    _check("gpt2_decode_step", _lib().gpt2_decode_step(_cfg(cfg), _ptr(params), _ptr(packed), _ptr(kvcache),
                                                       _ptr(tok), B, pos, _ptr(logits), _ptr(probs),
                                                       _ptr(workspace), ws_bytes, precision, _stream(stream)))


STAGES = ["encoder", "ln1", "qkv", "attention", "attproj", "ln2", "fc", "fcproj", "lnf", "lm_head", "softmax"]


def gpt2_train_workspace_size(cfg, B, T, precision) -> int:
    return _lib().gpt2_train_workspace_size(_cfg(cfg), B, T, precision)


def gpt2_forward_backward(cfg, params, grads, tok, targets, B, T, loss, workspace, ws_bytes, precision,
                          stream=None):
    _check("gpt2_forward_backward", _lib().gpt2_forward_backward(
        _cfg(cfg), _ptr(params), _ptr(grads), _ptr(tok), _ptr(targets), B, T, _ptr(loss), _ptr(workspace), ws_bytes,
        precision, _stream(stream)))


def gpt2_adamw(params, grads, m, v, n, lr, beta1, beta2, eps, weight_decay, t, stream=None):
    _check("gpt2_adamw", _lib().gpt2_adamw(_ptr(params), _ptr(grads), _ptr(m), _ptr(v), n, lr, beta1, beta2, eps,
                                           weight_decay, t, _stream(stream)))


def paged_kv(pool, block_table, num_blocks, block_size, max_blocks_per_seq) -> GPT2PagedKVCache:
    """The C struct describing a paged cache (pool and block_table: device
    tensors or addresses)."""
    return GPT2PagedKVCache(_ptr(pool), _ptr(block_table), num_blocks, block_size, max_blocks_per_seq)


def gpt2_paged_kvcache_size(cfg, num_blocks, block_size, precision) -> int:
    return _lib().gpt2_paged_kvcache_size(_cfg(cfg), num_blocks, block_size, precision)


def gpt2_prefill_paged(cfg, params, packed, tok, B, T, logits, probs, kv, workspace, ws_bytes, precision,
                       stream=None):
    _check("gpt2_prefill_paged", _lib().gpt2_prefill_paged(
        _cfg(cfg), _ptr(params), _ptr(packed), _ptr(tok), B, T, _ptr(logits), _ptr(probs),
        ctypes.byref(kv) if kv is not None else None, _ptr(workspace), ws_bytes, precision, _stream(stream)))


def gpt2_decode_step_paged(cfg, params, packed, kv, tok, pos, B, logits, probs, workspace, ws_bytes, precision,
                           stream=None):
    _check("gpt2_decode_step_paged", _lib().gpt2_decode_step_paged(
        _cfg(cfg), _ptr(params), _ptr(packed), ctypes.byref(kv) if kv is not None else None, _ptr(tok), _ptr(pos), B,
        _ptr(logits), _ptr(probs), _ptr(workspace), ws_bytes, precision, _stream(stream)))


def gpt2_forward_profile(cfg, params, packed, tok, B, T, logits, probs, workspace, ws_bytes, precision,
                         stream=None, probs_type=GPT2_PROBS_F32) -> dict:
    """Runs one forward pass with per-stage CUDA events; returns {stage: ms}."""
    ms = (ctypes.c_float * len(STAGES))()
    _check("gpt2_forward_profile", _lib().gpt2_forward_profile(
        _cfg(cfg), _ptr(params), _ptr(packed), _ptr(tok), B, T, _ptr(logits), _ptr(probs), probs_type,
        _ptr(workspace), ws_bytes, precision, _stream(stream), ctypes.cast(ms, ctypes.c_void_p), len(STAGES)))
    return dict(zip(STAGES, list(ms)))


def gpt2_get_error(stream=None) -> int:
    return _check("gpt2_get_error", _lib().gpt2_get_error(_stream(stream)))


def gpt2_strerror(code) -> str:
    return _lib().gpt2_strerror(code).decode()


def gpt2_last_cuda_error() -> str:
    return _lib().gpt2_last_cuda_error().decode()


def gpt2_diag_wait_timeout(limit_ns, gave_up, stream=None):
    """Runs the bounded-wait path once (see the header); gave_up: a device
    int32 tensor of one element."""
    _check("gpt2_diag_wait_timeout", _lib().gpt2_diag_wait_timeout(int(limit_ns), _ptr(gave_up), _stream(stream)))
