"""Device buffers around the C ABI: a GPT-2 model ready to run forward passes
and decode steps on one GPU.

PyTorch only provides device memory and the stream here; every kernel that
touches the data is the CUDA library's, reached through `binding`.
"""
from __future__ import annotations

import torch

from . import binding as ab

# the probabilities' element type from the output tensor's dtype
_PROBS_TYPE = {torch.float32: ab.GPT2_PROBS_F32, torch.float16: ab.GPT2_PROBS_F16,
               torch.bfloat16: ab.GPT2_PROBS_BF16}


def probs_type(probs) -> int:
    return ab.GPT2_PROBS_F32 if probs is None else _PROBS_TYPE[probs.dtype]


class GPT2Model:
    """Parameters (fp32, plus the packed bf16 weights in GPT2_BF16 mode) and a
    workspace sized for batches of up to B sequences of up to T tokens."""

    def __init__(self, cfg, params, B: int, T: int, precision: int = ab.GPT2_BF16, device="cuda"):
        ab.load()
        self.cfg = cfg
        self.precision = precision
        self.device = torch.device(device)
        p = torch.as_tensor(params)
        n = ab.gpt2_num_parameters(cfg)
        if p.numel() != n:
            raise ValueError(f"parameter buffer has {p.numel()} values, the config needs {n}")
        self.params = p.to(self.device, dtype=torch.float32).contiguous()
        nbytes = ab.gpt2_packed_weights_size(cfg, precision)
        self.packed = torch.empty(nbytes, dtype=torch.uint8, device=self.device) if nbytes else None
        if self.packed is not None:
            ab.gpt2_prepare_weights(cfg, self.params, self.packed, nbytes, precision)
        self.B, self.T = B, T
        self.ws_bytes = max(ab.gpt2_workspace_size(cfg, B, T, precision),
                            ab.gpt2_workspace_size(cfg, B, 1, precision))
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)

    # ---------------------------------------------------------------- buffers
    def new_outputs(self, B: int, T: int, probs: bool = True, probs_dtype=torch.float32):
        Vp = self.cfg.padded_vocab_size
        shape = (B, T, Vp) if T is not None else (B, Vp)
        logits = torch.empty(shape, dtype=torch.float32, device=self.device)
        pr = torch.empty(shape, dtype=probs_dtype, device=self.device) if probs else None
        return logits, pr

    def new_kvcache(self, B: int):
        nbytes = ab.gpt2_kvcache_size(self.cfg, B, self.precision)
        return torch.zeros(nbytes, dtype=torch.uint8, device=self.device)

    def new_paged_kvcache(self, num_blocks: int, block_size: int):
        """A zeroed pool of num_blocks blocks of block_size positions."""
        nbytes = ab.gpt2_paged_kvcache_size(self.cfg, num_blocks, block_size, self.precision)
        return torch.zeros(nbytes, dtype=torch.uint8, device=self.device)

    # ----------------------------------------------------------------- calls
    def forward(self, tok, logits, probs=None, kvcache=None, stream=None):
        """probs (optional): fp32, fp16 or bf16, [B, T, Vp]."""
        B, T = tok.shape
        ab.gpt2_forward_ex(self.cfg, self.params, self.packed, tok, B, T, logits, probs, probs_type(probs), kvcache,
                           self.workspace, self.ws_bytes, self.precision, stream)

    def forward_profile(self, tok, logits, probs=None, stream=None) -> dict:
        B, T = tok.shape
        return ab.gpt2_forward_profile(self.cfg, self.params, self.packed, tok, B, T, logits, probs,
                                       self.workspace, self.ws_bytes, self.precision, stream,
                                       probs_type=probs_type(probs))

    def decode_step(self, kvcache, tok, pos: int, logits, probs=None, stream=None):
        B = tok.shape[0]
        ab.gpt2_decode_step(self.cfg, self.params, self.packed, kvcache, tok, B, pos, logits, probs,
                            self.workspace, self.ws_bytes, self.precision, stream)

    def prefill_paged(self, tok, logits, kv, probs=None, stream=None):
        """gpt2_forward writing positions [0, T) through the paged cache kv
        (a binding.GPT2PagedKVCache)."""
        B, T = tok.shape
        ab.gpt2_prefill_paged(self.cfg, self.params, self.packed, tok, B, T, logits, probs, kv, self.workspace,
                              self.ws_bytes, self.precision, stream)

    def decode_step_paged(self, kv, tok, pos, logits, probs=None, stream=None):
        """One decode step, sequence b at position pos[b] (a device int32
        tensor)."""
        B = tok.shape[0]
        ab.gpt2_decode_step_paged(self.cfg, self.params, self.packed, kv, tok, pos, B, logits, probs, self.workspace,
                                  self.ws_bytes, self.precision, stream)
