"""The C-ABI library builds, loads and exports every function the header
declares; its host-only entry points answer without a GPU (no compute call
is made here)."""
import ctypes

import pytest

from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import build, inputs


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ab.load(build_if_missing=False)


def test_every_declared_function_is_exported(lib):
    names = ab.header_functions()
    assert len(names) == 33
    for n in names:
        assert hasattr(lib, n), n
        assert n in ab._SIGNATURES, n
    assert set(ab._SIGNATURES) == set(names)


def test_parameter_count_matches_layout():
    for cfg in (inputs.TINY, inputs.GPT2_124M, inputs.GPT2_MEDIUM):
        assert ab.gpt2_num_parameters(cfg) == inputs.num_params(cfg)
    assert ab.gpt2_num_parameters(inputs.GPT2_124M) == 124475904


def test_sizes_are_consistent():
    cfg = inputs.GPT2_124M
    C, L, Vp, maxT = cfg.channels, cfg.num_layers, cfg.padded_vocab_size, cfg.max_seq_len
    packed = ab.gpt2_packed_weights_size(cfg, ab.GPT2_BF16)
    assert packed >= 2 * (Vp * C + L * 12 * C * C)
    assert ab.gpt2_packed_weights_size(cfg, ab.GPT2_FP32) == 0
    kv = ab.gpt2_kvcache_size(cfg, 32, ab.GPT2_BF16)
    assert kv == L * 2 * 32 * maxT * C * 2
    assert ab.gpt2_kvcache_size(cfg, 32, ab.GPT2_FP32) == 2 * kv
    ws16 = ab.gpt2_workspace_size(cfg, 16, 1024, ab.GPT2_BF16)
    ws32 = ab.gpt2_workspace_size(cfg, 16, 1024, ab.GPT2_FP32)
    N = 16 * 1024
    assert ws16 >= N * C * 4 + N * C * 2 * (1 + 3 + 1 + 4)
    assert ws32 > ws16
    assert ab.matmul_workspace_size(100, 768, 2304, ab.GPT2_BF16) >= 2 * (100 * 768 + 2304 * 768)
    assert ab.matmul_workspace_size(100, 768, 2304, ab.GPT2_TF32) == 0
    assert ab.attention_workspace_size(2, 64, 768, ab.GPT2_FP32) == 0


def test_invalid_configs_are_rejected():
    bad = ab.GPT2Config(1024, 50257, 50304, 12, 7, 768)   # C % NH != 0
    assert ab.gpt2_num_parameters(bad) == 0
    assert ab.gpt2_workspace_size(bad, 1, 1, ab.GPT2_BF16) == 0
    worse = ab.GPT2Config(1024, 50257, 50000, 12, 12, 768)  # Vp < V
    assert ab.gpt2_num_parameters(worse) == 0


def test_argument_errors_before_any_launch(lib):
    # null pointers and bad shapes return an error code before CUDA is touched
    assert lib.encoder_forward(None, None, None, None, 1, 1, 8, 1, None) == -1
    assert lib.softmax_forward(None, None, 1, 5, 4, None) == -1
    assert lib.softmax_forward_ex(None, ab.GPT2_PROBS_F16, None, 1, 5, 4, None) == -1
    # a probabilities type outside GPT2ProbsType (aligned, never dereferenced pointers)
    assert lib.softmax_forward_ex(256, 3, 256, 1, 4, 4, None) == -1
    assert lib.softmax_forward_ex(256, -1, 256, 1, 4, 4, None) == -1
    cfg = ab.GPT2Config.of(inputs.TINY)
    assert lib.gpt2_forward(ctypes.byref(cfg), None, None, None, 1, 1, None, None, None, None, 0, 2, None) == -1
    bad = ab.GPT2Config(64, 512, 512, 2, 3, 64)
    assert lib.gpt2_forward(ctypes.byref(bad), 16, None, 16, 1, 1, 16, None, None, 16, 0, 2, None) == -2
    assert lib.gpt2_forward_ex(ctypes.byref(cfg), 256, 256, 256, 1, 8, 256, 256, 5, None, 256, 1 << 30, 2,
                               None) == -1
    # T > maxT
    assert lib.gpt2_forward(ctypes.byref(cfg), 256, 256, 256, 1, 65, 256, None, None, 256, 1 << 30, 2,
                            None) == -2
    # misaligned logits pointer
    assert lib.gpt2_forward(ctypes.byref(cfg), 256, 256, 256, 1, 8, 260, None, None, 256, 1 << 30, 2,
                            None) == -3
    # decode position beyond maxT
    assert lib.gpt2_decode_step(ctypes.byref(cfg), 256, 256, 256, 256, 1, 64, 256, None, 256, 1 << 30, 2,
                                None) == -2
    assert ab.gpt2_strerror(-4).startswith("workspace")


def test_wait_timeout_diagnostic_checks_its_arguments_on_the_host(lib):
    # rejected before anything is launched, so no GPU is needed
    with pytest.raises(ab.GPT2Error) as e:
        ab.gpt2_diag_wait_timeout(10, None, stream=0)
    assert e.value.code == -1
    assert lib.gpt2_diag_wait_timeout(999, None, None) == -1
    assert lib.gpt2_diag_wait_timeout(2_000_000_000, None, None) == -1


def test_paged_calls_check_their_arguments_on_the_host(lib):
    cfg = inputs.TINY
    assert ab.gpt2_paged_kvcache_size(cfg, 10, 16, ab.GPT2_FP16) == cfg.num_layers * 2 * 10 * cfg.channels * 16 * 2
    assert ab.gpt2_paged_kvcache_size(cfg, 10, 24, ab.GPT2_FP16) == 0  # not a power of two
    assert ab.gpt2_paged_kvcache_size(cfg, 0, 16, ab.GPT2_FP16) == 0
    fake = 1 << 20  # an aligned address that is never dereferenced: every call below fails its checks first
    for bs, nb, mb, code in [(24, 8, 4, -1), (16, 0, 4, -1), (16, 8, 0, -1), (16, 8, 2000, -2)]:
        kv = ab.paged_kv(fake, fake, nb, bs, mb)
        with pytest.raises(ab.GPT2Error) as e:
            ab.gpt2_decode_step_paged(cfg, fake, fake, kv, fake, fake, 2, fake, None, fake, 1 << 20, ab.GPT2_FP16,
                                      stream=0)
        assert e.value.code == code, (bs, nb, mb)
    # a prompt longer than one sequence's blocks (2 blocks of 16 positions)
    kv = ab.paged_kv(fake, fake, 8, 16, 2)
    with pytest.raises(ab.GPT2Error) as e:
        ab.gpt2_prefill_paged(cfg, fake, fake, fake, 2, 40, fake, None, kv, fake, 1 << 20, ab.GPT2_FP16, stream=0)
    assert e.value.code == -2
    with pytest.raises(ab.GPT2Error) as e:
        ab.gpt2_decode_step_paged(cfg, fake, fake, None, fake, fake, 2, fake, None, fake, 1 << 20, ab.GPT2_FP16,
                                  stream=0)
    assert e.value.code == -1


def test_training_calls_check_their_arguments_on_the_host(lib):
    cfg = inputs.TINY
    assert ab.gpt2_train_workspace_size(cfg, 2, 32, ab.GPT2_BF16) == 0  # fp32 activations only
    assert ab.gpt2_train_workspace_size(cfg, 2, 32, ab.GPT2_FP32) > 0
    fake = 1 << 20
    with pytest.raises(ab.GPT2Error) as e:
        ab.gpt2_forward_backward(cfg, fake, fake, fake, fake, 2, 32, fake, fake, 1 << 30, ab.GPT2_FP16, stream=0)
    assert e.value.code == -7
    with pytest.raises(ab.GPT2Error) as e:  # tf32 needs B*T % 4 == 0
        ab.gpt2_forward_backward(cfg, fake, fake, fake, fake, 1, 3, fake, fake, 1 << 30, ab.GPT2_TF32, stream=0)
    assert e.value.code == -2
    with pytest.raises(ab.GPT2Error) as e:
        ab.gpt2_forward_backward(cfg, fake, fake, fake, fake, 2, 32, fake, fake, 16, ab.GPT2_FP32, stream=0)
    assert e.value.code == -4
    with pytest.raises(ab.GPT2Error) as e:
        ab.gpt2_adamw(fake, fake, fake, fake, 10, 1e-3, 0.9, 0.95, 1e-8, 0.0, 0, stream=0)  # t starts at 1
    assert e.value.code == -1


def test_attention_backward_precisions_on_the_host(lib):
    B, T, C, NH = 2, 300, 768, 12
    Tp = 384  # T rounded up to 128
    assert ab.attention_backward_workspace_size(B, T, C, NH, ab.GPT2_FP32) == 2 * ((B * NH * T * 4 + 255) // 256 * 256)
    w16 = ab.attention_backward_workspace_size(B, T, C, NH, ab.GPT2_BF16)
    assert w16 >= B * T * (3 * C + 2 * C) * 2 + 2 * B * NH * Tp * 4
    assert ab.attention_backward_workspace_size(B, T, C, NH, ab.GPT2_TF32) == w16
    assert ab.attention_backward_workspace_size(B, T, C, NH, ab.GPT2_FP16) == 0  # not supported
    assert ab.attention_backward_workspace_size(B, T, 256, 8, ab.GPT2_BF16) == 0  # head size 32
    fake = 1 << 20
    for precision, nh in ((ab.GPT2_FP16, NH), (ab.GPT2_BF16, 24)):
        with pytest.raises(ab.GPT2Error) as e:
            ab.attention_backward(fake, fake, fake, fake, B, T, C, nh, precision, fake, 1 << 30, stream=0)
        assert e.value.code == -7
    with pytest.raises(ab.GPT2Error) as e:  # workspace too small for the 16-bit path
        ab.attention_backward(fake, fake, fake, fake, B, T, C, NH, ab.GPT2_BF16, fake, w16 - 1, stream=0)
    assert e.value.code == -4
