"""The kernels' bounded-wait path, run on the device on purpose.

Every pipeline wait in the library's kernels gives up after a time limit,
sets the timeout bit of the device error word and lets the kernel return,
instead of spinning forever.  gpt2_diag_wait_timeout() makes one such wait
run out (an mbarrier nothing completes, a limit of a few milliseconds);
the test checks that the wait ends, that gpt2_get_error() reports the
timeout bit (and clears it), and that the next calls run normally and give
correct results."""
import time

import numpy as np
import pytest
import torch

import oracle
from gpt_transformer_forward_gb300 import binding as ab
from gpt_transformer_forward_gb300 import inputs
from gpt_transformer_forward_gb300.runner import GPT2Model

from gpu_helpers import assert_close, dev, host, need_gpu

pytestmark = pytest.mark.gpu
TIMEOUT_BIT = 2  # GPT2_DEVERR_TIMEOUT_BIT


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def test_wait_gives_up_sets_the_bit_and_the_device_stays_usable():
    assert ab.gpt2_get_error() == 0
    gave_up = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    ab.gpt2_diag_wait_timeout(5_000_000, gave_up)  # 5 ms
    word = ab.gpt2_get_error()
    elapsed = time.perf_counter() - t0
    assert word == TIMEOUT_BIT, word
    assert int(host(gave_up)[0]) == 1
    assert elapsed < 5.0  # ended by its own limit, far inside the pipelines' ~1 s
    assert ab.gpt2_get_error() == 0  # reading the word cleared it
    # the next work runs normally
    w = inputs.WORKLOADS["tiny"]
    params, tok = inputs.workload_inputs(w, "perturbed")
    m = GPT2Model(w.cfg, params, w.B, w.T, ab.GPT2_FP16)
    logits, probs = m.new_outputs(w.B, w.T)
    m.forward(dev(tok), logits, probs)
    assert ab.gpt2_get_error() == 0
    rl, rp = oracle.forward(w.cfg, params, tok)
    assert_close(host(logits), rl, atol=2e-2, what="logits after a timed-out wait")
    assert_close(host(probs), rp, atol=1e-3, what="probs after a timed-out wait")


def test_repeated_timeouts_each_report_once():
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(3):
        ab.gpt2_diag_wait_timeout(1_000_000, gave_up)
        assert ab.gpt2_get_error() == TIMEOUT_BIT
        assert int(host(gave_up)[0]) == 1
    assert ab.gpt2_get_error() == 0
