"""Static checks on the CUDA sources (no GPU, no compiler).

A kernel launched with the programmatic-stream-serialization attribute may
start while the kernel ahead of it on the stream still runs; it is correct
only if its body waits (griddepcontrol.wait, pdl_wait()) before it touches
what that kernel writes.  Every kernel that can get the attribute must
therefore contain pdl_wait(): the kernels passed to launch_pdl, and the two
GEMM kernels that set the attribute in their own launch configuration.

Every barrier wait is bounded in time and no kernel traps: the checks below
keep a lost arrival or a failed check from hanging or faulting the GPU."""
import os
import re

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "gpt_transformer_forward_gb300",
                    "csrc")


def _sources():
    out = {}
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh")):
            with open(os.path.join(CSRC, f)) as fh:
                out[f] = fh.read()
    return out


def _kernel_body(src, name):
    """Text of the body of __global__ kernel `name` (first definition)."""
    m = re.search(r"__global__[^;{]*?\b" + re.escape(name) + r"\s*\(", src, re.S)
    if m is None:
        return None
    i = src.index("{", m.end())
    depth = 0
    for j in range(i, len(src)):
        if src[j] == "{":
            depth += 1
        elif src[j] == "}":
            depth -= 1
            if depth == 0:
                return src[i:j + 1]
    raise AssertionError(f"unbalanced braces in {name}")


def _pdl_kernels(srcs):
    names = set()
    for text in srcs.values():
        for m in re.finditer(r"launch_pdl\(\s*([A-Za-z_][A-Za-z_0-9]*)", text):
            if m.group(1) != "void":  # the helper's own declaration
                names.add(m.group(1))
    for f, text in srcs.items():
        if f.endswith(".cu") and "cudaLaunchAttributeProgrammaticStreamSerialization" in text:
            for m in re.finditer(r"auto\s+kern\s*=\s*([A-Za-z_][A-Za-z_0-9]*)\s*<", text):
                names.add(m.group(1))
    return sorted(names)


def test_pdl_kernels_are_found():
    names = _pdl_kernels(_sources())
    for expected in ("gemm_skinny_kernel", "gemm_tc_kernel", "decode_attn_kernel", "argmax_kernel",
                     "residual_layernorm_kernel", "softmax_from_stats_kernel"):
        assert expected in names, names


@pytest.mark.parametrize("name", _pdl_kernels(_sources()))
def test_every_programmatic_launch_waits(name):
    srcs = _sources()
    bodies = [b for b in (_kernel_body(t, name) for t in srcs.values()) if b is not None]
    assert bodies, f"kernel {name} not found"
    for body in bodies:
        assert "pdl_wait()" in body, f"{name} can start early but never waits for the kernel ahead"
        # nothing global is touched before the wait except loads of data no
        # kernel writes (weights, older cache rows), which the kernel marks
        head = body[:body.index("pdl_wait()")]
        assert "__stcs" not in head and "atomic" not in head, name


def test_the_check_sees_a_missing_wait():
    # the checker itself, on a planted source: a kernel launched early
    # without a wait is reported
    src = ("__global__ void good_kernel(float* x) { pdl_wait(); x[0] = 1.f; }\n"
           "__global__ void __launch_bounds__(256) bad_kernel(float* x) { if (x) { x[0] = 1.f; } }\n"
           "void go(cudaStream_t s, float* x) { launch_pdl(good_kernel, 1, 1, 0, s, x); "
           "launch_pdl(bad_kernel, 1, 1, 0, s, x); }\n")
    assert _pdl_kernels({"planted.cu": src}) == ["bad_kernel", "good_kernel"]
    assert "pdl_wait()" in _kernel_body(src, "good_kernel")
    assert "pdl_wait()" not in _kernel_body(src, "bad_kernel")


# Every wait on an mbarrier gives up after a time limit (about a second),
# records GPT2_DEVERR_TIMEOUT and returns, so that a lost arrival cannot
# hang the GPU.  The waiting instructions therefore appear only inside the
# bounded helpers of common.cuh, and every endless loop there checks the
# clock.

def _loops(text):
    """Bodies of the `for (;;)` and `while (true)` loops of a source."""
    out = []
    for m in re.finditer(r"for\s*\(\s*;\s*;\s*\)|while\s*\(\s*(true|1)\s*\)", text):
        i = text.index("{", m.end())
        depth = 0
        for j in range(i, len(text)):
            if text[j] == "{":
                depth += 1
            elif text[j] == "}":
                depth -= 1
                if depth == 0:
                    out.append(text[i:j + 1])
                    break
    return out


def test_barrier_waits_only_in_the_bounded_helpers():
    srcs = _sources()
    for f, text in srcs.items():
        if f == "common.cuh":
            continue
        for word in ("mbarrier.try_wait", "mbarrier.test_wait"):
            assert word not in text, f"{f} waits on a barrier outside the bounded helpers ({word})"


def test_every_endless_loop_has_a_time_limit():
    for f, text in _sources().items():
        for body in _loops(text):
            assert re.search(r"globaltimer_ns\(\)\s*-\s*t0\s*>", body), f"{f}: an endless loop without a time limit"


def test_the_loop_check_sees_an_unbounded_spin():
    bad = "__device__ void f(volatile int* p) { for (;;) { if (*p) return; } }"
    assert _loops(bad) and not re.search(r"globaltimer_ns\(\)\s*-\s*t0\s*>", _loops(bad)[0])


def test_no_device_traps():
    # no trap instruction and no device assert (a failed one traps): errors
    # are reported through the device error word
    for f, text in _sources().items():
        assert "__trap" not in text and "trap;" not in text, f"{f} traps"
        assert not re.search(r"(?<![A-Za-z_])assert\s*\(", text), f"{f} has a device assert"
