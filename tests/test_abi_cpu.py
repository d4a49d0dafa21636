"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, sizes workspaces, and rejects bad arguments on the host
(before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cv():
    import __graft_entry__
    __graft_entry__.build()
    import canvas_denoising_step_03_b300 as cv
    return cv


def header_symbols():
    with open(os.path.join(ROOT, "include", "canvas.h")) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(canvas_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(cv):
    syms = header_symbols()
    assert "canvas_attention" in syms and "canvas_sample" in syms
    for s in syms:
        assert hasattr(cv.lib, s), s
    assert sorted(cv.EXPORTED) == syms
    assert cv.canvas_version().startswith("canvas")


def test_workspace_sizes_are_positive_and_reject_bad_shapes(cv):
    assert cv.canvas_attention_workspace_size(cv.CANVAS_BF16, 1, 256, 2816, 16, 2, 512, 32768, 1) > 0
    assert cv.canvas_attention_workspace_size(cv.CANVAS_BF16, 1, 256, 2816, 16, 3, 512, 32768, 1) == 0
    assert cv.canvas_sample_workspace_size(cv.CANVAS_BF16, 256, 262144, 2816) > 256 * 262144 * 2
    assert cv.canvas_gemm_workspace_size(256, 2816, 262144) > 0
    assert cv.canvas_gemm_workspace_size(0, 1, 1) == 0


def test_host_validation_errors(cv):
    lib = cv.lib
    kv = cv.canvas_kv_cache()
    # null pointers -> CANVAS_ERR_ARG, message set, no CUDA work
    st = lib.canvas_attention(None, cv.CANVAS_BF16, 1, 16, 128, None, None, None, 2, 1, 64, None, None, 1e-6,
                              None, 0, ctypes.byref(kv), None, 0, 0, 1.0, 0, None, None, None, 0, None)
    assert st == cv.CANVAS_ERR_ARG
    assert "null" in cv.canvas_last_error()
    st = lib.canvas_sample(None, cv.CANVAS_BF16, 4, 512, None, 64, 0.3, 0, 0, 1.0, 0, 4, None, None, None, None,
                           None, None, None, None, 0, None, None, 0, None)
    assert st == cv.CANVAS_ERR_ARG
    st = lib.canvas_gemm_bf16(None, None, 0, None, 4, 8, 8, 0, None, 0, None)
    assert st == cv.CANVAS_ERR_ARG
    # unsupported K alignment, checked before the workspace
    fake = ctypes.c_void_p(256)
    st = lib.canvas_gemm_bf16(fake, fake, 0, fake, 4, 8, 12, 0, fake, 1 << 20, None)
    assert st == cv.CANVAS_ERR_UNSUPPORTED
    # workspace too small
    st = lib.canvas_gemm_bf16(fake, fake, 0, fake, 4, 8, 16, 0, fake, 16, None)
    assert st == cv.CANVAS_ERR_WORKSPACE


def test_misaligned_buffers_are_rejected_before_any_device_work(cv):
    lib = cv.lib
    good, bad = ctypes.c_void_p(256), ctypes.c_void_p(264)
    # GEMM entry points: A, B and C must be 16-byte aligned
    assert lib.canvas_gemm_bf16(good, good, 0, bad, 4, 8, 16, 0, good, 1 << 20, None) == cv.CANVAS_ERR_ARG
    assert "aligned" in cv.canvas_last_error()
    assert lib.canvas_gemm_bf16_to_bf16(good, bad, 0, good, 4, 8, 16, good, 1 << 20, None) == cv.CANVAS_ERR_ARG
    # the no-workspace GEMM: a C that is 4-byte but not 16-byte aligned (a
    # column-offset view) is rejected before the scratch lookup or any launch
    assert lib.canvas_gemm_bf16_noalloc(good, good, 0, ctypes.c_void_p(260), 128, 256, 4096, 0,
                                        None) == cv.CANVAS_ERR_ARG
    assert "aligned" in cv.canvas_last_error()
    # attention: x and out
    kv = cv.canvas_kv_cache()
    st = lib.canvas_attention(good, cv.CANVAS_BF16, 1, 16, 128, good, good, None, 2, 1, 64, good, good, 1e-6,
                              good, 1, ctypes.byref(kv), good, 0, 0, 1.0, 0, bad, None, good, 1 << 30, None)
    assert st == cv.CANVAS_ERR_ARG
    assert "aligned" in cv.canvas_last_error()
    # sampler: logits, probs_out, E and soft_emb
    st = lib.canvas_sample(good, cv.CANVAS_BF16, 4, 512, bad, 64, 0.3, 0, 0, 1.0, 0, 4, None, None, good, good,
                           good, good, None, None, cv.CANVAS_BF16, good, good, 1 << 30, None)
    assert st == cv.CANVAS_ERR_ARG
    assert "aligned" in cv.canvas_last_error()


def test_temperature_schedule_helper_matches_the_oracle(cv):
    # a host function: no device work
    from oracle import sampler as osamp
    for S, hi, lo in ((48, 1.5, 0.25), (12, 1.0, 0.1), (1, 0.7, 0.3), (2, 2.0, 1.0)):
        for s in range(S):
            want = osamp.temperature_schedule(s, S, hi, lo)
            assert abs(cv.canvas_temperature_at(s, S, hi, lo) - want) <= 1e-6 * want
