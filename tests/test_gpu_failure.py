"""Failure detection on the device without a GPU fault: a bounded wait that
cannot complete gives up, records CANVAS_ERR_TIMEOUT in the status word,
returns, and leaves the context usable."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cv():
    import __graft_entry__
    __graft_entry__.build()
    import canvas_denoising_step_03_b300 as cv
    return cv


def test_wait_that_never_completes_reports_timeout_and_the_context_survives(cv):
    assert cv.canvas_device_status() == cv.CANVAS_OK           # nothing pending from earlier tests
    t0 = time.perf_counter()
    cv.canvas_selftest_wait_timeout()
    st = cv.canvas_device_status()                              # synchronises, reads and clears
    waited = time.perf_counter() - t0
    assert st == cv.CANVAS_ERR_TIMEOUT, cv.canvas_last_error()
    assert 1.0 < waited < 30.0, waited                          # the 2 s wait limit, not a hang
    assert cv.canvas_device_status() == cv.CANVAS_OK           # the word was cleared
    # the context still runs work correctly
    A = torch.randn(128, 256, device="cuda").to(torch.bfloat16)
    B = torch.randn(64, 256, device="cuda").to(torch.bfloat16)
    C = torch.empty(128, 64, device="cuda")
    cv.canvas_gemm_bf16(A, B, 0, C, 0, cv.workspace(cv.canvas_gemm_workspace_size(128, 64, 256)))
    assert cv.canvas_device_status() == cv.CANVAS_OK
    ref = A.double() @ B.double().T
    assert float((C.double() - ref).norm() / ref.norm()) < 1e-5
