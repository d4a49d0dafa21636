"""canvas_gemm_bf16_noalloc: the GEMM entry point for callers that cannot
hand the library a device workspace (their host application owns all device
memory, or they must not allocate after start-up).  Its split-K scratch is a
static device array inside the library.

Checked through the C ABI against canvas_gemm_bf16 (the workspace entry
point) on the same operands, with the GEMM tests' tolerance, on two calls in a
row -- the second call reuses the scratch the first one left behind.  This
file is collected last on purpose.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cv():
    import __graft_entry__
    __graft_entry__.build()
    import canvas_denoising_step_03_b300 as cv
    return cv


def _operands(M, N, K, b_layout, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    shape = (N, K) if b_layout == 0 else (K, N)
    B = torch.randn(*shape, device="cuda", generator=g).to(torch.bfloat16)
    C0 = torch.randn(M, N, device="cuda", generator=g)
    return A, B, C0


def _compare(cv, M, N, K, b_layout, accumulate, seed):
    A, B, C0 = _operands(M, N, K, b_layout, seed)
    want = C0.clone()
    ws = cv.workspace(cv.canvas_gemm_workspace_size(M, N, K))
    cv.canvas_gemm_bf16(A, B, b_layout, want, accumulate, ws)
    got = C0.clone() if accumulate else torch.full((M, N), float("nan"), device="cuda")
    cv.canvas_gemm_bf16_noalloc(A, B, b_layout, got, accumulate)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    err = float((got.double() - want.double()).norm() / want.double().norm())
    mx = float((got.double() - want.double()).abs().max() / want.double().abs().max())
    # the tolerance of the GEMM tests (fp32 accumulation)
    assert err < 5e-5 and mx < 5e-4, (err, mx)


def test_noalloc_matches_workspace_gemm_twice(cv):
    # first call: K split across CTAs (the scratch holds the split partials);
    # second call: another shape and B layout, accumulating into C
    for M, N, K in ((128, 256, 4096), (200, 520, 2048)):
        assert cv.canvas_gemm_workspace_size(M, N, K) <= cv.CANVAS_GEMM_NOALLOC_SCRATCH_BYTES
    # more than the 256-byte alignment slack: the first shape does split K, so
    # its partials really go through the static array
    assert cv.canvas_gemm_workspace_size(128, 256, 4096) > 256
    _compare(cv, 128, 256, 4096, 0, 0, seed=1)
    _compare(cv, 200, 520, 2048, 1, 1, seed=2)


def test_noalloc_rejects_shapes_beyond_the_static_scratch(cv):
    M, N, K = 256, 8192, 2816
    assert cv.canvas_gemm_workspace_size(M, N, K) > cv.CANVAS_GEMM_NOALLOC_SCRATCH_BYTES
    A = torch.zeros(M, K, device="cuda", dtype=torch.bfloat16)
    B = torch.zeros(N, K, device="cuda", dtype=torch.bfloat16)
    C = torch.zeros(M, N, device="cuda")
    with pytest.raises(cv.CanvasError) as e:
        cv.canvas_gemm_bf16_noalloc(A, B, 0, C, 0)
    assert e.value.status == cv.CANVAS_ERR_WORKSPACE
    assert "static scratch" in str(e.value)


def test_noalloc_rejects_a_misaligned_output(cv):
    # C offset by one float: 4-byte aligned, not 16; the call returns before
    # anything is enqueued
    M, N, K = 128, 256, 4096
    A = torch.zeros(M, K, device="cuda", dtype=torch.bfloat16)
    B = torch.zeros(N, K, device="cuda", dtype=torch.bfloat16)
    Cbig = torch.zeros(M * N + 4, device="cuda")
    C = Cbig[1:1 + M * N].view(M, N)
    with pytest.raises(cv.CanvasError) as e:
        cv.canvas_gemm_bf16_noalloc(A, B, 0, C, 0)
    assert e.value.status == cv.CANVAS_ERR_ARG
    assert "aligned" in str(e.value)
