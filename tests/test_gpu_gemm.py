"""tcgen05 GEMM through the C ABI against a plain torch fp64 product of the
same bf16 operands."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cv():
    import __graft_entry__
    __graft_entry__.build()
    import canvas_denoising_step_03_b300 as cv
    return cv


def _run(cv, M, N, K, b_layout, accumulate=0, seed=0, scale=1.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    A = (torch.randn(M, K, device="cuda", generator=g) * scale).to(torch.bfloat16)
    if b_layout == 0:
        B = torch.randn(N, K, device="cuda", generator=g).to(torch.bfloat16)
        ref = A.double() @ B.double().T
    else:
        B = torch.randn(K, N, device="cuda", generator=g).to(torch.bfloat16)
        ref = A.double() @ B.double()
    C0 = torch.randn(M, N, device="cuda", generator=g)
    C = C0.clone() if accumulate else torch.full((M, N), float("nan"), device="cuda")
    if accumulate:
        ref = ref + C0.double()
    ws = cv.workspace(cv.canvas_gemm_workspace_size(M, N, K))
    cv.canvas_gemm_bf16(A, B, b_layout, C, accumulate, ws)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    err = (C.double() - ref).norm() / ref.norm()
    mx = (C.double() - ref).abs().max() / ref.abs().max()
    return float(err), float(mx)


@pytest.mark.parametrize("M,N,K,b_layout", [
    (128, 256, 64, 0),      # one tile, one k-block
    (256, 512, 1024, 0),    # two accumulators, split-K
    (256, 4096, 2816, 0),   # sliding-layer q projection shape
    (256, 1024, 2816, 0),   # global-layer k projection shape
    (100, 200, 136, 0),     # ragged M, N, K
    (300, 520, 1000, 0),    # two m-tiles, the second partly empty
    (256, 512, 1024, 1),    # B stored [K, N]
    (256, 2816, 65536, 1),  # soft-embedding shape (a quarter of the vocab)
    (40, 136, 8192, 1),     # ragged, B stored [K, N]
])
def test_gemm_matches_fp64(cv, M, N, K, b_layout):
    err, mx = _run(cv, M, N, K, b_layout)
    # fp32 accumulation over K terms: relative error grows like sqrt(K) * 2^-24
    assert err < 5e-5 and mx < 5e-4, (err, mx)


def test_gemm_accumulate(cv):
    err, mx = _run(cv, 256, 512, 2048, 0, accumulate=1)   # K split: the reduce kernel adds C
    assert err < 5e-5, err


@pytest.mark.parametrize("M,N,K", [(256, 512, 64), (100, 200, 120)])
def test_gemm_accumulate_single_split(cv, M, N, K):
    # one K split: the GEMM's own epilogue adds into C (ragged edges included)
    err, mx = _run(cv, M, N, K, 0, accumulate=1)
    assert err < 5e-5 and mx < 5e-4, (err, mx)


def test_gemm_repeatable_bitwise(cv):
    M, N, K = 256, 2816, 32768
    g = torch.Generator(device="cuda").manual_seed(3)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn(K, N, device="cuda", generator=g).to(torch.bfloat16)
    ws = cv.workspace(cv.canvas_gemm_workspace_size(M, N, K))
    outs = []
    for _ in range(3):
        C = torch.empty(M, N, device="cuda")
        cv.canvas_gemm_bf16(A, B, 1, C, 0, ws)
        outs.append(C)
    assert cv.canvas_device_status() == cv.CANVAS_OK
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("M,N,K,b_layout", [
    (1024, 4096, 2816, 0),  # K split: the reduce kernel rounds
    (256, 520, 64, 0),      # one split, ragged N: the epilogue's 64-column bf16 boxes are clipped
    (100, 200, 136, 1),     # ragged M, N, K, B stored [K, N]
])
def test_gemm_bf16_output_is_the_rounded_fp32_product(cv, M, N, K, b_layout):
    """canvas_gemm_bf16_to_bf16 equals canvas_gemm_bf16 rounded to bf16
    (nearest even), bit for bit: the same accumulation, one rounding."""
    g = torch.Generator(device="cuda").manual_seed(M + N)
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    B = (torch.randn(N, K, device="cuda", generator=g) if b_layout == 0 else
         torch.randn(K, N, device="cuda", generator=g)).to(torch.bfloat16)
    ws = cv.workspace(cv.canvas_gemm_workspace_size(M, N, K))
    C32 = torch.empty(M, N, device="cuda")
    cv.canvas_gemm_bf16(A, B, b_layout, C32, 0, ws)
    C16 = torch.full((M, N), float("nan"), device="cuda", dtype=torch.bfloat16)
    cv.canvas_gemm_bf16_to_bf16(A, B, b_layout, C16, ws)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    assert torch.equal(C16.view(torch.int16), C32.to(torch.bfloat16).view(torch.int16))
