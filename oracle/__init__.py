"""fp64 CPU oracle of the canvas refinement step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (the CUDA library and its Python binding) never imports, links
or calls anything here, and this package never touches the CUDA path: the two
share no code.  The only shared module is ``canvas_workloads`` (seeded random
draws).

Sources.  The method is described on five web pages about DiffusionGemma;
every function cites the page and the section it follows:

* [AIT] AI Trends summary of a hands-on DiffusionGemma 26B weights notebook
  (aitrends.kr/articles/94089): section "섹션별 상세" (the rms(), rotate()
  and attention-block snippets, the sampler paragraph) and the glossary
  "용어 해설" (scalar QK norm, partial RoPE, self-conditioning,
  sliding-window attention).
* [TC] ThakiCloud, "DiffusionGemma 26B-A4B" (thakicloud.github.io): section
  "아키텍처" (vocab 262,144, window 1,024, canvas 256).
* [VL] velog, "DiffusionGemma Self-conditioning": sections "Block diffusion",
  "Self-conditioning".
* [TR] "[논문리뷰] DiffusionGemma Technical Report" (blog.secrett2633.cloud):
  §1 key terms (canvas, adaptive stopping), §3.
* [AB] aibars news, "Google의 DiffusionGemma, 노이즈에서 텍스트 생성 및 자체
  수정 기능 탑재": section "블록 자동 회귀 노이즈 제거 및 자체 수정"
  (commit to the KV cache, uniform-state renoise of low-confidence tokens).

Modules: ``numerics`` (rms, rotate, RoPE spectrum, bf16 rounding),
``attention`` (the canvas attention layer), ``sampler`` (softmax, entropy,
argmax, commit/renoise, soft embedding), ``splitmix`` (the counter RNG),
``loop`` (one step of the multi-layer denoising loop, the self-conditioning
MLP), ``moe`` (a mixture-of-experts MLP block).

Parity status: every function is pinned by the CPU tests in
``tests/test_oracle_pins.py`` except where a docstring says "parity unpinned".
"""
from . import numerics, attention, sampler, splitmix, loop, moe  # noqa: F401
