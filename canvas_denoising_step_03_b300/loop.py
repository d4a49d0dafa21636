"""A batched multi-layer denoising loop built only from the library's C-ABI
calls (argument marshalling and buffer management here; every arithmetic step
runs in the library's kernels).

One step, for B canvases of C tokens:

1. ``canvas_embed_input``: v = E[tokens] + soft_emb of the previous step
   (bf16 copy for the layers, fp32 copy as the residual stream);
2. per layer: ``canvas_attention`` on the bf16 stream, then
   ``canvas_gemm_bf16`` adds out W_o^T to the fp32 stream and
   ``canvas_cast_bf16`` refreshes the bf16 copy;
3. tied LM head: ``canvas_gemm_bf16_to_bf16`` computes x E^T, accumulated in
   fp32 and stored once as bf16 logits;
4. ``canvas_sample`` with the step index; positions committed in earlier
   steps stay frozen with their tokens.

The method's sampling loop and self-conditioning are described in the AI
Trends summary of a DiffusionGemma 26B notebook (aitrends.kr/articles/94089),
section "섹션별 상세" (sampling-loop paragraph) and glossary "자기 조건화".
"""
from __future__ import annotations

import numpy as np
import torch

from . import (CANVAS_BF16, CANVAS_LAYER_GLOBAL, CANVAS_LAYER_SLIDING, canvas_attention,
               canvas_attention_workspace_size, canvas_cast_bf16, canvas_count_committed, canvas_embed_input,
               canvas_gelu_bf16, canvas_gemm_bf16, canvas_gemm_bf16_to_bf16, canvas_gemm_workspace_size,
               canvas_sample,
               canvas_sample_workspace_size, canvas_temperature_at, make_kv_cache, workspace)


def _bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


class CanvasLoop:
    """Device state of the loop for one set of inputs (the layout of
    ``canvas_workloads.LoopInputs``: bf16 bit patterns, caches holding
    positions cache_lo .. prefix-1 of every sequence)."""

    def __init__(self, inp, device="cuda", page_tokens: int = 64, seed_pages: int = 1234, schedule=None,
                 categorical: bool = False):
        """``schedule`` = (t_max, t_min, steps): the sampler temperature of
        step s is canvas_temperature_at(s, steps, t_max, t_min) (default: 1);
        ``categorical``: committed positions take a categorical draw from
        their probabilities instead of the argmax."""
        self.schedule = schedule
        self.commit_mode = 2 if categorical else 0
        import canvas_workloads as wl  # shapes and page tables of the seeded inputs
        cfg = inp.cfg
        self.cfg, self.dev = cfg, device
        B, C, D, V = cfg.B, cfg.C, cfg.D, cfg.V
        R = B * C
        self.layers = []
        attn_ws = 0
        for k, L in enumerate(inp.layers):
            lc = L.cfg
            table, npages = wl.page_layout_range(B, L.cache_lo, cfg.prefix, page_tokens, seed=seed_pages + k)
            kp = _bf16(wl.scatter_pages_range(L.cache_k, L.cache_lo, table, npages, page_tokens), device)
            vp = None if L.cache_v is None else _bf16(
                wl.scatter_pages_range(L.cache_v, L.cache_lo, table, npages, page_tokens), device)
            bt = torch.from_numpy(table).to(device)
            layer = dict(cfg=lc, W_q=_bf16(L.W_q, device), W_k=_bf16(L.W_k, device),
                         W_v=None if L.W_v is None else _bf16(L.W_v, device), W_o=_bf16(L.W_o, device),
                         gamma_q=torch.from_numpy(L.gamma_q).to(device), gamma_k=torch.from_numpy(L.gamma_k).to(device),
                         freq=torch.from_numpy(L.freq).to(device), k_pool=kp, v_pool=vp, table=bt,
                         kv=make_kv_cache(kp, vp, bt, page_tokens),
                         type=CANVAS_LAYER_GLOBAL if lc.layer == "global" else CANVAS_LAYER_SLIDING,
                         out=torch.empty((B, C, lc.Hq * lc.d), dtype=torch.bfloat16, device=device))
            self.layers.append(layer)
            attn_ws = max(attn_ws, canvas_attention_workspace_size(CANVAS_BF16, B, C, D, lc.Hq, lc.Hkv, lc.d,
                                                                   cfg.prefix, layer["type"]))
        self.prefix_len = torch.full((B,), cfg.prefix, dtype=torch.int32, device=device)
        self.E = _bf16(inp.E, device)
        self.tokens = torch.from_numpy(inp.tokens0.astype(np.int32)).to(device)
        self.x = torch.empty((B, C, D), dtype=torch.bfloat16, device=device)
        self.x32 = torch.empty((R, D), dtype=torch.float32, device=device)
        self.logits = torch.empty((R, V), dtype=torch.bfloat16, device=device)
        self.soft = torch.zeros((R, D), dtype=torch.float32, device=device)
        self.frozen = torch.zeros(R, dtype=torch.uint8, device=device)
        self.mask = torch.zeros(R, dtype=torch.uint8, device=device)
        self.next_tokens = torch.empty(R, dtype=torch.int32, device=device)
        self.entropy = torch.empty(R, dtype=torch.float32, device=device)
        self.conf = torch.empty(R, dtype=torch.float32, device=device)
        self.argmax = torch.empty(R, dtype=torch.int32, device=device)
        self.attn_ws = workspace(attn_ws, device)
        gws = max([canvas_gemm_workspace_size(R, D, L["cfg"].Hq * L["cfg"].d) for L in self.layers] +
                  [canvas_gemm_workspace_size(R, V, D)])
        self.gemm_ws = workspace(gws, device)
        self.samp_ws = workspace(canvas_sample_workspace_size(CANVAS_BF16, R, V, D), device)
        self.counts = torch.zeros(B, dtype=torch.int32, device=device)
        # self-conditioning MLP (optional): sc = W2 bf16(gelu(W1 bf16(soft)))
        self.sc = None
        if getattr(inp, "sc_W1", None) is not None:
            H = inp.sc_W1.shape[0]
            self.sc = dict(W1=_bf16(inp.sc_W1, device), W2=_bf16(inp.sc_W2, device),
                           s16=torch.empty((R, D), dtype=torch.bfloat16, device=device),
                           h=torch.empty((R, H), dtype=torch.float32, device=device),
                           g=torch.empty((R, H), dtype=torch.bfloat16, device=device),
                           out=torch.empty((R, D), dtype=torch.float32, device=device))
            gws2 = max(canvas_gemm_workspace_size(R, H, D), canvas_gemm_workspace_size(R, D, H))
            if gws2 > self.gemm_ws.numel():
                self.gemm_ws = workspace(gws2, device)
        self.step_index = 0

    # ---- the stages of a step (each one C-ABI call or two)
    def selfcond(self, soft: torch.Tensor) -> torch.Tensor:
        """The self-conditioning MLP on the previous soft embedding (fp32 out)."""
        s = self.sc
        canvas_cast_bf16(soft, s["s16"])
        canvas_gemm_bf16(s["s16"], s["W1"], 0, s["h"], 0, self.gemm_ws)
        canvas_gelu_bf16(s["h"], s["g"])
        canvas_gemm_bf16(s["g"], s["W2"], 0, s["out"], 0, self.gemm_ws)
        return s["out"]

    def embed(self, tokens: torch.Tensor, soft):
        """x, x32 = E[tokens] + soft (soft None: no self-conditioning input);
        with the self-conditioning MLP, soft passes through it first."""
        if soft is not None and self.sc is not None:
            soft = self.selfcond(soft)
        canvas_embed_input(tokens, self.E, soft, self.x, self.x32)

    def attention(self, k: int, x: torch.Tensor) -> torch.Tensor:
        """Layer k's attention on the bf16 canvas stream x [B, C, D]."""
        cfg, L = self.cfg, self.layers[k]
        lc = L["cfg"]
        canvas_attention(x, L["W_q"], L["W_k"], L["W_v"], lc.Hq, lc.Hkv, lc.d, L["gamma_q"], L["gamma_k"], lc.eps,
                         L["freq"], L["type"], L["kv"], self.prefix_len, cfg.prefix, lc.window, 1.0, 0, L["out"],
                         None, self.attn_ws)
        return L["out"]

    def residual(self, k: int, out: torch.Tensor, x32: torch.Tensor, x: torch.Tensor):
        """x32 += out W_o^T (fp32), x = bf16(x32)."""
        R = self.cfg.B * self.cfg.C
        canvas_gemm_bf16(out.view(R, -1), self.layers[k]["W_o"], 0, x32, 1, self.gemm_ws)
        canvas_cast_bf16(x32, x)

    def head(self, x: torch.Tensor) -> torch.Tensor:
        """bf16 logits of the tied LM head, x E^T."""
        R = self.cfg.B * self.cfg.C
        canvas_gemm_bf16_to_bf16(x.view(R, -1), self.E, 0, self.logits, self.gemm_ws)
        return self.logits

    def sample(self, logits: torch.Tensor, step: int, frozen: torch.Tensor, frozen_tokens: torch.Tensor):
        """The sampler of step ``step``; outputs in next_tokens, mask, entropy,
        conf, argmax, soft."""
        cfg = self.cfg
        canvas_sample(logits, self.E, cfg.bound, cfg.seed, step, self.temperature(step), self.commit_mode, cfg.C,
                      frozen, frozen_tokens, self.next_tokens, self.mask, self.entropy, self.conf, self.argmax, None,
                      CANVAS_BF16, self.soft, self.samp_ws)

    def temperature(self, step: int) -> float:
        if self.schedule is None:
            return 1.0
        t_max, t_min, steps = self.schedule
        return canvas_temperature_at(step, steps, t_max, t_min)

    def committed_counts(self) -> torch.Tensor:
        """Committed positions of each canvas after the last step (device)."""
        canvas_count_committed(self.mask, self.cfg.C, self.counts)
        return self.counts

    def run(self, max_steps: int, stop_when_committed: bool = True) -> int:
        """Steps until every canvas is fully committed (adaptive stopping) or
        max_steps; returns the number of steps run.  The stop test reads the
        per-canvas counts back to the host after each step."""
        for n in range(max_steps):
            self.step()
            if stop_when_committed:
                counts = self.committed_counts().cpu().numpy()   # device -> host copy, host-side test
                if bool(np.all(counts == self.cfg.C)):
                    return n + 1
        return max_steps

    def step(self, keep_attn: bool = False, mark=None):
        """Run one denoising step on the loop's own state; returns the
        attention outputs if asked.  ``mark(name)``, if given, is called on the
        host between the stages (``attention_begin``/``attention_end`` around
        each layer's attention call, ``sample_begin``/``sample_end`` around the
        sampler call), e.g. to record CUDA events on the stream."""
        mark = mark or (lambda name: None)
        self.embed(self.tokens, self.soft if self.step_index > 0 else None)
        outs = []
        for k in range(len(self.layers)):
            mark("attention_begin")
            out = self.attention(k, self.x)
            mark("attention_end")
            if keep_attn:
                outs.append(out.clone())
            self.residual(k, out, self.x32, self.x)
        logits = self.head(self.x)
        mark("sample_begin")
        self.sample(logits, self.step_index, self.frozen, self.tokens)
        mark("sample_end")
        # committed positions stay frozen with their tokens in the next step
        self.tokens, self.next_tokens = self.next_tokens, self.tokens
        self.frozen.copy_(self.mask)
        self.step_index += 1
        return outs
