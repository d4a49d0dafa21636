"""Shared helpers of the tests: move seeded workloads to the device, call the
C ABI through the binding, run the oracle on the same inputs, compare.

Nothing here computes any part of the method: device inputs come from
``canvas_workloads``; expected values come from ``oracle``.
"""
from __future__ import annotations

import numpy as np
import torch

import canvas_workloads as wl


def to_device(a: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def f64(a, dtype):
    return None if a is None else wl.as_f64(a, dtype)


class AttnCase:
    """Device-side buffers of one canvas_attention call."""

    def __init__(self, inp: wl.AttnInputs, device="cuda", page_seed=1234):
        import canvas_denoising_step_03_b300 as cv
        self.cv = cv
        self.inp = inp
        c = inp.cfg
        self.cfg = c
        dt = c.dtype
        self.x = to_device(inp.x, dt, device)
        self.W_q = to_device(inp.W_q, dt, device)
        self.W_k = to_device(inp.W_k, dt, device)
        self.W_v = None if inp.W_v is None else to_device(inp.W_v, dt, device)
        self.gamma_q = torch.from_numpy(inp.gamma_q).to(device)
        self.gamma_k = torch.from_numpy(inp.gamma_k).to(device)
        self.freq = torch.from_numpy(inp.freq).to(device)
        table, num_pages = wl.page_layout(c, seed=page_seed)
        self.table_np = table
        self.block_table = torch.from_numpy(table).to(device)
        self.k_pool = to_device(wl.scatter_pages(inp.cache_k, table, num_pages, c.page_tokens), dt, device)
        self.v_pool = None
        if inp.cache_v is not None:
            self.v_pool = to_device(wl.scatter_pages(inp.cache_v, table, num_pages, c.page_tokens), dt, device)
        self.kv = cv.make_kv_cache(self.k_pool, self.v_pool, self.block_table, c.page_tokens)
        self.prefix_len = torch.from_numpy(inp.prefix_len).to(device)
        tdt = torch.bfloat16 if dt == "bf16" else torch.float32
        self.out = torch.full((c.B, c.C, c.Hq * c.d), float("nan"), dtype=tdt, device=device)
        self.lse = torch.full((c.B, c.C, c.Hq), float("nan"), dtype=torch.float32, device=device)
        self.layer = cv.CANVAS_LAYER_GLOBAL if c.layer == "global" else cv.CANVAS_LAYER_SLIDING
        dcode = cv.CANVAS_BF16 if dt == "bf16" else cv.CANVAS_FP32
        ws = cv.canvas_attention_workspace_size(dcode, c.B, c.C, c.D, c.Hq, c.Hkv, c.d, c.max_prefix, self.layer)
        assert ws > 0
        self.ws = cv.workspace(ws, device)

    def run(self, v_unit_rms=0, scale=1.0, stream=None):
        c = self.cfg
        self.cv.canvas_attention(self.x, self.W_q, self.W_k, self.W_v, c.Hq, c.Hkv, c.d, self.gamma_q,
                                 self.gamma_k, c.eps, self.freq, self.layer, self.kv, self.prefix_len,
                                 c.max_prefix, c.window, scale, v_unit_rms, self.out, self.lse, self.ws, stream)
        return self

    def status(self):
        return self.cv.canvas_device_status()

    def out_f64(self):
        return self.out.float().cpu().numpy().astype(np.float64)


def oracle_attention(inp: wl.AttnInputs, rows=None, v_unit_rms=False, scale=1.0, slack_eps=None):
    """fp64 oracle on the same inputs; bf16 workloads use the bf16 storage
    model.  With ``slack_eps`` (bf16 only) returns (out, lse, slack)."""
    from oracle import attention as oatt
    c = inp.cfg
    dt = c.dtype
    storage = "bf16" if dt == "bf16" else "fp64"
    return oatt.canvas_attention(f64(inp.x, dt), f64(inp.W_q, dt), f64(inp.W_k, dt), f64(inp.W_v, dt), c.Hq,
                                 c.Hkv, c.d, inp.gamma_q.astype(np.float64), inp.gamma_k.astype(np.float64), c.eps,
                                 inp.freq.astype(np.float64), c.layer, f64(inp.cache_k, dt), f64(inp.cache_v, dt),
                                 inp.prefix_len, c.window, scale=scale, v_unit_rms=v_unit_rms, storage=storage,
                                 rows=rows, slack_eps=slack_eps if dt == "bf16" else None)


def attn_errors(got: np.ndarray, want: np.ndarray):
    """(max abs, relative Frobenius) over the finite entries of want."""
    m = np.isfinite(want)
    diff = got[m] - want[m]
    return float(np.max(np.abs(diff))), float(np.linalg.norm(diff) / max(np.linalg.norm(want[m]), 1e-300))
