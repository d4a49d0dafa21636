"""Encode mode and block commit through the C ABI against the fp64 oracle.

A finished canvas (the block) is first attended in encode mode
(canvas_attention_encode: causal inside the block), then committed to the
paged cache (canvas_kv_append: sliding layers append final keys and values,
global layers the raw shared rows), and the next canvas is attended in
decode mode over the extended prefix.

Bars: the attention bar of canvas_harness.attention_bar for both attention
calls; the appended cache rows bit-exact against the oracle's stored rows
except at rounding ties (where the row's pre-rounding value lies within the
path's fp32 error of a bf16 midpoint: either neighbour is a correct stored
value, and the next canvas's oracle carries their flips in its slack).
"""
import numpy as np
import pytest
import torch

import canvas_workloads as wl
from canvas_harness import SLACK_EPS, attention_bar, to_device
from oracle import attention as oatt

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cv():
    import __graft_entry__
    __graft_entry__.build()
    import canvas_denoising_step_03_b300 as cv
    return cv


def f64(a, dt="bf16"):
    return None if a is None else wl.as_f64(a, dt)


CASES = [
    dict(name="encode-sliding", B=2, C=48, prefix=(130, 64), D=256, Hq=4, Hkv=2, d=128, layer="sliding", window=96,
         theta=1e4, rotary_fraction=1.0, dtype="bf16", seed=31),
    dict(name="encode-sliding-d256", B=1, C=40, prefix=(300,), D=256, Hq=8, Hkv=2, d=256, layer="sliding",
         window=200, theta=1e4, rotary_fraction=1.0, dtype="bf16", seed=32),
    dict(name="encode-global-d512", B=2, C=64, prefix=(200, 0), D=256, Hq=8, Hkv=1, d=512, layer="global",
         window=0, theta=1e6, rotary_fraction=0.25, dtype="bf16", seed=33),
    dict(name="encode-global-d128", B=1, C=33, prefix=(150,), D=256, Hq=4, Hkv=2, d=128, layer="global", window=0,
         theta=1e6, rotary_fraction=0.25, dtype="bf16", seed=34),
]


@pytest.mark.parametrize("spec", CASES, ids=lambda s: s["name"])
def test_encode_commit_then_decode_the_next_canvas(cv, spec):
    cfg = wl.AttnConfig(**spec)
    inp = wl.make_attention_inputs(cfg)
    B, C, D, Hq, Hkv, d = cfg.B, cfg.C, cfg.D, cfg.Hq, cfg.Hkv, cfg.d
    glob = cfg.layer == "global"
    C2 = 24
    x2 = wl.f32_to_bf16_bits(np.random.default_rng(cfg.seed + 100).standard_normal((B, C2, D)).astype(np.float32))
    # a cache with room for the block and the next canvas
    cap = wl.replace(cfg, prefix=tuple(int(p) + C + C2 for p in cfg.prefix))
    table, npages = wl.page_layout(cap)
    dev = "cuda"
    kpool = to_device(wl.scatter_pages(inp.cache_k, table, npages, cfg.page_tokens), "bf16")
    vpool = None if glob else to_device(wl.scatter_pages(inp.cache_v, table, npages, cfg.page_tokens), "bf16")
    bt = torch.from_numpy(table).to(dev)
    kv = cv.make_kv_cache(kpool, vpool, bt, cfg.page_tokens)
    P0 = inp.prefix_len.astype(np.int64)
    prefix = torch.from_numpy(inp.prefix_len.astype(np.int32)).to(dev)
    cap_max = cap.max_prefix
    xs = to_device(inp.x, "bf16")
    Wq, Wk = to_device(inp.W_q, "bf16"), to_device(inp.W_k, "bf16")
    Wv = None if glob else to_device(inp.W_v, "bf16")
    gq, gk, fr = (torch.from_numpy(t).to(dev) for t in (inp.gamma_q, inp.gamma_k, inp.freq))
    layer = cv.CANVAS_LAYER_GLOBAL if glob else cv.CANVAS_LAYER_SLIDING
    ws = cv.workspace(max(cv.canvas_attention_workspace_size(cv.CANVAS_BF16, B, max(C, C2), D, Hq, Hkv, d, cap_max,
                                                             layer),
                          cv.canvas_kv_append_workspace_size(cv.CANVAS_BF16, B, C, D, Hkv, d, layer)))
    ora = dict(W_q=f64(inp.W_q), W_k=f64(inp.W_k), W_v=f64(inp.W_v), gq=inp.gamma_q.astype(np.float64),
               gk=inp.gamma_k.astype(np.float64), freq=inp.freq.astype(np.float64))
    ck0, cv0 = f64(inp.cache_k), f64(inp.cache_v)

    # 1. the block in encode mode
    out = torch.full((B, C, Hq * d), float("nan"), dtype=torch.bfloat16, device=dev)
    cv.canvas_attention_encode(xs, Wq, Wk, Wv, Hq, Hkv, d, gq, gk, cfg.eps, fr, layer, kv, prefix, cfg.max_prefix,
                               cfg.window, 1.0, 0, out, None, ws)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    args = (f64(inp.x), ora["W_q"], ora["W_k"], ora["W_v"], Hq, Hkv, d, ora["gq"], ora["gk"], cfg.eps, ora["freq"],
            cfg.layer)
    want, _, slack = oatt.canvas_attention(*args, ck0, cv0, P0, cfg.window, storage="bf16", slack_eps=SLACK_EPS,
                                           causal=True)
    want64, _ = oatt.canvas_attention(*args, ck0, cv0, P0, cfg.window, storage="fp64", causal=True)
    got = out.float().cpu().numpy().astype(np.float64)
    attention_bar(f"{cfg.name} block, encode mode", got, want, slack, want64)
    # the two modes differ on this workload by far more than the bar: the
    # comparison above tells them apart
    dec, _ = oatt.canvas_attention(*args, ck0, cv0, P0, cfg.window, storage="bf16")
    assert np.max(np.abs(want - dec)) > 0.1

    # 2. commit the block
    cv.canvas_kv_append(xs, Wk, Wv, Hkv, d, gk, cfg.eps, fr, layer, kv, prefix, cap_max, ws)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    np.testing.assert_array_equal(prefix.cpu().numpy(), P0 + C)
    res = oatt.kv_append(f64(inp.x), ora["W_k"], ora["W_v"], Hkv, d, ora["gk"], cfg.eps, ora["freq"], cfg.layer,
                         P0, storage="bf16", slack_eps=SLACK_EPS)
    rk, rv, dk, dv = res
    ex = oatt.kv_append(f64(inp.x), ora["W_k"], ora["W_v"], Hkv, d, ora["gk"], cfg.eps, ora["freq"], cfg.layer,
                        P0, storage="fp64")                         # the rows before rounding
    pools = [(kpool, rk, dk, ex[0])] + ([] if glob else [(vpool, rv, dv, ex[1])])
    n_ties = 0
    for pool, rows, delta, exact in pools:
        pool_np = pool.float().cpu().numpy().astype(np.float64)
        for b in range(B):
            for i in range(C):
                pos = int(P0[b]) + i
                page = table[b, pos // cfg.page_tokens]
                got_row = pool_np[page, :, pos % cfg.page_tokens, :]          # [Hkv, d]
                tie = delta[b, :, i, :] != 0
                diff = got_row != rows[b, :, i, :]
                assert not np.any(diff & ~tie), (b, i, int(np.sum(diff & ~tie)))
                # at a tie the row holds a correct rounding of a value within
                # the tie window of the exact one (for a value much smaller
                # than its row that can be more than one bf16 step away)
                x = exact[b, :, i, :]
                partner = np.concatenate([x[:, d // 2:], x[:, :d // 2]], axis=1)
                rms = np.sqrt(np.mean(x * x, axis=1, keepdims=True))
                window = SLACK_EPS * (np.abs(x) + np.abs(partner) + rms)
                spacing = np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(got_row), 1e-30))) - 8).astype(int))
                assert np.all((np.abs(got_row - x) <= window + spacing)[tie])
                n_ties += int(np.sum(diff))
    print(f"{cfg.name}: appended rows bit-exact except {n_ties} rounding-tie elements")

    # 3. the next canvas in decode mode over prefix P + C
    out2 = torch.full((B, C2, Hq * d), float("nan"), dtype=torch.bfloat16, device=dev)
    x2d = to_device(x2, "bf16")
    cv.canvas_attention(x2d, Wq, Wk, Wv, Hq, Hkv, d, gq, gk, cfg.eps, fr, layer, kv, prefix, cap_max, cfg.window,
                        1.0, 0, out2, None, ws)
    assert cv.canvas_device_status() == cv.CANVAS_OK, cv.canvas_last_error()
    Pm = int(P0.max()) + C
    ck = np.full((B, Hkv, Pm, d), np.nan)
    cvv = None if glob else np.full_like(ck, np.nan)
    dck = np.zeros_like(ck)
    dcv = None if glob else np.zeros_like(ck)
    for b in range(B):
        p = int(P0[b])
        ck[b, :, :p] = ck0[b, :, :p]
        ck[b, :, p:p + C] = rk[b]
        dck[b, :, p:p + C] = dk[b]
        if not glob:
            cvv[b, :, :p] = cv0[b, :, :p]
            cvv[b, :, p:p + C] = rv[b]
            dcv[b, :, p:p + C] = dv[b]
    args2 = (f64(x2), ora["W_q"], ora["W_k"], ora["W_v"], Hq, Hkv, d, ora["gq"], ora["gk"], cfg.eps, ora["freq"],
             cfg.layer, ck, cvv, P0 + C, cfg.window)
    want2, _, slack2 = oatt.canvas_attention(*args2, storage="bf16", slack_eps=SLACK_EPS, cache_dk=dck, cache_dv=dcv)
    want2_64, _ = oatt.canvas_attention(*args2, storage="fp64")
    attention_bar(f"{cfg.name} next canvas over the committed block", out2.float().cpu().numpy().astype(np.float64),
                    want2, slack2, want2_64)


def test_append_outside_the_mapped_pages_reports_bounds(cv):
    cfg = wl.AttnConfig(**CASES[0])
    inp = wl.make_attention_inputs(cfg)
    table, npages = wl.page_layout(cfg)          # pages for the prefix only: the block has no page
    dev = "cuda"
    kpool = to_device(wl.scatter_pages(inp.cache_k, table, npages, cfg.page_tokens), "bf16")
    vpool = to_device(wl.scatter_pages(inp.cache_v, table, npages, cfg.page_tokens), "bf16")
    bt = torch.from_numpy(np.concatenate([table, np.full((cfg.B, 4), -1, np.int32)], axis=1)).to(dev)
    kv = cv.make_kv_cache(kpool, vpool, bt, cfg.page_tokens)
    prefix = torch.from_numpy(inp.prefix_len.astype(np.int32)).to(dev)
    ws = cv.workspace(cv.canvas_kv_append_workspace_size(cv.CANVAS_BF16, cfg.B, cfg.C, cfg.D, cfg.Hkv, cfg.d,
                                                         cv.CANVAS_LAYER_SLIDING))
    before = kpool.clone()
    cv.canvas_kv_append(to_device(inp.x, "bf16"), to_device(inp.W_k, "bf16"), to_device(inp.W_v, "bf16"), cfg.Hkv,
                        cfg.d, torch.from_numpy(inp.gamma_k).to(dev), cfg.eps, torch.from_numpy(inp.freq).to(dev),
                        cv.CANVAS_LAYER_SLIDING, kv, prefix, int(bt.shape[1]) * cfg.page_tokens, ws)
    assert cv.canvas_device_status() == cv.CANVAS_ERR_BOUNDS
    # rows on mapped pages (the rest of each prefix's last page) were written;
    # nothing outside the pool was touched and the call's own pages are intact
    assert kpool.shape == before.shape
