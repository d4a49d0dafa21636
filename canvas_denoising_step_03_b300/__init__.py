"""Python binding of libcanvas.so -- argument marshalling only.

Every function here has the name of the C entry point it calls (see
include/canvas.h) and does nothing but turn tensors into device pointers, the
current torch stream into a cudaStream_t, and a non-OK status into a
``CanvasError``.  All arithmetic of the canvas step runs in the library's CUDA
kernels.  There is no fallback: if the shared library is missing or fails to
load, importing this package raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcanvas.so")

CANVAS_OK = 0
CANVAS_ERR_ARG = -1
CANVAS_ERR_UNSUPPORTED = -2
CANVAS_ERR_CUDA = -3
CANVAS_ERR_TIMEOUT = -4
CANVAS_ERR_WORKSPACE = -5
CANVAS_ERR_BOUNDS = -6
STATUS_NAMES = {0: "CANVAS_OK", -1: "CANVAS_ERR_ARG", -2: "CANVAS_ERR_UNSUPPORTED", -3: "CANVAS_ERR_CUDA",
                -4: "CANVAS_ERR_TIMEOUT", -5: "CANVAS_ERR_WORKSPACE", -6: "CANVAS_ERR_BOUNDS"}

CANVAS_BF16 = 0
CANVAS_FP32 = 1
CANVAS_LAYER_SLIDING = 0
CANVAS_LAYER_GLOBAL = 1

# every symbol include/canvas.h declares
EXPORTED = [
    "canvas_attention_workspace_size", "canvas_attention", "canvas_sample_workspace_size", "canvas_sample",
    "canvas_gemm_workspace_size", "canvas_gemm_bf16", "canvas_last_error", "canvas_device_status",
    "canvas_version", "canvas_profile_events", "canvas_kernel_launches", "canvas_gemm_bf16_noalloc",
    "canvas_embed_input", "canvas_cast_bf16", "canvas_gemm_bf16_to_bf16", "canvas_selftest_wait_timeout",
    "canvas_attention_encode", "canvas_kv_append_workspace_size", "canvas_kv_append", "canvas_count_committed",
    "canvas_temperature_at", "canvas_gelu_bf16", "canvas_moe_workspace_size", "canvas_moe",
]

# size of the static scratch behind canvas_gemm_bf16_noalloc (include/canvas.h)
CANVAS_GEMM_NOALLOC_SCRATCH_BYTES = 16 << 20

CANVAS_KERNEL_ATTENTION = 0
CANVAS_KERNEL_PREP = 1
CANVAS_KERNEL_SAMPLER = 2
CANVAS_KERNEL_SOFT_EMB = 3


class CanvasError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class canvas_kv_cache(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("max_pages_per_seq", ctypes.c_int32), ("page_tokens", ctypes.c_int32),
                ("num_pages", ctypes.c_int32)]


def _load(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"libcanvas.so not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    P, I, F, Z, U64, U32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64,
                            ctypes.c_uint32)
    lib.canvas_attention_workspace_size.argtypes = [I] * 9
    lib.canvas_attention_workspace_size.restype = Z
    lib.canvas_attention.argtypes = [P, I, I, I, I, P, P, P, I, I, I, P, P, F, P, I,
                                     ctypes.POINTER(canvas_kv_cache), P, I, I, F, I, P, P, P, Z, P]
    lib.canvas_attention.restype = I
    lib.canvas_attention_encode.argtypes = lib.canvas_attention.argtypes
    lib.canvas_attention_encode.restype = I
    lib.canvas_kv_append_workspace_size.argtypes = [I] * 7
    lib.canvas_kv_append_workspace_size.restype = Z
    lib.canvas_kv_append.argtypes = [P, I, I, I, I, P, P, I, I, P, F, P, I, ctypes.POINTER(canvas_kv_cache), P, I,
                                     P, Z, P]
    lib.canvas_kv_append.restype = I
    lib.canvas_moe_workspace_size.argtypes = [I] * 6
    lib.canvas_moe_workspace_size.restype = Z
    lib.canvas_moe.argtypes = [P, I, I, P, I, I, P, P, P, P, I, P, P, P, I, P, P, P, P, Z, P]
    lib.canvas_moe.restype = I
    lib.canvas_gelu_bf16.argtypes = [P, P, Z, P]
    lib.canvas_gelu_bf16.restype = I
    lib.canvas_count_committed.argtypes = [P, I, I, P, P]
    lib.canvas_count_committed.restype = I
    lib.canvas_temperature_at.argtypes = [I, I, F, F]
    lib.canvas_temperature_at.restype = F
    lib.canvas_sample_workspace_size.argtypes = [I, I, I, I]
    lib.canvas_sample_workspace_size.restype = Z
    lib.canvas_sample.argtypes = [P, I, I, I, P, I, F, U64, U32, F, I, I, P, P, P, P, P, P, P, P, I, P, P, Z, P]
    lib.canvas_sample.restype = I
    lib.canvas_gemm_workspace_size.argtypes = [I, I, I]
    lib.canvas_gemm_workspace_size.restype = Z
    lib.canvas_gemm_bf16.argtypes = [P, P, I, P, I, I, I, I, P, Z, P]
    lib.canvas_gemm_bf16.restype = I
    lib.canvas_selftest_wait_timeout.argtypes = [P]
    lib.canvas_selftest_wait_timeout.restype = I
    lib.canvas_gemm_bf16_to_bf16.argtypes = [P, P, I, P, I, I, I, P, Z, P]
    lib.canvas_gemm_bf16_to_bf16.restype = I
    lib.canvas_gemm_bf16_noalloc.argtypes = [P, P, I, P, I, I, I, I, P]
    lib.canvas_gemm_bf16_noalloc.restype = I
    lib.canvas_embed_input.argtypes = [P, P, P, I, I, I, P, P, P]
    lib.canvas_embed_input.restype = I
    lib.canvas_cast_bf16.argtypes = [P, P, Z, P]
    lib.canvas_cast_bf16.restype = I
    lib.canvas_last_error.argtypes = []
    lib.canvas_last_error.restype = ctypes.c_char_p
    lib.canvas_device_status.argtypes = [P]
    lib.canvas_device_status.restype = I
    lib.canvas_version.argtypes = []
    lib.canvas_version.restype = ctypes.c_char_p
    lib.canvas_profile_events.argtypes = [I, P, P]
    lib.canvas_profile_events.restype = I
    lib.canvas_kernel_launches.argtypes = []
    lib.canvas_kernel_launches.restype = U64
    return lib


lib = _load()


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("canvas calls take device tensors")
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int):
    if status != CANVAS_OK:
        raise CanvasError(status, lib.canvas_last_error().decode())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CANVAS_BF16
    if t.dtype == torch.float32:
        return CANVAS_FP32
    raise ValueError(f"unsupported dtype {t.dtype}")


def canvas_version() -> str:
    return lib.canvas_version().decode()


def canvas_last_error() -> str:
    return lib.canvas_last_error().decode()


def canvas_profile_events(kernel_id: int, start=None, stop=None):
    """Register torch.cuda.Event objects (or None) as timing hooks of a kernel.
    A torch event has a CUDA handle only once it has been recorded."""
    for e in (start, stop):
        if e is not None and not e.cuda_event:
            raise ValueError("canvas_profile_events: record the event once before registering it")
    hs = None if start is None else ctypes.c_void_p(start.cuda_event)
    he = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    _check(lib.canvas_profile_events(int(kernel_id), hs, he))


def canvas_kernel_launches() -> int:
    return int(lib.canvas_kernel_launches())


def canvas_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return lib.canvas_device_status(_stream(stream))


def canvas_attention_workspace_size(dtype: int, B, C, D, Hq, Hkv, d, max_prefix, layer_type) -> int:
    return lib.canvas_attention_workspace_size(dtype, B, C, D, Hq, Hkv, d, max_prefix, layer_type)


def canvas_sample_workspace_size(dtype: int, rows, V, D) -> int:
    return lib.canvas_sample_workspace_size(dtype, rows, V, D)


def canvas_gemm_workspace_size(M, N, K) -> int:
    return lib.canvas_gemm_workspace_size(M, N, K)


def make_kv_cache(k_pool, v_pool, block_table, page_tokens: int) -> canvas_kv_cache:
    return canvas_kv_cache(_ptr(k_pool), _ptr(v_pool), _ptr(block_table),
                           int(block_table.shape[1]) if block_table is not None else 0, int(page_tokens),
                           int(k_pool.shape[0]) if k_pool is not None else 0)


def canvas_attention(x, W_q, W_k, W_v, Hq, Hkv, d, gamma_q, gamma_k, eps, freq, layer_type, kv: canvas_kv_cache,
                     prefix_len, max_prefix, window, scale, v_unit_rms, out, lse, workspace, stream=None):
    B, C, D = x.shape
    _check(lib.canvas_attention(_ptr(x), _dtype_code(x), B, C, D, _ptr(W_q), _ptr(W_k), _ptr(W_v), Hq, Hkv, d,
                                _ptr(gamma_q), _ptr(gamma_k), float(eps), _ptr(freq), int(layer_type),
                                ctypes.byref(kv), _ptr(prefix_len), int(max_prefix), int(window), float(scale),
                                int(v_unit_rms), _ptr(out), _ptr(lse), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream(stream)))


def canvas_attention_encode(x, W_q, W_k, W_v, Hq, Hkv, d, gamma_q, gamma_k, eps, freq, layer_type,
                            kv: canvas_kv_cache, prefix_len, max_prefix, window, scale, v_unit_rms, out, lse,
                            workspace, stream=None):
    """canvas_attention in encode mode (causal inside the block); same arguments."""
    B, C, D = x.shape
    _check(lib.canvas_attention_encode(_ptr(x), _dtype_code(x), B, C, D, _ptr(W_q), _ptr(W_k), _ptr(W_v), Hq, Hkv,
                                       d, _ptr(gamma_q), _ptr(gamma_k), float(eps), _ptr(freq), int(layer_type),
                                       ctypes.byref(kv), _ptr(prefix_len), int(max_prefix), int(window),
                                       float(scale), int(v_unit_rms), _ptr(out), _ptr(lse), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


def canvas_kv_append_workspace_size(dtype: int, B, C, D, Hkv, d, layer_type) -> int:
    return lib.canvas_kv_append_workspace_size(dtype, B, C, D, Hkv, d, layer_type)


def canvas_kv_append(x, W_k, W_v, Hkv, d, gamma_k, eps, freq, layer_type, kv: canvas_kv_cache, prefix_len,
                     max_prefix, workspace, stream=None):
    """Write a committed block's cache rows; advances prefix_len by C."""
    B, C, D = x.shape
    _check(lib.canvas_kv_append(_ptr(x), _dtype_code(x), B, C, D, _ptr(W_k), _ptr(W_v), Hkv, d, _ptr(gamma_k),
                                float(eps), _ptr(freq), int(layer_type), ctypes.byref(kv), _ptr(prefix_len),
                                int(max_prefix), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(stream)))


def canvas_sample(logits, E, entropy_bound, seed, step, temperature, commit_mode, canvas_len, frozen,
                  frozen_tokens, tokens, commit_mask, entropy, confidence, argmax, probs_out, probs_dtype,
                  soft_emb, workspace, stream=None):
    rows, V = logits.shape
    D = E.shape[1]
    _check(lib.canvas_sample(_ptr(logits), _dtype_code(logits), rows, V, _ptr(E), D, float(entropy_bound),
                             int(seed) & (2 ** 64 - 1), int(step), float(temperature), int(commit_mode),
                             int(canvas_len), _ptr(frozen), _ptr(frozen_tokens), _ptr(tokens), _ptr(commit_mask),
                             _ptr(entropy), _ptr(confidence), _ptr(argmax), _ptr(probs_out), int(probs_dtype),
                             _ptr(soft_emb), _ptr(workspace), workspace.numel() * workspace.element_size(),
                             _stream(stream)))


def canvas_moe_workspace_size(R, D, E, F, k, Fs) -> int:
    return lib.canvas_moe_workspace_size(int(R), int(D), int(E), int(F), int(k), int(Fs))


def canvas_moe(x, router, k, expert_scale, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, out, topk_idx, topk_w,
               workspace, stream=None):
    """Mixture-of-experts block: x [R, D] bf16, router [E, D], W_gate / W_up
    [E*F, D], W_down [E*D, F], shared expert Ws_* (or None), out [R, D] fp32."""
    R, D = x.shape
    E = router.shape[0]
    F = W_gate.shape[0] // E
    Fs = 0 if Ws_gate is None else Ws_gate.shape[0]
    _check(lib.canvas_moe(_ptr(x), R, D, _ptr(router), E, int(k), _ptr(expert_scale), _ptr(W_gate), _ptr(W_up),
                          _ptr(W_down), F, _ptr(Ws_gate), _ptr(Ws_up), _ptr(Ws_down), Fs, _ptr(out), _ptr(topk_idx),
                          _ptr(topk_w), _ptr(workspace), workspace.numel() * workspace.element_size(),
                          _stream(stream)))


def canvas_gelu_bf16(inp, out, stream=None):
    """out = bf16(gelu(inp)) (tanh form), inp fp32."""
    _check(lib.canvas_gelu_bf16(_ptr(inp), _ptr(out), inp.numel(), _stream(stream)))


def canvas_count_committed(commit_mask, canvas_len, counts, stream=None):
    """counts[c] = committed positions of canvas c (commit_mask [rows] uint8)."""
    _check(lib.canvas_count_committed(_ptr(commit_mask), commit_mask.numel(), int(canvas_len), _ptr(counts),
                                      _stream(stream)))


def canvas_temperature_at(step: int, steps: int, t_max: float, t_min: float) -> float:
    """Sampler temperature of a step on the linear t_max -> t_min schedule."""
    return float(lib.canvas_temperature_at(int(step), int(steps), float(t_max), float(t_min)))


def canvas_gemm_bf16(A, B, b_layout, C, accumulate, workspace, stream=None):
    M, K = A.shape
    N = B.shape[0] if b_layout == 0 else B.shape[1]
    _check(lib.canvas_gemm_bf16(_ptr(A), _ptr(B), int(b_layout), _ptr(C), M, N, K, int(accumulate),
                                _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def canvas_gemm_bf16_to_bf16(A, B, b_layout, C, workspace, stream=None):
    """C (bf16) = bf16(A op(B)); the workspace of canvas_gemm_bf16."""
    M, K = A.shape
    N = B.shape[0] if b_layout == 0 else B.shape[1]
    _check(lib.canvas_gemm_bf16_to_bf16(_ptr(A), _ptr(B), int(b_layout), _ptr(C), M, N, K, _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream)))


def canvas_selftest_wait_timeout(stream=None):
    """Enqueue the diagnostic kernel whose bounded wait runs out (include/canvas.h)."""
    _check(lib.canvas_selftest_wait_timeout(_stream(stream)))


def canvas_gemm_bf16_noalloc(A, B, b_layout, C, accumulate, stream=None):
    """canvas_gemm_bf16 with the library's static scratch instead of a workspace."""
    M, K = A.shape
    N = B.shape[0] if b_layout == 0 else B.shape[1]
    _check(lib.canvas_gemm_bf16_noalloc(_ptr(A), _ptr(B), int(b_layout), _ptr(C), M, N, K, int(accumulate),
                                        _stream(stream)))


def canvas_embed_input(tokens, E, soft_emb, x, x32=None, stream=None):
    """x = bf16(E[tokens] + soft_emb), x32 = the fp32 sum (soft_emb, x32 may be None)."""
    rows = tokens.numel()
    V, D = E.shape
    _check(lib.canvas_embed_input(_ptr(tokens), _ptr(E), _ptr(soft_emb), rows, D, V, _ptr(x), _ptr(x32),
                                  _stream(stream)))


def canvas_cast_bf16(src, dst, stream=None):
    """dst (bf16) = src (fp32), element for element."""
    _check(lib.canvas_cast_bf16(_ptr(src), _ptr(dst), src.numel(), _stream(stream)))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A device byte buffer of at least ``nbytes`` (torch's allocator aligns it)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)
