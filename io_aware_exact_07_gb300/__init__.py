"""Exact IO-aware attention (forward + backward) for GB300 / sm_103a.

Thin ctypes binding over the C ABI in ``include/fa.h`` (libfa_gb300.so, built
in-tree by ``io_aware_exact_07_gb300.build``). Functions named ``fa_*`` mirror
the C entry points one to one and only marshal arguments (torch tensors ->
device pointers, the current torch CUDA stream); every step of the
computation runs in the library's CUDA kernels. There is no CPU fallback: if
the library is missing or fails to load, calls raise.

``fwd`` / ``bwd`` are conveniences that allocate the outputs (and the backward
workspace) with torch and call ``fa_fwd`` / ``fa_bwd``; ``decode`` does the
same for ``fa_decode`` (short query blocks over a K/V cache).
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_WORKSPACE = 4
FA_ERR_TIMEOUT = 5

# Symbols declared in include/fa.h.
EXPORTS = (
    "fa_fwd", "fa_bwd", "fa_fwd_gqa", "fa_bwd_gqa", "fa_fwd_window", "fa_bwd_window",
    "fa_bwd_workspace_size", "fa_bwd_preprocess",
    "fa_bwd_dkdv", "fa_bwd_dq", "fa_decode", "fa_decode_workspace_size",
    "fa_fp8_workspace_size", "fa_fp8_vt_stride", "fa_fp8_quantize", "fa_fwd_fp8",
    "fa_fp8_quantize_gqa", "fa_fwd_fp8_gqa",
    "fa_bwd_noalloc", "fa_dropout_p8", "fa_debug_dropout_keep",
    "fa_debug_philox", "fa_butterfly_mask", "fa_device_status", "fa_set_wait_timeout_ns",
    "fa_test_inject_stall", "fa_status_string",
)

_lock = threading.Lock()
_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def load(build_if_missing: bool = False):
    """Load libfa_gb300.so (optionally building it first). Raises if unavailable."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing or not os.path.exists(LIB_PATH):
            if not build_if_missing:
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m io_aware_exact_07_gb300.build`")
            from . import build as _b
            _b.build()
        lib = ctypes.CDLL(LIB_PATH)
        vp, i, f, u64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64,
                             ctypes.c_size_t)
        lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, f, u64, u64, vp, vp, vp]
        lib.fa_fwd.restype = i
        lib.fa_bwd_workspace_size.argtypes = [i, i, i, i]
        lib.fa_bwd_workspace_size.restype = sz
        lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, f, u64, u64,
                               vp, vp, vp, sz, vp]
        lib.fa_bwd.restype = i
        lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, f, u64, u64, vp, vp,
                                   vp]
        lib.fa_fwd_gqa.restype = i
        lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, f, u64,
                                   u64, vp, vp, vp, sz, vp]
        lib.fa_bwd_gqa.restype = i
        lib.fa_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, i, f, u64, u64,
                                      vp, vp, vp]
        lib.fa_fwd_window.restype = i
        lib.fa_bwd_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, i,
                                      f, u64, u64, vp, vp, vp, sz, vp]
        lib.fa_bwd_window.restype = i
        lib.fa_bwd_preprocess.argtypes = [vp, vp, i, i, i, i, vp, sz, vp]
        lib.fa_bwd_preprocess.restype = i
        lib.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, f, u64, u64, vp,
                                    vp, vp, sz, vp]
        lib.fa_bwd_dkdv.restype = i
        lib.fa_bwd_dq.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, f, u64, u64, vp, vp,
                                  vp, sz, vp]
        lib.fa_bwd_dq.restype = i
        lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, f,
                                       u64, u64, vp, vp, vp]
        lib.fa_bwd_noalloc.restype = i
        lib.fa_decode_workspace_size.argtypes = [i, i, i, i, i, i, i]
        lib.fa_decode_workspace_size.restype = sz
        lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, i, vp, sz, vp]
        lib.fa_decode.restype = i
        lib.fa_fp8_workspace_size.argtypes = [i, i, i]
        lib.fa_fp8_workspace_size.restype = sz
        lib.fa_fp8_vt_stride.argtypes = [i]
        lib.fa_fp8_vt_stride.restype = i
        lib.fa_fp8_quantize.argtypes = [vp, vp, vp, vp, i, i, i, i, vp, vp, vp, vp, vp, vp, vp, sz,
                                        vp]
        lib.fa_fp8_quantize.restype = i
        lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, vp]
        lib.fa_fwd_fp8.restype = i
        lib.fa_fp8_quantize_gqa.argtypes = [vp, vp, vp, vp, i, i, i, i, i, vp, vp, vp, vp, vp, vp,
                                            vp, sz, vp]
        lib.fa_fp8_quantize_gqa.restype = i
        lib.fa_fwd_fp8_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp]
        lib.fa_fwd_fp8_gqa.restype = i
        lib.fa_dropout_p8.argtypes = [f]
        lib.fa_dropout_p8.restype = i
        lib.fa_debug_dropout_keep.argtypes = [vp, i, i, i, f, u64, u64, vp]
        lib.fa_debug_dropout_keep.restype = i
        lib.fa_debug_philox.argtypes = [vp, vp, i, ctypes.c_uint32, ctypes.c_uint32, vp]
        lib.fa_debug_philox.restype = i
        lib.fa_butterfly_mask.argtypes = [vp, i]
        lib.fa_butterfly_mask.restype = i
        lib.fa_device_status.argtypes = [vp, i]
        lib.fa_device_status.restype = i
        lib.fa_set_wait_timeout_ns.argtypes = [u64]
        lib.fa_set_wait_timeout_ns.restype = None
        lib.fa_test_inject_stall.argtypes = [i]
        lib.fa_test_inject_stall.restype = None
        lib.fa_status_string.argtypes = [i]
        lib.fa_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().fa_status_string(int(status)).decode()


def fa_status_string(status: int) -> str:
    return status_string(status)


def _stream(stream=None):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(status: int, where: str):
    if status != FA_OK:
        raise FAError(status, where)


def _check_qkv(*ts):
    for t in ts:
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("expected contiguous 4-D bf16 CUDA tensors [B, H, N, d]")


def _kv_heads(q, k, v) -> int:
    """K/V head count; q [B, H, N, d] with k, v [B, H_kv, N, d], H a multiple of H_kv."""
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if tuple(k.shape) != (B, Hkv, N, d) or tuple(v.shape) != tuple(k.shape) or H % Hkv != 0:
        raise ValueError("k and v must be [B, H_kv, N, d] with H a multiple of H_kv")
    return Hkv


def _opt_ptrs(block_mask, seqlens_k, B, N):
    """Pointers of the optional block mask (uint8 [nb, nb], nb = ceil(N / 128))
    and key lengths (int32 [B]). The kernels index both without bounds (the C
    entry points cannot know their sizes), so their shapes are checked here."""
    if block_mask is not None:
        nb = (int(N) + 127) // 128
        if (block_mask.dtype != torch.uint8 or not block_mask.is_cuda
                or not block_mask.is_contiguous() or tuple(block_mask.shape) != (nb, nb)):
            raise ValueError(f"block_mask must be a contiguous uint8 CUDA tensor [{nb}, {nb}]")
    if seqlens_k is not None:
        if (seqlens_k.dtype != torch.int32 or not seqlens_k.is_cuda
                or not seqlens_k.is_contiguous() or tuple(seqlens_k.shape) != (int(B),)):
            raise ValueError(f"seqlens_k must be a contiguous int32 CUDA tensor [{int(B)}]")
    return _ptr(block_mask), _ptr(seqlens_k)


# ----------------------------------------------------------------- C mirrors

def fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal=False, dropout_p=0.0, seed=0, offset=0,
           block_mask=None, seqlens_k=None, stream=None) -> int:
    bm, sl = _opt_ptrs(block_mask, seqlens_k, B, N)
    return load().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                         int(bool(causal)), float(dropout_p), int(seed), int(offset), bm, sl,
                         _stream(stream))


def fa_bwd_workspace_size(B, H, N, d) -> int:
    return int(load().fa_bwd_workspace_size(B, H, N, d))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal=False, dropout_p=0.0,
           seed=0, offset=0, block_mask=None, seqlens_k=None, workspace=None, workspace_bytes=0,
           stream=None) -> int:
    bm, sl = _opt_ptrs(block_mask, seqlens_k, B, N)
    return load().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                         _ptr(dk), _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                         float(dropout_p), int(seed), int(offset), bm, sl, _ptr(workspace),
                         int(workspace_bytes), _stream(stream))


def fa_fwd_gqa(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal=False, dropout_p=0.0, seed=0,
               offset=0, block_mask=None, seqlens_k=None, stream=None) -> int:
    bm, sl = _opt_ptrs(block_mask, seqlens_k, B, N)
    return load().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv, N, d,
                             float(scale), int(bool(causal)), float(dropout_p), int(seed),
                             int(offset), bm, sl, _stream(stream))


def fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N, d, scale, causal=False,
               dropout_p=0.0, seed=0, offset=0, block_mask=None, seqlens_k=None, workspace=None,
               workspace_bytes=0, stream=None) -> int:
    bm, sl = _opt_ptrs(block_mask, seqlens_k, B, N)
    return load().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                             _ptr(dk), _ptr(dv), B, H, H_kv, N, d, float(scale),
                             int(bool(causal)), float(dropout_p), int(seed), int(offset), bm, sl,
                             _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_fwd_window(q, k, v, o, lse, B, H, H_kv, N, d, scale, causal=False, window_left=-1,
                  window_right=-1, dropout_p=0.0, seed=0, offset=0, block_mask=None,
                  seqlens_k=None, stream=None) -> int:
    bm, sl = _opt_ptrs(block_mask, seqlens_k, B, N)
    return load().fa_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, H_kv, N, d,
                                float(scale), int(bool(causal)), int(window_left),
                                int(window_right), float(dropout_p), int(seed), int(offset), bm,
                                sl, _stream(stream))


def fa_bwd_window(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, N, d, scale, causal=False,
                  window_left=-1, window_right=-1, dropout_p=0.0, seed=0, offset=0,
                  block_mask=None, seqlens_k=None, workspace=None, workspace_bytes=0,
                  stream=None) -> int:
    bm, sl = _opt_ptrs(block_mask, seqlens_k, B, N)
    return load().fa_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                _ptr(dq), _ptr(dk), _ptr(dv), B, H, H_kv, N, d, float(scale),
                                int(bool(causal)), int(window_left), int(window_right),
                                float(dropout_p), int(seed), int(offset), bm, sl, _ptr(workspace),
                                int(workspace_bytes), _stream(stream))


def fa_bwd_preprocess(o, dout, B, H, N, d, workspace, workspace_bytes, stream=None) -> int:
    return load().fa_bwd_preprocess(_ptr(o), _ptr(dout), B, H, N, d, _ptr(workspace),
                                    int(workspace_bytes), _stream(stream))


def fa_bwd_dkdv(q, k, v, dout, lse, dk, dv, B, H, N, d, scale, causal=False, dropout_p=0.0,
                seed=0, offset=0, block_mask=None, seqlens_k=None, workspace=None,
                workspace_bytes=0, stream=None) -> int:
    bm, sl = _opt_ptrs(block_mask, seqlens_k, B, N)
    return load().fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(dk),
                              _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                              float(dropout_p), int(seed), int(offset), bm, sl, _ptr(workspace),
                              int(workspace_bytes), _stream(stream))


def fa_bwd_dq(q, k, v, dout, lse, dq, B, H, N, d, scale, causal=False, dropout_p=0.0, seed=0,
              offset=0, block_mask=None, seqlens_k=None, workspace=None, workspace_bytes=0,
              stream=None) -> int:
    bm, sl = _opt_ptrs(block_mask, seqlens_k, B, N)
    return load().fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(lse), _ptr(dq), B, H, N,
                            d, float(scale), int(bool(causal)), float(dropout_p), int(seed),
                            int(offset), bm, sl, _ptr(workspace), int(workspace_bytes),
                            _stream(stream))


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal=False,
                   dropout_p=0.0, seed=0, offset=0, block_mask=None, seqlens_k=None,
                   stream=None) -> int:
    """fa_bwd for callers that cannot allocate device memory: the library uses
    its own static device scratch (B*H*N <= 2^22) instead of a workspace."""
    bm, sl = _opt_ptrs(block_mask, seqlens_k, B, N)
    return load().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, float(scale),
                                 int(bool(causal)), float(dropout_p), int(seed), int(offset), bm,
                                 sl, _stream(stream))


def fa_decode_workspace_size(B, H, H_kv, Nq, Nk, d, num_ctas=0) -> int:
    return int(load().fa_decode_workspace_size(B, H, H_kv, Nq, Nk, d, num_ctas))


def fa_decode(q, k_cache, v_cache, o, lse, B, H, H_kv, Nq, Nk, d, scale, causal=False,
              seqlens_k=None, num_ctas=0, workspace=None, workspace_bytes=0, stream=None,
              window_left=-1) -> int:
    if seqlens_k is not None and (seqlens_k.dtype != torch.int32 or not seqlens_k.is_cuda
                                  or not seqlens_k.is_contiguous()
                                  or tuple(seqlens_k.shape) != (int(B),)):
        raise ValueError(f"seqlens_k must be a contiguous int32 CUDA tensor [{int(B)}]")
    return load().fa_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), B, H, H_kv,
                            Nq, Nk, d, float(scale), int(bool(causal)), int(window_left),
                            _ptr(seqlens_k), int(num_ctas), _ptr(workspace), int(workspace_bytes),
                            _stream(stream))


def fa_fp8_workspace_size(B, H, d) -> int:
    return int(load().fa_fp8_workspace_size(B, H, d))


def fa_fp8_vt_stride(N) -> int:
    return int(load().fa_fp8_vt_stride(N))


def fa_fp8_quantize(q, k, v, signs, B, H, N, d, q8, k8, vt8, s_q, s_k, s_v, workspace,
                    workspace_bytes, stream=None) -> int:
    return load().fa_fp8_quantize(_ptr(q), _ptr(k), _ptr(v), _ptr(signs), B, H, N, d, _ptr(q8),
                                  _ptr(k8), _ptr(vt8), _ptr(s_q), _ptr(s_k), _ptr(s_v),
                                  _ptr(workspace), int(workspace_bytes), _stream(stream))


def fa_fwd_fp8(q8, k8, vt8, s_q, s_k, s_v, o, lse, B, H, N, d, scale, causal=False,
               seqlens_k=None, stream=None) -> int:
    _, sl = _opt_ptrs(None, seqlens_k, B, N)
    return load().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(s_q), _ptr(s_k), _ptr(s_v),
                             _ptr(o), _ptr(lse), B, H, N, d, float(scale), int(bool(causal)), sl,
                             _stream(stream))


def fa_fp8_quantize_gqa(q, k, v, signs, B, H, Hkv, N, d, q8, k8, vt8, s_q, s_k, s_v, workspace,
                        workspace_bytes, stream=None) -> int:
    return load().fa_fp8_quantize_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(signs), B, H, Hkv, N, d,
                                      _ptr(q8), _ptr(k8), _ptr(vt8), _ptr(s_q), _ptr(s_k),
                                      _ptr(s_v), _ptr(workspace), int(workspace_bytes),
                                      _stream(stream))


def fa_fwd_fp8_gqa(q8, k8, vt8, s_q, s_k, s_v, o, lse, B, H, Hkv, N, d, scale, causal=False,
                   seqlens_k=None, stream=None) -> int:
    _, sl = _opt_ptrs(None, seqlens_k, B, N)
    return load().fa_fwd_fp8_gqa(_ptr(q8), _ptr(k8), _ptr(vt8), _ptr(s_q), _ptr(s_k), _ptr(s_v),
                                 _ptr(o), _ptr(lse), B, H, Hkv, N, d, float(scale),
                                 int(bool(causal)), sl, _stream(stream))


def fa_dropout_p8(p: float) -> int:
    return int(load().fa_dropout_p8(float(p)))


def fa_debug_dropout_keep(keep, B, H, N, dropout_p, seed=0, offset=0, stream=None) -> int:
    return load().fa_debug_dropout_keep(_ptr(keep), B, H, N, float(dropout_p), int(seed),
                                        int(offset), _stream(stream))


def fa_debug_philox(counters, out, n, key0, key1, stream=None) -> int:
    return load().fa_debug_philox(_ptr(counters), _ptr(out), int(n), int(key0), int(key1),
                                  _stream(stream))


def fa_butterfly_mask(nb: int) -> torch.Tensor:
    """Host uint8 [nb, nb] butterfly block mask from the library's generator."""
    m = torch.zeros((nb, nb), dtype=torch.uint8)
    _check(load().fa_butterfly_mask(ctypes.c_void_p(m.data_ptr()), nb), "fa_butterfly_mask")
    return m


def fa_device_status(stream=None, clear=True) -> int:
    return int(load().fa_device_status(_stream(stream), int(bool(clear))))


def fa_set_wait_timeout_ns(ns: int) -> None:
    load().fa_set_wait_timeout_ns(int(ns))


def fa_test_inject_stall(mode: int) -> None:
    load().fa_test_inject_stall(int(mode))


# ----------------------------------------------------------- conveniences

def fwd(q, k, v, scale=None, causal=False, dropout_p=0.0, seed=0, offset=0, block_mask=None,
        seqlens_k=None, stream=None, window=(-1, -1)):
    """Allocate O and lse with torch and run fa_fwd (fa_fwd_gqa when k and v
    have fewer heads than q, fa_fwd_window when window = (left, right) is
    set). Returns (o, lse)."""
    _check_qkv(q, k, v)
    B, H, N, d = q.shape
    Hkv = _kv_heads(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if tuple(window) != (-1, -1):
        st = fa_fwd_window(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, window[0], window[1],
                           dropout_p, seed, offset, block_mask, seqlens_k, stream)
    elif Hkv == H:
        st = fa_fwd(q, k, v, o, lse, B, H, N, d, scale, causal, dropout_p, seed, offset,
                    block_mask, seqlens_k, stream)
    else:
        st = fa_fwd_gqa(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, dropout_p, seed, offset,
                        block_mask, seqlens_k, stream)
    _check(st, "fa_fwd")
    return o, lse


def bwd(q, k, v, o, dout, lse, scale=None, causal=False, dropout_p=0.0, seed=0, offset=0,
        block_mask=None, seqlens_k=None, workspace=None, stream=None, window=(-1, -1)):
    """Allocate dQ, dK, dV (and the workspace if not given) and run fa_bwd
    (fa_bwd_gqa when k and v have fewer heads than q, fa_bwd_window when
    window = (left, right) is set)."""
    _check_qkv(q, k, v, o, dout)
    B, H, N, d = q.shape
    Hkv = _kv_heads(q, k, v)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_bytes = fa_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    if tuple(window) != (-1, -1):
        st = fa_bwd_window(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal,
                           window[0], window[1], dropout_p, seed, offset, block_mask, seqlens_k,
                           workspace, workspace.numel(), stream)
    elif Hkv == H:
        st = fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, dropout_p, seed,
                    offset, block_mask, seqlens_k, workspace, workspace.numel(), stream)
    else:
        st = fa_bwd_gqa(q, k, v, o, dout, lse, dq, dk, dv, B, H, Hkv, N, d, scale, causal,
                        dropout_p, seed, offset, block_mask, seqlens_k, workspace,
                        workspace.numel(), stream)
    _check(st, "fa_bwd")
    return dq, dk, dv


def decode(q, k_cache, v_cache, scale=None, causal=False, seqlens_k=None, num_ctas=0,
           stream=None, window_left=-1):
    """Allocate O, lse (and the workspace, if the split needs one) with torch and
    run fa_decode: q [B, H, Nq, d] over k_cache, v_cache [B, H_kv, Nk, d].
    Returns (o, lse)."""
    _check_qkv(q, k_cache, v_cache)
    B, H, Nq, d = q.shape
    _, Hkv, Nk, _ = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or k_cache.shape[0] != B or \
            k_cache.shape[3] != d:
        raise ValueError("k_cache and v_cache must be [B, H_kv, Nk, d] like q's B and d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ws_bytes = fa_decode_workspace_size(B, H, Hkv, Nq, Nk, d, num_ctas)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device) if ws_bytes else None
    _check(fa_decode(q, k_cache, v_cache, o, lse, B, H, Hkv, Nq, Nk, d, scale, causal, seqlens_k,
                     num_ctas, ws, ws_bytes, stream, window_left), "fa_decode")
    return o, lse


def fp8_quantize(q, k, v, signs=None, stream=None):
    """Allocate the e4m3 tensors and scales with torch and run fa_fp8_quantize
    (fa_fp8_quantize_gqa when k and v have fewer heads than q).
    Returns dict(q8, k8, vt8, s_q, s_k, s_v) (uint8 codes, fp32 scales)."""
    _check_qkv(q, k, v)
    Hkv = _kv_heads(q, k, v)
    B, H, N, d = q.shape
    dev = q.device
    Np = fa_fp8_vt_stride(N)
    out = dict(q8=torch.empty((B, H, N, d), dtype=torch.uint8, device=dev),
               k8=torch.empty((B, Hkv, N, d), dtype=torch.uint8, device=dev),
               vt8=torch.empty((B, Hkv, d, Np), dtype=torch.uint8, device=dev),
               s_q=torch.empty((B, H), dtype=torch.float32, device=dev),
               s_k=torch.empty((B, Hkv), dtype=torch.float32, device=dev),
               s_v=torch.empty((B, Hkv, d), dtype=torch.float32, device=dev))
    wsb = fa_fp8_workspace_size(B, H, d)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    if Hkv == H:
        st = fa_fp8_quantize(q, k, v, signs, B, H, N, d, out["q8"], out["k8"], out["vt8"],
                             out["s_q"], out["s_k"], out["s_v"], ws, wsb, stream)
    else:
        st = fa_fp8_quantize_gqa(q, k, v, signs, B, H, Hkv, N, d, out["q8"], out["k8"],
                                 out["vt8"], out["s_q"], out["s_k"], out["s_v"], ws, wsb, stream)
    _check(st, "fa_fp8_quantize")
    return out


def fwd_fp8(qz, scale, causal=False, seqlens_k=None, stream=None):
    """Run fa_fwd_fp8 (fa_fwd_fp8_gqa with grouped K/V heads) on the output of
    fp8_quantize; returns (o bf16, lse)."""
    B, H, N, d = qz["q8"].shape
    Hkv = qz["k8"].shape[1]
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=qz["q8"].device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=qz["q8"].device)
    args = (qz["q8"], qz["k8"], qz["vt8"], qz["s_q"], qz["s_k"], qz["s_v"], o, lse)
    if Hkv == H:
        st = fa_fwd_fp8(*args, B, H, N, d, scale, causal, seqlens_k, stream)
    else:
        st = fa_fwd_fp8_gqa(*args, B, H, Hkv, N, d, scale, causal, seqlens_k, stream)
    _check(st, "fa_fwd_fp8")
    return o, lse
