"""CPU oracle for exact attention (fp64), with its ctypes binding.

TEST INFRASTRUCTURE ONLY: the plain definition that the GPU kernels are
checked against. Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the library itself
never does, and it shares no code with the CUDA sources.

Each function restates a definition from the pages (see ``oracle.c`` for the
citations): standard attention ("Algorithm 0", FlashAttention deep-read report
section 3.1) with the fused causal / key-padding / block-sparse / sliding-window masks and
dropout of section 3.2, its analytic backward, Philox4x32-10 (Salmon et al.,
SC'11) and the butterfly block mask of sections 2.6 / 3.5.

Parity status: every function here is pinned by tests in ``tests/`` against
closed forms, invariants, finite differences or an independent library
routine, except the absolute Philox stream on a CPU-only machine, which is
pinned on CPU only statistically and bit-exactly against cuRAND's device
Philox4_32_10 when a GPU is present.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc + OpenMP (no fast-math)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.POINTER
        dp = P(ctypes.c_double)
        ip = P(ctypes.c_int)
        u8 = P(ctypes.c_uint8)
        u32 = P(ctypes.c_uint32)
        lib.oracle_philox4x32_10.argtypes = [u32, u32, u32]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_p8.argtypes = [ctypes.c_double]
        lib.oracle_p8.restype = ctypes.c_int
        lib.oracle_butterfly.argtypes = [u8, ctypes.c_int]
        lib.oracle_butterfly.restype = None
        lib.oracle_dropout_keep.argtypes = [u8, ctypes.c_int, ip, ip, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64]
        lib.oracle_dropout_keep.restype = None
        common = [ctypes.c_int, ip, ip, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                  ctypes.c_int, ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, u8, ip,
                  ctypes.c_int, ctypes.c_int]
        lib.oracle_fwd.argtypes = [dp, dp, dp, dp, dp] + common
        lib.oracle_fwd.restype = ctypes.c_int
        lib.oracle_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp] + common
        lib.oracle_bwd.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _f64(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return np.ascontiguousarray(a)


def p8(p: float) -> int:
    """Dropout threshold in 1/256 units, round(256 p)."""
    return int(_load().oracle_p8(float(p)))


def philox4x32_10(counter, key) -> np.ndarray:
    """One Philox4x32-10 block: counter (4 x u32), key (2 x u32) -> 4 x u32."""
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c, ctypes.c_uint32), _ptr(k, ctypes.c_uint32),
                                 _ptr(out, ctypes.c_uint32))
    return out


def butterfly(nb: int) -> np.ndarray:
    """uint8 [nb, nb] butterfly block mask (r XOR c in {0} or a power of two < nb)."""
    m = np.zeros((nb, nb), dtype=np.uint8)
    _load().oracle_butterfly(_ptr(m, ctypes.c_uint8), int(nb))
    return m


def _heads(heads, B, H):
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    hb = np.ascontiguousarray(np.array([x[0] for x in heads], dtype=np.int32))
    hh = np.ascontiguousarray(np.array([x[1] for x in heads], dtype=np.int32))
    return heads, hb, hh


def dropout_keep(heads, H, N, p, seed=0, offset=0) -> np.ndarray:
    """uint8 [len(heads), N, N]: 1 where the element is kept."""
    heads, hb, hh = _heads(heads, None, None)
    out = np.zeros((len(heads), N, N), dtype=np.uint8)
    _load().oracle_dropout_keep(_ptr(out, ctypes.c_uint8), len(heads), _ptr(hb, ctypes.c_int),
                                _ptr(hh, ctypes.c_int), H, N, p8(p), seed, offset)
    return out


def _opt(block_mask, seqlens_k):
    bm = None if block_mask is None else np.ascontiguousarray(np.asarray(block_mask, np.uint8))
    sl = None if seqlens_k is None else np.ascontiguousarray(np.asarray(seqlens_k, np.int32))
    bmp = _ptr(bm, ctypes.c_uint8) if bm is not None else ctypes.POINTER(ctypes.c_uint8)()
    slp = _ptr(sl, ctypes.c_int) if sl is not None else ctypes.POINTER(ctypes.c_int)()
    return bm, sl, bmp, slp


def fwd(q, k, v, scale, causal=False, dropout_p=0.0, seed=0, offset=0, block_mask=None,
        seqlens_k=None, heads=None, H=None, window_left=-1, window_right=-1):
    """Standard attention forward in fp64.

    window_left / window_right: sliding window, key j visible to query i only
    if i - window_left <= j <= i + window_right (-1: that side unbounded).

    q, k, v: [n, N, d] arrays (one entry per head listed in ``heads``, a list
    of (b, h) pairs; default: all heads of a [B, H, N, d] tensor, in which
    case 4-D input is accepted). Returns (o [.., N, d], lse [.., N]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    shape4 = None
    if q.ndim == 4:
        B_, H_, N, d = q.shape
        shape4 = (B_, H_)
        heads, hb, hh = _heads(None, B_, H_)
        H = H_
        q, k, v = (x.reshape(B_ * H_, N, d) for x in (q, k, v))
    else:
        heads, hb, hh = _heads(heads, None, None)
        N, d = q.shape[1], q.shape[2]
    n = len(heads)
    o = np.zeros((n, N, d), dtype=np.float64)
    lse = np.zeros((n, N), dtype=np.float64)
    bm, sl, bmp, slp = _opt(block_mask, seqlens_k)
    rc = _load().oracle_fwd(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                            _ptr(v, ctypes.c_double), _ptr(o, ctypes.c_double),
                            _ptr(lse, ctypes.c_double), n, _ptr(hb, ctypes.c_int),
                            _ptr(hh, ctypes.c_int), int(H), N, d, float(scale), int(bool(causal)),
                            p8(dropout_p), int(seed), int(offset), bmp, slp, int(window_left),
                            int(window_right))
    if rc != 0:
        raise RuntimeError(f"oracle_fwd failed: {rc}")
    if shape4 is not None:
        o = o.reshape(shape4[0], shape4[1], N, d)
        lse = lse.reshape(shape4[0], shape4[1], N)
    return o, lse


def bwd(q, k, v, dout, scale, causal=False, dropout_p=0.0, seed=0, offset=0, block_mask=None,
        seqlens_k=None, heads=None, H=None, window_left=-1, window_right=-1):
    """Analytic backward of L = sum(O * dO) in fp64. Returns (dq, dk, dv, D)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    shape4 = None
    if q.ndim == 4:
        B_, H_, N, d = q.shape
        shape4 = (B_, H_)
        heads, hb, hh = _heads(None, B_, H_)
        H = H_
        q, k, v, dout = (x.reshape(B_ * H_, N, d) for x in (q, k, v, dout))
    else:
        heads, hb, hh = _heads(heads, None, None)
        N, d = q.shape[1], q.shape[2]
    n = len(heads)
    dq = np.zeros((n, N, d), dtype=np.float64)
    dk = np.zeros((n, N, d), dtype=np.float64)
    dv = np.zeros((n, N, d), dtype=np.float64)
    D = np.zeros((n, N), dtype=np.float64)
    bm, sl, bmp, slp = _opt(block_mask, seqlens_k)
    rc = _load().oracle_bwd(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                            _ptr(v, ctypes.c_double), _ptr(dout, ctypes.c_double),
                            _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                            _ptr(dv, ctypes.c_double), _ptr(D, ctypes.c_double), n,
                            _ptr(hb, ctypes.c_int), _ptr(hh, ctypes.c_int), int(H), N, d,
                            float(scale), int(bool(causal)), p8(dropout_p), int(seed),
                            int(offset), bmp, slp, int(window_left), int(window_right))
    if rc != 0:
        raise RuntimeError(f"oracle_bwd failed: {rc}")
    if shape4 is not None:
        dq, dk, dv = (x.reshape(shape4[0], shape4[1], N, d) for x in (dq, dk, dv))
        D = D.reshape(shape4[0], shape4[1], N)
    return dq, dk, dv, D


def _group(H: int, Hkv: int) -> int:
    if Hkv < 1 or H % Hkv != 0:
        raise ValueError(f"H={H} is not a multiple of H_kv={Hkv}")
    return H // Hkv


def fwd_gqa(q, k, v, scale, **kw):
    """Grouped-query attention forward (K/V heads shared by several query heads,
    which the page "Attention Kernel: FlashAttention 与它的后继者", section on
    FlashAttention's IO-aware insight, names as a further cut of K/V reads):
    q [B, H, N, d],
    k and v [B, H_kv, N, d] with H a multiple of H_kv; query head h of batch b
    attends with K/V head h // (H / H_kv). Written out from that definition:
    every query head gets its group's K/V and the per-head forward above runs
    unchanged (dropout keyed by the query head, as for H independent heads)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    G = _group(q.shape[1], k.shape[1])
    return fwd(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), scale, **kw)


def bwd_gqa(q, k, v, dout, scale, **kw):
    """Backward of fwd_gqa: dq per query head; dk and dv of a K/V head are the
    sums over the G query heads that share it (each of them used that K/V).
    Returns (dq [B, H, N, d], dk [B, H_kv, N, d], dv [B, H_kv, N, d], D)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    G = _group(H, Hkv)
    dq, dk, dv, D = bwd(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1), dout, scale, **kw)
    dk = dk.reshape(B, Hkv, G, N, d).sum(axis=2)
    dv = dv.reshape(B, Hkv, G, N, d).sum(axis=2)
    return dq, dk, dv, D


def fwd_decode(q, k, v, scale, causal=False, seqlens_k=None, heads=None, window_left=-1):
    """Attention of a short block of new query rows over a key/value cache, in
    fp64: the decode case that the page "FlashAttention — L3 Cross-Paper
    Synthesis" (section 3, the attack surface) names as left unoptimised,
    where one or a few query rows read a long cache.

    q [B, H, Nq, d]; k, v [B, H_kv, Nk, d] with H a multiple of H_kv (query
    head h reads K/V head h // (H / H_kv)); seqlens_k [B]: valid cache length
    L_b of each batch row (default Nk, clamped to [0, Nk]). The Nq query rows
    are the last Nq positions of the sequence: row i sits at position
    L_b - Nq + i. Without causal it sees keys j < L_b; with causal it sees
    j <= L_b - Nq + i as well. Written out row by row from the definition of
    softmax attention: scores scale * q . k_j over the allowed keys, their
    softmax, the weighted sum of V rows, and lse = log of the softmax
    denominator. A row with no allowed key has O = 0, lse = -inf.
    window_left >= 0 adds the sliding window: row i then sees only keys
    j >= L_b - Nq + i - window_left as well.

    heads: optional list of (b, h) to compute; the others stay O = 0,
    lse = -inf. Returns (o [B, H, Nq, d], lse [B, H, Nq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    G = _group(H, Hkv)
    o = np.zeros((B, H, Nq, d))
    lse = np.full((B, H, Nq), -np.inf)
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    for b, h in heads:
        L = Nk if seqlens_k is None else min(max(int(seqlens_k[b]), 0), Nk)
        kh, vh = k[b, h // G], v[b, h // G]
        for i in range(Nq):
            n = min(L, L - Nq + i + 1) if causal else L  # allowed keys are j < n
            j0 = max(0, L - Nq + i - window_left) if window_left >= 0 else 0  # ... and j >= j0
            if n <= j0:
                continue
            s = scale * (kh[j0:n] @ q[b, h, i])
            m = s.max()
            e = np.exp(s - m)
            den = e.sum()
            o[b, h, i] = (e @ vh[j0:n]) / den
            lse[b, h, i] = m + np.log(den)
    return o, lse


# ------------------------------------------------------------------ FP8 forward
# The cross-paper synthesis page on FlashAttention (section 2, the FA-3 entry)
# names FP8 with incoherent processing as FA-3's third Hopper technique. Read
# plainly: Q and K are multiplied by the same random orthogonal matrix M (a
# Hadamard matrix with random signs), which leaves Q K^T unchanged while
# spreading outlier channels, and Q, K, V are then stored as 8-bit floats
# (e4m3) with scales. The functions below restate those steps in fp64.

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Values of e4m3 byte codes: sign bit, 4 exponent bits (bias 7), 3
    mantissa bits; exponent 0 holds the subnormals 2^-6 * m/8; 0x7F / 0xFF
    are NaN (the format has no infinities)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


_E4M3_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # the 127 finite magnitudes, ascending


def e4m3_encode(x) -> np.ndarray:
    """Nearest e4m3 code to each finite x, ties to the even code (the one with
    mantissa bit 0), magnitudes above 448 saturated to 448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS, a, side="left")  # first magnitude >= a
    hi = np.minimum(hi, len(_E4M3_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS[hi] - a
    d_lo = a - _E4M3_POS[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return np.where(x < 0, code | 0x80, code).astype(np.uint8)


def hadamard(d: int) -> np.ndarray:
    """Sylvester's Hadamard matrix of order d (a power of two): H_1 = [1],
    H_2n = [[H_n, H_n], [H_n, -H_n]]."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotate(x, signs) -> np.ndarray:
    """x M with M = diag(signs) H / sqrt(d): an orthogonal matrix, so
    (q M)(k M)^T = q k^T; applied along the last axis. signs None: no
    rotation (M = I), the FP8 path without incoherent processing."""
    x = _f64(x)
    if signs is None:
        return x
    d = x.shape[-1]
    return (x * np.asarray(signs, dtype=np.float64)) @ hadamard(d) / np.sqrt(d)


def quantize_fp8(q, k, v, signs):
    """Quantisation for the FP8 forward, [B, H, N, d] inputs:
      Q' = Q M, K' = K M (M = I when signs is None); per-head scales s_q = amax|Q'| / 448, s_k likewise;
      per-(head, column) scales s_v[c] = amax_rows |V[:, c]| / 448;
      codes = nearest e4m3 of Q' / s_q, K' / s_k, V / s_v (a zero amax gives
      scale 1). Returns (q8, k8, v8 uint8 [B, H, N, d], s_q, s_k [B, H],
      s_v [B, H, d])."""
    qr, kr, v = rotate(q, signs), rotate(k, signs), _f64(v)

    def scale_of(amax):
        return np.where(amax > 0, amax / E4M3_MAX, 1.0)

    s_q = scale_of(np.abs(qr).max(axis=(2, 3)))
    s_k = scale_of(np.abs(kr).max(axis=(2, 3)))
    s_v = scale_of(np.abs(v).max(axis=2))
    q8 = e4m3_encode(qr / s_q[:, :, None, None])
    k8 = e4m3_encode(kr / s_k[:, :, None, None])
    v8 = e4m3_encode(v / s_v[:, :, None, :])
    return q8, k8, v8, s_q, s_k, s_v


def fwd_fp8(q8, k8, v8, s_q, s_k, s_v, scale, causal=False, seqlens_k=None):
    """Exact attention (the forward above, fp64) of the dequantised inputs
    Q^ = dec(q8) s_q, K^ = dec(k8) s_k, V^ = dec(v8) s_v: what the FP8 kernel
    computes before its own rounding of P. q8: uint8 [B, H, N, d]; k8, v8: uint8
    [B, Hkv, N, d] with Hkv dividing H (grouped K/V heads as in fwd_gqa)."""
    qh = e4m3_decode(q8) * np.asarray(s_q, dtype=np.float64)[:, :, None, None]
    kh = e4m3_decode(k8) * np.asarray(s_k, dtype=np.float64)[:, :, None, None]
    vh = e4m3_decode(v8) * np.asarray(s_v, dtype=np.float64)[:, :, None, :]
    return fwd_gqa(qh, kh, vh, scale, causal=causal, seqlens_k=seqlens_k)
