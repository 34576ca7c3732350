"""Shared helpers for the GPU-vs-oracle parity tests (inputs, tolerances)."""
import math

import numpy as np

import oracle
from io_aware_exact_07_gb300 import inputs

# Accuracy bars for bf16 inputs with fp32 accumulation: O max-abs, lse max-abs,
# and relative Frobenius error of dQ, dK, dV.
O_TOL = 1e-2
LSE_TOL = 1e-3
GRAD_RTOL = 2e-2


def make_case(B, H, N, d, seed=0, padding=None, with_grad=True):
    return inputs.draw_small(B, H, N, d, seed=seed, with_grad=with_grad, padding=padding)


def to_dev(x):
    return None if x is None else x.cuda()


def oracle_heads(x, heads):
    """Slice [B, H, N, d] bf16 tensor to fp64 [len(heads), N, d] for the given (b, h)."""
    return np.stack([x[b, h].double().numpy() for b, h in heads])


def o_within_tol(gpu, ref, o_abs=None):
    """O against the oracle: max-abs error 1e-2, except where the output's own
    bf16 storage cannot resolve that (|O| >= 4, where half a bf16 ulp is
    already 2**-6); there 1.5 half-ulps of the reference value are allowed.
    With o_abs = sum_j P_ij |v_j| (the oracle applied to |V|), the bound also
    holds the worst case of rounding each P weight to bf16 for the PV product,
    2**-8 * o_abs, which exceeds 1e-2 only in rows that see a few keys with
    large values. Returns (ok, worst excess of |gpu - ref| over the element's
    tolerance)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mag = np.maximum(np.abs(ref), 1e-30)
    half_ulp = np.exp2(np.floor(np.log2(mag)) - 8.0)
    bound = 1.5 * half_ulp
    if o_abs is not None:
        bound = bound + np.exp2(-8.0) * np.asarray(o_abs, dtype=np.float64)
    tol = np.maximum(O_TOL, bound)
    excess = np.abs(gpu - ref) - tol
    worst = float(np.max(excess)) if excess.size else -1.0
    return worst <= 0.0, worst


def rel_fro(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def lse_err(gpu, ref):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    both_inf = np.isneginf(gpu) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):
        diff = np.where(both_inf, 0.0, np.abs(gpu - ref))
    return float(np.max(diff)) if diff.size else 0.0


def butterfly_dev(N):
    from io_aware_exact_07_gb300 import fa_butterfly_mask
    nb = math.ceil(N / 128)
    return fa_butterfly_mask(nb).cuda()


def e4m3_gap(y):
    """Distance between the two e4m3 magnitudes around |y|."""
    mags = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    idx = np.minimum(np.searchsorted(mags, np.abs(y)), len(mags) - 1)
    return mags[idx] - mags[np.maximum(idx - 1, 0)]


def e4m3_code_tol(y):
    """Allowed |dec(code) - y| for a code of the value y (code units, GPU's
    scale): half a gap, plus the fp32 rounding of the GPU's rotation and
    scaling. The rotation is a 128-point Walsh-Hadamard transform in 7
    add/subtract stages after one multiply by sign / sqrt(128) / scale: each
    step rounds partial sums whose magnitudes add up to at most
    sum_j |x_j f_j| <= ||y_row||_2, so an element is off by at most about
    9 u ||y_row||_2 (u = 2^-24) before its e4m3 rounding, which can then go to
    the other side of a tie; 2^-20 leaves margin. The 2^-22 |y| term covers
    the rounding of 1 / scale."""
    row = np.sqrt((y ** 2).sum(axis=-1, keepdims=True))
    return e4m3_gap(y) / 2 + 2.0 ** -20 * row + 2.0 ** -22 * np.abs(y)


def fp8_contract(o, lse, o_ref, lse_ref, o_abs, vsum_abs):
    """|O - O^| <= 2^-4 sum P|v^| + 2^-15 sum |v^| + 1.5 bf16 half-ulps; lse 1e-3. The
    second term: P's e4m3 rounding is absolute (at most 2^-10, half the smallest
    subnormal) below 2^-6, relative to a row maximum of at least 2^5."""
    o = o.float().cpu().numpy().astype(np.float64)
    mag = np.maximum(np.abs(o_ref), 1e-30)
    half_ulp = np.exp2(np.floor(np.log2(mag)) - 8.0)
    tol = 2.0 ** -4 * o_abs + 2.0 ** -15 * vsum_abs + 1.5 * half_ulp + 1e-6
    excess = np.abs(o - o_ref) - tol
    assert excess.max() <= 0, f"FP8 contract exceeded by {excess.max()}"
    assert lse_err(lse.cpu().numpy(), lse_ref) <= LSE_TOL
    return float(np.abs(o - o_ref).max())


def fp8_dequantised(a):
    """Q^, K^, V^ (fp64) of (q8, k8, v8 [.., N, d] uint8, s_q, s_k, s_v) with V
    in key-major layout."""
    qh = oracle.e4m3_decode(a[0]) * a[3][:, :, None, None]
    kh = oracle.e4m3_decode(a[1]) * a[4][:, :, None, None]
    vh = oracle.e4m3_decode(a[2]) * a[5][:, :, None, :]
    return qh, kh, vh


def fp8_reference_terms(a, scale, causal, seqlens_k=None):
    """The oracle's FP8 forward of codes and scales `a` (see fp8_dequantised) and
    the two weights of the FP8 contract: sum_j P_ij |v^_j| and sum over each
    row's visible keys of |v^_j|."""
    B, _, N, _ = a[0].shape
    o_ref, lse_ref = oracle.fwd_fp8(*a, scale, causal=causal, seqlens_k=seqlens_k)
    qh, kh, vh = fp8_dequantised(a)
    o_abs, _ = oracle.fwd_gqa(qh, kh, np.abs(vh), scale, causal=causal, seqlens_k=seqlens_k)
    # uniform attention (q = 0) times the number of visible keys
    mean_abs, _ = oracle.fwd_gqa(np.zeros_like(qh), kh, np.abs(vh), scale, causal=causal,
                                 seqlens_k=seqlens_k)
    L = np.full(B, N) if seqlens_k is None else np.clip(seqlens_k, 0, N)
    rows = np.arange(N)
    count = np.minimum(rows[None, :] + 1, L[:, None]) if causal else np.repeat(L[:, None], N, 1)
    return o_ref, lse_ref, o_abs, mean_abs * count[:, None, :, None]


def check_grads_per_head(named):
    """named: (name, gpu, oracle) triples of [..., N, d] gradients. The relative
    Frobenius error is taken head by head over the leading axes, so one bad
    head cannot hide under the norm of the others. A head whose exact
    gradient is zero (one visible key: dS = P (dP - D) = 0; a key no query
    sees) must come back within 1e-2 of zero: its GPU value is the bf16
    rounding residue of D = rowsum(dO * O)."""
    for name, g, r in named:
        g = np.asarray(g, dtype=np.float64)
        r = np.asarray(r, dtype=np.float64)
        assert g.shape == r.shape, name
        assert np.isfinite(g).all(), name
        gh = g.reshape(-1, *g.shape[-2:])
        rh = r.reshape(-1, *r.shape[-2:])
        for n in range(gh.shape[0]):
            if np.linalg.norm(rh[n]) == 0:
                assert np.abs(gh[n]).max() <= 1e-2, f"{name} head {n}"
                continue
            e = rel_fro(gh[n], rh[n])
            assert e <= GRAD_RTOL, f"{name} head {n}: relative Frobenius error {e}"
