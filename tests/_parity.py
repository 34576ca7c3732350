"""Shared helpers for the GPU-vs-oracle parity tests (inputs, tolerances)."""
import math

import numpy as np
import torch

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
