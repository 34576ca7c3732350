"""Sliding-window attention (fa_fwd_window / fa_bwd_window) on the GPU against
the fp64 oracle: O, lse, dQ, dK, dV within their tolerances, for windows that
end on and off tile boundaries, one- and two-sided, with causal, key padding,
dropout, grouped K/V heads and a block mask."""
import math

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa
from io_aware_exact_07_gb300 import inputs
from _parity import LSE_TOL, check_grads_per_head, lse_err, butterfly_dev, o_within_tol

pytestmark = pytest.mark.gpu


def run(B, H, N, d, window, causal=False, p=0.0, padding=None, Hkv=None, butterfly=False,
        seed=0):
    Hkv = H if Hkv is None else Hkv
    xq = inputs.draw_small(B, H, N, d, seed=seed, with_grad=True, padding=padding)
    xk = inputs.draw_small(B, Hkv, N, d, seed=seed + 1000, with_grad=False)
    q, do, sl_cpu = xq["q"], xq["do"], xq["seqlens"]
    k, v = (xk["k"], xk["v"]) if Hkv != H else (xq["k"], xq["v"])
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    sl = None if sl_cpu is None else sl_cpu.cuda()
    bm = butterfly_dev(N) if butterfly else None
    scale = 1.0 / math.sqrt(d)
    kw = dict(causal=causal, dropout_p=p, seed=seed, offset=5, block_mask=bm, seqlens_k=sl,
              window=window)
    o, lse = fa.fwd(qd, kd, vd, scale, **kw)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, scale, **kw)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    okw = dict(causal=causal, dropout_p=p, seed=seed, offset=5,
               block_mask=None if bm is None else bm.cpu().numpy(),
               seqlens_k=None if sl_cpu is None else sl_cpu.numpy(),
               window_left=window[0], window_right=window[1])
    f64 = lambda t: t.double().numpy()
    o_ref, lse_ref = oracle.fwd_gqa(f64(q), f64(k), f64(v), scale, **okw)
    # sum_j P_ij |v_j|: the scale of the bf16 rounding of P in rows with few keys
    o_abs, _ = oracle.fwd_gqa(f64(q), f64(k), np.abs(f64(v)), scale, **okw)
    dq_ref, dk_ref, dv_ref, _ = oracle.bwd_gqa(f64(q), f64(k), f64(v), f64(do), scale, **okw)
    ok, worst = o_within_tol(o.float().cpu().numpy(), o_ref, o_abs)
    assert ok, f"O error exceeds its tolerance by {worst}"
    assert lse_err(lse.cpu().numpy(), lse_ref) <= LSE_TOL
    check_grads_per_head((name, g.float().cpu().numpy(), r) for name, g, r in
                         (("dQ", dq, dq_ref), ("dK", dk, dk_ref), ("dV", dv, dv_ref)))
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("wl", [0, 1, 127, 128, 200, 513])
def test_causal_sliding_window(wl, d):
    run(1, 2, 1000, d, (wl, -1), causal=True, seed=wl + d)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window", [(100, 300), (0, 0), (257, 5), (-1, 130), (64, -1)])
def test_two_sided_window(window, d):
    run(2, 2, 900, d, window, seed=sum(window) + d)


def test_window_with_padding_dropout_and_grouped_heads():
    run(2, 4, 1100, 64, (300, -1), causal=True, p=0.1, padding=(200, 1100), Hkv=2, seed=7)


def test_window_with_block_mask():
    run(1, 2, 1024, 64, (200, 200), butterfly=True, seed=8)


def test_window_rows_without_keys():
    # non-causal window (0, 0) with key padding: rows beyond the padded length see nothing
    run(2, 1, 384, 128, (0, 0), padding=(100, 300), seed=9)


def test_window_covering_everything_equals_no_window():
    B, H, N, d = 1, 2, 700, 64
    x = inputs.draw_small(B, H, N, d, seed=10, with_grad=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o1, l1 = fa.fwd(q, k, v, causal=True)
    o2, l2 = fa.fwd(q, k, v, causal=True, window=(N, N))
    g1 = fa.bwd(q, k, v, o1, do, l1, causal=True)
    g2 = fa.bwd(q, k, v, o2, do, l2, causal=True, window=(N, N))
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_window_rejects_bad_bounds():
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd_window(q, q, q, o, lse, 1, 1, 1, 128, 64, 0.125, window_left=-2) == \
        fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_window(q, q, q, o, lse, 1, 1, 1, 128, 64, 0.125, window_right=-3) == \
        fa.FA_ERR_INVALID_ARG
