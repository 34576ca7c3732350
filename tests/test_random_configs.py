"""Seeded sweep of random small configurations on the GPU against the fp64
oracle: head size, ragged N, causal, dropout, key padding, grouped K/V heads,
sliding windows and random block masks drawn together, so that option
combinations no hand-written case lists are also covered. Each case checks O
and lse, and dQ, dK, dV per head, at the parity tolerances."""
import math

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa
from io_aware_exact_07_gb300 import inputs
from _parity import LSE_TOL, check_grads_per_head, lse_err, o_within_tol

pytestmark = pytest.mark.gpu

N_CASES = 80


def _case(i):
    g = np.random.default_rng(1000 + i)
    d = int(g.choice([64, 128]))
    N = int(g.integers(1, 700))
    Hkv = int(g.choice([1, 2, 3]))
    G = int(g.choice([1, 1, 2, 4]))
    B = int(g.integers(1, 4))
    causal = bool(g.random() < 0.5)
    p = float(g.choice([0.0, 0.0, 0.1, 0.3]))
    padding = (int(g.integers(0, N + 1)), N) if g.random() < 0.4 else None
    window = (-1, -1)
    if g.random() < 0.35:
        window = (int(g.integers(-1, N + 1)), -1 if causal else int(g.integers(-1, N + 1)))
    nb = (N + 127) // 128
    block_mask = (g.random((nb, nb)) < 0.7).astype(np.uint8) if g.random() < 0.3 else None
    return dict(B=B, H=Hkv * G, Hkv=Hkv, N=N, d=d, causal=causal, p=p, padding=padding,
                window=window, block_mask=block_mask, seed=int(g.integers(0, 2**31)),
                offset=int(g.integers(0, 2**40)))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_config(i):
    c = _case(i)
    B, H, Hkv, N, d = c["B"], c["H"], c["Hkv"], c["N"], c["d"]
    xq = inputs.draw_small(B, H, N, d, seed=c["seed"] % 9973, with_grad=True, padding=c["padding"])
    xk = inputs.draw_small(B, Hkv, N, d, seed=c["seed"] % 9973 + 1, with_grad=False)
    q, do, sl_cpu = xq["q"], xq["do"], xq["seqlens"]
    k, v = xk["k"], xk["v"]
    scale = 1.0 / math.sqrt(d)
    bm = None if c["block_mask"] is None else torch.from_numpy(c["block_mask"]).cuda()
    sl = None if sl_cpu is None else sl_cpu.cuda()
    kw = dict(causal=c["causal"], dropout_p=c["p"], seed=c["seed"], offset=c["offset"],
              block_mask=bm, seqlens_k=sl, window=c["window"])
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    fa.fa_device_status(clear=True)
    o, lse = fa.fwd(qd, kd, vd, scale, **kw)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, scale, **kw)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK, c
    okw = dict(causal=c["causal"], dropout_p=c["p"], seed=c["seed"], offset=c["offset"],
               block_mask=c["block_mask"], seqlens_k=None if sl_cpu is None else sl_cpu.numpy(),
               window_left=c["window"][0], window_right=c["window"][1])
    f64 = lambda t: t.double().numpy()
    o_ref, lse_ref = oracle.fwd_gqa(f64(q), f64(k), f64(v), scale, **okw)
    o_abs, _ = oracle.fwd_gqa(f64(q), f64(k), np.abs(f64(v)), scale, **okw)
    dq_ref, dk_ref, dv_ref, _ = oracle.bwd_gqa(f64(q), f64(k), f64(v), f64(do), scale, **okw)
    ok, worst = o_within_tol(o.float().cpu().numpy(), o_ref, o_abs)
    assert ok, f"{c}: O error exceeds its tolerance by {worst}"
    assert lse_err(lse.cpu().numpy(), lse_ref) <= LSE_TOL, c
    check_grads_per_head((name, g.float().cpu().numpy(), r) for name, g, r in
                         (("dQ", dq, dq_ref), ("dK", dk, dk_ref), ("dV", dv, dv_ref)))
