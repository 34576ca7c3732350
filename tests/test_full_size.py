"""Parity at the benchmark's full sizes, in the launch configuration bench.py
times (its Step object: the same entry points, grid and workspace). Whole
sampled heads are checked against the fp64 oracle (O, lse, dQ, dK, dV; for
grouped K/V heads dK, dV against the oracle's sum over the group), and an
identity that holds for every head at any size is checked on all of them:
without dropout each row of P sums to 1, so sum_j dV_j = sum_i dO_i."""
import pytest
import torch

import bench
import oracle
import io_aware_exact_07_gb300 as fa
from io_aware_exact_07_gb300 import inputs
from _parity import LSE_TOL, GRAD_RTOL, lse_err, rel_fro, o_within_tol

pytestmark = pytest.mark.gpu

# workload -> heads checked whole against the oracle
SAMPLED = {
    "gpt2_medium": [(0, 0), (63, 15), (17, 9)],
    "causal_4k": [(0, 0), (7, 31)],
    "long_16k_d64": [(0, 0), (0, 15)],
    "long_16k_d128": [(0, 0), (0, 15)],
    "butterfly_16k": [(0, 0), (3, 15)],
    "gqa_causal_4k": [(7, 31)],
    "sliding_16k": [(1, 31)],
}


@pytest.mark.parametrize("name", list(SAMPLED))
def test_full_size_workload(name):
    w = inputs.ALL[name]
    x = inputs.draw(w, with_grad=True)
    step = bench.Step(w, x, torch.device("cuda", 0))
    step.run()
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    G = w.H // w.kv_heads
    sl = None if x["seqlens"] is None else x["seqlens"].numpy()
    bm = None if step.bm is None else step.bm.cpu().numpy()
    kw = dict(causal=w.causal, dropout_p=w.dropout_p, seed=0, offset=0, block_mask=bm,
              seqlens_k=sl, H=w.H, window_left=w.window[0], window_right=w.window[1])
    f64 = lambda t: t.double().numpy()[None]
    for b, h in SAMPLED[name]:
        # the oracle on every query head of the sampled head's K/V group
        kvh = h // G
        group = [(b, kvh * G + g) for g in range(G)] if G > 1 else [(b, h)]
        kk, vv = f64(x["k"][b, kvh]), f64(x["v"][b, kvh])
        dk_sum = dv_sum = 0.0
        for bb, hh in group:
            q, do = f64(x["q"][bb, hh]), f64(x["do"][bb, hh])
            o_ref, lse_ref = oracle.fwd(q, kk, vv, w.scale, heads=[(bb, hh)], **kw)
            dq_ref, dk_ref, dv_ref, _ = oracle.bwd(q, kk, vv, do, w.scale, heads=[(bb, hh)], **kw)
            dk_sum = dk_sum + dk_ref[0]
            dv_sum = dv_sum + dv_ref[0]
            ok, worst = o_within_tol(step.o[bb, hh].float().cpu().numpy(), o_ref[0])
            assert ok, f"{name} head {(bb, hh)}: O error exceeds its tolerance by {worst}"
            assert lse_err(step.lse[bb, hh].cpu().numpy(), lse_ref[0]) <= LSE_TOL
            e = rel_fro(step.dq[bb, hh].float().cpu().numpy(), dq_ref[0])
            assert e <= GRAD_RTOL, f"{name} head {(bb, hh)}: dQ relative Frobenius error {e}"
        for nm, g, r in (("dK", step.dk, dk_sum), ("dV", step.dv, dv_sum)):
            e = rel_fro(g[b, kvh].float().cpu().numpy(), r)
            assert e <= GRAD_RTOL, f"{name} K/V head {(b, kvh)}: {nm} relative Frobenius error {e}"
    if w.dropout_p == 0.0:
        # every head: sum over keys of dV equals the sum over query rows of dO
        # (each query row here sees at least one key)
        dv_tot = step.dv.float().sum(dim=2)                                # [B, H_kv, d]
        do_tot = step.do.float().sum(dim=2).view(w.B, w.kv_heads, G, w.d).sum(dim=2)
        err = (dv_tot - do_tot).norm(dim=-1) / do_tot.norm(dim=-1).clamp_min(1e-6)
        assert float(err.max()) < 1e-2, f"{name}: worst head {float(err.max())}"
