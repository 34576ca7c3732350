"""The longest sequences: N = 131072 (1024 key tiles per head, the row index
of the last head near 2^18), d = 64 and 128, with and without the causal mask,
through fa_fwd / fa_bwd. Sampled query rows are checked against the fp64
oracle one block at a time: a block of the last rows is the oracle's
short-query case (query rows at the end of the key sequence, which is where
the causal mask of a square problem places them), a middle block likewise
without the mask, and under the mask the first 128 rows see only the first 128
keys (a square problem of its own). On every head the backward is checked
through an identity that holds at any size without dropout: each row of P
sums to 1, so the sum over keys of dV equals the sum over query rows of dO."""
import math

import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa
from io_aware_exact_07_gb300 import inputs
from _parity import LSE_TOL, lse_err, o_within_tol

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_longest_sequence(d, causal):
    B, H, N = 1, 2, 131072
    x = inputs.draw_small(B, H, N, d, seed=d + int(causal), with_grad=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, scale, causal=causal)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, scale, causal=causal)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    f64 = lambda t: t.double().numpy()
    kk, vv = f64(x["k"]), f64(x["v"])
    blocks = [(N - 128, N)] + ([] if causal else [(N // 2 - 64, N // 2 + 64)])
    o_cpu, lse_cpu = o.float().cpu().numpy(), lse.cpu().numpy()
    for r0, r1 in blocks:
        # rows r0 .. r1-1 at the end of a key sequence of length r1 (keys >= r1 unused
        # without the mask only when r1 = N)
        kv_len = N if not causal else r1
        ro, rl = oracle.fwd_decode(f64(x["q"][:, :, r0:r1]), kk[:, :, :kv_len], vv[:, :, :kv_len],
                                   scale, causal=causal)
        ok, worst = o_within_tol(o_cpu[:, :, r0:r1], ro)
        assert ok, f"rows {r0}..{r1}: O error exceeds its tolerance by {worst}"
        assert lse_err(lse_cpu[:, :, r0:r1], rl) <= LSE_TOL
    if causal:
        ro, rl = oracle.fwd(f64(x["q"][:, :, :128]), kk[:, :, :128], vv[:, :, :128], scale,
                            causal=True)
        ok, worst = o_within_tol(o_cpu[:, :, :128], ro)
        assert ok, f"first rows: O error exceeds its tolerance by {worst}"
        assert lse_err(lse_cpu[:, :, :128], rl) <= LSE_TOL
    dv_tot = dv.float().sum(dim=2)
    do_tot = do.float().sum(dim=2)
    err = (dv_tot - do_tot).norm(dim=-1) / do_tot.norm(dim=-1).clamp_min(1e-6)
    assert float(err.max()) < 1e-2, float(err.max())
    for g in (dq, dk, dv):
        assert bool(torch.isfinite(g).all())
