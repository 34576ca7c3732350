"""Grouped-query attention (shared K/V heads) on the GPU against the fp64 oracle."""
import math

import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa
from io_aware_exact_07_gb300 import inputs
from _parity import LSE_TOL, check_grads_per_head, lse_err, rel_fro, butterfly_dev, o_within_tol

pytestmark = pytest.mark.gpu


def draw(B, H, Hkv, N, d, seed, padding=None):
    """Q, dO with H heads and K, V with H_kv heads, from the seeded input recipe."""
    xq = inputs.draw_small(B, H, N, d, seed=seed, with_grad=True, padding=padding)
    xk = inputs.draw_small(B, Hkv, N, d, seed=seed + 1000, with_grad=False)
    return xq["q"], xk["k"], xk["v"], xq["do"], xq["seqlens"]


def run(B, H, Hkv, N, d, causal=False, p=0.0, padding=None, butterfly=False, seed=0):
    q, k, v, do, sl_cpu = draw(B, H, Hkv, N, d, seed, padding)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    sl = None if sl_cpu is None else sl_cpu.cuda()
    bm = butterfly_dev(N) if butterfly else None
    scale = 1.0 / math.sqrt(d)
    kw = dict(causal=causal, dropout_p=p, seed=seed, offset=3, block_mask=bm, seqlens_k=sl)
    o, lse = fa.fwd(qd, kd, vd, scale, **kw)
    dq, dk, dv = fa.bwd(qd, kd, vd, o, dod, lse, scale, **kw)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    okw = dict(causal=causal, dropout_p=p, seed=seed, offset=3,
               block_mask=None if bm is None else bm.cpu().numpy(),
               seqlens_k=None if sl_cpu is None else sl_cpu.numpy())
    f64 = lambda t: t.double().numpy()
    o_ref, lse_ref = oracle.fwd_gqa(f64(q), f64(k), f64(v), scale, **okw)
    dq_ref, dk_ref, dv_ref, _ = oracle.bwd_gqa(f64(q), f64(k), f64(v), f64(do), scale, **okw)
    ok, worst = o_within_tol(o.float().cpu().numpy(), o_ref)
    assert ok, f"O error exceeds its tolerance by {worst}"
    assert lse_err(lse.cpu().numpy(), lse_ref) <= LSE_TOL
    check_grads_per_head((name, g.float().cpu().numpy(), r) for name, g, r in
                         (("dQ", dq, dq_ref), ("dK", dk, dk_ref), ("dV", dv, dv_ref)))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hkv", [(4, 2), (4, 1), (8, 2)])
def test_gqa_dense(H, Hkv, d):
    run(1, H, Hkv, 300, d, seed=1)


@pytest.mark.parametrize("d", [64, 128])
def test_gqa_causal(d):
    run(2, 4, 2, 384, d, causal=True, seed=2)


def test_gqa_padding_dropout():
    run(2, 6, 3, 256, 64, p=0.1, padding=(100, 256), seed=3)


def test_mqa_causal_dropout_d128():
    run(1, 4, 1, 260, 128, causal=True, p=0.1, seed=4)


def test_gqa_block_mask():
    run(1, 4, 2, 1024, 64, butterfly=True, seed=5)


def test_gqa_equal_to_per_head_with_repeated_kv():
    # H_kv < H must give the same result as per-head attention on K/V repeated
    # over each group, with dK / dV summed over the group.
    B, H, Hkv, N, d = 1, 4, 2, 200, 64
    q, k, v, do, _ = draw(B, H, Hkv, N, d, seed=6)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o1, l1 = fa.fwd(qd, kd, vd, causal=True)
    dq1, dk1, dv1 = fa.bwd(qd, kd, vd, o1, dod, l1, causal=True)
    kr = kd.repeat_interleave(H // Hkv, dim=1).contiguous()
    vr = vd.repeat_interleave(H // Hkv, dim=1).contiguous()
    o2, l2 = fa.fwd(qd, kr, vr, causal=True)
    dq2, dk2, dv2 = fa.bwd(qd, kr, vr, o2, dod, l2, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(dq1, dq2)
    dk2s = dk2.float().view(B, Hkv, H // Hkv, N, d).sum(2)
    dv2s = dv2.float().view(B, Hkv, H // Hkv, N, d).sum(2)
    assert rel_fro(dk1.float().cpu().numpy(), dk2s.cpu().numpy()) < 1e-2
    assert rel_fro(dv1.float().cpu().numpy(), dv2s.cpu().numpy()) < 1e-2


def test_gqa_rejects_bad_head_counts():
    q = torch.zeros((1, 4, 128, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 3, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 4, 128), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd_gqa(q, k, k, o, lse, 1, 4, 3, 128, 64, 0.125) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd_gqa(q, k, k, o, lse, 1, 4, 0, 128, 64, 0.125) == fa.FA_ERR_INVALID_ARG
