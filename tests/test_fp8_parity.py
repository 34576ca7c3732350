"""FP8 forward (fa_fp8_quantize, fa_fwd_fp8) on the GPU against the fp64
oracle. The quantiser: scales as the oracle's, every code within half an e4m3
gap of the oracle's rotated, scaled value. The forward, on e4m3 codes drawn by
the input module: within the FP8 accuracy contract of exact attention of the
dequantised inputs. End to end from bf16 inputs with outlier channels: the
rotation lowers the error against exact attention."""
import math

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa
from io_aware_exact_07_gb300 import inputs
from _parity import e4m3_code_tol, fp8_contract, fp8_reference_terms

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,rot,Hkv", [(300, True, 3), (1000, True, 3), (129, False, 3),
                                       (300, True, 1), (520, False, 2)])
def test_quantiser_matches_oracle(N, rot, Hkv):
    B, H, d = 2, 3 if Hkv != 2 else 4, 128
    x = inputs.draw_small(B, H, N, d, seed=N, with_grad=False)
    q, k, v = x["q"], x["k"][:, :Hkv].contiguous(), x["v"][:, :Hkv].contiguous()
    k[..., 5] *= 30  # an outlier channel
    signs = inputs.rotation_signs(d, seed=1)
    z = fa.fp8_quantize(q.cuda(), k.cuda(), v.cuda(), signs.cuda() if rot else None)
    torch.cuda.synchronize()
    f64 = lambda t: t.double().numpy()
    s_np = f64(signs) if rot else None
    q8r, k8r, v8r, sq, sk, sv = oracle.quantize_fp8(f64(q), f64(k), f64(v), s_np)
    for name, ref in (("s_q", sq), ("s_k", sk), ("s_v", sv)):
        assert np.allclose(z[name].cpu().numpy(), ref, rtol=2e-6, atol=0), name
    Np = fa.fa_fp8_vt_stride(N)
    vt = z["vt8"].cpu().numpy()
    assert vt.shape == (B, Hkv, d, Np) and np.all(vt[..., N:] == 0)
    v8 = np.ascontiguousarray(np.swapaxes(vt[..., :N], 2, 3))
    for name, codes, xr, sc in (("q8", z["q8"].cpu().numpy(), oracle.rotate(f64(q), s_np),
                                 z["s_q"].cpu().numpy()[:, :, None, None]),
                                ("k8", z["k8"].cpu().numpy(), oracle.rotate(f64(k), s_np),
                                 z["s_k"].cpu().numpy()[:, :, None, None]),
                                ("v8", v8, f64(v), z["s_v"].cpu().numpy()[:, :, None, :])):
        y = xr / sc.astype(np.float64)  # the value in code units, with the GPU's scale
        err = np.abs(oracle.e4m3_decode(codes) - y)
        tol = e4m3_code_tol(y)
        assert np.all(err <= tol), (name, float((err - tol).max()))


@pytest.mark.parametrize("N,causal,padding", [(256, False, None), (1000, True, None),
                                              (777, False, (100, 777)), (2048, True, (900, 2048)),
                                              (1, False, None), (17, True, None),
                                              (300, False, (0, 40))])
def test_fp8_forward_within_contract(N, causal, padding):
    B, H, d = 2, 2, 128
    x = inputs.draw_fp8_codes(B, H, N, d, seed=N)
    Np = fa.fa_fp8_vt_stride(N)
    vt = torch.zeros((B, H, d, Np), dtype=torch.uint8)
    vt[..., :N] = x["v8"].transpose(2, 3)
    sl = None
    if padding is not None:
        sl = inputs.draw_small(B, 1, N, 64, seed=N, with_grad=False, padding=padding)["seqlens"]
    scale = 1.0 / math.sqrt(d)
    z = dict(q8=x["q8"].cuda(), k8=x["k8"].cuda(), vt8=vt.contiguous().cuda(),
             s_q=x["s_q"].cuda(), s_k=x["s_k"].cuda(), s_v=x["s_v"].cuda())
    o, lse = fa.fwd_fp8(z, scale, causal=causal, seqlens_k=None if sl is None else sl.cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    a = [t.numpy() for t in (x["q8"], x["k8"], x["v8"], x["s_q"].double(), x["s_k"].double(),
                             x["s_v"].double())]
    sl_np = None if sl is None else sl.numpy()
    fp8_contract(o, lse, *fp8_reference_terms(a, scale, causal, sl_np))


@pytest.mark.parametrize("H,Hkv,N,causal,padding", [(8, 2, 1000, True, None),
                                                    (6, 1, 777, False, (100, 777)),
                                                    (4, 2, 300, True, (0, 300))])
def test_fp8_grouped_heads_within_contract(H, Hkv, N, causal, padding):
    """Grouped K/V heads: q8 [B, H, N, d] with k8, vt8 [B, Hkv, ...]."""
    B, d = 2, 128
    xq = inputs.draw_fp8_codes(B, H, N, d, seed=N + H)
    xk = inputs.draw_fp8_codes(B, Hkv, N, d, seed=N + 100 * Hkv)
    Np = fa.fa_fp8_vt_stride(N)
    vt = torch.zeros((B, Hkv, d, Np), dtype=torch.uint8)
    vt[..., :N] = xk["v8"].transpose(2, 3)
    sl = None
    if padding is not None:
        sl = inputs.draw_small(B, 1, N, 64, seed=N, with_grad=False, padding=padding)["seqlens"]
    scale = 1.0 / math.sqrt(d)
    z = dict(q8=xq["q8"].cuda(), k8=xk["k8"].cuda(), vt8=vt.contiguous().cuda(),
             s_q=xq["s_q"].cuda(), s_k=xk["s_k"].cuda(), s_v=xk["s_v"].cuda())
    o, lse = fa.fwd_fp8(z, scale, causal=causal, seqlens_k=None if sl is None else sl.cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    a = [t.numpy() for t in (xq["q8"], xk["k8"], xk["v8"], xq["s_q"].double(),
                             xk["s_k"].double(), xk["s_v"].double())]
    sl_np = None if sl is None else sl.numpy()
    fp8_contract(o, lse, *fp8_reference_terms(a, scale, causal, sl_np))


def test_fp8_grouped_heads_equal_repeated_heads():
    """From bf16 inputs: quantising and running the forward with Hkv K/V heads
    gives bit for bit what the same calls give with each K/V head repeated for
    its group (the per-head scales, codes and every product are the same)."""
    B, H, Hkv, N, d = 2, 6, 2, 700, 128
    xq = inputs.draw_small(B, H, N, d, seed=41, with_grad=False)
    xk = inputs.draw_small(B, Hkv, N, d, seed=42, with_grad=False)
    q, k, v = xq["q"].cuda(), xk["k"].cuda(), xk["v"].cuda()
    signs = inputs.rotation_signs(d, seed=3).cuda()
    G = H // Hkv
    kr, vr = (t.repeat_interleave(G, dim=1).contiguous() for t in (k, v))
    zg = fa.fp8_quantize(q, k, v, signs)
    zr = fa.fp8_quantize(q, kr, vr, signs)
    og, lg = fa.fwd_fp8(zg, 0.09, causal=True)
    orr, lr = fa.fwd_fp8(zr, 0.09, causal=True)
    torch.cuda.synchronize()
    for name in ("k8", "vt8", "s_k", "s_v"):
        assert torch.equal(zg[name].repeat_interleave(G, dim=1), zr[name]), name
    assert torch.equal(zg["q8"], zr["q8"]) and torch.equal(zg["s_q"], zr["s_q"])
    assert torch.equal(og, orr) and torch.equal(lg, lr)


def test_fp8_end_to_end_rotation_helps_with_outliers():
    """bf16 inputs whose K has outlier channels: quantised with the rotation the
    FP8 forward lands closer to exact attention than quantised without it, in
    the scores (lse) and in O. (e4m3 is a floating-point format, so a large
    scale does not coarsen the small channels as an integer grid would; the
    gain is modest, and O's error is dominated by the e4m3 rounding of P.)"""
    B, H, N, d = 1, 4, 1024, 128
    x = inputs.draw_small(B, H, N, d, seed=77, with_grad=False)
    q, k, v = x["q"], x["k"], x["v"]
    k[..., 3] *= 40
    k[..., 77] *= 25
    scale = 1.0 / math.sqrt(d)
    f64 = lambda t: t.double().numpy()
    o_exact, lse_exact = oracle.fwd(f64(q), f64(k), f64(v), scale, causal=True)
    errs = {}
    for rot in (True, False):
        signs = inputs.rotation_signs(d, seed=5).cuda() if rot else None
        z = fa.fp8_quantize(q.cuda(), k.cuda(), v.cuda(), signs)
        o, lse = fa.fwd_fp8(z, scale, causal=True)
        torch.cuda.synchronize()
        errs[rot] = (float(np.sqrt(np.mean((o.float().cpu().numpy() - o_exact) ** 2))),
                     float(np.sqrt(np.mean((lse.cpu().numpy() - lse_exact) ** 2))))
    print("FP8 RMS error vs exact (O, lse): rotated", errs[True], "not rotated", errs[False])
    assert errs[True][0] < errs[False][0] and errs[True][1] < errs[False][1], errs


def test_fp8_long_runs_of_empty_units():
    """Key lengths 0 for all batch rows but the last, with several work units per
    CTA: the empty rows give O = 0 and lse = -inf, and the last row equals the
    same kernel run on it alone, bit for bit."""
    B, H, N, d = 16, 16, 1024, 128
    x = inputs.draw_fp8_codes(B, H, N, d, seed=5)
    Np = fa.fa_fp8_vt_stride(N)
    vt = torch.zeros((B, H, d, Np), dtype=torch.uint8)
    vt[..., :N] = x["v8"].transpose(2, 3)
    sl = torch.zeros(B, dtype=torch.int32)
    sl[-1] = N - 5
    z = dict(q8=x["q8"].cuda(), k8=x["k8"].cuda(), vt8=vt.contiguous().cuda(),
             s_q=x["s_q"].cuda(), s_k=x["s_k"].cuda(), s_v=x["s_v"].cuda())
    z1 = {n: t[-1:].contiguous() for n, t in z.items()}
    o, lse = fa.fwd_fp8(z, 0.088, seqlens_k=sl.cuda())
    o1, lse1 = fa.fwd_fp8(z1, 0.088, seqlens_k=sl[-1:].cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    assert torch.all(o[:-1] == 0) and torch.all(torch.isneginf(lse[:-1]))
    assert torch.equal(o[-1:], o1) and torch.equal(lse[-1:], lse1)


def test_fp8_rejects_bad_arguments():
    q8 = torch.zeros((1, 1, 128, 64), dtype=torch.uint8, device="cuda")
    o = torch.empty((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    s = torch.ones(128, dtype=torch.float32, device="cuda")
    assert fa.fa_fwd_fp8(q8, q8, q8, s, s, s, o, lse, 1, 1, 128, 64, 0.125) == \
        fa.FA_ERR_UNSUPPORTED
    assert fa.fa_fwd_fp8(q8, q8, q8, s, s, s, o, lse, 1, 1, 0, 128, 0.125) == \
        fa.FA_ERR_INVALID_ARG
    assert fa.fa_fp8_workspace_size(1, 1, 64) == 0
    kv = torch.zeros((1, 3, 128, 128), dtype=torch.uint8, device="cuda")
    q3 = torch.zeros((1, 4, 128, 128), dtype=torch.uint8, device="cuda")
    o4 = torch.empty((1, 4, 128, 128), dtype=torch.bfloat16, device="cuda")
    l4 = torch.empty((1, 4, 128), dtype=torch.float32, device="cuda")
    # 4 query heads cannot share 3 K/V heads
    assert fa.fa_fwd_fp8_gqa(q3, kv, kv, s, s, s, o4, l4, 1, 4, 3, 128, 128, 0.125) == \
        fa.FA_ERR_INVALID_ARG
