"""FP8 forward at the benchmark's full size (B=8 H=32 N=4096 d=128, causal), in
the launch configuration bench.py times (fa_fp8_quantize then fa_fwd_fp8 on
the bench's own inputs and rotation signs). Sampled heads are checked whole
against the oracle: the quantiser's scales and codes, and the forward within
the FP8 accuracy contract on the GPU's own codes. On every head, a property
that holds at any size: causal row 0 sees key 0 alone, so its P is 2^5
exactly, O_0 is the dequantised V row of key 0 (up to bf16 rounding) and lse_0
is that one score."""
import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa
from io_aware_exact_07_gb300 import inputs
from _parity import e4m3_code_tol, fp8_contract, fp8_reference_terms

pytestmark = pytest.mark.gpu

SAMPLED = [(0, 0), (7, 31), (3, 17)]


def test_fp8_full_size_workload():
    w = inputs.FP8_CAUSAL
    assert w.causal and w.d == 128
    x = inputs.draw(w, with_grad=False)
    dev = torch.device("cuda", 0)
    signs = inputs.rotation_signs(w.d, seed=0)
    z = fa.fp8_quantize(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), signs.to(dev))
    o, lse = fa.fwd_fp8(z, w.scale, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    zc = {k: t.cpu() for k, t in z.items()}
    N = w.N
    v8 = zc["vt8"][..., :N].transpose(2, 3).contiguous()  # [B, H, N, d] key-major codes
    f64 = lambda t: t.double().numpy()
    s_np = f64(signs)
    for b, h in SAMPLED:
        q, k, v = (f64(x[n][b:b + 1, h:h + 1]) for n in ("q", "k", "v"))
        _, _, _, sq, sk, sv = oracle.quantize_fp8(q, k, v, s_np)
        assert np.allclose(zc["s_q"][b, h].item(), sq[0, 0], rtol=2e-6, atol=0)
        assert np.allclose(zc["s_k"][b, h].item(), sk[0, 0], rtol=2e-6, atol=0)
        assert np.allclose(zc["s_v"][b, h].numpy(), sv[0, 0], rtol=2e-6, atol=0)
        for name, codes, xr, sc in (
                ("q8", zc["q8"][b, h].numpy(), oracle.rotate(q[0, 0], s_np), zc["s_q"][b, h].item()),
                ("k8", zc["k8"][b, h].numpy(), oracle.rotate(k[0, 0], s_np), zc["s_k"][b, h].item()),
                ("v8", v8[b, h].numpy(), v[0, 0], zc["s_v"][b, h].double().numpy()[None, :])):
            y = xr / np.asarray(sc, dtype=np.float64)
            err = np.abs(oracle.e4m3_decode(codes) - y)
            tol = e4m3_code_tol(y)
            assert np.all(err <= tol), (name, (b, h), float((err - tol).max()))
        a = [zc["q8"][b:b + 1, h:h + 1].numpy(), zc["k8"][b:b + 1, h:h + 1].numpy(),
             v8[b:b + 1, h:h + 1].numpy(), zc["s_q"][b:b + 1, h:h + 1].double().numpy(),
             zc["s_k"][b:b + 1, h:h + 1].double().numpy(),
             zc["s_v"][b:b + 1, h:h + 1].double().numpy()]
        fp8_contract(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1],
                     *fp8_reference_terms(a, w.scale, True))
    # every head: row 0 attends to key 0 only
    q0 = oracle.e4m3_decode(zc["q8"][:, :, 0].numpy()) * zc["s_q"].double().numpy()[..., None]
    k0 = oracle.e4m3_decode(zc["k8"][:, :, 0].numpy()) * zc["s_k"].double().numpy()[..., None]
    v0 = oracle.e4m3_decode(v8[:, :, 0].numpy()) * zc["s_v"].double().numpy()
    lse0 = w.scale * (q0 * k0).sum(-1)
    o0 = o[:, :, 0].float().cpu().numpy().astype(np.float64)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(v0), 1e-30))) - 8.0)
    assert np.all(np.abs(o0 - v0) <= 1.5 * half_ulp + 1e-6), float(np.abs(o0 - v0).max())
    assert float(np.abs(lse[:, :, 0].cpu().numpy() - lse0).max()) <= 1e-3
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())
