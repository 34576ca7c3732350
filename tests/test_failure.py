"""Failure detection without a GPU fault: a device-side wait that nothing
completes runs out after a short limit, the kernel records FA_ERR_TIMEOUT and
returns, and the context stays usable for the next call."""
import math

import numpy as np
import pytest
import torch

import io_aware_exact_07_gb300 as fa
import oracle
from _parity import GRAD_RTOL, make_case, oracle_heads, rel_fro

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d", [64, 128])  # the two forward kernels
def test_stalled_wait_times_out_and_context_survives(d):
    x = make_case(1, 2, 512, d, with_grad=False)
    q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
    fa.fa_device_status(clear=True)
    fa.fa_set_wait_timeout_ns(200_000_000)  # 0.2 s
    try:
        fa.fa_test_inject_stall(1)
        o, lse = fa.fwd(q, k, v)
        assert fa.fa_device_status(clear=True) == fa.FA_ERR_TIMEOUT
    finally:
        fa.fa_test_inject_stall(0)
        fa.fa_set_wait_timeout_ns(4_000_000_000)
    # the hook was consumed: the next call is a normal, correct forward
    o, lse = fa.fwd(q, k, v)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    heads = [(0, 0), (0, 1)]
    ro, _ = oracle.fwd(oracle_heads(x["q"], heads), oracle_heads(x["k"], heads),
                       oracle_heads(x["v"], heads), 1 / math.sqrt(d), heads=heads, H=2)
    got = np.stack([o[0, h].float().cpu().numpy() for h in range(2)])
    assert np.abs(got - ro).max() <= 1e-2


def _stalled(call):
    """Run `call` with the stall hook armed and a 0.2 s wait limit; return the
    recorded device status."""
    fa.fa_device_status(clear=True)
    fa.fa_set_wait_timeout_ns(200_000_000)
    try:
        fa.fa_test_inject_stall(1)
        call()
        return fa.fa_device_status(clear=True)
    finally:
        fa.fa_test_inject_stall(0)
        fa.fa_set_wait_timeout_ns(4_000_000_000)


def test_decode_stall_times_out_and_next_call_is_correct():
    q = torch.randn((2, 4, 1, 128), device="cuda").to(torch.bfloat16)
    k, v = (torch.randn((2, 2, 3000, 128), device="cuda").to(torch.bfloat16) for _ in range(2))
    assert _stalled(lambda: fa.decode(q, k, v, num_ctas=5)) == fa.FA_ERR_TIMEOUT
    o, lse = fa.decode(q, k, v, num_ctas=5)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    f64 = lambda t: t.double().cpu().numpy()
    ro, rl = oracle.fwd_decode(f64(q), f64(k), f64(v), 1 / math.sqrt(128))
    assert np.abs(o.float().cpu().numpy() - ro).max() <= 1e-2
    assert np.abs(lse.cpu().numpy() - rl).max() <= 1e-3


def test_fp8_forward_stall_times_out_and_next_call_works():
    x = make_case(1, 2, 512, 128, with_grad=False)
    q, k, v = (t.cuda() for t in (x["q"], x["k"], x["v"]))
    z = fa.fp8_quantize(q, k, v, None)
    assert _stalled(lambda: fa.fwd_fp8(z, 1 / math.sqrt(128))) == fa.FA_ERR_TIMEOUT
    o, lse = fa.fwd_fp8(z, 1 / math.sqrt(128))
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    assert torch.isfinite(lse).all() and torch.isfinite(o.float()).all()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mode,kernel", [(2, "dK/dV"), (3, "dQ")])
def test_backward_stall_times_out_and_next_call_is_correct(d, mode, kernel):
    """The backward kernels' bounded waits: the armed kernel (mode 2: dK/dV,
    mode 3: dQ) gives up after the short limit and returns FA_ERR_TIMEOUT; the
    hook is consumed, so the next backward runs normally and matches the
    oracle."""
    B, H, N = 1, 2, 384
    x = make_case(B, H, N, d, seed=d + mode)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    scale = 1 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, scale, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    fa.fa_device_status(clear=True)
    fa.fa_set_wait_timeout_ns(200_000_000)
    try:
        fa.fa_test_inject_stall(mode)
        fa.bwd(q, k, v, o, do, lse, scale, causal=True)
        assert fa.fa_device_status(clear=True) == fa.FA_ERR_TIMEOUT, kernel
    finally:
        fa.fa_test_inject_stall(0)
        fa.fa_set_wait_timeout_ns(4_000_000_000)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, scale, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    heads = [(0, h) for h in range(H)]
    ref = oracle.bwd(oracle_heads(x["q"], heads), oracle_heads(x["k"], heads),
                     oracle_heads(x["v"], heads), oracle_heads(x["do"], heads), scale,
                     causal=True, heads=heads, H=H)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref[:3]):
        for h in range(H):
            e = rel_fro(g[0, h].float().cpu().numpy(), r[h])
            assert e <= GRAD_RTOL, f"{name} head {h}: {e}"


def test_stall_hook_waits_for_its_own_kind_of_launch():
    """A hook armed for the dQ kernel is not taken by a forward or a dK/dV
    launch: those complete normally, and the next dQ kernel takes it."""
    x = make_case(1, 1, 256, 64)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    fa.fa_device_status(clear=True)
    fa.fa_set_wait_timeout_ns(200_000_000)
    try:
        fa.fa_test_inject_stall(3)
        o, lse = fa.fwd(q, k, v)
        ws = torch.empty(fa.fa_bwd_workspace_size(1, 1, 256, 64), dtype=torch.uint8,
                         device="cuda")
        dk, dv = torch.empty_like(k), torch.empty_like(v)
        assert fa.fa_bwd_preprocess(o, do, 1, 1, 256, 64, ws, ws.numel()) == fa.FA_OK
        assert fa.fa_bwd_dkdv(q, k, v, do, lse, dk, dv, 1, 1, 256, 64, 0.125, workspace=ws,
                              workspace_bytes=ws.numel()) == fa.FA_OK
        assert fa.fa_device_status(clear=True) == fa.FA_OK
        dq = torch.empty_like(q)
        assert fa.fa_bwd_dq(q, k, v, do, lse, dq, 1, 1, 256, 64, 0.125, workspace=ws,
                            workspace_bytes=ws.numel()) == fa.FA_OK
        assert fa.fa_device_status(clear=True) == fa.FA_ERR_TIMEOUT
    finally:
        fa.fa_test_inject_stall(0)
        fa.fa_set_wait_timeout_ns(4_000_000_000)
