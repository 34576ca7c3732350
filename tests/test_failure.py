"""Failure detection without a GPU fault: a device-side wait that nothing
completes runs out after a short limit, the kernel records FA_ERR_TIMEOUT and
returns, and the context stays usable for the next call."""
import math

import numpy as np
import pytest
import torch

import io_aware_exact_07_gb300 as fa
import oracle
from _parity import make_case, oracle_heads

pytestmark = pytest.mark.gpu


def test_stalled_wait_times_out_and_context_survives():
    x = make_case(1, 2, 512, 64, with_grad=False)
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
                       oracle_heads(x["v"], heads), 1 / math.sqrt(64), heads=heads, H=2)
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
