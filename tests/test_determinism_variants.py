"""Bitwise determinism of the paths beyond the per-head forward and backward:
grouped-query dK/dV (group sums formed on chip), the sliding window, the decode
split and combine, and the FP8 forward. Each is run twice on the same inputs."""
import torch
import pytest

import io_aware_exact_07_gb300 as fa
from io_aware_exact_07_gb300 import inputs

pytestmark = pytest.mark.gpu


def _pair(fn):
    a = fn()
    b = fn()
    torch.cuda.synchronize()
    return a, b


def test_gqa_and_window_backward_are_deterministic():
    x = inputs.draw_small(2, 8, 900, 64, seed=21, with_grad=True, padding=(300, 900))
    q, do = x["q"].cuda(), x["do"].cuda()
    k, v = (x[n][:, :2].contiguous().cuda() for n in ("k", "v"))  # 2 K/V heads for 8 query heads
    sl = x["seqlens"].cuda()
    kw = dict(causal=True, dropout_p=0.1, seed=3, seqlens_k=sl, window=(200, -1))

    def run():
        o, lse = fa.fwd(q, k, v, **kw)
        return (o, lse) + fa.bwd(q, k, v, o, do, lse, **kw)
    a, b = _pair(run)
    for s, t in zip(a, b):
        assert torch.equal(s, t)


@pytest.mark.parametrize("ctas", [0, 7])
def test_decode_is_deterministic(ctas):
    w = inputs.DecodeWorkload("t", 2, 8, 2, 3, 3000, 128, causal=True, lengths=(100, 3000), seed=22)
    x = inputs.draw_decode(w)
    q, k, v, sl = x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["seqlens"].cuda()
    a, b = _pair(lambda: fa.decode(q, k, v, causal=True, seqlens_k=sl, num_ctas=ctas))
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_forward_is_deterministic():
    x = inputs.draw_small(1, 4, 1000, 128, seed=23, with_grad=False)
    z = fa.fp8_quantize(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(),
                        inputs.rotation_signs(128).cuda())
    a, b = _pair(lambda: fa.fwd_fp8(z, 0.0884, causal=True))
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
