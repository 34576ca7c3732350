"""fa_bwd_noalloc, the backward entry point for callers that cannot allocate
device memory (for example a plugin inside a framework that owns all device
memory and hands out no workspace, or code that must avoid cudaMalloc/cudaFree
because they can synchronise the device). It must give the same gradients as
fa_bwd with a caller-provided workspace, on consecutive calls that share its
static scratch array.

This file is collected last so that, in a run that stops at the first
failure, every other test has already run."""
import ctypes
import math

import numpy as np
import pytest
import torch

import io_aware_exact_07_gb300 as fa
from _parity import GRAD_RTOL, make_case, rel_fro

pytestmark = pytest.mark.gpu


def _noalloc_raw(lib, q, k, v, o, do, lse, dq, dk, dv, B, H, N, d, scale, causal, p, seed,
                 offset, bm, sl):
    vp = ctypes.c_void_p
    ptr = lambda t: None if t is None else vp(t.data_ptr())
    stream = vp(torch.cuda.current_stream().cuda_stream)
    return lib.fa_bwd_noalloc(ptr(q), ptr(k), ptr(v), ptr(o), ptr(do), ptr(lse), ptr(dq),
                              ptr(dk), ptr(dv), B, H, N, d, scale, int(causal), p, seed, offset,
                              ptr(bm), ptr(sl), stream)


@pytest.mark.parametrize("case", [
    dict(B=2, H=3, N=700, d=64, causal=True, p=0.0, padding=None),
    dict(B=4, H=2, N=384, d=128, causal=False, p=0.1, padding=(100, 384)),
])
def test_noalloc_matches_workspace_backward_on_consecutive_calls(case):
    lib = fa.load()
    B, H, N, d = case["B"], case["H"], case["N"], case["d"]
    scale = 1.0 / math.sqrt(d)
    for call, seed in enumerate((21, 22)):  # two calls in a row on the shared scratch
        x = make_case(B, H, N, d, seed=seed, padding=case["padding"])
        q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
        sl = None if x["seqlens"] is None else x["seqlens"].cuda()
        kw = dict(causal=case["causal"], dropout_p=case["p"], seed=seed, offset=call,
                  seqlens_k=sl)
        o, lse = fa.fwd(q, k, v, scale, **kw)
        ref = fa.bwd(q, k, v, o, do, lse, scale, **kw)
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        st = _noalloc_raw(lib, q, k, v, o, do, lse, got[0], got[1], got[2], B, H, N, d, scale,
                          case["causal"], case["p"], seed, call, None, sl)
        assert st == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.fa_device_status() == fa.FA_OK
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            g = g.float().cpu().numpy()
            r = r.float().cpu().numpy()
            assert np.isfinite(g).all(), name
            assert rel_fro(g, r) <= GRAD_RTOL, name


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    lib = fa.load()
    vp = ctypes.c_void_p
    a = vp(1 << 20)  # never dereferenced: the size check comes first
    st = lib.fa_bwd_noalloc(a, a, a, a, a, a, a, a, a, 64, 64, 1025, 64, 0.125, 0, 0.0, 0, 0,
                            None, None, None)
    assert st == fa.FA_ERR_WORKSPACE
