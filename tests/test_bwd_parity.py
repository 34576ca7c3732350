"""Backward pass on the GPU against the fp64 oracle (relative Frobenius error)."""
import math

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa
from _parity import check_grads_per_head, make_case, oracle_heads, butterfly_dev

pytestmark = pytest.mark.gpu


def run_bwd(B, H, N, d, causal=False, p=0.0, padding=None, mask=None, seed=0, offset=0,
            heads=None):
    x = make_case(B, H, N, d, seed=seed, padding=padding, with_grad=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    sl = None if x["seqlens"] is None else x["seqlens"].cuda()
    bm = None
    if isinstance(mask, str) and mask == "butterfly":
        bm = butterfly_dev(N)
    elif mask is not None:
        bm = torch.as_tensor(mask, dtype=torch.uint8).cuda()
    scale = 1.0 / math.sqrt(d)
    kw = dict(causal=causal, dropout_p=p, seed=seed, offset=offset, block_mask=bm, seqlens_k=sl)
    o, lse = fa.fwd(q, k, v, scale, **kw)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, scale, **kw)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    ref = oracle.bwd(oracle_heads(x["q"], heads), oracle_heads(x["k"], heads),
                     oracle_heads(x["v"], heads), oracle_heads(x["do"], heads), scale,
                     causal=causal, dropout_p=p, seed=seed, offset=offset,
                     block_mask=None if bm is None else bm.cpu().numpy(),
                     seqlens_k=None if sl is None else x["seqlens"].numpy(), heads=heads, H=H)
    got = [np.stack([t[b, h].float().cpu().numpy() for b, h in heads]) for t in (dq, dk, dv)]
    return got, ref[:3]


def check(got, ref):
    check_grads_per_head(zip(("dQ", "dK", "dV"), got, ref))


def test_tiny_config():
    check(*run_bwd(1, 1, 128, 64))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 127, 130, 256, 300, 640])
def test_dense_shapes(N, d):
    check(*run_bwd(2, 2, N, d, seed=N + d))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [128, 200, 513, 1024])
def test_causal(N, d):
    check(*run_bwd(1, 3, N, d, causal=True, seed=7 + N))


@pytest.mark.parametrize("d", [64, 128])
def test_key_padding(d):
    check(*run_bwd(4, 2, 700, d, padding=(1, 700), seed=3))


@pytest.mark.parametrize("d", [64, 128])
def test_butterfly_block_mask(d):
    check(*run_bwd(1, 2, 1024, d, mask="butterfly", seed=5))


def test_key_padding_many_units_every_head():
    # 16 x 16 heads x 8 key tiles = 2048 key-tile units over the persistent grid:
    # under key padding the key-tile kernels walk a rotated schedule through many
    # rounds. Every head is checked through an identity that holds at any size
    # (without dropout each query row's P sums to 1 over its visible keys, so
    # sum_j dV_j = sum_i dO_i), a few heads against the oracle.
    B, H, N, d = 16, 16, 1024, 64
    x = make_case(B, H, N, d, seed=21, padding=(1, N))
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    sl = x["seqlens"].cuda()
    o, lse = fa.fwd(q, k, v, seqlens_k=sl)
    dq, dk, dv = fa.bwd(q, k, v, o, do, lse, seqlens_k=sl)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    dv_tot = dv.double().sum(dim=2)
    do_tot = do.double().sum(dim=2)
    err = (dv_tot - do_tot).norm(dim=-1) / do_tot.norm(dim=-1).clamp_min(1e-6)
    assert float(err.max()) < 1e-2, f"worst head {float(err.max())}"
    # keys past a row's length get no gradient
    for b in range(B):
        L = int(x["seqlens"][b])
        assert torch.count_nonzero(dk[b, :, L:]) == 0 and torch.count_nonzero(dv[b, :, L:]) == 0
    heads = [(0, 0), (7, 9), (15, 15)]
    ref = oracle.bwd(oracle_heads(x["q"], heads), oracle_heads(x["k"], heads),
                     oracle_heads(x["v"], heads), oracle_heads(x["do"], heads), 1.0 / math.sqrt(d),
                     seqlens_k=x["seqlens"].numpy(), heads=heads, H=H)
    got = [np.stack([t[b, h].float().cpu().numpy() for b, h in heads]) for t in (dq, dk, dv)]
    check(got, ref[:3])


@pytest.mark.parametrize("d", [64, 128])
def test_long_runs_of_empty_units(d):
    """Backward with key length 0 for all batch rows but the last, several work
    units per CTA and most of them without any key: the empty rows' gradients are
    zero, and the last row equals the same kernels run on it alone (bit for bit:
    without dropout a row's result does not depend on which CTA computes it) and
    the oracle."""
    B, H, N = 16, 16, 1024
    x = make_case(B, H, N, d, seed=23, with_grad=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    sl = torch.zeros(B, dtype=torch.int32)
    sl[-1] = N - 7
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, scale, seqlens_k=sl.cuda())
    grads = fa.bwd(q, k, v, o, do, lse, scale, seqlens_k=sl.cuda())
    one = lambda t: t[-1:].contiguous()
    o1, l1 = fa.fwd(one(q), one(k), one(v), scale, seqlens_k=sl[-1:].cuda())
    grads1 = fa.bwd(one(q), one(k), one(v), o1, one(do), l1, scale, seqlens_k=sl[-1:].cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    for name, g, g1 in zip(("dQ", "dK", "dV"), grads, grads1):
        assert torch.all(g[:-1] == 0), f"{name}: nonzero gradient in a row without keys"
        assert torch.equal(g[-1:], g1), f"{name}: last row differs from the single-row run"
    heads = [(B - 1, 0), (B - 1, H - 1)]
    ref = oracle.bwd(oracle_heads(x["q"], heads), oracle_heads(x["k"], heads),
                     oracle_heads(x["v"], heads), oracle_heads(x["do"], heads), scale,
                     seqlens_k=sl.numpy(), heads=heads, H=H)
    got = [np.stack([t[b, h].float().cpu().numpy() for b, h in heads]) for t in grads]
    check(got, ref[:3])


def test_random_block_mask_with_empty_rows_and_columns():
    nb = 5
    g = np.random.default_rng(1)
    m = (g.random((nb, nb)) < 0.5).astype(np.uint8)
    m[2, :] = 0  # a query block with no key
    m[:, 4] = 0  # a key block no query sees: dK = dV = 0 there
    check(*run_bwd(2, 2, 640, 64, mask=m, seed=9))


@pytest.mark.parametrize("d", [64, 128])
def test_dropout(d):
    check(*run_bwd(2, 2, 384, d, p=0.1, seed=11, offset=3))


def test_all_options_together():
    N = 700
    nb = math.ceil(N / 128)
    m = np.ones((nb, nb), dtype=np.uint8)
    m[3, 1] = 0
    m[5, 0] = 0
    check(*run_bwd(3, 2, N, 64, causal=True, p=0.2, padding=(300, 700), mask=m, seed=13))


def test_determinism():
    x = make_case(2, 2, 1000, 64)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v, causal=True)
    r1 = fa.bwd(q, k, v, o, do, lse, causal=True)
    r2 = fa.bwd(q, k, v, o, do, lse, causal=True)
    torch.cuda.synchronize()
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


def test_workspace_validation():
    x = make_case(1, 1, 128, 64)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = fa.fwd(q, k, v)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    st = fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, 1, 1, 128, 64, 0.125, workspace=small,
                   workspace_bytes=16)
    assert st == fa.FA_ERR_WORKSPACE
