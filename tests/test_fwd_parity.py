"""Forward pass on the GPU against the fp64 oracle, element by element."""
import math

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa
from _parity import (LSE_TOL, make_case, oracle_heads, lse_err, butterfly_dev, o_within_tol)

pytestmark = pytest.mark.gpu


def run_fwd(B, H, N, d, causal=False, p=0.0, padding=None, mask=None, seed=0, heads=None,
            offset=0):
    x = make_case(B, H, N, d, seed=seed, padding=padding, with_grad=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    sl = None if x["seqlens"] is None else x["seqlens"].cuda()
    bm = None
    if isinstance(mask, str) and mask == "butterfly":
        bm = butterfly_dev(N)
    elif mask is not None:
        bm = torch.as_tensor(mask, dtype=torch.uint8).cuda()
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, scale, causal=causal, dropout_p=p, seed=seed, offset=offset,
                    block_mask=bm, seqlens_k=sl)
    torch.cuda.synchronize()
    if heads is None:
        heads = [(b, h) for b in range(B) for h in range(H)]
    ro, rl = oracle.fwd(oracle_heads(x["q"], heads), oracle_heads(x["k"], heads),
                        oracle_heads(x["v"], heads), scale, causal=causal, dropout_p=p, seed=seed,
                        offset=offset, block_mask=None if bm is None else bm.cpu().numpy(),
                        seqlens_k=None if sl is None else x["seqlens"].numpy(), heads=heads, H=H)
    go = np.stack([o[b, h].float().cpu().numpy() for b, h in heads])
    gl = np.stack([lse[b, h].cpu().numpy() for b, h in heads])
    return go, gl, ro, rl


def check(go, gl, ro, rl):
    ok_o, worst = o_within_tol(go, ro)
    err_l = lse_err(gl, rl)
    assert np.isfinite(go).all()
    assert ok_o, f"O error exceeds its tolerance by {worst}"
    assert err_l <= LSE_TOL, f"lse max-abs error {err_l}"


def test_tiny_config():
    """B=1, H=1, N=128, d=64, non-causal, no dropout: checked in full."""
    check(*run_fwd(1, 1, 128, 64))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 127, 128, 130, 256, 300, 640])
def test_dense_shapes(N, d):
    check(*run_fwd(2, 2, N, d, seed=N + d))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [128, 200, 513, 1024])
def test_causal(N, d):
    check(*run_fwd(1, 3, N, d, causal=True, seed=7 + N))


@pytest.mark.parametrize("d", [64, 128])
def test_key_padding(d):
    check(*run_fwd(4, 2, 700, d, padding=(1, 700), seed=3))


def test_key_padding_zero_length():
    x = make_case(2, 1, 256, 64, with_grad=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    sl = torch.tensor([0, 100], dtype=torch.int32).cuda()
    o, lse = fa.fwd(q, k, v, 0.125, seqlens_k=sl)
    torch.cuda.synchronize()
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ro, rl = oracle.fwd(oracle_heads(x["q"], [(1, 0)]), oracle_heads(x["k"], [(1, 0)]),
                        oracle_heads(x["v"], [(1, 0)]), 0.125, seqlens_k=[0, 100],
                        heads=[(1, 0)], H=1)
    check(o[1:2, 0].float().cpu().numpy(), lse[1:2, 0].cpu().numpy(), ro, rl)


@pytest.mark.parametrize("d", [64, 128])
def test_long_runs_of_empty_units(d):
    """Key lengths 0 for all batch rows but the last, with several work units per
    CTA: each CTA meets runs of units without any key tile (epilogues that wait
    for no product) before the last batch row's real ones. Empty rows give O = 0
    and lse = -inf; the last row equals the same kernel run on it alone (bit for
    bit: a row's result does not depend on which CTA computes it) and the oracle."""
    B, H, N = 16, 16, 1024
    x = make_case(B, H, N, d, seed=21, with_grad=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    sl = torch.zeros(B, dtype=torch.int32)
    sl[-1] = N - 3
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fwd(q, k, v, scale, seqlens_k=sl.cuda())
    o1, lse1 = fa.fwd(q[-1:].contiguous(), k[-1:].contiguous(), v[-1:].contiguous(), scale,
                      seqlens_k=sl[-1:].cuda())
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    assert torch.all(o[:-1] == 0) and torch.all(torch.isneginf(lse[:-1]))
    assert torch.equal(o[-1:], o1) and torch.equal(lse[-1:], lse1)
    heads = [(B - 1, 0), (B - 1, H - 1)]
    ro, rl = oracle.fwd(oracle_heads(x["q"], heads), oracle_heads(x["k"], heads),
                        oracle_heads(x["v"], heads), scale, seqlens_k=sl.numpy(), heads=heads,
                        H=H)
    check(np.stack([o[b, h].float().cpu().numpy() for b, h in heads]),
          np.stack([lse[b, h].cpu().numpy() for b, h in heads]), ro, rl)


@pytest.mark.parametrize("d", [64, 128])
def test_butterfly_block_mask(d):
    check(*run_fwd(1, 2, 1024, d, mask="butterfly", seed=5))


def test_random_block_mask_with_empty_rows():
    N = 640
    nb = 5
    g = np.random.default_rng(0)
    m = (g.random((nb, nb)) < 0.5).astype(np.uint8)
    m[2, :] = 0  # query block 2 sees no key: O = 0, lse = -inf
    check(*run_fwd(2, 2, N, 64, mask=m, seed=9))


@pytest.mark.parametrize("d", [64, 128])
def test_dropout(d):
    check(*run_fwd(2, 2, 384, d, p=0.1, seed=11, offset=3))


def test_all_options_together():
    N = 700
    nb = math.ceil(N / 128)
    m = np.ones((nb, nb), dtype=np.uint8)
    m[3, 1] = 0
    m[5, 0] = 0
    check(*run_fwd(3, 2, N, 64, causal=True, p=0.2, padding=(300, 700), mask=m, seed=13))


def test_determinism():
    x = make_case(2, 4, 1000, 128, with_grad=False)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = fa.fwd(q, k, v, causal=True)
    o2, l2 = fa.fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
