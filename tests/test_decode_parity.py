"""Short-query attention over a K/V cache (fa_decode) on the GPU against the
fp64 oracle: O within the O tolerance, lse within 1e-3, rows without keys
exactly O = 0 and lse = -inf, for every way the work is split among CTAs."""
import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa
from io_aware_exact_07_gb300 import inputs
from _parity import LSE_TOL, o_within_tol

pytestmark = pytest.mark.gpu


def run(B, H, Hkv, Nq, Nk, d, causal=False, lengths=None, num_ctas=0, seed=0, window_left=-1):
    w = inputs.DecodeWorkload("t", B, H, Hkv, Nq, Nk, d, causal=causal, lengths=lengths,
                              seed=seed)
    x = inputs.draw_decode(w)
    sl = None if x["seqlens"] is None else x["seqlens"].cuda()
    o, lse = fa.decode(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), w.scale, causal=causal,
                       seqlens_k=sl, num_ctas=num_ctas, window_left=window_left)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    f64 = lambda t: t.double().numpy()
    o_ref, lse_ref = oracle.fwd_decode(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.scale,
                                       causal=causal,
                                       seqlens_k=None if x["seqlens"] is None
                                       else x["seqlens"].numpy(), window_left=window_left)
    check(o, lse, o_ref, lse_ref)
    return o, lse


def check(o, lse, o_ref, lse_ref):
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), "rows without keys differ"
    assert np.all(o[empty] == 0)
    ok, worst = o_within_tol(o, o_ref)
    assert ok, f"O error exceeds its tolerance by {worst}"
    if (~empty).any():
        assert np.max(np.abs(lse[~empty] - lse_ref[~empty])) <= LSE_TOL


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,causal,lengths", [
    (1, 4, 2, 1, 300, 64, False, None),          # ragged last tile
    (2, 8, 2, 3, 1000, 128, True, None),         # several query rows, causal offsets
    (3, 4, 1, 16, 129, 64, True, (0, 129)),      # MQA, ragged and empty caches
    (2, 32, 8, 1, 4100, 128, False, (1, 4100)),  # grouped heads, ragged lengths
    (1, 2, 2, 64, 5000, 128, True, None),        # 64 rows per head, causal
    (1, 128, 1, 1, 777, 64, False, None),        # 128 query heads over one K/V head
    (4, 16, 16, 1, 128, 64, False, None),        # one key tile per head
    (1, 8, 1, 16, 2048, 128, True, (10, 2048)),  # 8 x 16 = 128 rows: a full query tile
    (3, 2, 2, 1, 1, 64, False, None),             # a one-key cache
    (2, 2, 1, 5, 1, 128, True, None),             # one key, more query rows than keys
])
def test_decode_matches_oracle(B, H, Hkv, Nq, Nk, d, causal, lengths):
    run(B, H, Hkv, Nq, Nk, d, causal, lengths, seed=B + Nk)


@pytest.mark.parametrize("num_ctas", [1, 2, 5, 16, 1000])
def test_decode_any_split_matches_oracle(num_ctas):
    # 8 K/V heads x 17 key tiles = 136 (head, tile) pairs: 1 and 2 CTAs hold
    # whole heads (direct path); 5 and 16 CTAs cut heads into 2-3 pieces; 1000
    # gives one tile per CTA, 17 pieces per head.
    run(2, 8, 4, 2, 17 * 128 - 5, 64, causal=True, lengths=(300, 2171), num_ctas=num_ctas,
        seed=11)


def test_decode_one_cta_per_head_is_direct():
    # B * H_kv CTAs over whole heads: no piece is cut, no workspace, no combine.
    assert fa.fa_decode_workspace_size(2, 8, 4, 1, 1000, 128, 8) == 0
    run(2, 8, 4, 1, 1000, 128, num_ctas=8, seed=12)


def test_decode_empty_caches():
    q = torch.randn((2, 4, 3, 64), device="cuda").to(torch.bfloat16)
    k = torch.randn((2, 2, 500, 64), device="cuda").to(torch.bfloat16)
    sl = torch.zeros(2, dtype=torch.int32, device="cuda")
    for ctas in (0, 1, 3):
        o, lse = fa.decode(q, k, k, causal=True, seqlens_k=sl, num_ctas=ctas)
        torch.cuda.synchronize()
        assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_decode_bench_workload_matches_oracle():
    # The bench's decode step at full size, every row checked: in the launch
    # configuration the bench times (automatic split: 128 whole K/V heads on
    # 128 CTAs) and with one CTA per SM (heads cut, combine kernel).
    w = inputs.DECODE
    x = inputs.draw_decode(w)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    f64 = lambda t: t.double().numpy()
    o_ref, lse_ref = oracle.fwd_decode(f64(x["q"]), f64(x["k"]), f64(x["v"]), w.scale,
                                       causal=w.causal)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for ctas in (0, sms):
        o, lse = fa.decode(q, k, v, w.scale, causal=w.causal, num_ctas=ctas)
        torch.cuda.synchronize()
        assert fa.fa_device_status() == fa.FA_OK
        check(o, lse, o_ref, lse_ref)
    assert fa.fa_decode_workspace_size(w.B, w.H, w.Hkv, w.Nq, w.Nk, w.d, sms) > 0


def test_decode_rejects_bad_arguments():
    q = torch.zeros((1, 4, 64, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 2, 256, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 4, 64), dtype=torch.float32, device="cuda")
    s = 0.125
    # 2 query heads x 64 rows = 128: allowed; 4 x 64 over one K/V head = 256: not
    assert fa.fa_decode(q, k, k, o, lse, 1, 4, 1, 64, 256, 64, s) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_decode(q, k, k, o, lse, 1, 4, 3, 64, 256, 64, s) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_decode(q, k, k, o, lse, 1, 4, 2, 64, 256, 96, s) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_decode(q, k, k, o, lse, 1, 4, 2, 64, 0, 64, s) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_decode(q, k, k, o, lse, 1, 4, 2, 64, 256, 64, -1.0) == fa.FA_ERR_INVALID_ARG
    # a split that cuts heads needs the workspace
    assert fa.fa_decode_workspace_size(1, 4, 2, 64, 256, 64, 4) > 0
    assert fa.fa_decode(q, k, k, o, lse, 1, 4, 2, 64, 256, 64, s, num_ctas=4) == \
        fa.FA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK


@pytest.mark.parametrize("B,H,Hkv,Nq,Nk,d,causal,lengths,wl,ctas", [
    (2, 8, 2, 1, 5000, 128, True, None, 0, 0),           # a window of one key
    (2, 8, 2, 4, 5000, 64, True, (100, 5000), 300, 0),   # ragged caches, 301-key window
    (1, 4, 1, 16, 3000, 128, False, None, 1000, 7),      # non-causal, heads cut over 7 CTAs
    (2, 4, 4, 1, 4100, 128, True, None, 127, 1000),      # window on a tile edge, one tile per CTA
    (1, 2, 2, 64, 2000, 64, True, None, 4095, 0),        # window wider than the cache
])
def test_decode_sliding_window(B, H, Hkv, Nq, Nk, d, causal, lengths, wl, ctas):
    run(B, H, Hkv, Nq, Nk, d, causal, lengths, num_ctas=ctas, seed=wl + Nk, window_left=wl)

