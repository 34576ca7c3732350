"""Pins for the oracle's sliding-window mask (key j visible to query i only if
i - window_left <= j <= i + window_right): closed forms whose counts carry the
window edges, the separately written decode oracle on the window's keys,
torch's fp64 scaled_dot_product_attention with a band mask built here (forward
and autograd backward), and finite differences."""
import numpy as np
import pytest
import torch

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def band(N, wl, wr, causal=False, seqlen=None):
    """Boolean [N, N] allowed set written from the window definition."""
    a = np.zeros((N, N), dtype=bool)
    for i in range(N):
        lo = 0 if wl < 0 else max(0, i - wl)
        hi = N - 1 if wr < 0 else min(N - 1, i + wr)
        if causal:
            hi = min(hi, i)
        if seqlen is not None:
            hi = min(hi, seqlen - 1)
        if hi >= lo:
            a[i, lo:hi + 1] = True
    return a


def test_causal_window_of_zero_sees_only_itself():
    N, d = 70, 5
    r = rng(20)
    q, k, v = r.standard_normal((3, 1, N, d))
    o, lse = oracle.fwd(q, k, v, 0.6, causal=True, window_left=0, heads=[(0, 0)], H=1)
    assert np.max(np.abs(o[0] - v[0])) < 1e-15
    assert np.max(np.abs(lse[0] - 0.6 * np.einsum("id,id->i", q[0], k[0]))) < 1e-12


@pytest.mark.parametrize("wl,wr,causal", [(5, -1, True), (0, 3, False), (7, 2, False),
                                          (-1, 4, False), (130, 130, False), (200, -1, True)])
def test_identical_keys_give_mean_over_the_window(wl, wr, causal):
    """Every key equal: row i's softmax is uniform over its window, so O is the
    mean of those V rows and lse = s + ln(count)."""
    N, d = 260, 4
    r = rng(21)
    q = r.standard_normal((1, N, d))
    k = np.broadcast_to(r.standard_normal(d), (1, N, d)).copy()
    v = r.standard_normal((1, N, d))
    o, lse = oracle.fwd(q, k, v, 0.8, causal=causal, window_left=wl, window_right=wr,
                        heads=[(0, 0)], H=1)
    for i in range(N):
        lo = 0 if wl < 0 else max(0, i - wl)
        hi = N - 1 if wr < 0 else min(N - 1, i + wr)
        if causal:
            hi = min(hi, i)
        assert np.max(np.abs(o[0, i] - v[0, lo:hi + 1].mean(axis=0))) < 1e-12
        assert abs(lse[0, i] - (0.8 * q[0, i] @ k[0, 0] + np.log(hi - lo + 1))) < 1e-12


def test_window_covering_everything_is_no_window():
    N, d = 150, 6
    r = rng(22)
    q, k, v = r.standard_normal((3, 2, 1, N, d))[:3]
    o1, l1 = oracle.fwd(q, k, v, 0.3, causal=True)
    o2, l2 = oracle.fwd(q, k, v, 0.3, causal=True, window_left=N - 1, window_right=0)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_causal_window_row_is_decode_over_its_keys():
    """Row i of causal attention with window W is one query over the cache
    k[i - W .. i], computed by the separately written decode oracle."""
    N, d, W = 200, 8, 37
    r = rng(23)
    q, k, v = r.standard_normal((3, 1, 1, N, d))
    o, lse = oracle.fwd(q, k, v, 0.45, causal=True, window_left=W)
    for i in (0, 5, 36, 37, 38, 120, 199):
        lo = max(0, i - W)
        od, ld = oracle.fwd_decode(q[:, :, i:i + 1], k[:, :, lo:i + 1], v[:, :, lo:i + 1], 0.45)
        assert np.max(np.abs(od[0, 0, 0] - o[0, 0, i])) < 1e-12
        assert abs(ld[0, 0, 0] - lse[0, 0, i]) < 1e-12


@pytest.mark.parametrize("wl,wr,causal,seqlens", [(50, -1, True, None), (20, 30, False, None),
                                                  (140, 5, False, [200, 131]),
                                                  (0, 0, False, None), (129, -1, True, [260, 200])])
def test_matches_torch_sdpa_fp64(wl, wr, causal, seqlens):
    B, H, N, d = 2, 2, 260, 8
    r = rng(24)
    q, k, v, do = r.standard_normal((4, B, H, N, d))
    kw = dict(causal=causal, seqlens_k=seqlens, window_left=wl, window_right=wr)
    o, lse = oracle.fwd(q, k, v, 0.33, **kw)
    dq, dk, dv, _ = oracle.bwd(q, k, v, do, 0.33, **kw)
    mask = np.zeros((B, 1, N, N), dtype=bool)
    for b in range(B):
        mask[b, 0] = band(N, wl, wr, causal, None if seqlens is None else seqlens[b])
    assert mask.any(-1).all()
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ot = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.tensor(mask),
                                                          scale=0.33)
    assert np.max(np.abs(ot.detach().numpy() - o)) < 1e-12
    (ot * torch.tensor(do)).sum().backward()
    for mine, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        assert np.max(np.abs(mine - ref.numpy())) < 1e-11
    s = 0.33 * np.einsum("bhid,bhjd->bhij", q, k)
    ref_lse = torch.logsumexp(torch.tensor(np.where(mask, s, -np.inf)), dim=-1).numpy()
    assert np.max(np.abs(ref_lse - lse)) < 1e-12


@pytest.mark.parametrize("wl,wr,causal,p", [(2, -1, True, 0.0), (1, 2, False, 0.3),
                                            (3, 0, False, 0.0)])
def test_backward_matches_finite_differences(wl, wr, causal, p):
    N, d = 9, 3
    r = rng(25)
    q, k, v, do = r.standard_normal((4, 1, N, d))
    kw = dict(causal=causal, dropout_p=p, seed=3, offset=1, window_left=wl, window_right=wr,
              heads=[(0, 0)], H=1)
    dq, dk, dv, _ = oracle.bwd(q, k, v, do, 0.5, **kw)

    def loss(q_, k_, v_):
        o, _ = oracle.fwd(q_, k_, v_, 0.5, **kw)
        return float((o * do).sum())

    eps = 1e-6
    for grad, idx in ((dq, 0), (dk, 1), (dv, 2)):
        num = np.zeros_like(grad)
        for i in range(N):
            for c in range(d):
                args = [q.copy(), k.copy(), v.copy()]
                args[idx][0, i, c] += eps
                lp = loss(*args)
                args[idx][0, i, c] -= 2 * eps
                lm = loss(*args)
                num[0, i, c] = (lp - lm) / (2 * eps)
        assert np.max(np.abs(num - grad)) < 1e-6 * max(1.0, np.max(np.abs(grad)))
