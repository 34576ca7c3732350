"""Pins for the oracle's short-query (decode) attention over a K/V cache. Each
test checks it against something other than itself: the separately written
full-attention oracle where the two cases coincide, a closed form whose count
of visible keys depends on the position offset of the query rows, the merge
identity of the online softmax, and torch's fp64 scaled_dot_product_attention
with an explicit mask built here."""
import numpy as np
import pytest
import torch

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def visible_keys(L, Nq, i, causal):
    """Number of cache keys query row i sees: rows are the last Nq positions."""
    if not causal:
        return L
    return max(0, min(L, L - Nq + i + 1))


@pytest.mark.parametrize("causal", [False, True])
def test_whole_sequence_as_query_block_is_full_attention(causal):
    """Nq = Nk = L: the query block is the whole sequence, so decode attention is
    ordinary (causal) attention, computed by the C oracle."""
    B, H, N, d = 2, 3, 150, 8
    r = rng(10)
    q, k, v = r.standard_normal((3, B, H, N, d))
    o, lse = oracle.fwd_decode(q, k, v, 0.31, causal=causal)
    o2, lse2 = oracle.fwd(q, k, v, 0.31, causal=causal)
    assert np.max(np.abs(o - o2)) < 1e-12
    assert np.max(np.abs(lse - lse2)) < 1e-12


def test_padding_without_causal_is_key_padding():
    """Without causal, a cache length L_b masks keys j >= L_b for every row, the
    key-padding mask of the full-attention oracle."""
    B, H, N, d = 2, 2, 140, 4
    r = rng(11)
    q, k, v = r.standard_normal((3, B, H, N, d))
    o, lse = oracle.fwd_decode(q, k, v, 0.5, seqlens_k=[97, 140])
    o2, lse2 = oracle.fwd(q, k, v, 0.5, seqlens_k=[97, 140])
    assert np.max(np.abs(o - o2)) < 1e-12
    assert np.max(np.abs(lse - lse2)) < 1e-12


@pytest.mark.parametrize("Nq,L,causal", [(1, 37, False), (1, 37, True), (5, 37, True),
                                         (5, 3, True), (8, 200, False), (16, 16, True)])
def test_identical_keys_give_mean_of_visible_values(Nq, L, causal):
    """With every key equal, each row's softmax is uniform over the keys it sees:
    O = mean of those V rows and lse = s + ln(count). The count carries the
    position offset of the query block (row i sits at L - Nq + i)."""
    Nk, d = 210, 6
    r = rng(12)
    q = r.standard_normal((1, 2, Nq, d))
    k = np.broadcast_to(r.standard_normal(d), (1, 1, Nk, d)).copy()
    v = r.standard_normal((1, 1, Nk, d))
    o, lse = oracle.fwd_decode(q, k, v, 0.7, causal=causal, seqlens_k=[L])
    for h in range(2):
        for i in range(Nq):
            n = visible_keys(L, Nq, i, causal)
            if n == 0:
                assert np.all(o[0, h, i] == 0) and np.isneginf(lse[0, h, i])
                continue
            assert np.max(np.abs(o[0, h, i] - v[0, 0, :n].mean(axis=0))) < 1e-12
            s = 0.7 * q[0, h, i] @ k[0, 0, 0]
            assert abs(lse[0, h, i] - (s + np.log(n))) < 1e-12


def test_one_visible_key_returns_its_value():
    r = rng(13)
    q, k, v = r.standard_normal((3, 1, 1, 1, 5))
    o, lse = oracle.fwd_decode(q, k, v, 0.9)
    assert np.max(np.abs(o[0, 0, 0] - v[0, 0, 0])) < 1e-15
    assert abs(lse[0, 0, 0] - 0.9 * q[0, 0, 0] @ k[0, 0, 0]) < 1e-12


def test_rows_before_the_cache_start_see_nothing():
    """Causal rows at positions < 0 (L < Nq) and an empty cache get O = 0, lse = -inf."""
    r = rng(14)
    q = r.standard_normal((2, 1, 4, 3))
    k, v = r.standard_normal((2, 2, 1, 9, 3))
    o, lse = oracle.fwd_decode(q, k, v, 1.0, causal=True, seqlens_k=[2, 0])
    assert np.all(np.isneginf(lse[0, 0, :2])) and np.all(o[0, 0, :2] == 0)
    assert np.all(np.isfinite(lse[0, 0, 2:]))
    assert np.all(np.isneginf(lse[1])) and np.all(o[1] == 0)


def test_split_cache_merges_to_the_whole():
    """Two halves of the cache, each attended alone and merged with the online
    softmax's update rule, give the whole-cache result (split-KV decode)."""
    B, H, Hkv, Nq, Nk, d, a = 1, 4, 2, 3, 300, 8, 113
    r = rng(15)
    q = r.standard_normal((B, H, Nq, d)) * 1.3
    k, v = r.standard_normal((2, B, Hkv, Nk, d))
    o, lse = oracle.fwd_decode(q, k, v, 0.4)
    o1, l1 = oracle.fwd_decode(q, k[:, :, :a], v[:, :, :a], 0.4)
    o2, l2 = oracle.fwd_decode(q, k[:, :, a:], v[:, :, a:], 0.4)
    m = np.maximum(l1, l2)
    w1, w2 = np.exp(l1 - m), np.exp(l2 - m)
    om = (w1[..., None] * o1 + w2[..., None] * o2) / (w1 + w2)[..., None]
    assert np.max(np.abs(om - o)) < 1e-12
    assert np.max(np.abs(m + np.log(w1 + w2) - lse)) < 1e-12


@pytest.mark.parametrize("H,Hkv,Nq,causal", [(4, 4, 1, False), (8, 2, 1, True),
                                             (8, 2, 6, True), (6, 1, 9, False),
                                             (4, 2, 33, True)])
def test_matches_torch_sdpa_fp64(H, Hkv, Nq, causal):
    """torch's fp64 CPU scaled_dot_product_attention on K/V repeated over each
    group, with the cache-length and causal offsets written as a boolean mask."""
    B, Nk, d = 2, 190, 16
    L = [190, 57]
    r = rng(16)
    q = r.standard_normal((B, H, Nq, d))
    k, v = r.standard_normal((2, B, Hkv, Nk, d))
    o, lse = oracle.fwd_decode(q, k, v, 0.23, causal=causal, seqlens_k=L)
    mask = np.zeros((B, 1, Nq, Nk), dtype=bool)
    for b in range(B):
        for i in range(Nq):
            mask[b, 0, i, :visible_keys(L[b], Nq, i, causal)] = True
    G = H // Hkv
    kr = torch.tensor(k).repeat_interleave(G, dim=1)
    vr = torch.tensor(v).repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), kr, vr, attn_mask=torch.tensor(mask), scale=0.23).numpy()
    s = 0.23 * torch.einsum("bhid,bhjd->bhij", torch.tensor(q), kr)
    ref_lse = torch.logsumexp(s.masked_fill(~torch.tensor(mask), -np.inf), dim=-1).numpy()
    rows = mask.any(-1)[:, 0]  # rows with at least one key
    for b in range(B):
        assert np.max(np.abs(o[b][:, rows[b]] - ref[b][:, rows[b]])) < 1e-12
        assert np.max(np.abs(lse[b][:, rows[b]] - ref_lse[b][:, rows[b]])) < 1e-12
        assert np.all(np.isneginf(lse[b][:, ~rows[b]]))


@pytest.mark.parametrize("causal", [True, False])
def test_decode_window_is_the_full_window_oracle_on_the_whole_block(causal):
    """Nq = Nk: the window decode equals the C oracle's sliding window (a
    separately written mask) on full attention."""
    B, H, N, d, W = 1, 2, 300, 8, 37
    r = rng(17)
    q, k, v = r.standard_normal((3, B, H, N, d))
    o, lse = oracle.fwd_decode(q, k, v, 0.3, causal=causal, window_left=W)
    o2, lse2 = oracle.fwd(q, k, v, 0.3, causal=causal, window_left=W)
    assert np.max(np.abs(o - o2)) < 1e-12
    assert np.max(np.abs(lse - lse2)) < 1e-12


@pytest.mark.parametrize("Nq,L,W", [(1, 200, 0), (1, 200, 63), (4, 200, 10), (3, 5, 2)])
def test_decode_window_identical_keys_closed_form(Nq, L, W):
    """Identical keys: mean of V over j in [max(0, L - Nq + i - W), L - Nq + i]."""
    Nk, d = 210, 5
    r = rng(18)
    q = r.standard_normal((1, 1, Nq, d))
    k = np.broadcast_to(r.standard_normal(d), (1, 1, Nk, d)).copy()
    v = r.standard_normal((1, 1, Nk, d))
    o, lse = oracle.fwd_decode(q, k, v, 0.5, causal=True, seqlens_k=[L], window_left=W)
    for i in range(Nq):
        hi = L - Nq + i
        lo = max(0, hi - W)
        assert np.max(np.abs(o[0, 0, i] - v[0, 0, lo:hi + 1].mean(axis=0))) < 1e-12
        assert abs(lse[0, 0, i] - (0.5 * q[0, 0, i] @ k[0, 0, 0] + np.log(hi - lo + 1))) < 1e-12
