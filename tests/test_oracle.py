"""Pins for the CPU oracle: each test checks it against something other than
itself (closed forms, invariants from the pages, finite differences, or an
independent library routine), chosen so that a dropped term, a wrong sign or
index, or a transposed operand fails at least one of them."""
import math

import numpy as np
import pytest
import torch

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def heads_of(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


def allowed_matrix(N, causal, seqlen=None, block_mask=None):
    """Boolean [N, N] allowed set, built independently of the oracle."""
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    a = np.ones((N, N), dtype=bool)
    if causal:
        a &= j <= i
    if seqlen is not None:
        a &= j < seqlen
    if block_mask is not None:
        a &= block_mask[i // 128, j // 128].astype(bool)
    return a


# --------------------------------------------------------------------- forward

@pytest.mark.parametrize("opts", [
    dict(), dict(causal=True), dict(seqlens_k=[70]), dict(block_mask="diag"),
    dict(causal=True, seqlens_k=[200]),
])
def test_softmax_rows_sum_to_one(opts):
    """Softmax rows sum to 1: with V = 1, every row with an allowed key has O = 1."""
    N, d = 300, 8
    r = rng(1)
    q, k = r.standard_normal((2, 1, N, d))
    v = np.ones((1, N, d))
    opts = dict(opts)
    if opts.get("block_mask") == "diag":
        nb = math.ceil(N / 128)
        opts["block_mask"] = np.eye(nb, dtype=np.uint8)
    o, lse = oracle.fwd(q, k, v, 0.3, heads=[(0, 0)], H=1, **opts)
    seqlen = opts.get("seqlens_k", [None])[0]
    a = allowed_matrix(N, opts.get("causal", False), seqlen, opts.get("block_mask"))
    has = a.any(axis=1)
    assert np.all(has)  # every case above leaves at least one key per row
    assert np.max(np.abs(o[0] - 1.0)) < 1e-12


def test_identical_keys_give_mean_of_values():
    """All keys equal: softmax is uniform over the allowed keys, O_i = mean of those v_j."""
    N, d = 260, 16
    r = rng(2)
    q = r.standard_normal((1, N, d))
    k = np.tile(r.standard_normal((1, 1, d)), (1, N, 1))
    v = r.standard_normal((1, N, d))
    for causal, seqlen in [(False, None), (True, None), (False, 131), (True, 200)]:
        o, lse = oracle.fwd(q, k, v, 0.125, causal=causal,
                            seqlens_k=None if seqlen is None else [seqlen], heads=[(0, 0)], H=1)
        a = allowed_matrix(N, causal, seqlen)
        expect = (a.astype(np.float64) @ v[0]) / a.sum(axis=1, keepdims=True)
        assert np.max(np.abs(o[0] - expect)) < 1e-12
        s = 0.125 * float(q[0, 0] @ k[0, 0])
        # lse of n equal scores s is s + ln n
        assert abs(lse[0, 0] - (s + math.log(a[0].sum()))) < 1e-12


def test_dominant_score_selects_one_value_row():
    """One score above all others by 60 gives O_i = v_j* (error <= N e^-60 max|v|)."""
    N = 64
    r = rng(3)
    target = (np.arange(N) * 7 + 3) % N
    # k_j = e_j and q_i = 60 e_target(i): s_ij = 60 at j = target(i), 0 elsewhere
    k = np.eye(N)[None]
    q = np.zeros((1, N, N))
    q[0, np.arange(N), target] = 60.0
    v = r.standard_normal((1, N, N))
    o, lse = oracle.fwd(q, k, v, 1.0, heads=[(0, 0)], H=1)
    assert np.max(np.abs(o[0] - v[0][target])) < math.exp(-40) * np.abs(v).max()
    assert np.max(np.abs(lse[0] - 60.0)) < 1e-12


def test_two_block_merge_identity():
    """Split the keys into two blocks; merging the per-block (m, l, O) with the
    update rule of the online softmax reproduces the full result."""
    N, d, n1 = 200, 12, 77
    r = rng(4)
    q, k, v = r.standard_normal((3, 1, N, d)) * 1.5
    scale = 0.4
    o, lse = oracle.fwd(q, k, v, scale, heads=[(0, 0)], H=1)
    # per-block normalised results; the first block is the key prefix [0, n1):
    o1, lse1 = oracle.fwd(q, k, v, scale, seqlens_k=[n1], heads=[(0, 0)], H=1)
    # second block: move keys [n1, N) to the front and mask the rest
    perm = np.concatenate([np.arange(n1, N), np.arange(0, n1)])
    o2, lse2 = oracle.fwd(q, k[:, perm], v[:, perm], scale, seqlens_k=[N - n1],
                          heads=[(0, 0)], H=1)
    # lse = m + ln l, so (m, l) of a block is recovered up to the free choice of m.
    m1, m2 = lse1[0], lse2[0]
    l1 = np.ones_like(m1)
    l2 = np.ones_like(m2)
    m_new = np.maximum(m1, m2)
    l_new = l1 * np.exp(m1 - m_new) + l2 * np.exp(m2 - m_new)
    o_new = (l1 * np.exp(m1 - m_new))[:, None] * o1[0] + (l2 * np.exp(m2 - m_new))[:, None] * o2[0]
    o_new /= l_new[:, None]
    assert np.max(np.abs(o_new - o[0])) < 1e-12
    assert np.max(np.abs(m_new + np.log(l_new) - lse[0])) < 1e-12


def test_prefix_invariant():
    """After seeing the first t keys, the running output equals the softmax
    over that prefix; extending the prefix one block at a time ends at the full O."""
    N, d = 256, 8
    r = rng(5)
    q, k, v = r.standard_normal((3, 1, N, d))
    o_full, lse_full = oracle.fwd(q, k, v, 0.35, heads=[(0, 0)], H=1)
    m = np.full(N, -np.inf)
    l = np.zeros(N)
    acc = np.zeros((N, d))
    for t in range(64, N + 1, 64):
        o_t, lse_t = oracle.fwd(q, k, v, 0.35, seqlens_k=[t], heads=[(0, 0)], H=1)
        # running statistics built from the previous prefix and the new block only
        s_blk = 0.35 * q[0] @ k[0, t - 64:t].T
        m_blk = s_blk.max(axis=1)
        m_new = np.maximum(m, m_blk)
        p_blk = np.exp(s_blk - m_new[:, None])
        l = l * np.exp(m - m_new) + p_blk.sum(axis=1)
        acc = acc * np.exp(m - m_new)[:, None] + p_blk @ v[0, t - 64:t]
        m = m_new
        assert np.max(np.abs(acc / l[:, None] - o_t[0])) < 1e-12
        assert np.max(np.abs(m + np.log(l) - lse_t[0])) < 1e-12
    assert np.max(np.abs(acc / l[:, None] - o_full[0])) < 1e-12


def test_fully_masked_row_is_zero():
    N, d = 8, 4
    r = rng(6)
    q, k, v = r.standard_normal((3, 1, N, d))
    o, lse = oracle.fwd(q, k, v, 1.0, seqlens_k=[0], heads=[(0, 0)], H=1)
    assert np.all(o == 0) and np.all(np.isneginf(lse))
    dq, dk, dv, D = oracle.bwd(q, k, v, r.standard_normal((1, N, d)), 1.0, seqlens_k=[0],
                               heads=[(0, 0)], H=1)
    assert np.all(dq == 0) and np.all(dk == 0) and np.all(dv == 0)


# ----------------------------------------------------- library special case

def _torch_sdpa(q, k, v, scale, mask):
    qt, kt, vt = (torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q, k, v))
    m = torch.tensor(mask)
    # the math backend: softmax(scale Q K^T + mask) V as plain tensor ops, the same
    # on every run (a blocked CPU kernel could otherwise be picked)
    from torch.nn.attention import SDPBackend, sdpa_kernel
    with sdpa_kernel(SDPBackend.MATH):
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    return qt, kt, vt, o


@pytest.mark.parametrize("case", ["dense", "causal", "padding", "block", "all"])
def test_matches_torch_sdpa_fp64(case):
    """No dropout: the oracle equals torch's fp64 CPU scaled_dot_product_attention
    with an explicit boolean mask, forward and autograd backward."""
    B, H, N, d = 2, 2, 260, 16
    r = rng(7)
    q, k, v, do = r.standard_normal((4, B, H, N, d))
    scale = 0.27
    causal = case in ("causal", "all")
    seqlens = [200, 131] if case in ("padding", "all") else None
    nb = math.ceil(N / 128)
    bm = None
    if case in ("block", "all"):
        bm = np.ones((nb, nb), dtype=np.uint8)
        bm[0, 1] = 0
        bm[2, 0] = 0
        bm[1, 2] = 0
    o, lse = oracle.fwd(q, k, v, scale, causal=causal, seqlens_k=seqlens, block_mask=bm)
    dq, dk, dv, D = oracle.bwd(q, k, v, do, scale, causal=causal, seqlens_k=seqlens,
                               block_mask=bm)
    mask = np.zeros((B, 1, N, N), dtype=bool)
    for b in range(B):
        mask[b, 0] = allowed_matrix(N, causal, None if seqlens is None else seqlens[b], bm)
    assert mask.any(axis=-1).all()
    qt, kt, vt, ot = _torch_sdpa(q, k, v, scale, mask)
    assert np.max(np.abs(ot.detach().numpy() - o)) < 1e-12
    (ot * torch.tensor(do)).sum().backward()
    for mine, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        assert np.max(np.abs(mine - ref.numpy())) < 1e-11
    # lse against a direct logsumexp of the masked scores
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    s = np.where(mask, s, -np.inf)
    ref_lse = torch.logsumexp(torch.tensor(s), dim=-1).numpy()
    assert np.max(np.abs(ref_lse - lse)) < 1e-12
    # D_i = dO_i . O_i
    assert np.max(np.abs(D - (do * o).sum(-1))) < 1e-11


def test_dropout_application_matches_masked_softmax():
    """With dropout, O = (softmax(S) * Z / (1 - p8/256)) V for the oracle's own Z."""
    B, H, N, d = 1, 2, 150, 8
    r = rng(8)
    q, k, v = r.standard_normal((3, B, H, N, d))
    p = 0.3
    o, lse = oracle.fwd(q, k, v, 0.5, dropout_p=p, seed=11, offset=5)
    keep = oracle.dropout_keep(heads_of(B, H), H, N, p, seed=11, offset=5).reshape(B, H, N, N)
    s = 0.5 * np.einsum("bhid,bhjd->bhij", q, k)
    P = torch.softmax(torch.tensor(s), dim=-1).numpy()
    phat = oracle.p8(p) / 256.0
    expect = np.einsum("bhij,bhjd->bhid", P * keep / (1 - phat), v)
    assert np.max(np.abs(expect - o)) < 1e-12


# ----------------------------------------------------- finite differences

def _loss(q, k, v, do, opts):
    o, _ = oracle.fwd(q, k, v, opts["scale"], causal=opts.get("causal", False),
                      dropout_p=opts.get("p", 0.0), seed=3, offset=7,
                      block_mask=opts.get("bm"), seqlens_k=opts.get("seqlens"))
    return float((o * do).sum())


FD_CASES = [
    dict(N=1, d=1), dict(N=2, d=4), dict(N=3, d=1, causal=True), dict(N=5, d=4, causal=True),
    dict(N=17, d=4, seqlens=[11]), dict(N=17, d=1, p=0.25), dict(N=5, d=4, p=0.5, causal=True),
    dict(N=130, d=1, causal=True), dict(N=130, d=1, seqlens=[129], p=0.1),
    dict(N=256, d=2, bm=np.array([[1, 0], [1, 1]], dtype=np.uint8)),
]


@pytest.mark.parametrize("case", FD_CASES, ids=lambda c: "-".join(
    f"{k}{v if not isinstance(v, np.ndarray) else 'mask'}" for k, v in c.items()))
def test_backward_matches_finite_differences(case):
    N, d = case["N"], case["d"]
    r = rng(100 + N * 10 + d)
    q, k, v, do = (x for x in r.standard_normal((4, 1, 1, N, d)))
    opts = dict(scale=0.7, causal=case.get("causal", False), p=case.get("p", 0.0),
                bm=case.get("bm"), seqlens=case.get("seqlens"))
    dq, dk, dv, D = oracle.bwd(q, k, v, do, opts["scale"], causal=opts["causal"],
                               dropout_p=opts["p"], seed=3, offset=7, block_mask=opts["bm"],
                               seqlens_k=opts["seqlens"])
    h = 1e-6
    grads = []
    for which in range(3):
        g = np.zeros((1, 1, N, d))
        for idx in np.ndindex(N, d):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][0, 0][idx] += h
            lp = _loss(*args, do, opts)
            args[which][0, 0][idx] -= 2 * h
            lm = _loss(*args, do, opts)
            g[0, 0][idx] = (lp - lm) / (2 * h)
        grads.append(g)
    for mine, fd in zip((dq, dk, dv), grads):
        denom = max(np.linalg.norm(fd), 1e-30)
        if np.linalg.norm(fd) == 0:
            assert np.linalg.norm(mine) < 1e-9
        else:
            assert np.linalg.norm(mine - fd) / denom < 1e-6
    o, _ = oracle.fwd(q, k, v, opts["scale"], causal=opts["causal"], dropout_p=opts["p"], seed=3,
                      offset=7, block_mask=opts["bm"], seqlens_k=opts["seqlens"])
    assert np.max(np.abs(D - (do * o).sum(-1))) < 1e-12


# ------------------------------------------------------------------ dropout

def test_p8_rounding():
    assert oracle.p8(0.0) == 0
    assert oracle.p8(0.1) == 26          # p-hat = 0.1015625
    assert oracle.p8(0.5) == 128
    assert oracle.p8(1.0 / 512) == 1     # round half up at the boundary
    assert oracle.p8(0.999) == 256


def test_philox_is_bijective_on_a_counter_sample():
    seen = set()
    for c in range(4096):
        out = tuple(int(x) for x in oracle.philox4x32_10([c, 7, 0, 0], [1, 2]))
        seen.add(out)
    assert len(seen) == 4096


def test_philox_key_and_counter_both_matter():
    base = oracle.philox4x32_10([1, 2, 3, 4], [5, 6])
    for pos in range(4):
        c = [1, 2, 3, 4]
        c[pos] ^= 1
        assert not np.array_equal(oracle.philox4x32_10(c, [5, 6]), base)
    for pos in range(2):
        key = [5, 6]
        key[pos] ^= 1
        assert not np.array_equal(oracle.philox4x32_10([1, 2, 3, 4], key), base)


def test_philox_bit_balance():
    """Every output bit is 1 with frequency 1/2 within 5 sigma over 2^15 blocks."""
    n = 1 << 15
    bits = np.zeros(128)
    for c in range(n):
        out = oracle.philox4x32_10([c, 0, 0, 0], [0x12345678, 0x9ABCDEF0])
        b = np.unpackbits(out.view(np.uint8))
        bits += b
    sigma = math.sqrt(n * 0.25)
    assert np.max(np.abs(bits - n / 2)) < 5 * sigma


@pytest.mark.parametrize("p", [0.1, 0.5])
def test_dropout_keep_statistics(p):
    H, N = 2, 2048
    keep = oracle.dropout_keep([(0, 0), (3, 1)], H, N, p, seed=0, offset=0).astype(np.float64)
    phat = oracle.p8(p) / 256.0
    n = keep.size
    frac = keep.mean()
    sigma = math.sqrt(phat * (1 - phat) / n)
    assert abs(frac - (1 - phat)) < 5 * sigma
    # no row / column structure: per-row keep counts are binomial
    rows = keep.reshape(-1, N).mean(axis=1)
    row_sigma = math.sqrt(phat * (1 - phat) / N)
    assert np.max(np.abs(rows - (1 - phat))) < 6 * row_sigma
    cols = keep.mean(axis=1).reshape(-1)
    assert np.max(np.abs(cols - (1 - phat))) < 6 * row_sigma
    # neighbouring columns (same Philox block and across blocks) are uncorrelated
    x = keep[..., :-1].reshape(-1) - keep.mean()
    y = keep[..., 1:].reshape(-1) - keep.mean()
    corr = (x * y).mean() / keep.var()
    assert abs(corr) < 5 / math.sqrt(x.size)


def test_dropout_streams_differ_by_seed_offset_and_head():
    N = 256
    a = oracle.dropout_keep([(0, 0)], 1, N, 0.5, seed=1, offset=0)
    b = oracle.dropout_keep([(0, 0)], 1, N, 0.5, seed=2, offset=0)
    c = oracle.dropout_keep([(0, 0)], 1, N, 0.5, seed=1, offset=1)
    d = oracle.dropout_keep([(1, 0)], 1, N, 0.5, seed=1, offset=0)
    for other in (b, c, d):
        assert (a != other).mean() > 0.4


def test_zero_dropout_keeps_everything():
    keep = oracle.dropout_keep([(0, 0)], 1, 300, 0.0)
    assert keep.all()


# ---------------------------------------------------------------- butterfly

@pytest.mark.parametrize("nb", [1, 2, 4, 8, 16, 128])
def test_butterfly_closed_form(nb):
    m = oracle.butterfly(nb).astype(int)
    k = int(round(math.log2(nb)))
    assert np.array_equal(m, m.T)
    assert np.all(np.diag(m) == 1)
    assert np.all(m.sum(axis=0) == 1 + k) and np.all(m.sum(axis=1) == 1 + k)
    assert m.sum() == nb * (1 + k)
    if nb == 128:
        assert m.sum() == 1024  # 6.25 % of the 16384 blocks at N = 16384


def test_butterfly_non_power_of_two():
    m = oracle.butterfly(6).astype(int)
    # strides 1, 2, 4; pairs whose partner falls outside [0, 6) are dropped
    assert np.array_equal(m, m.T) and np.all(np.diag(m) == 1)
    for r in range(6):
        for c in range(6):
            x = r ^ c
            assert m[r, c] == int(x in (0, 1, 2, 4))


# -------------------------------------------------------- worked example

def test_pages_worked_example_score_matrix_size():
    """Attention Kernel page, question 1: 32 heads x (32K)^2 x 2 bytes ~ 64 GB,
    the size of S that standard attention (the oracle's definition) materialises."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "pages_worked_examples.json")
    with open(path) as f:
        g = json.load(f)["score_matrix_bytes"]
    n_bytes = g["heads"] * g["seq_len"] ** 2 * g["bytes_per_element"]
    assert n_bytes == g["bytes"]
    assert abs(n_bytes / 2 ** 30 - g["approx_GiB"]) < 1e-9


# ------------------------------------------------------- grouped-query heads

def _loss_gqa(q, k, v, do, opts):
    o, _ = oracle.fwd_gqa(q, k, v, opts["scale"], causal=opts["causal"], dropout_p=opts["p"],
                          seed=3, offset=7)
    return float((o * do).sum())


@pytest.mark.parametrize("H,Hkv,causal,p", [(2, 1, False, 0.0), (4, 2, True, 0.0),
                                            (3, 1, True, 0.25)])
def test_gqa_backward_matches_finite_differences(H, Hkv, causal, p):
    # dK / dV of a shared K/V head must be the sum over its query heads: a
    # dropped sum or a wrong head map fails the finite-difference check.
    N, d = 5, 2
    r = rng(7 + H * 3 + Hkv)
    q = r.standard_normal((1, H, N, d))
    k = r.standard_normal((1, Hkv, N, d))
    v = r.standard_normal((1, Hkv, N, d))
    do = r.standard_normal((1, H, N, d))
    opts = dict(scale=0.6, causal=causal, p=p)
    dq, dk, dv, _ = oracle.bwd_gqa(q, k, v, do, opts["scale"], causal=causal, dropout_p=p,
                                   seed=3, offset=7)
    h = 1e-6
    for which, mine in ((0, dq), (1, dk), (2, dv)):
        base = (q, k, v)[which]
        fd = np.zeros_like(base)
        for idx in np.ndindex(*base.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = _loss_gqa(*args, do, opts)
            args[which][idx] -= 2 * h
            lm = _loss_gqa(*args, do, opts)
            fd[idx] = (lp - lm) / (2 * h)
        assert np.linalg.norm(mine - fd) / max(np.linalg.norm(fd), 1e-30) < 1e-6


def test_gqa_with_one_group_is_per_head_attention():
    # H_kv = H: the grouped form reduces to independent heads.
    r = rng(11)
    q, k, v, do = (r.standard_normal((2, 3, 9, 4)) for _ in range(4))
    o1, l1 = oracle.fwd_gqa(q, k, v, 0.5, causal=True)
    o2, l2 = oracle.fwd(q, k, v, 0.5, causal=True)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_mqa_heads_share_keys():
    # H_kv = 1: two query heads with equal queries see the same K/V, so their
    # outputs are equal; with different queries they generally differ.
    r = rng(12)
    q1 = r.standard_normal((1, 1, 7, 4))
    q = np.concatenate([q1, q1, r.standard_normal((1, 1, 7, 4))], axis=1)
    k, v = r.standard_normal((2, 1, 1, 7, 4))
    o, _ = oracle.fwd_gqa(q, k, v, 0.5)
    assert np.max(np.abs(o[0, 0] - o[0, 1])) < 1e-15
    assert np.max(np.abs(o[0, 0] - o[0, 2])) > 1e-3
