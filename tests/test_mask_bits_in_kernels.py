"""The masks the production kernels apply, read back bit for bit.

The dropout keep mask and the block / causal / padding / window masks are fused
into the forward, dK/dV and dQ kernels (FlashAttention deep-read report,
section 3.2, Algorithm 1 with its fused masking and dropout). Tolerance-based
parity cannot prove those masks exact: one wrong keep bit moves O by a few
thousandths. These tests pick inputs under which every output element of a
kernel is one mask bit times a nonzero number, so `output != 0` is the mask:

  * Q = 0, so every allowed score is 0 and P_ij = 1 / (number of allowed keys
    of row i), which is nonzero and far from bf16 underflow;
  * forward: V = the one-hot rows of a chunk of keys (v_j = e_{j - c0} for
    c0 <= j < c0 + d, else 0), so O_ic = P_i,c0+c Z_i,c0+c / (1 - p);
  * dK/dV kernel: dO = one-hot rows of a chunk of query rows, so
    dV_jc = P_r0+c,j Z_r0+c,j / (1 - p) (with grouped K/V heads the columns
    are split between the query heads of a group, because dV sums over them);
  * dQ kernel: K, V = one-hot rows of a key chunk, dO = all ones and O passed
    as zeros (so D = rowsum(dO * O) = 0), so dS_ij = P_ij Z_ij / (1 - p) on the
    chunk and dQ_ic = scale dS_i,c0+c.

The expected bits come from the fp64 oracle run on the same inputs
(Q = K = 0, V = the N x N identity): its output is nonzero exactly where the
oracle's own mask and its own Philox stream keep the element. Exact zeros
on dropped or masked elements hold on the GPU because each such product is
0 * P and every other term of the sum is 0 * 0.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa

pytestmark = pytest.mark.gpu


def _expected(B, H, N, causal, p, seed, offset, block_mask, seqlens, window):
    """bool [B, H, N, N]: element (i, j) allowed by every mask and kept by dropout,
    from the oracle's forward with Q = K = 0 and V = I."""
    z = np.zeros((B, H, N, N))
    eye = np.broadcast_to(np.eye(N), (B, H, N, N))
    o, _ = oracle.fwd(z, z, eye, 1.0, causal=causal, dropout_p=p, seed=seed, offset=offset,
                      block_mask=block_mask, seqlens_k=seqlens, window_left=window[0],
                      window_right=window[1])
    return o != 0


def _one_hot_chunk(shape_lead, N, d, c0):
    """bf16 [*shape_lead, N, d] CUDA tensor: row j is e_{j - c0} for c0 <= j < c0 + d."""
    x = torch.zeros((*shape_lead, N, d), dtype=torch.bfloat16)
    n = min(d, N - c0)
    idx = torch.arange(n)
    x[..., c0 + idx, idx] = 1.0
    return x.cuda()


CASES = [
    # d = 64: split dK/dV kernel and d = 64 dQ; ragged last key group (200 = 12*16 + 8)
    dict(id="d64_dense_drop", B=2, H=3, Hkv=3, N=200, d=64, causal=False, p=0.1, seed=7,
         offset=5),
    # d = 128: single-issuer dK/dV kernel; N = 120 is not a multiple of 16
    dict(id="d128_causal_drop", B=2, H=3, Hkv=3, N=120, d=128, causal=True, p=0.1, seed=3,
         offset=2**33 + 1),
    # row index r = (b H + h) N + i beyond 2^16 (up to 67,599)
    dict(id="d64_rows_past_2_16", B=2, H=260, Hkv=260, N=130, d=64, causal=False, p=0.25,
         seed=2**40 + 1, offset=9),
    dict(id="d128_rows_past_2_16", B=1, H=520, Hkv=520, N=130, d=128, causal=True, p=0.1,
         seed=11, offset=0),
    # grouped K/V heads (dK/dV sums the group on chip)
    dict(id="d128_gqa_causal_drop", B=2, H=8, Hkv=2, N=200, d=128, causal=True, p=0.1, seed=5,
         offset=1),
    dict(id="d64_gqa_drop", B=1, H=4, Hkv=1, N=150, d=64, causal=False, p=0.5, seed=9, offset=4),
    # sliding-window instances
    dict(id="d64_window_drop", B=1, H=2, Hkv=2, N=300, d=64, causal=False, p=0.1, seed=13,
         offset=6, window=(50, 20)),
    dict(id="d128_window_causal_drop", B=1, H=2, Hkv=1, N=300, d=128, causal=True, p=0.2,
         seed=14, offset=0, window=(70, -1)),
    # random block mask (with empty block rows / columns), key padding, dropout
    dict(id="d64_blockmask_padding_drop", B=2, H=2, Hkv=2, N=400, d=64, causal=False, p=0.1,
         seed=15, offset=3, block_mask=17, seqlens=(400, 203)),
    dict(id="d128_blockmask_causal_drop", B=1, H=2, Hkv=2, N=390, d=128, causal=True, p=0.1,
         seed=16, offset=0, block_mask=18),
    # masks without dropout (the no-dropout kernel instances)
    dict(id="d64_blockmask_padding_nodrop", B=2, H=2, Hkv=2, N=400, d=64, causal=True, p=0.0,
         seed=0, offset=0, block_mask=19, seqlens=(333, 129)),
    dict(id="d128_blockmask_nodrop", B=1, H=3, Hkv=3, N=300, d=128, causal=False, p=0.0, seed=0,
         offset=0, block_mask=20),
    dict(id="d128_window_padding_nodrop", B=2, H=2, Hkv=2, N=260, d=128, causal=False, p=0.0,
         seed=0, offset=0, window=(0, 0), seqlens=(260, 100)),
]


def _block_mask(N, seed):
    nb = math.ceil(N / 128)
    g = np.random.default_rng(seed)
    m = (g.random((nb, nb)) < 0.6).astype(np.uint8)
    for r in range(1, nb):
        m[r, r] = 1   # every diagonal block but the first: causal cases keep some pairs
    m[nb - 1, :] = 0  # a query block that sees no key
    m[:, 0] = 0       # a key block that no query sees
    m[0, 1 % nb] = 1
    return m


@pytest.mark.parametrize("case", CASES, ids=[c["id"] for c in CASES])
def test_kernel_masks_bit_exact(case):
    B, H, Hkv, N, d = case["B"], case["H"], case["Hkv"], case["N"], case["d"]
    G = H // Hkv
    causal, p, seed, offset = case["causal"], case["p"], case["seed"], case["offset"]
    window = case.get("window", (-1, -1))
    bm_np = None if case.get("block_mask") is None else _block_mask(N, case["block_mask"])
    sl_np = None if case.get("seqlens") is None else np.array(case["seqlens"], dtype=np.int32)
    bm = None if bm_np is None else torch.from_numpy(bm_np).cuda()
    sl = None if sl_np is None else torch.from_numpy(sl_np).cuda()
    scale = 1.0 / math.sqrt(d)
    kw = dict(causal=causal, dropout_p=p, seed=seed, offset=offset, block_mask=bm,
              seqlens_k=sl, window=window)

    want = _expected(B, H, N, causal, p, seed, offset, bm_np, sl_np, window)

    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    zeros_o = torch.zeros_like(q)
    ones_do = torch.ones_like(q)
    chunks = range(0, N, d)

    fa.fa_device_status(clear=True)
    lse = None
    fwd_bits = np.zeros((B, H, N, N), dtype=bool)
    dq_bits = np.zeros((B, H, N, N), dtype=bool)
    for c0 in chunks:
        n = min(d, N - c0)
        kv = _one_hot_chunk((B, Hkv), N, d, c0)
        # forward: O_ic is nonzero iff (i, c0 + c) is allowed and kept
        o, lse_c = fa.fwd(q, kv, kv, scale, **kw)
        if lse is None:
            lse = lse_c
        fwd_bits[..., c0:c0 + n] = (o[..., :n] != 0).cpu().numpy()
        # dQ kernel: K = V = one-hot chunk, dO = 1, O = 0 (D = 0)
        dq, _, _ = fa.bwd(q, kv, kv, zeros_o, ones_do, lse, scale, **kw)
        dq_bits[..., c0:c0 + n] = (dq[..., :n] != 0).cpu().numpy()

    # dK/dV kernel: dO = one-hot rows of a chunk of w query rows per query head,
    # each head of a K/V group owning its own w of the d columns.
    w = d // G
    dv_bits = np.zeros((B, H, N, N), dtype=bool)
    kv_any = torch.zeros((B, Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    for r0 in range(0, N, w):
        n = min(w, N - r0)
        do = torch.zeros((B, H, N, d), dtype=torch.bfloat16)
        t = torch.arange(n)
        for g in range(G):
            do[:, g::G, r0 + t, g * w + t] = 1.0
        _, _, dv = fa.bwd(q, kv_any, kv_any, zeros_o, do.cuda(), lse, scale, **kw)
        dv_c = dv.cpu()  # [B, Hkv, N(keys), d]
        for g in range(G):
            # query head hk*G + g, query row r0 + t, key j  <->  dv[b, hk, j, g*w + t]
            blk = (dv_c[..., g * w:g * w + n] != 0).numpy()  # [B, Hkv, N, n]
            dv_bits[:, g::G, r0:r0 + n, :] = blk.transpose(0, 1, 3, 2)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK

    # the construction keeps at least some of each kind, so none of the three
    # checks below can pass vacuously
    assert want.any() and (~want).any()
    for name, got in (("forward", fwd_bits), ("dQ kernel", dq_bits), ("dK/dV kernel", dv_bits)):
        if not np.array_equal(got, want):
            bad = np.argwhere(got != want)
            b, h, i, j = bad[0]
            raise AssertionError(f"{name}: {len(bad)} mask bits differ, first at b={b} h={h} "
                                 f"i={i} j={j} (want {want[b, h, i, j]})")
