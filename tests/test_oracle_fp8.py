"""Pins for the oracle's FP8 pieces: the e4m3 codec against torch's
float8_e4m3fn (an independent implementation of the format) and the format's
closed forms, Sylvester's Hadamard matrix against its closed form, the
rotation against orthogonality, the quantiser against its half-ulp bound and
the FP8 forward against the plain forward on exactly representable inputs."""
import numpy as np
import pytest
import torch

import oracle


def rng(seed):
    return np.random.default_rng(seed)


def torch_e4m3(x):
    return torch.tensor(np.asarray(x, dtype=np.float64)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()


def test_decode_every_code_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    dec = oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(dec), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(dec[ok], ref[ok])
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert dec[0x7E] == 448.0 and dec[0x01] == 2.0 ** -9 and dec[0x08] == 2.0 ** -6


def test_encode_matches_torch_in_range():
    r = rng(30)
    x = np.concatenate([r.standard_normal(200000) * 60, r.standard_normal(20000) * 0.004,
                        r.uniform(-448, 448, 20000)])
    assert np.array_equal(oracle.e4m3_encode(x), torch_e4m3(x))


def test_ties_go_to_the_even_code_and_codes_round_trip():
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # 0 .. 448 ascending
    mids = (vals[:-1] + vals[1:]) / 2
    enc = oracle.e4m3_encode(mids).astype(int)
    lo = np.arange(len(mids))
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(enc, expect)
    assert np.array_equal(enc, torch_e4m3(mids).astype(int))
    finite = [c for c in range(256) if c not in (0x7F, 0xFF, 0x80)]
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_decode(np.array(finite, np.uint8))),
                          np.array(finite, np.uint8))


def test_encode_saturates_at_448():
    enc = oracle.e4m3_encode([448.0, 460.0, 500.0, 1e9, -1e9, -449.0])
    assert list(enc) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


@pytest.mark.parametrize("d", [1, 2, 8, 64, 128])
def test_hadamard_closed_form_and_orthogonality(d):
    h = oracle.hadamard(d)
    i, j = np.meshgrid(np.arange(d), np.arange(d), indexing="ij")
    popc = np.vectorize(lambda t: bin(int(t)).count("1"))(i & j)
    assert np.array_equal(h, (-1.0) ** popc)
    assert np.array_equal(h @ h.T, d * np.eye(d))


def test_rotation_keeps_dot_products():
    r = rng(31)
    d = 128
    q, k = r.standard_normal((2, 50, d))
    s = r.choice([-1.0, 1.0], d)
    qr, kr = oracle.rotate(q, s), oracle.rotate(k, s)
    assert np.max(np.abs(qr @ kr.T - q @ k.T)) < 1e-11
    assert np.max(np.abs(np.linalg.norm(qr, axis=1) - np.linalg.norm(q, axis=1))) < 1e-12
    # spreading: one outlier channel becomes d equal-magnitude entries
    e = np.zeros(d)
    e[5] = 100.0
    assert np.allclose(np.abs(oracle.rotate(e, s)), 100.0 / np.sqrt(d))


def test_quantiser_is_within_half_an_ulp():
    r = rng(32)
    B, H, N, d = 2, 3, 70, 64
    q, k, v = r.standard_normal((3, B, H, N, d))
    v[..., 7] *= 40.0  # an outlier column gets its own V scale
    s = r.choice([-1.0, 1.0], d)
    q8, k8, v8, sq, sk, sv = oracle.quantize_fp8(q, k, v, s)
    for x, c, sc in ((oracle.rotate(q, s), q8, sq[:, :, None, None]),
                     (oracle.rotate(k, s), k8, sk[:, :, None, None]), (v, v8, sv[:, :, None, :])):
        y = x / sc                                   # in code units, |y| <= 448
        dec = oracle.e4m3_decode(c)
        # the scale maps each head's (V: each column's) largest magnitude to exactly 448
        red = (2, 3) if c is not v8 else (2,)
        assert np.allclose(np.abs(y).max(axis=red), 448.0, rtol=1e-12, atol=0)
        # the gap to the next e4m3 magnitude above |y| bounds the rounding error by half of it
        mags = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
        idx = np.minimum(np.searchsorted(mags, np.abs(y)), len(mags) - 1)
        gap = mags[idx] - mags[np.maximum(idx - 1, 0)]
        assert np.all(np.abs(dec - y) <= gap / 2 + 1e-12)
    # each head's largest |Q'| element maps to exactly 448
    qr = oracle.rotate(q, s)
    for b in range(B):
        for h in range(H):
            t = np.unravel_index(np.argmax(np.abs(qr[b, h])), qr[b, h].shape)
            assert abs(oracle.e4m3_decode(q8[b, h][t])) == 448.0


def test_fp8_forward_on_representable_inputs_is_the_plain_forward():
    r = rng(33)
    B, H, N, d = 1, 2, 150, 16
    q8, k8, v8 = (r.integers(0, 0x7F, (B, H, N, d)).astype(np.uint8) |
                  (r.integers(0, 2, (B, H, N, d)).astype(np.uint8) << 7) for _ in range(3))
    sq, sk = r.uniform(0.001, 0.01, (2, B, H))
    sv = r.uniform(0.001, 0.01, (B, H, d))
    o, lse = oracle.fwd_fp8(q8, k8, v8, sq, sk, sv, 0.25, causal=True)
    qh = oracle.e4m3_decode(q8) * sq[:, :, None, None]
    kh = oracle.e4m3_decode(k8) * sk[:, :, None, None]
    vh = oracle.e4m3_decode(v8) * sv[:, :, None, :]
    o2, lse2 = oracle.fwd(qh, kh, vh, 0.25, causal=True)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)


def test_no_rotation_quantises_the_inputs_themselves():
    r = rng(34)
    q, k, v = r.standard_normal((3, 1, 2, 40, 16))
    q8, k8, v8, sq, sk, sv = oracle.quantize_fp8(q, k, v, None)
    assert np.array_equal(q8, oracle.e4m3_encode(q / sq[:, :, None, None]))
    assert np.array_equal(k8, oracle.e4m3_encode(k / sk[:, :, None, None]))
    assert np.allclose(sq, np.abs(q).max(axis=(2, 3)) / 448.0, rtol=1e-15)


def test_fp8_forward_grouped_heads_is_the_grouped_plain_forward():
    """Grouped K/V heads: the FP8 oracle on Hkv K/V heads is, per query head
    h, the plain fp64 forward of that head against K/V head h // (H / Hkv),
    written here head by head (not through the repeat in fwd_gqa)."""
    r = rng(35)
    B, H, Hkv, N, d = 2, 6, 2, 90, 16
    q8 = r.integers(0, 256, (B, H, N, d)).astype(np.uint8)
    k8, v8 = (r.integers(0, 256, (B, Hkv, N, d)).astype(np.uint8) for _ in range(2))
    for c in (q8, k8, v8):
        c[(c & 0x7F) == 0x7F] = 0  # no NaN codes
    sq = r.uniform(0.001, 0.01, (B, H))
    sk = r.uniform(0.001, 0.01, (B, Hkv))
    sv = r.uniform(0.001, 0.01, (B, Hkv, d))
    sl = np.array([90, 41])
    o, lse = oracle.fwd_fp8(q8, k8, v8, sq, sk, sv, 0.3, causal=True, seqlens_k=sl)
    G = H // Hkv
    for b in range(B):
        for h in range(H):
            j = h // G
            qh = oracle.e4m3_decode(q8[b, h]) * sq[b, h]
            kh = oracle.e4m3_decode(k8[b, j]) * sk[b, j]
            vh = oracle.e4m3_decode(v8[b, j]) * sv[b, j][None, :]
            o1, l1 = oracle.fwd(qh[None, None], kh[None, None], vh[None, None], 0.3, causal=True,
                                seqlens_k=sl[b:b + 1])
            assert np.array_equal(o[b, h], o1[0, 0]) and np.array_equal(lse[b, h], l1[0, 0])
    # the quantiser's K/V scales are per K/V head: a K/V head with 10x the values
    # gets 10x the scale and the same codes
    x = r.standard_normal((1, 1, 40, 16))
    y = np.concatenate([x, 10 * x], axis=1)
    _, k8q, v8q, _, skq, svq = oracle.quantize_fp8(np.zeros((1, 4, 40, 16)), y, y, None)
    assert np.allclose(skq[0, 1], 10 * skq[0, 0], rtol=1e-14) and np.array_equal(k8q[0, 0], k8q[0, 1])
    assert np.allclose(svq[0, 1], 10 * svq[0, 0], rtol=1e-14) and np.array_equal(v8q[0, 0], v8q[0, 1])
