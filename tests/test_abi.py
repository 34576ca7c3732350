"""The C-ABI library loads and exports every symbol include/fa.h declares;
host-side validation and host helpers work without a GPU (no compute calls)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import io_aware_exact_07_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from io_aware_exact_07_gb300 import build
    build.build()
    return fa.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "fa.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(fa.EXPORTS)


def test_status_strings(lib):
    for s in range(6):
        assert fa.status_string(s)
    assert fa.status_string(fa.FA_ERR_TIMEOUT) == "device-side wait timed out"


def test_dropout_threshold_matches_oracle(lib):
    for p in (0.0, 0.05, 0.1, 0.3, 0.5, 0.9, 255.4 / 256):
        assert fa.fa_dropout_p8(p) == oracle.p8(p)
    assert fa.fa_dropout_p8(-0.1) == -1
    assert fa.fa_dropout_p8(1.0) == -1
    assert fa.fa_dropout_p8(0.999) == -1  # rounds to 256: everything dropped, rejected


@pytest.mark.parametrize("nb", [1, 2, 3, 6, 8, 64, 128])
def test_library_butterfly_equals_oracle_butterfly(lib, nb):
    assert np.array_equal(fa.fa_butterfly_mask(nb).numpy(), oracle.butterfly(nb))


def test_workspace_size(lib):
    assert fa.fa_bwd_workspace_size(2, 3, 5, 64) == 256
    assert fa.fa_bwd_workspace_size(64, 16, 1024, 64) == 64 * 16 * 1024 * 4
    assert fa.fa_bwd_workspace_size(0, 1, 1, 64) == 0


def _fwd_raw(lib, q=1 << 20, k=1 << 20, v=1 << 20, o=1 << 20, lse=1 << 20, B=1, H=1, N=128,
             d=64, scale=0.125, p=0.0):
    vp = ctypes.c_void_p
    return lib.fa_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, N, d, scale, 0, p, 0, 0, None,
                      None, None)


def test_host_validation_rejects_bad_arguments(lib):
    # every case is rejected on the host before any device work
    assert _fwd_raw(lib, q=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd_raw(lib, q=(1 << 20) + 8) == fa.FA_ERR_INVALID_ARG  # not 16-byte aligned
    assert _fwd_raw(lib, lse=(1 << 20) + 2) == fa.FA_ERR_INVALID_ARG
    assert _fwd_raw(lib, N=0) == fa.FA_ERR_INVALID_ARG
    assert _fwd_raw(lib, B=-1) == fa.FA_ERR_INVALID_ARG
    assert _fwd_raw(lib, B=1 << 16, H=1 << 8, N=1 << 8) == fa.FA_ERR_INVALID_ARG  # B*H*N >= 2^31
    assert _fwd_raw(lib, scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert _fwd_raw(lib, scale=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert _fwd_raw(lib, p=1.0) == fa.FA_ERR_INVALID_ARG
    assert _fwd_raw(lib, d=96) == fa.FA_ERR_UNSUPPORTED
    assert _fwd_raw(lib, d=256) == fa.FA_ERR_UNSUPPORTED
    vp = ctypes.c_void_p
    a = vp(1 << 20)
    # missing workspace for the backward
    st = lib.fa_bwd(a, a, a, a, a, a, a, a, a, 1, 1, 128, 64, 0.125, 0, 0.0, 0, 0, None, None,
                    None, 0, None)
    assert st == fa.FA_ERR_WORKSPACE
    st = lib.fa_bwd(a, a, a, a, a, a, a, a, a, 1, 1, 128, 64, 0.125, 0, 0.0, 0, 0, None, None, a,
                    16, None)
    assert st == fa.FA_ERR_WORKSPACE
    assert lib.fa_debug_philox(vp(0), a, 4, 0, 0, None) == fa.FA_ERR_INVALID_ARG


def test_fp8_grouped_entry_points_validate_on_the_host(lib):
    # rejected before any device work: H not a multiple of H_kv, H_kv < 1, d != 128
    vp = ctypes.c_void_p
    a = vp(1 << 20)
    quant = lambda H, Hkv, d: lib.fa_fp8_quantize_gqa(a, a, a, None, 1, H, Hkv, 128, d, a, a, a,
                                                      a, a, a, a, 1 << 20, None)
    fwd8 = lambda H, Hkv, d: lib.fa_fwd_fp8_gqa(a, a, a, a, a, a, a, a, 1, H, Hkv, 128, d, 0.125,
                                                0, None, None)
    for call in (quant, fwd8):
        assert call(4, 3, 128) == fa.FA_ERR_INVALID_ARG
        assert call(4, 0, 128) == fa.FA_ERR_INVALID_ARG
        assert call(4, 2, 64) == fa.FA_ERR_UNSUPPORTED
    # the H_kv = H entry points are the same calls
    assert lib.fa_fwd_fp8(a, a, a, a, a, a, a, a, 1, 4, 128, 64, 0.125, 0, None, None) == \
        fa.FA_ERR_UNSUPPORTED


def test_window_and_decode_validate_on_the_host(lib):
    vp = ctypes.c_void_p
    a = vp(1 << 20)
    win = lambda wl, wr: lib.fa_fwd_window(a, a, a, a, a, 1, 1, 1, 128, 64, 0.125, 0, wl, wr, 0.0,
                                           0, 0, None, None, None)
    assert win(-2, -1) == fa.FA_ERR_INVALID_ARG
    assert win(-1, -3) == fa.FA_ERR_INVALID_ARG

    def dec(q=1 << 20, H=8, Hkv=2, Nq=1, d=128, scale=0.125, wl=-1, ctas=4, ws=None, wsb=0):
        return lib.fa_decode(vp(q), a, a, a, a, 1, H, Hkv, Nq, 1024, d, scale, 0, wl, None, ctas,
                             ws, wsb, None)
    # explicit CTA counts: the split is planned without asking the device
    assert dec(wl=-2) == fa.FA_ERR_INVALID_ARG
    assert dec(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert dec(q=(1 << 20) + 8) == fa.FA_ERR_INVALID_ARG       # not 16-byte aligned
    assert dec(Hkv=3) == fa.FA_ERR_INVALID_ARG                 # 8 heads do not share 3
    assert dec(ctas=-1) == fa.FA_ERR_INVALID_ARG
    assert dec(Nq=64) == fa.FA_ERR_UNSUPPORTED                 # 4 x 64 rows > one 128-row tile
    assert dec(d=96) == fa.FA_ERR_UNSUPPORTED
    # 2 K/V heads x 8 key tiles over 64 CTAs cuts the heads: partial results need a workspace
    assert dec(ctas=64) == fa.FA_ERR_WORKSPACE


def test_fp8_workspace_covers_grouped_heads(lib):
    # include/fa.h: fa_fp8_workspace_size(B, H, 128) also covers H_kv < H; the
    # quantiser uses B*H + 129*B*H_kv 32-bit words (maxima of Q, K and V's columns)
    for B in (1, 3, 8):
        for H in range(1, 65):
            for Hkv in (g for g in range(1, H + 1) if H % g == 0):
                assert fa.fa_fp8_workspace_size(B, H, 128) >= 4 * (B * H + 129 * B * Hkv)
    assert fa.fa_fp8_workspace_size(1, 1, 64) == 0


def test_product_path_has_no_fallback(monkeypatch, tmp_path):
    """Without the built library the binding raises instead of computing elsewhere."""
    import io_aware_exact_07_gb300 as mod
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_lib", None)
    with pytest.raises(RuntimeError):
        mod.load()


def test_decode_workspace_size(lib):
    """Host-side work split of fa_decode, with an explicit CTA count (no device
    query): B*H_kv*ceil(Nk/128) (K/V head, key tile) pairs in runs of
    ceil(pairs / CTAs); a run length that is a multiple of the tiles per head
    cuts no head and needs no workspace; otherwise each query row gets
    min(runs, (tiles - 1) // run + 2) slots of d + 1 floats (256-byte rounded)."""
    # 1 x 2 heads x 3 tiles = 6 pairs
    assert fa.fa_decode_workspace_size(1, 4, 2, 1, 300, 64, 2) == 0       # runs of 3
    assert fa.fa_decode_workspace_size(1, 4, 2, 1, 300, 64, 1) == 0       # one run of 6
    # runs of 1: 4 slots x 4 rows: 16 x 64 floats + 16 floats
    assert fa.fa_decode_workspace_size(1, 4, 2, 1, 300, 64, 6) == 4096 + 256
    # runs of 2 (3 runs): 3 slots x 4 rows
    assert fa.fa_decode_workspace_size(1, 4, 2, 1, 300, 64, 4) == 3072 + 256
    assert fa.fa_decode_workspace_size(1, 4, 2, 1, 300, 64, 1000) == 4096 + 256  # clamped to 6
    # invalid shapes report 0 (fa_decode itself returns the error)
    assert fa.fa_decode_workspace_size(1, 3, 2, 1, 300, 64, 4) == 0       # H % H_kv
    assert fa.fa_decode_workspace_size(1, 4, 1, 64, 300, 64, 4) == 0      # 4 x 64 rows > 128
    assert fa.fa_decode_workspace_size(1, 4, 2, 1, 300, 96, 4) == 0       # d
    assert fa.fa_decode_workspace_size(1, 4, 2, 1, 0, 64, 4) == 0         # empty cache dim



@pytest.mark.gpu
def test_binding_checks_the_shapes_of_block_mask_and_key_lengths(lib):
    """The kernels index block_mask [nb, nb] and seqlens_k [B] without bounds,
    so the binding refuses wrongly sized ones before any launch."""
    import torch
    B, H, N, d = 2, 1, 300, 64  # nb = 3
    q = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    good_bm = torch.ones((3, 3), dtype=torch.uint8, device="cuda")
    good_sl = torch.full((B,), N, dtype=torch.int32, device="cuda")
    fa.fwd(q, q, q, block_mask=good_bm, seqlens_k=good_sl)
    for bm in (torch.ones((2, 2), dtype=torch.uint8, device="cuda"),
               torch.ones((9,), dtype=torch.uint8, device="cuda"),
               torch.ones((3, 6), dtype=torch.uint8, device="cuda")[:, ::2]):
        with pytest.raises(ValueError):
            fa.fwd(q, q, q, block_mask=bm)
    for sl in (torch.full((1,), N, dtype=torch.int32, device="cuda"),
               torch.full((B, 1), N, dtype=torch.int32, device="cuda"),
               torch.full((B,), N, dtype=torch.int64, device="cuda")):
        with pytest.raises(ValueError):
            fa.fwd(q, q, q, seqlens_k=sl)
        with pytest.raises(ValueError):
            fa.decode(q[:, :, :1], q, q, seqlens_k=sl)
    torch.cuda.synchronize()
