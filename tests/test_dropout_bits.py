"""Dropout mask: the device Philox stream and the keep mask it yields must match
the oracle's independent implementation bit for bit; and the oracle's Philox is
pinned to cuRAND's device Philox4_32_10 generator (an external library
implementation of the same published algorithm)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import io_aware_exact_07_gb300 as fa

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("p,seed,offset", [(0.1, 0, 0), (0.5, 12345, 7), (0.9, 2**40 + 3, 2**33)])
@pytest.mark.parametrize("B,H,N", [(1, 1, 128), (2, 3, 130), (1, 2, 257)])
def test_keep_mask_matches_oracle(B, H, N, p, seed, offset):
    keep = torch.empty((B, H, N, N), dtype=torch.uint8, device="cuda")
    assert fa.fa_debug_dropout_keep(keep, B, H, N, p, seed, offset) == fa.FA_OK
    torch.cuda.synchronize()
    heads = [(b, h) for b in range(B) for h in range(H)]
    ref = oracle.dropout_keep(heads, H, N, p, seed=seed, offset=offset).reshape(B, H, N, N)
    assert np.array_equal(keep.cpu().numpy(), ref)


def test_raw_philox_matches_oracle():
    g = np.random.default_rng(0)
    n = 4096
    ctr = g.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    key = (0x243F6A88, 0x85A308D3)
    dc = torch.from_numpy(ctr.view(np.int32)).cuda()
    out = torch.empty_like(dc)
    assert fa.fa_debug_philox(dc, out, n, key[0], key[1]) == fa.FA_OK
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    for t in range(0, n, 97):
        assert np.array_equal(got[t], oracle.philox4x32_10(ctr[t], key))


def _curand_helper():
    src = os.path.join(HERE, "curand_philox_ref.cu")
    lib = os.path.join(HERE, "_build_curand_philox_ref.so")
    if not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                        "-Xcompiler", "-fPIC", src, "-o", lib], check=True)
    h = ctypes.CDLL(lib)
    h.curand_philox_blocks.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
                                       ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
    h.curand_philox_blocks.restype = ctypes.c_int
    return h


@pytest.mark.parametrize("seed,row,offset", [(0, 0, 0), (12345, 77, 3), (2**40 + 5, 1023, 2**35)])
def test_oracle_philox_pinned_to_curand(seed, row, offset):
    """cuRAND's Philox4_32_10 state after curand_init(seed, subsequence=offset,
    skip=4*(row<<32)) has key (lo32 seed, hi32 seed) and counter (0, row, lo32
    offset, hi32 offset); successive curand4() calls advance the low counter
    word. That is exactly the counter layout of one query row of the dropout
    mask, so the oracle's keep bits for that row follow from cuRAND's output."""
    h = _curand_helper()
    nblk = 16
    out = torch.empty((nblk, 4), dtype=torch.int32, device="cuda")
    assert h.curand_philox_blocks(out.data_ptr(), nblk, seed, offset, row, 0) == 0
    torch.cuda.synchronize()
    blocks = out.cpu().numpy().view(np.uint32)
    for t in range(nblk):
        ctr = [t, row, offset & 0xFFFFFFFF, offset >> 32]
        key = [seed & 0xFFFFFFFF, seed >> 32]
        assert np.array_equal(oracle.philox4x32_10(ctr, key), blocks[t]), t
    # and the oracle's keep mask for that row is the byte-wise threshold of those blocks
    N = nblk * 16
    p = 0.3
    p8 = oracle.p8(p)
    H = 1
    b, hh, i = 0, 0, row  # row index r = (b*H + h)*N + i with N > row
    Nrow = max(N, row + 1)
    keep = oracle.dropout_keep([(b, hh)], H, Nrow, p, seed=seed, offset=offset)[0, i, :N]
    bytes_ = blocks.reshape(-1).view(np.uint8)  # little-endian bytes, 16 per block
    assert np.array_equal(keep, (bytes_ >= p8).astype(np.uint8))
