"""Pin of the oracle's Philox4x32-10 on the CPU against an external
implementation of the same published generator: cuRAND's host-API generator
CURAND_RNG_PSEUDO_PHILOX4_32_10 (it runs on the host, no GPU needed). Its
stream, after an offset of 4 t0 values, holds in block t = t0 + i (four 32-bit
values) Philox4x32-10 with key (lo32 seed, hi32 seed) and counter
(lo32(t >> 16), t >> 48, t mod 2^16, 0); the test compares the oracle with
that for several seeds, offsets and stream lengths, so the counter words 0, 1
and 2 and both key words take non-zero values (every round mixes all four
words, so word 3 is exercised from the second round on)."""
import ctypes
import os

import numpy as np
import pytest

import oracle

_PHILOX4_32_10 = 161  # curandRngType_t value of CURAND_RNG_PSEUDO_PHILOX4_32_10


def _curand():
    names = []
    for base in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        if base:
            names += [os.path.join(base, "lib64", "libcurand.so"),
                      os.path.join(base, "targets", "sbsa-linux", "lib", "libcurand.so"),
                      os.path.join(base, "targets", "x86_64-linux", "lib", "libcurand.so")]
    names.append("libcurand.so")
    for n in names:
        try:
            return ctypes.CDLL(n)
        except OSError:
            continue
    return None


def host_blocks(lib, seed, t0, nblk):
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), _PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(4 * t0)) == 0
        out = np.zeros(4 * nblk, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(4 * nblk)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out.reshape(nblk, 4)


@pytest.mark.parametrize("seed,t0,nblk", [
    (0x123456789ABCDEF0, 0, 64),
    (0xDEADBEEFCAFEF00D, 65536 - 8, 24),          # word 2 wraps into word 0
    (0x0123456789ABCDEF, (1 << 32) + 2, 16),
    (0xFFFFFFFFFFFFFFFF, (1 << 48) + 3, 16),      # word 1 non-zero
    (42, (5 << 48) + (77 << 16) + 65530, 16),
])
def test_oracle_philox_matches_curand_host_generator(seed, t0, nblk):
    lib = _curand()
    if lib is None:
        pytest.skip("cuRAND library not found")
    blocks = host_blocks(lib, seed, t0, nblk)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for i in range(nblk):
        t = t0 + i
        ctr = [(t >> 16) & 0xFFFFFFFF, t >> 48, t & 0xFFFF, 0]
        assert np.array_equal(oracle.philox4x32_10(ctr, key), blocks[i]), (seed, t)


@pytest.mark.parametrize("seed,offset,rows,p", [
    (0x5EED5EED12345678, 0, [(0, 0), (0, 7), (1, 44)], 0.1),
    (77, 4321, [(0, 1), (3, 232), (63, 255)], 0.3),   # r = b N + i up to 16383
])
def test_oracle_dropout_keep_from_curand_host_blocks(seed, offset, rows, p):
    """The dropout mapping of include/fa.h (row r = (b H + h) N + i, keys 16 g ..
    16 g + 15 use the Philox block with counter (g, r, lo32 offset, hi32 offset);
    key 16 g + e is kept iff byte e of the block, little-endian, is >= p8)
    rebuilt from cuRAND's host generator: with hi32 offset = 0, r < 2^14 and
    lo32 offset < 2^16 that block is block t = (r << 48) | (g << 16) | offset of
    its stream."""
    lib = _curand()
    if lib is None:
        pytest.skip("cuRAND library not found")
    N = 256
    p8 = oracle.p8(p)
    for b, i in rows:
        keep = oracle.dropout_keep([(b, 0)], 1, N, p, seed=seed, offset=offset)[0, i]
        r = b * N + i
        expect = np.zeros(N, dtype=np.uint8)
        for g in range(N // 16):
            blk = host_blocks(lib, seed, (r << 48) | (g << 16) | offset, 1)[0]
            expect[16 * g:16 * g + 16] = (blk.view(np.uint8) >= p8).astype(np.uint8)
        assert np.array_equal(keep, expect), (b, i)
