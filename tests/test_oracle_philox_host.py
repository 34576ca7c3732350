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
