"""Pins of the oracle's Philox4x32-10 and its 24-bit uniforms.

The independent reference is curand's host-side PHILOX4_32_10 generator (a
library routine): block n of its output stream is the Philox bijection of the
counter (n >> 16 as a 64-bit value in words 0-1, n & 0xffff in word 2, 0 in
word 3) keyed by the 64-bit seed.  Word 3 of the counter is the high half of
the round number in the verify step's layout and stays 0 in every workload.
"""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest
from scipy import stats


def _curand():
    cands = []
    for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/sbsa-linux/lib",
              "/usr/local/cuda/targets/x86_64-linux/lib"):
        cands += [os.path.join(d, n) for n in ("libcurand.so", "libcurand.so.10")]
    found = ctypes.util.find_library("curand")
    if found:
        cands.append(found)
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    pytest.skip("libcurand not found")


def _curand_host_stream(lib, seed: int, offset_blocks: int, nblocks: int) -> np.ndarray:
    CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(4 * offset_blocks)) == 0
        out = np.zeros(4 * nblocks, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.c_size_t(out.size)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out.reshape(nblocks, 4)


def _counters(offset_blocks: int, nblocks: int) -> np.ndarray:
    n = np.arange(offset_blocks, offset_blocks + nblocks, dtype=np.uint64)
    hi = n >> np.uint64(16)
    c = np.zeros((nblocks, 4), dtype=np.uint32)
    c[:, 0] = (hi & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    c[:, 1] = (hi >> np.uint64(32)).astype(np.uint32)
    c[:, 2] = (n & np.uint64(0xFFFF)).astype(np.uint32)
    return c


@pytest.mark.parametrize("seed,offset", [
    (0, 0), (1, 0), (2, 65530), (0x123456789ABCDEF, 3 * 65536 + 17),
    (0xFFFFFFFFFFFFFFFF, (1 << 48) + 5), (0x0BADC0FFEE123457, (7 << 48) + (3 << 32) + 12345),
])
def test_philox_matches_curand_host_generator(orc, seed, offset):
    lib = _curand()
    nblocks = 4096
    want = _curand_host_stream(lib, seed, offset, nblocks)
    got = orc.philox_batch(seed, _counters(offset, nblocks))
    np.testing.assert_array_equal(got, want)


def test_philox_key_and_counter_sensitivity(orc):
    """Every counter word and both key words change every output word."""
    base = np.array([[5, 6, 7, 8]], dtype=np.uint32)
    ref = orc.philox_batch(0x1111222233334444, base)
    for w in range(4):
        c = base.copy()
        c[0, w] ^= 1
        out = orc.philox_batch(0x1111222233334444, c)
        assert np.all(out != ref)
        # about half the 128 output bits flip (avalanche)
        flips = sum(bin(int(a) ^ int(b)).count("1") for a, b in zip(out[0], ref[0]))
        assert 32 <= flips <= 96
    for seed in (0x1111222233334445, 0x1111222333334444):
        assert np.all(orc.philox_batch(seed, base) != ref)


def test_u24_is_exact_and_uniform(orc):
    assert orc.u24(0) == 0.0
    assert orc.u24(0xFF) == 0.0
    assert orc.u24(0x100) == 2.0 ** -24
    assert orc.u24(0xFFFFFFFF) == 1.0 - 2.0 ** -24
    n = 1 << 18
    ctr = np.zeros((n, 4), np.uint32)
    ctr[:, 0] = np.arange(n, dtype=np.uint32) << 2
    ctr[:, 1] = 12345
    words = orc.philox_batch(7, ctr)
    u = (words >> np.uint32(8)).astype(np.float64) * 2.0 ** -24
    for col in range(4):
        counts = np.bincount((u[:, col] * 1024).astype(np.int64), minlength=1024)
        p = stats.chisquare(counts).pvalue
        assert p > 1e-3, (col, p)
    # words 0 and 1 (accept / sample uniforms of one slot) are uncorrelated
    r = np.corrcoef(u[:, 0], u[:, 1])[0, 1]
    assert abs(r) < 4.0 / np.sqrt(n)
