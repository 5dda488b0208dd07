"""Pins of the oracle's Philox4x32-10 and of the uniform mapping.

Philox is pinned bit-for-bit against NVIDIA's cuRAND host generator
(CURAND_RNG_PSEUDO_PHILOX4_32_10, generated on the CPU, no GPU needed): its
output block i is Philox(counter = (i // 65536 + offset carry, ., i % 65536, 0),
key = (lo32(seed), hi32(seed))), which covers counter words 0..2 and both key
words.  Counter word 3 is covered by the GPU test against cuRAND's device API.
"""
import ctypes
import ctypes.util
import os

import numpy as np
import pytest

import oracle

CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161  # curand.h


def _curand():
    cands = []
    for d in ("/usr/local/cuda/lib64", "/usr/local/cuda/targets/sbsa-linux/lib",
              "/usr/local/cuda/targets/x86_64-linux/lib"):
        cands += [os.path.join(d, "libcurand.so"), os.path.join(d, "libcurand.so.10")]
    found = ctypes.util.find_library("curand")
    if found:
        cands.append(found)
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    pytest.skip("libcurand not found")


def curand_host_philox(seed: int, offset: int, n: int) -> np.ndarray:
    L = _curand()
    gen = ctypes.c_void_p()
    assert L.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert L.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert L.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, np.uint32)
        assert L.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(n)) == 0
    finally:
        L.curandDestroyGenerator(gen)
    return out.reshape(-1, 4)


@pytest.mark.parametrize("seed", [0, 7, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_philox_matches_curand_host(seed):
    key = [seed & 0xFFFFFFFF, seed >> 32]
    blocks = curand_host_philox(seed, 0, 4 * 70000)  # crosses the c2 -> c0 wrap at 65536
    rng = np.random.default_rng(seed & 0xFFFF)
    idx = np.concatenate([np.arange(8), np.arange(65530, 65545), rng.integers(0, 70000, 200)])
    for i in idx:
        ctr = [i // 65536, 0, i % 65536, 0]
        assert (oracle.philox4x32_10(ctr, key) == blocks[i]).all(), (seed, i)


def test_philox_counter_word1_via_offset():
    # offset 2^50 values = 2^48 blocks = 2^32 steps of c0 -> carries into c1
    off = 2**50 + 4 * 65536 * 5 + 4 * 3
    blocks = curand_host_philox(7, off, 16)
    assert (oracle.philox4x32_10([5, 1, 3, 0], [7, 0]) == blocks[0]).all()
    assert (oracle.philox4x32_10([5, 1, 4, 0], [7, 0]) == blocks[1]).all()


def test_uniform_mapping_properties():
    u = oracle.uniform_row(123, 1, 4, 9, 77, 0, 50_000)
    assert np.all(u > 0) and np.all(u < 1)
    k = u * 2**24
    assert np.all(k == np.round(k)) and np.all(np.round(k) % 2 == 1)  # odd multiples of 2^-24
    # lane/c0 layout: entry v uses block v>>2, lane v&3
    blk = oracle.philox4x32_10([3, (1 << 24) | 4, 9, 77], [123, 0])
    np.testing.assert_array_equal(u[12:16], (2.0 * (blk >> 9) + 1) * 2.0**-24)
    # acceptance draws: tag 0, c0 = 0, lane 0
    a = oracle.uniform(5, 0, 2, 11, 3, 0, 0)
    blk = oracle.philox4x32_10([0, 2, 11, 3], [5, 0])
    assert a == (2.0 * (blk[0] >> 9) + 1) * 2.0**-24


def test_uniform_statistics():
    from scipy import stats
    u = np.concatenate([oracle.uniform_row(s, 1, p, b, r, 0, 40_000)
                        for s, p, b, r in [(0, 0, 0, 0), (1, 3, 5, 7), (2**40, 8, 63, 99)]])
    counts, _ = np.histogram(u, bins=256, range=(0, 1))
    assert stats.chisquare(counts).pvalue > 1e-4
    assert stats.kstest(u, "uniform").pvalue > 1e-4
    # lag-1 correlation along the vocabulary index
    x = u - 0.5
    assert abs(np.mean(x[1:] * x[:-1]) / np.var(x)) < 5.0 / np.sqrt(u.size)


def test_streams_are_distinct():
    base = oracle.uniform_row(1, 1, 2, 3, 4, 0, 64)
    for args in [(2, 1, 2, 3, 4), (1, 0, 2, 3, 4), (1, 1, 3, 3, 4), (1, 1, 2, 4, 4), (1, 1, 2, 3, 5)]:
        assert not np.array_equal(base, oracle.uniform_row(*args, 0, 64))
