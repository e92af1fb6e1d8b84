"""Pins of the oracle's Philox4x32-10 and its (seed, row, element, offset)
stream layout against things other than itself.

Philox4x32-10 is defined by Salmon et al., "Parallel Random Numbers: As Easy as
1, 2, 3" (SC'11). The library pin is cuRAND's host-side PHILOX4_32_10 generator
(run on the CPU, no GPU needed): its value n at generator offset o is word
(o + n) & 3 of the block whose counter is
    (lo32(j >> 16), hi32(j >> 16), j & 0xffff, 0),  j = (o + n) >> 2,
keyed by (lo32(seed), hi32(seed)); the test establishes that layout and the
block function together, since neither could match by accident.
"""
import ctypes
import ctypes.util
import glob
import os

import numpy as np
import pytest

import oracle

CURAND_RNG_PSEUDO_PHILOX4_32_10 = 161


def _find_curand():
    cands = []
    name = ctypes.util.find_library("curand")
    if name:
        cands.append(name)
    cands += sorted(glob.glob("/usr/local/cuda/lib64/libcurand.so*"))
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    return None


_CURAND = _find_curand()


def curand_host_words(seed: int, offset: int, n: int) -> np.ndarray:
    lib = _CURAND
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), CURAND_RNG_PSEUDO_PHILOX4_32_10) == 0
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(n, dtype=np.uint32)
        assert lib.curandGenerate(gen, ctypes.c_void_p(out.ctypes.data), ctypes.c_size_t(n)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out


def curand_layout_counters(offset: int, n: int):
    pos = np.arange(n, dtype=np.uint64) + np.uint64(offset)
    j = pos >> np.uint64(2)
    hi = j >> np.uint64(16)
    ctr = np.stack([(hi & np.uint64(0xFFFFFFFF)).astype(np.uint32),
                    (hi >> np.uint64(32)).astype(np.uint32),
                    (j & np.uint64(0xFFFF)).astype(np.uint32),
                    np.zeros(n, dtype=np.uint32)], axis=1)
    return ctr, (pos & np.uint64(3)).astype(np.int64)


@pytest.mark.skipif(_CURAND is None, reason="cuRAND host library not found")
@pytest.mark.parametrize("seed", [0, 1234, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF,
                                  0x63CBE1E459320DD7])
@pytest.mark.parametrize("offset", [0, 4 * 65536 * 3 + 8, (1 << 50) + 12, (1 << 62) + (5 << 18)])
def test_philox_matches_curand_host_generator(seed, offset):
    n = 4 * 70000  # spans a wrap of the 16-bit subsequence field
    got = curand_host_words(seed, offset, n)
    ctr, word = curand_layout_counters(offset, n)
    blocks = oracle.philox_blocks(seed & 0xFFFFFFFF, seed >> 32, ctr)
    mine = blocks[np.arange(n), word]
    bad = np.nonzero(mine != got)[0]
    assert bad.size == 0, "first mismatch at value %d: oracle %08x curand %08x" % (
        bad[0], mine[bad[0]], got[bad[0]])


def test_stream_word_layout():
    """Element i of row r at offset o is word i&3 of the block with counter
    (i>>2, r, lo32(o), hi32(o)) under key (lo32(seed), hi32(seed))."""
    rng = np.random.default_rng(0)
    for _ in range(200):
        seed = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        row = int(rng.integers(0, 2**31))
        off = int(rng.integers(0, 2**63))
        i = int(rng.integers(0, 2**31))
        blk = oracle.philox4x32_10((seed & 0xFFFFFFFF, seed >> 32),
                                   (i >> 2, row, off & 0xFFFFFFFF, off >> 32))
        assert oracle.stream_words(seed, row, off, i, 1)[0] == blk[i & 3]


def test_stream_statistics():
    """Uniformity of the raw words (byte histogram chi-square) and no
    correlation between neighbouring rows or offsets."""
    from scipy import stats

    w = oracle.stream_words(7, 3, 11, 0, 1 << 20)
    counts = np.bincount((w & 0xFF).astype(np.int64), minlength=256)
    assert stats.chisquare(counts).pvalue > 1e-4
    counts = np.bincount((w >> 24).astype(np.int64), minlength=256)
    assert stats.chisquare(counts).pvalue > 1e-4
    a = oracle.stream_words(7, 3, 11, 0, 1 << 16).astype(np.float64)
    for other in (oracle.stream_words(7, 4, 11, 0, 1 << 16), oracle.stream_words(7, 3, 12, 0, 1 << 16),
                  oracle.stream_words(8, 3, 11, 0, 1 << 16)):
        r = np.corrcoef(a, other.astype(np.float64))[0, 1]
        assert abs(r) < 5.0 / np.sqrt(a.size)
    # distinct rows / offsets / seeds give different streams
    assert not np.array_equal(oracle.stream_words(7, 3, 11, 0, 64), oracle.stream_words(7, 4, 11, 0, 64))
