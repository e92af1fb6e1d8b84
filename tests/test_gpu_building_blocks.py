"""The kernels' Philox4x32-10 and Gumbel transform, compared one by one with
the CPU oracle (independent code): raw words bit-exact over millions of
counters, and the binary32 Gumbel of every one of the 2^23 uniform cells
against the oracle's double, with the pruning bound checked on each cell."""
import numpy as np
import pytest

import oracle
import token_sampling_logits_gb300 as gs
from tests import oracle_pool

pytestmark = pytest.mark.gpu


def _philox_job(args):
    import oracle as o

    key0, key1, row, offset, g0, n = args
    j = np.arange(g0, g0 + n, dtype=np.uint64)
    ctr = np.stack([(j & np.uint64(0xFFFFFFFF)).astype(np.uint32),
                    np.full(n, row, dtype=np.uint32),
                    np.full(n, offset & 0xFFFFFFFF, dtype=np.uint32),
                    np.full(n, offset >> 32, dtype=np.uint32)], axis=1)
    return o.philox_blocks(key0, key1, ctr)


@pytest.mark.parametrize("seed,row,offset,group0", [
    (1234, 0, 0, 0),
    (0x63CBE1E459320DD7, 511, 999_999, 1 << 20),
    (0xFFFFFFFFFFFFFFFF, 0x7FFFFFFF, (1 << 40) + 3, (1 << 29) - (1 << 22)),
])
def test_philox_bit_exact(seed, row, offset, group0):
    n = 1 << 22  # 16.7M words per case
    got = gs.debug_philox(seed, row, offset, group0, n).cpu().numpy().view(np.uint32)
    chunks = 32
    jobs = [(seed & 0xFFFFFFFF, seed >> 32, row, offset, group0 + k * (n // chunks), n // chunks)
            for k in range(chunks)]
    want = np.concatenate(list(oracle_pool.pool().map(_philox_job, jobs)))
    bad = np.nonzero((got != want).any(axis=1))[0]
    assert bad.size == 0, "first mismatch at group %d" % (group0 + bad[0])


def test_gumbel_transform_all_cells():
    torch = pytest.importorskip("torch")
    k = np.arange(1 << 23, dtype=np.uint32)
    words = (k << np.uint32(9)) | np.uint32(0x1FF) * (k & np.uint32(1))  # low bits must not matter
    g_dev, bound_dev = gs.debug_gumbel(torch.from_numpy(words.view(np.int32)).cuda())
    g = g_dev.cpu().numpy().astype(np.float64)
    bound = bound_dev.cpu().numpy().astype(np.float64)
    ref = oracle.gumbel_of_words(words)
    err = np.abs(g - ref)
    assert err.max() < 2e-6, err.max()
    # the pruning constants: max g below 16.64, and the per-word bound holds
    assert g.max() < 16.64
    assert np.all(bound >= ref - 4e-6)  # -log(1-u) >= g exactly; binary32 rounding aside
    assert np.all(g <= bound + 1e-3)
