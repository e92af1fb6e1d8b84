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


def _word_test(x, w, L, T):
    torch = pytest.importorskip("torch")
    xd = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    wd = torch.from_numpy(np.ascontiguousarray(w, np.uint32).view(np.int32)).cuda()
    thr = torch.zeros(x.size, dtype=torch.int32, device="cuda")
    flags = torch.zeros(x.size, dtype=torch.uint8, device="cuda")
    st = gs.lib().gsample_debug_word_test(xd.data_ptr(), wd.data_ptr(), x.size, L, T,
                                          thr.data_ptr(), flags.data_ptr(),
                                          torch.cuda.current_stream().cuda_stream)
    assert st == gs.OK
    torch.cuda.synchronize()
    return thr.cpu().numpy().view(np.uint32).astype(np.int64), flags.cpu().numpy()


@pytest.mark.parametrize("L,T", [(12.5, 1.0), (12.5, 0.05), (3.0, 0.7), (-40.0, 3.0),
                                 (float("-inf"), 1.0)])
def test_group_word_threshold_covers_the_element_test(L, T):
    """The group test (largest word >= an integer threshold computed from the
    largest logit before the Philox block is known) must pass every word the
    element test passes, and may pass more only just below the boundary."""
    rng = np.random.default_rng(abs(hash((L, T))) % (1 << 32))
    top = (L + 1) * T if np.isfinite(L) else 10.0
    x = np.concatenate([rng.uniform(top - 20 * T - 5, top, 4000),
                        [np.nan, np.inf, -np.inf, 0.0, -0.0]]).astype(np.float32)
    thr, _ = _word_test(x, np.zeros(x.size, np.uint32), L, T)
    offsets = np.array([-2000, -1700, -1300, -1024, -600, -513, -512, -511, -1, 0, 1, 511, 512,
                        1700, 100000], np.int64)
    xs = np.repeat(x, offsets.size + 8)
    near = (thr[:, None] + offsets[None, :]).clip(0, 0xFFFFFFFF)
    rand = rng.integers(0, 1 << 32, (x.size, 8), dtype=np.int64)
    ws = np.concatenate([near, rand], axis=1).reshape(-1)
    thr2, flags = _word_test(xs, ws.astype(np.uint32), L, T)
    assert np.array_equal(thr2, np.repeat(thr, offsets.size + 8))
    elem, grp = (flags & 1) != 0, (flags & 2) != 0
    missed = elem & ~grp
    assert not missed.any(), list(zip(xs[missed][:5], ws[missed][:5], thr2[missed][:5]))
    # extra group passes sit within the rounding slack below the exact boundary
    extra = grp & ~elem & ~np.isnan(xs)
    assert (ws[extra] - thr2[extra] < 1700).all()
    assert elem[(ws - thr2 >= 1700) & ~np.isnan(xs)].all()
    # specials: +inf always passes; so does a NaN maximum (the exact pass then
    # rejects it), and the element test never passes NaN
    assert (thr[x == np.inf] == 0).all()
    if np.isfinite(L):
        assert (thr[np.isnan(x)] == 0).all()
    assert not elem[np.isnan(xs)].any()
