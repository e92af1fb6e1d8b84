"""Top-k / top-p on the Gumbel path (gsample_filtered_gumbel_argmax) against
the oracle's definition: the Gumbel-max over the filter set K ("Softmax-free
GPU sampling", Background: the rejection-based top-k/top-p follow-up).

Sampled rows must return the oracle's index except where the oracle's top-two
scores within K are closer than 1e-5 (the plain sampler's near-tie rule), or
where the nucleus boundary sits within 1e-5 of the row's mass from moving by
one element (binary32 masses on the GPU; the oracle sums in double). Both
exemptions are counted and must stay below 1e-4 of the rows on the workload
tests. Greedy rows must match exactly."""
import numpy as np
import pytest

import oracle
import token_sampling_logits_gb300 as gs
import workloads as W
from tests import oracle_pool
from tests.gpu_util import Tally, register, rows_to_device, to_device
from tests.stats_util import P_THRESHOLD, chi_square

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

NEAR_EDGE = 1e-5


def _gpu(batch, K, P, x=None, ws=None, cluster=0):
    x = to_device(batch.logits, batch.dtype) if x is None else x
    T, S, O = rows_to_device(batch)
    Kt = None if K is None else torch.from_numpy(np.asarray(K, np.int32)).cuda()
    Pt = None if P is None else torch.from_numpy(np.asarray(P, np.float32)).cuda()
    out = gs.filtered_gumbel_argmax(x, T, S, O, top_k=Kt, top_p=Pt, workspace=ws,
                                    cluster=cluster)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _check(b, K, P, tally, where, x=None, cluster=0):
    Kf = np.zeros(b.B, np.int32) if K is None else np.asarray(K, np.int32)
    Pf = np.ones(b.B, np.float32) if P is None else np.asarray(P, np.float32)
    got = _gpu(b, K, P, x=x, cluster=cluster)
    ref, gap, edge = _oracle(b, Kf, Pf)
    greedy = ~(b.temperature > 0)
    # rows on a nucleus edge are exempted like near-ties (gap set to 0) and counted
    tally.add(got, ref, np.where(edge < NEAR_EDGE, 0.0, gap), greedy_mask=greedy, where=where)
    tally.edge = getattr(tally, "edge", 0) + int(((edge < NEAR_EDGE) & ~greedy).sum())


def _oracle(b, Kf, Pf):
    res = [oracle_pool.pool().submit(oracle.filtered_sample_row, np.ascontiguousarray(b.logits[r]),
                                     float(b.temperature[r]), int(b.seed[r]), r,
                                     int(b.offset[r]), int(Kf[r]), float(Pf[r]), b.dtype)
           for r in range(b.B)]
    out = [f.result() for f in res]
    return (np.array([o[0] for o in out], np.int64), np.array([o[1] for o in out]),
            np.array([o[2] for o in out]))


def _small(B, V, dtype, seed, sigma=3.0):
    rng = np.random.default_rng([seed, B, V, dtype])
    x = (rng.standard_normal((B, V)) * sigma).astype(np.float32)
    x[rng.random((B, V)) < 0.01] = -np.inf
    T = rng.uniform(0.3, 2.0, B).astype(np.float32)
    T[::5] = 0.0
    return W.Batch("filt", W.encode(x, dtype), dtype, T, W.splitmix64(seed + 3, B),
                   np.full(B, seed, np.uint64)), rng


@pytest.mark.parametrize("dtype", [W.F32, W.BF16, W.F16])
@pytest.mark.parametrize("B,V", [(1, 1), (3, 7), (5, 64), (7, 1000), (9, 4099), (3, 65536 + 13),
                                 (70, 3000)])
def test_filtered_shapes(dtype, B, V):
    t = Tally()
    for seed in range(2):
        b, rng = _small(B, V, dtype, seed)
        K = rng.choice([0, 1, 2, 5, 40, 10**6], B).astype(np.int32)
        P = rng.choice([1.0, 0.0, 0.3, 0.9, 0.99, np.nan, 2.0], B).astype(np.float32)
        _check(b, K, P, t, "B=%d V=%d" % (B, V))
        _check(b, K, None, t, "top-k only")
        _check(b, None, P, t, "top-p only")
    register("6 filtered (edge cases)", t, assert_bound=False)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16, W.F16])
@pytest.mark.parametrize("cluster", [1, 3, 16])
def test_forced_cluster_sizes(dtype, cluster):
    """The filter at forced cluster sizes: one CTA per row (slices of 240-480 KB
    at V = 120001, re-read from global memory in every phase), an odd size,
    and sixteen CTAs (some of them with an empty slice on the small rows).
    Logits on a coarse grid put many entries on K's last key, so the tie rule
    (lower index first) splits a tie group across CTA slices."""
    t = Tally()
    for B, V in ((6, 20000), (3, 37), (4, 120001)):
        rng = np.random.default_rng([cluster, B, V, dtype])
        x = (rng.standard_normal((B, V)) * 2.0).astype(np.float32)
        x[::2] = np.round(x[::2] * 2.0) / 2.0  # coarse grid: large tie groups
        x[rng.random((B, V)) < 0.01] = -np.inf
        x[rng.random((B, V)) < 0.005] = np.nan
        T = rng.uniform(0.5, 2.0, B).astype(np.float32)
        b = W.Batch("cluster", W.encode(x, dtype), dtype, T, W.splitmix64(cluster, B),
                    np.full(B, 3, np.uint64))
        K = rng.choice([1, 2, 7, 100, 3000], B).astype(np.int32)
        P = rng.choice([1.0, 0.3, 0.8, 0.95], B).astype(np.float32)
        for step in range(3):
            bs = b.at_step(step)
            _check(bs, K, P, t, "cluster=%d B=%d V=%d" % (cluster, B, V), cluster=cluster)
            _check(bs, K, None, t, "cluster=%d top-k" % cluster, cluster=cluster)
            _check(bs, None, P, t, "cluster=%d top-p" % cluster, cluster=cluster)
    register("6 filtered (edge cases)", t, assert_bound=False)


def test_signed_zeros_tie():
    """-0 and +0 are equal logits: the order puts the lower index first whatever
    the sign, so top_k = 2 over a row topped by three zeros keeps the first two."""
    B, V = 4, 3000
    x = np.full((B, V), -5.0, np.float32)
    x[:, [100, 1700, 2900]] = [[-0.0, 0.0, -0.0], [0.0, -0.0, 0.0], [-0.0, -0.0, 0.0],
                               [0.0, 0.0, -0.0]]
    b = W.Batch("zeros", x, W.F32, np.full(B, 0.25, np.float32), W.splitmix64(4, B),
                np.zeros(B, np.uint64))
    t = Tally()
    for step in range(40):
        bs = b.at_step(step)
        got = _gpu(bs, np.full(B, 2, np.int32), None)
        assert np.isin(got, [100, 1700]).all(), got
        _check(bs, np.full(B, 2, np.int32), None, t, "zeros")
        _check(bs, np.full(B, 2, np.int32), None, t, "zeros cluster 2", cluster=2)


def test_filtered_ld_and_misaligned_rows():
    """Rows in a wider buffer (ld > V) and shifted by 1-3 elements: the filter
    then takes the element-by-element load path for every dtype."""
    B, V, ld = 5, 3001, 3008
    rng = np.random.default_rng(12)
    base = (rng.standard_normal((B, ld + 8)) * 2).astype(np.float32)
    K = np.array([3, 0, 40, 1, 7], np.int32)
    P = np.array([0.5, 0.9, 1.0, 0.2, 0.99], np.float32)
    t = Tally()
    for dtype in (W.F32, W.BF16, W.F16):
        enc = W.encode(base, dtype)
        dev = to_device(enc, dtype)
        for shift in (0, 1, 3):
            view = dev[:, shift:shift + V]
            host = np.ascontiguousarray(enc[:, shift:shift + V])
            T = np.array([0.5, 1.0, 0.0, 2.0, 1.5], np.float32)
            b = W.Batch("ld", host, dtype, T, W.splitmix64(9, B), np.full(B, 7, np.uint64))
            for step in range(3):
                _check(b.at_step(step), K, P, t, "ld shift=%d dt=%d" % (shift, dtype), x=view)
    register("6 filtered (edge cases)", t, assert_bound=False)


def test_filtered_large_batch():
    """4100 rows (32,800 CTAs of filter clusters) with mixed filters."""
    b, rng = _small(4100, 1000, W.BF16, 21)
    K = rng.choice([0, 1, 5, 50], b.B).astype(np.int32)
    P = rng.choice([1.0, 0.5, 0.9], b.B).astype(np.float32)
    t = Tally()
    _check(b, K, P, t, "B=4100")
    register("6 filtered (edge cases)", t, assert_bound=False)


def test_rejections_and_acceptances_both_exercised():
    """Flat rows with a tight top-k reject nearly every proposal (the exact
    path); one dominant logit makes every proposal stand (the fast path)."""
    B, V = 16, 20000
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((B, V)) * 0.1).astype(np.float32)
    x[8:, 123] = 30.0
    b = W.Batch("rej", x, W.F32, np.ones(B, np.float32), W.splitmix64(2, B),
                np.zeros(B, np.uint64))
    t = Tally()
    K = np.array([1, 2, 3, 5, 10, 50, 100, 500] * 2, np.int32)
    P = np.array([0.001, 0.01, 0.05, 0.1] * 4, np.float32)
    for step in range(4):
        _check(b.at_step(step), K, None, t, "tight top-k")
        _check(b.at_step(step), None, P, t, "tight top-p")
        _check(b.at_step(step), K, P, t, "both")
    register("6 filtered (edge cases)", t, assert_bound=False)


def test_special_rows():
    B, V = 6, 999
    x = np.random.default_rng(4).standard_normal((B, V)).astype(np.float32)
    x[0, :] = -np.inf
    x[1, 10] = np.inf
    x[1, 900] = np.inf
    x[2, ::3] = np.nan
    x[3, :] = -np.inf
    x[3, 998] = 0.5
    x[4, :] = 1.0  # flat: ties everywhere
    x[5, 7] = x[5, 500] = 40.0  # a tie at the top
    b = W.Batch("special", x, W.F32, np.ones(B, np.float32), W.splitmix64(7, B),
                np.ones(B, np.uint64))
    for K, P in ((3, 0.5), (1, 1.0), (0, 0.0), (7, 0.9)):
        got = _gpu(b, np.full(B, K, np.int32), np.full(B, P, np.float32))
        assert got[0] == -1 and got[1] == 10 and got[3] == 998
        assert not np.isnan(x[2][got[2]])
        ref, gap, edge = _oracle(b, np.full(B, K, np.int32), np.full(B, P, np.float32))
        Tally().add(got, ref, np.where(edge < NEAR_EDGE, 0.0, gap), where="special")


def test_workspace_clean_and_deterministic():
    b, _ = _small(96, 30000, W.BF16, 11)
    rng = np.random.default_rng(9)
    K = rng.choice([1, 3, 20], b.B).astype(np.int32)
    P = rng.choice([0.2, 0.7], b.B).astype(np.float32)
    ws = gs.new_workspace(b.B)
    x = to_device(b.logits, b.dtype)
    a1 = _gpu(b, K, P, x=x, ws=ws)
    assert int(ws.count_nonzero()) == 0
    a2 = _gpu(b, K, P, x=x, ws=ws)
    assert np.array_equal(a1, a2)


def test_throughput_workload_filtered():
    """Full-size bf16 batches (B = 64, 128, 256; the flat split above 64 rows)
    with per-row filters, every row at 45 decode steps (20,160 rows)."""
    t = Tally()
    for B in W.THROUGHPUT_B:
        base = W.throughput(B)
        x = to_device(base.logits, base.dtype)
        rng = np.random.default_rng(B)
        K = rng.choice([0, 1, 10, 50, 200], B).astype(np.int32)
        P = rng.choice([1.0, 0.5, 0.9, 0.95], B).astype(np.float32)
        steps = range(0, 90, 2)
        for s in steps:
            b = base.at_step(s)
            got = _gpu(b, K, P, x=x)
            ref, gap, edge = _oracle(b, K, P)
            t.add(got, ref, np.where(edge < NEAR_EDGE, 0.0, gap), where="B=%d step %d" % (B, s))
            t.edge = getattr(t, "edge", 0) + int((edge < NEAR_EDGE).sum())
    print("nucleus-edge rows: %d" % getattr(t, "edge", 0))
    register("6 filtered (throughput workload)", t)


@pytest.mark.parametrize("K,P", [(3, 1.0), (5, 0.9)])
def test_tiny_statistical_filtered(K, P):
    """3e4 draws of the tiny workload at T = 1: index-exact against the
    oracle, never outside K, and chi-square against the truncated softmax."""
    tiny = W.tiny_statistical()
    x = to_device(tiny.logits, tiny.dtype)
    n = 30_000
    B = tiny.B
    T = torch.ones(B, device="cuda")
    S = gs.seeds_as_tensor(tiny.seed, "cuda")
    Kt = torch.full((B,), K, dtype=torch.int32, device="cuda")
    Pt = torch.full((B,), P, dtype=torch.float32, device="cuda")
    ws = gs.new_workspace(B)
    outs = torch.empty((n, B), dtype=torch.int64, device="cuda")
    offs = torch.arange(n, dtype=torch.int64, device="cuda")[:, None].expand(n, B).contiguous()
    for k in range(n):
        gs.filtered_gumbel_argmax(x, T, S, offs[k], top_k=Kt, top_p=Pt, out=outs[k], workspace=ws)
    torch.cuda.synchronize()
    got = outs.cpu().numpy()
    ref = oracle_pool.filtered_steps(tiny.logits, 1.0, 1234, 0, n, dtype=W.F32, top_k=K,
                                     top_p=P)
    assert np.mean(got == ref) > 1 - 1e-4
    from tests.test_oracle_filter import _k_set

    for r in range(B):
        Kset = _k_set(tiny.logits[r], 1.0, K, P)
        assert np.isin(got[:, r], Kset).all()
        if Kset.size > 1:
            p = np.zeros(tiny.V)
            xk = tiny.logits[r][Kset].astype(np.float64)
            p[Kset] = np.exp(xk - xk.max())
            p /= p.sum()
            pval, _ = chi_square(got[:, r], p)
            assert pval >= P_THRESHOLD, (r, K, P, pval)
