"""CUDA path vs the CPU oracle, element by element, on the workloads' input
recipes and on edge cases. Sampled rows must return the oracle's index except
where the oracle's top-two scores are closer than 1e-5 (binary32 vs double);
greedy rows must match exactly."""
import numpy as np
import pytest

import oracle
import token_sampling_logits_gb300 as gs
import workloads as W
from tests import oracle_pool
from tests.gpu_util import (Tally, gpu_gumbel, gpu_gumbel_steps, register, rows_to_device,
                            to_device)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _oracle_rows(batch, rows=None, kind="gumbel", extra=None):
    return oracle_pool.rows(kind, batch.logits, batch.dtype, batch.temperature, batch.seed,
                            batch.offset, extra=extra, row_ids=rows)


def _check_batch(batch, tally=None, rows=None, ctas=0, where="", cluster=0):
    gpu = gpu_gumbel(batch, ctas=ctas, cluster=cluster)
    rows = np.arange(batch.B) if rows is None else np.asarray(rows)
    ref, gap = _oracle_rows(batch, rows)
    t = tally or Tally()
    t.add(gpu[rows], ref, gap, greedy_mask=~(batch.temperature[rows] > 0), where=where)
    if tally is None:
        register("edge cases", t, assert_bound=False)
    return t


def _small(B, V, dtype, sigma=3.0, inf_frac=0.01, seed=0, T=None):
    rng = np.random.default_rng([seed, B, V, dtype])
    x = (rng.standard_normal((B, V)) * sigma).astype(np.float32)
    if inf_frac:
        x[rng.random((B, V)) < inf_frac] = -np.inf
    if T is None:
        T = rng.uniform(0.3, 2.0, B).astype(np.float32)
    return W.Batch("small", W.encode(x, dtype), dtype, np.asarray(T, np.float32),
                   W.splitmix64(seed + 11, B), np.full(B, seed, np.uint64))


@pytest.mark.parametrize("dtype", [W.F32, W.BF16, W.F16])
@pytest.mark.parametrize("B,V", [(1, 1), (3, 2), (2, 3), (5, 7), (4, 17), (7, 64), (3, 1000),
                                 (9, 4099), (2, 65536 + 13)])
def test_small_shapes(dtype, B, V):
    t = Tally()
    for step in range(3):
        _check_batch(_small(B, V, dtype, seed=step), t, where="B=%d V=%d" % (B, V))
    register("edge cases", t, assert_bound=False)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("ctas", [1, 2, 3, 7, 64, 1000])
def test_forced_cta_counts_and_split_ties(dtype, ctas):
    """Rows split over many CTAs, with the row maximum copied to positions in
    different CTA slices: greedy rows must still take the lowest index."""
    B, V = 6, 20000
    rng = np.random.default_rng(ctas)
    x = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    x = W.roundtrip(x, dtype)
    W.plant_ties(rng, x, range(B))
    T = np.array([0, 0.7, 0, 1.3, 0, 0.4], np.float32)
    b = W.Batch("ties", W.encode(x, dtype), dtype, T, W.splitmix64(3, B), np.full(B, 5, np.uint64))
    _check_batch(b, ctas=ctas, where="ctas=%d" % ctas)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("cluster", [1, 2, 7, 16])
def test_cluster_per_row_kernel(dtype, cluster):
    """The small-batch kernel (one cluster per row) at forced cluster sizes,
    with the row maximum copied into different CTA slices and lanes, mixed
    greedy and sampled rows, and a batch larger than it is chosen for."""
    for B, V in ((6, 20000), (3, 4099), (40, 3000)):
        rng = np.random.default_rng([cluster, B, V])
        x = (rng.standard_normal((B, V)) * 3).astype(np.float32)
        x[rng.random((B, V)) < 0.01] = -np.inf
        x = W.roundtrip(x, dtype)
        W.plant_ties(rng, x, range(min(B, 6)))
        T = rng.uniform(0.3, 2.0, B).astype(np.float32)
        T[::3] = 0.0
        b = W.Batch("cluster", W.encode(x, dtype), dtype, T, W.splitmix64(9, B),
                    np.full(B, 2, np.uint64))
        _check_batch(b, cluster=cluster, where="cluster=%d B=%d V=%d" % (cluster, B, V))


def test_ld_and_misaligned_rows():
    B, V, ld = 5, 3001, 3008
    rng = np.random.default_rng(1)
    base = (rng.standard_normal((B, ld + 8)) * 2).astype(np.float32)
    for dtype in (W.F32, W.BF16, W.F16):
        enc = W.encode(base, dtype)
        dev = to_device(enc, dtype)
        for shift in (0, 1, 3):
            view = dev[:, shift:shift + V]  # ld = ld + 8, row start shifted by `shift` elements
            host = np.ascontiguousarray(enc[:, shift:shift + V])
            T = np.array([0.5, 1.0, 0.0, 2.0, 1.5], np.float32)
            b = W.Batch("ld", host, dtype, T, W.splitmix64(9, B), np.full(B, 7, np.uint64))
            Tt, S, O = rows_to_device(b)
            got = gs.gumbel_argmax(view, Tt, S, O).cpu().numpy()
            ref, gap = _oracle_rows(b)
            Tally().add(got, ref, gap, greedy_mask=~(T > 0), where="shift=%d dt=%d" % (shift, dtype))


@pytest.mark.parametrize("ctas", [3, 40, 400])
def test_flat_split_on_rows_off_128_byte_lines(ctas):
    """The flat split moves each warp's split point down to a unit that starts a
    128-byte line of its row. Here the row stride is 8144 bytes, so successive
    rows start at every 16-byte offset within a line, and the base pointer is
    shifted by 0..112 bytes; with 400 CTAs the warps' ranges shrink to 8 units."""
    B, V = 11, 4000
    rng = np.random.default_rng(ctas)
    base = (rng.standard_normal((B, V + 72)) * 2).astype(np.float32)
    enc = W.encode(base, W.BF16)
    dev = to_device(enc, W.BF16)
    T = rng.uniform(0.3, 2.0, B).astype(np.float32)
    T[::3] = 0.0
    for shift in (0, 8, 24, 56):  # elements: 0, 16, 48 and 112 bytes
        view = dev[:, shift:shift + V]
        host = np.ascontiguousarray(enc[:, shift:shift + V])
        b = W.Batch("lines", host, W.BF16, T, W.splitmix64(ctas, B), np.full(B, shift, np.uint64))
        Tt, S, O = rows_to_device(b)
        got = gs.gumbel_argmax(view, Tt, S, O, ctas=ctas).cpu().numpy()
        ref, gap = _oracle_rows(b)
        Tally().add(got, ref, gap, greedy_mask=~(T > 0), where="ctas=%d shift=%d" % (ctas, shift))


def test_special_values():
    B, V = 8, 777
    x = np.random.default_rng(2).standard_normal((B, V)).astype(np.float32)
    x[0, :] = -np.inf
    x[1, :] = np.nan
    x[2, :] = np.nan
    x[2, 500] = -1.0  # the only candidate
    x[3, 100] = np.inf
    x[3, 50] = np.inf
    x[4, ::2] = np.nan
    x[5, :] = 0.0  # flat
    x[6, :] = -np.inf
    x[6, 776] = 3.0  # last element is the only candidate
    x[7, 3] = 1e30  # huge finite logit dominates
    for T in (1.0, 0.0):
        b = W.Batch("special", x, W.F32, np.full(B, T, np.float32), W.splitmix64(1, B),
                    np.full(B, 3, np.uint64))
        got = gpu_gumbel(b)
        ref, gap = _oracle_rows(b)
        assert got[0] == -1 and got[1] == -1
        assert got[2] == 500 and got[3] == 50 and got[6] == 776 and got[7] == 3
        Tally().add(got, ref, gap, greedy_mask=np.full(B, T <= 0), where="T=%g" % T)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
@pytest.mark.parametrize("path", ["flat", "cluster"])
def test_nan_runs_beside_live_groups(dtype, path):
    """Runs of NaN logits covering whole 4-element groups, in the same tiles as
    logits within reach of the row's best (the dense path's word test lets
    such groups through to the exact pass, which must reject them), at T = 1
    and at a high temperature where many groups pass."""
    B, V = 6, 40000
    rng = np.random.default_rng([dtype, len(path)])
    x = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    for r in range(B):
        starts = rng.integers(0, V // 8, 200) * 8
        for s0 in starts:
            x[r, s0:s0 + 8 * (1 + r % 3)] = np.nan
    x[0, : V // 2] = np.nan
    x = W.roundtrip(x, dtype)
    for T in (1.0, 50.0):
        b = W.Batch("nanruns", W.encode(x, dtype), dtype, np.full(B, T, np.float32),
                    W.splitmix64(5, B), np.full(B, 11, np.uint64))
        got = gpu_gumbel(b, ctas=64) if path == "flat" else gpu_gumbel(b, cluster=8)
        ref, gap = _oracle_rows(b)
        assert not np.isnan(x[np.arange(B), got]).any()
        Tally().add(got, ref, gap, where="%s T=%g" % (path, T))


def test_temperature_edge_values_route_to_greedy():
    B, V = 6, 4096
    b = _small(B, V, W.F32, seed=4, T=np.array([0.0, -1.0, np.nan, -0.0, 1e-30, 3.0], np.float32))
    got = gpu_gumbel(b)
    ref, _ = oracle.argmax(b.logits)
    assert np.array_equal(got[:4], ref[:4])


def test_argmax_entry_matches_library_argmax():
    for dtype in (W.F32, W.BF16, W.F16):
        b = _small(33, 12345, dtype, seed=8)
        x = to_device(b.logits, dtype)
        got = gs.argmax(x).cpu().numpy()
        ref, _ = oracle.argmax(b.logits, dtype=dtype)
        assert np.array_equal(got, ref)
        # torch's argmax returns the first maximal index on this NaN-free data
        xm = x.float().masked_fill(torch.isneginf(x.float()), -3e38)
        assert np.array_equal(got, xm.argmax(dim=1).cpu().numpy())


def test_workspace_left_clean_and_deterministic():
    b = _small(16, 50000, W.BF16, seed=6)
    ws = gs.new_workspace(b.B)
    x = to_device(b.logits, b.dtype)
    a1 = gpu_gumbel(b, logits_dev=x, workspace=ws)
    assert int(ws.count_nonzero()) == 0
    a2 = gpu_gumbel(b, logits_dev=x, workspace=ws)
    assert np.array_equal(a1, a2)
    b2 = b.at_step(1)
    a3 = gpu_gumbel(b2, logits_dev=x, workspace=ws)
    assert not np.array_equal(a1, a3)


def test_sweep_workload():
    """The vocab x batch sweep at every one of its 1000 decode steps, every row:
    39,000 rows against the oracle, under one near-tie bound for the config."""
    steps = range(1000)
    t = Tally()
    for V in W.VOCAB_SWEEP:
        for B in W.BATCH_SWEEP:
            base = W.sweep(V, B)
            got = gpu_gumbel_steps(base, steps)
            ref, gap = oracle_pool.rows_at_steps("gumbel", base.logits, base.dtype,
                                                 base.temperature, base.seed, steps)
            t.add(got.ravel(), ref.ravel(), gap.ravel(), where="sweep V=%d B=%d" % (V, B))
    register("2 sweep", t)


def test_throughput_workload_all_rows():
    """Full-size bf16 batches in the launch configuration the benchmark times:
    every row of B = 64, 128 and 256 at 50 of the 100 decode steps (22,400 rows)."""
    steps = list(range(0, 100, 2))
    t = Tally()
    for B in W.THROUGHPUT_B:
        base = W.throughput(B)
        got = gpu_gumbel_steps(base, steps)
        ref, gap = oracle_pool.rows_at_steps("gumbel", base.logits, base.dtype, base.temperature,
                                             base.seed, steps)
        t.add(got.ravel(), ref.ravel(), gap.ravel(), where="throughput B=%d" % B)
    register("3 throughput", t)


def test_mixed_greedy_workload():
    """Every row of the mixed batch at 80 of its 100 steps: greedy rows byte-exact
    (ties planted on rows 0, 2, 4, 6), sampled rows under the near-tie rule
    (20,480 of them)."""
    base = W.mixed_greedy()
    x = to_device(base.logits, base.dtype)
    greedy = ~(base.temperature > 0)
    steps = [s for s in range(100) if s % 5]
    got = gpu_gumbel_steps(base, steps, logits_dev=x)
    gref, _ = oracle.argmax(base.logits, dtype=base.dtype)
    for k, s in enumerate(steps):
        assert np.array_equal(got[k][greedy], gref[greedy]), "greedy rows differ at step %d" % s
    sampled = np.flatnonzero(~greedy)
    ref, gap = oracle_pool.rows_at_steps("gumbel", base.logits, base.dtype, base.temperature,
                                         base.seed, steps, row_ids=sampled)
    t = Tally()
    t.add(got[:, sampled].ravel(), ref.ravel(), gap.ravel(), where="mixed")
    register("5 mixed greedy (sampled rows)", t)
    g = Tally()
    g.add(got[:, greedy].ravel(), np.tile(gref[greedy], len(steps)),
          np.zeros(greedy.sum() * len(steps)), greedy_mask=np.ones(greedy.sum() * len(steps), bool),
          where="mixed greedy rows")
    register("5 mixed greedy (greedy rows)", g, assert_bound=False)
