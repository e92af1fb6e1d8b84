"""The categorical baseline kernel (softmax + inverse CDF, "Softmax-free GPU
sampling", Background and Performance validation) against the oracle.

Binary32 sums cannot reproduce a double-precision CDF at V ~ 1e5 (the
intervals of small weights are narrower than the sums' rounding), so every
GPU index is located against the oracle's exact CDF: it must be the inverse
CDF of a target within TOL * S of the exact u * S. Greedy and special rows
must match exactly, and 1e6 draws per row and temperature must fit softmax."""
import numpy as np
import pytest

import oracle
import token_sampling_logits_gb300 as gs
import workloads as W
from tests.gpu_util import rows_to_device, to_device
from tests.stats_util import P_THRESHOLD, chi_square, softmax64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TOL = 1e-5  # binary32 CDF error budget, relative to the row's weight sum
N_DRAWS = 1_000_000
CHUNK = 1000


def gpu_cat(batch, logits_dev=None, cluster=0):
    x = logits_dev if logits_dev is not None else to_device(batch.logits, batch.dtype)
    T, S, O = rows_to_device(batch)
    out = gs.categorical(x, T, S, O, cluster=cluster)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def check(batch, got, where=""):
    ref, margin, dist = oracle.categorical(batch.logits, batch.temperature, batch.seed,
                                           batch.offset, probe=got, dtype=batch.dtype)
    greedy = ~(batch.temperature > 0)
    assert np.array_equal(got[greedy], ref[greedy]), where
    bad = (~greedy) & ~(dist <= TOL)
    assert not bad.any(), "%s: %s" % (where, [(int(b), int(got[b]), int(ref[b]), float(dist[b]))
                                            for b in np.nonzero(bad)[0][:5]])
    return int(np.sum(got == ref)), got.size


def _small(B, V, dtype, seed, sigma=3.0):
    rng = np.random.default_rng([seed, B, V, dtype])
    x = (rng.standard_normal((B, V)) * sigma).astype(np.float32)
    x[rng.random((B, V)) < 0.01] = -np.inf
    T = rng.uniform(0.3, 2.0, B).astype(np.float32)
    T[0] = 0.0
    return W.Batch("cat_small", W.encode(x, dtype), dtype, T, W.splitmix64(seed + 3, B),
                   np.full(B, seed, np.uint64))


@pytest.mark.parametrize("dtype", [W.F32, W.BF16, W.F16])
@pytest.mark.parametrize("B,V", [(1, 1), (2, 3), (3, 7), (4, 64), (3, 1000), (5, 4099),
                                 (2, 65536 + 13)])
def test_small_shapes(dtype, B, V):
    for step in range(3):
        b = _small(B, V, dtype, step)
        check(b, gpu_cat(b), "B=%d V=%d" % (B, V))


@pytest.mark.parametrize("cluster", [1, 2, 5, 16])
def test_forced_cluster_sizes(cluster):
    b = _small(4, 30000, W.F32, 7)
    check(b, gpu_cat(b, cluster=cluster), "cluster=%d" % cluster)


@pytest.mark.parametrize("V", W.VOCAB_SWEEP)
@pytest.mark.parametrize("B", W.BATCH_SWEEP)
def test_sweep_workload(V, B):
    base = W.sweep(V, B)
    x = to_device(base.logits, base.dtype)
    same = total = 0
    for step in (0, 1, 999):
        b = base.at_step(step)
        s, t = check(b, gpu_cat(b, logits_dev=x), "sweep V=%d B=%d step %d" % (V, B, step))
        same += s
        total += t
    print("sweep V=%d B=%d: index equal to the double-precision CDF's in %d of %d rows"
          % (V, B, same, total))


def test_special_rows():
    x = np.array([[1.0, 3.0, 3.0, -2.0],                       # greedy (T = 0) below
                  [0.0, np.inf, 5.0, np.inf],                  # +inf: lowest +inf index
                  [-np.inf, -np.inf, -np.inf, -np.inf],        # nothing to draw
                  [np.nan, np.nan, 2.0, np.nan],               # NaN never drawn
                  [-np.inf, 0.5, -np.inf, -np.inf]], np.float32)
    T = np.array([0.0, 1.0, 1.0, 1.0, 0.7], np.float32)
    b = W.Batch("cat_special", x, W.F32, T, W.splitmix64(1, 5), np.arange(5, dtype=np.uint64))
    got = gpu_cat(b)
    assert got.tolist() == [1, 1, -1, 2, 1]


def _draws(batch, T, n):
    B = batch.B
    x = to_device(batch.logits, batch.dtype)
    Tt = torch.full((B,), T, dtype=torch.float32, device="cuda")
    S = gs.seeds_as_tensor(batch.seed, "cuda")
    off = torch.zeros((CHUNK, B), dtype=torch.int64, device="cuda")
    out = torch.zeros((CHUNK, B), dtype=torch.int64, device="cuda")
    L = gs.lib()
    dt, _, V, ld = gs._logits_args(x)
    ramp = torch.arange(CHUNK, dtype=torch.int64, device="cuda")[:, None].expand(CHUNK, B)

    def launch_all():
        st = torch.cuda.current_stream().cuda_stream
        for k in range(CHUNK):
            rc = L.gsample_categorical(x.data_ptr(), dt, B, V, ld, Tt.data_ptr(), S.data_ptr(),
                                       off.data_ptr() + 8 * B * k, out.data_ptr() + 8 * B * k, st)
            assert rc == 0

    launch_all()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        launch_all()
    res = torch.empty((n, B), dtype=torch.int64, device="cuda")
    for c0 in range(0, n, CHUNK):
        off.copy_(ramp + c0)
        g.replay()
        res[c0:c0 + CHUNK].copy_(out)
    torch.cuda.synchronize()
    return res.cpu().numpy()


@pytest.mark.parametrize("T", [0.5, 1.0, 1.5])
def test_tiny_statistical(T):
    b = W.tiny_statistical()
    draws = _draws(b, T, N_DRAWS)
    for r in range(b.B):
        d = draws[:, r]
        assert np.all(d >= 0)
        assert not np.any(np.isneginf(b.logits[r][d])), "a -inf logit was drawn"
        pval, df = chi_square(d, softmax64(b.logits[r], T))
        assert pval >= P_THRESHOLD, (r, T, pval, df)
    # the first draws against the oracle's exact CDF
    for k in range(0, 2000, 97):
        bk = W.Batch(b.name, b.logits, b.dtype, np.full(b.B, T, np.float32), b.seed,
                     np.full(b.B, k, np.uint64))
        check(bk, draws[k], "tiny T=%g step %d" % (T, k))
