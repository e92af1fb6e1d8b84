"""HLG kernel vs the CPU oracle on the hlg workload recipe and edge cases,
plus the pages' neutrality gate on the GPU ("HLG sampling", "The degeneracies
are the safety anchors", "Correctness & evaluation" 1)."""
import ctypes

import numpy as np
import pytest

import oracle
import token_sampling_logits_gb300 as gs
import workloads as W
from tests import oracle_pool
from tests.gpu_util import Tally, gpu_gumbel, gpu_hlg, gpu_hlg_steps, register, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

P = W.HLG_PARAMS


def params(mode=gs.PIVOT_TOP, **kw):
    d = dict(m=P["m"], w=P["w"], beta_t=P["beta_t"], beta_h=P["beta_h"], pivot_offset=P["c"],
             pivot_mode=mode)
    d.update(kw)
    return gs.HlgParams(**d)


def _oracle(batch, hp, rows=None):
    extra = dict(m=hp.m, w=hp.w, beta_t=hp.beta_t, beta_h=hp.beta_h, c=hp.pivot_offset,
                 pivot_mode=hp.pivot_mode)
    return oracle_pool.rows("hlg", batch.logits, batch.dtype, batch.temperature, batch.seed,
                            batch.offset, extra=extra, row_ids=rows)


@pytest.mark.parametrize("mode", [gs.PIVOT_TOP, gs.PIVOT_ENTROPY])
def test_hlg_workload(mode):
    """The HLG workload at 2500 decode steps per pivot, every row: 20,000 rows
    against the oracle, with the near-tie share reported per pivot."""
    base = W.hlg()
    x = to_device(base.logits, base.dtype)
    hp = params(mode)
    steps = range(2500)
    got = gpu_hlg_steps(base, hp, steps, logits_dev=x)
    extra = dict(m=hp.m, w=hp.w, beta_t=hp.beta_t, beta_h=hp.beta_h, c=hp.pivot_offset,
                 pivot_mode=hp.pivot_mode)
    ref, gap = oracle_pool.rows_at_steps("hlg", base.logits, base.dtype, base.temperature,
                                         base.seed, steps, extra=extra)
    t = Tally()
    t.add(got.ravel(), ref.ravel(), gap.ravel(), where="hlg mode %d" % mode)
    register("4 hlg (%s pivot)" % ("top" if mode == gs.PIVOT_TOP else "entropy"), t)


@pytest.mark.parametrize("dtype", [W.F32, W.BF16, W.F16])
@pytest.mark.parametrize("B,V,cluster", [(1, 5, 0), (3, 100, 0), (4, 4099, 0), (2, 70001, 0),
                                         (3, 30000, 1), (3, 30000, 2), (2, 50000, 16)])
def test_hlg_shapes(dtype, B, V, cluster):
    rng = np.random.default_rng([B, V, dtype])
    x = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    x[rng.random((B, V)) < 0.01] = -np.inf
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    T[0] = 0.0  # greedy row
    b = W.Batch("hlg_small", W.encode(x, dtype), dtype, T, W.splitmix64(5, B),
                np.full(B, 9, np.uint64))
    for mode in (gs.PIVOT_TOP, gs.PIVOT_ENTROPY):
        hp = params(mode)
        got = gpu_hlg(b, hp, cluster=cluster)
        ref, gap = _oracle(b, hp)
        Tally().add(got, ref, gap, greedy_mask=~(T > 0), where="hlg B=%d V=%d" % (B, V))


def test_hlg_large_row_streams_twice():
    """A row too long for the cluster's shared memory takes the re-reading path."""
    B, V = 2, 1_500_000
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    b = W.Batch("hlg_long", x, W.F32, np.ones(B, np.float32), W.splitmix64(6, B),
                np.full(B, 2, np.uint64))
    hp = params()
    got = gpu_hlg(b, hp)
    ref, gap = _oracle(b, hp)
    Tally().add(got, ref, gap, where="hlg long")


def test_hlg_special_rows():
    B, V = 5, 999
    x = np.random.default_rng(4).standard_normal((B, V)).astype(np.float32)
    x[0, :] = -np.inf
    x[1, 10] = np.inf
    x[1, 900] = np.inf
    x[2, ::3] = np.nan
    x[3, :] = -np.inf
    x[3, 998] = 0.5
    b = W.Batch("hlg_special", x, W.F32, np.ones(B, np.float32), W.splitmix64(7, B),
                np.full(B, 1, np.uint64))
    for mode in (gs.PIVOT_TOP, gs.PIVOT_ENTROPY):
        got = gpu_hlg(b, params(mode))
        assert got[0] == -1 and got[1] == 10 and got[3] == 998
        ref, gap = _oracle(b, params(mode))
        Tally().add(got, ref, gap, where="hlg special")


def test_hlg_neutrality_on_gpu():
    """Rolloff off and m = 1: the HLG kernel draws what the plain kernel draws."""
    base = W.sweep(65536, 8)
    x = to_device(base.logits, base.dtype)
    hp = params(w=float("inf"), m=1.0, pivot_offset=3.0)
    same = total = 0
    for step in range(5):
        b = base.at_step(step)
        h = gpu_hlg(b, hp, logits_dev=x)
        g = gpu_gumbel(b, logits_dev=x)
        ref, gap = oracle_pool.rows("gumbel", b.logits, b.dtype, b.temperature, b.seed, b.offset)
        Tally().add(h, ref, gap, where="neutral hlg")
        same += int((h == g).sum())
        total += b.B
    assert same >= total - 1


def test_hlg_greedy_rows_untouched():
    base = W.hlg(B=4, V=20000)
    b = W.Batch(base.name, base.logits, base.dtype, np.zeros(4, np.float32), base.seed, base.offset)
    got = gpu_hlg(b, params())
    ref, _ = oracle.argmax(b.logits)
    assert np.array_equal(got, ref)


def _rows_oracle(b, curves):
    ref, gap = oracle.hlg_gumbel_argmax(
        b.logits, b.temperature, b.seed, b.offset, m=[c.m for c in curves], w=[c.w for c in curves],
        beta_t=[c.beta_t for c in curves], beta_h=[c.beta_h for c in curves],
        c=[c.pivot_offset for c in curves], pivot_mode=[c.pivot_mode for c in curves],
        dtype=b.dtype)
    return ref, gap


@pytest.mark.parametrize("dtype", [W.F32, W.BF16])
def test_hlg_per_row_curves(dtype):
    """One curve per row ("HLG sampling", "Where it lands in the code": batched
    rows carry per-request parameters): each row matches the oracle with its
    own curve, and equals a launch-wide call made with that curve."""
    rng = np.random.default_rng([41, dtype])
    B, V = 6, 20000
    x = (rng.standard_normal((B, V)) * 3).astype(np.float32)
    x[rng.random((B, V)) < 0.005] = -np.inf
    T = np.array([1.0, 0.7, 0.0, 1.3, 1.0, 0.9], np.float32)
    b = W.Batch("hlg_rows", W.encode(x, dtype), dtype, T, W.splitmix64(8, B),
                np.full(B, 3, np.uint64))
    curves = [params(gs.PIVOT_TOP), params(gs.PIVOT_ENTROPY, m=0.8, w=1.0),
              params(gs.PIVOT_TOP, m=5.0), params(gs.PIVOT_TOP, m=2.0, w=0.5, beta_t=0.5,
                                                  beta_h=3.0, pivot_offset=3.0),
              params(gs.PIVOT_ENTROPY, m=1.0, w=float("inf")), params(gs.PIVOT_TOP, pivot_offset=-2.0)]
    xd = to_device(b.logits, b.dtype)
    got = gs.hlg_gumbel_argmax_rows(xd, torch.from_numpy(T).cuda(),
                                    gs.seeds_as_tensor(b.seed, "cuda"),
                                    gs.seeds_as_tensor(b.offset, "cuda"), curves)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    ref, gap = _rows_oracle(b, curves)
    Tally().add(got, ref, gap, greedy_mask=~(T > 0), where="per-row curves")
    for r in range(B):
        single = gpu_hlg(b, curves[r], logits_dev=xd)
        assert single[r] == got[r], (r, single[r], got[r])


def test_hlg_per_row_invalid_curve_gives_minus_one():
    rng = np.random.default_rng(5)
    B, V = 4, 3000
    x = (rng.standard_normal((B, V)) * 2).astype(np.float32)
    T = np.array([1.0, 1.0, 0.0, 1.0], np.float32)
    b = W.Batch("hlg_bad", x, W.F32, T, W.splitmix64(2, B), np.zeros(B, np.uint64))
    curves = [params(), params(m=-1.0), params(pivot_mode=7), params(beta_h=float("nan"))]
    got = gs.hlg_gumbel_argmax_rows(to_device(x, W.F32), torch.from_numpy(T).cuda(),
                                    gs.seeds_as_tensor(b.seed, "cuda"),
                                    gs.seeds_as_tensor(b.offset, "cuda"), curves)
    torch.cuda.synchronize()
    got = got.cpu().numpy()
    assert got[1] == -1 and got[3] == -1          # sampled rows with a failing curve
    assert got[2] == int(np.argmax(x[2]))         # a greedy row ignores its curve
    ref, gap = _rows_oracle(b, [curves[0]] * B)
    Tally().add(got[:1], ref[:1], gap[:1], where="valid row beside invalid ones")


def test_hlg_score_error_budget():
    """The kernel's exact HLG score tone(x + shift)/T + g against the oracle's
    double-precision curve and Gumbel transform, over all three branches of the
    curve ("HLG sampling", "The transfer function"), within the binary32 budget
    of every step: the rounded z (at most half an ulp of z, times the slope m),
    the curve's own arithmetic (at most 4 ulps of the curve value), the IEEE
    division by T (half an ulp), the Gumbel transform (2e-6, its pinned bound
    over all 2^23 cells) and the final sum (half an ulp of the score)."""
    rng = np.random.default_rng(77)
    n = 1_000_000
    f32 = np.float32
    for T in (1.0, 0.7, 1.6):
        m, w, bt, bh = 1.3, 2.0, 1.0, 1.5
        shift = f32(6.0 - rng.uniform(5, 25))           # c - M for a range of row maxima
        z = np.concatenate([rng.uniform(-60, 12, n // 2), rng.uniform(-w - 1, w + 1, n // 2)])
        x = (z - np.float64(shift)).astype(f32)
        words = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
        words[:64] = np.arange(64, dtype=np.uint32) | np.uint32(0xFFFFFF00)  # largest g
        xd = torch.from_numpy(x).cuda()
        wd = torch.from_numpy(words.view(np.int32)).cuda()
        out = torch.empty(n, dtype=torch.float32, device="cuda")
        hp = gs.HlgParams(m=m, w=w, beta_t=bt, beta_h=bh).to_c()
        rc = gs.lib().gsample_debug_hlg_score(xd.data_ptr(), wd.data_ptr(), n,
                                              ctypes.byref(hp), T, float(shift), out.data_ptr(),
                                              torch.cuda.current_stream().cuda_stream)
        assert rc == gs.OK
        got = out.cpu().numpy().astype(np.float64)
        zd = x.astype(np.float64) + np.float64(shift)
        y = oracle.hlg_curve(zd, m, w, bt, bh)
        Tq = np.float64(f32(T))
        ref = y / Tq + oracle.gumbel_of_words(words)
        ulp = lambda v: np.spacing(np.abs(v).astype(f32)).astype(np.float64)  # noqa: E731
        zf = x.astype(f32) + f32(shift)                   # the kernel's rounded z
        bound = (m * 0.5 * ulp(zf) + 4 * ulp(y)) / Tq + 0.5 * ulp(y / Tq) + 2e-6 + 0.5 * ulp(ref)
        err = np.abs(got - ref)
        worst = int(np.argmax(err / bound))
        print("T=%g: max |score error| %.2e, largest share of the budget %.2f" %
              (T, err.max(), (err / bound).max()))
        assert (err <= bound).all(), (T, float(z[worst]), float(err[worst]), float(bound[worst]))
