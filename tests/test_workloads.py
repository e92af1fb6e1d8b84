"""The seeded input recipes: shapes, dtypes, value distributions and per-row
parameters of every workload match their stated recipe, and generation is
deterministic. The CUDA path and the oracle both consume these bytes, so a
silent change here would change what every parity and timing number means."""
import numpy as np
import pytest

import workloads as W


def _f32(b):
    if b.dtype == W.F32:
        return b.logits
    assert b.dtype == W.BF16
    return W.bf16_bits_to_f32(b.logits.view(np.uint16))


def test_generation_is_deterministic():
    for make in (lambda: W.sweep(32768, 4), lambda: W.throughput(64), W.hlg, W.tiny_statistical):
        a, b = make(), make()
        assert np.array_equal(a.logits, b.logits)
        assert np.array_equal(a.temperature, b.temperature)
        assert np.array_equal(a.seed, b.seed) and np.array_equal(a.offset, b.offset)


def test_splitmix64_reference_values():
    # splitmix64 from state 0: the first outputs of the published generator
    got = W.splitmix64(0, 3)
    assert got.dtype == np.uint64
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


@pytest.mark.parametrize("V,B", [(32768, 1), (65536, 4), (151936, 8)])
def test_sweep_recipe(V, B):
    b = W.sweep(V, B)
    assert b.logits.shape == (B, V) and b.dtype == W.F32
    x = b.logits
    inf = np.isneginf(x)
    assert abs(inf.mean() - 0.01) < 0.004  # 1% -inf at uniform positions
    fin = x[~inf]
    assert abs(fin.std() - 3.0) < 0.05 and abs(fin.mean()) < 0.05  # N(0, 3^2)
    assert ((b.temperature >= 0.5) & (b.temperature <= 1.5)).all()
    assert (b.offset == 0).all()
    assert np.array_equal(b.seed, W.splitmix64(7, B))


def test_throughput_recipe():
    b = W.throughput(64)
    assert b.logits.shape == (64, W.THROUGHPUT_V) and b.dtype == W.BF16
    x = _f32(b)
    assert np.isfinite(x).all()
    assert (b.temperature == 1.0).all()
    # 32 bumped ids per row: the base draw is N(0, 4^2), so a +6 bump shows as
    # a heavy right tail; the row's bulk keeps sigma 4
    assert abs(np.median(np.abs(x[0])) / 0.6745 - 4.0) < 0.1
    # the bumps are applied before the bf16 rounding: re-derive them
    rng = np.random.default_rng([3, W.THROUGHPUT_V, 64])
    base = rng.standard_normal((64, W.THROUGHPUT_V), dtype=np.float32) * np.float32(4.0)
    ids = W.zipf_ids(rng, W.THROUGHPUT_V, 32)
    assert len(set(ids.tolist())) == 32 and ids.min() >= 0 and ids.max() < W.THROUGHPUT_V
    row0 = base[0].copy()
    row0[ids] += 6.0
    assert np.array_equal(W.encode(row0[None, :], W.BF16)[0], b.logits[0])


def test_hlg_recipe():
    b = W.hlg()
    assert b.logits.shape == (8, 262144) and b.dtype == W.F32
    assert abs(np.isneginf(b.logits).mean() - 0.005) < 0.001
    assert b.hlg == W.HLG_PARAMS
    assert W.HLG_PARAMS == dict(m=1.3, w=2.0, beta_t=1.0, beta_h=1.5, c=6.0)


def test_mixed_greedy_recipe():
    b = W.mixed_greedy(B=16, V=4096)
    T = b.temperature
    assert (T[0::2] == 0.0).all()
    assert ((T[1::2] >= 0.3) & (T[1::2] <= 2.0)).all()
    x = _f32(b)
    for r in range(8):  # planted ties: the row maximum appears at least three times
        fin = x[r][np.isfinite(x[r])]
        assert (fin == fin.max()).sum() >= 3
    for r in range(8, 16):
        fin = x[r][np.isfinite(x[r])]
        assert (fin == fin.max()).sum() >= 1


def test_tiny_statistical_recipe():
    b = W.tiny_statistical()
    x = b.logits
    assert x.shape == (4, 64)
    assert (x[0] == 8.0).sum() == 1
    assert (x[1] == 0.0).all()
    assert (x[2] == 4.0).sum() == 2
    assert np.isneginf(x[3]).sum() == 16
    assert (b.seed == 1234).all()


def test_at_step_sets_every_offset():
    b = W.sweep(32768, 4).at_step(17)
    assert (b.offset == 17).all()
