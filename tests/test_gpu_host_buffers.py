"""The host-buffer entry point (gsample_gumbel_argmax_host): logits, per-row
arrays and indices live in pinned host memory, and the kernels read and write
them through their device mapping, with no staging copy. The indices must equal
the device-buffer call's on the same inputs, element by element (the same
kernels run on the same values), and the oracle's under the near-tie rule."""
import numpy as np
import pytest

import token_sampling_logits_gb300 as gs
import workloads as W
from tests import oracle_pool
from tests.gpu_util import Tally, gpu_gumbel, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _pinned_logits(x: np.ndarray, dtype: int):
    if dtype == W.F32:
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).pin_memory()
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).pin_memory()
    return t.view(torch.bfloat16 if dtype == W.BF16 else torch.float16)


def _pinned_rows(batch: W.Batch):
    T = torch.from_numpy(np.ascontiguousarray(batch.temperature, np.float32)).pin_memory()
    S = torch.from_numpy(batch.seed.view(np.int64).copy()).pin_memory()
    O = torch.from_numpy(batch.offset.view(np.int64).copy()).pin_memory()
    return T, S, O


def _host_gumbel(batch: W.Batch, logits=None):
    x = logits if logits is not None else _pinned_logits(batch.logits, batch.dtype)
    T, S, O = _pinned_rows(batch)
    out = gs.gumbel_argmax_host(x, T, S, O)
    return out.numpy().copy()


def _mixed(B, V, dtype, seed):
    rng = np.random.default_rng([seed, B, V, dtype, 77])
    x = (rng.standard_normal((B, V)) * 3.0).astype(np.float32)
    x[rng.random((B, V)) < 0.01] = -np.inf
    T = rng.uniform(0.3, 2.0, B).astype(np.float32)
    T[::5] = 0.0  # greedy rows in the same batch
    return W.Batch("host_mixed", W.encode(x, dtype), dtype, T, W.splitmix64(seed + 5, B),
                   np.full(B, seed + 1, np.uint64))


# B <= 64 takes the cluster-per-row kernel, larger batches the flat split
@pytest.mark.parametrize("dtype,B,V", [(W.F32, 4, 4099), (W.BF16, 9, 151936), (W.F16, 64, 1000),
                                       (W.BF16, 100, 32768), (W.F32, 130, 5003)])
def test_matches_device_path_and_oracle(dtype, B, V):
    b = _mixed(B, V, dtype, seed=B)
    host = _host_gumbel(b)
    dev = gpu_gumbel(b)
    assert np.array_equal(host, dev), np.nonzero(host != dev)[0][:10]
    ref, gap = oracle_pool.rows("gumbel", b.logits, b.dtype, b.temperature, b.seed, b.offset)
    Tally().add(host, ref, gap, greedy_mask=~(b.temperature > 0), where="host buffers")


def test_headline_shape_sampled_rows():
    """The e2e workload (bf16, V = 151936, B = 256): every index equals the
    device path's; 32 rows are checked against the oracle."""
    b = W.throughput(256)
    x = _pinned_logits(b.logits, b.dtype)
    host = _host_gumbel(b, logits=x)
    dev = gpu_gumbel(b)
    assert np.array_equal(host, dev)
    rows = np.arange(0, 256, 8)
    ref, gap = oracle_pool.rows("gumbel", b.logits, b.dtype, b.temperature, b.seed, b.offset,
                                row_ids=rows)
    Tally().add(host[rows], ref, gap, where="headline host buffers")


def test_strided_rows():
    """Rows of a wider pinned matrix (ld > V, rows not 16-byte aligned)."""
    b = _mixed(6, 3001, W.BF16, seed=3)
    wide = np.zeros((6, 3011), np.uint16)
    wide[:, :3001] = b.logits
    xw = _pinned_logits(wide, W.BF16)
    host = gs.gumbel_argmax_host(xw[:, :3001], *_pinned_rows(b)).numpy().copy()
    dev = gpu_gumbel(b, logits_dev=to_device(wide, W.BF16)[:, :3001])
    assert np.array_equal(host, dev)


def test_rejects_buffers_that_are_not_pinned_host_memory():
    L = gs.lib()
    B, V = 4, 256
    x_pin = torch.zeros((B, V), dtype=torch.float32).pin_memory()
    x_pageable = torch.zeros((B, V), dtype=torch.float32)
    x_dev = torch.zeros((B, V), dtype=torch.float32, device="cuda")
    T = torch.ones(B, dtype=torch.float32).pin_memory()
    S = torch.zeros(B, dtype=torch.int64).pin_memory()
    out = torch.zeros(B, dtype=torch.int64).pin_memory()
    ws = gs.new_workspace(B)
    ws_host = torch.zeros(gs.workspace_bytes(B), dtype=torch.uint8).pin_memory()
    st = torch.cuda.current_stream().cuda_stream

    def call(x=x_pin, t=T, o=out, w=ws):
        return L.gsample_gumbel_argmax_host(x.data_ptr(), gs.F32, B, V, V, t.data_ptr(),
                                            S.data_ptr(), S.data_ptr(), o.data_ptr(),
                                            w.data_ptr(), st)

    assert call(x=x_pageable) == gs.ERR_INVALID_ARG
    assert call(x=x_dev) == gs.ERR_INVALID_ARG
    assert call(t=torch.ones(B, dtype=torch.float32, device="cuda")) == gs.ERR_INVALID_ARG
    assert call(o=torch.zeros(B, dtype=torch.int64)) == gs.ERR_INVALID_ARG
    assert call(w=ws_host) == gs.ERR_WORKSPACE
    T0 = torch.zeros(B, dtype=torch.float32).pin_memory()
    assert call(t=T0) == gs.OK
    torch.cuda.synchronize()
    assert out.tolist() == [0, 0, 0, 0]  # greedy on all-equal rows: the lowest index
    with pytest.raises(ValueError):
        gs.gumbel_argmax_host(x_pageable, T, S, S)
