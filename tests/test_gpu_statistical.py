"""GPU draws on the tiny statistical workload: chi-square of 1e6 draws per row
per temperature against exact softmax, masked logits never drawn, and the
first draws bit-identical to the oracle's ("Softmax-free GPU sampling",
Regression guard)."""
import numpy as np
import pytest

import token_sampling_logits_gb300 as gs
import workloads as W
from tests import oracle_pool
from tests.gpu_util import Tally, register, to_device
from tests.stats_util import P_THRESHOLD, chi_square, softmax64

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

N_DRAWS = 1_000_000
CHUNK = 1000
N_ORACLE = 200_000


def gpu_draws(batch, T, n):
    """n decode steps (offset = step) of the whole batch, replayed through a
    captured CUDA graph of CHUNK launches."""
    B = batch.B
    x = to_device(batch.logits, batch.dtype)
    Tt = torch.full((B,), T, dtype=torch.float32, device="cuda")
    S = gs.seeds_as_tensor(batch.seed, "cuda")
    off = torch.zeros((CHUNK, B), dtype=torch.int64, device="cuda")
    out = torch.zeros((CHUNK, B), dtype=torch.int64, device="cuda")
    ws = gs.new_workspace(B)
    L = gs.lib()
    dt, _, V, ld = gs._logits_args(x)
    ramp = torch.arange(CHUNK, dtype=torch.int64, device="cuda")[:, None].expand(CHUNK, B)

    def launch_all():
        st = torch.cuda.current_stream().cuda_stream
        for k in range(CHUNK):
            rc = L.gsample_gumbel_argmax(x.data_ptr(), dt, B, V, ld, Tt.data_ptr(), S.data_ptr(),
                                         off.data_ptr() + 8 * B * k, out.data_ptr() + 8 * B * k,
                                         ws.data_ptr(), st)
            assert rc == 0

    launch_all()  # warm-up outside capture
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
    draws = gpu_draws(b, T, N_DRAWS)
    for r in range(b.B):
        d = draws[:, r]
        assert np.all(d >= 0)
        assert not np.any(np.isneginf(b.logits[r][d])), "a -inf logit was drawn"
        pval, df = chi_square(d, softmax64(b.logits[r], T))
        assert pval >= P_THRESHOLD, (r, T, pval, df)
    ref, gap = oracle_pool.gumbel_argmax_steps(b.logits, T, 1234, 0, N_ORACLE, dtype=W.F32,
                                               want_gap=True)
    t = Tally()
    t.add(draws[:N_ORACLE].ravel(), ref.ravel(), gap.ravel(), where="tiny T=%g" % T)
    register("1 tiny statistical T=%g" % T, t)
