"""gsample_gumbel_argmax_static: the entry point for callers that cannot
allocate device memory (plugins inside a host engine that owns all device
memory, fixed memory budgets, decode loops that must not stall on
cudaMalloc/cudaFree). It keeps its merge state in an array inside the library
instead of a caller workspace. Called through the C ABI, its indices must equal
those of gsample_gumbel_argmax on the same inputs, on two calls in a row (the
second call reuses whatever the first left in the shared array).

This file is named so that pytest collects it last."""
import numpy as np
import pytest

import token_sampling_logits_gb300 as gs
import workloads as W
from tests.gpu_util import rows_to_device, to_device

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

MAX_ROWS = 4096  # GSAMPLE_STATIC_WS_MAX_ROWS in include/gsample.h


def _call_static(x, T, S, O, out):
    dt, B, V, ld = gs._logits_args(x)
    return gs.lib().gsample_gumbel_argmax_static(
        x.data_ptr(), dt, B, V, ld, T.data_ptr(), S.data_ptr(), O.data_ptr(), out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


# Both batches take the flat split (more than 64 rows), whose merge state lives
# in the shared array; smaller batches take a kernel that needs none.
@pytest.mark.parametrize("make", [lambda: W.mixed_greedy(B=96), lambda: W.sweep(151936, 128)])
def test_static_workspace_matches_caller_workspace(make):
    base = make()
    x = to_device(base.logits, base.dtype)
    for step in (0, 1):  # two calls in a row on the shared array
        b = base.at_step(step)
        T, S, O = rows_to_device(b)
        out_static = torch.full((b.B,), -7, dtype=torch.int64, device="cuda")
        assert _call_static(x, T, S, O, out_static) == gs.OK
        ref = gs.gumbel_argmax(x, T, S, O)
        torch.cuda.synchronize()
        assert np.array_equal(out_static.cpu().numpy(), ref.cpu().numpy()), step


def test_larger_batch_after_smaller_one():
    """A call that uses more rows of the shared array than the call before it,
    on the same stream: the rows the first call never touched must be cleared
    like the others."""
    small = W.throughput(80)
    large = W.mixed_greedy(B=300)
    xs = to_device(small.logits, small.dtype)
    xl = to_device(large.logits, large.dtype)
    for step in (3, 4):
        for base, x in ((small, xs), (large, xl)):
            b = base.at_step(step)
            T, S, O = rows_to_device(b)
            out_static = torch.full((b.B,), -7, dtype=torch.int64, device="cuda")
            assert _call_static(x, T, S, O, out_static) == gs.OK
            ref = gs.gumbel_argmax(x, T, S, O)
            torch.cuda.synchronize()
            assert np.array_equal(out_static.cpu().numpy(), ref.cpu().numpy()), (b.B, step)


def test_static_workspace_size_limit():
    x = torch.zeros((MAX_ROWS + 1, 16), dtype=torch.float32, device="cuda")
    T = torch.ones(MAX_ROWS + 1, device="cuda")
    S = torch.zeros(MAX_ROWS + 1, dtype=torch.int64, device="cuda")
    out = torch.zeros(MAX_ROWS + 1, dtype=torch.int64, device="cuda")
    assert _call_static(x, T, S, S, out) == gs.ERR_INVALID_ARG
    # the largest accepted batch works
    assert _call_static(x[:MAX_ROWS], T[:MAX_ROWS], S[:MAX_ROWS], S[:MAX_ROWS],
                        out[:MAX_ROWS]) == gs.OK
    torch.cuda.synchronize()
    ref = gs.gumbel_argmax(x[:MAX_ROWS], T[:MAX_ROWS], S[:MAX_ROWS], S[:MAX_ROWS])
    assert torch.equal(out[:MAX_ROWS], ref)
