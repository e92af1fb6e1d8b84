"""Helpers for the GPU parity tests: move a workloads.Batch to the device, run
the CUDA path through the C ABI, and compare with the CPU oracle under the
agreed rule (indices equal, except rows whose top-two perturbed scores differ
by less than NEAR_TIE in the oracle's exact arithmetic; greedy rows exact)."""
from __future__ import annotations

import numpy as np

import token_sampling_logits_gb300 as gs
import workloads as W

NEAR_TIE = 1e-5
# The parity rule's bound on the share of exempted (near-tie) rows, per config.
MAX_NEAR_FRACTION = 1e-4
# Rows checked per config over the whole session (name -> Tally); printed as a
# table at the end of the run (tests/conftest.py) and written as JSON to the
# path in GSAMPLE_PARITY_TABLE if that variable is set.
PARITY = {}


def torch_mod():
    import torch

    return torch


def to_device(x: np.ndarray, dtype: int, device="cuda"):
    torch = torch_mod()
    if dtype == W.F32:
        return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(device)
    t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(device)
    return t.view(torch.bfloat16 if dtype == W.BF16 else torch.float16)


def rows_to_device(batch: W.Batch, device="cuda"):
    torch = torch_mod()
    T = torch.from_numpy(np.ascontiguousarray(batch.temperature, dtype=np.float32)).to(device)
    S = gs.seeds_as_tensor(batch.seed, device)
    O = gs.seeds_as_tensor(batch.offset, device)
    return T, S, O


def gpu_gumbel(batch: W.Batch, logits_dev=None, ctas: int = 0, workspace=None, cluster: int = 0):
    torch = torch_mod()
    x = logits_dev if logits_dev is not None else to_device(batch.logits, batch.dtype)
    T, S, O = rows_to_device(batch)
    out = gs.gumbel_argmax(x, T, S, O, workspace=workspace, ctas=ctas, cluster=cluster)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def gpu_hlg(batch: W.Batch, params: gs.HlgParams, logits_dev=None, cluster: int = 0,
            workspace=None):
    torch = torch_mod()
    x = logits_dev if logits_dev is not None else to_device(batch.logits, batch.dtype)
    T, S, O = rows_to_device(batch)
    out = gs.hlg_gumbel_argmax(x, T, S, O, params, workspace=workspace, cluster=cluster)
    torch.cuda.synchronize()
    return out.cpu().numpy()


class Tally:
    """Mismatch bookkeeping across many rows."""

    def __init__(self):
        self.rows = 0
        self.near = 0
        self.near_mismatch = 0

    def add(self, gpu, ref, gap, greedy_mask=None, where=""):
        gpu = np.asarray(gpu)
        ref = np.asarray(ref)
        gap = np.asarray(gap)
        greedy = np.zeros(gpu.shape, bool) if greedy_mask is None else np.asarray(greedy_mask)
        bad_greedy = greedy & (gpu != ref)
        assert not bad_greedy.any(), "%s greedy rows differ: %s" % (
            where, list(zip(np.nonzero(bad_greedy)[0][:5], gpu[bad_greedy][:5], ref[bad_greedy][:5])))
        near = (~greedy) & (gap < NEAR_TIE)
        bad = (~greedy) & (gpu != ref) & ~near
        assert not bad.any(), "%s sampled rows differ beyond the near-tie rule: %s" % (
            where, [(int(i), int(gpu[i]), int(ref[i]), float(gap[i])) for i in np.nonzero(bad)[0][:5]])
        self.rows += gpu.size
        self.near += int(near.sum())
        self.near_mismatch += int(((gpu != ref) & near).sum())

    def merge(self, other: "Tally"):
        self.rows += other.rows
        self.near += other.near
        self.near_mismatch += other.near_mismatch
        return self

    @property
    def near_fraction(self):
        return self.near / max(1, self.rows)

    def summary(self):
        return "rows %d, near-tie rows %d (fraction %.2e), near-tie mismatches %d" % (
            self.rows, self.near, self.near_fraction, self.near_mismatch)


def register(config: str, tally: Tally, assert_bound: bool = True):
    """Add a test's rows to its config's session total. With assert_bound, the
    test's own rows must already meet the near-tie bound; the workload tests
    check at least 2e4 rows each, so that one exempted row stays within it."""
    PARITY.setdefault(config, Tally()).merge(tally)
    print("%s: %s" % (config, tally.summary()))
    if assert_bound:
        assert tally.rows >= int(2 / MAX_NEAR_FRACTION), (config, tally.rows)
        assert tally.near_fraction < MAX_NEAR_FRACTION, (config, tally.summary())


def gpu_gumbel_steps(batch: W.Batch, steps, logits_dev=None):
    """The CUDA path at every decode step in `steps` (offset = step for every
    row): int64[len(steps), B]."""
    torch = torch_mod()
    x = logits_dev if logits_dev is not None else to_device(batch.logits, batch.dtype)
    T, S, _ = rows_to_device(batch)
    outs = []
    for s in steps:
        O = torch.full((batch.B,), int(s), dtype=torch.int64, device=x.device)
        outs.append(gs.gumbel_argmax(x, T, S, O))
    torch.cuda.synchronize()
    return torch.stack(outs).cpu().numpy()


def gpu_hlg_steps(batch: W.Batch, params, steps, logits_dev=None):
    """The HLG kernel at every decode step in `steps`: int64[len(steps), B]."""
    torch = torch_mod()
    x = logits_dev if logits_dev is not None else to_device(batch.logits, batch.dtype)
    T, S, _ = rows_to_device(batch)
    outs = []
    for s in steps:
        O = torch.full((batch.B,), int(s), dtype=torch.int64, device=x.device)
        outs.append(gs.hlg_gumbel_argmax(x, T, S, O, params))
    torch.cuda.synchronize()
    return torch.stack(outs).cpu().numpy()
