"""Helpers for the GPU parity tests: move a workloads.Batch to the device, run
the CUDA path through the C ABI, and compare with the CPU oracle under the
agreed rule (indices equal, except rows whose top-two perturbed scores differ
by less than NEAR_TIE in the oracle's exact arithmetic; greedy rows exact)."""
from __future__ import annotations

import numpy as np

import token_sampling_logits_gb300 as gs
import workloads as W

NEAR_TIE = 1e-5


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

    @property
    def near_fraction(self):
        return self.near / max(1, self.rows)
