"""Seeded synthetic inputs for the sampler's workloads.

This module only builds inputs: logits matrices, per-row temperatures, seeds
and offsets. It holds none of the sampler's arithmetic, and both the CUDA path
and the CPU oracle consume exactly the bytes it produces.

Workloads (the sampling step of LLM decoding over a [B, V] logits matrix):

  tiny_statistical   B=4, V=64, f32. Row 0 peaked (one logit 8.0, rest N(0,1)),
                     row 1 flat (all 0), row 2 bimodal (two logits 4.0, rest
                     N(0,1)), row 3 N(0, 2^2) with 16 entries at -inf.
                     seed 1234 for every row; offsets 0..n-1.
  sweep              V in {32768, 65536, 151936} x B in {1, 4, 8}, f32,
                     N(0, 3^2) with 1% of entries at -inf, T ~ U[0.5, 1.5],
                     seeds from splitmix64(7), offset = decode step.
  throughput         V=151936, B in {64, 128, 256}, bf16, N(0, 4^2) plus +6 on
                     32 distinct Zipf(1.1)-ranked token ids per row, T = 1.0.
  hlg                B=8, V=262144, f32, N(0, 3^2) with 0.5% at -inf; curve
                     m=1.3, w=2.0, beta_t=1.0, beta_h=1.5, pivot offset c=6.0.
  mixed_greedy       B=512, V=151936, bf16, N(0, 3^2) with 1% at -inf; even rows
                     T=0 (greedy), odd rows T ~ U[0.3, 2.0]; exact ties of the
                     row maximum planted on rows 0..7.

16-bit inputs are returned as uint16 bit patterns (round-to-nearest-even from
float32), which is how both the oracle and the CUDA library read them.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32, BF16, F16 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", BF16: "bf16", F16: "f16"}

VOCAB_SWEEP = (32768, 65536, 151936)
BATCH_SWEEP = (1, 4, 8)
THROUGHPUT_V = 151936
THROUGHPUT_B = (64, 128, 256)
HLG_PARAMS = dict(m=1.3, w=2.0, beta_t=1.0, beta_h=1.5, c=6.0)

_MASK64 = (1 << 64) - 1


def splitmix64(state: int, n: int) -> np.ndarray:
    """First n outputs of SplitMix64 (Steele, Lea and Flood, "Fast splittable
    pseudorandom number generators", OOPSLA 2014) started at `state`; used to
    derive per-row sampler seeds."""
    out = np.zeros(n, dtype=np.uint64)
    s = state & _MASK64
    for k in range(n):
        s = (s + 0x9E3779B97F4A7C15) & _MASK64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        out[k] = z ^ (z >> 31)
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (NaN kept NaN)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.uint64)
    rounded = ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        rounded[nan] = ((bits[nan] >> 16) | 0x40).astype(np.uint16)
    return rounded


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def encode(x: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == BF16:
        return to_bf16_bits(x)
    if dtype == F16:
        return to_f16_bits(x)
    raise ValueError(dtype)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def roundtrip(x: np.ndarray, dtype: int) -> np.ndarray:
    """float32 values rounded to `dtype` and widened back to float32."""
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == BF16:
        return bf16_bits_to_f32(to_bf16_bits(x))
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).astype(np.float32)


@dataclass
class Batch:
    """One batch of sampler inputs. `logits` is float32 [B, V] or uint16 bit
    patterns [B, V]; `dtype` says which."""
    name: str
    logits: np.ndarray
    dtype: int
    temperature: np.ndarray  # float32 [B]
    seed: np.ndarray  # uint64 [B]
    offset: np.ndarray  # uint64 [B]
    hlg: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return self.logits.shape[0]

    @property
    def V(self) -> int:
        return self.logits.shape[1]

    def at_step(self, step: int) -> "Batch":
        """The same batch at decode step `step` (offset = step for every row)."""
        return Batch(self.name, self.logits, self.dtype, self.temperature, self.seed,
                     np.full(self.B, step, dtype=np.uint64), self.hlg)


def _normal_logits(rng, B, V, sigma, inf_frac):
    x = rng.standard_normal((B, V), dtype=np.float32) * np.float32(sigma)
    if inf_frac > 0:
        x[rng.random((B, V), dtype=np.float32) < inf_frac] = -np.inf
    return x


def tiny_statistical() -> Batch:
    rng = np.random.default_rng(1234)
    B, V = 4, 64
    x = np.zeros((B, V), dtype=np.float32)
    x[0] = rng.standard_normal(V)
    x[0, rng.integers(V)] = 8.0
    x[1] = 0.0
    x[2] = rng.standard_normal(V)
    x[2, rng.choice(V, 2, replace=False)] = 4.0
    x[3] = 2.0 * rng.standard_normal(V)
    x[3, rng.choice(V, 16, replace=False)] = -np.inf
    return Batch("tiny_statistical", x, F32, np.ones(B, dtype=np.float32),
                 np.full(B, 1234, dtype=np.uint64), np.zeros(B, dtype=np.uint64))


def sweep(V: int, B: int, seed: int = 2) -> Batch:
    rng = np.random.default_rng([seed, V, B])
    x = _normal_logits(rng, B, V, 3.0, 0.01)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    return Batch("sweep_V%d_B%d" % (V, B), x, F32, T, splitmix64(7, B),
                 np.zeros(B, dtype=np.uint64))


def zipf_ids(rng, V: int, count: int, s: float = 1.1) -> np.ndarray:
    """`count` distinct token ids drawn by Zipf(s) rank over ranks 1..V
    (id = rank - 1), duplicates and out-of-range ranks rejected."""
    ids: list[int] = []
    seen = set()
    while len(ids) < count:
        r = int(rng.zipf(s))
        if r > V or r in seen:
            continue
        seen.add(r)
        ids.append(r - 1)
    return np.array(ids, dtype=np.int64)


def throughput(B: int, V: int = THROUGHPUT_V, dtype: int = BF16, seed: int = 3) -> Batch:
    rng = np.random.default_rng([seed, V, B])
    x = _normal_logits(rng, B, V, 4.0, 0.0)
    for b in range(B):
        x[b, zipf_ids(rng, V, 32)] += 6.0
    return Batch("throughput_V%d_B%d" % (V, B), encode(x, dtype), dtype,
                 np.ones(B, dtype=np.float32), splitmix64(7, B), np.zeros(B, dtype=np.uint64))


def hlg(B: int = 8, V: int = 262144, seed: int = 4) -> Batch:
    rng = np.random.default_rng([seed, V, B])
    x = _normal_logits(rng, B, V, 3.0, 0.005)
    return Batch("hlg_V%d_B%d" % (V, B), x, F32, np.ones(B, dtype=np.float32),
                 splitmix64(7, B), np.zeros(B, dtype=np.uint64), dict(HLG_PARAMS))


def plant_ties(rng, x: np.ndarray, rows) -> None:
    """Copy each listed row's maximum to three more positions: one below the
    original argmax (so the lowest-index rule decides), its neighbour, and one
    half a row away (a different slice of the row)."""
    V = x.shape[1]
    for b in rows:
        p = int(np.argmax(x[b]))
        v = x[b, p]
        targets = {(p + 1) % V, (p + V // 2) % V}
        if p > 0:
            targets.add(int(rng.integers(0, p)))
        for t in targets:
            x[b, t] = v


def mixed_greedy(B: int = 512, V: int = THROUGHPUT_V, dtype: int = BF16, seed: int = 5,
                 tie_rows: int = 8) -> Batch:
    rng = np.random.default_rng([seed, V, B])
    x = _normal_logits(rng, B, V, 3.0, 0.01)
    x = roundtrip(x, dtype)  # plant ties on the values the kernel will see
    plant_ties(rng, x, range(min(tie_rows, B)))
    T = rng.uniform(0.3, 2.0, B).astype(np.float32)
    T[0::2] = 0.0
    return Batch("mixed_greedy_V%d_B%d" % (V, B), encode(x, dtype), dtype, T, splitmix64(7, B),
                 np.zeros(B, dtype=np.uint64))
