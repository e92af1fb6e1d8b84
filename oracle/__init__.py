"""CPU oracle for the batch Gumbel-max / HLG sampler (test infrastructure).

A plain, slow, single-threaded C restatement (``oracle.c``) of what the sampler
computes, in double precision, with a thin ctypes/numpy wrapper. Only the test
suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg use it;
the CUDA library never does and shares no code with it.

Sources (page title, section):
  * "Softmax-free GPU sampling: Gumbel-max categorical sampling kernel"
    (lablup/mlxcel issue #900), Background and Task: score = logits/T + g,
    g = -log(-log u), argmax per row, counter-based Philox stream per
    (seed, row, element, offset), greedy argmax at temperature 0.
  * Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11),
    section 3: Philox4x32-10.
  * "HLG sampling -- a piecewise tone curve on the logits" (mlx-bun
    docs/design/hlg-sampling.md), "The transfer function" and "The pivot".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F16 = 0, 1, 2
PIVOT_TOP, PIVOT_ENTROPY = 0, 1

_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64
_u32 = ctypes.c_uint32
_int = ctypes.c_int
_dbl = ctypes.c_double
_flt = ctypes.c_float
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with plain gcc (no fast-math, no FMA
    contraction, so x86 and Arm hosts give the same doubles)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        sig = {
            "oracle_philox4x32_10": (None, [_vp, _vp, _vp]),
            "oracle_stream_word": (_u32, [_u64, _u32, _u64, _u64]),
            "oracle_uniform": (_dbl, [_u32]),
            "oracle_gumbel": (_dbl, [_dbl]),
            "oracle_load": (_dbl, [_vp, _int, _i64]),
            "oracle_sample_row": (_i64, [_vp, _int, _i64, _flt, _u64, _u32, _u64, _vp, _vp]),
            "oracle_gumbel_argmax": (None, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
            "oracle_argmax": (None, [_vp, _int, _i64, _i64, _i64, _vp, _vp]),
            "oracle_gumbel_argmax_steps": (None, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _u64,
                                                  _i64, _vp, _vp]),
            "oracle_hlg_curve": (_dbl, [_dbl, _dbl, _dbl, _dbl, _dbl]),
            "oracle_hlg_pivot": (_int, [_vp, _int, _i64, _int, _dbl, _vp, _vp]),
            "oracle_hlg_transform_row": (_int, [_vp, _int, _i64, _dbl, _dbl, _dbl, _dbl, _dbl,
                                                _int, _vp, _vp, _vp]),
            "oracle_hlg_sample_row": (_i64, [_vp, _int, _i64, _flt, _u64, _u32, _u64, _dbl, _dbl,
                                             _dbl, _dbl, _dbl, _int, _vp, _vp]),
            "oracle_hlg_gumbel_argmax": (None, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                                _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
            "oracle_categorical_row": (_i64, [_vp, _int, _i64, _flt, _u64, _u32, _u64, _i64,
                                              _vp, _vp]),
            "oracle_categorical": (None, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp,
                                          _vp, _vp]),
            "oracle_filtered_sample_row": (_i64, [_vp, _int, _i64, _flt, _u64, _u32, _u64,
                                                  ctypes.c_int32, _flt, _vp, _vp]),
            "oracle_filtered_gumbel_argmax": (None, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp,
                                                     _vp, _vp, _vp, _vp, _vp]),
            "oracle_filtered_steps": (None, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _u64, _i64,
                                             _vp, _vp, _vp]),
            "oracle_philox_blocks": (None, [_u32, _u32, _vp, _i64, _vp]),
            "oracle_stream_words": (None, [_u64, _u32, _u64, _i64, _i64, _vp]),
            "oracle_gumbel_of_words": (None, [_vp, _i64, _vp]),
            "oracle_uniform_of_words": (None, [_vp, _i64, _vp]),
            "oracle_hlg_curve_many": (None, [_vp, _i64, _dbl, _dbl, _dbl, _dbl, _vp]),
            "oracle_decode": (None, [_vp, _int, _i64, _vp]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def _dtype_code(x: np.ndarray, dtype: int | None) -> int:
    if dtype is not None:
        return dtype
    if x.dtype == np.float32:
        return F32
    raise TypeError("pass dtype=BF16 or F16 for 16-bit inputs given as uint16 bit patterns")


def _logits_2d(x: np.ndarray):
    """Return (array, B, V, ld) for a 2-D row-major array whose rows may be
    strided (ld >= V elements)."""
    if x.ndim != 2:
        raise ValueError("logits must be 2-D [B, V]")
    if x.strides[1] != x.itemsize:
        raise ValueError("logits rows must be contiguous")
    if x.strides[0] % x.itemsize:
        raise ValueError("row stride must be a whole number of elements")
    return x, x.shape[0], x.shape[1], x.strides[0] // x.itemsize


def philox4x32_10(key, ctr):
    """One Philox4x32-10 block: key = (k0, k1), ctr = (c0, c1, c2, c3)."""
    lib = _load()
    k = np.asarray(key, dtype=np.uint32)
    c = np.asarray(ctr, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(_ptr(k), _ptr(c), _ptr(out))
    return out


def philox_blocks(key0: int, key1: int, ctrs: np.ndarray) -> np.ndarray:
    lib = _load()
    ctrs = np.ascontiguousarray(ctrs, dtype=np.uint32).reshape(-1, 4)
    out = np.zeros_like(ctrs)
    lib.oracle_philox_blocks(key0, key1, _ptr(ctrs), ctrs.shape[0], _ptr(out))
    return out


def stream_words(seed: int, row: int, offset: int, i0: int, n: int) -> np.ndarray:
    lib = _load()
    out = np.zeros(n, dtype=np.uint32)
    lib.oracle_stream_words(seed, row, offset, i0, n, _ptr(out))
    return out


def uniform_of_words(words: np.ndarray) -> np.ndarray:
    lib = _load()
    w = np.ascontiguousarray(words, dtype=np.uint32)
    out = np.zeros(w.shape, dtype=np.float64)
    lib.oracle_uniform_of_words(_ptr(w), w.size, _ptr(out))
    return out


def gumbel_of_words(words: np.ndarray) -> np.ndarray:
    lib = _load()
    w = np.ascontiguousarray(words, dtype=np.uint32)
    out = np.zeros(w.shape, dtype=np.float64)
    lib.oracle_gumbel_of_words(_ptr(w), w.size, _ptr(out))
    return out


def gumbel(u: float) -> float:
    return _load().oracle_gumbel(u)


def decode(x: np.ndarray, dtype: int) -> np.ndarray:
    lib = _load()
    x = np.ascontiguousarray(x)
    out = np.zeros(x.size, dtype=np.float64)
    lib.oracle_decode(_ptr(x), dtype, x.size, _ptr(out))
    return out.reshape(x.shape)


def argmax(logits: np.ndarray, dtype: int | None = None):
    """Greedy argmax per row -> (idx int64[B], gap float64[B])."""
    lib = _load()
    x, B, V, ld = _logits_2d(logits)
    dt = _dtype_code(x, dtype)
    idx = np.zeros(B, dtype=np.int64)
    gap = np.zeros(B, dtype=np.float64)
    lib.oracle_argmax(_ptr(x), dt, B, V, ld, _ptr(idx), _ptr(gap))
    return idx, gap


def sample_row(row: np.ndarray, temperature: float, seed: int, row_id: int, offset: int,
               dtype: int | None = None):
    """Gumbel-max sample of one row whose Philox row word is `row_id`.
    -> (idx, gap, best score)."""
    lib = _load()
    row = np.ascontiguousarray(row)
    dt = _dtype_code(row, dtype)
    gap = ctypes.c_double()
    best = ctypes.c_double()
    idx = lib.oracle_sample_row(_ptr(row), dt, row.size, temperature, seed, row_id, offset,
                                ctypes.byref(gap), ctypes.byref(best))
    return int(idx), gap.value, best.value


def hlg_sample_row(row: np.ndarray, temperature: float, seed: int, row_id: int, offset: int,
                   m: float, w: float, beta_t: float, beta_h: float, c: float,
                   pivot_mode: int = PIVOT_TOP, dtype: int | None = None):
    """HLG + Gumbel-max sample of one row. -> (idx, gap, best score)."""
    lib = _load()
    row = np.ascontiguousarray(row)
    dt = _dtype_code(row, dtype)
    gap = ctypes.c_double()
    best = ctypes.c_double()
    idx = lib.oracle_hlg_sample_row(_ptr(row), dt, row.size, temperature, seed, row_id, offset,
                                    m, w, beta_t, beta_h, c, pivot_mode, ctypes.byref(gap),
                                    ctypes.byref(best))
    return int(idx), gap.value, best.value


def categorical_row(row: np.ndarray, temperature: float, seed: int, row_id: int, offset: int,
                    probe: int = -1, dtype: int | None = None):
    """Inverse-CDF sample of softmax(row / T) with element 0's uniform.
    -> (idx, margin, probe_dist): margin and probe_dist relative to the row's sum."""
    lib = _load()
    row = np.ascontiguousarray(row)
    dt = _dtype_code(row, dtype)
    margin = ctypes.c_double()
    pd = ctypes.c_double()
    idx = lib.oracle_categorical_row(_ptr(row), dt, row.size, temperature, seed, row_id, offset,
                                     probe, ctypes.byref(pd), ctypes.byref(margin))
    return int(idx), margin.value, pd.value


def categorical(logits: np.ndarray, temperature, seed, offset, probe=None,
                dtype: int | None = None):
    """Categorical (inverse-CDF) sample per row. probe: optional int64[B] of
    indices to locate against the exact CDF. -> (idx, margin, probe_dist)."""
    lib = _load()
    x, B, V, ld = _logits_2d(logits)
    dt = _dtype_code(x, dtype)
    T, S, O = _row_arrays(B, temperature, seed, offset)
    pr = None if probe is None else np.ascontiguousarray(np.asarray(probe, dtype=np.int64))
    idx = np.zeros(B, dtype=np.int64)
    margin = np.zeros(B, dtype=np.float64)
    pd = np.zeros(B, dtype=np.float64)
    lib.oracle_categorical(_ptr(x), dt, B, V, ld, _ptr(T), _ptr(S), _ptr(O), _ptr(pr), _ptr(idx),
                           _ptr(margin), _ptr(pd))
    return idx, margin, pd


def _row_arrays(B, temperature, seed, offset):
    T = np.ascontiguousarray(np.broadcast_to(np.asarray(temperature, dtype=np.float32), (B,)))
    S = np.ascontiguousarray(np.broadcast_to(np.asarray(seed, dtype=np.uint64), (B,)))
    O = np.ascontiguousarray(np.broadcast_to(np.asarray(offset, dtype=np.uint64), (B,)))
    return T, S, O


def gumbel_argmax(logits: np.ndarray, temperature, seed, offset, dtype: int | None = None):
    """Gumbel-max sample per row -> (idx int64[B], top-2 score gap float64[B])."""
    lib = _load()
    x, B, V, ld = _logits_2d(logits)
    dt = _dtype_code(x, dtype)
    T, S, O = _row_arrays(B, temperature, seed, offset)
    idx = np.zeros(B, dtype=np.int64)
    gap = np.zeros(B, dtype=np.float64)
    lib.oracle_gumbel_argmax(_ptr(x), dt, B, V, ld, _ptr(T), _ptr(S), _ptr(O), _ptr(idx),
                             _ptr(gap))
    return idx, gap


def gumbel_argmax_steps(logits: np.ndarray, temperature, seed, base_offset: int, steps: int,
                        dtype: int | None = None, want_gap: bool = False):
    """steps consecutive decode steps (offset = base_offset + k for every row).
    Returns idx int64[steps, B] (and gap float64[steps, B] if want_gap)."""
    lib = _load()
    x, B, V, ld = _logits_2d(logits)
    dt = _dtype_code(x, dtype)
    T = np.ascontiguousarray(np.broadcast_to(np.asarray(temperature, dtype=np.float32), (B,)))
    S = np.ascontiguousarray(np.broadcast_to(np.asarray(seed, dtype=np.uint64), (B,)))
    idx = np.zeros((steps, B), dtype=np.int64)
    gap = np.zeros((steps, B), dtype=np.float64) if want_gap else None
    lib.oracle_gumbel_argmax_steps(_ptr(x), dt, B, V, ld, _ptr(T), _ptr(S), base_offset, steps,
                                   _ptr(idx), _ptr(gap))
    return (idx, gap) if want_gap else idx


def hlg_curve(z, m: float, w: float, beta_t: float, beta_h: float) -> np.ndarray:
    lib = _load()
    z = np.ascontiguousarray(np.atleast_1d(np.asarray(z, dtype=np.float64)))
    out = np.zeros_like(z)
    lib.oracle_hlg_curve_many(_ptr(z), z.size, m, w, beta_t, beta_h, _ptr(out))
    return out


def hlg_pivot(row: np.ndarray, c: float, pivot_mode: int = PIVOT_TOP, dtype: int | None = None):
    """(lse, mu) of one row; None if the row has no finite logit."""
    lib = _load()
    row = np.ascontiguousarray(row)
    dt = _dtype_code(row, dtype)
    lse = ctypes.c_double()
    mu = ctypes.c_double()
    rc = lib.oracle_hlg_pivot(_ptr(row), dt, row.size, pivot_mode, c, ctypes.byref(lse),
                              ctypes.byref(mu))
    return None if rc else (lse.value, mu.value)


def hlg_transform_row(row: np.ndarray, m, w, beta_t, beta_h, c, pivot_mode=PIVOT_TOP,
                      dtype: int | None = None):
    """Tone-mapped log-probs g(l - mu) of one row (float64[V]); None if the row
    has no finite logit."""
    lib = _load()
    row = np.ascontiguousarray(row)
    dt = _dtype_code(row, dtype)
    out = np.zeros(row.size, dtype=np.float64)
    rc = lib.oracle_hlg_transform_row(_ptr(row), dt, row.size, m, w, beta_t, beta_h, c,
                                      pivot_mode, _ptr(out), None, None)
    return None if rc else out


def hlg_gumbel_argmax(logits: np.ndarray, temperature, seed, offset, m, w, beta_t, beta_h, c,
                      pivot_mode=PIVOT_TOP, dtype: int | None = None):
    """HLG tone curve + Gumbel-max per row; curve parameters are scalars or
    per-row arrays. -> (idx int64[B], gap float64[B])."""
    lib = _load()
    x, B, V, ld = _logits_2d(logits)
    dt = _dtype_code(x, dtype)
    T, S, O = _row_arrays(B, temperature, seed, offset)

    def per_row(v, dtype=np.float64):
        return np.ascontiguousarray(np.broadcast_to(np.asarray(v, dtype=dtype), (B,)))

    pm, pw, pbt, pbh, pc = (per_row(v) for v in (m, w, beta_t, beta_h, c))
    pmode = per_row(pivot_mode, np.int32)
    idx = np.zeros(B, dtype=np.int64)
    gap = np.zeros(B, dtype=np.float64)
    lib.oracle_hlg_gumbel_argmax(_ptr(x), dt, B, V, ld, _ptr(T), _ptr(S), _ptr(O), _ptr(pm),
                                 _ptr(pw), _ptr(pbt), _ptr(pbh), _ptr(pc), _ptr(pmode), _ptr(idx),
                                 _ptr(gap))
    return idx, gap


def filtered_sample_row(row: np.ndarray, temperature: float, seed: int, row_id: int,
                        offset: int, top_k: int = 0, top_p: float = 1.0,
                        dtype: int | None = None):
    """Top-k / top-p Gumbel-max sample of one row (see oracle.c, [FILTER]).
    -> (idx, gap within the filter set, nucleus edge margin)."""
    lib = _load()
    row = np.ascontiguousarray(row)
    dt = _dtype_code(row, dtype)
    gap = ctypes.c_double()
    edge = ctypes.c_double()
    idx = lib.oracle_filtered_sample_row(_ptr(row), dt, row.size, temperature, seed, row_id,
                                         offset, int(top_k), float(top_p), ctypes.byref(gap),
                                         ctypes.byref(edge))
    return int(idx), gap.value, edge.value


def filtered_gumbel_argmax(logits: np.ndarray, temperature, seed, offset, top_k=0, top_p=1.0,
                           dtype: int | None = None):
    """Per-row top-k / top-p Gumbel-max. -> (idx int64[B], gap float64[B], edge float64[B])."""
    lib = _load()
    x, B, V, ld = _logits_2d(logits)
    dt = _dtype_code(x, dtype)
    T, S, O = _row_arrays(B, temperature, seed, offset)
    K = np.ascontiguousarray(np.broadcast_to(np.asarray(top_k, dtype=np.int32), (B,)))
    P = np.ascontiguousarray(np.broadcast_to(np.asarray(top_p, dtype=np.float32), (B,)))
    idx = np.zeros(B, dtype=np.int64)
    gap = np.zeros(B, dtype=np.float64)
    edge = np.zeros(B, dtype=np.float64)
    lib.oracle_filtered_gumbel_argmax(_ptr(x), dt, B, V, ld, _ptr(T), _ptr(S), _ptr(O), _ptr(K),
                                      _ptr(P), _ptr(idx), _ptr(gap), _ptr(edge))
    return idx, gap, edge


def filtered_steps(logits: np.ndarray, temperature, seed, base_offset: int, steps: int,
                   top_k=0, top_p=1.0, dtype: int | None = None):
    """steps decode steps of a filtered batch -> idx int64[steps, B]."""
    lib = _load()
    x, B, V, ld = _logits_2d(logits)
    dt = _dtype_code(x, dtype)
    T = np.ascontiguousarray(np.broadcast_to(np.asarray(temperature, dtype=np.float32), (B,)))
    S = np.ascontiguousarray(np.broadcast_to(np.asarray(seed, dtype=np.uint64), (B,)))
    K = np.ascontiguousarray(np.broadcast_to(np.asarray(top_k, dtype=np.int32), (B,)))
    P = np.ascontiguousarray(np.broadcast_to(np.asarray(top_p, dtype=np.float32), (B,)))
    idx = np.zeros((steps, B), dtype=np.int64)
    lib.oracle_filtered_steps(_ptr(x), dt, B, V, ld, _ptr(T), _ptr(S), base_offset, steps,
                              _ptr(K), _ptr(P), _ptr(idx))
    return idx
