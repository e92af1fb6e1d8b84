"""gsample: batch Gumbel-max / HLG token sampling on GB300 (sm_103a).

Thin ctypes binding over the C ABI of ``libgsample.so`` (declared in
``include/gsample.h``). Every step of the sampling runs in the library's CUDA
kernels; this module only checks tensors, passes device pointers and the
current CUDA stream, and turns status codes into exceptions. PyTorch supplies
device memory and streams.

    import torch, token_sampling_logits_gb300 as gs
    idx = gs.gumbel_argmax(logits, temperature, seed, offset)   # int64 [B]

All calls are asynchronous on ``torch.cuda.current_stream()``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

from . import build as _build

__all__ = [
    "GSampleError", "HlgParams", "PIVOT_TOP", "PIVOT_ENTROPY", "F32", "BF16", "F16",
    "lib", "library_path", "workspace_bytes", "workspace_init", "new_workspace", "argmax",
    "gumbel_argmax", "hlg_gumbel_argmax", "hlg_gumbel_argmax_rows", "hlg_rows_tensor",
    "categorical", "filtered_gumbel_argmax", "status_string",
]

F32, BF16, F16 = 0, 1, 2
PIVOT_TOP, PIVOT_ENTROPY = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA = 0, 1, 2, 3, 4

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_u32 = ctypes.c_uint32
_u64 = ctypes.c_uint64
_vp = ctypes.c_void_p
_int = ctypes.c_int


class _HlgParamsC(ctypes.Structure):
    _fields_ = [("m", ctypes.c_float), ("w", ctypes.c_float), ("beta_t", ctypes.c_float),
                ("beta_h", ctypes.c_float), ("pivot_offset", ctypes.c_float),
                ("pivot_mode", ctypes.c_int32)]


@dataclass(frozen=True)
class HlgParams:
    """HLG tone-curve knobs in nats ("HLG sampling", "The transfer function"
    and "The pivot"). w = inf turns the rolloff off."""
    m: float = 1.0
    w: float = 4.0
    beta_t: float = 6.0
    beta_h: float = 4.0
    pivot_offset: float = 6.0
    pivot_mode: int = PIVOT_TOP

    def to_c(self) -> _HlgParamsC:
        return _HlgParamsC(self.m, self.w, self.beta_t, self.beta_h, self.pivot_offset,
                           self.pivot_mode)


class GSampleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__("%s failed: %s" % (what, status_string(status)))
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib() -> ctypes.CDLL:
    """Load libgsample.so (building it first if its sources are newer).
    Raises if the library cannot be built or loaded: there is no fallback."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.build() if _build.is_stale() else _build.LIB
        L = ctypes.CDLL(path)
        sigs = {
            "gsample_workspace_bytes": (ctypes.c_size_t, [_i64]),
            "gsample_workspace_init": (_int, [_vp, _i64, _vp]),
            "gsample_argmax": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp]),
            "gsample_gumbel_argmax": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp,
                                             _vp]),
            "gsample_hlg_gumbel_argmax": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                                 _vp, _vp, _vp]),
            "gsample_hlg_gumbel_argmax_rows": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp,
                                                      _vp, _vp, _vp, _vp]),
            "gsample_categorical": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
            "gsample_debug_categorical_ex": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp,
                                                    _vp, _i32, _vp]),
            "gsample_debug_sample_cluster": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp,
                                                    _vp, _vp, _i32, _vp]),
            "gsample_status_string": (ctypes.c_char_p, [_int]),
            "gsample_debug_philox": (_int, [_u64, _u32, _u64, _i64, _i64, _vp, _vp]),
            "gsample_debug_gumbel": (_int, [_vp, _i64, _vp, _vp, _vp]),
            "gsample_debug_word_test": (_int, [_vp, _vp, _i64, ctypes.c_float, ctypes.c_float, _vp,
                                               _vp, _vp]),
            "gsample_debug_sample_ex": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                               _vp, _vp, _i32, _vp]),
            "gsample_debug_planned_ctas": (_i32, [_int, _i64, _i64, _i64, _vp, _i32]),
            "gsample_debug_philox_rate": (_int, [_i32, _u32, _vp, _vp]),
            "gsample_debug_philox_alu_mix": (_int, [_i32, _u32, _i32, _i32, _vp, _vp]),
            "gsample_debug_blocks_computed": (_int, [_vp, _i32]),
            "gsample_debug_hlg_score": (_int, [_vp, _vp, _i64, _vp, ctypes.c_float, ctypes.c_float,
                                               _vp, _vp]),
            "gsample_gumbel_argmax_static": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp,
                                                    _vp, _vp]),
            "gsample_gumbel_argmax_host": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp,
                                                  _vp, _vp, _vp]),
            "gsample_filtered_gumbel_argmax": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp,
                                                      _vp, _vp, _vp, _vp, _vp]),
            "gsample_debug_filtered_ex": (_int, [_vp, _int, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                                 _vp, _vp, _vp, _i32, _vp]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
        return L


def status_string(status: int) -> str:
    return lib().gsample_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise GSampleError(status, what)


# --------------------------------------------------------------------------
# torch marshalling
# --------------------------------------------------------------------------
def _torch():
    import torch

    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    m = {torch.float32: F32, torch.bfloat16: BF16, torch.float16: F16}
    if t.dtype not in m:
        raise TypeError("logits must be float32, bfloat16 or float16, got %s" % t.dtype)
    return m[t.dtype]


def _stream_ptr(device) -> int:
    torch = _torch()
    return torch.cuda.current_stream(device).cuda_stream


def _logits_args(logits):
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    if logits.dim() != 2:
        raise ValueError("logits must be 2-D [B, V]")
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous (stride(1) == 1)")
    B, V = logits.shape
    ld = logits.stride(0) if B > 1 else V
    return _dtype_code(logits), B, V, ld


def _row_tensor(x, B, dtype, device, name):
    torch = _torch()
    if not torch.is_tensor(x):
        x = torch.full((B,), x, dtype=dtype, device=device)
    if x.dtype != dtype or x.device != device or x.shape != (B,) or not x.is_contiguous():
        raise ValueError("%s must be a contiguous %s tensor of shape [%d] on %s" %
                         (name, dtype, B, device))
    return x


def workspace_bytes(B: int) -> int:
    return int(lib().gsample_workspace_bytes(B))


def new_workspace(B: int, device=None):
    """A zeroed workspace for up to B rows (uint8 tensor, 16-byte aligned)."""
    torch = _torch()
    n = max(16, workspace_bytes(B))
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def workspace_init(ws, B: int) -> None:
    _check(lib().gsample_workspace_init(ws.data_ptr(), B, _stream_ptr(ws.device)),
           "gsample_workspace_init")


def _prepare(logits, out, workspace, need_ws: bool = True):
    torch = _torch()
    dt, B, V, ld = _logits_args(logits)
    dev = logits.device
    if out is None:
        out = torch.empty(B, dtype=torch.int64, device=dev)
    elif out.dtype != torch.int64 or out.device != dev or out.shape != (B,) or not out.is_contiguous():
        raise ValueError("out must be a contiguous int64 tensor of shape [B] on the logits' device")
    if not need_ws:
        return dt, B, V, ld, out, None
    if workspace is None:
        workspace = new_workspace(B, dev)
    elif workspace.device != dev or workspace.numel() * workspace.element_size() < workspace_bytes(B):
        raise ValueError("workspace too small or on another device")
    return dt, B, V, ld, out, workspace


def argmax(logits, out=None, workspace=None):
    """Greedy argmax per row (lowest index on ties; -1 for an all-masked row)."""
    dt, B, V, ld, out, ws = _prepare(logits, out, workspace)
    _check(lib().gsample_argmax(logits.data_ptr(), dt, B, V, ld, out.data_ptr(), ws.data_ptr(),
                                _stream_ptr(logits.device)), "gsample_argmax")
    return out


def gumbel_argmax(logits, temperature, seed, offset, out=None, workspace=None, ctas: int = 0,
                  cluster: int = 0):
    """Gumbel-max sample per row: argmax_i(logits[i]/T + g_i). temperature
    (float32), seed (uint64 as int64 bits) and offset (uint64 as int64 bits)
    are per-row tensors or scalars. Rows with T <= 0 are greedy. Diagnostics:
    ctas > 0 forces the flat split with that many CTAs; cluster > 0 forces the
    cluster-per-row kernel with that many CTAs per row."""
    torch = _torch()
    dt, B, V, ld, out, ws = _prepare(logits, out, workspace)
    dev = logits.device
    T = _row_tensor(temperature, B, torch.float32, dev, "temperature")
    S = _row_tensor(seed, B, torch.int64, dev, "seed")
    O = _row_tensor(offset, B, torch.int64, dev, "offset")
    L = lib()
    if cluster:
        st = L.gsample_debug_sample_cluster(logits.data_ptr(), dt, B, V, ld, T.data_ptr(),
                                            S.data_ptr(), O.data_ptr(), out.data_ptr(),
                                            ws.data_ptr(), cluster, _stream_ptr(dev))
    elif ctas:
        st = L.gsample_debug_sample_ex(logits.data_ptr(), dt, B, V, ld, T.data_ptr(), S.data_ptr(),
                                       O.data_ptr(), None, out.data_ptr(), ws.data_ptr(), ctas,
                                       _stream_ptr(dev))
    else:
        st = L.gsample_gumbel_argmax(logits.data_ptr(), dt, B, V, ld, T.data_ptr(), S.data_ptr(),
                                     O.data_ptr(), out.data_ptr(), ws.data_ptr(), _stream_ptr(dev))
    _check(st, "gsample_gumbel_argmax")
    return out


def filtered_gumbel_argmax(logits, temperature, seed, offset, top_k=None, top_p=None, out=None,
                           workspace=None, cluster: int = 0):
    """Top-k / top-p Gumbel-max sample per row (gsample_filtered_gumbel_argmax):
    the Gumbel-max over the row's filter set K (the top_k largest logits and/or
    the smallest prefix whose softmax mass reaches top_p). top_k (int32) and
    top_p (float32) are per-row tensors, scalars, or None (filter off).
    Diagnostics: cluster > 0 forces that many filter CTAs per row."""
    torch = _torch()
    dt, B, V, ld, out, ws = _prepare(logits, out, workspace)
    dev = logits.device
    T = _row_tensor(temperature, B, torch.float32, dev, "temperature")
    S = _row_tensor(seed, B, torch.int64, dev, "seed")
    O = _row_tensor(offset, B, torch.int64, dev, "offset")
    K = None if top_k is None else _row_tensor(top_k, B, torch.int32, dev, "top_k")
    P = None if top_p is None else _row_tensor(top_p, B, torch.float32, dev, "top_p")
    args = (logits.data_ptr(), dt, B, V, ld, T.data_ptr(), S.data_ptr(), O.data_ptr(),
            None if K is None else K.data_ptr(), None if P is None else P.data_ptr(),
            out.data_ptr(), ws.data_ptr())
    if cluster:
        st = lib().gsample_debug_filtered_ex(*args, cluster, _stream_ptr(dev))
    else:
        st = lib().gsample_filtered_gumbel_argmax(*args, _stream_ptr(dev))
    _check(st, "gsample_filtered_gumbel_argmax")
    return out


def _pinned_row(x, B, dtype, name):
    torch = _torch()
    if not torch.is_tensor(x):
        x = torch.full((B,), x, dtype=dtype).pin_memory()
    if x.dtype != dtype or x.is_cuda or x.shape != (B,) or not x.is_contiguous() or \
            not x.is_pinned():
        raise ValueError("%s must be a contiguous pinned %s host tensor of shape [%d]" %
                         (name, dtype, B))
    return x


def gumbel_argmax_host(logits, temperature, seed, offset, out=None, workspace=None,
                       sync: bool = True):
    """gumbel_argmax on pinned HOST tensors: the kernel reads the logits and the
    per-row arrays over the CPU-GPU link and writes the indices straight into
    `out` (a pinned int64 host tensor), with no device copy of the logits. The
    workspace is a device tensor. With sync=False the call only enqueues on the
    current CUDA stream, and `out` is ready once that stream is synchronised."""
    torch = _torch()
    if logits.is_cuda or not logits.is_pinned():
        raise ValueError("logits must be a pinned host tensor")
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be 2-D [B, V] with contiguous rows")
    dt = _dtype_code(logits)
    B, V = logits.shape
    ld = logits.stride(0) if B > 1 else V
    T = _pinned_row(temperature, B, torch.float32, "temperature")
    S = _pinned_row(seed, B, torch.int64, "seed")
    O = _pinned_row(offset, B, torch.int64, "offset")
    if out is None:
        out = torch.empty(B, dtype=torch.int64).pin_memory()
    else:
        _pinned_row(out, B, torch.int64, "out")
    dev = torch.device("cuda", torch.cuda.current_device())
    if workspace is None:
        workspace = new_workspace(B, dev)
    elif not workspace.is_cuda or workspace.numel() * workspace.element_size() < workspace_bytes(B):
        raise ValueError("workspace must be a device tensor of at least workspace_bytes(B) bytes")
    stream = torch.cuda.current_stream(dev)
    _check(lib().gsample_gumbel_argmax_host(logits.data_ptr(), dt, B, V, ld, T.data_ptr(),
                                            S.data_ptr(), O.data_ptr(), out.data_ptr(),
                                            workspace.data_ptr(), stream.cuda_stream),
           "gsample_gumbel_argmax_host")
    if sync:
        stream.synchronize()
    return out


def hlg_gumbel_argmax(logits, temperature, seed, offset, hlg: HlgParams, out=None,
                      workspace=None, cluster: int = 0):
    """HLG tone curve on the row's log-probs, then Gumbel-max."""
    torch = _torch()
    dt, B, V, ld, out, ws = _prepare(logits, out, workspace)
    dev = logits.device
    T = _row_tensor(temperature, B, torch.float32, dev, "temperature")
    S = _row_tensor(seed, B, torch.int64, dev, "seed")
    O = _row_tensor(offset, B, torch.int64, dev, "offset")
    hp = hlg.to_c()
    L = lib()
    if cluster:
        st = L.gsample_debug_sample_ex(logits.data_ptr(), dt, B, V, ld, T.data_ptr(), S.data_ptr(),
                                       O.data_ptr(), ctypes.byref(hp), out.data_ptr(),
                                       ws.data_ptr(), cluster, _stream_ptr(dev))
    else:
        st = L.gsample_hlg_gumbel_argmax(logits.data_ptr(), dt, B, V, ld, T.data_ptr(),
                                         S.data_ptr(), O.data_ptr(), ctypes.byref(hp),
                                         out.data_ptr(), ws.data_ptr(), _stream_ptr(dev))
    _check(st, "gsample_hlg_gumbel_argmax")
    return out


def categorical(logits, temperature, seed, offset, out=None, cluster: int = 0):
    """The categorical baseline: softmax(logits / T) drawn by the inverse CDF of
    element 0's uniform. cluster: CTAs per row (0 = the library's choice)."""
    torch = _torch()
    dt, B, V, ld, out, _ = _prepare(logits, out, None, need_ws=False)
    dev = logits.device
    T = _row_tensor(temperature, B, torch.float32, dev, "temperature")
    S = _row_tensor(seed, B, torch.int64, dev, "seed")
    O = _row_tensor(offset, B, torch.int64, dev, "offset")
    L = lib()
    if cluster:
        st = L.gsample_debug_categorical_ex(logits.data_ptr(), dt, B, V, ld, T.data_ptr(),
                                            S.data_ptr(), O.data_ptr(), out.data_ptr(), cluster,
                                            _stream_ptr(dev))
    else:
        st = L.gsample_categorical(logits.data_ptr(), dt, B, V, ld, T.data_ptr(), S.data_ptr(),
                                   O.data_ptr(), out.data_ptr(), _stream_ptr(dev))
    _check(st, "gsample_categorical")
    return out


def hlg_rows_tensor(params, device):
    """Per-row curves as the device array gsample_hlg_gumbel_argmax_rows reads:
    B records of 24 bytes (five float32 fields, then the int32 pivot mode)."""
    import numpy as np

    torch = _torch()
    rec = np.dtype([("m", "<f4"), ("w", "<f4"), ("beta_t", "<f4"), ("beta_h", "<f4"),
                    ("pivot_offset", "<f4"), ("pivot_mode", "<i4")])
    a = np.zeros(len(params), dtype=rec)
    for i, h in enumerate(params):
        a[i] = (h.m, h.w, h.beta_t, h.beta_h, h.pivot_offset, h.pivot_mode)
    return torch.from_numpy(a.view(np.uint8).copy()).to(device)


def hlg_gumbel_argmax_rows(logits, temperature, seed, offset, params, out=None, workspace=None):
    """HLG + Gumbel-max with one curve per row. `params`: a list of B HlgParams,
    or a uint8 device tensor from hlg_rows_tensor."""
    torch = _torch()
    dt, B, V, ld, out, ws = _prepare(logits, out, workspace)
    dev = logits.device
    T = _row_tensor(temperature, B, torch.float32, dev, "temperature")
    S = _row_tensor(seed, B, torch.int64, dev, "seed")
    O = _row_tensor(offset, B, torch.int64, dev, "offset")
    if not torch.is_tensor(params):
        params = hlg_rows_tensor(params, dev)
    if params.device != dev or params.dtype != torch.uint8 or params.numel() != 24 * B:
        raise ValueError("per-row HLG parameters: a uint8 tensor of 24*B bytes on the logits' device")
    st = lib().gsample_hlg_gumbel_argmax_rows(logits.data_ptr(), dt, B, V, ld, T.data_ptr(),
                                              S.data_ptr(), O.data_ptr(), params.data_ptr(),
                                              out.data_ptr(), ws.data_ptr(), _stream_ptr(dev))
    _check(st, "gsample_hlg_gumbel_argmax_rows")
    return out


def seeds_as_tensor(seeds, device):
    """uint64 seeds (numpy or ints) as an int64 tensor holding the same bits."""
    import numpy as np

    torch = _torch()
    a = np.ascontiguousarray(np.asarray(seeds, dtype=np.uint64)).view(np.int64)
    return torch.from_numpy(a.copy()).to(device)


def debug_philox(seed: int, row: int, offset: int, group0: int, n_groups: int, device=None):
    """Raw Philox4x32-10 blocks of the kernels' stream -> int32 tensor [n, 4]
    (bit patterns of uint32)."""
    torch = _torch()
    out = torch.empty((n_groups, 4), dtype=torch.int32, device=device or "cuda")
    _check(lib().gsample_debug_philox(seed, row, offset, group0, n_groups, out.data_ptr(),
                                      _stream_ptr(out.device)), "gsample_debug_philox")
    return out


def debug_gumbel(words, with_bound: bool = True):
    """The kernels' binary32 Gumbel transform (and pruning bound) of raw words
    (int32 tensor of uint32 bit patterns)."""
    torch = _torch()
    g = torch.empty(words.shape, dtype=torch.float32, device=words.device)
    bnd = torch.empty_like(g) if with_bound else None
    _check(lib().gsample_debug_gumbel(words.data_ptr(), words.numel(), g.data_ptr(),
                                      bnd.data_ptr() if bnd is not None else None,
                                      _stream_ptr(words.device)), "gsample_debug_gumbel")
    return g, bnd


def planned_ctas(dtype: int, B: int, V: int, ld: int | None = None, ptr: int = 0) -> int:
    return int(lib().gsample_debug_planned_ctas(dtype, B, V, ld or V, ptr or None, 0))
