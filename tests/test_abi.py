"""Host-side checks of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every function declared in include/*.h, and rejects
bad arguments with the documented status before touching the device."""
import ctypes
import glob
import os
import re

import pytest

import token_sampling_logits_gb300 as gs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"\b(gsample_[a-z0-9_]+)\s*\(", src):
            names.add(m.group(1))
    return sorted(names)


def test_library_exports_every_declared_function():
    L = gs.lib()
    names = _declared_functions()
    assert {"gsample_argmax", "gsample_gumbel_argmax", "gsample_hlg_gumbel_argmax",
            "gsample_workspace_bytes", "gsample_status_string"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_library_is_built_for_sm103a():
    # cuobjdump is not used: the build flags name the one target
    from token_sampling_logits_gb300 import build

    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(gs.library_path())


def test_workspace_size_and_status_strings():
    assert gs.workspace_bytes(0) == 0
    assert gs.workspace_bytes(1) == 16
    assert gs.workspace_bytes(512) == 16 * 512
    seen = {gs.status_string(s) for s in range(5)}
    assert len(seen) == 5 and all(s.startswith("GSAMPLE_") for s in seen)
    assert "UNKNOWN" in gs.status_string(99)


FAKE = 1 << 20  # 16-byte aligned fake device address; never dereferenced below


def _gumbel(**kw):
    a = dict(logits=FAKE, dtype=gs.F32, B=4, V=100, ld=100, T=FAKE, seed=FAKE, off=FAKE,
             out=FAKE, ws=FAKE)
    a.update(kw)
    return gs.lib().gsample_gumbel_argmax(a["logits"], a["dtype"], a["B"], a["V"], a["ld"], a["T"],
                                          a["seed"], a["off"], a["out"], a["ws"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(logits=None), gs.ERR_INVALID_ARG),
    (dict(out=None), gs.ERR_INVALID_ARG),
    (dict(ws=None), gs.ERR_INVALID_ARG),
    (dict(T=None), gs.ERR_INVALID_ARG),
    (dict(seed=None), gs.ERR_INVALID_ARG),
    (dict(off=None), gs.ERR_INVALID_ARG),
    (dict(dtype=7), gs.ERR_INVALID_ARG),
    (dict(B=-1), gs.ERR_INVALID_ARG),
    (dict(V=0), gs.ERR_INVALID_ARG),
    (dict(V=1 << 31), gs.ERR_INVALID_ARG),
    (dict(ld=99), gs.ERR_INVALID_ARG),
    (dict(B=1 << 31), gs.ERR_INVALID_ARG),
    (dict(logits=FAKE + 2), gs.ERR_INVALID_ARG),  # f32 logits must be 4-byte aligned
    (dict(out=FAKE + 4), gs.ERR_INVALID_ARG),
    (dict(ws=FAKE + 8), gs.ERR_WORKSPACE),
    (dict(B=0), gs.OK),  # empty batch: nothing to do, nothing launched
    (dict(B=0, logits=None, out=None, ws=None, T=None), gs.OK),
])
def test_invalid_arguments_rejected_on_host(kw, status):
    assert _gumbel(**kw) == status


def test_hlg_parameter_validation():
    L = gs.lib()

    def call(**kw):
        p = gs.HlgParams(**{**dict(m=1.3, w=2.0, beta_t=1.0, beta_h=1.5, pivot_offset=6.0), **kw})
        c = p.to_c()
        return L.gsample_hlg_gumbel_argmax(FAKE, gs.F32, 0, 100, 100, FAKE, FAKE, FAKE,
                                           ctypes.byref(c), FAKE, FAKE, None)

    assert call() == gs.OK  # B = 0 after a full parameter check
    for bad in (dict(m=0.0), dict(m=-1.0), dict(m=float("inf")), dict(w=-0.5),
                dict(w=float("nan")), dict(beta_t=0.0), dict(beta_h=float("inf")),
                dict(pivot_offset=float("nan")), dict(pivot_mode=5)):
        assert call(**bad) == gs.ERR_INVALID_ARG, bad
    assert call(w=float("inf")) == gs.OK  # rolloff off is allowed
    assert L.gsample_hlg_gumbel_argmax(FAKE, gs.F32, 0, 100, 100, FAKE, FAKE, FAKE, None, FAKE,
                                       FAKE, None) == gs.ERR_INVALID_ARG


def test_no_device_is_an_error_not_a_fallback():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # valid-looking arguments reach the device query, which must fail loudly
    assert _gumbel() == gs.ERR_CUDA
    assert gs.lib().gsample_argmax(FAKE, gs.BF16, 2, 64, 64, FAKE, FAKE, None) == gs.ERR_CUDA


def test_per_row_hlg_entry_validation():
    L = gs.lib()

    def call(B=4, rows=FAKE, out=FAKE, logits=FAKE):
        return L.gsample_hlg_gumbel_argmax_rows(logits, gs.F32, B, 100, 100, FAKE, FAKE, FAKE,
                                                rows, out, FAKE, None)

    assert call(B=0, rows=None) == gs.OK              # empty batch: nothing to do
    assert call(rows=None) == gs.ERR_INVALID_ARG       # B > 0 needs the per-row array
    assert call(rows=FAKE + 2) == gs.ERR_INVALID_ARG   # 24-byte records of 4-byte fields
    assert call(out=None) == gs.ERR_INVALID_ARG
    assert call(logits=None) == gs.ERR_INVALID_ARG


def test_categorical_entry_validation():
    L = gs.lib()

    def call(B=4, logits=FAKE, T=FAKE, out=FAKE):
        return L.gsample_categorical(logits, gs.F32, B, 100, 100, T, FAKE, FAKE, out, None)

    assert call(B=0) == gs.OK                      # empty batch: nothing to do
    assert call(logits=None) == gs.ERR_INVALID_ARG
    assert call(out=None) == gs.ERR_INVALID_ARG
    assert call(T=None) == gs.ERR_INVALID_ARG
    assert L.gsample_debug_categorical_ex(FAKE, gs.F32, 4, 100, 100, FAKE, FAKE, FAKE, FAKE, -1,
                                          None) == gs.ERR_INVALID_ARG
    assert L.gsample_debug_sample_cluster(FAKE, gs.F32, 4, 100, 100, FAKE, FAKE, FAKE, FAKE, FAKE,
                                          0, None) == gs.ERR_INVALID_ARG


def test_host_buffer_entry_validation():
    L = gs.lib()

    def call(B=4, logits=FAKE, T=FAKE, out=FAKE, ws=FAKE):
        return L.gsample_gumbel_argmax_host(logits, gs.F32, B, 100, 100, T, FAKE, FAKE, out, ws,
                                            None)

    assert call(B=0) == gs.OK                       # empty batch: nothing to do
    assert call(logits=None) == gs.ERR_INVALID_ARG
    assert call(T=None) == gs.ERR_INVALID_ARG
    assert call(out=FAKE + 4) == gs.ERR_INVALID_ARG
    assert call(ws=None) == gs.ERR_INVALID_ARG
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        # the pointer checks need the device: without one the call fails loudly
        assert call() == gs.ERR_CUDA


def test_host_buffer_binding_rejects_pageable_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros((2, 64), dtype=torch.float32)  # pageable host memory
    with pytest.raises(ValueError):
        gs.gumbel_argmax_host(x, 1.0, 0, 0)
    with pytest.raises(ValueError):
        gs.gumbel_argmax_host(torch.zeros(64), 1.0, 0, 0)  # not 2-D (and not pinned)


def test_word_test_debug_entry_validation():
    L = gs.lib()

    def call(n=4, x=FAKE, w=FAKE, T=1.0, thr=FAKE, flags=FAKE):
        return L.gsample_debug_word_test(x, w, n, 10.0, T, thr, flags, None)

    assert call(n=0) == gs.OK                      # nothing to do
    assert call(n=-1) == gs.ERR_INVALID_ARG
    assert call(T=0.0) == gs.ERR_INVALID_ARG       # the test is defined for T > 0
    assert call(T=float("nan")) == gs.ERR_INVALID_ARG
    assert call(x=None) == gs.ERR_INVALID_ARG
    assert call(flags=None) == gs.ERR_INVALID_ARG


def test_static_workspace_entry_validation():
    """gsample_gumbel_argmax_static checks every argument the regular entry point
    checks before it sets anything up or enqueues anything (no device is touched
    for a bad argument; on this CPU-only host a valid call fails at the device)."""
    L = gs.lib()

    def call(B=4, logits=FAKE, dtype=gs.F32, V=100, ld=100, T=FAKE, seed=FAKE, off=FAKE,
             out=FAKE):
        return L.gsample_gumbel_argmax_static(logits, dtype, B, V, ld, T, seed, off, out, None)

    assert call(B=0) == gs.OK
    assert call(B=-1) == gs.ERR_INVALID_ARG
    assert call(B=4097) == gs.ERR_INVALID_ARG         # past the static array
    assert call(logits=None) == gs.ERR_INVALID_ARG
    assert call(out=None) == gs.ERR_INVALID_ARG
    assert call(T=None) == gs.ERR_INVALID_ARG
    assert call(seed=None) == gs.ERR_INVALID_ARG
    assert call(off=None) == gs.ERR_INVALID_ARG
    assert call(V=0) == gs.ERR_INVALID_ARG
    assert call(ld=99) == gs.ERR_INVALID_ARG
    assert call(dtype=7) == gs.ERR_INVALID_ARG
    assert call(logits=FAKE + 2) == gs.ERR_INVALID_ARG  # f32 logits must be 4-byte aligned
    assert call(out=FAKE + 4) == gs.ERR_INVALID_ARG
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert call() == gs.ERR_CUDA


def test_philox_rate_and_block_counter_validation():
    L = gs.lib()
    assert L.gsample_debug_philox_rate(0, 10, FAKE, None) == gs.ERR_INVALID_ARG
    assert L.gsample_debug_philox_rate(33, 10, FAKE, None) == gs.ERR_INVALID_ARG
    assert L.gsample_debug_philox_rate(8, 0, FAKE, None) == gs.ERR_INVALID_ARG
    assert L.gsample_debug_philox_rate(8, 10, None, None) == gs.ERR_INVALID_ARG
    assert L.gsample_debug_blocks_computed(None, 0) == gs.ERR_INVALID_ARG
    # the regular build has no counter
    c = ctypes.c_uint64(7)
    assert L.gsample_debug_blocks_computed(ctypes.byref(c), 0) == gs.ERR_UNSUPPORTED
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert L.gsample_debug_philox_rate(8, 10, FAKE, None) == gs.ERR_CUDA


def test_philox_alu_mix_validation():
    L = gs.lib()
    f = L.gsample_debug_philox_alu_mix
    assert f(0, 10, 2, 1, FAKE, None) == gs.ERR_INVALID_ARG
    assert f(33, 10, 2, 1, FAKE, None) == gs.ERR_INVALID_ARG
    assert f(16, 0, 2, 1, FAKE, None) == gs.ERR_INVALID_ARG
    assert f(16, 10, 3, 1, FAKE, None) == gs.ERR_INVALID_ARG
    assert f(16, 10, 2, 2, FAKE, None) == gs.ERR_INVALID_ARG
    assert f(16, 10, 0, 0, FAKE, None) == gs.ERR_INVALID_ARG  # nothing to run
    assert f(16, 10, 2, 1, None, None) == gs.ERR_INVALID_ARG
    assert f(16, 10, 2, 1, FAKE + 2, None) == gs.ERR_INVALID_ARG
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert f(16, 10, 2, 1, FAKE, None) == gs.ERR_CUDA


def test_hlg_score_debug_validation():
    L = gs.lib()
    hp = gs.HlgParams().to_c()
    bad = gs.HlgParams(m=-1.0).to_c()
    st = None
    assert L.gsample_debug_hlg_score(FAKE, FAKE, 4, ctypes.byref(hp), 0.0, 1.0, FAKE, st) == \
        gs.ERR_INVALID_ARG                                             # T must be > 0
    assert L.gsample_debug_hlg_score(FAKE, FAKE, 4, ctypes.byref(hp), 1.0, float("inf"), FAKE,
                                     st) == gs.ERR_INVALID_ARG         # shift must be finite
    assert L.gsample_debug_hlg_score(FAKE, FAKE, 4, ctypes.byref(bad), 1.0, 1.0, FAKE, st) == \
        gs.ERR_INVALID_ARG
    assert L.gsample_debug_hlg_score(FAKE, FAKE, 4, None, 1.0, 1.0, FAKE, st) == gs.ERR_INVALID_ARG
    assert L.gsample_debug_hlg_score(None, FAKE, 4, ctypes.byref(hp), 1.0, 1.0, FAKE, st) == \
        gs.ERR_INVALID_ARG
    assert L.gsample_debug_hlg_score(FAKE, FAKE, 0, ctypes.byref(hp), 1.0, 1.0, FAKE, st) == gs.OK


def test_filtered_entry_validation():
    L = gs.lib()

    def call(B=4, logits=FAKE, T=FAKE, k=FAKE, p=FAKE, out=FAKE, ws=FAKE):
        return L.gsample_filtered_gumbel_argmax(logits, gs.F32, B, 100, 100, T, FAKE, FAKE, k, p,
                                                out, ws, None)

    assert call(B=0) == gs.OK
    assert call(logits=None) == gs.ERR_INVALID_ARG
    assert call(T=None) == gs.ERR_INVALID_ARG
    assert call(k=FAKE + 2) == gs.ERR_INVALID_ARG       # int32 array, 4-byte aligned
    assert call(p=FAKE + 1) == gs.ERR_INVALID_ARG
    assert call(out=FAKE + 4) == gs.ERR_INVALID_ARG
    assert call(ws=None) == gs.ERR_INVALID_ARG
    assert call(ws=FAKE + 8) == gs.ERR_WORKSPACE
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        assert call(k=None, p=None) == gs.ERR_CUDA
