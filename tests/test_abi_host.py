"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point declared in include/nvfp4.h, the pure host helpers agree
with the oracle, and argument validation rejects bad calls before anything
is launched (validation runs before any CUDA call)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

import oracle


@pytest.fixture(scope="module")
def nv():
    from nvfp4_block_scaled_29_b300 import build
    build.build()
    import nvfp4_block_scaled_29_b300 as m
    return m


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_path_calls():
    names = _declared_functions()
    for required in ["nvfp4_amax", "nvfp4_quantize_1d", "nvfp4_quantize_2d", "nvfp4_rht_quantize",
                     "nvfp4_amax_dual", "nvfp4_quantize_dual",
                     "nvfp4_dequantize", "nvfp4_gemm"]:
        assert required in names


def test_library_exports_every_declared_symbol(nv):
    lib = ctypes.CDLL(nv.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_rht_mask_from_seed_matches_oracle(nv):
    for seed in [0, 1, 2002, 2**40 + 3, 2**64 - 1]:
        assert nv.nvfp4_rht_mask_from_seed(seed) == oracle.rht_mask_from_seed(seed)


def test_scale_bytes_matches_oracle(nv):
    for rows, k in [(1, 16), (128, 64), (129, 80), (8192, 5120), (20480, 8192), (5, 1040)]:
        assert nv.nvfp4_scale_bytes(rows, k) == oracle.scale_bytes(rows, k)
    assert nv.nvfp4_scale_bytes(0, 64) == 0


def test_status_strings(nv):
    for s in range(9):
        assert nv.status_string(s) and "unknown" not in nv.status_string(s)
    assert "unknown" in nv.status_string(9)


@pytest.fixture(scope="module")
def guarded():
    """The index-guarded debug build (libnvfp4_guarded.so)."""
    from nvfp4_block_scaled_29_b300 import build
    lib = ctypes.CDLL(build.build(guards=True))
    lib.nvfp4_debug_guard_record.restype = ctypes.c_int
    lib.nvfp4_debug_guard_shrink.restype = ctypes.c_int
    return lib


def test_guarded_library_exports_every_declared_symbol(guarded):
    for name in _declared_functions():
        assert hasattr(guarded, name), name


def test_guard_entry_points(nv, guarded):
    """Which build is which, and the calls that need no GPU in either."""
    from nvfp4_block_scaled_29_b300 import build
    normal = ctypes.CDLL(build.LIB)
    normal.nvfp4_debug_guard_record.restype = ctypes.c_int
    normal.nvfp4_debug_guard_shrink.restype = ctypes.c_int
    assert normal.nvfp4_debug_guards_enabled() == 0
    assert guarded.nvfp4_debug_guards_enabled() == 1
    site, off = ctypes.c_uint32(7), ctypes.c_uint64(9)
    assert normal.nvfp4_debug_guard_record(ctypes.byref(site), ctypes.byref(off), None) == nv.NVFP4_OK
    assert site.value == 0 and off.value == 0
    assert normal.nvfp4_debug_guard_shrink(ctypes.c_uint64(8)) == nv.NVFP4_ERR_INVALID_ARG
    assert guarded.nvfp4_debug_guard_record(None, None, None) == nv.NVFP4_ERR_INVALID_ARG
    assert normal.nvfp4_debug_guard_record(None, None, None) == nv.NVFP4_ERR_INVALID_ARG
    assert nv.NVFP4_ERR_GUARD == 8 and "guard" in nv.status_string(nv.NVFP4_ERR_GUARD)


def test_guard_sites_are_documented():
    """The public header names the range of guard sites that csrc/guard.cuh
    defines."""
    text = open(os.path.join(ROOT, "nvfp4_block_scaled_29_b300", "csrc", "guard.cuh")).read()
    sites = [int(v) for v in re.findall(r"kGuard\w+ = (\d+),", text)]
    assert sites == list(range(1, len(sites) + 1))
    hdr = open(os.path.join(ROOT, "include", "nvfp4.h")).read()
    assert f"1..{len(sites)}" in hdr


def _view(nv, ptr, rows, cols, ld, tr=0):
    return nv.Bf16View(ptr, rows, cols, ld, tr)


def _q(nv, rows, k, codes=0x1000, scales=0x2000, gs=0x3000):
    return nv.QStruct(codes, scales, gs, rows, k, 0)


def test_validation_rejects_bad_calls(nv):
    L = nv.lib
    good = _view(nv, 0x10000, 32, 64, 64)
    q = _q(nv, 32, 64)
    # k not a multiple of 16
    assert L.nvfp4_quantize_1d(_view(nv, 0x10000, 32, 40, 40), None, 0, 0, 0,
                               ctypes.byref(_q(nv, 32, 40)), None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    # misaligned input pointer / leading dimension
    assert L.nvfp4_quantize_1d(_view(nv, 0x10002, 32, 64, 64), None, 0, 0, 0, ctypes.byref(q),
                               None) == nv.NVFP4_ERR_MISALIGNED
    assert L.nvfp4_quantize_1d(_view(nv, 0x10000, 32, 64, 68), None, 0, 0, 0, ctypes.byref(q),
                               None) == nv.NVFP4_ERR_MISALIGNED
    # ld smaller than the row
    assert L.nvfp4_quantize_1d(_view(nv, 0x10000, 32, 64, 32), None, 0, 0, 0, ctypes.byref(q),
                               None) == nv.NVFP4_ERR_INVALID_ARG
    # output shape mismatch, null output, bad rounding mode
    assert L.nvfp4_quantize_1d(good, None, 0, 0, 0, ctypes.byref(_q(nv, 16, 64)), None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_quantize_1d(good, None, 0, 0, 0, None, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_quantize_1d(good, None, 7, 0, 0, ctypes.byref(q), None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_quantize_1d(good, None, 3, 0, 0, ctypes.byref(q), None) == nv.NVFP4_ERR_INVALID_ARG
    # amax aliasing the output global scale
    assert L.nvfp4_quantize_1d(good, ctypes.c_void_p(0x3000), 0, 0, 0, ctypes.byref(q), None) == nv.NVFP4_ERR_INVALID_ARG
    # RHT mask out of range / zero for rht_quantize
    assert L.nvfp4_rht_quantize(good, 0x10000, None, 0, 0, 0, ctypes.byref(q), None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_rht_quantize(good, 0, None, 0, 0, 0, ctypes.byref(q), None) == nv.NVFP4_ERR_INVALID_ARG
    # 2D transposed emit needs rows % 16 == 0
    bad_rows = _view(nv, 0x10000, 24, 64, 64)
    assert L.nvfp4_quantize_2d(bad_rows, None, 0, 0, 0, ctypes.byref(_q(nv, 24, 64)),
                               ctypes.byref(_q(nv, 64, 24)), None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    # GEMM: k mismatch, K % 32, misaligned output leading dimension
    a, b = _q(nv, 128, 256), _q(nv, 256, 256)
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(_q(nv, 256, 224)), 0x4000, 0, 256, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_gemm(ctypes.byref(_q(nv, 128, 48)), ctypes.byref(_q(nv, 256, 48)), 0x4000, 0, 256, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), 0x4000, 1, 260, None) == nv.NVFP4_ERR_MISALIGNED
    assert L.nvfp4_gemm(ctypes.byref(a), ctypes.byref(b), 0x4000, 0, 128, None) == nv.NVFP4_ERR_INVALID_ARG
    # dequantize: misaligned output
    assert L.nvfp4_dequantize(ctypes.byref(q), ctypes.c_void_p(0x4004), 0, 64, None) == nv.NVFP4_ERR_MISALIGNED
    # amax: null output
    assert L.nvfp4_amax(good, 0, None, None) == nv.NVFP4_ERR_INVALID_ARG


def test_dual_validation_rejects_bad_calls(nv):
    L = nv.lib
    good = _view(nv, 0x10000, 32, 64, 64)
    q, qt = _q(nv, 32, 64), _q(nv, 64, 32, 0x5000, 0x6000, 0x7000)
    A, AT = ctypes.c_void_p(0x8000), ctypes.c_void_p(0x8004)
    # amax_dual: transposed view, rows % 16, aliased or null outputs
    assert L.nvfp4_amax_dual(_view(nv, 0x10000, 32, 64, 32, 1), 0, A, AT, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_amax_dual(_view(nv, 0x10000, 24, 64, 64), 0, A, AT, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert L.nvfp4_amax_dual(good, 0, A, A, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_amax_dual(good, 0, None, AT, None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_amax_dual(good, 0x10000, A, AT, None) == nv.NVFP4_ERR_INVALID_ARG
    # quantize_dual: shapes of the two outputs, required amaxes, aliasing
    args = lambda q_, qt_, a_, at_, mask=0, rnd=0: (good, a_, rnd, 0, 0, ctypes.byref(q_), mask, at_, 0, 0, 0,
                                                    ctypes.byref(qt_), None)
    assert L.nvfp4_quantize_dual(*args(q, _q(nv, 32, 64, 0x5000, 0x6000, 0x7000), A, AT)) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_quantize_dual(*args(q, qt, None, AT)) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_quantize_dual(*args(q, qt, A, None)) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_quantize_dual(*args(q, qt, ctypes.c_void_p(0x3000), AT)) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_quantize_dual(*args(q, _q(nv, 64, 32, 0x5000, 0x6000, 0x3000), A, AT)) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_quantize_dual(*args(q, qt, A, AT, mask=0x10000)) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_quantize_dual(*args(q, qt, A, AT, rnd=5)) == nv.NVFP4_ERR_INVALID_ARG
    odd = _view(nv, 0x10000, 24, 64, 64)
    assert L.nvfp4_quantize_dual(odd, A, 0, 0, 0, ctypes.byref(_q(nv, 24, 64)), 0, AT, 0, 0, 0,
                                 ctypes.byref(_q(nv, 64, 24, 0x5000, 0x6000, 0x7000)), None) == \
        nv.NVFP4_ERR_UNSUPPORTED_SHAPE


def test_mx_helpers_and_validation(nv):
    for rows, k in [(1, 32), (128, 64), (129, 96), (8192, 5120)]:
        assert nv.nvfp4_mx_scale_bytes(rows, k) == oracle.mx_scale_bytes(rows, k)
    L = nv.lib
    q = nv.QStruct(0x1000, 0x2000, None, 32, 64, 0)
    good = _view(nv, 0x10000, 32, 64, 64)
    assert L.nvfp4_mx_quantize(_view(nv, 0x10000, 32, 48, 48), 0, ctypes.byref(nv.QStruct(0x1000, 0x2000, None, 32, 48, 0)),
                               None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE
    assert L.nvfp4_mx_quantize(_view(nv, 0x10000, 32, 64, 32, 1), 0, ctypes.byref(q), None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_mx_quantize(good, 0x10000, ctypes.byref(q), None) == nv.NVFP4_ERR_INVALID_ARG
    assert L.nvfp4_mx_quantize(good, 0, ctypes.byref(nv.QStruct(0x1008, 0x2000, None, 32, 64, 0)), None) == \
        nv.NVFP4_ERR_MISALIGNED
    a, b = nv.QStruct(0x1000, 0x2000, None, 128, 96, 0), nv.QStruct(0x3000, 0x4000, None, 256, 64, 0)
    assert L.nvfp4_mx_gemm(ctypes.byref(a), ctypes.byref(b), 0x5000, 0, 256, None) == nv.NVFP4_ERR_INVALID_ARG
    a2 = nv.QStruct(0x1000, 0x2000, None, 128, 48, 0)
    b2 = nv.QStruct(0x3000, 0x4000, None, 256, 48, 0)
    assert L.nvfp4_mx_gemm(ctypes.byref(a2), ctypes.byref(b2), 0x5000, 0, 256, None) == nv.NVFP4_ERR_UNSUPPORTED_SHAPE


def test_build_tracks_every_kernel_header(tmp_path, monkeypatch):
    """Every header under csrc/ is an input of the build, so editing one of
    them (the CTA-pair GEMM, the dual quantiser, MXFP4, ...) rebuilds the
    library instead of keeping a stale one."""
    from nvfp4_block_scaled_29_b300 import build
    inputs = set(build._inputs())
    for f in os.listdir(build.CSRC):
        if f.endswith((".cuh", ".cu", ".h")):
            assert os.path.join(build.CSRC, f) in inputs, f
    fake = tmp_path / "libnvfp4.so"
    fake.write_bytes(b"")
    monkeypatch.setattr(build, "LIB", str(fake))
    newest = max(os.path.getmtime(f) for f in inputs)
    os.utime(fake, (newest + 10, newest + 10))
    assert build.up_to_date()
    dual = os.path.join(build.CSRC, "dual.cuh")
    t = os.path.getmtime(dual)
    os.utime(fake, (t - 10, t - 10))       # dual.cuh is now newer than the library
    assert not build.up_to_date()


def test_launch_status_has_its_own_code(nv):
    lib = ctypes.CDLL(nv.LIB_PATH)
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    assert nv.NVFP4_ERR_LAUNCH == 7
    assert b"shared memory" in lib.nvfp4_status_string(nv.NVFP4_ERR_LAUNCH)
    assert lib.nvfp4_status_string(nv.NVFP4_ERR_TIMEOUT) != lib.nvfp4_status_string(nv.NVFP4_ERR_LAUNCH)
