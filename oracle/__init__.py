"""CPU oracle of the NVFP4 linear-layer path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The library path never does,
and the oracle shares no code with it.

The arithmetic lives in plain C (``nvfp4_oracle.c``, built by ``build()``);
this module only marshals numpy arrays into it.  Each call documents which
step of the method it computes; citations are in ``nvfp4_oracle.h``:

* [NVB] NVIDIA technical blog "NVFP4 Trains with Precision of 16-Bit and Speed
  and Efficiency of 4-Bit" (Chinese edition), section "NVFP4 quantization
  recipe for pre-training", bullets 1-5.
* [SAI] prism.simon-ai.net article 7890 "From MVFP4 to the essence of compute
  precision": two-level scale, 16x16 weight blocks, Hadamard transform and
  stochastic rounding sections.
* [PHX] Salmon et al., SC'11, Philox4x32-10.

Functions with no independent pin say "parity unpinned"; at present every
function below is pinned by a ``-m "not gpu"`` test (tests/test_oracle_pins.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_c_u8p = ctypes.POINTER(ctypes.c_uint8)
_c_u16p = ctypes.POINTER(ctypes.c_uint16)
_c_u32p = ctypes.POINTER(ctypes.c_uint32)
_c_i64p = ctypes.POINTER(ctypes.c_int64)
_c_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile nvfp4_oracle.c into liboracle.so (plain C, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "nvfp4_oracle.h"))
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-Wall",
             "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            L.orc_e2m1_value.restype = ctypes.c_double
            L.orc_e2m1_value.argtypes = [ctypes.c_uint8]
            L.orc_e2m1_rne.restype = ctypes.c_uint8
            L.orc_e2m1_rne.argtypes = [ctypes.c_float]
            L.orc_e2m1_sr.restype = ctypes.c_uint8
            L.orc_e2m1_sr.argtypes = [ctypes.c_float, ctypes.c_uint32]
            L.orc_e4m3_value.restype = ctypes.c_float
            L.orc_e4m3_value.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_rne_satfinite.restype = ctypes.c_uint8
            L.orc_e4m3_rne_satfinite.argtypes = [ctypes.c_float]
            L.orc_bf16_to_f32.restype = ctypes.c_float
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f32_to_bf16_rne.restype = ctypes.c_uint16
            L.orc_f32_to_bf16_rne.argtypes = [ctypes.c_float]
            L.orc_philox4x32_10.restype = None
            L.orc_philox4x32_10.argtypes = [_c_u32p, _c_u32p, _c_u32p]
            L.orc_rht_mask_from_seed.restype = ctypes.c_uint32
            L.orc_rht_mask_from_seed.argtypes = [ctypes.c_uint64]
            L.orc_sr_r16_of_word.restype = ctypes.c_uint32
            L.orc_sr_r16_of_word.argtypes = [ctypes.c_uint32, ctypes.c_int]
            L.orc_sr_bits16_hw.restype = ctypes.c_uint32
            L.orc_sr_bits16_hw.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            L.orc_sr_bits16.restype = ctypes.c_uint32
            L.orc_sr_bits16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            L.orc_rht16.restype = None
            L.orc_rht16.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_uint32,
                                    ctypes.POINTER(ctypes.c_float)]
            L.orc_amax.restype = ctypes.c_float
            L.orc_amax.argtypes = [_c_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int, ctypes.c_uint32]
            L.orc_global_scale.restype = ctypes.c_int
            L.orc_global_scale.argtypes = [ctypes.c_float, ctypes.POINTER(ctypes.c_float)]
            L.orc_quantize.restype = ctypes.c_int
            L.orc_quantize.argtypes = [_c_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int, ctypes.c_uint32, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64,
                                       ctypes.c_int64, ctypes.c_int64, _c_u8p, _c_u8p]
            L.orc_scale_bytes.restype = ctypes.c_size_t
            L.orc_scale_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
            L.orc_swizzle_scales.restype = None
            L.orc_swizzle_scales.argtypes = [_c_u8p, ctypes.c_int64, ctypes.c_int64, _c_u8p]
            L.orc_unswizzle_scales.restype = None
            L.orc_unswizzle_scales.argtypes = [_c_u8p, ctypes.c_int64, ctypes.c_int64, _c_u8p]
            L.orc_transpose_codes.restype = None
            L.orc_transpose_codes.argtypes = [_c_u8p, ctypes.c_int64, ctypes.c_int64, _c_u8p]
            L.orc_dequantize.restype = None
            L.orc_dequantize.argtypes = [_c_u8p, _c_u8p, ctypes.c_float, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_void_p, ctypes.c_int, ctypes.c_int64]
            L.orc_gemm_points.restype = None
            L.orc_gemm_points.argtypes = [_c_u8p, _c_u8p, ctypes.c_float, _c_u8p, _c_u8p,
                                          ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_int64, _c_i64p, _c_i64p,
                                          _c_f64p, _c_f64p]
            L.orc_gemm_full.restype = None
            L.orc_gemm_full.argtypes = [_c_u8p, _c_u8p, ctypes.c_float, _c_u8p, _c_u8p,
                                        ctypes.c_float, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                        _c_f64p, _c_f64p]
            L.orc_e8m0_value.restype = ctypes.c_double
            L.orc_e8m0_value.argtypes = [ctypes.c_uint8]
            L.orc_mx_scale_code.restype = ctypes.c_uint8
            L.orc_mx_scale_code.argtypes = [ctypes.c_float]
            L.orc_mx_quantize.restype = ctypes.c_int
            L.orc_mx_quantize.argtypes = [_c_u16p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int, ctypes.c_uint32, ctypes.c_int64, ctypes.c_int64,
                                          _c_u8p, _c_u8p]
            L.orc_mx_scale_bytes.restype = ctypes.c_size_t
            L.orc_mx_scale_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
            L.orc_mx_swizzle_scales.restype = None
            L.orc_mx_swizzle_scales.argtypes = [_c_u8p, ctypes.c_int64, ctypes.c_int64, _c_u8p]
            L.orc_mx_unswizzle_scales.restype = None
            L.orc_mx_unswizzle_scales.argtypes = [_c_u8p, ctypes.c_int64, ctypes.c_int64, _c_u8p]
            L.orc_mx_dequantize.restype = None
            L.orc_mx_dequantize.argtypes = [_c_u8p, _c_u8p, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(ctypes.c_float),
                                            ctypes.c_int64]
            L.orc_mx_gemm_points.restype = None
            L.orc_mx_gemm_points.argtypes = [_c_u8p, _c_u8p, _c_u8p, _c_u8p, ctypes.c_int64, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int64, _c_i64p, _c_i64p, _c_f64p,
                                             _c_f64p]
            _lib = L
    return _lib


def _p(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"] or a.ndim == 1
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---------------------------------------------------------------- scalars --
def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e2m1_rne(v: float) -> int:
    return lib().orc_e2m1_rne(v)


def e2m1_sr(v: float, u16: int) -> int:
    """Stochastic E2M1 code of v: up iff u16 < floor(frac * 2^16)."""
    return lib().orc_e2m1_sr(v, u16)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def e4m3_rne_satfinite(t: float) -> int:
    return lib().orc_e4m3_rne_satfinite(t)


def f32_to_bf16_rne(f: float) -> int:
    return lib().orc_f32_to_bf16_rne(f)


def philox4x32_10(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    o = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_p(c, ctypes.c_uint32), _p(k, ctypes.c_uint32), _p(o, ctypes.c_uint32))
    return o


def rht_mask_from_seed(seed: int) -> int:
    return lib().orc_rht_mask_from_seed(seed)


def sr_bits16(seed: int, stream_id: int, idx: int) -> int:
    return lib().orc_sr_bits16(seed, stream_id, idx)


def sr_r16_of_word(w: int, p: int) -> int:
    """Second layout: integer r of element p (0..3) of the 32-bit word w."""
    return lib().orc_sr_r16_of_word(w, p)


def sr_bits16_hw(seed: int, stream_id: int, idx: int) -> int:
    """Second layout: the u16 (= 65535 - r) of element idx."""
    return lib().orc_sr_bits16_hw(seed, stream_id, idx)


def rht16(x, mask: int) -> np.ndarray:
    a = np.ascontiguousarray(x, dtype=np.float32)
    assert a.shape == (16,)
    o = np.zeros(16, dtype=np.float32)
    lib().orc_rht16(_p(a, ctypes.c_float), mask, _p(o, ctypes.c_float))
    return o


# ---------------------------------------------------------------- tensors --
def _view_dims(x: np.ndarray, transposed: bool):
    """x is the stored bf16 array (uint16).  Returns (rows, k, ld) of the
    logical operand [rows x k]."""
    assert x.dtype == np.uint16 and x.ndim == 2 and x.flags["C_CONTIGUOUS"]
    if transposed:
        return x.shape[1], x.shape[0], x.shape[1]
    return x.shape[0], x.shape[1], x.shape[1]


def amax(x: np.ndarray, transposed: bool = False, rht_mask: int = 0) -> float:
    """Step 1 (+2): max |x| over the tensor, or over RHT16 of every 16-chunk
    along k of the logical operand when rht_mask != 0."""
    rows, k, ld = _view_dims(x, transposed)
    return float(lib().orc_amax(_p(x, ctypes.c_uint16), rows, k, ld, int(transposed), rht_mask))


def global_scale(amax_v: float):
    """Step 3: (status, S_enc)."""
    s = ctypes.c_float(0.0)
    st = lib().orc_global_scale(amax_v, ctypes.byref(s))
    return st, s.value


def scale_bytes(rows: int, k: int) -> int:
    return int(lib().orc_scale_bytes(rows, k))


def swizzle_scales(plain: np.ndarray, rows: int, k: int) -> np.ndarray:
    plain = np.ascontiguousarray(plain, dtype=np.uint8)
    out = np.zeros(scale_bytes(rows, k), dtype=np.uint8)
    lib().orc_swizzle_scales(_p(plain, ctypes.c_uint8), rows, k, _p(out, ctypes.c_uint8))
    return out


def unswizzle_scales(swz: np.ndarray, rows: int, k: int) -> np.ndarray:
    swz = np.ascontiguousarray(swz, dtype=np.uint8)
    out = np.zeros((rows, k // 16), dtype=np.uint8)
    lib().orc_unswizzle_scales(_p(swz, ctypes.c_uint8), rows, k, _p(out, ctypes.c_uint8))
    return out


def transpose_codes(codes: np.ndarray, rows: int, k: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros((k, rows // 2), dtype=np.uint8)
    lib().orc_transpose_codes(_p(codes, ctypes.c_uint8), rows, k, _p(out, ctypes.c_uint8))
    return out


class Quantized:
    """A quantised operand: codes [rows x k/2], plain scales [rows x k/16],
    swizzled scales, and the global encode scale S_enc."""

    def __init__(self, codes, scales_plain, s_enc, rows, k, swizzle=True):
        self.codes = codes
        self.scales_plain = scales_plain
        self.s_enc = s_enc
        self.rows = rows
        self.k = k
        self.scales = swizzle_scales(scales_plain, rows, k) if swizzle else None


def _row_chunks(rows: int, threads: int, align: int):
    n = max(1, min(threads, (rows + align - 1) // align))
    step = ((rows + n - 1) // n + align - 1) // align * align
    return [(r, min(rows, r + step)) for r in range(0, rows, step)]


def quantize(x: np.ndarray, *, transposed: bool = False, rht_mask: int = 0, block2d: bool = False,
             amax_v: float | None = None, sr: bool = False, seed: int = 0, stream_id: int = 0,
             threads: int | None = None, rows_range=None, ranges=None,
             swizzle: bool = True, sr_hw: bool = False) -> Quantized:
    """Steps 1-6: quantise the logical operand of bf16 array x.

    sr: stochastic rounding with 16 independent random bits per element;
    sr_hw (with sr): the second random-bit layout (sr_bits16_hw).

    amax_v defaults to ``amax(x, transposed, rht_mask)``.  ``rows_range`` (or
    a list ``ranges`` of (lo, hi)) restricts the rows computed -- the other
    rows of the outputs stay 0 -- which the full-size parity tests use to
    check sampled rows only.  swizzle=False skips building the swizzled
    scale buffer."""
    rows, k, ld = _view_dims(x, transposed)
    if amax_v is None:
        amax_v = amax(x, transposed, rht_mask)
    st, s_enc = global_scale(amax_v)
    if st != 0:
        raise ValueError("non-finite amax")
    codes = np.zeros((rows, k // 2), dtype=np.uint8)
    scales = np.zeros((rows, k // 16), dtype=np.uint8)
    if ranges is None:
        ranges = [rows_range if rows_range is not None else (0, rows)]
    align = 16 if block2d else 1
    chunks = []
    for r_lo, r_hi in ranges:
        chunks += [(r_lo + a, r_lo + b)
                   for a, b in _row_chunks(r_hi - r_lo, threads or default_threads(), align)]

    def run(ch):
        return lib().orc_quantize(_p(x, ctypes.c_uint16), rows, k, ld, int(transposed), rht_mask,
                                  int(block2d), amax_v, (2 if sr_hw else 1) if sr else 0, seed, stream_id, ch[0], ch[1],
                                  _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8))

    if len(chunks) == 1:
        rcs = [run(chunks[0])]
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            rcs = list(ex.map(run, chunks))
    if any(rcs):
        raise ValueError("non-finite amax")
    return Quantized(codes, scales, s_enc, rows, k, swizzle=swizzle)


def dequantize(q: Quantized, out_bf16: bool = False) -> np.ndarray:
    """Dequantisation: x_hat = fp32(fp32(q * s_b) * fp32(1/S_enc))."""
    out = np.zeros((q.rows, q.k), dtype=np.uint16 if out_bf16 else np.float32)
    lib().orc_dequantize(_p(q.codes, ctypes.c_uint8), _p(q.scales, ctypes.c_uint8), q.s_enc,
                         q.rows, q.k, 0, q.rows, out.ctypes.data_as(ctypes.c_void_p),
                         int(out_bf16), q.k)
    return out


def gemm_points(qa: np.ndarray, sa_swz: np.ndarray, s_a: float, qb: np.ndarray,
                sb_swz: np.ndarray, s_b: float, m: int, n: int, k: int, ms, ns,
                threads: int | None = None):
    """FP64 reference y[i] = sum_k a[ms[i],k] b[ns[i],k] / (S_A S_B) and the
    matching sum of |a b| for the error bound."""
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    y = np.zeros(len(ms), dtype=np.float64)
    ab = np.zeros(len(ms), dtype=np.float64)
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sa_swz = np.ascontiguousarray(sa_swz, dtype=np.uint8)
    sb_swz = np.ascontiguousarray(sb_swz, dtype=np.uint8)
    nthr = max(1, min(threads or default_threads(), len(ms)))
    bounds = np.linspace(0, len(ms), nthr + 1).astype(np.int64)

    def run(i):
        lo, hi = int(bounds[i]), int(bounds[i + 1])
        if hi <= lo:
            return
        lib().orc_gemm_points(_p(qa, ctypes.c_uint8), _p(sa_swz, ctypes.c_uint8), s_a,
                              _p(qb, ctypes.c_uint8), _p(sb_swz, ctypes.c_uint8), s_b, m, n, k,
                              hi - lo, _p(ms[lo:hi], ctypes.c_int64), _p(ns[lo:hi], ctypes.c_int64),
                              _p(y[lo:hi], ctypes.c_double), _p(ab[lo:hi], ctypes.c_double))

    with ThreadPoolExecutor(nthr) as ex:
        list(ex.map(run, range(nthr)))
    return y, ab


def gemm_full(qa, sa_swz, s_a, qb, sb_swz, s_b, m: int, n: int, k: int,
              threads: int | None = None):
    """FP64 reference of the whole [m x n] output (small shapes only)."""
    y = np.zeros((m, n), dtype=np.float64)
    ab = np.zeros((m, n), dtype=np.float64)
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sa_swz = np.ascontiguousarray(sa_swz, dtype=np.uint8)
    sb_swz = np.ascontiguousarray(sb_swz, dtype=np.uint8)
    chunks = _row_chunks(m, threads or default_threads(), 1)

    def run(ch):
        lib().orc_gemm_full(_p(qa, ctypes.c_uint8), _p(sa_swz, ctypes.c_uint8), s_a,
                            _p(qb, ctypes.c_uint8), _p(sb_swz, ctypes.c_uint8), s_b, m, n, k,
                            ch[0], ch[1], _p(y, ctypes.c_double), _p(ab, ctypes.c_double))

    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(run, chunks))
    return y, ab


# ------------------------------------------------------------------ MXFP4 --
# The comparison format of [NVB] bullets 1-2 and [SAI] "MVFP4 and MXFP4":
# 32-element blocks with one power-of-two (E8M0) scale each, no tensor scale.
def e8m0_value(code: int) -> float:
    return float(lib().orc_e8m0_value(code))


def mx_scale_code(amax_b: float) -> int:
    """E8M0 code of a block: X = floor(log2 amax_b) - 2, clamped to
    [-127, 127]; code X + 127."""
    return int(lib().orc_mx_scale_code(amax_b))


def mx_scale_bytes(rows: int, k: int) -> int:
    return int(lib().orc_mx_scale_bytes(rows, k))


def mx_swizzle_scales(plain: np.ndarray, rows: int, k: int) -> np.ndarray:
    plain = np.ascontiguousarray(plain, dtype=np.uint8)
    out = np.zeros(mx_scale_bytes(rows, k), dtype=np.uint8)
    lib().orc_mx_swizzle_scales(_p(plain, ctypes.c_uint8), rows, k, _p(out, ctypes.c_uint8))
    return out


def mx_unswizzle_scales(swz: np.ndarray, rows: int, k: int) -> np.ndarray:
    swz = np.ascontiguousarray(swz, dtype=np.uint8)
    out = np.zeros((rows, k // 32), dtype=np.uint8)
    lib().orc_mx_unswizzle_scales(_p(swz, ctypes.c_uint8), rows, k, _p(out, ctypes.c_uint8))
    return out


class MxQuantized:
    """An MXFP4 operand: codes [rows x k/2], plain E8M0 scales [rows x k/32]
    and the swizzled scale buffer."""

    def __init__(self, codes, scales_plain, rows, k):
        self.codes, self.scales_plain, self.rows, self.k = codes, scales_plain, rows, k
        self.scales = mx_swizzle_scales(scales_plain, rows, k)


def mx_quantize(x: np.ndarray, *, transposed: bool = False, rht_mask: int = 0,
                threads: int | None = None) -> MxQuantized:
    """1x32 MXFP4 quantisation (RNE) of the logical operand of bf16 array x,
    optionally after RHT16 of every 16-chunk along k."""
    rows, k, ld = _view_dims(x, transposed)
    if k % 32:
        raise ValueError("k must be a multiple of 32")
    codes = np.zeros((rows, k // 2), dtype=np.uint8)
    scales = np.zeros((rows, k // 32), dtype=np.uint8)
    chunks = _row_chunks(rows, threads or default_threads(), 1)

    def run(ch):
        return lib().orc_mx_quantize(_p(x, ctypes.c_uint16), rows, k, ld, int(transposed), rht_mask,
                                     ch[0], ch[1], _p(codes, ctypes.c_uint8), _p(scales, ctypes.c_uint8))

    with ThreadPoolExecutor(len(chunks)) as ex:
        rcs = list(ex.map(run, chunks))
    if any(rcs):
        raise ValueError("non-finite block amax")
    return MxQuantized(codes, scales, rows, k)


def mx_dequantize(q: MxQuantized) -> np.ndarray:
    out = np.zeros((q.rows, q.k), dtype=np.float32)
    lib().orc_mx_dequantize(_p(q.codes, ctypes.c_uint8), _p(q.scales, ctypes.c_uint8), q.rows, q.k,
                            0, q.rows, out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), q.k)
    return out


def mx_gemm_points(qa, sa_swz, qb, sb_swz, m: int, n: int, k: int, ms, ns, threads: int | None = None):
    """FP64 reference y[i] = sum_k a[ms[i],k] b[ns[i],k] of MXFP4 operands
    and the matching sum of |a b|."""
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    y = np.zeros(len(ms), dtype=np.float64)
    ab = np.zeros(len(ms), dtype=np.float64)
    qa, qb = np.ascontiguousarray(qa, dtype=np.uint8), np.ascontiguousarray(qb, dtype=np.uint8)
    sa_swz, sb_swz = np.ascontiguousarray(sa_swz, dtype=np.uint8), np.ascontiguousarray(sb_swz, dtype=np.uint8)
    nthr = max(1, min(threads or default_threads(), len(ms)))
    bounds = np.linspace(0, len(ms), nthr + 1).astype(np.int64)

    def run(i):
        lo, hi = int(bounds[i]), int(bounds[i + 1])
        if hi > lo:
            lib().orc_mx_gemm_points(_p(qa, ctypes.c_uint8), _p(sa_swz, ctypes.c_uint8), _p(qb, ctypes.c_uint8),
                                     _p(sb_swz, ctypes.c_uint8), m, n, k, hi - lo, _p(ms[lo:hi], ctypes.c_int64),
                                     _p(ns[lo:hi], ctypes.c_int64), _p(y[lo:hi], ctypes.c_double),
                                     _p(ab[lo:hi], ctypes.c_double))

    with ThreadPoolExecutor(nthr) as ex:
        list(ex.map(run, range(nthr)))
    return y, ab


def mx_gemm_full(qa, sa_swz, qb, sb_swz, m: int, n: int, k: int, threads: int | None = None):
    mm, nn = np.meshgrid(np.arange(m), np.arange(n), indexing="ij")
    y, ab = mx_gemm_points(qa, sa_swz, qb, sb_swz, m, n, k, mm.ravel(), nn.ravel(), threads)
    return y.reshape(m, n), ab.reshape(m, n)
