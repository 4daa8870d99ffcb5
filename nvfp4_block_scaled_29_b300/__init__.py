"""Python binding of libnvfp4 (the NVFP4 linear-layer path on one B300).

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libnvfp4.so`` (built in-tree by ``build.py``).  PyTorch provides device
memory and streams.  There is no CPU fallback: importing this package on a
machine where the library cannot be loaded raises, and every call checks the
status the C ABI returns.

The functions carry the C names of ``include/nvfp4.h``:

  nvfp4_amax, nvfp4_quantize_1d, nvfp4_quantize_2d, nvfp4_rht_quantize,
  nvfp4_amax_dual, nvfp4_quantize_dual, nvfp4_dequantize, nvfp4_gemm,
  nvfp4_mx_quantize, nvfp4_mx_dequantize, nvfp4_mx_gemm, nvfp4_mx_scale_bytes,
  nvfp4_rht_mask_from_seed, nvfp4_get_status, nvfp4_scale_bytes

Sources of the method: NVIDIA blog "NVFP4 Trains with Precision of 16-Bit and
Speed and Efficiency of 4-Bit" (recipe bullets 1-5, Figure 1) and the
prism.simon-ai.net article 7890 (two-level scale, 16x16 weight blocks,
Hadamard transform, stochastic rounding).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# NVFP4_DEBUG_GUARDS=1 in the environment loads the debug build, whose kernels
# check every plain global access against its buffer's extent (same entry
# points, same results; see include/nvfp4.h, "Index guards").
GUARDED = os.environ.get("NVFP4_DEBUG_GUARDS", "0") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "libnvfp4_guarded.so" if GUARDED else "libnvfp4.so")

NVFP4_OK = 0
NVFP4_ERR_INVALID_ARG = 1
NVFP4_ERR_UNSUPPORTED_SHAPE = 2
NVFP4_ERR_MISALIGNED = 3
NVFP4_ERR_NONFINITE = 4
NVFP4_ERR_TIMEOUT = 5
NVFP4_ERR_CUDA = 6
NVFP4_ERR_LAUNCH = 7
NVFP4_ERR_GUARD = 8
NVFP4_RNE = 0
NVFP4_SR = 1
NVFP4_SR_HW = 2              # the same rule, random bits in the hardware conversion's layout


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class Bf16View(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ld", ctypes.c_int64), ("transposed", ctypes.c_int)]


class QStruct(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("global_scale", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("k", ctypes.c_int64), ("block2d", ctypes.c_int)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run "
                          "`python -m nvfp4_block_scaled_29_b300.build` (needs nvcc)")
    L = ctypes.CDLL(LIB_PATH)
    st = ctypes.c_int
    vp = ctypes.c_void_p
    u64 = ctypes.c_uint64
    L.nvfp4_amax.argtypes = [Bf16View, ctypes.c_uint32, vp, vp]
    L.nvfp4_amax.restype = st
    L.nvfp4_quantize_1d.argtypes = [Bf16View, vp, ctypes.c_int, u64, u64, ctypes.POINTER(QStruct), vp]
    L.nvfp4_quantize_1d.restype = st
    L.nvfp4_quantize_2d.argtypes = [Bf16View, vp, ctypes.c_int, u64, u64, ctypes.POINTER(QStruct),
                                    ctypes.POINTER(QStruct), vp]
    L.nvfp4_quantize_2d.restype = st
    L.nvfp4_rht_quantize.argtypes = [Bf16View, ctypes.c_uint32, vp, ctypes.c_int, u64, u64,
                                     ctypes.POINTER(QStruct), vp]
    L.nvfp4_rht_quantize.restype = st
    L.nvfp4_amax_dual.argtypes = [Bf16View, ctypes.c_uint32, vp, vp, vp]
    L.nvfp4_amax_dual.restype = st
    L.nvfp4_quantize_dual.argtypes = [Bf16View, vp, ctypes.c_int, u64, u64, ctypes.POINTER(QStruct),
                                      ctypes.c_uint32, vp, ctypes.c_int, u64, u64, ctypes.POINTER(QStruct), vp]
    L.nvfp4_quantize_dual.restype = st
    L.nvfp4_mx_scale_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    L.nvfp4_mx_scale_bytes.restype = ctypes.c_size_t
    L.nvfp4_mx_quantize.argtypes = [Bf16View, ctypes.c_uint32, ctypes.POINTER(QStruct), vp]
    L.nvfp4_mx_quantize.restype = st
    L.nvfp4_mx_dequantize.argtypes = [ctypes.POINTER(QStruct), vp, ctypes.c_int, ctypes.c_int64, vp]
    L.nvfp4_mx_dequantize.restype = st
    L.nvfp4_mx_gemm.argtypes = [ctypes.POINTER(QStruct), ctypes.POINTER(QStruct), vp, ctypes.c_int,
                                ctypes.c_int64, vp]
    L.nvfp4_mx_gemm.restype = st
    L.nvfp4_dequantize.argtypes = [ctypes.POINTER(QStruct), vp, ctypes.c_int, ctypes.c_int64, vp]
    L.nvfp4_dequantize.restype = st
    L.nvfp4_gemm.argtypes = [ctypes.POINTER(QStruct), ctypes.POINTER(QStruct), vp, ctypes.c_int,
                             ctypes.c_int64, vp]
    L.nvfp4_gemm.restype = st
    L.nvfp4_rht_mask_from_seed.argtypes = [u64]
    L.nvfp4_rht_mask_from_seed.restype = ctypes.c_uint32
    L.nvfp4_get_status.argtypes = [vp]
    L.nvfp4_get_status.restype = st
    L.nvfp4_scale_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    L.nvfp4_scale_bytes.restype = ctypes.c_size_t
    L.nvfp4_status_string.argtypes = [st]
    L.nvfp4_status_string.restype = ctypes.c_char_p
    L.nvfp4_debug_inject.argtypes = [ctypes.c_int]
    L.nvfp4_debug_inject.restype = st
    L.nvfp4_debug_check_div6.argtypes = [ctypes.c_uint32, ctypes.c_uint32, vp, vp, vp]
    L.nvfp4_debug_check_div6.restype = st
    L.nvfp4_debug_guards_enabled.argtypes = []
    L.nvfp4_debug_guards_enabled.restype = ctypes.c_int
    L.nvfp4_debug_guard_record.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint64), vp]
    L.nvfp4_debug_guard_record.restype = st
    L.nvfp4_debug_guard_shrink.argtypes = [u64]
    L.nvfp4_debug_guard_shrink.restype = st
    return L


lib = _load()


def status_string(s: int) -> str:
    return lib.nvfp4_status_string(s).decode()


def _check(status: int, what: str, raise_on_error: bool = True) -> int:
    if status != NVFP4_OK and raise_on_error:
        raise Nvfp4Error(status, what)
    return status


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


# ----------------------------------------------------------------- views ---
def bf16_view(x: torch.Tensor, transposed: bool = False) -> Bf16View:
    """View a 2-D bf16 tensor (stored row-major with unit column stride) as
    the logical operand [rows x cols]; with transposed=True the logical operand
    is x^T (x stored as [k x rows])."""
    if x.dim() != 2 or x.stride(1) != 1 or x.element_size() != 2:
        raise ValueError("expected a 2-D 16-bit tensor with unit column stride")
    r, c = x.shape
    if transposed:
        return Bf16View(x.data_ptr(), c, r, x.stride(0), 1)
    return Bf16View(x.data_ptr(), r, c, x.stride(0), 0)


class QTensor:
    """A quantised operand in device memory (torch-allocated): codes
    [rows, k/2] uint8, swizzled scales (nvfp4_scale_bytes) uint8, global
    encode scale [1] float32."""

    def __init__(self, rows: int, k: int, block2d: bool = False, device="cuda"):
        self.rows, self.k, self.block2d = rows, k, block2d
        self.codes = torch.empty((rows, k // 2), dtype=torch.uint8, device=device)
        self.scales = torch.empty((max(1, nvfp4_scale_bytes(rows, k)),), dtype=torch.uint8, device=device)
        self.global_scale = torch.empty((1,), dtype=torch.float32, device=device)

    def c(self) -> QStruct:
        return QStruct(self.codes.data_ptr(), self.scales.data_ptr(), self.global_scale.data_ptr(),
                       self.rows, self.k, int(self.block2d))


class MxQTensor:
    """An MXFP4 operand in device memory: codes [rows, k/2] uint8 and swizzled
    E8M0 scales (nvfp4_mx_scale_bytes) uint8; no tensor scale."""

    def __init__(self, rows: int, k: int, device="cuda"):
        self.rows, self.k = rows, k
        self.codes = torch.empty((rows, k // 2), dtype=torch.uint8, device=device)
        self.scales = torch.empty((max(1, nvfp4_mx_scale_bytes(rows, k)),), dtype=torch.uint8, device=device)

    def c(self) -> QStruct:
        return QStruct(self.codes.data_ptr(), self.scales.data_ptr(), None, self.rows, self.k, 0)


def _as_view(x, transposed):
    return x if isinstance(x, Bf16View) else bf16_view(x, transposed)


# ------------------------------------------------------------ the calls ----
def nvfp4_amax(x, rht_mask: int = 0, amax: torch.Tensor | None = None, *, transposed=False,
               stream=None, check=True) -> torch.Tensor:
    v = _as_view(x, transposed)
    if amax is None:
        amax = torch.empty((1,), dtype=torch.float32, device="cuda")
    _check(lib.nvfp4_amax(v, rht_mask, amax.data_ptr(), _stream(stream)), "nvfp4_amax", check)
    return amax


def nvfp4_quantize_1d(x, amax: torch.Tensor | None, rnd: int, seed: int, stream_id: int,
                      out: QTensor, *, transposed=False, stream=None, check=True) -> int:
    q = out.c()
    return _check(lib.nvfp4_quantize_1d(_as_view(x, transposed), _ptr(amax), rnd, seed, stream_id,
                                        ctypes.byref(q), _stream(stream)), "nvfp4_quantize_1d", check)


def nvfp4_quantize_2d(w, amax: torch.Tensor | None, rnd: int, seed: int, stream_id: int,
                      out: QTensor, out_t: QTensor | None = None, *, transposed=False, stream=None,
                      check=True) -> int:
    q = out.c()
    qt = out_t.c() if out_t is not None else None
    return _check(lib.nvfp4_quantize_2d(_as_view(w, transposed), _ptr(amax), rnd, seed, stream_id,
                                        ctypes.byref(q), ctypes.byref(qt) if qt is not None else None,
                                        _stream(stream)), "nvfp4_quantize_2d", check)


def nvfp4_rht_quantize(x, rht_mask: int, amax: torch.Tensor | None, rnd: int, seed: int,
                       stream_id: int, out: QTensor, *, transposed=False, stream=None,
                       check=True) -> int:
    q = out.c()
    return _check(lib.nvfp4_rht_quantize(_as_view(x, transposed), rht_mask, _ptr(amax), rnd, seed,
                                         stream_id, ctypes.byref(q), _stream(stream)),
                  "nvfp4_rht_quantize", check)


def nvfp4_amax_dual(x, rht_mask: int = 0, amax: torch.Tensor | None = None,
                    amax_t: torch.Tensor | None = None, *, stream=None, check=True):
    """Both amaxes of a stored tensor S in one read: (max |S|, max |RHT16 of
    S^T along its k = S's rows|)."""
    v = _as_view(x, False)
    if amax is None:
        amax = torch.empty((1,), dtype=torch.float32, device="cuda")
    if amax_t is None:
        amax_t = torch.empty((1,), dtype=torch.float32, device="cuda")
    _check(lib.nvfp4_amax_dual(v, rht_mask, amax.data_ptr(), amax_t.data_ptr(), _stream(stream)),
           "nvfp4_amax_dual", check)
    return amax, amax_t


def nvfp4_quantize_dual(x, amax: torch.Tensor, rnd: int, seed: int, stream_id: int, out: QTensor,
                        rht_mask_t: int, amax_t: torch.Tensor, rnd_t: int, seed_t: int,
                        stream_id_t: int, out_t: QTensor, *, stream=None, check=True) -> int:
    """Row-wise operand S (out) and column-wise operand S^T with optional
    RHT (out_t) from one read of S."""
    q, qt = out.c(), out_t.c()
    return _check(lib.nvfp4_quantize_dual(_as_view(x, False), _ptr(amax), rnd, seed, stream_id,
                                          ctypes.byref(q), rht_mask_t, _ptr(amax_t), rnd_t, seed_t,
                                          stream_id_t, ctypes.byref(qt), _stream(stream)),
                  "nvfp4_quantize_dual", check)


def nvfp4_dequantize(q: QTensor, out: torch.Tensor, *, stream=None, check=True) -> int:
    if out.dtype not in (torch.float32, torch.bfloat16) or out.dim() != 2 or out.stride(1) != 1:
        raise ValueError("out must be a 2-D float32 or bfloat16 tensor with unit column stride")
    qs = q.c()
    return _check(lib.nvfp4_dequantize(ctypes.byref(qs), out.data_ptr(), int(out.dtype == torch.bfloat16),
                                       out.stride(0), _stream(stream)), "nvfp4_dequantize", check)


def nvfp4_gemm(a: QTensor, b: QTensor, d: torch.Tensor, *, stream=None, check=True) -> int:
    if d.dtype not in (torch.float32, torch.bfloat16) or d.dim() != 2 or d.stride(1) != 1:
        raise ValueError("d must be a 2-D float32 or bfloat16 tensor with unit column stride")
    qa, qb = a.c(), b.c()
    return _check(lib.nvfp4_gemm(ctypes.byref(qa), ctypes.byref(qb), d.data_ptr(),
                                 int(d.dtype == torch.bfloat16), d.stride(0), _stream(stream)),
                  "nvfp4_gemm", check)


def nvfp4_mx_scale_bytes(rows: int, k: int) -> int:
    return int(lib.nvfp4_mx_scale_bytes(rows, k))


def nvfp4_mx_quantize(x, rht_mask: int, out: MxQTensor, *, stream=None, check=True) -> int:
    q = out.c()
    return _check(lib.nvfp4_mx_quantize(_as_view(x, False), rht_mask, ctypes.byref(q), _stream(stream)),
                  "nvfp4_mx_quantize", check)


def nvfp4_mx_dequantize(q: MxQTensor, out: torch.Tensor, *, stream=None, check=True) -> int:
    if out.dtype not in (torch.float32, torch.bfloat16) or out.dim() != 2 or out.stride(1) != 1:
        raise ValueError("out must be a 2-D float32 or bfloat16 tensor with unit column stride")
    qs = q.c()
    return _check(lib.nvfp4_mx_dequantize(ctypes.byref(qs), out.data_ptr(), int(out.dtype == torch.bfloat16),
                                          out.stride(0), _stream(stream)), "nvfp4_mx_dequantize", check)


def nvfp4_mx_gemm(a: MxQTensor, b: MxQTensor, d: torch.Tensor, *, stream=None, check=True) -> int:
    if d.dtype not in (torch.float32, torch.bfloat16) or d.dim() != 2 or d.stride(1) != 1:
        raise ValueError("d must be a 2-D float32 or bfloat16 tensor with unit column stride")
    qa, qb = a.c(), b.c()
    return _check(lib.nvfp4_mx_gemm(ctypes.byref(qa), ctypes.byref(qb), d.data_ptr(),
                                    int(d.dtype == torch.bfloat16), d.stride(0), _stream(stream)),
                  "nvfp4_mx_gemm", check)


def nvfp4_rht_mask_from_seed(seed: int) -> int:
    return int(lib.nvfp4_rht_mask_from_seed(seed))


def nvfp4_get_status(stream=None) -> int:
    return int(lib.nvfp4_get_status(_stream(stream)))


def nvfp4_debug_inject(mode: int) -> int:
    """Test-only: mode 1 makes the next streamed amax launch skip the copy of
    its first tile, so that its bounded wait expires and nvfp4_get_status
    reports NVFP4_ERR_TIMEOUT; mode 2 makes the next dual quantise take its
    64-bit Philox block-index path; mode 0 clears both (see include/nvfp4.h)."""
    return _check(int(lib.nvfp4_debug_inject(mode)), "nvfp4_debug_inject")


def nvfp4_debug_guards_enabled() -> bool:
    """True when the loaded library is the guarded debug build."""
    return bool(lib.nvfp4_debug_guards_enabled())


def nvfp4_debug_guard_record(stream=None):
    """(site, byte offset) of the first access an index guard refused since
    the last call, or None; clears the record (debug build; None otherwise)."""
    site = ctypes.c_uint32(0)
    off = ctypes.c_uint64(0)
    _check(lib.nvfp4_debug_guard_record(ctypes.byref(site), ctypes.byref(off), _stream(stream)),
           "nvfp4_debug_guard_record")
    return None if site.value == 0 else (int(site.value), int(off.value))


def nvfp4_debug_guard_shrink(nbytes: int) -> int:
    """Test-only (debug build): every guard checks against its extent minus
    nbytes, so in-bounds accesses near a buffer's end are refused and
    reported; 0 restores the extents."""
    return _check(int(lib.nvfp4_debug_guard_shrink(nbytes)), "nvfp4_debug_guard_shrink")


def nvfp4_debug_check_div6(lo_bits: int, hi_bits: int, *, stream=None):
    """Test-only: (mismatches, smallest mismatching bit pattern or None) of the
    kernels' amax_b / 6 against IEEE division, over float bit patterns in
    [lo_bits, hi_bits) (see include/nvfp4.h)."""
    cnt = torch.empty((1,), dtype=torch.int64, device="cuda")
    first = torch.empty((1,), dtype=torch.int32, device="cuda")
    _check(lib.nvfp4_debug_check_div6(lo_bits, hi_bits, cnt.data_ptr(), first.data_ptr(), _stream(stream)),
           "nvfp4_debug_check_div6")
    n = int(cnt.cpu()[0])
    f = int(first.cpu()[0]) & 0xFFFFFFFF
    return n, (None if f == 0xFFFFFFFF else f)


def nvfp4_scale_bytes(rows: int, k: int) -> int:
    return int(lib.nvfp4_scale_bytes(rows, k))


# ------------------------------------------------------------------ tracing --
# NVFP4_TRACE=1: every call of the functions above logs its name, its tensor
# arguments' shapes and its host enqueue time (the calls are asynchronous) to
# stderr.  NVFP4_TRACE=sync also synchronises the device before and after the
# call, so the logged time covers its kernels.
def _trace_wrap(fn, sync: bool):
    import functools
    import sys
    import time

    def desc(a):
        if isinstance(a, torch.Tensor):
            return "x".join(map(str, a.shape)) + ":" + str(a.dtype).replace("torch.", "")
        if isinstance(a, (QTensor, MxQTensor)):
            return f"q{a.rows}x{a.k}"
        return repr(a) if isinstance(a, (int, float)) else type(a).__name__

    @functools.wraps(fn)
    def traced(*args, **kw):
        if sync and torch.cuda.is_available():
            torch.cuda.synchronize()
        t0 = time.perf_counter()
        r = fn(*args, **kw)
        if sync and torch.cuda.is_available():
            torch.cuda.synchronize()
        us = (time.perf_counter() - t0) * 1e6
        print(f"[nvfp4] {fn.__name__}({', '.join(desc(a) for a in args)}) {us:.1f} us"
              f"{' (device)' if sync else ' (enqueue)'}", file=sys.stderr)
        return r

    return traced


_TRACE = os.environ.get("NVFP4_TRACE", "")
if _TRACE in ("1", "sync"):
    for _name in [n for n in list(globals()) if n.startswith("nvfp4_") and callable(globals()[n])]:
        globals()[_name] = _trace_wrap(globals()[_name], _TRACE == "sync")
