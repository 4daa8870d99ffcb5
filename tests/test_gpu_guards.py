"""Memory safety of the kernels, checked without a memory checker.

* Red zones (either build): every output of a call is carved out of one
  larger device buffer filled with a canary byte, 4 KB from its neighbours.
  After the call every byte outside the outputs must still hold the canary,
  and the outputs must equal those of the same call on separately allocated
  tensors.  Shapes have ragged row and column tails.
* The guarded build (libnvfp4_guarded.so, loaded when NVFP4_DEBUG_GUARDS=1):
  a child process runs the GPU parity modules against it; the conftest there
  fails any test after which an index guard refused an access.  In that child
  the shrink tests below also run: with every guard's extent cut short by a
  few bytes, each kernel family must refuse exactly the accesses that touch
  the cut-off tail (the stores are skipped, so those bytes keep their
  canary), report NVFP4_ERR_GUARD and record the site, and write every other
  byte as the unguarded call does.  No access ever leaves its buffer.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import synth
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
RED = 4096
CANARY = 0xA5
MASK = 0x9D2B

# guard sites (the site field of nvfp4_debug_guard_record)
AMAX_X = 1
Q2D = {2, 3, 4, 5}
DUAL = {6, 7, 8, 9}
DEQ = {10, 11}
MX_Q = {12, 13, 14}
GEMM_D = 17


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


class Arena:
    """Outputs carved from one canary-filled device buffer, RED bytes apart."""

    def __init__(self, capacity=1 << 23):
        self.buf = torch.full((capacity,), CANARY, dtype=torch.uint8, device="cuda")
        self.pos = RED
        self.spans = []

    def take(self, nbytes, dtype=torch.uint8, shape=None):
        nbytes = max(1, int(nbytes))
        assert self.pos + nbytes + RED <= self.buf.numel()
        t = self.buf[self.pos:self.pos + nbytes]
        self.spans.append((self.pos, nbytes))
        self.pos += (nbytes + 255) // 256 * 256 + RED
        if dtype != torch.uint8:
            t = t.view(dtype)
        return t.view(shape) if shape is not None else t

    def qtensor(self, nv, rows, k, block2d=False):
        q = nv.QTensor.__new__(nv.QTensor)
        q.rows, q.k, q.block2d = rows, k, block2d
        q.codes = self.take(rows * k // 2, shape=(rows, k // 2))
        q.scales = self.take(nv.nvfp4_scale_bytes(rows, k))
        q.global_scale = self.take(4, torch.float32)
        return q

    def mx_qtensor(self, nv, rows, k):
        q = nv.MxQTensor.__new__(nv.MxQTensor)
        q.rows, q.k = rows, k
        q.codes = self.take(rows * k // 2, shape=(rows, k // 2))
        q.scales = self.take(nv.nvfp4_mx_scale_bytes(rows, k))
        return q

    def check(self):
        torch.cuda.synchronize()
        host = self.buf.cpu().numpy()
        outside = np.ones(host.size, dtype=bool)
        for o, n in self.spans:
            outside[o:o + n] = False
        bad = np.flatnonzero(outside & (host != CANARY))
        assert bad.size == 0, f"{bad.size} bytes written outside the outputs; first at arena byte {bad[0]}"


def _x(rows, cols, seed):
    return synth.normal_bf16((rows, cols), seed, 1.0, 0.002, 60.0)


def _ok(nv):
    torch.cuda.synchronize()
    st = nv.nvfp4_get_status()
    assert st == nv.NVFP4_OK, nv.status_string(st)


def _same_q(a, b):
    assert torch.equal(a.codes, b.codes)
    n = b.scales.numel()
    assert torch.equal(a.scales[:n], b.scales[:n])


# ---------------------------------------------------------- red zones ------
@pytest.mark.parametrize("rows,cols,transposed,mask,ld_pad", [
    (64, 256, False, 0, 0), (200, 208, False, 0, 8), (199, 208, True, 0, 0),
    (200, 208, False, MASK, 8), (199, 208, True, MASK, 8)])
def test_red_zone_amax(nv, rows, cols, transposed, mask, ld_pad):
    x = _x(rows, cols, rows + cols)
    stored = x.T.copy() if transposed else x
    ld = (stored.shape[1] + 7) // 8 * 8 + ld_pad
    d = dev_bf16(stored, ld)
    ar = Arena()
    amax = ar.take(4, torch.float32)
    nv.nvfp4_amax(d, mask, amax, transposed=transposed)
    _ok(nv)
    ar.check()
    assert float(amax.cpu()[0]) == float(nv.nvfp4_amax(d, mask, transposed=transposed).cpu()[0])


@pytest.mark.parametrize("rows,k,transposed,mask,sr", [
    (200, 208, False, 0, False), (200, 208, False, 0, True), (200, 208, True, 0, True),
    (199, 208, True, 0, False), (199, 208, True, 0, True), (200, 208, False, MASK, True),
    (199, 208, True, MASK, False)])
def test_red_zone_quantize_1d(nv, rows, k, transposed, mask, sr):
    x = _x(rows, k, 7 * rows + k)
    d = dev_bf16(x.T.copy(), ((rows + 7) // 8) * 8) if transposed else dev_bf16(x)
    amax = nv.nvfp4_amax(d, mask, transposed=transposed)
    rnd = nv.NVFP4_SR if sr else nv.NVFP4_RNE
    ar = Arena()
    q = ar.qtensor(nv, rows, k)
    ref = nv.QTensor(rows, k)
    for out in (q, ref):
        if mask:
            nv.nvfp4_rht_quantize(d, mask, amax, rnd, 3, 4, out, transposed=transposed)
        else:
            nv.nvfp4_quantize_1d(d, amax, rnd, 3, 4, out, transposed=transposed)
    _ok(nv)
    ar.check()
    _same_q(q, ref)


@pytest.mark.parametrize("rows,k,emit_t,sr", [(200, 208, False, False), (208, 272, True, False),
                                              (208, 272, True, True), (112, 1040, True, False)])
def test_red_zone_quantize_2d(nv, rows, k, emit_t, sr):
    x = _x(rows, k, 11 * rows + k)
    d = dev_bf16(x)
    amax = nv.nvfp4_amax(d)
    rnd = nv.NVFP4_SR if sr else nv.NVFP4_RNE
    ar = Arena()
    q = ar.qtensor(nv, rows, k, True)
    qt = ar.qtensor(nv, k, rows, True) if emit_t else None
    ref = nv.QTensor(rows, k, True)
    ref_t = nv.QTensor(k, rows, True) if emit_t else None
    nv.nvfp4_quantize_2d(d, amax, rnd, 5, 6, q, qt)
    nv.nvfp4_quantize_2d(d, amax, rnd, 5, 6, ref, ref_t)
    _ok(nv)
    ar.check()
    _same_q(q, ref)
    if emit_t:
        _same_q(qt, ref_t)


@pytest.mark.parametrize("rows,cols,mask", [(144, 272, MASK), (400, 784, 0)])
def test_red_zone_quantize_dual(nv, rows, cols, mask):
    x = _x(rows, cols, rows * 3 + cols)
    d = dev_bf16(x, (cols + 7) // 8 * 8 + 8)
    a, at = nv.nvfp4_amax_dual(d, mask)
    ar = Arena()
    q, qt = ar.qtensor(nv, rows, cols), ar.qtensor(nv, cols, rows)
    ref, ref_t = nv.QTensor(rows, cols), nv.QTensor(cols, rows)
    for o, ot in ((q, qt), (ref, ref_t)):
        nv.nvfp4_quantize_dual(d, a, nv.NVFP4_SR, 1, 2, o, mask, at, nv.NVFP4_SR, 3, 4, ot)
    _ok(nv)
    ar.check()
    _same_q(q, ref)
    _same_q(qt, ref_t)


@pytest.mark.parametrize("bf16", [False, True])
def test_red_zone_dequantize(nv, bf16):
    rows, k, ld = 200, 208, 216
    d = dev_bf16(_x(rows, k, 17))
    q = nv.QTensor(rows, k)
    nv.nvfp4_quantize_1d(d, nv.nvfp4_amax(d), nv.NVFP4_RNE, 0, 0, q)
    dt = torch.bfloat16 if bf16 else torch.float32
    ar = Arena()
    out = ar.take(((rows - 1) * ld + k) * (2 if bf16 else 4), dt)
    out2d = out.as_strided((rows, k), (ld, 1))
    ref = torch.empty((rows, k), dtype=dt, device="cuda")
    nv.nvfp4_dequantize(q, out2d)
    nv.nvfp4_dequantize(q, ref)
    _ok(nv)
    ar.check()
    assert torch.equal(out2d, ref)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("M,N,K", [(200, 200, 256), (136, 392, 320),
                                   # odd 128-row tile counts: the last CTA pair holds an empty tile
                                   (300, 136, 256), (72, 520, 96)])
def test_red_zone_gemm(nv, bf16, M, N, K):
    da, db = dev_bf16(_x(M, K, 19)), dev_bf16(_x(N, K, 23))
    qa, qb = nv.QTensor(M, K), nv.QTensor(N, K)
    nv.nvfp4_quantize_1d(da, nv.nvfp4_amax(da), nv.NVFP4_RNE, 0, 0, qa)
    nv.nvfp4_quantize_2d(db, nv.nvfp4_amax(db), nv.NVFP4_RNE, 0, 0, qb)
    dt = torch.bfloat16 if bf16 else torch.float32
    ldd = (N + 7) // 8 * 8 + 8
    ar = Arena()
    out = ar.take(((M - 1) * ldd + N) * (2 if bf16 else 4), dt).as_strided((M, N), (ldd, 1))
    ref = torch.empty((M, N), dtype=dt, device="cuda")
    nv.nvfp4_gemm(qa, qb, out)
    nv.nvfp4_gemm(qa, qb, ref)
    _ok(nv)
    ar.check()
    assert torch.equal(out, ref)


@pytest.mark.parametrize("mask", [0, MASK])
def test_red_zone_mx(nv, mask):
    M, N, K = 200, 136, 224
    da, db = dev_bf16(_x(M, K, 29)), dev_bf16(_x(N, K, 31))
    ar = Arena()
    qa, qb = ar.mx_qtensor(nv, M, K), ar.mx_qtensor(nv, N, K)
    ra, rb = nv.MxQTensor(M, K), nv.MxQTensor(N, K)
    for q, r, x in ((qa, ra, da), (qb, rb, db)):
        nv.nvfp4_mx_quantize(x, mask, q)
        nv.nvfp4_mx_quantize(x, mask, r)
    deq = ar.take(M * K * 4, torch.float32, (M, K))
    out = ar.take(M * N * 2, torch.bfloat16, (M, N))
    nv.nvfp4_mx_dequantize(qa, deq)
    nv.nvfp4_mx_gemm(qa, qb, out)
    ref_deq = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ref_out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_mx_dequantize(ra, ref_deq)
    nv.nvfp4_mx_gemm(ra, rb, ref_out)
    _ok(nv)
    ar.check()
    _same_q(qa, ra)
    _same_q(qb, rb)
    assert torch.equal(deq, ref_deq) and torch.equal(out, ref_out)


# ------------------------------------------------ the guarded build --------
def test_guarded_build_runs_the_parity_modules(nv):
    """The parity modules and this one, against libnvfp4_guarded.so in a child
    process: every test passes and no guard refuses an access."""
    if nv.GUARDED:
        pytest.skip("already running against the guarded build")
    from nvfp4_block_scaled_29_b300 import build
    if not os.path.exists(build.LIB_GUARDED):
        pytest.fail("libnvfp4_guarded.so is not built (build_all() builds it)")
    env = dict(os.environ, NVFP4_DEBUG_GUARDS="1")
    mods = ["tests/test_gpu_parity.py", "tests/test_gpu_dual.py", "tests/test_gpu_mx.py",
            "tests/test_gpu_linear.py", "tests/test_gpu_guards.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-rA", "-m", "gpu and not slow",
                        "-p", "no:cacheprovider", *mods], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=1800)
    report = "\n".join(l for l in r.stdout.splitlines() if not l.startswith("PASSED"))
    assert r.returncode == 0, report[-8000:] + r.stderr[-2000:]
    for name in ("test_guard_shrink_quantize_1d", "test_guard_shrink_quantize_2d", "test_guard_shrink_dual",
                 "test_guard_shrink_dequantize", "test_guard_shrink_gemm", "test_guard_shrink_amax",
                 "test_guard_shrink_quantize_1d_transposed_odd", "test_guard_shrink_mx"):
        assert f"PASSED tests/test_gpu_guards.py::{name}" in r.stdout, name


@pytest.fixture
def shrink(nv):
    if not nv.GUARDED:
        pytest.skip("runs against the guarded build (NVFP4_DEBUG_GUARDS=1)")
    assert nv.nvfp4_debug_guards_enabled()
    nv.nvfp4_get_status()
    nv.nvfp4_debug_guard_record()
    yield nv.nvfp4_debug_guard_shrink
    nv.nvfp4_debug_guard_shrink(0)
    nv.nvfp4_debug_guard_record()
    nv.nvfp4_get_status()


def _refused(nv, sites):
    torch.cuda.synchronize()
    rec = nv.nvfp4_debug_guard_record()
    assert rec is not None and rec[0] in sites, rec
    assert nv.nvfp4_get_status() == nv.NVFP4_ERR_GUARD
    return rec


def _tail_check(got, ref, n_tail):
    """got equals ref except its last n_tail bytes, which kept the canary."""
    g, r = got.reshape(-1).view(torch.uint8), ref.reshape(-1).view(torch.uint8)
    assert torch.equal(g[:-n_tail], r[:-n_tail])
    assert bool((g[-n_tail:] == CANARY).all())


def _canary_q(nv, rows, k, block2d=False):
    q = nv.QTensor(rows, k, block2d)
    q.codes.fill_(CANARY)
    q.scales.fill_(CANARY)
    return q


def test_guard_shrink_quantize_1d(nv, shrink):
    # [200 x 512]: the last row's last 32-byte code store and the last two
    # 4-byte scale words (rows 223 and 255 of the 128-row padding) reach into
    # the last 8 bytes
    d = dev_bf16(_x(200, 512, 41))
    amax = nv.nvfp4_amax(d)
    ref = nv.QTensor(200, 512)
    nv.nvfp4_quantize_1d(d, amax, nv.NVFP4_SR, 1, 1, ref)
    _ok(nv)
    q = _canary_q(nv, 200, 512)
    shrink(8)
    nv.nvfp4_quantize_1d(d, amax, nv.NVFP4_SR, 1, 1, q)
    _refused(nv, DUAL)
    _tail_check(q.codes, ref.codes, 32)
    _tail_check(q.scales, ref.scales, 8)


def test_guard_shrink_quantize_1d_transposed_odd(nv, shrink):
    # transposed view with an odd row count (the column-wise path of the
    # TMA-fed kernel, the last logical row paired with a padding row):
    # logical [199 x 512], stored [512 x 199] with ld 200.  The last 16-byte
    # code store (row 198, blocks 30-31) and the padding scale halves of rows
    # 223 and 255 reach into the last 8 bytes and are refused.
    x = _x(199, 512, 43)
    d = dev_bf16(x.T.copy(), 200)
    amax = nv.nvfp4_amax(d, transposed=True)
    ref = nv.QTensor(199, 512)
    nv.nvfp4_quantize_1d(d, amax, nv.NVFP4_SR, 3, 4, ref, transposed=True)
    _ok(nv)
    q = _canary_q(nv, 199, 512)
    shrink(8)
    nv.nvfp4_quantize_1d(d, amax, nv.NVFP4_SR, 3, 4, q, transposed=True)
    _refused(nv, DUAL)
    _tail_check(q.codes, ref.codes, 16)
    _tail_check(q.scales, ref.scales, 8)


def test_guard_shrink_quantize_2d(nv, shrink):
    d = dev_bf16(_x(208, 512, 47))
    amax = nv.nvfp4_amax(d)
    ref, ref_t = nv.QTensor(208, 512, True), nv.QTensor(512, 208, True)
    nv.nvfp4_quantize_2d(d, amax, nv.NVFP4_RNE, 0, 0, ref, ref_t)
    _ok(nv)
    q, qt = _canary_q(nv, 208, 512, True), _canary_q(nv, 512, 208, True)
    shrink(8)
    nv.nvfp4_quantize_2d(d, amax, nv.NVFP4_RNE, 0, 0, q, qt)
    _refused(nv, Q2D)
    _tail_check(q.codes, ref.codes, 32)
    _tail_check(q.scales, ref.scales, 8)
    _tail_check(qt.codes, ref_t.codes, 8)
    _tail_check(qt.scales, ref_t.scales, 8)


def test_guard_shrink_dual(nv, shrink):
    d = dev_bf16(_x(208, 512, 53))
    a, at = nv.nvfp4_amax_dual(d, MASK)
    ref, ref_t = nv.QTensor(208, 512), nv.QTensor(512, 208)
    nv.nvfp4_quantize_dual(d, a, nv.NVFP4_SR, 1, 2, ref, MASK, at, nv.NVFP4_SR, 3, 4, ref_t)
    _ok(nv)
    q, qt = _canary_q(nv, 208, 512), _canary_q(nv, 512, 208)
    shrink(8)
    nv.nvfp4_quantize_dual(d, a, nv.NVFP4_SR, 1, 2, q, MASK, at, nv.NVFP4_SR, 3, 4, qt)
    _refused(nv, DUAL)
    _tail_check(q.codes, ref.codes, 32)
    _tail_check(q.scales, ref.scales, 8)
    _tail_check(qt.codes, ref_t.codes, 8)          # k = 208: the last store is one 8-byte block
    _tail_check(qt.scales, ref_t.scales, 8)


def test_guard_shrink_dequantize(nv, shrink):
    # rows 200: the scale buffer's last 8 bytes are padding rows, never read.
    # The last two 4-byte code loads (row 199, elements 496..511) are refused
    # and read zeros; of the two 32-byte stores of those elements, the last
    # one reaches into the last 8 bytes and is refused.
    d = dev_bf16(_x(200, 512, 59))
    q = nv.QTensor(200, 512)
    nv.nvfp4_quantize_1d(d, nv.nvfp4_amax(d), nv.NVFP4_RNE, 0, 0, q)
    ref = torch.empty((200, 512), dtype=torch.float32, device="cuda")
    nv.nvfp4_dequantize(q, ref)
    _ok(nv)
    ref.view(-1)[-16:-8] = 0.0
    out = torch.empty_like(ref)
    out.view(torch.uint8).fill_(CANARY)
    shrink(8)
    nv.nvfp4_dequantize(q, out)
    _refused(nv, DEQ)
    _tail_check(out, ref, 32)


def test_guard_shrink_gemm(nv, shrink):
    # FP32 D [200 x 200] (plain-store epilogue): the last row's last chunk
    # (columns 192..199, 32 bytes) is refused
    da, db = dev_bf16(_x(200, 256, 61)), dev_bf16(_x(200, 256, 67))
    qa, qb = nv.QTensor(200, 256), nv.QTensor(200, 256)
    nv.nvfp4_quantize_1d(da, nv.nvfp4_amax(da), nv.NVFP4_RNE, 0, 0, qa)
    nv.nvfp4_quantize_1d(db, nv.nvfp4_amax(db), nv.NVFP4_RNE, 0, 0, qb)
    ref = torch.empty((200, 200), dtype=torch.float32, device="cuda")
    nv.nvfp4_gemm(qa, qb, ref)
    _ok(nv)
    out = torch.empty_like(ref)
    out.view(torch.uint8).fill_(CANARY)
    shrink(8)
    nv.nvfp4_gemm(qa, qb, out)
    assert _refused(nv, {GEMM_D}) == (GEMM_D, 200 * 200 * 4 - 32)
    _tail_check(out, ref, 32)


def test_guard_shrink_amax(nv, shrink):
    # contiguous x: the last 16-byte load (8 elements) reaches into the last
    # 8 bytes and is refused, so a maximum planted there is not seen
    x = _x(64, 256, 71)
    body = np.abs(synth.bf16_bits_to_f32(x).reshape(-1)[:-8]).max()
    x.reshape(-1)[-1] = 0x447A                      # bf16 1000.0
    d = dev_bf16(x)
    assert float(nv.nvfp4_amax(d).cpu()[0]) == 1000.0
    _ok(nv)
    shrink(8)
    got = float(nv.nvfp4_amax(d).cpu()[0])
    _refused(nv, {AMAX_X})
    assert got == float(body)


def test_guard_shrink_mx(nv, shrink):
    # [200 x 512]: the last row's last 128-byte load (columns 448..511) and
    # its 32-byte code store are refused, and the two blocks are encoded from
    # zeros (scale code 0); the last 8 scale bytes are padding rows 223, 255
    x = _x(200, 512, 73)
    d = dev_bf16(x)
    x_mod = x.copy()
    x_mod[199, 448:] = 0
    ref = nv.MxQTensor(200, 512)
    nv.nvfp4_mx_quantize(dev_bf16(x_mod), 0, ref)
    _ok(nv)
    q = nv.MxQTensor(200, 512)
    q.codes.fill_(CANARY)
    q.scales.fill_(CANARY)
    shrink(8)
    nv.nvfp4_mx_quantize(d, 0, q)
    _refused(nv, MX_Q)
    _tail_check(q.codes, ref.codes, 32)
    _tail_check(q.scales, ref.scales, 8)
