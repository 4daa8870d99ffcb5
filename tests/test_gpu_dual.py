"""Dual-axis calls vs the CPU oracle: one read of a stored tensor S [R x C]
gives the row-wise 1x16 operand S and the column-wise (optionally RHT) 1x16
operand S^T, each bit for bit what the oracle makes for that view; the dual
amax gives both views' amaxes exactly.

Shapes span several 128 x 256 tiles with ragged row and column tails (rows
and columns are multiples of 16, as the column-wise operand's k = R needs).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_q_equal, dev_bf16

pytestmark = pytest.mark.gpu

MASK = 0x9D2B
SHAPES = [(16, 16), (32, 48), (128, 256), (144, 272), (256, 528), (1040, 96), (64, 4096), (400, 784)]


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


def _data(rows, cols, seed, kind="normal"):
    if kind == "t":
        return synth.student_t_bf16((rows, cols), seed, 3, 1e-3)
    return synth.normal_bf16((rows, cols), seed, 1.0, 0.002, 60.0)


def _ld(cols):
    return ((cols + 7) // 8) * 8 + 8                      # a strided view with NaN padding


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("mask", [0, MASK])
def test_amax_dual(nv, rows, cols, mask):
    s = _data(rows, cols, 7 * rows + cols)
    d = dev_bf16(s, _ld(cols))
    a, at = nv.nvfp4_amax_dual(d, mask)
    torch.cuda.synchronize()
    assert float(a.cpu()[0]) == oracle.amax(s)
    assert float(at.cpu()[0]) == oracle.amax(s, transposed=True, rht_mask=mask)


def test_amax_dual_nonfinite(nv):
    s = _data(64, 96, 11)
    s[17, 40] = 0x7F80                                     # +Inf
    a, at = nv.nvfp4_amax_dual(dev_bf16(s), MASK)
    torch.cuda.synchronize()
    assert float(a.cpu()[0]) == float("inf")
    assert float(at.cpu()[0]) == oracle.amax(s, transposed=True, rht_mask=MASK) or \
        (np.isnan(float(at.cpu()[0])) and np.isnan(oracle.amax(s, transposed=True, rht_mask=MASK)))
    s[3, 3] = 0xFFC1                                       # NaN
    a, at = nv.nvfp4_amax_dual(dev_bf16(s), MASK)
    torch.cuda.synchronize()
    assert np.isnan(float(a.cpu()[0])) and np.isnan(float(at.cpu()[0]))


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("sr,sr_t,mask", [(False, False, MASK), (True, True, MASK), (False, True, 0),
                                           (True, False, 0)])
def test_quantize_dual(nv, rows, cols, sr, sr_t, mask):
    s = _data(rows, cols, 3000 + rows + cols, "t" if sr else "normal")
    d = dev_bf16(s, _ld(cols))
    a, at = nv.nvfp4_amax_dual(d, mask)
    q, qt = nv.QTensor(rows, cols), nv.QTensor(cols, rows)
    rnd = lambda b: nv.NVFP4_SR if b else nv.NVFP4_RNE
    nv.nvfp4_quantize_dual(d, a, rnd(sr), 91, 1, q, mask, at, rnd(sr_t), 92, 2, qt)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    ref = oracle.quantize(s, sr=sr, seed=91, stream_id=1)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, f"dual rows {rows}x{cols} sr={sr}")
    ref_t = oracle.quantize(s, transposed=True, rht_mask=mask, sr=sr_t, seed=92, stream_id=2)
    assert_q_equal(qt, ref_t.codes, ref_t.scales, ref_t.s_enc, f"dual cols {rows}x{cols} sr={sr_t} rht={mask}")


def test_quantize_dual_matches_separate_calls(nv):
    """The dual call and the two separate calls write identical bytes."""
    rows, cols = 384, 1280
    s = _data(rows, cols, 5, "t")
    d = dev_bf16(s)
    a, at = nv.nvfp4_amax_dual(d, MASK)
    q, qt = nv.QTensor(rows, cols), nv.QTensor(cols, rows)
    nv.nvfp4_quantize_dual(d, a, nv.NVFP4_SR, 5, 1, q, MASK, at, nv.NVFP4_SR, 5, 2, qt)
    q2, qt2 = nv.QTensor(rows, cols), nv.QTensor(cols, rows)
    nv.nvfp4_quantize_1d(d, a, nv.NVFP4_SR, 5, 1, q2)
    nv.nvfp4_rht_quantize(d, MASK, at, nv.NVFP4_SR, 5, 2, qt2, transposed=True)
    torch.cuda.synchronize()
    for x, y in ((q, q2), (qt, qt2)):
        assert torch.equal(x.codes, y.codes)
        assert torch.equal(x.scales, y.scales)
        assert torch.equal(x.global_scale, y.global_scale)


def test_quantize_dual_zero_tensor(nv):
    """amax = 0: S_enc = 1 and every code a zero.  The sign flip of the RHT
    turns +0 into -0, so the transformed operand holds sign-kept zeros (code
    0x8) exactly where the oracle puts them."""
    s = np.zeros((48, 80), np.uint16)
    d = dev_bf16(s)
    a, at = nv.nvfp4_amax_dual(d, MASK)
    q, qt = nv.QTensor(48, 80), nv.QTensor(80, 48)
    nv.nvfp4_quantize_dual(d, a, nv.NVFP4_SR, 1, 1, q, MASK, at, nv.NVFP4_RNE, 0, 0, qt)
    torch.cuda.synchronize()
    ref = oracle.quantize(s, sr=True, seed=1, stream_id=1)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "zero rows")
    ref_t = oracle.quantize(s, transposed=True, rht_mask=MASK)
    assert_q_equal(qt, ref_t.codes, ref_t.scales, ref_t.s_enc, "zero cols")
    for t, (r, k) in ((q, (48, 80)), (qt, (80, 48))):
        assert not (t.codes & 0x77).any()                  # magnitudes all zero
        assert not t.scales[:nv.nvfp4_scale_bytes(r, k)].any()
        assert float(t.global_scale.cpu()[0]) == 1.0


def test_quantize_dual_nonfinite_one_side(nv):
    """A non-finite amax stops only its own operand, publishes NaN for it and
    reports NVFP4_ERR_NONFINITE; the other operand is still exact."""
    s = _data(64, 64, 9)
    d = dev_bf16(s)
    a, at = nv.nvfp4_amax_dual(d, 0)
    at.fill_(float("inf"))
    q, qt = nv.QTensor(64, 64), nv.QTensor(64, 64)
    nv.nvfp4_quantize_dual(d, a, nv.NVFP4_RNE, 0, 0, q, 0, at, nv.NVFP4_RNE, 0, 0, qt)
    assert nv.nvfp4_get_status() == nv.NVFP4_ERR_NONFINITE
    ref = oracle.quantize(s)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "finite side")
    assert np.isnan(float(qt.global_scale.cpu()[0]))


def test_dual_rejects_bad_calls(nv):
    s = _data(40, 64, 1)                                   # rows % 16 != 0
    d = dev_bf16(s)
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_amax_dual(d, MASK)
    q, qt = nv.QTensor(40, 64), nv.QTensor(64, 40)
    a = torch.ones(1, device="cuda")
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_quantize_dual(d, a, 0, 0, 0, q, 0, a.clone(), 0, 0, 0, qt)


def test_quantize_dual_many_tiles_per_cta(nv):
    """1024 x 16384: 1024 tiles of 64 x 256, several per persistent CTA, so the
    shared-memory ring wraps; SR on both sides and RHT on the column side."""
    rows, cols = 1024, 16384
    s = _data(rows, cols, 77, "t")
    d = dev_bf16(s)
    a, at = nv.nvfp4_amax_dual(d, MASK)
    q, qt = nv.QTensor(rows, cols), nv.QTensor(cols, rows)
    nv.nvfp4_quantize_dual(d, a, nv.NVFP4_SR, 17, 1, q, MASK, at, nv.NVFP4_SR, 17, 2, qt)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    ref = oracle.quantize(s, sr=True, seed=17, stream_id=1)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "dual rows, many tiles")
    ref_t = oracle.quantize(s, transposed=True, rht_mask=MASK, sr=True, seed=17, stream_id=2)
    assert_q_equal(qt, ref_t.codes, ref_t.scales, ref_t.s_enc, "dual cols, many tiles")


@pytest.mark.parametrize("hw", [False, True])
def test_quantize_dual_wide_seed_and_stream(nv, hw):
    """Seeds and Philox stream ids with both 32-bit words set: the kernels fold
    the counter's stream words and the first keys into constants made on the
    host, so every word of the key and of the counter must reach the draws."""
    rows, cols = 256, 528
    s = _data(rows, cols, 41, "t")
    d = dev_bf16(s)
    seed, sid, seed_t, sid_t = 0xDEADBEEF12345678, 0x123456789ABCDEF0, 0x0F1E2D3C4B5A6978, 0xFEDCBA9876543210
    a, at = nv.nvfp4_amax_dual(d, MASK)
    q, qt = nv.QTensor(rows, cols), nv.QTensor(cols, rows)
    rnd = nv.NVFP4_SR_HW if hw else nv.NVFP4_SR
    nv.nvfp4_quantize_dual(d, a, rnd, seed, sid, q, MASK, at, rnd, seed_t, sid_t, qt)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    ref = oracle.quantize(s, sr=True, seed=seed, stream_id=sid, sr_hw=hw)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "wide seed rows")
    ref_t = oracle.quantize(s, transposed=True, rht_mask=MASK, sr=True, seed=seed_t, stream_id=sid_t, sr_hw=hw)
    assert_q_equal(qt, ref_t.codes, ref_t.scales, ref_t.s_enc, "wide seed cols")


@pytest.mark.parametrize("rnd_name", ["NVFP4_SR", "NVFP4_SR_HW", "NVFP4_RNE"])
def test_quantize_dual_general_index_path(nv, rnd_name):
    """The path for Philox block indices of 64 bits (taken only for operands of
    more than 2^35 elements) writes the same bytes as the 32-bit-index path;
    the test-only injection mode 2 makes one call take it on a small tensor."""
    rows, cols = 384, 1280
    s = _data(rows, cols, 43, "t")
    d = dev_bf16(s)
    rnd = getattr(nv, rnd_name)
    a, at = nv.nvfp4_amax_dual(d, MASK)
    outs = []
    for force in (False, True):
        q, qt = nv.QTensor(rows, cols), nv.QTensor(cols, rows)
        if force:
            nv.nvfp4_debug_inject(2)
        nv.nvfp4_quantize_dual(d, a, rnd, 7, 3, q, MASK, at, rnd, 8, 4, qt)
        torch.cuda.synchronize()
        assert nv.nvfp4_get_status() == nv.NVFP4_OK
        outs.append((q, qt))
    for x, y in zip(outs[0], outs[1]):
        assert torch.equal(x.codes, y.codes) and torch.equal(x.scales, y.scales)
    ref = oracle.quantize(s, sr=rnd != nv.NVFP4_RNE, seed=7, stream_id=3, sr_hw=rnd == nv.NVFP4_SR_HW)
    assert_q_equal(outs[1][0], ref.codes, ref.scales, ref.s_enc, "general path rows")
