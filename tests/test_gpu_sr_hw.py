"""Rounding mode NVFP4_SR_HW vs the CPU oracle: stochastic rounding with the
random bits in the layout of the hardware FP4 stochastic-rounding conversion
(32 Philox bits per 4 elements), through every quantise call that takes a
rounding mode.  Bit-exact, like NVFP4_SR.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import assert_q_equal, dev_bf16, expected_transpose, gpu_quantize

pytestmark = pytest.mark.gpu

MASK = 0x9D2B


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


@pytest.mark.parametrize("rows,k", [(16, 16), (100, 80), (130, 272), (257, 1040), (64, 4096)])
@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("mask", [0, MASK])
def test_quantize_1d_sr_hw(nv, rows, k, transposed, mask):
    if transposed and rows % 16:
        pytest.skip("a transposed view needs rows % 16 == 0 (its stored k)")
    x = synth.student_t_bf16((k, rows) if transposed else (rows, k), 500 + rows + k, 3, 1e-3)
    q, _, _ = gpu_quantize(nv, dev_bf16(x), transposed=transposed, mask=mask, sr=True, sr_hw=True, seed=41, sid=3)
    ref = oracle.quantize(x, transposed=transposed, rht_mask=mask, sr=True, sr_hw=True, seed=41, stream_id=3)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, f"1d sr_hw {rows}x{k} t={transposed} rht={mask}")


@pytest.mark.parametrize("rows,k", [(16, 16), (48, 80), (144, 272), (4096, 4096)])
@pytest.mark.parametrize("emit_t", [False, True])
def test_quantize_2d_sr_hw(nv, rows, k, emit_t):
    w = synth.normal_bf16((rows, k), 2100 + rows + k, 0.02)
    q, qt, _ = gpu_quantize(nv, dev_bf16(w, k + 8), block2d=True, sr=True, sr_hw=True, seed=9, sid=2,
                            emit_t=emit_t)
    ref = oracle.quantize(w, block2d=True, sr=True, sr_hw=True, seed=9, stream_id=2)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, f"2d sr_hw {rows}x{k}")
    if emit_t:
        codes_t, scales_t = expected_transpose(ref)
        assert_q_equal(qt, codes_t, scales_t, ref.s_enc, f"2d-T sr_hw {rows}x{k}")


def test_quantize_2d_transposed_view_sr_hw(nv):
    """A transposed view indexes the random bits in the view's logical layout."""
    stored = synth.normal_bf16((96, 64), 77, 0.02)
    q, qt, _ = gpu_quantize(nv, dev_bf16(stored), transposed=True, block2d=True, sr=True, sr_hw=True, seed=4,
                            emit_t=True)
    ref = oracle.quantize(stored, transposed=True, block2d=True, sr=True, sr_hw=True, seed=4)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "2d transposed view sr_hw")
    codes_t, scales_t = expected_transpose(ref)
    assert_q_equal(qt, codes_t, scales_t, ref.s_enc, "2d transposed view sr_hw, out_t")


@pytest.mark.parametrize("rows,cols", [(16, 16), (144, 272), (400, 784), (1024, 16384)])
@pytest.mark.parametrize("modes", [("hw", "hw"), ("sw", "hw"), ("hw", "rne")])
def test_quantize_dual_sr_hw(nv, rows, cols, modes):
    s = synth.student_t_bf16((rows, cols), 3300 + rows + cols, 3, 1e-3)
    d = dev_bf16(s)
    a, at = nv.nvfp4_amax_dual(d, MASK)
    q, qt = nv.QTensor(rows, cols), nv.QTensor(cols, rows)
    code = {"hw": nv.NVFP4_SR_HW, "sw": nv.NVFP4_SR, "rne": nv.NVFP4_RNE}
    nv.nvfp4_quantize_dual(d, a, code[modes[0]], 91, 1, q, MASK, at, code[modes[1]], 92, 2, qt)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    kw = lambda m: dict(sr=m != "rne", sr_hw=m == "hw")
    ref = oracle.quantize(s, seed=91, stream_id=1, **kw(modes[0]))
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, f"dual rows {rows}x{cols} {modes[0]}")
    ref_t = oracle.quantize(s, transposed=True, rht_mask=MASK, seed=92, stream_id=2, **kw(modes[1]))
    assert_q_equal(qt, ref_t.codes, ref_t.scales, ref_t.s_enc, f"dual cols {rows}x{cols} {modes[1]}")


def test_sr_hw_differs_from_sr(nv):
    """The two layouts draw different bits: same input, same seed, different codes."""
    x = synth.student_t_bf16((128, 256), 5, 3, 1e-3)
    q1, _, _ = gpu_quantize(nv, dev_bf16(x), sr=True, seed=7, sid=1)
    q2, _, _ = gpu_quantize(nv, dev_bf16(x), sr=True, sr_hw=True, seed=7, sid=1)
    assert not torch.equal(q1.codes, q2.codes)
    assert torch.equal(q1.scales, q2.scales)
