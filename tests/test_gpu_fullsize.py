"""Parity at the full 12B-hybrid FFN shapes, in the launch sequence bench.py
times: forward (X 8192x5120 1x16 RNE, W 20480x5120 16x16 with W^T, Y bf16),
dgrad (dY 8192x20480 1x16 SR, dX bf16) and wgrad (RHT-16 along the 8192
tokens, dY^T SR and X^T RNE read transposed, dW bf16).

The oracle cannot quantise 168M elements per case in test time, so codes and
scales are compared bit for bit on sampled row ranges (aligned to 16 for the
16x16 weight) after the oracle has computed the exact full-tensor amax; the
GEMMs are compared on 2^14 random output points plus two full 128x128 tiles,
each an exact FP64 dot product over the whole k.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import check_sampled as _check_sampled, dev_bf16, gemm_bound_check, sample_ranges as _ranges

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOK, HID, FFN = synth.TOKENS, synth.HIDDEN, synth.FFN
SR_SEED, RHT_SEED = 1003, 2004


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


@pytest.fixture(scope="module")
def step(nv):
    """Run one full step through the C ABI, keep host copies of what the
    checks need."""
    x = synth.activations(2)
    w = synth.weights(3)
    dy = synth.grad_output(3 + 7919)
    dx_, dw_, ddy = dev_bf16(x), dev_bf16(w), dev_bf16(dy)
    Q = nv.QTensor
    qx, qw, qwt = Q(TOK, HID), Q(FFN, HID, True), Q(HID, FFN, True)
    qdy, qdyt, qxt = Q(TOK, FFN), Q(FFN, TOK), Q(HID, TOK)
    mask = nv.nvfp4_rht_mask_from_seed(RHT_SEED)
    a = torch.empty((8,), dtype=torch.float32, device="cuda")
    rne, sr = nv.NVFP4_RNE, nv.NVFP4_SR
    y = torch.empty((TOK, FFN), dtype=torch.bfloat16, device="cuda")
    dxo = torch.empty((TOK, HID), dtype=torch.bfloat16, device="cuda")
    dwo = torch.empty((FFN, HID), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_amax(dx_, 0, a[0:1])
    nv.nvfp4_quantize_1d(dx_, a[0:1], rne, 0, 0, qx)
    nv.nvfp4_amax(dw_, 0, a[1:2])
    nv.nvfp4_quantize_2d(dw_, a[1:2], rne, 0, 0, qw, qwt)
    nv.nvfp4_gemm(qx, qw, y)
    nv.nvfp4_amax(ddy, 0, a[2:3])
    nv.nvfp4_quantize_1d(ddy, a[2:3], sr, SR_SEED, 1, qdy)
    nv.nvfp4_gemm(qdy, qwt, dxo)
    nv.nvfp4_amax(ddy, mask, a[3:4], transposed=True)
    nv.nvfp4_rht_quantize(ddy, mask, a[3:4], sr, SR_SEED, 2, qdyt, transposed=True)
    nv.nvfp4_amax(dx_, mask, a[4:5], transposed=True)
    nv.nvfp4_rht_quantize(dx_, mask, a[4:5], rne, 0, 0, qxt, transposed=True)
    nv.nvfp4_gemm(qdyt, qxt, dwo)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    host = lambda q: (q.codes.cpu().numpy(), q.scales.cpu().numpy(), float(q.global_scale.cpu()[0]))
    out = {"x": x, "w": w, "dy": dy, "mask": mask, "amax": a.cpu().numpy(),
           "qx": host(qx), "qw": host(qw), "qwt": host(qwt), "qdy": host(qdy), "qdyt": host(qdyt),
           "qxt": host(qxt), "y": y.float().cpu().numpy(), "dx": dxo.float().cpu().numpy(),
           "dw": dwo.float().cpu().numpy()}
    return out


def test_amax_values(step):
    s = step
    assert s["amax"][0] == oracle.amax(s["x"])
    assert s["amax"][1] == oracle.amax(s["w"])
    assert s["amax"][2] == oracle.amax(s["dy"])
    assert s["amax"][3] == oracle.amax(s["dy"], transposed=True, rht_mask=s["mask"])
    assert s["amax"][4] == oracle.amax(s["x"], transposed=True, rht_mask=s["mask"])


def test_forward_quantisation(step):
    s = step
    rx = _ranges(TOK, 3, 24, 1, 1)
    ref = oracle.quantize(s["x"], amax_v=float(s["amax"][0]), ranges=rx, swizzle=False)
    _check_sampled(s["qx"], ref, rx, TOK, HID, "X")
    rw = _ranges(FFN, 3, 32, 16, 2)
    ref = oracle.quantize(s["w"], block2d=True, amax_v=float(s["amax"][1]), ranges=rw, swizzle=False)
    _check_sampled(s["qw"], ref, rw, FFN, HID, "W")
    # W^T: rows of W^T are k indices of W; check sampled rows against the
    # oracle's 16x16 quantisation of the transposed view (RNE: identical)
    rwt = _ranges(HID, 2, 32, 16, 3)
    ref = oracle.quantize(s["w"], block2d=True, transposed=True, amax_v=float(s["amax"][1]), ranges=rwt,
                          swizzle=False)
    _check_sampled(s["qwt"], ref, rwt, HID, FFN, "W^T")


def test_dgrad_quantisation(step):
    s = step
    r = _ranges(TOK, 3, 16, 1, 4)
    ref = oracle.quantize(s["dy"], amax_v=float(s["amax"][2]), sr=True, seed=SR_SEED, stream_id=1, ranges=r,
                          swizzle=False)
    _check_sampled(s["qdy"], ref, r, TOK, FFN, "dY")


def test_wgrad_quantisation(step):
    s = step
    r = _ranges(FFN, 3, 16, 1, 5)
    ref = oracle.quantize(s["dy"], transposed=True, rht_mask=s["mask"], amax_v=float(s["amax"][3]), sr=True,
                          seed=SR_SEED, stream_id=2, ranges=r, swizzle=False)
    _check_sampled(s["qdyt"], ref, r, FFN, TOK, "dY^T")
    r = _ranges(HID, 3, 16, 1, 6)
    ref = oracle.quantize(s["x"], transposed=True, rht_mask=s["mask"], amax_v=float(s["amax"][4]), ranges=r,
                          swizzle=False)
    _check_sampled(s["qxt"], ref, r, HID, TOK, "X^T")


def _gemm_points(qa, qb, M, N, K, y, seed, what):
    rng = np.random.default_rng(seed)
    ms = rng.integers(0, M, 1 << 14)
    ns = rng.integers(0, N, 1 << 14)
    tiles = [(0, 0), ((M // 128 - 1) * 128, (N // 128 - 1) * 128)]
    for m0, n0 in tiles:
        mm, nn = np.meshgrid(np.arange(m0, m0 + 128), np.arange(n0, n0 + 128), indexing="ij")
        ms = np.concatenate([ms, mm.ravel()])
        ns = np.concatenate([ns, nn.ravel()])
    yr, ab = oracle.gemm_points(qa[0], qa[1], qa[2], qb[0], qb[1], qb[2], M, N, K, ms, ns)
    gemm_bound_check(y[ms, ns], yr, ab, True, what)


def test_forward_gemm(step):
    s = step
    _gemm_points(s["qx"], s["qw"], TOK, FFN, HID, s["y"], 7, "Y = X W^T")


def test_dgrad_gemm(step):
    s = step
    _gemm_points(s["qdy"], s["qwt"], TOK, HID, FFN, s["dx"], 8, "dX = dY W")


def test_wgrad_gemm(step):
    s = step
    _gemm_points(s["qdyt"], s["qxt"], FFN, HID, TOK, s["dw"], 9, "dW = dY^T X")


def test_dual_axis_path_matches(step, nv):
    """The dual-axis calls on the full-size X and dY write exactly the bytes
    of the separate calls above (which are checked against the oracle)."""
    s = step
    dx_, ddy = dev_bf16(s["x"]), dev_bf16(s["dy"])
    Q = nv.QTensor
    a = torch.zeros((4,), dtype=torch.float32, device="cuda")
    qx, qxt, qdy, qdyt = Q(TOK, HID), Q(HID, TOK), Q(TOK, FFN), Q(FFN, TOK)
    nv.nvfp4_amax_dual(dx_, s["mask"], a[0:1], a[1:2])
    nv.nvfp4_quantize_dual(dx_, a[0:1], nv.NVFP4_RNE, 0, 0, qx, s["mask"], a[1:2], nv.NVFP4_RNE, 0, 0, qxt)
    nv.nvfp4_amax_dual(ddy, s["mask"], a[2:3], a[3:4])
    nv.nvfp4_quantize_dual(ddy, a[2:3], nv.NVFP4_SR, SR_SEED, 1, qdy, s["mask"], a[3:4], nv.NVFP4_SR, SR_SEED, 2,
                           qdyt)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    am = a.cpu().numpy()
    assert am[0] == s["amax"][0] and am[1] == s["amax"][4]
    assert am[2] == s["amax"][2] and am[3] == s["amax"][3]
    for got, key in ((qx, "qx"), (qxt, "qxt"), (qdy, "qdy"), (qdyt, "qdyt")):
        codes, scales, gs = s[key]
        assert np.array_equal(got.codes.cpu().numpy(), codes), key
        assert np.array_equal(got.scales.cpu().numpy(), scales), key
        assert float(got.global_scale.cpu()[0]) == gs, key
