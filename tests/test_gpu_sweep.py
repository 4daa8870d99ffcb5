"""Quantise-only sweep: bf16 tensors of n = 2^20 ... 2^30 elements shaped
[n/8192 x 8192] (k = 8192), drawn as Student-t(3) (unscaled) and as N(0,1)
with 0.05% of the entries x100, each quantised in every combination of
{1x16, 16x16 blocks} x {RNE, stochastic (NVFP4_SR)} x {no RHT, RHT-16}.

The amax is compared exactly.  The oracle cannot quantise 2^28 elements per
case in test time, so codes and scales are compared bit for bit on sampled
row ranges (aligned to 16), with the full tensor's amax.  Sizes up to 2^28
are drawn on the host (numpy); 2^29 and 2^30 are drawn on the device by the
seeded device generators (the host ones take minutes there) and copied to
the host for the oracle.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import check_sampled, dev_bf16, sample_ranges

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

K = 8192
SIZES = [1 << 20, 1 << 23, 1 << 26, 1 << 28]
MASK = 0x9D2B


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


def sweep_tensor(n: int, dist: str) -> np.ndarray:
    rows, seed = n // K, n.bit_length()
    if dist == "t3":
        return synth.student_t_bf16((rows, K), seed, 3, 1.0)
    return synth.normal_bf16((rows, K), seed + 100, 1.0, 0.0005, 100.0)


def quantise_point(nv, d, rows, block2d, sr, mask, seed):
    """One sweep point through the C ABI: amax, then the quantiser of that
    mode.  Returns (amax, (codes, swizzled scales, S_enc)) on the host."""
    amax = nv.nvfp4_amax(d, mask)
    q = nv.QTensor(rows, K, block2d)
    rnd = nv.NVFP4_SR if sr else nv.NVFP4_RNE
    if mask:
        nv.nvfp4_rht_quantize(d, mask, amax, rnd, seed, 1, q)
    elif block2d:
        nv.nvfp4_quantize_2d(d, amax, rnd, seed, 1, q)
    else:
        nv.nvfp4_quantize_1d(d, amax, rnd, seed, 1, q)
    torch.cuda.synchronize()
    st = nv.nvfp4_get_status()
    assert st == nv.NVFP4_OK, nv.status_string(st)
    return float(amax.cpu()[0]), (q.codes.cpu().numpy(), q.scales.cpu().numpy(), float(q.global_scale.cpu()[0]))


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("dist", ["t3", "normal_outliers"])
def test_sweep_point(nv, n, dist):
    x = sweep_tensor(n, dist)
    rows = n // K
    d = dev_bf16(x)
    ref_amax = {m: oracle.amax(x, rht_mask=m) for m in (0, MASK)}
    for block2d, sr, mask in itertools.product((False, True), (False, True), (0, MASK)):
        what = f"n=2^{n.bit_length() - 1} {dist} {'16x16' if block2d else '1x16'} {'SR' if sr else 'RNE'} " \
               f"rht={mask:#x}"
        seed = 1000 + n.bit_length()
        amax, got = quantise_point(nv, d, rows, block2d, sr, mask, seed)
        assert amax == ref_amax[mask], what
        r = sample_ranges(rows, 3, 16, 16, n.bit_length() + int(block2d) + 2 * int(sr))
        ref = oracle.quantize(x, block2d=block2d, rht_mask=mask, amax_v=amax, sr=sr, seed=seed, stream_id=1,
                              ranges=r, swizzle=False)
        check_sampled(got, ref, r, rows, K, what)


LARGE = [1 << 29, 1 << 30]


@pytest.mark.parametrize("n", LARGE)
@pytest.mark.parametrize("dist", ["t3", "normal_outliers"])
def test_sweep_point_large(nv, n, dist):
    rows, seed = n // K, n.bit_length()
    d = (synth.student_t_bf16_device((rows, K), seed, 1.0) if dist == "t3"
         else synth.normal_bf16_device((rows, K), seed + 100, 1.0, 0.0005, 100.0))
    x = d.view(torch.int16).cpu().numpy().view(np.uint16)
    ref_amax = {m: oracle.amax(x, rht_mask=m) for m in (0, MASK)}
    for block2d, sr, mask in itertools.product((False, True), (False, True), (0, MASK)):
        what = f"n=2^{n.bit_length() - 1} {dist} {'16x16' if block2d else '1x16'} {'SR' if sr else 'RNE'} " \
               f"rht={mask:#x}"
        qseed = 1000 + n.bit_length()
        amax, got = quantise_point(nv, d, rows, block2d, sr, mask, qseed)
        assert amax == ref_amax[mask], what
        r = sample_ranges(rows, 3, 16, 16, n.bit_length() + int(block2d) + 2 * int(sr))
        ref = oracle.quantize(x, block2d=block2d, rht_mask=mask, amax_v=amax, sr=sr, seed=qseed, stream_id=1,
                              ranges=r, swizzle=False)
        check_sampled(got, ref, r, rows, K, what)
