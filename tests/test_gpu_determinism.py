"""Run-to-run reproducibility of the GPU path.

The oracle tests fix what each call computes; these fix that it computes it
the same way every time.  The block-scaled GEMM sums each output tile's k
blocks in a fixed order inside one accumulator (no split-k, no atomics), so
repeated launches, with other work queued between them, write identical
bits.  The stochastic-rounding quantisers
draw their random bits from Philox keyed by (seed, element index, stream), so
a repeat gives identical codes and another seed or stream changes them.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev_bf16, gpu_quantize

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


def _operand(nv, rows, k, seed, s_enc):
    codes, scales = synth.random_operand(rows, k, seed)
    q = nv.QTensor(rows, k)
    q.codes.copy_(torch.from_numpy(codes))
    q.scales.copy_(torch.from_numpy(oracle.swizzle_scales(scales, rows, k)))
    q.global_scale.fill_(float(s_enc))
    return q


@pytest.mark.parametrize("M,N,K", [
    (300, 520, 320),        # odd count of 128-row tiles, ragged N and k
    (2048, 4096, 2048),     # many tiles per CTA pair (persistent walk)
])
@pytest.mark.parametrize("bf16", [False, True])
def test_gemm_repeats_bit_identical(nv, M, N, K, bf16):
    qa = _operand(nv, M, K, M + 3 * K, 1.75)
    qb = _operand(nv, N, K, N + 5 * K, 0.625)
    dt = torch.bfloat16 if bf16 else torch.float32
    outs = []
    for rep in range(3):
        d = torch.full((M, N), float("nan"), dtype=dt, device="cuda")
        if rep == 2:
            # other work queued in between: the walk and the order of the k
            # blocks per tile do not depend on it
            ld = ((M + 7) // 8) * 8                       # rows of the output start 16-byte aligned
            nv.nvfp4_gemm(qb, qa, torch.empty((N, ld), dtype=dt, device="cuda")[:, :M])
        nv.nvfp4_gemm(qa, qb, d)
        outs.append(d)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    assert not torch.isnan(outs[0].float()).any()
    for d in outs[1:]:
        assert torch.equal(d.view(torch.int16 if bf16 else torch.int32),
                           outs[0].view(torch.int16 if bf16 else torch.int32))


@pytest.mark.parametrize("block2d", [False, True])
def test_stochastic_rounding_repeats_and_seeds(nv, block2d):
    x = dev_bf16(synth.student_t_bf16((256, 512), 11, 3, 1e-3))
    a, _, _ = gpu_quantize(nv, x, block2d=block2d, sr=True, seed=12345, sid=1)
    b, _, _ = gpu_quantize(nv, x, block2d=block2d, sr=True, seed=12345, sid=1)
    c, _, _ = gpu_quantize(nv, x, block2d=block2d, sr=True, seed=12346, sid=1)
    d, _, _ = gpu_quantize(nv, x, block2d=block2d, sr=True, seed=12345, sid=2)
    assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
    # the scales do not depend on the random bits; the codes do
    assert torch.equal(a.scales, c.scales) and torch.equal(a.scales, d.scales)
    for other in (c, d):
        frac = (a.codes != other.codes).float().mean().item()
        assert 0.05 < frac < 0.95, frac


def test_dual_quantise_repeats(nv):
    x = dev_bf16(synth.student_t_bf16((256, 1024), 13, 3, 1e-3))
    mask = 0x6A5C
    amax = nv.nvfp4_amax(x)
    amax_t = nv.nvfp4_amax(x, mask, transposed=True)
    res = []
    for _ in range(2):
        q, qt = nv.QTensor(256, 1024), nv.QTensor(1024, 256)
        nv.nvfp4_quantize_dual(x, amax, nv.NVFP4_SR, 99, 1, q, mask, amax_t, nv.NVFP4_SR, 99, 2, qt)
        res.append((q, qt))
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    for t0, t1 in zip(res[0], res[1]):
        assert torch.equal(t0.codes, t1.codes) and torch.equal(t0.scales, t1.scales)
