"""MXFP4 (32-element blocks, E8M0 scales) on the GPU vs the CPU oracle:
quantisation and dequantisation bit-exact, the kind::mxf4 GEMM within
|y - y_ref| <= 2e-5 * sum_k |a_k b_k| (FP32 out; BF16 out adds its rounding)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev_bf16, gemm_bound_check

pytestmark = pytest.mark.gpu
MASK = 0x9D2B


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


def _mx(nv, x_dev, mask=0):
    r, k = x_dev.shape
    q = nv.MxQTensor(r, k)
    nv.nvfp4_mx_quantize(x_dev, mask, q)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    return q


@pytest.mark.parametrize("rows,k", [(1, 32), (3, 96), (130, 288), (257, 1056), (64, 4096)])
@pytest.mark.parametrize("mask", [0, MASK])
def test_mx_quantize(nv, rows, k, mask):
    x = synth.normal_bf16((rows, k), 50 + rows + k, 1.0, 0.002, 60.0)
    ld = k + 8
    q = _mx(nv, dev_bf16(x, ld), mask)
    ref = oracle.mx_quantize(x, rht_mask=mask)
    assert np.array_equal(q.codes.cpu().numpy(), ref.codes)
    assert np.array_equal(q.scales.cpu().numpy()[:ref.scales.size], ref.scales)


def test_mx_dequantize(nv):
    x = synth.student_t_bf16((200, 320), 9, 3, 1e-3)
    q = _mx(nv, dev_bf16(x))
    out = torch.empty((200, 320), dtype=torch.float32, device="cuda")
    nv.nvfp4_mx_dequantize(q, out)
    torch.cuda.synchronize()
    ref = oracle.mx_dequantize(oracle.mx_quantize(x))
    assert np.array_equal(out.cpu().numpy(), ref)


def test_mx_nonfinite_block_is_reported(nv):
    x = synth.normal_bf16((32, 64), 3, 1.0, 0.0, 1.0)
    x[5, 40] = 0x7FC1
    q = nv.MxQTensor(32, 64)
    nv.nvfp4_mx_quantize(dev_bf16(x), 0, q)
    assert nv.nvfp4_get_status() == nv.NVFP4_ERR_NONFINITE
    plain = oracle.mx_unswizzle_scales(q.scales.cpu().numpy(), 32, 64)
    assert plain[5, 1] == 0xFF


def _upload_mx(nv, codes, scales_plain, rows, k):
    q = nv.MxQTensor(rows, k)
    q.codes.copy_(torch.from_numpy(codes))
    swz = oracle.mx_swizzle_scales(scales_plain, rows, k)
    q.scales[:swz.size].copy_(torch.from_numpy(swz))
    return q, swz


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (200, 300, 96), (130, 260, 320),
                                   (512, 512, 512), (1024, 768, 1280), (2048, 256, 512), (1, 1, 32)])
@pytest.mark.parametrize("bf16", [False, True])
def test_mx_gemm(nv, M, N, K, bf16):
    xa = synth.normal_bf16((M, K), M + K, 1.0, 0.002, 60.0)
    xb = synth.normal_bf16((N, K), N + 3 * K, 0.02, 0.0, 1.0)
    ga, gb = _mx(nv, dev_bf16(xa)), _mx(nv, dev_bf16(xb))
    qa, qb = oracle.mx_quantize(xa), oracle.mx_quantize(xb)
    d = torch.empty((M, ((N + 7) // 8) * 8 + 8), dtype=torch.bfloat16 if bf16 else torch.float32,
                    device="cuda")[:, :N]
    d.fill_(float("nan"))
    nv.nvfp4_mx_gemm(ga, gb, d)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    y_ref, ab = oracle.mx_gemm_full(qa.codes, qa.scales, qb.codes, qb.scales, M, N, K)
    gemm_bound_check(d.float().cpu().numpy(), y_ref, ab, bf16, f"mx gemm {M}x{N}x{K} bf16={bf16}")


def test_mx_gemm_integer_exact(nv):
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 512
    pick = np.array([0, 2, 10], np.uint8)
    av, bv = rng.integers(0, 3, (M, K)), rng.integers(0, 3, (N, K))
    pack = lambda v: (pick[v[:, 0::2]] | (pick[v[:, 1::2]] << 4)).astype(np.uint8)
    ga, _ = _upload_mx(nv, pack(av), np.full((M, K // 32), 127, np.uint8), M, K)
    gb, _ = _upload_mx(nv, pack(bv), np.full((N, K // 32), 127, np.uint8), N, K)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nv.nvfp4_mx_gemm(ga, gb, d)
    torch.cuda.synchronize()
    sv = np.array([0, 1, -1])
    np.testing.assert_array_equal(d.cpu().numpy(), (sv[av] @ sv[bv].T).astype(np.float32))


def test_mx_gemm_per_block_scales(nv):
    """Every 32-block of A and B carries its own power of two: a wrong byte
    of the scale words (the two MMAs that share one) shows up in D."""
    rng = np.random.default_rng(6)
    M, N, K = 256, 256, 512
    ca = np.full((M, K // 2), 0x22, np.uint8)                 # all elements 1.0
    cb = np.full((N, K // 2), 0x22, np.uint8)
    sa = rng.integers(120, 135, (M, K // 32)).astype(np.uint8)
    sb = rng.integers(120, 135, (N, K // 32)).astype(np.uint8)
    ga, swa = _upload_mx(nv, ca, sa, M, K)
    gb, swb = _upload_mx(nv, cb, sb, N, K)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nv.nvfp4_mx_gemm(ga, gb, d)
    torch.cuda.synchronize()
    y_ref, ab = oracle.mx_gemm_full(ca, swa, cb, swb, M, N, K)
    gemm_bound_check(d.cpu().numpy(), y_ref, ab, False, "mx per-block scales")
