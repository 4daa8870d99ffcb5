"""GPU path vs CPU oracle on the same seeded inputs, element by element.

Sizes span several tiles and ragged tails; quantised codes and scales must
be bit-exact, GEMM outputs within |y - y_ref| <= 2e-5 * sum_k |a_k b_k|.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (assert_q_equal, dev_bf16, expected_transpose, gemm_bound_check,
                      gpu_quantize)

pytestmark = pytest.mark.gpu

MASK = 0x9D2B


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


def _data(rows, k, seed, kind="normal"):
    if kind == "t":
        return synth.student_t_bf16((rows, k), seed, 3, 1e-3)
    return synth.normal_bf16((rows, k), seed, 1.0, 0.002, 60.0)


# ------------------------------------------------------------------- amax --
@pytest.mark.parametrize("rows,k", [(1, 16), (7, 48), (130, 272), (512, 1024), (3, 4096)])
@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("mask", [0, MASK])
def test_amax(nv, rows, k, transposed, mask):
    x = _data(rows, k, rows * 31 + k)
    stored = x.T.copy() if transposed else x                 # stored array of the view
    ld = ((stored.shape[1] + 7) // 8) * 8 + (8 if rows % 2 else 0)
    d = dev_bf16(stored, ld)
    a = nv.nvfp4_amax(d, mask, transposed=transposed)
    torch.cuda.synchronize()
    assert float(a.cpu()[0]) == oracle.amax(stored, transposed=transposed, rht_mask=mask)


def test_amax_nan_and_inf(nv):
    x = _data(64, 64, 5)
    x[10, 17] = 0x7F80                                        # +Inf
    a = nv.nvfp4_amax(dev_bf16(x))
    assert float(a.cpu()[0]) == float("inf")
    x[3, 3] = 0xFFC1                                          # NaN
    a = nv.nvfp4_amax(dev_bf16(x))
    assert np.isnan(float(a.cpu()[0]))


def test_nonfinite_amax_is_reported(nv):
    x = _data(32, 64, 6)
    x[1, 1] = 0x7F80
    d = dev_bf16(x)
    q = nv.QTensor(32, 64)
    a = nv.nvfp4_amax(d)
    nv.nvfp4_quantize_1d(d, a, nv.NVFP4_RNE, 0, 0, q)
    assert nv.nvfp4_get_status() == nv.NVFP4_ERR_NONFINITE
    assert nv.nvfp4_get_status() == nv.NVFP4_OK                # read clears it
    assert np.isnan(float(q.global_scale.cpu()[0]))


# ------------------------------------------------------- 1x16 quantisation --
SHAPES_1D = [(1, 16), (3, 48), (100, 80), (128, 256), (130, 272), (257, 1040), (64, 4096)]


@pytest.mark.parametrize("rows,k", SHAPES_1D)
@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("sr", [False, True])
@pytest.mark.parametrize("mask", [0, MASK])
def test_quantize_1d(nv, rows, k, transposed, sr, mask):
    x = _data(rows, k, 1000 + rows + k, "t" if sr else "normal")   # logical [rows x k]
    stored = x.T.copy() if transposed else x
    ld = ((stored.shape[1] + 7) // 8) * 8 + 8
    d = dev_bf16(stored, ld)
    q, _, _ = gpu_quantize(nv, d, transposed=transposed, mask=mask, sr=sr, seed=77, sid=5)
    ref = oracle.quantize(stored, transposed=transposed, rht_mask=mask, sr=sr, seed=77, stream_id=5)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, f"1d {rows}x{k} t={transposed} sr={sr} rht={mask}")


@pytest.mark.parametrize("transposed", [False, True])
def test_quantize_own_amax(nv, transposed):
    """amax == NULL: the call computes the amax itself."""
    x = _data(96, 128, 3)
    stored = x.T.copy() if transposed else x
    q, _, _ = gpu_quantize(nv, dev_bf16(stored), transposed=transposed, own_amax=True)
    ref = oracle.quantize(stored, transposed=transposed)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "own amax")
    q, _, _ = gpu_quantize(nv, dev_bf16(stored), transposed=transposed, own_amax=True, mask=MASK, sr=True, seed=3)
    ref = oracle.quantize(stored, transposed=transposed, rht_mask=MASK, sr=True, seed=3)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "own amax rht sr")


def test_quantize_edge_values(nv):
    """Zero blocks, ties of the E2M1 grid, signed zeros and a zero tensor."""
    rows, k = 32, 64
    base = np.zeros((rows, k), np.float32)
    base[0, :16] = [6, 0.25 * 6 / 6, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.0, -0.1, 0.1, 4, 3, 2, 1, 0.5]
    base[1, 16:32] = -np.linspace(0, 6, 16)
    base[2, :] = 1e-3
    base[3, :] = -1e-30
    x = synth._to_bf16_bits(base)
    q, _, _ = gpu_quantize(nv, dev_bf16(x))
    ref = oracle.quantize(x)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "edge values")
    z = np.zeros((16, 32), np.uint16)
    q, _, _ = gpu_quantize(nv, dev_bf16(z))
    ref = oracle.quantize(z)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "zero tensor")


def test_quantize_tiny_amax(nv):
    """amax in the bf16 subnormal range: S_enc saturates to FLT_MAX."""
    x = np.zeros((16, 32), np.uint16)
    x[0, 0] = 0x0001
    x[5, 7] = 0x8003
    q, _, _ = gpu_quantize(nv, dev_bf16(x))
    ref = oracle.quantize(x)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "tiny amax")


def test_quantize_op_order_golden(nv, golden_dir):
    """The golden rows that separate the two plausible operation orders of the
    block scale and of the element encode: the kernels give the bytes derived
    by hand from t = fp32(fp32(amax_b / 6) * S_enc) and v = fp32(x * r_b)."""
    from conftest import read_golden
    import os
    for kind, a, b, x, expect, _ in read_golden(os.path.join(golden_dir, "op_order.txt")):
        row = np.zeros((1, 32), np.uint16)
        row[0, 0], row[0, 16], row[0, 17] = int(a, 16), int(b, 16), int(x, 16)
        q, _, _ = gpu_quantize(nv, dev_bf16(row))
        if kind == "scale":
            plain = oracle.unswizzle_scales(q.scales.cpu().numpy()[:oracle.scale_bytes(1, 32)], 1, 32)
            assert int(plain[0, 1]) == int(expect, 0), (a, b)
        else:
            assert (int(q.codes.cpu().numpy()[0, 8]) >> 4) & 0xF == int(expect, 0), (a, b, x)


# ------------------------------------------------------ 16x16 quantisation --
SHAPES_2D = [(16, 16), (32, 48), (48, 80), (128, 256), (144, 272), (256, 1040), (80, 192)]


@pytest.mark.parametrize("rows,k", SHAPES_2D)
@pytest.mark.parametrize("sr", [False, True])
@pytest.mark.parametrize("emit_t", [False, True])
def test_quantize_2d(nv, rows, k, sr, emit_t):
    w = synth.normal_bf16((rows, k), 2000 + rows + k, 0.02)
    q, qt, _ = gpu_quantize(nv, dev_bf16(w, k + 8), block2d=True, sr=sr, seed=9, sid=2, emit_t=emit_t)
    ref = oracle.quantize(w, block2d=True, sr=sr, seed=9, stream_id=2)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, f"2d {rows}x{k} sr={sr}")
    if emit_t:
        codes_t, scales_t = expected_transpose(ref)
        assert_q_equal(qt, codes_t, scales_t, ref.s_enc, f"2d-T {rows}x{k} sr={sr}")


@pytest.mark.parametrize("sr", [False, True])
def test_quantize_2d_many_tiles_per_cta(nv, sr):
    """4096 x 4096: 2048 tiles of 64 x 128, several per persistent CTA, so the
    shared-memory ring wraps; with the transposed emit."""
    rows, k = 4096, 4096
    w = synth.normal_bf16((rows, k), 31, 0.02)
    q, qt, _ = gpu_quantize(nv, dev_bf16(w), block2d=True, sr=sr, seed=3, sid=2, emit_t=True)
    ref = oracle.quantize(w, block2d=True, sr=sr, seed=3, stream_id=2)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, f"2d many tiles sr={sr}")
    codes_t, scales_t = expected_transpose(ref)
    assert_q_equal(qt, codes_t, scales_t, ref.s_enc, f"2d-T many tiles sr={sr}")


@pytest.mark.parametrize("rows,k", [(37, 64), (5, 16), (130, 96)])
def test_quantize_2d_ragged_rows(nv, rows, k):
    w = synth.normal_bf16((rows, k), 3000 + rows, 0.02)
    q, _, _ = gpu_quantize(nv, dev_bf16(w), block2d=True)
    ref = oracle.quantize(w, block2d=True)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "2d ragged")


@pytest.mark.parametrize("sr", [False, True])
def test_quantize_2d_transposed_view(nv, sr):
    """16x16 blocks of W^T read from W stored [k x rows]; out_t is W itself."""
    stored = synth.normal_bf16((96, 160), 41, 0.02)      # logical operand [160 x 96]
    q, qt, _ = gpu_quantize(nv, dev_bf16(stored), transposed=True, block2d=True, sr=sr, seed=4,
                            emit_t=True)
    ref = oracle.quantize(stored, transposed=True, block2d=True, sr=sr, seed=4)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "2d transposed view")
    codes_t, scales_t = expected_transpose(ref)
    assert_q_equal(qt, codes_t, scales_t, ref.s_enc, "2d transposed view, out_t")


@pytest.mark.parametrize("rows,k", [(32, 64), (144, 272)])
@pytest.mark.parametrize("sr", [False, True])
def test_rht_quantize_2d(nv, rows, k, sr):
    w = synth.normal_bf16((rows, k), 4000 + rows, 0.02, 0.01, 30.0)
    q, _, _ = gpu_quantize(nv, dev_bf16(w), block2d=True, mask=MASK, sr=sr, seed=1)
    ref = oracle.quantize(w, block2d=True, rht_mask=MASK, sr=sr, seed=1)
    assert_q_equal(q, ref.codes, ref.scales, ref.s_enc, "rht 2d")


def test_dequant_consistency_2d(nv):
    """dequant(W^T q) == dequant(W q)^T bit for bit (forward and backward see
    the same quantised weight)."""
    w = synth.normal_bf16((64, 128), 77, 0.02)
    q, qt, _ = gpu_quantize(nv, dev_bf16(w), block2d=True, sr=True, seed=8, emit_t=True)
    a = torch.empty((64, 128), dtype=torch.float32, device="cuda")
    b = torch.empty((128, 64), dtype=torch.float32, device="cuda")
    nv.nvfp4_dequantize(q, a)
    nv.nvfp4_dequantize(qt, b)
    torch.cuda.synchronize()
    assert torch.equal(a.T.cpu(), b.cpu())


# ---------------------------------------------------------- dequantise ----
@pytest.mark.parametrize("rows,k", [(1, 16), (100, 80), (257, 1040)])
@pytest.mark.parametrize("bf16", [False, True])
def test_dequantize(nv, rows, k, bf16):
    codes, scales = synth.random_operand(rows, k, rows + k, 0x01, 0x7E)
    q = oracle.Quantized(codes, scales, np.float32(3.7e2), rows, k)
    g = nv.QTensor(rows, k)
    g.codes.copy_(torch.from_numpy(codes))
    g.scales.copy_(torch.from_numpy(q.scales))
    g.global_scale.fill_(float(q.s_enc))
    ld = k + 8
    out = torch.empty((rows, ld), dtype=torch.bfloat16 if bf16 else torch.float32, device="cuda")[:, :k]
    nv.nvfp4_dequantize(g, out)
    torch.cuda.synchronize()
    ref = oracle.dequantize(q, out_bf16=bf16)
    got = out.cpu().view(torch.int16).numpy().view(np.uint16) if bf16 else out.cpu().numpy()
    np.testing.assert_array_equal(got, ref)


# -------------------------------------------------------------------- GEMM --
def _upload_operand(nv, codes, scales_plain, s_enc, rows, k):
    g = nv.QTensor(rows, k)
    g.codes.copy_(torch.from_numpy(codes))
    sw = oracle.swizzle_scales(scales_plain, rows, k)
    g.scales.copy_(torch.from_numpy(sw))
    g.global_scale.fill_(float(s_enc))
    return g, sw


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 512), (200, 300, 96), (1, 1, 32),
                                   (130, 260, 320), (384, 256, 1024), (128, 128, 4160),
                                   # several CTA-pair units, M- and N-fastest tile walks
                                   (512, 512, 512), (500, 300, 96), (1024, 768, 1280), (2048, 256, 512),
                                   (512, 4096, 256),
                                   # 384-column pair tiles, several units per pair
                                   (2048, 6144, 512)])
@pytest.mark.parametrize("bf16", [False, True])
def test_gemm_random_operands(nv, M, N, K, bf16):
    ca, sa = synth.random_operand(M, K, M + 7 * K)
    cb, sb = synth.random_operand(N, K, N + 13 * K)
    SA, SB = np.float32(2.5), np.float32(0.375)
    ga, swa = _upload_operand(nv, ca, sa, SA, M, K)
    gb, swb = _upload_operand(nv, cb, sb, SB, N, K)
    d = torch.empty((M, ((N + 7) // 8) * 8 + 8), dtype=torch.bfloat16 if bf16 else torch.float32,
                    device="cuda")[:, :N]
    d.fill_(float("nan"))
    nv.nvfp4_gemm(ga, gb, d)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    y_ref, ab = oracle.gemm_full(ca, swa, SA, cb, swb, SB, M, N, K)
    gemm_bound_check(d.float().cpu().numpy(), y_ref, ab, bf16, f"gemm {M}x{N}x{K} bf16={bf16}")


def test_gemm_integer_exact(nv):
    """Scales 1.0 and codes in {0, +1, -1}: an exact integer GEMM."""
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 512
    pick = np.array([0, 2, 10], np.uint8)
    av, bv = rng.integers(0, 3, (M, K)), rng.integers(0, 3, (N, K))
    pack = lambda v: (pick[v[:, 0::2]] | (pick[v[:, 1::2]] << 4)).astype(np.uint8)
    ga, _ = _upload_operand(nv, pack(av), np.full((M, K // 16), 0x38, np.uint8), 1.0, M, K)
    gb, _ = _upload_operand(nv, pack(bv), np.full((N, K // 16), 0x38, np.uint8), 1.0, N, K)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nv.nvfp4_gemm(ga, gb, d)
    torch.cuda.synchronize()
    sv = np.array([0, 1, -1])
    ref = sv[av].astype(np.int64) @ sv[bv].astype(np.int64).T
    np.testing.assert_array_equal(d.cpu().numpy(), ref.astype(np.float32))


@pytest.mark.parametrize("M", [256, 512, 1024])
def test_gemm_scale_rows_are_distinct(nv, M):
    """Each row of A and of B gets its own scale (power of two by row): a
    wrong scale layout in shared or tensor memory shows up as a wrong row or
    column of D (M = 512, 1024: several CTA pairs)."""
    N, K = 256, 256
    rng = np.random.default_rng(6)
    ca = np.full((M, K // 2), 0x22, np.uint8)                 # all elements 1.0
    cb = np.full((N, K // 2), 0x22, np.uint8)
    ea = rng.integers(0x20, 0x50, size=(M, 1)).repeat(K // 16, 1).astype(np.uint8)
    eb = rng.integers(0x20, 0x50, size=(N, 1)).repeat(K // 16, 1).astype(np.uint8)
    ea[:, 3] = 0x38                                           # one block of each row at 1.0
    ga, swa = _upload_operand(nv, ca, ea, 1.0, M, K)
    gb, swb = _upload_operand(nv, cb, eb, 1.0, N, K)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nv.nvfp4_gemm(ga, gb, d)
    torch.cuda.synchronize()
    y_ref, ab = oracle.gemm_full(ca, swa, 1.0, cb, swb, 1.0, M, N, K)
    gemm_bound_check(d.cpu().numpy(), y_ref, ab, False, "per-row scales")


def _full_range_scales(rows, k, seed):
    """E4M3 decode-scale bytes over the whole finite range 0x00-0x7E: uniform
    draws, then whole zero-scale blocks (0x00), subnormal codes 0x01-0x07 and
    the largest code 0x7E (448) planted in about 6%, 12% and 3% of the blocks."""
    rng = np.random.default_rng(seed)
    s = rng.integers(0x00, 0x7F, size=(rows, k // 16), dtype=np.uint8)
    u = rng.random(s.shape)
    s[u < 0.06] = 0x00
    sub = (u >= 0.06) & (u < 0.18)
    s[sub] = rng.integers(0x01, 0x08, size=int(sub.sum()), dtype=np.uint8)
    s[(u >= 0.18) & (u < 0.21)] = 0x7E
    return s


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (128, 256, 320), (1024, 768, 1280), (384, 200, 4096)])
@pytest.mark.parametrize("bf16", [False, True])
def test_gemm_full_e4m3_scale_range(nv, M, N, K, bf16):
    """Block scales over every finite E4M3 code, including zero-scale blocks,
    the subnormal codes 0x01-0x07 (2^-9 .. 7 * 2^-9) and 0x7E: the tensor
    core's UE4M3 scale decoding must match the format's value set ([NVB]
    recipe bullet 2: E4M3 block scales; [SAI] "Core architectural changes of
    the MVFP4 format").  (128, 256, 320) and (384, 200, 4096) have an odd
    128-row tile count: their last CTA pair holds one empty tile."""
    rng = np.random.default_rng(M * 3 + N + K)
    ca = rng.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    cb = rng.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    sa, sb = _full_range_scales(M, K, M + K), _full_range_scales(N, K, N + 2 * K)
    assert (sa == 0).any() and ((sa >= 1) & (sa <= 7)).any() and (sa == 0x7E).any()
    SA, SB = np.float32(2.5), np.float32(0.375)
    ga, swa = _upload_operand(nv, ca, sa, SA, M, K)
    gb, swb = _upload_operand(nv, cb, sb, SB, N, K)
    d = torch.empty((M, ((N + 7) // 8) * 8), dtype=torch.bfloat16 if bf16 else torch.float32,
                    device="cuda")[:, :N]
    d.fill_(float("nan"))
    nv.nvfp4_gemm(ga, gb, d)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    y_ref, ab = oracle.gemm_full(ca, swa, SA, cb, swb, SB, M, N, K)
    gemm_bound_check(d.float().cpu().numpy(), y_ref, ab, bf16, f"full scale range {M}x{N}x{K} bf16={bf16}")


def test_gemm_subnormal_scale_products_exact(nv):
    """Only subnormal and zero scales, codes 1.0: every product of two block
    scales is a small exact binary64 number and the FP32 sums are exact, so
    D must equal the oracle exactly."""
    M, N, K = 256, 256, 256
    rng = np.random.default_rng(11)
    ca = np.full((M, K // 2), 0x22, np.uint8)
    cb = np.full((N, K // 2), 0x22, np.uint8)
    sa = rng.integers(0, 8, size=(M, K // 16), dtype=np.uint8)
    sb = rng.integers(0, 8, size=(N, K // 16), dtype=np.uint8)
    ga, swa = _upload_operand(nv, ca, sa, 1.0, M, K)
    gb, swb = _upload_operand(nv, cb, sb, 1.0, N, K)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nv.nvfp4_gemm(ga, gb, d)
    torch.cuda.synchronize()
    y_ref, _ = oracle.gemm_full(ca, swa, 1.0, cb, swb, 1.0, M, N, K)
    np.testing.assert_array_equal(d.cpu().numpy().astype(np.float64), y_ref)


def _tiny_amax_data(rows, k, seed, magnitude):
    """bf16 data ~ N(0,1) * magnitude (a magnitude below 7.9e-36 makes the
    tensor's S_enc = 2688 / amax overflow to FLT_MAX)."""
    g = np.random.default_rng(seed)
    x = (g.standard_normal((rows, k)) * magnitude).astype(np.float32)
    return synth._to_bf16_bits(x)


@pytest.mark.parametrize("tiny", ["a", "ab"])
@pytest.mark.parametrize("bf16", [False, True])
def test_gemm_alpha_from_saturated_global_scale(nv, tiny, bf16):
    """An operand whose amax is tiny (S_enc saturates to FLT_MAX): alpha =
    1 / (S_A S_B) falls into FP32's subnormal range ("a") or below it ("ab",
    both operands tiny: the exact products underflow FP32 altogether).  The
    quantised operands must equal the oracle's and D must stay within the
    bound of the binary64 reference."""
    M, N, K = 256, 256, 512
    x = _tiny_amax_data(M, K, 21, 1e-37)
    w = _tiny_amax_data(N, K, 22, 1e-37) if tiny == "ab" else synth.normal_bf16((N, K), 23, 0.02)
    qx, _, _ = gpu_quantize(nv, dev_bf16(x))
    qw, _, _ = gpu_quantize(nv, dev_bf16(w), block2d=True)
    ox, ow = oracle.quantize(x), oracle.quantize(w, block2d=True)
    assert_q_equal(qx, ox.codes, ox.scales, ox.s_enc, "tiny X")
    assert_q_equal(qw, ow.codes, ow.scales, ow.s_enc, "W")
    assert ox.s_enc == np.float32(np.finfo(np.float32).max)
    d = torch.empty((M, N), dtype=torch.bfloat16 if bf16 else torch.float32, device="cuda")
    nv.nvfp4_gemm(qx, qw, d)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    y_ref, ab = oracle.gemm_full(ox.codes, ox.scales, ox.s_enc, ow.codes, ow.scales, ow.s_enc, M, N, K)
    alpha = 1.0 / (float(ox.s_enc) * float(ow.s_enc))
    assert alpha < 2.0 ** -126                                 # outside FP32's normal range
    gemm_bound_check(d.float().cpu().numpy(), y_ref, ab, bf16, f"saturated S_enc ({tiny}) bf16={bf16}")
    if tiny == "a":
        assert np.count_nonzero(d.float().cpu().numpy()) > 0.9 * M * N


def test_quantize_gemm_subnormal_block_scales(nv):
    """Quantise -> GEMM with subnormal E4M3 block scales made by the
    quantiser itself: one huge outlier sets S_enc, and blocks of small values
    beside it get decode scales 0x01-0x07 (or 0).  Codes and scales must equal
    the oracle's, and D must be within the bound."""
    M, N, K = 256, 256, 1024
    g = np.random.default_rng(31)
    xf = (g.standard_normal((M, K)) * 0.05).astype(np.float32)
    xf[7, 100] = 1.0e4
    x = synth._to_bf16_bits(xf)
    w = synth.normal_bf16((N, K), 32, 0.02)
    qx, _, _ = gpu_quantize(nv, dev_bf16(x))
    qw, _, _ = gpu_quantize(nv, dev_bf16(w), block2d=True)
    ox, ow = oracle.quantize(x), oracle.quantize(w, block2d=True)
    assert_q_equal(qx, ox.codes, ox.scales, ox.s_enc, "X with subnormal block scales")
    assert_q_equal(qw, ow.codes, ow.scales, ow.s_enc, "W")
    plain = ox.scales_plain
    assert ((plain >= 1) & (plain <= 7)).mean() > 0.5, "the case must produce subnormal scales"
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    nv.nvfp4_gemm(qx, qw, d)
    torch.cuda.synchronize()
    y_ref, ab = oracle.gemm_full(ox.codes, ox.scales, ox.s_enc, ow.codes, ow.scales, ow.s_enc, M, N, K)
    gemm_bound_check(d.cpu().numpy(), y_ref, ab, False, "subnormal block scales")


# --------------------------------------------------- tiny forward linear ---
def test_tiny_forward_linear(nv):
    """The tiny forward workload end to end: X [128 x 256] 1x16 RNE, W
    [256 x 256] 16x16, Y = X W^T with FP32 accumulation and FP32 output."""
    x, w = synth.tiny_forward(0)
    dx, dw = dev_bf16(x), dev_bf16(w)
    qx, _, _ = gpu_quantize(nv, dx)
    qw, _, _ = gpu_quantize(nv, dw, block2d=True)
    y = torch.empty((128, 256), dtype=torch.float32, device="cuda")
    nv.nvfp4_gemm(qx, qw, y)
    torch.cuda.synchronize()
    ox, ow = oracle.quantize(x), oracle.quantize(w, block2d=True)
    assert_q_equal(qx, ox.codes, ox.scales, ox.s_enc, "X")
    assert_q_equal(qw, ow.codes, ow.scales, ow.s_enc, "W")
    yr, ab = oracle.gemm_full(ox.codes, ox.scales, ox.s_enc, ow.codes, ow.scales, ow.s_enc, 128, 256, 256)
    gemm_bound_check(y.cpu().numpy(), yr, ab, False, "tiny forward")
