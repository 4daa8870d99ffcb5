"""Helpers shared by the GPU parity tests: moving seeded host inputs to the
device, running one quantisation through the C ABI, and comparing a
quantised operand with the oracle's byte for byte."""
import numpy as np
import torch

import oracle


def dev_bf16(a: np.ndarray, ld: int | None = None) -> torch.Tensor:
    """Upload a bf16 bit array [r x c]; with ld > c the device array is
    [r x ld] and the returned tensor is its [:, :c] slice (stride ld)."""
    r, c = a.shape
    if ld is None or ld == c:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    pad = np.full((r, ld), 0x7FC0, dtype=np.uint16)      # NaN padding must never be read
    pad[:, :c] = a
    t = torch.from_numpy(pad.view(np.int16)).cuda().view(torch.bfloat16)
    return t[:, :c]


def gpu_quantize(nv, x_dev, *, transposed=False, mask=0, block2d=False, sr=False, seed=0, sid=0,
                 own_amax=False, emit_t=False, sr_hw=False):
    """Quantise through the C ABI; returns (q, q_t or None, amax tensor or None)."""
    r, c = x_dev.shape
    rows, k = (c, r) if transposed else (r, c)
    out = nv.QTensor(rows, k, block2d)
    out_t = nv.QTensor(k, rows, True) if emit_t else None
    rnd = (nv.NVFP4_SR_HW if sr_hw else nv.NVFP4_SR) if sr else nv.NVFP4_RNE
    amax = None if own_amax else nv.nvfp4_amax(x_dev, mask, transposed=transposed)
    if mask:
        nv.nvfp4_rht_quantize(x_dev, mask, amax, rnd, seed, sid, out, transposed=transposed)
    elif block2d:
        nv.nvfp4_quantize_2d(x_dev, amax, rnd, seed, sid, out, out_t, transposed=transposed)
    else:
        nv.nvfp4_quantize_1d(x_dev, amax, rnd, seed, sid, out, transposed=transposed)
    torch.cuda.synchronize()
    st = nv.nvfp4_get_status()
    assert st == nv.NVFP4_OK, nv.status_string(st)
    return out, out_t, amax


def assert_q_equal(q_gpu, codes, scales_swz, s_enc, what=""):
    gc = q_gpu.codes.cpu().numpy()
    gs = q_gpu.scales.cpu().numpy()[:scales_swz.size]
    if not np.array_equal(gc, codes):
        bad = np.argwhere(gc != codes)
        r, c = bad[0]
        raise AssertionError(f"{what}: {len(bad)} code bytes differ; first at row {r} byte {c}: "
                             f"gpu {gc[r, c]:#04x} oracle {codes[r, c]:#04x}")
    if not np.array_equal(gs, scales_swz):
        bad = np.flatnonzero(gs != scales_swz)
        raise AssertionError(f"{what}: {len(bad)} scale bytes differ; first at {bad[0]}: "
                             f"gpu {gs[bad[0]]:#04x} oracle {scales_swz[bad[0]]:#04x}")
    g = float(q_gpu.global_scale.cpu().numpy()[0])
    assert g == np.float32(s_enc), f"{what}: S_enc gpu {g!r} oracle {s_enc!r}"


def expected_transpose(q: "oracle.Quantized"):
    """The transposed operand made from the same 16x16 encoding: codes
    transposed nibble by nibble, each block scale copied to the rows of the
    transposed operand."""
    rows, k = q.rows, q.k
    codes_t = oracle.transpose_codes(q.codes, rows, k)
    blk = q.scales_plain[::16, :]                          # [rows/16 x k/16]
    plain_t = np.repeat(blk.T, 16, axis=0)                  # [k x rows/16]
    return codes_t, oracle.swizzle_scales(plain_t, k, rows)


def gemm_bound_check(y_gpu: np.ndarray, y_ref: np.ndarray, ab: np.ndarray, bf16: bool, what=""):
    """|y - y_ref| <= 2e-5 * sum|a b| (FP32 output).  BF16 output adds the
    BF16 rounding of the result: + 2^-8 |y_ref| (unit roundoff of an 8-bit
    significand), with the FP32 bound scaled by (1 + 2^-8).

    Both add the smallest subnormal of the output format (2^-149 for FP32,
    2^-133 for BF16): an exact result below that spacing has no closer
    representable output, so the relative bound alone cannot hold there (it
    only matters when both operands have a tiny amax and alpha is near FP32's
    underflow)."""
    y = y_gpu.astype(np.float64)
    err = np.abs(y - y_ref)
    bound = 2e-5 * ab + 2.0 ** -149
    if bf16:
        bound = bound * (1 + 2.0 ** -8) + 2.0 ** -8 * np.abs(y_ref) + 2.0 ** -133
    ok = err <= bound
    if not ok.all():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {np.count_nonzero(~ok)} of {ok.size} outside the bound; worst at "
                             f"{i}: gpu {y[i]!r} ref {y_ref[i]!r} sum|ab| {ab[i]!r}")


def sample_ranges(rows, n, length, align, seed):
    """Row ranges for sampled checks: the first and last `length` rows and n
    random ranges in between, starts aligned to `align`."""
    rng = np.random.default_rng(seed)
    starts = sorted(set(int(s) // align * align for s in rng.integers(0, rows - length, n)))
    return [(0, length)] + [(s, s + length) for s in starts] + [(rows - length, rows)]


def check_sampled(gpu, ref, ranges, rows, k, what):
    """Codes and scales of a GPU operand (codes, swizzled scales, S_enc) equal
    the oracle's on the sampled row ranges; S_enc equal; scale padding zero."""
    codes, scales_swz, s_enc = gpu
    plain = oracle.unswizzle_scales(scales_swz[:oracle.scale_bytes(rows, k)], rows, k)
    for lo, hi in ranges:
        np.testing.assert_array_equal(codes[lo:hi], ref.codes[lo:hi], err_msg=f"{what} codes rows {lo}:{hi}")
        np.testing.assert_array_equal(plain[lo:hi], ref.scales_plain[lo:hi], err_msg=f"{what} scales rows {lo}:{hi}")
    assert s_enc == np.float32(ref.s_enc), what
    # padding of the scale layout is zero
    full = np.zeros(oracle.scale_bytes(rows, k), np.uint8)
    pad_mask = oracle.swizzle_scales(np.ones((rows, k // 16), np.uint8), rows, k) == 0
    assert not scales_swz[:full.size][pad_mask].any(), f"{what}: non-zero scale padding"
