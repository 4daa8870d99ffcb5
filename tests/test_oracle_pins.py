"""Pins of the CPU oracle against what the sources and the mathematics fix.

Each test is chosen so that a plausible mistake in the oracle (a wrong tie
rule, a swapped nibble, a dropped Hadamard stage, a transposed index, a wrong
scale op order) fails it.  None of these tests uses the CUDA library.
"""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
import synth
from conftest import ROOT, read_golden

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


# ----------------------------------------------------------------- formats --
def test_e2m1_value_set_matches_pages(golden_dir):
    rows = read_golden(os.path.join(golden_dir, "e2m1_values.txt"))
    assert len(rows) == 16
    for code, val in rows:
        v = oracle.e2m1_value(int(code))
        assert v == float(val) and math.copysign(1, v) == math.copysign(1, float(val))
    mags = sorted({abs(oracle.e2m1_value(c)) for c in range(16)})
    assert mags == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_rne_ties_and_saturation(golden_dir):
    for v, code in read_golden(os.path.join(golden_dir, "e2m1_rne_ties.txt")):
        assert oracle.e2m1_rne(np.float32(float(v))) == int(code), v


def test_e2m1_rne_is_nearest_by_brute_force():
    """Nearest-value property over a dense sweep: the chosen value is never
    farther than any other value of the set."""
    vals = np.array([oracle.e2m1_value(c) for c in range(16)])
    rng = np.random.default_rng(1)
    xs = np.concatenate([np.linspace(-7, 7, 20001), rng.uniform(-6.5, 6.5, 20000)]).astype(np.float32)
    for x in xs:
        c = oracle.e2m1_rne(x)
        d = abs(vals[c] - float(x))
        if abs(float(x)) <= 6:
            assert d <= np.min(np.abs(vals - float(x))) + 0.0
        else:
            assert abs(vals[c]) == 6.0


def _host_conv_binary(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("hc") / "host_conversions")
    subprocess.check_call([nvcc, "-O2", "-o", out,
                           os.path.join(ROOT, "tests", "helpers", "host_conversions.cu")])
    return out


@pytest.fixture(scope="module")
def host_conv(tmp_path_factory):
    return _host_conv_binary(tmp_path_factory)


def _run_conv(binary, mode, xs):
    r = subprocess.run([binary, mode], input=np.asarray(xs, np.float32).tobytes(),
                       capture_output=True, check=True)
    return np.frombuffer(r.stdout, dtype=np.uint8)


def test_e2m1_rne_matches_cuda_host_library(host_conv):
    rng = np.random.default_rng(2)
    xs = np.concatenate([
        rng.uniform(-8, 8, 50000), rng.normal(0, 1e-3, 2000), [0.0, -0.0, 1e-40, -1e-40],
        np.arange(-6.5, 6.5, 0.125)]).astype(np.float32)
    lib = _run_conv(host_conv, "e2m1", xs)
    ours = np.array([oracle.e2m1_rne(x) for x in xs], dtype=np.uint8)
    np.testing.assert_array_equal(ours, lib)


def test_e4m3_values_match_torch_float8():
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    np.testing.assert_array_equal(ours, ref)
    assert oracle.e4m3_value(0x7E) == 448.0


def test_e4m3_rne_satfinite_matches_libraries(host_conv):
    rng = np.random.default_rng(3)
    grid = np.array([oracle.e4m3_value(c) for c in range(0x7F)])
    mids = (grid[1:] + grid[:-1]) / 2
    xs = np.concatenate([rng.uniform(0, 460, 20000), 10 ** rng.uniform(-4, 2.7, 20000), grid, mids,
                         [448.0, 448.5, 463.9, 464.0, 1e6, 3e38, 0.0, 1e-30]]).astype(np.float32)
    ours = np.array([oracle.e4m3_rne_satfinite(x) for x in xs], dtype=np.uint8)
    np.testing.assert_array_equal(ours, _run_conv(host_conv, "e4m3", xs))
    below = xs < 448
    ref = torch.from_numpy(xs[below]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours[below], ref)


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(4)
    xs = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e30, 1000), [0.0, -0.0, 1e-40, 3.4e38]]).astype(np.float32)
    ours = np.array([oracle.f32_to_bf16_rne(x) for x in xs], dtype=np.uint16)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


# ------------------------------------------------------------------ Philox --
def test_philox_known_answers(golden_dir):
    for row in read_golden(os.path.join(golden_dir, "philox4x32_10_kat.txt")):
        w = [int(t, 16) for t in row]
        np.testing.assert_array_equal(oracle.philox4x32_10(w[:4], w[4:6]), np.array(w[6:], np.uint32))


def test_philox_matches_curand_host_call(tmp_path_factory):
    """The oracle's Philox4x32-10 equals the CUDA toolkit's cuRAND block
    function (called on the host, black box) on random and edge counters/keys."""
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("hp") / "host_philox")
    subprocess.check_call([nvcc, "-O2", "-o", exe, os.path.join(ROOT, "tests", "helpers", "host_philox.cu")])
    rng = np.random.default_rng(21)
    recs = rng.integers(0, 1 << 32, (2000, 6), dtype=np.uint64).astype(np.uint32)
    edge = np.array([[0, 0, 0, 0, 0, 0], [0xFFFFFFFF] * 6, [1, 0, 0, 0, 0, 0], [0, 0, 0, 1, 0xDEADBEEF, 0]],
                    np.uint32)
    recs = np.concatenate([recs, edge])
    r = subprocess.run([exe], input=recs.tobytes(), capture_output=True, check=True)
    lib = np.frombuffer(r.stdout, dtype=np.uint32).reshape(-1, 4)
    for rec, want in zip(recs, lib):
        np.testing.assert_array_equal(oracle.philox4x32_10(rec[:4], rec[4:6]), want)


def test_philox_bit_statistics():
    bits = np.array([oracle.sr_bits16(123, 7, i) for i in range(200000)], dtype=np.uint32)
    # every one of the 16 bit positions is set about half the time (5 sigma)
    for b in range(16):
        p = ((bits >> b) & 1).mean()
        assert abs(p - 0.5) < 5 * math.sqrt(0.25 / len(bits))
    # byte chi-square, 255 dof: mean 255, sd ~22.6
    hist = np.bincount((bits & 0xFF).astype(np.int64), minlength=256)
    e = len(bits) / 256
    chi2 = ((hist - e) ** 2 / e).sum()
    assert chi2 < 255 + 6 * 22.6


def test_sr_bits_follow_counter_layout():
    """Element idx takes 16-bit slice idx%8 of Philox(counter=(idx/8, stream), key=seed)."""
    seed, sid = 0x1234_5678_9ABC, 0xDEAD_BEEF_01
    for idx in [0, 1, 2, 7, 8, 9, 12345, 2**33 + 5]:
        g = idx >> 3
        o = oracle.philox4x32_10([g & 0xFFFFFFFF, g >> 32, sid & 0xFFFFFFFF, sid >> 32],
                                 [seed & 0xFFFFFFFF, seed >> 32])
        w = int(o[(idx & 7) >> 1])
        exp = (w >> 16) if idx & 1 else (w & 0xFFFF)
        assert oracle.sr_bits16(seed, sid, idx) == exp


def test_sr_hw_bits_follow_counter_layout():
    """Second layout: element idx takes position idx%4 of word (idx%16)/4 of
    Philox(counter=(idx/16, stream), key=seed), as u16 = 65535 - r."""
    seed, sid = 0x1234_5678_9ABC, 0xDEAD_BEEF_01
    for idx in [0, 1, 2, 3, 4, 7, 15, 16, 17, 12345, 2**33 + 5]:
        g = idx >> 4
        o = oracle.philox4x32_10([g & 0xFFFFFFFF, g >> 32, sid & 0xFFFFFFFF, sid >> 32],
                                 [seed & 0xFFFFFFFF, seed >> 32])
        r = oracle.sr_r16_of_word(int(o[(idx & 15) >> 2]), idx & 3)
        assert oracle.sr_bits16_hw(seed, sid, idx) == 65535 - r


def test_sr_word_layout_single_bits():
    """Worked single-bit cases of the second layout: H = (byte 3, byte 1) and
    L = (byte 2, byte 0); positions 0..3 take L, reversed L, H, reversed H."""
    cases = [  # (word bit, position, r16)
        (0, 0, 0x0001), (7, 0, 0x0080), (16, 0, 0x0100), (23, 0, 0x8000),
        (0, 1, 0x8000), (7, 1, 0x0100), (16, 1, 0x0080), (23, 1, 0x0001),
        (8, 2, 0x0001), (15, 2, 0x0080), (24, 2, 0x0100), (31, 2, 0x8000),
        (8, 3, 0x8000), (15, 3, 0x0100), (24, 3, 0x0080), (31, 3, 0x0001),
    ]
    for bit, pos, r in cases:
        assert oracle.sr_r16_of_word(1 << bit, pos) == r, (bit, pos)
    # a position ignores the two bytes it does not read
    for pos, other in ((0, 0xFF00FF00), (1, 0xFF00FF00), (2, 0x00FF00FF), (3, 0x00FF00FF)):
        assert oracle.sr_r16_of_word(other, pos) == 0


def test_sr_word_layout_is_a_bijection_per_position():
    """Second layout: over all 2^16 settings of the 16 bits a position reads,
    its r16 takes every value exactly once, so a uniform word gives a uniform
    r16 (and u16)."""
    t = np.arange(1 << 16, dtype=np.uint32)
    lo_bytes = (t & 0xFF) | ((t >> 8) << 16)            # bytes 0 and 2
    hi_bytes = lo_bytes << 8                            # bytes 1 and 3
    for pos, words in ((0, lo_bytes), (1, lo_bytes), (2, hi_bytes), (3, hi_bytes)):
        r = np.array([oracle.sr_r16_of_word(int(w), pos) for w in words], dtype=np.int64)
        assert np.array_equal(np.sort(r), np.arange(1 << 16))


# ------------------------------------------------------ stochastic rounding --
def test_sr_pages_example_probability(golden_dir):
    """0.3 on a grid {0, 1}: P(up) = 0.3 over 10^6 Philox draws, within 5 sigma.

    In E2M1 code units the grid {0, 1} is {0, 0.5}, so the value is 0.15."""
    (row,) = read_golden(os.path.join(golden_dir, "sr_example.txt"))
    val, p_up, lo, hi = map(float, row)
    unit = 0.5 / (hi - lo)
    v = np.float32(val * unit)
    n = 1_000_000
    ups = sum(oracle.e2m1_value(oracle.e2m1_sr(v, oracle.sr_bits16(99, 0, i))) == 0.5 for i in range(n))
    sigma = math.sqrt(p_up * (1 - p_up) / n)
    assert abs(ups / n - p_up) < 5 * sigma


def test_sr_pages_example_through_quantizer():
    """Same example end to end: blocks of one 12.0 and fifteen bf16(0.3).  With
    amax 12, S_enc = 224, s_b = 448, so dequantised values are exactly {0, 1}."""
    x_bits = synth._to_bf16_bits(np.full((4168, 256), 0.3, np.float32))
    x_bits[:, ::16] = synth._to_bf16_bits(np.array([12.0], np.float32))[0]
    q = oracle.quantize(x_bits, sr=True, seed=5, stream_id=1)
    assert q.s_enc == np.float32(224.0)
    xh = oracle.dequantize(q)
    mask = np.ones_like(xh, dtype=bool)
    mask[:, ::16] = False
    vals = xh[mask]
    assert set(np.unique(vals)) <= {0.0, 1.0}
    x03 = float(synth.bf16_bits_to_f32(x_bits[0, 1]))
    n = vals.size
    assert n >= 1_000_000
    sigma = math.sqrt(x03 * (1 - x03) / n)
    assert abs(vals.mean() - x03) < 5 * sigma
    # 6 * 448 * fp32(1/224): one rounding of the reciprocal away from 12
    np.testing.assert_allclose(xh[:, ::16], 12.0, rtol=2.0 ** -23)


def test_sr_is_unbiased_and_brackets_value():
    rng = np.random.default_rng(6)
    for v in rng.uniform(-6, 6, 40).astype(np.float32):
        codes = [oracle.e2m1_sr(v, oracle.sr_bits16(1, 3, i)) for i in range(20000)]
        got = np.array([oracle.e2m1_value(c) for c in codes])
        assert len(np.unique(got)) <= 2
        assert got.min() <= v <= got.max()
        spread = got.max() - got.min()
        if spread:
            sd = spread * 0.5 / math.sqrt(len(got))
            assert abs(got.mean() - float(v)) < 5 * sd + 1e-12


def test_sr_exact_grid_values_never_move():
    for c in range(16):
        v = np.float32(oracle.e2m1_value(c))
        for u in [0, 1, 0x7FFF, 0xFFFF]:
            assert oracle.e2m1_value(oracle.e2m1_sr(v, u)) == float(v)


def test_sr_rule_exact_over_all_random_values():
    """For a value a fraction k/2^16 of the way from lo to hi, exactly k of the
    2^16 values of u16 round it up, so the mean over them is the value itself
    (the rounding is unbiased, exactly); larger magnitudes saturate."""
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    rng = np.random.default_rng(12)
    for lo_i in range(7):
        lo, hi = grid[lo_i], grid[lo_i + 1]
        for k in [0, 1, 2, 0x4000, 0x8000, 0xFFFF, int(rng.integers(0, 1 << 16))]:
            for sgn in (1.0, -1.0):
                v = np.float32(sgn * (lo + (hi - lo) * k / 65536.0))
                assert float(v) == sgn * (lo + (hi - lo) * k / 65536.0)
                codes = np.array([oracle.e2m1_sr(v, u) for u in range(1 << 16)])
                ups = int(((codes & 7) == lo_i + 1).sum())
                assert ups == k and int(((codes & 7) == lo_i).sum()) == 65536 - k
                assert ((codes & 8) == (8 if sgn < 0 else 0)).all()
                vals = np.array([oracle.e2m1_value(c) for c in np.unique(codes)])
                cnt = np.array([(codes == c).sum() for c in np.unique(codes)])
                assert (vals * cnt).sum() / 65536.0 == float(v)
    for v in (6.0, 6.5, 100.0):
        assert oracle.e2m1_sr(np.float32(v), 0) == 7 and oracle.e2m1_sr(np.float32(-v), 0xFFFF) == 15


def test_sr_hw_layout_statistics():
    """The second layout through the quantiser: the pages' 0.3 example rounds
    up with probability 0.3 within 5 sigma, as with the first layout."""
    n = 400_000
    v = np.float32(0.15)                   # 0.3 of the way from 0 to 0.5
    ups = sum(oracle.e2m1_value(oracle.e2m1_sr(v, oracle.sr_bits16_hw(99, 0, i))) == 0.5 for i in range(n))
    sigma = math.sqrt(0.3 * 0.7 / n)
    assert abs(ups / n - 0.3) < 5 * sigma


# --------------------------------------------------------------------- RHT --
def _rht_matrix(mask):
    return np.stack([oracle.rht16(np.eye(16, dtype=np.float32)[j], mask) for j in range(16)], axis=1)


def test_rht_is_scaled_sylvester_hadamard():
    H = _rht_matrix(0).astype(np.float64)
    np.testing.assert_array_equal(H, scipy.linalg.hadamard(16) / 4.0)
    np.testing.assert_array_equal(H.T @ H, np.eye(16))


def test_rht_signs_and_orthogonality():
    mask = 0b1010_0110_0001_1101
    R = _rht_matrix(mask).astype(np.float64)
    D = np.diag([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)])
    np.testing.assert_array_equal(R, scipy.linalg.hadamard(16) @ D / 4.0)
    np.testing.assert_array_equal(R.T @ R, np.eye(16))


def test_rht_norm_and_dot_product_preserved():
    rng = np.random.default_rng(7)
    for _ in range(200):
        a = rng.standard_normal(16).astype(np.float32)
        b = rng.standard_normal(16).astype(np.float32)
        m = int(rng.integers(0, 1 << 16))
        ta, tb = oracle.rht16(a, m).astype(np.float64), oracle.rht16(b, m).astype(np.float64)
        a64, b64 = a.astype(np.float64), b.astype(np.float64)
        assert abs(np.linalg.norm(ta) - np.linalg.norm(a64)) <= 1e-6 * np.linalg.norm(a64)
        assert abs(ta @ tb - a64 @ b64) <= 1e-6 * np.linalg.norm(a64) * np.linalg.norm(b64)


def test_rht_exact_on_integers_and_inverse():
    rng = np.random.default_rng(8)
    for _ in range(100):
        a = rng.integers(-512, 512, 16).astype(np.float32)
        m = int(rng.integers(0, 1 << 16))
        D = np.array([-1.0 if (m >> j) & 1 else 1.0 for j in range(16)])
        ref = scipy.linalg.hadamard(16) @ (D * a) / 4.0
        t = oracle.rht16(a, m)
        np.testing.assert_array_equal(t.astype(np.float64), ref)
        # inverse: x = D H y / 4  (H symmetric, H H = 16 I)
        back = D * (scipy.linalg.hadamard(16) @ t.astype(np.float64)) / 4.0
        np.testing.assert_array_equal(back, a)


def test_rht_mask_from_seed_is_philox_word0():
    for seed in [0, 1, 2002, 2**40 + 3]:
        o = oracle.philox4x32_10([0, 0, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.rht_mask_from_seed(seed) == int(o[0]) & 0xFFFF


# -------------------------------------------------------------------- amax --
def test_amax_plain_matches_numpy():
    x = synth.normal_bf16((64, 96), 11, 1.0, 0.01, 50.0)
    ref = np.abs(synth.bf16_bits_to_f32(x)).max()
    assert oracle.amax(x) == ref
    assert oracle.amax(x, transposed=True) == ref


def test_amax_rht_matches_hadamard_matmul():
    rng = np.random.default_rng(12)
    xi = rng.integers(-100, 100, size=(32, 64)).astype(np.float32)
    x = synth._to_bf16_bits(xi)
    mask = 0x5A3C
    D = np.array([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)])
    H = scipy.linalg.hadamard(16)
    # rows layout: chunks along the stored rows
    ref_rows = np.abs((H @ (D[:, None] * xi.reshape(32, 4, 16).transpose(2, 0, 1).reshape(16, -1)))).max() / 4
    assert oracle.amax(x, rht_mask=mask) == ref_rows
    # transposed view: logical k runs down the stored columns
    ref_t = np.abs((H @ (D[:, None] * xi.reshape(2, 16, 64).transpose(1, 0, 2).reshape(16, -1)))).max() / 4
    assert oracle.amax(x, transposed=True, rht_mask=mask) == ref_t


def test_amax_nan_propagates():
    x = synth.normal_bf16((16, 32), 13)
    x[3, 5] = 0x7FC1
    assert math.isnan(oracle.amax(x))
    assert oracle.global_scale(float("nan"))[0] != 0
    assert oracle.global_scale(float("inf"))[0] != 0


def test_global_scale_closed_form():
    assert oracle.global_scale(0.0) == (0, 1.0)
    for a in [1.0, 6.0, 12.0, 448.0, 3.7e-3]:
        st, s = oracle.global_scale(a)
        assert st == 0 and s == np.float32(np.float32(2688.0) / np.float32(a))
    st, s = oracle.global_scale(1e-40)
    assert st == 0 and s == np.finfo(np.float32).max


# --------------------------------------------------- scales and block coverage --
def test_max_element_dequantises_within_e4m3_rounding():
    """Per block, the largest |x| maps to code 6 and dequantises within the
    E4M3 relative rounding error 2^-4 of the block amax."""
    x = synth.normal_bf16((64, 256), 21, 1.0, 0.001, 50.0)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    q = oracle.quantize(x)
    xh = oracle.dequantize(q).astype(np.float64)
    blocks = np.abs(xf).reshape(64, 16, 16)
    amax_b = blocks.max(axis=2)
    idx = blocks.argmax(axis=2)
    got = np.abs(xh.reshape(64, 16, 16))[np.arange(64)[:, None], np.arange(16)[None, :], idx]
    ok = amax_b > 0
    assert np.all(np.abs(got[ok] - amax_b[ok]) <= 2.0 ** -4 * amax_b[ok] * (1 + 1e-6))


def test_tensor_max_maps_to_448_scale_and_code_6():
    x = synth.normal_bf16((32, 64), 22)
    q = oracle.quantize(x)
    xf = synth.bf16_bits_to_f32(x)
    r, c = np.unravel_index(np.argmax(np.abs(xf)), xf.shape)
    assert q.scales_plain[r, c // 16] == 0x7E        # 448
    code = (q.codes[r, c // 2] >> (4 * (c % 2))) & 0xF
    assert code & 7 == 7                             # magnitude 6


@pytest.mark.parametrize("block2d", [False, True])
def test_block_coverage(block2d):
    """Changing one element changes at most its own scale and only the codes of
    its 16-element (1x16) or 256-element (16x16) block."""
    x = synth.normal_bf16((48, 64), 31)
    amax_v = oracle.amax(x) * 2
    base = oracle.quantize(x, block2d=block2d, amax_v=amax_v)
    rng = np.random.default_rng(32)
    for _ in range(12):
        r, c = int(rng.integers(0, 48)), int(rng.integers(0, 64))
        y = x.copy()
        y[r, c] = synth._to_bf16_bits(np.array([float(synth.bf16_bits_to_f32(x[r, c])) * 7 + 3.0], np.float32))[0]
        q = oracle.quantize(y, block2d=block2d, amax_v=amax_v)
        rows = slice(r // 16 * 16, r // 16 * 16 + 16) if block2d else slice(r, r + 1)
        cols = slice(c // 16 * 16, c // 16 * 16 + 16)
        unpack = lambda cd: np.stack([cd & 0xF, cd >> 4], axis=-1).reshape(48, 64)
        d_codes = unpack(q.codes) != unpack(base.codes)
        outside = d_codes.copy()
        outside[rows, cols] = False
        assert not outside.any()
        d_sc = q.scales_plain != base.scales_plain
        sc_out = d_sc.copy()
        sc_out[rows, c // 16] = False
        assert not sc_out.any()
        if block2d:
            # the scale is shared by all 16 rows of the block
            assert len(np.unique(q.scales_plain[rows, c // 16])) == 1


def test_2d_transposed_view_is_exact_transpose():
    """Quantising W^T (transposed view, 16x16 blocks) gives exactly the
    transposed codes and the same scales: forward and backward see one
    quantised weight."""
    w = synth.normal_bf16((64, 96), 41, 0.02)
    q = oracle.quantize(w, block2d=True)
    qt = oracle.quantize(w, block2d=True, transposed=True)
    np.testing.assert_array_equal(qt.codes, oracle.transpose_codes(q.codes, 64, 96))
    np.testing.assert_array_equal(oracle.dequantize(qt), oracle.dequantize(q).T)


def test_quantize_1d_differs_from_2d_only_by_scale_sharing():
    w = synth.normal_bf16((32, 64), 42)
    q1, q2 = oracle.quantize(w), oracle.quantize(w, block2d=True)
    # the 2D scale is the max over the 16 rows of the 1D scales of that block
    s1 = np.array([[oracle.e4m3_value(v) for v in row] for row in q1.scales_plain])
    s2 = np.array([[oracle.e4m3_value(v) for v in row] for row in q2.scales_plain])
    for rb in range(2):
        np.testing.assert_array_equal(s2[rb * 16], s1[rb * 16:rb * 16 + 16].max(axis=0))


def test_zero_block_and_zero_tensor():
    x = synth.normal_bf16((16, 64), 43)
    x[:, 16:32] = 0
    q = oracle.quantize(x)
    assert np.all(q.scales_plain[:, 1] == 0)
    z = np.zeros((16, 32), np.uint16)
    qz = oracle.quantize(z)
    assert qz.s_enc == 1.0 and not qz.codes.any() and not qz.scales_plain.any()


def test_rht_quantize_uses_transformed_values():
    x = synth.normal_bf16((16, 32), 44)
    m = 0x1234
    q = oracle.quantize(x, rht_mask=m)
    xf = synth.bf16_bits_to_f32(x)
    t = np.stack([oracle.rht16(xf[r, c:c + 16], m) for r in range(16) for c in (0, 16)]).reshape(16, 32)
    # dequantised values approximate the transformed tensor (E2M1 + E4M3 rounding)
    xh = oracle.dequantize(q)
    amax_b = np.abs(t).reshape(16, 2, 16).max(axis=2)
    err = np.abs(xh - t).reshape(16, 2, 16).max(axis=2)
    assert np.all(err <= amax_b * (1 / 6 + 2 ** -4) * 1.07 + 1e-30)


# ---------------------------------------------------------- swizzle layout --
def test_swizzle_roundtrip_and_padding():
    rng = np.random.default_rng(51)
    for rows, k in [(1, 16), (128, 64), (130, 80), (257, 272), (64, 1024)]:
        plain = rng.integers(1, 255, size=(rows, k // 16), dtype=np.uint8)
        swz = oracle.swizzle_scales(plain, rows, k)
        assert swz.size == -(-rows // 128) * 128 * (-(-(k // 16) // 4) * 4)
        np.testing.assert_array_equal(oracle.unswizzle_scales(swz, rows, k), plain)
        assert np.count_nonzero(swz) == plain.size      # padding stays 0


def test_swizzle_tile_structure():
    """Each 512-byte tile holds exactly the 128 rows x 4 columns of its tile,
    with the 4 scales of one row contiguous."""
    rows, k = 256, 256
    plain = np.zeros((rows, k // 16), np.uint16)
    for r in range(rows):
        for c in range(k // 16):
            plain[r, c] = (r // 128) * 4 + c // 4          # tile id
    swz = oracle.swizzle_scales(plain.astype(np.uint8), rows, k)
    tiles = swz.reshape(-1, 512)
    for t in range(tiles.shape[0]):
        assert np.all(tiles[t] == t)
    plain2 = np.arange(rows)[:, None].repeat(k // 16, 1).astype(np.uint8)
    swz2 = oracle.swizzle_scales(plain2, rows, k).reshape(-1, 128, 4)
    assert np.all(swz2 == swz2[:, :, :1])               # 4 scales of a row are adjacent


def test_transpose_codes_involution():
    rng = np.random.default_rng(52)
    c = rng.integers(0, 256, size=(32, 48), dtype=np.uint8)
    t = oracle.transpose_codes(c, 32, 96)
    np.testing.assert_array_equal(oracle.transpose_codes(t, 96, 32), c)


# ------------------------------------------------------------ dequantise --
def test_dequantize_matches_library_decoders(golden_dir):
    table = {int(a): float(b) for a, b in read_golden(os.path.join(golden_dir, "e2m1_values.txt"))}
    codes, scales = synth.random_operand(40, 64, 53)
    q = oracle.Quantized(codes, scales, np.float32(37.25), 40, 64)
    xh = oracle.dequantize(q)
    lo, hi = codes & 0xF, codes >> 4
    qv = np.stack([np.vectorize(table.get)(lo), np.vectorize(table.get)(hi)], -1).reshape(40, 64).astype(np.float32)
    sv = torch.from_numpy(scales).view(torch.float8_e4m3fn).float().numpy().repeat(16, axis=1)
    ref = (qv * sv) * (np.float32(1) / np.float32(37.25))
    np.testing.assert_array_equal(xh, ref.astype(np.float32))
    xb = oracle.dequantize(q, out_bf16=True)
    np.testing.assert_array_equal(xb, torch.from_numpy(ref).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_quantize_dequantize_error_bound():
    """|x_hat - x| <= half an E2M1 step at the scale, plus the scale's rounding."""
    x = synth.normal_bf16((64, 128), 54, 1.0, 0.001, 50.0)
    q = oracle.quantize(x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    xh = oracle.dequantize(q).astype(np.float64)
    sb = np.array([[oracle.e4m3_value(v) for v in row] for row in q.scales_plain]).repeat(16, 1)
    unit = sb / q.s_enc                 # dequantised value of code magnitude 1
    assert np.all(np.abs(xh - xf) <= 1.0 * unit * 1.0001 + 1e-30)   # max grid gap is 2 -> half is 1


# --------------------------------------------------------------- GEMM ref --
def test_gemm_integer_special_case_exact():
    """Scales all 1.0 (E4M3 0x38) and codes in {0, +1, -1}: the reference is an
    integer GEMM, compared exactly with numpy."""
    rng = np.random.default_rng(61)
    M, N, K = 40, 24, 128
    pick = np.array([0, 2, 10], np.uint8)                    # 0, +1, -1
    av = rng.integers(0, 3, size=(M, K)); bv = rng.integers(0, 3, size=(N, K))
    pack = lambda v: (pick[v[:, 0::2]] | (pick[v[:, 1::2]] << 4)).astype(np.uint8)
    ones_a = oracle.swizzle_scales(np.full((M, K // 16), 0x38, np.uint8), M, K)
    ones_b = oracle.swizzle_scales(np.full((N, K // 16), 0x38, np.uint8), N, K)
    y, ab = oracle.gemm_full(pack(av), ones_a, 1.0, pack(bv), ones_b, 1.0, M, N, K)
    sv = np.array([0, 1, -1])
    ref = sv[av].astype(np.int64) @ sv[bv].astype(np.int64).T
    np.testing.assert_array_equal(y, ref.astype(np.float64))
    np.testing.assert_array_equal(ab, (np.abs(sv[av]) @ np.abs(sv[bv]).T).astype(np.float64))


def test_gemm_matches_numpy_on_dequantised_operands():
    M, N, K = 48, 40, 96
    ca, sa = synth.random_operand(M, K, 62)
    cb, sb = synth.random_operand(N, K, 63)
    table = np.array([oracle.e2m1_value(c) for c in range(16)])
    deq = lambda c, s, r: (np.stack([table[c & 0xF], table[c >> 4]], -1).reshape(r, K) *
                           torch.from_numpy(s).view(torch.float8_e4m3fn).double().numpy().repeat(16, 1))
    A, B = deq(ca, sa, M), deq(cb, sb, N)
    SA, SB = np.float32(3.5), np.float32(0.75)
    y, ab = oracle.gemm_full(ca, oracle.swizzle_scales(sa, M, K), SA, cb,
                             oracle.swizzle_scales(sb, N, K), SB, M, N, K)
    ref = A @ B.T / (float(SA) * float(SB))
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    np.testing.assert_allclose(ab, np.abs(A) @ np.abs(B).T / (float(SA) * float(SB)), rtol=1e-12)
    ms = np.array([0, 5, 47, 13]); ns = np.array([0, 39, 7, 13])
    yp, abp = oracle.gemm_points(ca, oracle.swizzle_scales(sa, M, K), SA, cb,
                                 oracle.swizzle_scales(sb, N, K), SB, M, N, K, ms, ns)
    np.testing.assert_array_equal(yp, y[ms, ns])
    np.testing.assert_array_equal(abp, ab[ms, ns])


def test_gemm_end_to_end_approximates_bf16_matmul():
    """Quantised GEMM of the tiny forward workload approximates the bf16 matmul
    (relative Frobenius error of a 4-bit format, a loose sanity bound)."""
    x, w = synth.tiny_forward(0)
    qx, qw = oracle.quantize(x), oracle.quantize(w, block2d=True)
    y, _ = oracle.gemm_full(qx.codes, qx.scales, qx.s_enc, qw.codes, qw.scales, qw.s_enc, 128, 256, 256)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ synth.bf16_bits_to_f32(w).astype(np.float64).T
    assert np.linalg.norm(y - ref) / np.linalg.norm(ref) < 0.2


# ------------------------------------------------------------------ MXFP4 --
def test_mx_scale_examples_from_pages(golden_dir):
    for amax_b, scale in read_golden(os.path.join(golden_dir, "mx_scale_examples.txt")):
        assert oracle.e8m0_value(oracle.mx_scale_code(float(amax_b))) == float(scale)


def test_mx_scale_rule_closed_form():
    """The block max lands in [4, 8) after scaling by 2^-X, away from the
    clamps; zero gives the smallest scale."""
    rng = np.random.default_rng(3)
    vals = np.concatenate([np.exp2(rng.uniform(-120, 120, 2000)), [1.0, 4.0, 6.0, 7.99, 8.0, 2.0 ** -125]])
    for a in vals.astype(np.float32):
        s = oracle.e8m0_value(oracle.mx_scale_code(float(a)))
        assert 4.0 <= float(a) / s < 8.0, a
        assert math.log2(s) == math.floor(math.log2(float(a))) - 2
    assert oracle.mx_scale_code(0.0) == 0
    assert oracle.mx_scale_code(2.0 ** -126) == 0                # X = -128 clamps to -127
    assert oracle.mx_scale_code(1e-45) == 0
    assert oracle.e8m0_value(255) != oracle.e8m0_value(255)      # NaN code


def _grid():
    return np.array([oracle.e2m1_value(c) for c in range(16)])


def test_mx_quantize_is_nearest_grid_point_by_brute_force():
    """Every element dequantises to the E2M1 grid point nearest to x / 2^X
    (ties to the even code, saturating at 6), times 2^X."""
    x = synth.normal_bf16((8, 256), 5, 1.0, 0.01, 30.0)
    q = oracle.mx_quantize(x)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    deq = oracle.mx_dequantize(q).astype(np.float64)
    grid = _grid()
    for r in range(8):
        for b in range(256 // 32):
            blk = xf[r, 32 * b:32 * b + 32]
            s = 2.0 ** (math.floor(math.log2(np.abs(blk).max())) - 2)
            for j, v in enumerate(blk / s):
                d = np.abs(grid - np.clip(v, -6, 6))
                best = np.flatnonzero(d == d.min())
                best = [c for c in best if (grid[c] < 0) == (v < 0) or grid[c] == 0] or list(best)
                code = min(best, key=lambda c: (c & 1, c))          # ties: even code
                assert deq[r, 32 * b + j] == grid[code] * s, (r, b, j, v)


def test_mx_exact_on_grid_values():
    """A block whose values are grid points times 2^X is represented exactly."""
    rng = np.random.default_rng(7)
    grid = _grid()
    vals = grid[rng.integers(0, 16, (4, 64))] * 2.0 ** 5
    vals[:, 0] = 6 * 2.0 ** 5                                 # block max -> scale 2^5
    vals[:, 32] = -4 * 2.0 ** 5
    x = np.vectorize(lambda f: oracle.f32_to_bf16_rne(float(f)))(vals.astype(np.float32)).astype(np.uint16)
    q = oracle.mx_quantize(x)
    assert np.array_equal(oracle.mx_dequantize(q), vals.astype(np.float32))


def test_mx_swizzle_roundtrip():
    rng = np.random.default_rng(8)
    for rows, k in [(1, 32), (130, 96), (256, 512)]:
        plain = rng.integers(1, 255, (rows, k // 32)).astype(np.uint8)
        swz = oracle.mx_swizzle_scales(plain, rows, k)
        assert swz.size == oracle.mx_scale_bytes(rows, k)
        assert np.array_equal(oracle.mx_unswizzle_scales(swz, rows, k), plain)
        assert np.count_nonzero(swz) == plain.size                # padding is zero


def test_mx_gemm_integer_special_case_exact():
    rng = np.random.default_rng(9)
    M, N, K = 16, 24, 128
    pick = np.array([0, 2, 10], np.uint8)                       # codes of 0, +1, -1
    av, bv = rng.integers(0, 3, (M, K)), rng.integers(0, 3, (N, K))
    pack = lambda v: (pick[v[:, 0::2]] | (pick[v[:, 1::2]] << 4)).astype(np.uint8)
    one = np.full((M, K // 32), 127, np.uint8)                  # 2^0
    sa = oracle.mx_swizzle_scales(one, M, K)
    sb = oracle.mx_swizzle_scales(np.full((N, K // 32), 127, np.uint8), N, K)
    y, _ = oracle.mx_gemm_full(pack(av), sa, pack(bv), sb, M, N, K)
    sv = np.array([0, 1, -1])
    assert np.array_equal(y, (sv[av] @ sv[bv].T).astype(np.float64))


def test_mx_gemm_matches_numpy_on_dequantised_operands():
    a = synth.normal_bf16((32, 256), 10, 1.0, 0.01, 30.0)
    b = synth.normal_bf16((48, 256), 11, 0.02, 0.0, 1.0)
    qa, qb = oracle.mx_quantize(a), oracle.mx_quantize(b)
    y, ab = oracle.mx_gemm_full(qa.codes, qa.scales, qb.codes, qb.scales, 32, 48, 256)
    da, db = oracle.mx_dequantize(qa).astype(np.float64), oracle.mx_dequantize(qb).astype(np.float64)
    ref = da @ db.T
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * np.abs(da) @ np.abs(db).T + 1e-300)
    assert np.allclose(ab, np.abs(da) @ np.abs(db).T, rtol=1e-12)


# ------------------------------------------------------ operation order ----
def _op_order_cases(golden_dir):
    from conftest import read_golden
    return [(k, int(a, 16), int(b, 16), int(x, 16), int(e, 0), int(o, 0))
            for k, a, b, x, e, o in read_golden(os.path.join(golden_dir, "op_order.txt"))]


def _op_order_row(a_bits, b_bits, x_bits):
    row = np.zeros((1, 32), np.uint16)
    row[0, 0], row[0, 16], row[0, 17] = a_bits, b_bits, x_bits
    return row


def test_op_order_cases_discriminate(golden_dir):
    """Each golden case separates the two operation orders: computed here with
    numpy binary32 arithmetic and torch's float -> E4M3 cast (independent of
    the oracle), the left-to-right order gives the stated byte and the other
    order the stated other byte."""
    import torch
    f32 = np.float32
    bf = lambda b: np.array([b << 16], np.uint32).view(np.float32)[0]
    e4m3 = lambda t: int(torch.tensor([float(t)]).to(torch.float8_e4m3fn).view(torch.uint8)[0])
    e4m3v = lambda c: float(torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float()[0])
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]

    def e2m1(v):                                   # nearest, ties to the even code (v >= 0)
        d = [abs(float(v) - g) for g in grid]
        best = min(d)
        return min(i for i in range(8) if d[i] == best and (d.count(best) == 1 or i % 2 == 0))

    cases = _op_order_cases(golden_dir)
    assert {c[0] for c in cases} == {"scale", "code"}
    for kind, a, b, x, expect, other in cases:
        A, ab, xv = bf(a), bf(b), bf(x)
        s = f32(f32(2688.0) / A)
        t_lr = f32(f32(ab / f32(6.0)) * s)
        t_alt = f32(f32(ab * s) / f32(6.0))
        if kind == "scale":
            assert (e4m3(t_lr), e4m3(t_alt)) == (expect, other)
        else:
            sb = f32(e4m3v(e4m3(t_lr)))
            v_lr = f32(xv * f32(s / sb))
            v_alt = f32(f32(xv * s) / sb)
            assert (e2m1(v_lr), e2m1(v_alt)) == (expect, other)


def test_oracle_takes_the_specified_op_order(golden_dir):
    """The oracle's block scale and element code on the golden rows are the
    left-to-right ones: t = fp32(fp32(amax_b / 6) * S_enc) and
    v = fp32(x * fp32(S_enc / s_b))."""
    for kind, a, b, x, expect, other in _op_order_cases(golden_dir):
        q = oracle.quantize(_op_order_row(a, b, x))
        if kind == "scale":
            assert int(q.scales_plain[0, 1]) == expect, (kind, hex(a), hex(b))
        else:
            code = (int(q.codes[0, 8]) >> 4) & 0xF        # element 17: high nibble of byte 8
            assert code == expect, (kind, hex(a), hex(b), hex(x))
