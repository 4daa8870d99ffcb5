"""The kernels' fp32(amax_b / 6) against CUDA's IEEE-rounded division, over
every non-negative finite float.

The block decode scale is t = fp32(fp32(amax_b / 6) * S_enc) (NVIDIA blog
"NVFP4 Trains with Precision of 16-Bit and Speed and Efficiency of 4-Bit",
recipe bullet 2: E4M3 block scales; the constants 6 and 448 fixed for this
path).  The kernels compute the quotient with Markstein's correction instead
of a division; this must give the correctly rounded quotient bit for bit.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


def test_div6_matches_ieee_division_exhaustively(nv):
    # 2^31 - 2^23 patterns: +0, every subnormal and normal float below +Inf
    n, first = nv.nvfp4_debug_check_div6(0x00000000, 0x7F800000)
    assert n == 0, f"{n} mismatches, first at bit pattern {first:#010x}"


def test_div6_check_reports_a_range_and_rejects_bad_args(nv):
    assert nv.nvfp4_debug_check_div6(0x3F800000, 0x3F800000) == (0, None)   # empty range
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_debug_check_div6(0x7F800000, 0x7F800001)                  # Inf is not allowed
