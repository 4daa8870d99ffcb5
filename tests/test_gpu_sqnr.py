"""The quantisation-error harness (NVFP4 vs MXFP4, with and without RHT-16):
its dequantised values are the oracle's bit for bit, its Hadamard reference
agrees with the oracle's transform, and on the step's synthetic tensors it
shows the pages' claim that NVFP4 (16-element blocks, E4M3 scales)
represents values more precisely than MXFP4 (32-element blocks, power-of-two
scales)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu
MASK = 0x6A39


@pytest.fixture(scope="module")
def sq():
    from nvfp4_block_scaled_29_b300 import sqnr
    assert torch.cuda.is_available()
    return sqnr


@pytest.mark.parametrize("mask", [0, MASK])
def test_dequantised_values_are_the_oracles(sq, mask):
    x = synth.normal_bf16((96, 320), 4, 1.0, 0.002, 60.0)
    d = dev_bf16(x)
    got = sq._dequant_nvfp4(d, mask).cpu().numpy()
    assert np.array_equal(got, oracle.dequantize(oracle.quantize(x, rht_mask=mask)))
    got = sq._dequant_mxfp4(d, mask).cpu().numpy()
    assert np.array_equal(got, oracle.mx_dequantize(oracle.mx_quantize(x, rht_mask=mask)))


def test_hadamard_reference_matches_oracle_transform(sq):
    x = synth.normal_bf16((4, 64), 5, 1.0, 0.0, 1.0)
    ref = sq._reference(dev_bf16(x), MASK).cpu().numpy()
    xf = synth.bf16_bits_to_f32(x)
    for r in range(4):
        for c in range(0, 64, 16):
            np.testing.assert_allclose(oracle.rht16(xf[r, c:c + 16], MASK), ref[r, c:c + 16], rtol=1e-6, atol=1e-6)


def test_nvfp4_beats_mxfp4_on_the_step_tensors(sq):
    tensors = {"X": dev_bf16(synth.activations(2, tokens=512)), "W": dev_bf16(synth.weights(3, ffn=512)),
               "dY": dev_bf16(synth.grad_output(3 + 7919, tokens=512))}
    rows = sq.table(tensors, MASK)
    by = {(r["tensor"], r["format"], r["rht"]): r["sqnr_db"] for r in rows}
    for name in tensors:
        for rht in (False, True):
            assert by[(name, "nvfp4", rht)] > by[(name, "mxfp4", rht)], (name, rht, by)
    assert all(8.0 < v < 40.0 for v in by.values()), by
