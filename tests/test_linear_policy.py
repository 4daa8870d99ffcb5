"""Host-side logic of the NVFP4 linear module (no GPU): the per-layer
precision opt-out and the shape rules."""
import pytest
import torch

from nvfp4_block_scaled_29_b300.linear import NVFP4Linear, _check_shapes, apply_precision_policy


def _model(n):
    return torch.nn.Sequential(*[NVFP4Linear(64, 64, device="cpu", seed=i) for i in range(n)])


@pytest.mark.parametrize("n,frac,expect", [(20, 0.15, 3), (10, 0.15, 2), (7, 0.15, 2), (4, 0.0, 0),
                                           (4, 1.0, 4), (1, 0.15, 1), (100, 0.15, 15)])
def test_policy_keeps_the_last_layers_in_bf16(n, frac, expect):
    m = _model(n)
    names = apply_precision_policy(m, frac)
    assert len(names) == expect
    prec = [layer.precision for layer in m]
    assert prec == ["nvfp4"] * (n - expect) + ["bf16"] * expect
    assert names == [str(i) for i in range(n - expect, n)]


def test_policy_rejects_bad_fraction():
    with pytest.raises(ValueError):
        apply_precision_policy(_model(2), 1.5)


def test_shape_rules():
    _check_shapes(64, 32, 96)
    for bad in [(48, 32, 32), (32, 16, 32), (32, 32, 80)]:
        with pytest.raises(ValueError):
            _check_shapes(*bad)


def test_call_seeds_differ_per_call():
    layer = NVFP4Linear(64, 64, device="cpu", seed=7)
    s0 = layer.call_seed()
    layer.calls += 1
    assert layer.call_seed() != s0
