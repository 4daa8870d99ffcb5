"""Failure detection on the GPU without a fault: a wait whose copy is never
issued (test-only injection, nvfp4_debug_inject) expires after its bounded
limit, the kernel returns, nvfp4_get_status reports NVFP4_ERR_TIMEOUT, and
the context stays usable for the next call.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

MASK = 0x9D2B


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_29_b300 as m
    assert torch.cuda.is_available()
    return m


def test_dropped_copy_reports_timeout_and_context_survives(nv):
    s = synth.normal_bf16((512, 1024), 13, 1.0, 0.002, 60.0)
    d = dev_bf16(s)
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    nv.nvfp4_debug_inject(1)
    t0 = time.monotonic()
    nv.nvfp4_amax_dual(d, MASK)
    st = nv.nvfp4_get_status()                 # synchronises
    waited = time.monotonic() - t0
    assert st == nv.NVFP4_ERR_TIMEOUT, nv.status_string(st)
    assert waited < 30.0                       # bounded: about 2 s of wait plus 2 s of drain
    # the injection applied once; the next call is exact
    a, at = nv.nvfp4_amax_dual(d, MASK)
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    assert float(a.cpu()[0]) == oracle.amax(s)
    assert float(at.cpu()[0]) == oracle.amax(s, transposed=True, rht_mask=MASK)


def test_debug_inject_rejects_unknown_modes(nv):
    with pytest.raises(nv.Nvfp4Error):
        nv.nvfp4_debug_inject(3)
    nv.nvfp4_debug_inject(0)
