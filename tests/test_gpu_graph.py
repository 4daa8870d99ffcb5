"""The path's calls inside a CUDA graph.

Every call is asynchronous and stream-ordered (host validation, a launch or a
memset on the caller's stream, no host synchronisation), so a whole linear
layer step can be captured once and replayed.  The replay must write the
same bytes as the same calls run eagerly.  The cold case captures before any
eager call, so the first-use work inside the calls (kernel attributes, the
GEMM's cached cluster occupancy) happens during capture.
"""
import os
import subprocess
import sys

import pytest
import torch

import synth
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _inputs():
    tok, hid, ffn = 512, 1024, 768
    x = dev_bf16(synth.normal_bf16((tok, hid), 21, 1.0, 0.0005, 100.0))
    w = dev_bf16(synth.normal_bf16((ffn, hid), 22, 0.02))
    dy = dev_bf16(synth.student_t_bf16((tok, ffn), 23, 3, 1e-3))
    return tok, hid, ffn, x, w, dy


class _Step:
    """Forward, dgrad and wgrad of one NVFP4 linear layer, every buffer
    allocated up front (a graph replays fixed addresses)."""

    def __init__(self, nv, tok, hid, ffn, x, w, dy):
        self.nv, self.x, self.w, self.dy = nv, x, w, dy
        self.mask = nv.nvfp4_rht_mask_from_seed(2023) or 1
        self.amax = torch.zeros(6, dtype=torch.float32, device="cuda")
        self.qx, self.qxt = nv.QTensor(tok, hid), nv.QTensor(hid, tok)
        self.qw, self.qwt = nv.QTensor(ffn, hid, block2d=True), nv.QTensor(hid, ffn, block2d=True)
        self.qdy, self.qdyt = nv.QTensor(tok, ffn), nv.QTensor(ffn, tok)
        self.y = torch.empty(tok, ffn, dtype=torch.bfloat16, device="cuda")
        self.dx = torch.empty(tok, hid, dtype=torch.bfloat16, device="cuda")
        self.dw = torch.empty(ffn, hid, dtype=torch.bfloat16, device="cuda")

    def run(self):
        nv, a = self.nv, self.amax
        nv.nvfp4_amax(self.w, 0, a[1:2])
        nv.nvfp4_quantize_2d(self.w, a[1:2], nv.NVFP4_RNE, 0, 0, self.qw, self.qwt)
        nv.nvfp4_amax_dual(self.x, self.mask, a[0:1], a[4:5])
        nv.nvfp4_quantize_dual(self.x, a[0:1], nv.NVFP4_RNE, 0, 0, self.qx, self.mask, a[4:5], nv.NVFP4_RNE, 0, 0,
                               self.qxt)
        nv.nvfp4_gemm(self.qx, self.qw, self.y)
        nv.nvfp4_amax_dual(self.dy, self.mask, a[2:3], a[3:4])
        nv.nvfp4_quantize_dual(self.dy, a[2:3], nv.NVFP4_SR, 77, 1, self.qdy, self.mask, a[3:4], nv.NVFP4_SR, 77,
                               2, self.qdyt)
        nv.nvfp4_gemm(self.qdy, self.qwt, self.dx)
        nv.nvfp4_gemm(self.qdyt, self.qxt, self.dw)

    def outputs(self):
        out = [self.amax.clone(), self.y.clone(), self.dx.clone(), self.dw.clone()]
        for q in (self.qx, self.qxt, self.qw, self.qwt, self.qdy, self.qdyt):
            out += [q.codes.clone(), q.scales.clone(), q.global_scale.clone()]
        return out

    def clear(self):
        for t in (self.amax, self.y, self.dx, self.dw):
            t.zero_()
        for q in (self.qx, self.qxt, self.qw, self.qwt, self.qdy, self.qdyt):
            q.codes.zero_(), q.scales.zero_(), q.global_scale.zero_()


def _same(a, b):
    return all(torch.equal(u.view(torch.uint8), v.view(torch.uint8)) for u, v in zip(a, b))


def capture_and_compare(cold: bool) -> None:
    import nvfp4_block_scaled_29_b300 as nv
    step = _Step(nv, *_inputs())
    if not cold:
        step.run()                         # eager first: the calls' first-use work happens here
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):              # the calls take torch's current (capturing) stream
        step.run()
    torch.cuda.synchronize()
    step.clear()
    g.replay()
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    replayed = step.outputs()
    step.clear()
    g.replay()
    torch.cuda.synchronize()
    assert _same(step.outputs(), replayed), "two replays differ"
    step.clear()
    step.run()
    torch.cuda.synchronize()
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    assert _same(step.outputs(), replayed), "replay and eager calls differ"
    assert float(replayed[0].abs().sum()) > 0 and float(replayed[1].float().abs().sum()) > 0


def test_graph_replay_matches_eager():
    capture_and_compare(cold=False)


def test_graph_capture_before_any_eager_call():
    # a fresh process: nothing of the library has run on the device yet
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "import test_gpu_graph as t; t.capture_and_compare(cold=True); print('cold capture ok')"
            % (ROOT, HERE))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0 and "cold capture ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
