"""The NVFP4 linear layer (autograd) on the GPU: forward and backward equal
the C-ABI call sequence byte for byte, and are within the GEMM bound of the
oracle's quantisation of the same operands (forward 1x16 RNE X, 16x16 RNE W;
dgrad 1x16 SR dY with W^T; wgrad RHT-16 SR dY^T with RHT RNE X^T)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev_bf16, gemm_bound_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lin():
    from nvfp4_block_scaled_29_b300 import linear
    assert torch.cuda.is_available()
    return linear


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _qdq(q):
    return q.codes, q.scales, q.s_enc


@pytest.mark.parametrize("tokens,k_in,k_out", [(256, 256, 512), (384, 640, 256)])
def test_linear_matches_oracle(lin, tokens, k_in, k_out):
    xb = synth.normal_bf16((tokens, k_in), 11, 1.0, 0.002, 60.0)
    wb = synth.normal_bf16((k_out, k_in), 12, 0.02, 0.0, 1.0)
    dyb = synth.student_t_bf16((tokens, k_out), 13, 3, 1e-3)
    x = dev_bf16(xb).requires_grad_(True)
    w = dev_bf16(wb).requires_grad_(True)
    seed, mask = 4242, 0x6A39
    y = lin.NVFP4LinearFunction.apply(x, w, seed, mask)
    y.backward(dev_bf16(dyb))
    torch.cuda.synchronize()
    import nvfp4_block_scaled_29_b300 as nv
    assert nv.nvfp4_get_status() == nv.NVFP4_OK
    # forward
    qx = oracle.quantize(xb)
    qw = oracle.quantize(wb, block2d=True)
    yr, ab = oracle.gemm_full(*_qdq(qx), *_qdq(qw), tokens, k_out, k_in)
    gemm_bound_check(y.float().detach().cpu().numpy(), yr, ab, True, "linear forward")
    # dgrad: dX = dY W
    qdy = oracle.quantize(dyb, sr=True, seed=seed, stream_id=lin.STREAM_DGRAD)
    qwt = oracle.quantize(wb, block2d=True, transposed=True)
    dxr, ab = oracle.gemm_full(*_qdq(qdy), *_qdq(qwt), tokens, k_in, k_out)
    gemm_bound_check(x.grad.float().cpu().numpy(), dxr, ab, True, "linear dgrad")
    # wgrad: dW = dY^T X with the RHT along the tokens on both operands
    qdyt = oracle.quantize(dyb, transposed=True, rht_mask=mask, sr=True, seed=seed, stream_id=lin.STREAM_WGRAD)
    qxt = oracle.quantize(xb, transposed=True, rht_mask=mask)
    dwr, ab = oracle.gemm_full(*_qdq(qdyt), *_qdq(qxt), k_out, k_in, tokens)
    gemm_bound_check(w.grad.float().cpu().numpy(), dwr, ab, True, "linear wgrad")


def test_linear_matches_direct_calls(lin):
    """Byte equality with the explicit C-ABI sequence of the training step."""
    import nvfp4_block_scaled_29_b300 as nv
    tokens, k_in, k_out = 512, 384, 256
    xb = synth.normal_bf16((tokens, k_in), 21, 1.0, 0.002, 60.0)
    wb = synth.normal_bf16((k_out, k_in), 22, 0.02, 0.0, 1.0)
    dyb = synth.student_t_bf16((tokens, k_out), 23, 3, 1e-3)
    x, w, dy = dev_bf16(xb), dev_bf16(wb), dev_bf16(dyb)
    seed, mask = 77, 0x1F2E
    xg, wg = x.clone().requires_grad_(True), w.clone().requires_grad_(True)
    y = lin.NVFP4LinearFunction.apply(xg, wg, seed, mask)
    y.backward(dy)
    Q = nv.QTensor
    a = torch.zeros(8, device="cuda")
    qx, qxt, qw, qwt = Q(tokens, k_in), Q(k_in, tokens), Q(k_out, k_in, True), Q(k_in, k_out, True)
    nv.nvfp4_amax(x, mask, a[0:1], transposed=True)
    nv.nvfp4_rht_quantize(x, mask, a[0:1], nv.NVFP4_RNE, 0, 0, qxt, transposed=True)
    nv.nvfp4_amax(x, 0, a[1:2])
    nv.nvfp4_quantize_1d(x, a[1:2], nv.NVFP4_RNE, 0, 0, qx)
    nv.nvfp4_amax(w, 0, a[2:3])
    nv.nvfp4_quantize_2d(w, a[2:3], nv.NVFP4_RNE, 0, 0, qw, qwt)
    y2 = torch.empty((tokens, k_out), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(qx, qw, y2)
    qdy, qdyt = Q(tokens, k_out), Q(k_out, tokens)
    nv.nvfp4_amax(dy, 0, a[3:4])
    nv.nvfp4_quantize_1d(dy, a[3:4], nv.NVFP4_SR, seed, lin.STREAM_DGRAD, qdy)
    nv.nvfp4_amax(dy, mask, a[4:5], transposed=True)
    nv.nvfp4_rht_quantize(dy, mask, a[4:5], nv.NVFP4_SR, seed, lin.STREAM_WGRAD, qdyt, transposed=True)
    dx2 = torch.empty((tokens, k_in), dtype=torch.bfloat16, device="cuda")
    dw2 = torch.empty((k_out, k_in), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(qdy, qwt, dx2)
    nv.nvfp4_gemm(qdyt, qxt, dw2)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(y.detach()), _bits(y2))
    assert np.array_equal(_bits(xg.grad), _bits(dx2))
    assert np.array_equal(_bits(wg.grad), _bits(dw2))


def test_module_policy_and_training_step(lin):
    """A small model: the last 15% of its layers run in BF16; one SGD step
    through the NVFP4 layers lowers the loss of a fixed regression target."""
    torch.manual_seed(0)
    layers = [lin.NVFP4Linear(256, 256, seed=i) for i in range(7)]
    model = torch.nn.Sequential(*layers)
    bf16 = lin.apply_precision_policy(model, 0.15)
    assert bf16 == ["5", "6"]
    x = torch.randn(128, 256, device="cuda", dtype=torch.bfloat16)
    target = torch.randn(128, 256, device="cuda", dtype=torch.bfloat16) * 0.01
    losses = []
    for _ in range(3):
        y = model(x)
        loss = ((y.float() - target.float()) ** 2).mean()
        losses.append(float(loss.detach()))
        model.zero_grad()
        loss.backward()
        with torch.no_grad():
            for p in model.parameters():
                p -= 0.2 * p.grad
    assert all(np.isfinite(losses)) and losses[-1] < losses[0]
    assert all(layer.calls == 3 for layer in layers)
