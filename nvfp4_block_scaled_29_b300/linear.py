"""NVFP4 linear layer for training, over the libnvfp4 C ABI.

The forward, dgrad and wgrad products of a linear layer run as NVFP4 GEMMs
with the recipe of NVIDIA blog "NVFP4 Trains with Precision of 16-Bit and
Speed and Efficiency of 4-Bit", section "NVFP4 quantization recipe for
pre-training":

  * activations X and output gradients dY in 1x16 blocks (bullet 1), E4M3
    block scales under an FP32 per-tensor scale (bullet 2);
  * the weight W in 16x16 blocks, so that the forward operand W and the dgrad
    operand W^T come from one encoding (bullet 4);
  * the 16-point random Hadamard transform on the wgrad inputs dY^T and X^T,
    one sign mask shared by both (bullet 3);
  * stochastic rounding of dY (bullet 5); X and W round to nearest.  The
    rounding mode of dY is NVFP4_SR (16 independent Philox bits per element)
    or NVFP4_SR_HW (the same rule with the random bits in the layout of the
    hardware FP4 stochastic-rounding conversion, 32 bits per 4 elements;
    faster).

X and dY are each read once for both of their operands (nvfp4_amax_dual /
nvfp4_quantize_dual).  The forward saves the quantised X^T and W^T for the
backward instead of the BF16 tensors.

Per-layer precision opt-out: the prism.simon-ai.net article 7890, section
"Training stability and protection of sensitive layers", states that
quantising every linear layer to FP4 diverges and that the last 15% of the
network's layers need higher precision.  `apply_precision_policy` marks the
last fraction of a model's NVFP4Linear layers (15% by default) to run in
BF16.
"""
from __future__ import annotations

import math

import torch

from . import (NVFP4_RNE, NVFP4_SR, NVFP4_SR_HW, QTensor, nvfp4_amax, nvfp4_amax_dual, nvfp4_gemm,
               nvfp4_quantize_2d, nvfp4_quantize_dual, nvfp4_rht_mask_from_seed)

# Philox stream ids of the two stochastic-rounding draws of a step
STREAM_DGRAD, STREAM_WGRAD = 1, 2


_SIDE_STREAMS: dict = {}


def _side_stream(device) -> "torch.cuda.Stream":
    """One side stream per device, for the weight's quantisation."""
    idx = torch.device(device).index
    idx = torch.cuda.current_device() if idx is None else idx
    if idx not in _SIDE_STREAMS:
        _SIDE_STREAMS[idx] = torch.cuda.Stream(device=idx)
    return _SIDE_STREAMS[idx]


def _check_shapes(tokens: int, k_in: int, k_out: int):
    # every GEMM reduction dimension (k_in: fprop, k_out: dgrad, tokens:
    # wgrad) must be a multiple of 32
    for name, v in (("tokens", tokens), ("in_features", k_in), ("out_features", k_out)):
        if v % 32 != 0:
            raise ValueError(f"NVFP4 linear needs {name} % 32 == 0 (got {v})")


class NVFP4LinearFunction(torch.autograd.Function):
    """y = x w^T with x [tokens x in], w [out x in] (bf16, CUDA); returns y bf16.

    seed selects the Philox stream of this call's stochastic rounding; rht_mask
    the 16-bit Hadamard sign mask (one per call, shared by dY^T and X^T);
    sr_round the rounding mode of dY (NVFP4_SR or NVFP4_SR_HW)."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, w: torch.Tensor, seed: int, rht_mask: int, sr_round: int = NVFP4_SR):
        tokens, k_in = x.shape
        k_out = w.shape[0]
        _check_shapes(tokens, k_in, k_out)
        x = x.contiguous()
        w = w.contiguous()
        amax = torch.empty((3,), dtype=torch.float32, device=x.device)
        qx, qxt = QTensor(tokens, k_in), QTensor(k_in, tokens)
        qw, qwt = QTensor(k_out, k_in, True), QTensor(k_in, k_out, True)
        # W's amax and 16x16 quantise run on a side stream beside X's
        main, side = torch.cuda.current_stream(x.device), _side_stream(x.device)
        fork = torch.cuda.Event()
        fork.record(main)
        side.wait_event(fork)
        with torch.cuda.stream(side):
            nvfp4_amax(w, 0, amax[2:3])
            nvfp4_quantize_2d(w, amax[2:3], NVFP4_RNE, 0, 0, qw, qwt)
        # buffers made on the main stream and used on the side stream
        for t in (w, amax, qw.codes, qw.scales, qw.global_scale, qwt.codes, qwt.scales, qwt.global_scale):
            t.record_stream(side)
        nvfp4_amax_dual(x, rht_mask, amax[0:1], amax[1:2])
        nvfp4_quantize_dual(x, amax[0:1], NVFP4_RNE, 0, 0, qx, rht_mask, amax[1:2], NVFP4_RNE, 0, 0, qxt)
        join = torch.cuda.Event()
        join.record(side)
        main.wait_event(join)
        y = torch.empty((tokens, k_out), dtype=torch.bfloat16, device=x.device)
        nvfp4_gemm(qx, qw, y)
        ctx.q = (qxt, qwt)
        ctx.seed, ctx.rht_mask, ctx.sr_round = seed, rht_mask, sr_round
        return y

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        qxt, qwt = ctx.q
        dy = dy.contiguous().to(torch.bfloat16)
        tokens, k_out = dy.shape
        k_in = qwt.rows
        amax = torch.empty((2,), dtype=torch.float32, device=dy.device)
        qdy, qdyt = QTensor(tokens, k_out), QTensor(k_out, tokens)
        nvfp4_amax_dual(dy, ctx.rht_mask, amax[0:1], amax[1:2])
        nvfp4_quantize_dual(dy, amax[0:1], ctx.sr_round, ctx.seed, STREAM_DGRAD, qdy, ctx.rht_mask, amax[1:2],
                            ctx.sr_round, ctx.seed, STREAM_WGRAD, qdyt)
        dx = torch.empty((tokens, k_in), dtype=torch.bfloat16, device=dy.device)
        dw = torch.empty((k_out, k_in), dtype=torch.bfloat16, device=dy.device)
        nvfp4_gemm(qdy, qwt, dx)                  # dX = dY W
        nvfp4_gemm(qdyt, qxt, dw)                 # dW = dY^T X, k = tokens, RHT on both
        ctx.q = None
        return dx, dw, None, None, None


class NVFP4Linear(torch.nn.Module):
    """Linear layer (no bias) whose three products run in NVFP4, or in BF16
    when `precision` is "bf16" (the per-layer opt-out).  Inputs of any
    leading shape are flattened to [tokens x in_features].

    Each forward call draws a fresh stochastic-rounding seed and Hadamard
    mask from the layer's seed and its call counter, so consecutive steps see
    independent rounding noise while a run stays reproducible."""

    def __init__(self, in_features: int, out_features: int, *, precision: str = "nvfp4",
                 seed: int = 0, device="cuda", dtype=torch.bfloat16, sr_round: int = NVFP4_SR):
        super().__init__()
        if precision not in ("nvfp4", "bf16"):
            raise ValueError("precision must be 'nvfp4' or 'bf16'")
        if sr_round not in (NVFP4_SR, NVFP4_SR_HW):
            raise ValueError("sr_round must be NVFP4_SR or NVFP4_SR_HW")
        self.sr_round = sr_round
        self.in_features, self.out_features = in_features, out_features
        self.precision = precision
        self.seed = seed
        self.calls = 0
        w = torch.empty((out_features, in_features), device=device, dtype=dtype)
        torch.nn.init.normal_(w, std=1.0 / math.sqrt(in_features))
        self.weight = torch.nn.Parameter(w)

    def extra_repr(self) -> str:
        return f"in_features={self.in_features}, out_features={self.out_features}, precision={self.precision}"

    def call_seed(self) -> int:
        return (self.seed * 0x9E3779B97F4A7C15 + self.calls) & 0xFFFFFFFFFFFFFFFF

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        lead = x.shape[:-1]
        x2 = x.reshape(-1, self.in_features)
        if self.precision == "bf16":
            y = x2.to(torch.bfloat16) @ self.weight.t()
        else:
            s = self.call_seed()
            # mask 0 would switch the transform off in the C ABI: use 1 instead
            mask = nvfp4_rht_mask_from_seed(s ^ 0x5EED) or 1
            y = NVFP4LinearFunction.apply(x2.to(torch.bfloat16), self.weight, s, mask, self.sr_round)
        self.calls += 1
        return y.reshape(*lead, self.out_features)


def apply_precision_policy(model: torch.nn.Module, keep_last_fraction: float = 0.15) -> list[str]:
    """Run the last `keep_last_fraction` of the model's NVFP4Linear layers (in
    module registration order, rounded up to whole layers) in BF16, the rest
    in NVFP4.  Returns the names of the BF16 layers."""
    if not 0.0 <= keep_last_fraction <= 1.0:
        raise ValueError("keep_last_fraction must be in [0, 1]")
    layers = [(n, m) for n, m in model.named_modules() if isinstance(m, NVFP4Linear)]
    n_bf16 = math.ceil(len(layers) * keep_last_fraction - 1e-9)
    cut = len(layers) - n_bf16
    for i, (_, m) in enumerate(layers):
        m.precision = "nvfp4" if i < cut else "bf16"
    return [n for n, _ in layers[cut:]]
