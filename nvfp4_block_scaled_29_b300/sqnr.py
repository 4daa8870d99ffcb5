"""Quantisation-error harness: NVFP4 against MXFP4, with and without the
16-point random Hadamard transform, on the path's own quantisers.

The pages' claims it measures:
  * NVIDIA blog "NVFP4 Trains with Precision of 16-Bit and Speed and
    Efficiency of 4-Bit", recipe bullets 1-2: 16-element blocks and E4M3
    scales represent values more precisely than MXFP4's 32-element blocks
    with power-of-two scales;
  * the same blog, bullet 3, and prism.simon-ai.net article 7890,
    "Techniques against outliers and rounding error": the Hadamard transform
    reshapes outlier-heavy distributions so that they quantise better.

For each tensor and setting the harness quantises on the GPU (the C-ABI
calls), dequantises, and reports SQNR = 10 log10(sum x^2 / sum (x - x_hat)^2)
and the MSE against the exact reference, in float64.  With the RHT the
reference is RHT16(x) along k (the transform is orthogonal, so the error
energy equals the error of inverting it back).
"""
from __future__ import annotations

import math

import torch

from . import (MxQTensor, QTensor, nvfp4_amax, nvfp4_dequantize, nvfp4_mx_dequantize,
               nvfp4_mx_quantize, nvfp4_quantize_1d, nvfp4_rht_quantize, NVFP4_RNE)


def hadamard16(mask: int, device="cuda") -> torch.Tensor:
    """The 16 x 16 matrix of x -> H16 diag(s) x / 4 (Sylvester order, s_j = -1
    where bit j of mask is set), float64: RHT16(x) = x @ M for a row x."""
    idx = torch.arange(16, device=device)
    pop = torch.tensor([bin(int(v)).count("1") for v in (idx[:, None] & idx[None, :]).flatten()],
                       device=device).reshape(16, 16)
    h = torch.where(pop % 2 == 0, 1.0, -1.0).to(torch.float64)
    s = torch.tensor([-1.0 if (mask >> j) & 1 else 1.0 for j in range(16)], dtype=torch.float64, device=device)
    # y_i = 1/4 sum_j H[i, j] s_j x_j  ->  y = x @ (diag(s) H^T) / 4
    return (torch.diag(s) @ h.t()) / 4.0


def _reference(x: torch.Tensor, mask: int) -> torch.Tensor:
    xd = x.to(torch.float64)
    if not mask:
        return xd
    r, k = xd.shape
    return (xd.reshape(r, k // 16, 16) @ hadamard16(mask, x.device)).reshape(r, k)


def _dequant_nvfp4(x: torch.Tensor, mask: int) -> torch.Tensor:
    r, k = x.shape
    q = QTensor(r, k)
    amax = nvfp4_amax(x, mask)
    if mask:
        nvfp4_rht_quantize(x, mask, amax, NVFP4_RNE, 0, 0, q)
    else:
        nvfp4_quantize_1d(x, amax, NVFP4_RNE, 0, 0, q)
    out = torch.empty((r, k), dtype=torch.float32, device=x.device)
    nvfp4_dequantize(q, out)
    return out


def _dequant_mxfp4(x: torch.Tensor, mask: int) -> torch.Tensor:
    r, k = x.shape
    q = MxQTensor(r, k)
    nvfp4_mx_quantize(x, mask, q)
    out = torch.empty((r, k), dtype=torch.float32, device=x.device)
    nvfp4_mx_dequantize(q, out)
    return out


def measure(x: torch.Tensor, fmt: str, mask: int = 0) -> dict:
    """SQNR (dB) and MSE of one quantisation of the bf16 tensor x [rows x k]
    (k % 32 == 0): fmt "nvfp4" (1x16, E4M3 scales, FP32 tensor scale, RNE) or
    "mxfp4" (1x32, E8M0 scales, RNE); mask != 0 applies RHT-16 along k."""
    if fmt not in ("nvfp4", "mxfp4"):
        raise ValueError("fmt must be 'nvfp4' or 'mxfp4'")
    deq = (_dequant_nvfp4 if fmt == "nvfp4" else _dequant_mxfp4)(x, mask).to(torch.float64)
    ref = _reference(x, mask)
    err = float(((ref - deq) ** 2).sum())
    sig = float((ref ** 2).sum())
    return {"format": fmt, "rht": bool(mask), "sqnr_db": 10.0 * math.log10(sig / err) if err > 0 else math.inf,
            "mse": err / ref.numel()}


def table(tensors: dict, mask: int) -> list[dict]:
    """measure() for every tensor x {NVFP4, MXFP4} x {no RHT, RHT}."""
    rows = []
    for name, x in tensors.items():
        for fmt in ("nvfp4", "mxfp4"):
            for m in (0, mask):
                rows.append({"tensor": name, **measure(x, fmt, m)})
    return rows


def main(argv=None) -> int:
    """Print the SQNR table for the linear step's synthetic tensors (a
    1024-token slice of X, W's first 1024 rows and a 1024-token slice of dY,
    k = the GEMM reduction dimension of each) as a markdown table."""
    import argparse
    import os
    import sys

    import numpy as np

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import synth
    from . import nvfp4_rht_mask_from_seed

    ap = argparse.ArgumentParser()
    ap.add_argument("--rows", type=int, default=1024)
    ap.add_argument("--rht-seed", type=int, default=2004)
    args = ap.parse_args(argv)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    tensors = {
        "X: N(0,1) + 0.05% x100 outliers": dev(synth.activations(2, tokens=args.rows)),
        "W: N(0, 0.02^2)": dev(synth.weights(3, ffn=args.rows)),
        "dY: 1e-3 t3": dev(synth.grad_output(3 + 7919, tokens=args.rows)),
    }
    rows = table(tensors, nvfp4_rht_mask_from_seed(args.rht_seed))
    print("| tensor | format | RHT-16 | SQNR dB | MSE |")
    print("|---|---|---|---|---|")
    for r in rows:
        print(f"| {r['tensor']} | {r['format']} | {'yes' if r['rht'] else 'no'} | {r['sqnr_db']:.2f} | {r['mse']:.4e} |")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
