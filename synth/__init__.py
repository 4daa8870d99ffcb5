"""Seeded synthetic inputs for the NVFP4 linear-layer path.

This module is the one thing the CUDA path and the CPU oracle share: it makes
bf16 tensors (as raw uint16 bit patterns) and random quantised operands, and
holds none of the method's arithmetic.  The recipe:

* draw in float32 with numpy's PCG64 generator seeded by ``seed``;
* normal:      N(0, sigma^2), optionally with a fraction of entries (chosen
               uniformly without replacement, round(frac*n) of them)
               multiplied by ``outlier_mult``, sign kept;
* student_t:   z / sqrt(chi2_nu / nu) with nu = 3, times ``scale``;
* round float32 -> bf16 to nearest-even on the bit pattern (input encoding).

The workload shapes are those of a 12B-class hybrid model's FFN up-projection
(hidden 5120, FFN 20480, 8192 tokens per micro-batch).
"""
from __future__ import annotations

import numpy as np

HIDDEN = 5120
FFN = 20480
TOKENS = 8192


def _to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(shape, seed: int, sigma: float = 1.0, outlier_frac: float = 0.0,
                outlier_mult: float = 1.0) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seed))
    x = g.standard_normal(size=shape, dtype=np.float32)
    if sigma != 1.0:
        x *= np.float32(sigma)
    n = x.size
    n_out = int(round(outlier_frac * n))
    if n_out:
        idx = g.choice(n, size=n_out, replace=False)
        flat = x.reshape(-1)
        flat[idx] *= np.float32(outlier_mult)
    return _to_bf16_bits(x)


def student_t_bf16(shape, seed: int, nu: int = 3, scale: float = 1e-3) -> np.ndarray:
    g = np.random.Generator(np.random.PCG64(seed))
    z = g.standard_normal(size=shape, dtype=np.float32)
    chi2 = g.chisquare(nu, size=shape).astype(np.float32)
    x = z / np.sqrt(chi2 / np.float32(nu))
    x *= np.float32(scale)
    return _to_bf16_bits(x)


def random_operand(rows: int, k: int, seed: int, scale_lo: int = 0x20, scale_hi: int = 0x50):
    """A random quantised operand for GEMM tests: uniform 4-bit codes, and
    decode-scale bytes drawn uniformly from the E4M3 code range
    [scale_lo, scale_hi] (finite, non-NaN codes) in the plain [rows x k/16]
    layout.  Returns (codes [rows x k/2] uint8, scales_plain uint8)."""
    g = np.random.Generator(np.random.PCG64(seed))
    codes = g.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)
    scales = g.integers(scale_lo, scale_hi + 1, size=(rows, k // 16), dtype=np.uint8)
    return codes, scales


# --- the configurations of the linear-layer workload ------------------------
def tiny_forward(seed: int = 0):
    """128x256 activations N(0,1) with 0.1% x50 outliers; 256x256 weights N(0, 0.02^2)."""
    x = normal_bf16((128, 256), seed, 1.0, 0.001, 50.0)
    w = normal_bf16((256, 256), seed + 7919, 0.02)
    return x, w


def activations(seed: int, tokens: int = TOKENS, hidden: int = HIDDEN):
    """X [tokens x hidden] ~ N(0,1) with 0.05% x100 outliers."""
    return normal_bf16((tokens, hidden), seed, 1.0, 0.0005, 100.0)


def weights(seed: int, ffn: int = FFN, hidden: int = HIDDEN):
    """W [ffn x hidden] ~ N(0, 0.02^2)."""
    return normal_bf16((ffn, hidden), seed, 0.02)


def grad_output(seed: int, tokens: int = TOKENS, ffn: int = FFN):
    """dY [tokens x ffn] ~ 1e-3 * Student-t(3)."""
    return student_t_bf16((tokens, ffn), seed, 3, 1e-3)


# --- device-side generators (for inputs too large to draw on the host) -----
# Same distributions as above, drawn with torch's seeded CUDA generator
# (Philox-based) instead of numpy's PCG64, so the values differ from the host
# generators' but the recipe is the same:
#   normal:    N(0, sigma^2), then round(frac * n) entries chosen uniformly
#              without replacement (the first entries of a seeded random
#              permutation) multiplied by outlier_mult;
#   student_t: z / sqrt(chi2_3 / 3) with chi2_3 = z1^2 + z2^2 + z3^2 (the
#              definition of a chi-square variable with 3 degrees of freedom),
#              times scale;
# then float32 -> bf16 round to nearest even.  Generation runs in row chunks
# to bound the temporary memory.
def _device_generator(seed: int, device: str):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16_device(shape, seed: int, sigma: float = 1.0, outlier_frac: float = 0.0,
                       outlier_mult: float = 1.0, device: str = "cuda"):
    import torch
    rows, cols = shape
    g = _device_generator(seed, device)
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    chunk = max(1, (1 << 26) // cols)
    n = rows * cols
    n_out = int(round(outlier_frac * n))
    idx = torch.randperm(n, generator=g, device=device)[:n_out] if n_out else None
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        x = torch.randn((r1 - r0, cols), generator=g, dtype=torch.float32, device=device)
        if sigma != 1.0:
            x *= sigma
        if idx is not None:
            lo, hi = r0 * cols, r1 * cols
            sel = idx[(idx >= lo) & (idx < hi)] - lo
            x.view(-1)[sel] *= outlier_mult
        out[r0:r1] = x.to(torch.bfloat16)
    return out


def student_t_bf16_device(shape, seed: int, scale: float = 1e-3, device: str = "cuda"):
    import torch
    rows, cols = shape
    g = _device_generator(seed, device)
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=device)
    chunk = max(1, (1 << 25) // cols)
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        z = torch.randn((4, r1 - r0, cols), generator=g, dtype=torch.float32, device=device)
        chi2 = z[1] * z[1] + z[2] * z[2] + z[3] * z[3]
        x = z[0] / torch.sqrt(chi2 / 3.0)
        if scale != 1.0:
            x *= scale
        out[r0:r1] = x.to(torch.bfloat16)
    return out
