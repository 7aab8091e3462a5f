"""Seeded synthetic inputs for the NF4 linear layer.

This module draws random numbers and nothing else: it holds none of the NF4 arithmetic (no table,
no scale rule, no rounding of weights), so the CPU oracle and the CUDA library can both be fed
from it without sharing any of the method's code.

Distributions follow the workloads the NF4 pages run: weights W ~ N(0, 0.02) in fp32, optionally
with a fraction of outliers drawn from N(0, 0.2); activations x ~ N(0, 1) rounded to bf16 (the
rounding is torch's own float32 -> bfloat16 cast).
"""
from __future__ import annotations

import numpy as np
import torch

WEIGHT_STD = 0.02
OUTLIER_STD = 0.2


def weights(seed: int, n: int, k: int, std: float = WEIGHT_STD, outlier_frac: float = 0.0,
            outlier_std: float = OUTLIER_STD) -> np.ndarray:
    """fp32 [n, k] host weights from numpy's PCG64 stream ``seed``."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((n, k), dtype=np.float32) * np.float32(std)
    if outlier_frac > 0.0:
        mask = rng.random((n, k), dtype=np.float32) < outlier_frac
        w[mask] = rng.standard_normal(int(mask.sum()), dtype=np.float32) * np.float32(outlier_std)
    return w


def activations_bf16(seed: int, m: int, k: int) -> np.ndarray:
    """bf16 bit patterns (uint16) [m, k] of x ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((m, k), dtype=np.float32))
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def device_weights(seed: int, n: int, k: int, device, std: float = WEIGHT_STD,
                   outlier_frac: float = 0.0, outlier_std: float = OUTLIER_STD) -> torch.Tensor:
    """fp32 [n, k] weights drawn on ``device`` with torch's counter-based (Philox) CUDA generator.

    Used for the multi-gigabyte layer sweeps; a test that checks such a layer copies the same fp32
    tensor back to the host, so both sides see identical bytes.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w = torch.randn((n, k), generator=g, device=device, dtype=torch.float32) * std
    if outlier_frac > 0.0:
        mask = torch.rand((n, k), generator=g, device=device) < outlier_frac
        w = torch.where(mask, torch.randn((n, k), generator=g, device=device) * outlier_std, w)
    return w


def device_activations_bf16(seed: int, m: int, k: int, device) -> torch.Tensor:
    """bf16 [m, k] x ~ N(0, 1) drawn on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn((m, k), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def device_packed(seed: int, n: int, k: int, device, scale_lo: float = 0.01, scale_hi: float = 0.1):
    """Random packed weights drawn on ``device``: uint8 code bytes [n, k/2], uniform over all 256
    values, and fp16 scales [n, k/64], uniform in [scale_lo, scale_hi) rounded by torch's cast.

    For runs too large to quantize from fp32 weights (tens of GB); a test that checks such a linear
    copies the rows it checks back to the host, so both sides see identical bytes.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    codes = torch.randint(0, 256, (n, k // 2), generator=g, device=device, dtype=torch.uint8)
    scales = (torch.rand((n, k // 64), generator=g, device=device) * (scale_hi - scale_lo) + scale_lo).to(torch.float16)
    return codes, scales
