"""Layer shapes of the synthetic workloads (K = in-features, N = out-features, M = tokens).

The shapes are those of the dense models the NF4 pages run (Qwen2.5-3B/14B/32B-shaped decode and a
20B-shaped prefill); the weights are random, never a checkpoint.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Tuple


@dataclass(frozen=True)
class Linear:
    name: str
    k: int  # in-features
    n: int  # out-features


@dataclass(frozen=True)
class Workload:
    name: str
    linears: Tuple[Linear, ...]
    layers: int
    tokens: Tuple[int, ...]
    seed: int
    outlier_frac: float = 0.0

    def weights_per_layer(self) -> int:
        return sum(l.n * l.k for l in self.linears)

    def packed_bytes_per_pass(self) -> int:
        """Codes (K/2 bytes per row) plus fp16 scales (K/64 per row), all layers."""
        per_layer = sum(l.n * (l.k // 2) + l.n * (l.k // 64) * 2 for l in self.linears)
        return per_layer * self.layers


def _decode_layer(hidden: int, kv: int, inter: int) -> Tuple[Linear, ...]:
    return (Linear("q", hidden, hidden), Linear("k", hidden, kv), Linear("v", hidden, kv),
            Linear("o", hidden, hidden), Linear("gate", hidden, inter), Linear("up", hidden, inter),
            Linear("down", inter, hidden))


SINGLE_2048 = Workload("single linear 2048x2048, M=1", (Linear("linear", 2048, 2048),), 1, (1,), 0)
DECODE_3B = Workload("3B-shaped decode, hidden 2048, 36 layers, M=1", _decode_layer(2048, 256, 11008),
                     36, (1,), 1)
DECODE_14B = Workload("14B-shaped decode, hidden 5120, 48 layers, M in {1,4,8}",
                      _decode_layer(5120, 1024, 13824), 48, (1, 4, 8), 2)
SWEEP_32B = Workload("32B-shaped decode sweep, hidden 5120, intermediate 27648, 64 layers, M=1",
                     _decode_layer(5120, 1024, 27648), 64, (1,), 3)
PREFILL_20B = Workload("20B-shaped prefill, hidden 6144, intermediate 16384, M in {32,512}",
                       (Linear("gate", 6144, 16384), Linear("up", 6144, 16384),
                        Linear("down", 16384, 6144), Linear("qkv", 6144, 8192)),
                       1, (32, 512), 4, outlier_frac=0.01)

ALL: List[Workload] = [SINGLE_2048, DECODE_3B, DECODE_14B, SWEEP_32B, PREFILL_20B]
