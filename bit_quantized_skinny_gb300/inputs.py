"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds none of the product's arithmetic: it only draws the random weights and
activations of the workloads (weights W ~ N(0, 0.02^2) in fp32, activations X ~ N(0, 1)
rounded to bf16), from torch's CPU generator so that every run and every machine sees the
same numbers.  Weight rows are drawn in fixed chunks of ROWS_PER_CHUNK rows, chunk c from its
own seed, so a consumer can stream a large matrix (the 248320-row vocabulary projection)
through any buffer size and still get the same matrix.
"""
from __future__ import annotations

import numpy as np
import torch

ROWS_PER_CHUNK = 4096
WEIGHT_STD = 0.02


def _chunk_seed(seed: int, chunk: int) -> int:
    return (seed * 1_000_003 + chunk * 7919 + 17) & 0x7FFF_FFFF_FFFF


def weight_chunks(N: int, K: int, seed: int):
    """Yield (row0, W_chunk) with W_chunk an fp32 numpy array of shape (rows, K)."""
    g = torch.Generator(device="cpu")
    for c, row0 in enumerate(range(0, N, ROWS_PER_CHUNK)):
        rows = min(ROWS_PER_CHUNK, N - row0)
        g.manual_seed(_chunk_seed(seed, c))
        w = torch.randn(rows, K, generator=g, dtype=torch.float32) * WEIGHT_STD
        yield row0, w.numpy()


def weights_f32(N: int, K: int, seed: int) -> np.ndarray:
    """The whole N x K fp32 weight matrix (only for sizes that fit comfortably in memory)."""
    out = np.empty((N, K), dtype=np.float32)
    for row0, w in weight_chunks(N, K, seed):
        out[row0:row0 + w.shape[0]] = w
    return out


def activations_bf16_bits(M: int, K: int, seed: int) -> np.ndarray:
    """M x K bf16 activations ~ N(0, 1) as uint16 bit patterns (round to nearest even)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(_chunk_seed(seed, 1 << 20))
    x = torch.randn(M, K, generator=g, dtype=torch.float32).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round an fp32 array to bf16 (nearest even) and return the uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


# Seeds of the workloads: seed 0 for the tiny 256 x 512 check, 1000*workload + matrix index
# for the others (workload 2 = one FFN layer, 3 = verify sweep, 4 = 64-layer pass,
# 5 = vocabulary projection).
def seed_for(workload: int, matrix_index: int = 0) -> int:
    return 0 if workload == 1 else 1000 * workload + matrix_index
