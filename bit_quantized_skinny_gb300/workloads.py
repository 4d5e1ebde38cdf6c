"""Synthetic workloads: the matrix shapes of the benchmark configurations and a streaming
generate -> pack -> upload helper that keeps host memory bounded for the 248320-row
vocabulary projection.  Weights follow inputs.weight_chunks (W ~ N(0, 0.02^2)), packed with
the library's host packer.
"""
from __future__ import annotations

import numpy as np

from . import inputs

# One transformer layer's Q4K matrices of the 27B hybrid model the pages run
# (attention projections and the FFN), as (name, N, K).
LAYER_SHAPES = [
    ("q", 5120, 5120),
    ("k", 1024, 5120),
    ("v", 1024, 5120),
    ("o", 5120, 5120),
    ("gate_up", 34816, 5120),
    ("down", 5120, 17408),
]
LM_HEAD = ("lm_head", 248320, 5120)
TINY = ("tiny", 256, 512)


def packed_weights(N: int, K: int, seed: int, device=None, keep_host: bool = False, threads: int = 0):
    """Pack W(N, K, seed) chunk by chunk.  Returns (device_tensor or None, host_bytes or None)."""
    import torch
    from . import qmm

    rowbytes = (K // 256) * 144
    dev = torch.empty(N * rowbytes, dtype=torch.uint8, device=device) if device is not None else None
    host = np.empty(N * rowbytes, dtype=np.uint8) if (keep_host or device is None) else None
    for row0, w in inputs.weight_chunks(N, K, seed):
        rows = w.shape[0]
        buf = qmm.pack(w, threads=threads)
        if host is not None:
            host[row0 * rowbytes:(row0 + rows) * rowbytes] = buf
        if dev is not None:
            dev[row0 * rowbytes:(row0 + rows) * rowbytes].copy_(torch.from_numpy(buf), non_blocking=False)
    return dev, host


def packed_weights_fmt(fmt: int, N: int, K: int, seed: int, device="cuda"):
    """A device buffer of an N x K matrix in weight format `fmt` for timing: the first
    min(N, ROWS_PER_CHUNK) rows of W(N, K, seed) packed with the library's packer, their bytes
    repeated down to row N (the kernels have no data-dependent paths, so the content does not
    change the timing).  INT4 and Q6K repeat both of their planes; NVFP4 keeps the first chunk's
    tensor scale."""
    import torch
    from . import qmm

    rows = min(N, inputs.ROWS_PER_CHUNK)
    _, w = next(inputs.weight_chunks(N, K, seed))
    chunk = torch.from_numpy(qmm.fmt_pack(fmt, w[:rows])).to(device)
    out = torch.empty(qmm.fmt_packed_bytes(fmt, N, K), dtype=torch.uint8, device=device)
    if fmt == qmm.FMT_INT4:
        planes = [(K // 2, 0, 0), (K // 64, N * (K // 2), rows * (K // 2))]   # (row bytes, out offset, chunk offset)
    elif fmt == qmm.FMT_Q6K:
        rb = (K // 256) * 208
        planes = [(rb, 0, 0), ((K // 256) * 2, N * rb, rows * rb)]
    else:
        rb = (K // 256) * (176 if fmt == qmm.FMT_Q5K else 144)
        planes = [(rb, 0, 0)]
    for row_bytes, off, coff in planes:
        src = chunk[coff:coff + rows * row_bytes]
        for r0 in range(0, N, rows):
            n = min(rows, N - r0)
            out[off + r0 * row_bytes:off + (r0 + n) * row_bytes].copy_(src[:n * row_bytes])
    if fmt == qmm.FMT_NVFP4:
        out[-16:].copy_(chunk[-16:])
    return out


def activations(M: int, K: int, seed: int, device=None):
    """(torch bf16 tensor on `device`, host uint16 bits) of M x K activations."""
    import torch
    bits = inputs.activations_bf16_bits(M, K, seed)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16)
    return (t.to(device) if device is not None else t), bits
