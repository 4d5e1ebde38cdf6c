"""Randomized parity: seeded random shapes, row counts, weight formats and kernel families, as
single products and as mixed batches, against the oracle (every output within
1e-4 * sum_k |w_k x_k|).  The draws span ragged N, K from one to 40 super-blocks (the K-split
path of single products included), every M from 1 to 32, and random weights of random scale.
"""
import numpy as np
import pytest
import torch

from bit_quantized_skinny_gb300 import build_lib, inputs

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module")
def qmm():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    build_lib.build()
    from bit_quantized_skinny_gb300 import qmm as q
    q.load()
    return q


def dev_bytes(host_u8):
    a = np.ascontiguousarray(host_u8)
    return torch.from_numpy(a if a.flags.writeable else a.copy()).cuda()


def dev_x(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).cuda().view(torch.bfloat16)


def draw(rng):
    fmt = int(rng.integers(0, 5))
    N = int(rng.choice([1, 2, 127, 128, 129, 300, 640, 1000, 1500]))
    K = 256 * int(rng.choice([1, 2, 3, 5, 8, 9, 17, 24, 40]))
    M = int(rng.integers(1, 33))
    scale = float(np.exp(rng.uniform(-6, 4)))
    return fmt, N, K, M, scale


def weights(N, K, seed, scale):
    return (inputs.weights_f32(N, K, seed) * np.float32(scale / 0.02)).astype(np.float32)


def check(Y, Yref, S, what):
    err = np.abs(Y.astype(np.float64) - Yref)
    bad = err > TOL * S
    assert not bad.any(), f"{what}: {bad.sum()} out of bound, max err / S = {np.max(err / np.maximum(S, 1e-300))}"
    assert np.all(np.isfinite(Y))


@pytest.mark.parametrize("seed", range(6))
def test_random_single_products(qmm, oracle_lib, seed):
    rng = np.random.default_rng(1000 + seed)
    for case in range(12):
        fmt, N, K, M, scale = draw(rng)
        Wq = oracle_lib.fmt_pack(fmt, weights(N, K, 10 * seed + case, scale))
        X = inputs.activations_bf16_bits(M, K, 77 * seed + case)
        Yref, S = oracle_lib.fmt_matmul(fmt, Wq, N, K, X)
        Wd, Xd = dev_bytes(Wq), dev_x(X)
        variants = [qmm.VARIANT_FMA, qmm.VARIANT_TC] if fmt == qmm.FMT_Q4K else [None]
        for v in variants:
            Y = torch.full((M * N + 32,), 4242.0, dtype=torch.float32, device="cuda")
            if v is None:
                qmm.fmt_run(fmt, Wd, N, K, Xd, Y, M=M)
            else:
                qmm.run(Wd, N, K, Xd, Y, M=M, variant=v)
            torch.cuda.synchronize()
            assert qmm.device_status() == 0
            yh = Y.cpu().numpy()
            assert np.all(yh[M * N:] == 4242.0), "write past the end of Y"
            check(yh[:M * N].reshape(M, N), Yref, S, f"fmt={fmt} N={N} K={K} M={M} scale={scale:.3g} variant={v}")


@pytest.mark.parametrize("seed", range(3))
def test_random_mixed_batches(qmm, oracle_lib, seed):
    rng = np.random.default_rng(2000 + seed)
    M = int(rng.integers(1, 33))
    items, refs = [], []
    Xs = {}
    for case in range(10):
        fmt, N, K, _, scale = draw(rng)
        Wq = oracle_lib.fmt_pack(fmt, weights(N, K, 500 + 10 * seed + case, scale))
        if K not in Xs:
            bits = inputs.activations_bf16_bits(M, K, 900 + K)
            Xs[K] = (bits, dev_x(bits))
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        items.append((fmt, dev_bytes(Wq), Xs[K][1], Y, N, K))
        refs.append((fmt, Wq, N, K, Xs[K][0]))
    qmm.fmt_run_batched(qmm.make_fmt_entries(items), M)
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    for (fmt, _, _, Y, N, K), (_, Wq, _, _, Xb) in zip(items, refs):
        Yref, S = oracle_lib.fmt_matmul(fmt, Wq, N, K, Xb)
        check(Y.cpu().numpy(), Yref, S, f"batched fmt={fmt} N={N} K={K} M={M}")
