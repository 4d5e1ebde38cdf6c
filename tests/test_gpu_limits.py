"""The largest sizes the C ABI accepts: K = 2^20 (4096 super-blocks per row: the longest K
split and the most chunk partials) for every weight format and both kernel families, and a
batched call of QMM_MAX_BATCH = 512 entries (four launches of at most 160 products), against
the oracle and against single calls.
"""
import numpy as np
import pytest
import torch

from bit_quantized_skinny_gb300 import build_lib, inputs

pytestmark = pytest.mark.gpu
TOL = 1e-4
K_MAX = 1 << 20


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


def check(Y, Yref, S, what):
    err = np.abs(Y.astype(np.float64) - Yref)
    assert np.all(err <= TOL * S), f"{what}: max err / S = {np.max(err / np.maximum(S, 1e-300))}"
    assert np.all(np.isfinite(Y))


@pytest.mark.parametrize("fmt_name", ["q4k", "q5k", "q6k", "nvfp4", "int4"])
def test_longest_rows(qmm, oracle_lib, fmt_name):
    fmt = qmm.FORMATS[fmt_name]
    N = 3
    Wq = oracle_lib.fmt_pack(fmt, inputs.weights_f32(N, K_MAX, 91))
    Wd = dev_bytes(Wq)
    for M in (1, 8, 32):
        X = inputs.activations_bf16_bits(M, K_MAX, 92 + M)
        Yref, S = oracle_lib.fmt_matmul(fmt, Wq, N, K_MAX, X)
        variants = [qmm.VARIANT_FMA, qmm.VARIANT_TC] if fmt == qmm.FMT_Q4K else [None]
        for v in variants:
            Y = torch.full((M * N + 16,), 4242.0, dtype=torch.float32, device="cuda")
            if v is None:
                qmm.fmt_run(fmt, Wd, N, K_MAX, dev_x(X), Y, M=M)
            else:
                qmm.run(Wd, N, K_MAX, dev_x(X), Y, M=M, variant=v)
            torch.cuda.synchronize()
            assert qmm.device_status() == 0
            yh = Y.cpu().numpy()
            assert np.all(yh[M * N:] == 4242.0)
            check(yh[:M * N].reshape(M, N), Yref, S, f"{fmt_name} K=2^20 M={M} variant={v}")


def test_largest_batch(qmm, oracle_lib):
    """512 entries (the maximum) of assorted small shapes sharing M; each result equals the
    single call with the same kernel family bit for bit and the oracle within tolerance."""
    M = 6
    rng = np.random.default_rng(5)
    shapes = [(int(rng.choice([1, 64, 129, 256])), 256 * int(rng.integers(1, 5))) for _ in range(512)]
    Xs = {K: dev_x(inputs.activations_bf16_bits(M, K, 300 + K)) for K in {k for _, k in shapes}}
    packs = {}
    items, ys = [], []
    for i, (N, K) in enumerate(shapes):
        if (N, K) not in packs:
            packs[(N, K)] = oracle_lib.pack(inputs.weights_f32(N, K, 40 + N + K))
        Wd = dev_bytes(packs[(N, K)])
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        items.append((Wd, Xs[K], Y, N, K))
        ys.append(Y)
    entries = qmm.make_entries(items)
    variant = qmm.select_variant_batched(entries, M)
    qmm.run_batched(entries, M)
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    for idx in list(range(0, 512, 37)) + [159, 160, 319, 320, 479, 480, 511]:
        Wd, Xd, Y, N, K = items[idx]
        Ys = torch.empty((M, N), dtype=torch.float32, device="cuda")
        qmm.run(Wd, N, K, Xd, Ys, M=M, variant=variant)
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int32), Ys.view(torch.int32)), idx
        X = inputs.activations_bf16_bits(M, K, 300 + K)
        Yref, S = oracle_lib.matmul(packs[(N, K)], N, K, X)
        check(Y.cpu().numpy(), Yref, S, f"entry {idx}")
