"""GPU parity of the other weight formats (Q5K, Q6K, NVFP4, INT4 with one scale per 128 columns):
the CUDA path through the C ABI (qmm_fmt_run, qmm_fmt_dequant) against the oracle.

Acceptance as for Q4K: dequantized weights bit-exact; every output element within
|Y - Y_ref| <= 1e-4 * S, S = sum_k |w_k x_k|.
"""
import numpy as np
import pytest
import torch

from bit_quantized_skinny_gb300 import build_lib, inputs

pytestmark = pytest.mark.gpu
TOL = 1e-4
FMTS = ["q5k", "q6k", "nvfp4", "int4"]


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


def fmt_codes(qmm, oracle_lib, name):
    return qmm.FORMATS[name], oracle_lib.FORMATS[name]


def gpu_run(qmm, fmt, Wq_d, N, K, X_d, M):
    pad = 64
    Yfull = torch.full((M * N + pad,), 12345.0, dtype=torch.float32, device="cuda")
    qmm.fmt_run(fmt, Wq_d, N, K, X_d, Yfull, M=M)
    torch.cuda.synchronize()
    Yh = Yfull.cpu().numpy()
    assert np.all(Yh[M * N:] == 12345.0), "write past the end of Y"
    assert qmm.device_status() == 0
    return Yh[:M * N].reshape(M, N)


def assert_within(Y, Yref, S, what=""):
    err = np.abs(Y.astype(np.float64) - Yref)
    bad = err > TOL * S
    if bad.any():
        i, n = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of bound; first at (i={i}, n={n}) "
                             f"y={Y[i, n]!r} ref={Yref[i, n]!r} S={S[i, n]!r}")
    assert np.all(np.isfinite(Y))


_packs = {}


def packed(oracle_lib, ofmt, N, K, seed):
    key = (ofmt, N, K, seed)
    if key not in _packs:
        _packs[key] = oracle_lib.fmt_pack(ofmt, inputs.weights_f32(N, K, seed))
    return _packs[key]


# ------------------------------------------------------------------ dequant ----------------

@pytest.mark.parametrize("fmt_name", FMTS)
@pytest.mark.parametrize("shape", [(256, 512), (33, 2304), (1, 256)])
def test_dequant_bit_exact(qmm, oracle_lib, fmt_name, shape):
    fmt, ofmt = fmt_codes(qmm, oracle_lib, fmt_name)
    N, K = shape
    Wq = packed(oracle_lib, ofmt, N, K, 7 + N)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    qmm.fmt_dequant(fmt, dev_bytes(Wq), N, K, out)
    torch.cuda.synchronize()
    ref = oracle_lib.fmt_dequant(ofmt, Wq, N, K)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("fmt_name", FMTS)
def test_dequant_random_bytes_bit_exact(qmm, oracle_lib, fmt_name):
    """Every field value, not only the packer's: random bytes with the non-finite scale codes
    replaced (NaN E4M3 scales, non-finite binary16 d / dmin / scales)."""
    fmt, ofmt = fmt_codes(qmm, oracle_lib, fmt_name)
    N, K = 64, 1024
    rng = np.random.default_rng(31)
    raw = rng.integers(0, 256, qmm.fmt_packed_bytes(fmt, N, K), dtype=np.uint8)
    if fmt_name == "q5k":
        blocks = raw.reshape(-1, 176)
        for c in (1, 3):
            blocks[:, c] &= 0xFB                    # even exponent field (below 31): finite d, dmin
    elif fmt_name == "nvfp4":
        blocks = raw[:N * (K // 256) * 144].reshape(-1, 144)
        nan = (blocks[:, :16] & 0x7F) == 0x7F
        blocks[:, :16][nan] &= 0xFE
        raw[N * (K // 256) * 144:] = np.frombuffer(np.float32(0.75).tobytes() + bytes(12), np.uint8)
    elif fmt_name == "q6k":
        dp = raw[N * (K // 256) * 208:]
        dp[1::2] &= 0xFB                             # even exponent field: finite d
    else:
        sc = raw[N * K // 2:]
        sc[1::2] &= 0xFB                             # even exponent field: finite scales
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    qmm.fmt_dequant(fmt, dev_bytes(raw), N, K, out)
    torch.cuda.synchronize()
    ref = oracle_lib.fmt_dequant(ofmt, raw, N, K)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------ the product ------------

@pytest.mark.parametrize("fmt_name", FMTS)
@pytest.mark.parametrize("M", [1, 2, 5, 8, 9, 13, 16, 17, 24, 32])
def test_ragged_shape_every_width(qmm, oracle_lib, fmt_name, M):
    """N not a multiple of the 128-row tile, K = 9 super-blocks (a partial 4-block chunk)."""
    fmt, ofmt = fmt_codes(qmm, oracle_lib, fmt_name)
    N, K = 1001, 2304
    Wq = packed(oracle_lib, ofmt, N, K, 41)
    X = inputs.activations_bf16_bits(M, K, 1000 + M)
    Yref, S = oracle_lib.fmt_matmul(ofmt, Wq, N, K, X)
    Y = gpu_run(qmm, fmt, dev_bytes(Wq), N, K, dev_x(X), M)
    assert_within(Y, Yref, S, f"{fmt_name} M={M}")


@pytest.mark.parametrize("fmt_name", FMTS)
@pytest.mark.parametrize("shape,M", [((300, 17408), 3), ((130, 5120), 16), ((64, 2560), 32), ((1, 256), 1)])
def test_split_and_small_shapes(qmm, oracle_lib, fmt_name, shape, M):
    """Few tiles and long rows (the K-split path with its last-arriver reduction), a single
    row, a single super-block."""
    fmt, ofmt = fmt_codes(qmm, oracle_lib, fmt_name)
    N, K = shape
    Wq = packed(oracle_lib, ofmt, N, K, 51 + N)
    X = inputs.activations_bf16_bits(M, K, 77 + M)
    Yref, S = oracle_lib.fmt_matmul(ofmt, Wq, N, K, X)
    Y = gpu_run(qmm, fmt, dev_bytes(Wq), N, K, dev_x(X), M)
    assert_within(Y, Yref, S, f"{fmt_name} {shape} M={M}")


@pytest.mark.parametrize("fmt_name", ["nvfp4", "int4"])
def test_exact_cases_are_bit_exact(qmm, oracle_lib, fmt_name):
    """NVFP4 with g = 1 and power-of-two scales, INT4 with unit scales, integer activations:
    every product and partial sum is an exactly representable number, so the GPU result must
    equal the oracle's bit for bit; one-hot activations reproduce the dequantized weights."""
    fmt, ofmt = fmt_codes(qmm, oracle_lib, fmt_name)
    N, K, M = 384, 1024, 6
    rng = np.random.default_rng(3)
    if fmt_name == "nvfp4":
        raw = rng.integers(0, 256, qmm.fmt_packed_bytes(fmt, N, K), dtype=np.uint8)
        blocks = raw[:N * (K // 256) * 144].reshape(-1, 144)
        blocks[:, :16] = rng.integers(0x30, 0x48, (blocks.shape[0], 16)) & 0xF8   # 2^-1 .. 2^1
        raw[N * (K // 256) * 144:] = np.frombuffer(np.float32(1.0).tobytes() + bytes(12), np.uint8)
    else:
        raw = rng.integers(0, 256, qmm.fmt_packed_bytes(fmt, N, K), dtype=np.uint8)
        raw[N * K // 2:] = np.frombuffer(np.full(N * K // 128, 0x3C00, np.uint16).tobytes(), np.uint8)
    xi = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    X = inputs.bf16_bits_from_f32(xi)
    Yref, _ = oracle_lib.fmt_matmul(ofmt, raw, N, K, X)
    Y = gpu_run(qmm, fmt, dev_bytes(raw), N, K, dev_x(X), M)
    assert np.array_equal(Y.astype(np.float64), Yref)
    ks = [0, 1, 15, 16, 127, 128, 255, 256, 1023]
    eye = np.zeros((len(ks), K), np.float32)
    for r, k in enumerate(ks):
        eye[r, k] = 1.0
    Y1 = gpu_run(qmm, fmt, dev_bytes(raw), N, K, dev_x(inputs.bf16_bits_from_f32(eye)), len(ks))
    w = oracle_lib.fmt_dequant(ofmt, raw, N, K)
    for r, k in enumerate(ks):
        assert np.array_equal(Y1[r], w[:, k]), k


@pytest.mark.parametrize("fmt_name", FMTS)
def test_row_independence_bitwise(qmm, oracle_lib, fmt_name):
    """A row's result does not depend on the other rows of the batch (same kernel width)."""
    fmt, ofmt = fmt_codes(qmm, oracle_lib, fmt_name)
    N, K = 777, 5120
    Wd = dev_bytes(packed(oracle_lib, ofmt, N, K, 61))
    X = inputs.activations_bf16_bits(8, K, 62)
    Y8 = gpu_run(qmm, fmt, Wd, N, K, dev_x(X), 8)
    X2 = X.copy()
    X2[1:] = inputs.activations_bf16_bits(7, K, 63)
    Y8b = gpu_run(qmm, fmt, Wd, N, K, dev_x(X2), 8)
    assert np.array_equal(Y8[0], Y8b[0])


# ------------------------------------------------------------------ full shapes --------------

FULL = [("gate_up", 34816, 5120, [1, 8, 16, 32]), ("down", 5120, 17408, [1, 8])]


@pytest.mark.parametrize("fmt_name", FMTS)
@pytest.mark.parametrize("name,N,K,Ms", FULL, ids=[f[0] for f in FULL])
def test_full_size_sampled_rows(qmm, oracle_lib, fmt_name, name, N, K, Ms):
    """The configurations' FFN shapes in the launch the benchmark times: every output computed
    on the GPU, sampled rows (first, last, random) checked against the oracle."""
    fmt, ofmt = fmt_codes(qmm, oracle_lib, fmt_name)
    seed = inputs.seed_for(2, 0 if name == "gate_up" else 1)
    Wh = qmm.fmt_pack(fmt, inputs.weights_f32(N, K, seed))
    Wd = dev_bytes(Wh)
    rng = np.random.default_rng(N)
    rows = np.unique(np.concatenate([[0, 1, N - 1, N - 2], rng.integers(0, N, 64)])).astype(np.int64)
    for M in Ms:
        X = inputs.activations_bf16_bits(M, K, seed + M)
        Yref, S = oracle_lib.fmt_matmul(ofmt, Wh, N, K, X, rows=rows)
        Y = gpu_run(qmm, fmt, Wd, N, K, dev_x(X), M)
        assert_within(Y[:, rows], Yref, S, f"{fmt_name} {name} M={M}")
    del Wd
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ batched ------------------

@pytest.mark.parametrize("fmt_name", FMTS)
@pytest.mark.parametrize("M", [3, 8, 16, 32])
def test_batched_equals_single_calls(qmm, oracle_lib, fmt_name, M):
    """One launch over several products of one format (shared and distinct X, a product that a
    single call splits along K) gives every product's single-call bits."""
    fmt, ofmt = fmt_codes(qmm, oracle_lib, fmt_name)
    shapes = [(1001, 2304), (300, 17408), (130, 5120), (64, 2560)]
    Xs = {K: dev_x(inputs.activations_bf16_bits(M, K, 300 + K % 97)) for _, K in shapes}
    X2 = dev_x(inputs.activations_bf16_bits(M, 2304, 999))
    items, singles = [], []
    for idx, (N, K) in enumerate(shapes + [(1001, 2304)]):
        Wd = dev_bytes(packed(oracle_lib, ofmt, N, K, 41 if (N, K) == (1001, 2304) else 51 + N))
        X = X2 if idx == len(shapes) else Xs[K]
        Y = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
        items.append((fmt, Wd, X, Y, N, K))
        singles.append(gpu_run(qmm, fmt, Wd, N, K, X, M))
    qmm.fmt_run_batched(qmm.make_fmt_entries(items), M)
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    for (f, Wd, X, Y, N, K), ys in zip(items, singles):
        assert np.array_equal(Y.cpu().numpy().view(np.uint32), ys.view(np.uint32)), (N, K)


def test_batched_many_entries_and_mixed_formats(qmm, oracle_lib):
    """More entries than one launch takes (170 of one format), and every format in one call;
    the Q4K entries go through the library's dispatcher and are checked against the oracle."""
    M = 5
    N, K = 128, 512
    X = inputs.activations_bf16_bits(M, K, 55)
    Xd = dev_x(X)
    items, refs = [], []
    for i in range(170):
        Wq = oracle_lib.fmt_pack(oracle_lib.FMT_NVFP4, inputs.weights_f32(N, K, 1000 + i % 7))
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        items.append((qmm.FMT_NVFP4, dev_bytes(Wq), Xd, Y, N, K))
        refs.append(Wq)
    for name in ["q4k", "q5k", "q6k", "int4", "q4k"]:
        fmt, ofmt = fmt_codes(qmm, oracle_lib, name)
        Wq = oracle_lib.fmt_pack(ofmt, inputs.weights_f32(N, K, 77 + fmt))
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        items.append((fmt, dev_bytes(Wq), Xd, Y, N, K))
        refs.append(Wq)
    qmm.fmt_run_batched(qmm.make_fmt_entries(items), M)
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    for (fmt, Wd, _, Y, _, _), Wq in zip(items, refs):
        ofmt = fmt   # the format codes of the library and of the oracle agree
        Yref, S = oracle_lib.fmt_matmul(ofmt, Wq, N, K, X)
        assert_within(Y.cpu().numpy(), Yref, S, f"fmt {fmt}")
        if fmt != qmm.FMT_Q4K:
            ys = gpu_run(qmm, fmt, Wd, N, K, Xd, M)
            assert np.array_equal(Y.cpu().numpy().view(np.uint32), ys.view(np.uint32))
