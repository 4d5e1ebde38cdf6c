"""GPU parity: the CUDA path (through the C ABI) against the oracle.

Acceptance (the product's stated bar): dequantized weights bit-exact; every output element
within |Y - Y_ref| <= 1e-4 * S with S = sum_k |w_k x_k| (S = 0 demands an exact 0).
"""
import numpy as np
import pytest
import torch

from bit_quantized_skinny_gb300 import build_lib, inputs, workloads

pytestmark = pytest.mark.gpu
TOL = 1e-4
FMA, TC = 1, 2
VARIANTS = [pytest.param(FMA, id="fma"), pytest.param(TC, id="tc")]


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


def gpu_run(qmm, Wq_d, N, K, X_d, M, variant=0, canary=True):
    pad = 64
    Yfull = torch.full((M * N + pad,), 12345.0, dtype=torch.float32, device="cuda")
    qmm.run(Wq_d, N, K, X_d, Yfull, M=M, variant=variant)
    torch.cuda.synchronize()
    Yh = Yfull.cpu().numpy()
    if canary:
        assert np.all(Yh[M * N:] == 12345.0), "write past the end of Y"
    assert qmm.device_status() == 0
    return Yh[:M * N].reshape(M, N)


def assert_within(Y, Yref, S, what=""):
    err = np.abs(Y.astype(np.float64) - Yref)
    bound = TOL * S
    bad = err > bound
    if bad.any():
        i, n = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of bound; first at (i={i}, n={n}) "
                             f"y={Y[i, n]!r} ref={Yref[i, n]!r} S={S[i, n]!r}")
    assert np.all(np.isfinite(Y))


# ------------------------------------------------------------------ dequant ----------------

@pytest.mark.parametrize("shape", [(256, 512), (33, 2304), (1, 256)])
def test_dequant_bit_exact(qmm, oracle_lib, shape):
    N, K = shape
    Wq = oracle_lib.pack(inputs.weights_f32(N, K, 7 + N))
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    qmm.dequant(dev_bytes(Wq), N, K, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = oracle_lib.dequant(Wq, N, K)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_extreme_fields_bit_exact(qmm, oracle_lib):
    from test_oracle_pins import EXTREME_BLOCKS, make_block, read_golden_block
    blocks = [make_block(*b) for b in EXTREME_BLOCKS] + [read_golden_block()]
    rng = np.random.default_rng(0)
    blocks += [bytes(rng.integers(0, 256, 144, dtype=np.uint8)) for _ in range(64)]
    blocks = [b for b in blocks if np.isfinite(np.frombuffer(b[:4], np.float16)).all()]
    Wq = np.frombuffer(b"".join(blocks), dtype=np.uint8)
    N = len(blocks)
    out = torch.empty((N, 256), dtype=torch.float32, device="cuda")
    qmm.dequant(dev_bytes(Wq), N, 256, out)
    torch.cuda.synchronize()
    ref = oracle_lib.dequant(Wq, N, 256)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


# ------------------------------------------------------------------ the product ------------

@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_config(qmm, oracle_lib, variant):
    """256 x 512 weights from W ~ N(0, 0.02^2), seed 0; M = 1 and 4."""
    N, K = 256, 512
    Wq = oracle_lib.pack(inputs.weights_f32(N, K, inputs.seed_for(1)))
    Wd = dev_bytes(Wq)
    for M in (1, 4):
        X = inputs.activations_bf16_bits(M, K, inputs.seed_for(1))
        Yref, S = oracle_lib.matmul(Wq, N, K, X)
        Y = gpu_run(qmm, Wd, N, K, dev_x(X), M, variant=variant)
        assert_within(Y, Yref, S, f"tiny M={M}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M", list(range(1, 33)))
def test_every_M_ragged_shape(qmm, oracle_lib, M, variant):
    """N not a multiple of the 4-row box, K = 9 super-blocks (a partial 4-block chunk)."""
    N, K = 1001, 2304
    Wq = _cached_pack(oracle_lib, N, K, 41)
    X = inputs.activations_bf16_bits(M, K, 1000 + M)
    Yref, S = oracle_lib.matmul(Wq, N, K, X)
    Y = gpu_run(qmm, dev_bytes(Wq), N, K, dev_x(X), M, variant=variant)
    assert_within(Y, Yref, S, f"M={M}")


_pack_cache = {}


def _cached_pack(oracle_lib, N, K, seed):
    key = (N, K, seed)
    if key not in _pack_cache:
        _pack_cache[key] = oracle_lib.pack(inputs.weights_f32(N, K, seed))
    return _pack_cache[key]


@pytest.mark.parametrize("shape", [(1, 256), (3, 256), (5, 512), (4, 1024), (7, 1280), (130, 4352)])
@pytest.mark.parametrize("M", [1, 2, 3, 32])
@pytest.mark.parametrize("variant", VARIANTS)
def test_small_and_degenerate_shapes(qmm, oracle_lib, shape, M, variant):
    N, K = shape
    Wq = _cached_pack(oracle_lib, N, K, 5)
    X = inputs.activations_bf16_bits(M, K, 77)
    Yref, S = oracle_lib.matmul(Wq, N, K, X)
    Y = gpu_run(qmm, dev_bytes(Wq), N, K, dev_x(X), M, variant=variant)
    assert_within(Y, Yref, S, f"{shape} M={M}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_integer_activations_are_exact(qmm, oracle_lib, variant):
    """Constant blocks (w = 0.25*3*5 - 0.125*7 = 2.875) and small integer x: every partial sum
    is exact in fp32, so the GPU must equal the closed form w0 * sum_k x bit for bit."""
    from test_oracle_pins import make_block
    N, K, M = 70, 3072, 5
    blk = make_block(0x3400, 0x3000, [3] * 8, [7] * 8, [5] * 256)
    Wq = np.frombuffer(blk * (N * K // 256), dtype=np.uint8)
    xi = np.random.default_rng(2).integers(-20, 21, size=(M, K)).astype(np.float32)
    X = inputs.bf16_bits_from_f32(xi)
    Y = gpu_run(qmm, dev_bytes(Wq), N, K, dev_x(X), M, variant=variant)
    expect = (2.875 * xi.astype(np.float64).sum(axis=1))[:, None] * np.ones((1, N))
    assert np.array_equal(Y.astype(np.float64), expect)


@pytest.mark.parametrize("variant", VARIANTS)
def test_zero_weights_give_exact_zero(qmm, variant):
    N, K, M = 40, 1024, 3
    Wq = np.zeros(N * K // 256 * 144, np.uint8)
    X = inputs.activations_bf16_bits(M, K, 3)
    Y = gpu_run(qmm, dev_bytes(Wq), N, K, dev_x(X), M, variant=variant)
    assert np.all(Y == 0.0)


@pytest.mark.parametrize("variant", VARIANTS)
def test_one_hot_activations_reproduce_dequant(qmm, oracle_lib, variant):
    N, K = 96, 2048
    Wq = _cached_pack(oracle_lib, N, K, 13)
    ks = [0, 1, 255, 256, 1023, 1024, 2047, 517]
    eye = np.zeros((len(ks), K), np.float32)
    for r, k in enumerate(ks):
        eye[r, k] = 1.0
    Y = gpu_run(qmm, dev_bytes(Wq), N, K, dev_x(inputs.bf16_bits_from_f32(eye)), len(ks), variant=variant)
    w = oracle_lib.dequant(Wq, N, K)
    for r, k in enumerate(ks):
        assert np.array_equal(Y[r], w[:, k])


@pytest.mark.parametrize("variant", VARIANTS)
def test_row_independence_bitwise(qmm, oracle_lib, variant):
    """For a fixed variant, an M-row product equals M one-row products bit for bit."""
    N, K, M = 777, 5120, 9
    Wq = _cached_pack(oracle_lib, N, K, 17)
    Wd = dev_bytes(Wq)
    X = inputs.activations_bf16_bits(M, K, 18)
    Yall = gpu_run(qmm, Wd, N, K, dev_x(X), M, variant=variant)
    for i in range(M):
        Yi = gpu_run(qmm, Wd, N, K, dev_x(X[i:i + 1]), 1, variant=variant)
        assert np.array_equal(Yi[0].view(np.uint32), Yall[i].view(np.uint32)), i


@pytest.mark.parametrize("M", [4, 24])
def test_batched_equals_single_calls(qmm, oracle_lib, M):
    """One batched launch equals the single-matrix calls of the kernel family that ran it, bit
    for bit (each family's arithmetic does not depend on how the work is split), and every
    entry is within the tolerance of the oracle."""
    shapes = [(512, 5120), (128, 5120), (96, 17408), (1001, 2304), (3, 256), (2048, 512)]
    items, singles, refs = [], {FMA: [], TC: []}, []
    for k, (N, K) in enumerate(shapes):
        Wq = _cached_pack(oracle_lib, N, K, 300 + k)
        X = inputs.activations_bf16_bits(M, K, 400 + k)
        Wd, Xd = dev_bytes(Wq), dev_x(X)
        Y = torch.full((M, N), -1.0, device="cuda")
        items.append((Wd, Xd, Y, N, K))
        for v in (FMA, TC):
            singles[v].append(gpu_run(qmm, Wd, N, K, Xd, M, variant=v))
        refs.append(oracle_lib.matmul(Wq, N, K, X))
    ents = qmm.make_entries(items)
    qmm.run_batched(ents, M)
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    got = [Y.cpu().numpy() for (_, _, Y, _, _) in items]
    same = {v: all(np.array_equal(g.view(np.uint32), s.view(np.uint32)) for g, s in zip(got, singles[v]))
            for v in (FMA, TC)}
    assert same[FMA] or same[TC], "batched launch differs from the single calls of both families"
    for g, (Yref, S), (N, K) in zip(got, refs, shapes):
        assert_within(g, Yref, S, f"batched {N}x{K}")


def test_batched_shared_x(qmm, oracle_lib):
    """Entries may share one X (the q/k/v projections of a layer read the same activations)."""
    K, M = 5120, 8
    X = inputs.activations_bf16_bits(M, K, 55)
    Xd = dev_x(X)
    items, checks = [], []
    for k, N in enumerate([5120, 1024, 1024]):
        Wq = _cached_pack(oracle_lib, N, K, 500 + k)
        Y = torch.empty((M, N), device="cuda")
        items.append((dev_bytes(Wq), Xd, Y, N, K))
        checks.append((Wq, N, Y))
    qmm.run_batched(qmm.make_entries(items), M)
    torch.cuda.synchronize()
    for Wq, N, Y in checks:
        rows = np.arange(0, N, 7)
        Yref, S = oracle_lib.matmul(Wq, N, K, X, rows=rows)
        assert_within(Y.cpu().numpy()[:, rows], Yref, S, f"shared-x {N}")


def test_misaligned_pointers_rejected(qmm):
    N, K = 8, 256
    Wd = torch.zeros(N * 144 + 32, dtype=torch.uint8, device="cuda")
    Xd = torch.zeros(K + 16, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(N + 4, device="cuda")
    st = qmm.run_raw(Wd.data_ptr() + 8, N, K, Xd.data_ptr(), Y.data_ptr(), 1)
    assert st == 4
    st = qmm.run_raw(Wd.data_ptr(), N, K, Xd.data_ptr() + 2, Y.data_ptr(), 1)
    assert st == 4
    assert qmm.run_raw(Wd.data_ptr(), N, K, Xd.data_ptr(), Y.data_ptr(), 1) == 0
    torch.cuda.synchronize()


def test_release_frees_the_workspaces_and_calls_allocate_again(qmm, oracle_lib):
    """After qmm_release the tensor-core workspaces are gone (0 bytes held, the device memory
    back); the next call allocates again and computes the same bits."""
    N, K, M = 1001, 5120, 8
    Wq = _cached_pack(oracle_lib, N, K, 19)
    X = inputs.activations_bf16_bits(M, K, 20)
    Wd, Xd = dev_bytes(Wq), dev_x(X)
    Y1 = gpu_run(qmm, Wd, N, K, Xd, M, variant=TC)
    assert qmm.workspace_bytes_held() > 0
    free_before = torch.cuda.mem_get_info()[0]
    held = qmm.workspace_bytes_held()
    qmm.release()
    assert qmm.workspace_bytes_held() == 0
    assert torch.cuda.mem_get_info()[0] >= free_before + held - (2 << 20)
    Y2 = gpu_run(qmm, Wd, N, K, Xd, M, variant=TC)
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
    assert qmm.workspace_bytes_held() > 0


# ------------------------------------------------------------------ full sizes --------------

FULL = [
    ("gate_up", 34816, 5120, [1, 2, 8, 16]),
    ("down", 5120, 17408, [1, 3, 8]),
    ("q", 5120, 5120, [1, 4, 12]),
    ("k", 1024, 5120, [1, 7, 16]),
    ("lm_head", 248320, 5120, [1, 7]),
]


@pytest.mark.parametrize("name,N,K,Ms", FULL, ids=[f[0] for f in FULL])
def test_full_size_sampled_rows(qmm, oracle_lib, name, N, K, Ms):
    """Both variants and the automatic choice, on the configurations' full shapes."""
    """The configurations' full shapes, in the launch the benchmark times: every output is
    computed on the GPU; sampled rows (first, last, random) are checked against the oracle.
    The sampled rows' packed bytes are also checked against the oracle's packer."""
    seed = inputs.seed_for(5 if name == "lm_head" else 2, 0)
    Wd, Wh = workloads.packed_weights(N, K, seed, device="cuda", keep_host=True)
    rng = np.random.default_rng(N)
    rows = np.unique(np.concatenate([[0, 1, N - 1, N - 2], rng.integers(0, N, 96)])).astype(np.int64)
    rowbytes = K // 256 * 144
    W = inputs.weights_f32(min(N, 4096), K, seed)          # first chunk of rows, same draw
    first = rows[rows < W.shape[0]]
    assert np.array_equal(oracle_lib.pack(W[first]), Wh.reshape(N, rowbytes)[first].reshape(-1))
    for M in Ms:
        X = inputs.activations_bf16_bits(M, K, seed + M)
        Yref, S = oracle_lib.matmul(Wh, N, K, X, rows=rows)
        for variant in (0, FMA, TC):
            Y = gpu_run(qmm, Wd, N, K, dev_x(X), M, variant=variant)
            assert_within(Y[:, rows], Yref, S, f"{name} M={M} variant={variant}")
    del Wd
    torch.cuda.empty_cache()
