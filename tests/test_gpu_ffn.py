"""GPU parity of the feed-forward chain (qmm_run_ffn): gate/up product -> SiLU-gated bf16
activations -> down product, through the C ABI, against the oracle step by step.

The chain is checked where each result is defined:
  G (fp32, the gate/up product)  within 1e-4 * sum|w x| of the oracle, per element;
  H (bf16)                       within one bf16 step of the oracle's fp64 SwiGLU of the GPU's G
                                 (the GPU rounds an fp32 value, the oracle an fp64 one);
  Y (fp32, the down product)     within 1e-4 * sum|w x| of the oracle fed the GPU's H.
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


def _dev_bytes(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _dev_x(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).cuda().view(torch.bfloat16)


def _within(Y, Yref, S, what):
    err = np.abs(Y.astype(np.float64) - Yref)
    bad = err > TOL * S
    assert not bad.any(), f"{what}: {bad.sum()} elements out of bound, max err {err.max()}"
    assert np.all(np.isfinite(Y))


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("F,K,Ms", [(512, 256, [1, 3, 8]), (768, 512, [16, 32]), (1024, 1024, [2, 9])])
def test_ffn_chain_step_by_step(qmm, oracle_lib, F, K, Ms):
    Wgu = oracle_lib.pack(inputs.weights_f32(2 * F, K, 700 + F))
    Wdn = oracle_lib.pack(inputs.weights_f32(K, F, 800 + F))
    Wgu_d, Wdn_d = _dev_bytes(Wgu), _dev_bytes(Wdn)
    for M in Ms:
        X = inputs.activations_bf16_bits(M, K, 900 + M)
        Y = torch.full((M, K), 7.0, dtype=torch.float32, device="cuda")
        ws = torch.zeros(qmm.ffn_workspace_bytes(M, F), dtype=torch.uint8, device="cuda")
        qmm.run_ffn(Wgu_d, Wdn_d, F, K, _dev_x(X), Y, ws, M=M)
        torch.cuda.synchronize()
        assert qmm.device_status() == 0
        wsh = ws.cpu().numpy()
        g_bytes = (M * 2 * F * 4 + 15) // 16 * 16
        G = wsh[:M * 2 * F * 4].view(np.float32).reshape(M, 2 * F)
        H = wsh[g_bytes:g_bytes + M * F * 2].view(np.uint16).reshape(M, F)
        Gref, SG = oracle_lib.matmul(Wgu, 2 * F, K, X)
        _within(G, Gref, SG, f"gate/up M={M}")
        href = oracle_lib.swiglu(G.astype(np.float64), F)
        hg = _bf16_to_f64(H)
        step = np.ldexp(1.0, np.frexp(np.abs(href))[1] - 8)       # one bf16 step at |href|
        assert np.all(np.abs(hg - href) <= step), f"H off by more than one bf16 step at M={M}"
        assert np.mean(H == oracle_lib.bf16_round(href)) > 0.99   # nearly all round identically
        Yref, SY = oracle_lib.matmul(Wdn, K, F, H)
        _within(Y.cpu().numpy(), Yref, SY, f"down M={M}")


def test_ffn_argument_errors(qmm):
    F, K, M = 256, 256, 2
    W = torch.zeros(2 * F * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    X = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((M, K), device="cuda")
    small = torch.zeros(qmm.ffn_workspace_bytes(M, F) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qmm.QmmError) as ei:
        qmm.run_ffn(W, W, F, K, X, Y, small, M=M)
    assert ei.value.status == 5   # QMM_ERR_BUFSIZE
    assert qmm.ffn_workspace_bytes(M, 100) == 0   # F not a multiple of 256


def _interleave_rows(packed, F, K):
    """Packed (2F) x K Q4K rows (gate 0..F-1, up F..2F-1) -> rows 2f = gate f, 2f+1 = up f."""
    rows = packed.reshape(2 * F, (K // 256) * 144)
    out = np.empty_like(rows)
    out[0::2] = rows[:F]
    out[1::2] = rows[F:]
    return out.reshape(-1)


@pytest.mark.parametrize("F,K,Ms", [(512, 256, [1, 3, 8]), (768, 512, [16, 32]), (1536, 1024, [2, 9, 24])])
def test_fused_ffn_matches_the_chain(qmm, oracle_lib, F, K, Ms):
    """qmm_run_ffn_fused on the row-interleaved gate/up matrix: H is the SwiGLU of the gate/up
    product's fp32 results (checked against the oracle's fp64 SwiGLU of the tensor-core product
    of the same rows, within one bf16 step and nearly always identical), equal bit for bit to
    the unfused chain's H whenever that chain's gate/up product runs on the tensor cores too, and
    Y is the down product of H."""
    Wgu = oracle_lib.pack(inputs.weights_f32(2 * F, K, 710 + F))
    Wdn = oracle_lib.pack(inputs.weights_f32(K, F, 810 + F))
    Wgu_d, Wint_d, Wdn_d = _dev_bytes(Wgu), _dev_bytes(_interleave_rows(Wgu, F, K)), _dev_bytes(Wdn)
    for M in Ms:
        X = inputs.activations_bf16_bits(M, K, 910 + M)
        Xd = _dev_x(X)
        Yf = torch.full((M, K), 7.0, dtype=torch.float32, device="cuda")
        wsf = torch.full((qmm.ffn_fused_workspace_bytes(M, F),), 255, dtype=torch.uint8, device="cuda")
        qmm.run_ffn_fused(Wint_d, Wdn_d, F, K, Xd, Yf, wsf, M=M)
        Gtc = torch.empty((M, 2 * F), dtype=torch.float32, device="cuda")
        qmm.run(Wgu_d, 2 * F, K, Xd, Gtc, M=M, variant=qmm.VARIANT_TC)
        Yu = torch.full((M, K), 7.0, dtype=torch.float32, device="cuda")
        wsu = torch.zeros(qmm.ffn_workspace_bytes(M, F), dtype=torch.uint8, device="cuda")
        qmm.run_ffn(Wgu_d, Wdn_d, F, K, Xd, Yu, wsu, M=M)
        torch.cuda.synchronize()
        assert qmm.device_status() == 0
        Hf = wsf.cpu().numpy()[:M * F * 2].view(np.uint16).reshape(M, F)
        G = Gtc.cpu().numpy()
        Gref, SG = oracle_lib.matmul(Wgu, 2 * F, K, X)
        _within(G, Gref, SG, f"gate/up M={M}")
        href = oracle_lib.swiglu(G.astype(np.float64), F)
        step = np.ldexp(1.0, np.frexp(np.abs(href))[1] - 8)
        assert np.all(np.abs(_bf16_to_f64(Hf) - href) <= step), f"fused H off by more than one bf16 step, M={M}"
        assert np.mean(Hf == oracle_lib.bf16_round(href)) > 0.99
        if qmm.select_variant(M, 2 * F, K) == qmm.VARIANT_TC:
            g_bytes = (M * 2 * F * 4 + 15) // 16 * 16
            Hu = wsu.cpu().numpy()[g_bytes:g_bytes + M * F * 2].view(np.uint16).reshape(M, F)
            assert np.array_equal(Hf, Hu), f"fused and chained H differ, M={M}"
            assert torch.equal(Yf.view(torch.int32), Yu.view(torch.int32))
        Yref, SY = oracle_lib.matmul(Wdn, K, F, Hf)
        _within(Yf.cpu().numpy(), Yref, SY, f"fused down M={M}")


def test_fused_ffn_argument_errors(qmm):
    F, K, M = 256, 256, 2
    W = torch.zeros(2 * F * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    X = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((M, K), device="cuda")
    small = torch.zeros(qmm.ffn_fused_workspace_bytes(M, F) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(qmm.QmmError) as ei:
        qmm.run_ffn_fused(W, W, F, K, X, Y, small, M=M)
    assert ei.value.status == 5
    assert qmm.ffn_fused_workspace_bytes(M, 100) == 0
    assert qmm.ffn_fused_workspace_bytes(M, F) == M * F * 2


@pytest.mark.parametrize("M", [1, 8, 32])
def test_full_size_ffn_chain_and_fused(qmm, oracle_lib, M):
    """The configurations' FFN layer (gate/up 34816 x 5120, down 5120 x 17408) through qmm_run_ffn
    and qmm_run_ffn_fused, on sampled rows: G within 1e-4 * sum|w x| of the oracle; H within one
    bf16 step of the oracle's SwiGLU of the GPU's G (and of the fused block's own H: identical
    when both gate/up products run on the tensor cores); Y within 1e-4 * sum|w x| of the oracle's
    down product of the GPU's H.  The sampled rows' packed bytes equal the oracle packer's."""
    from bit_quantized_skinny_gb300 import workloads
    F, K = 17408, 5120
    Wgu_d, Wgu = workloads.packed_weights(2 * F, K, inputs.seed_for(2, 0), device="cuda", keep_host=True)
    Wdn_d, Wdn = workloads.packed_weights(K, F, inputs.seed_for(2, 1), device="cuda", keep_host=True)
    rowbytes = (K // 256) * 144
    W0 = inputs.weights_f32(64, K, inputs.seed_for(2, 0))          # the first rows of the same draw
    assert np.array_equal(oracle_lib.pack(W0), Wgu[:64 * rowbytes])
    Wint_d = _dev_bytes(_interleave_rows(Wgu, F, K))
    rng = np.random.default_rng(M)
    fs = np.unique(np.concatenate([[0, F - 1], rng.integers(0, F, 62)])).astype(np.int64)
    ys = np.unique(np.concatenate([[0, K - 1], rng.integers(0, K, 62)])).astype(np.int64)
    X = inputs.activations_bf16_bits(M, K, 950 + M)
    Xd = _dev_x(X)
    Y = torch.full((M, K), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.zeros(qmm.ffn_workspace_bytes(M, F), dtype=torch.uint8, device="cuda")
    qmm.run_ffn(Wgu_d, Wdn_d, F, K, Xd, Y, ws, M=M)
    Yf = torch.full((M, K), 7.0, dtype=torch.float32, device="cuda")
    wsf = torch.full((qmm.ffn_fused_workspace_bytes(M, F),), 255, dtype=torch.uint8, device="cuda")
    qmm.run_ffn_fused(Wint_d, Wdn_d, F, K, Xd, Yf, wsf, M=M)
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    wsh = ws.cpu().numpy()
    g_bytes = (M * 2 * F * 4 + 15) // 16 * 16
    G = wsh[:M * 2 * F * 4].view(np.float32).reshape(M, 2 * F)
    H = wsh[g_bytes:g_bytes + M * F * 2].view(np.uint16).reshape(M, F)
    Hf = wsf.cpu().numpy()[:M * F * 2].view(np.uint16).reshape(M, F)
    rows = np.concatenate([fs, F + fs])
    Gref, SG = oracle_lib.matmul(Wgu, 2 * F, K, X, rows=rows)
    _within(G[:, rows], Gref, SG, f"full gate/up M={M}")
    href = oracle_lib.swiglu(G[:, rows].astype(np.float64), len(fs))
    step = np.ldexp(1.0, np.frexp(np.abs(href))[1] - 8)
    for what, HH in (("chained", H), ("fused", Hf)):
        assert np.all(np.abs(_bf16_to_f64(HH[:, fs]) - href) <= step), f"{what} H off by more than one bf16 step"
    assert np.mean(H[:, fs] == oracle_lib.bf16_round(href)) > 0.99
    if qmm.select_variant(M, 2 * F, K) == qmm.VARIANT_TC:
        assert np.array_equal(H, Hf), "fused and chained H differ"
    for what, HH, YY in (("chained", H, Y), ("fused", Hf, Yf)):
        Yref, SY = oracle_lib.matmul(Wdn, K, F, HH, rows=ys)
        _within(YY.cpu().numpy()[:, ys], Yref, SY, f"full {what} down M={M}")
    del Wgu_d, Wdn_d, Wint_d
    torch.cuda.empty_cache()
