"""GPU parity on the inputs where a fast kernel's arithmetic could lose the acceptance bound.

The bound |Y - Y_ref| <= 1e-4 * S, S = sum_k |w_k x_k|, is per element (S = 0 demands an exact
0), so it is tightest where S is small against the magnitudes the arithmetic handles:
  * k-quant blocks whose fields cancel, d*sc_j*q = dmin*m_j: such weights are exactly 0, and a
    row whose weights all cancel must give exactly 0; near-cancelling fields give tiny weights;
  * random field bytes pushed through the product: every d/dmin ratio and every field value;
  * activations spanning far more than fp16's range inside one super-block (bf16 subnormals
    included), paired with weights so that S is made of the small products only.
Both kernel families, both k-quant widths, and for the activation range every weight format.
The blocks are built from their fields by the written layouts (the helpers of the oracle pins).
"""
import numpy as np
import pytest
import torch

from bit_quantized_skinny_gb300 import build_lib, inputs
from test_oracle_formats import q5k_block
from test_oracle_pins import make_block

pytestmark = pytest.mark.gpu
TOL = 1e-4
FMA, TC = 1, 2


@pytest.fixture(scope="module")
def qmm():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    build_lib.build()
    from bit_quantized_skinny_gb300 import qmm as q
    q.load()
    return q


def dev_bytes(host_u8):
    return torch.from_numpy(np.ascontiguousarray(host_u8).copy()).cuda()


def dev_x(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).cuda().view(torch.bfloat16)


def run(qmm, fmt, Wq, N, K, X, variant=0):
    M = X.shape[0]
    pad = 64
    Yfull = torch.full((M * N + pad,), 12345.0, dtype=torch.float32, device="cuda")
    Wd, Xd = dev_bytes(Wq), dev_x(X)
    if fmt == "q4k":
        qmm.run(Wd, N, K, Xd, Yfull, M=M, variant=variant)
    else:
        qmm.fmt_run(qmm.FORMATS[fmt], Wd, N, K, Xd, Yfull, M=M)
    torch.cuda.synchronize()
    Yh = Yfull.cpu().numpy()
    assert np.all(Yh[M * N:] == 12345.0), "write past the end of Y"
    assert qmm.device_status() == 0
    return Yh[:M * N].reshape(M, N)


def assert_within(Y, Yref, S, what):
    assert np.all(np.isfinite(Y)), what
    err = np.abs(Y.astype(np.float64) - Yref)
    bad = err > TOL * S
    if bad.any():
        i, n = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of bound; first (i={i}, n={n}) "
                             f"y={Y[i, n]!r} ref={Yref[i, n]!r} S={S[i, n]!r} err/S={err[i, n] / max(S[i, n], 1e-300):.3g}")


def h16(v):
    b = int(np.array([v], dtype=np.float16).view(np.uint16)[0])
    assert float(np.array([b], np.uint16).view(np.float16)[0]) == v, v
    return b


def next16(bits, step):
    """The fp16 pattern `step` units of the last place away from a positive fp16 pattern."""
    return bits + step


# Triples (sc, q*, m) with sc * q* = m * 2^p for p = -2..2: with dmin = d * 2^p every weight
# d*sc*q* - dmin*m of such a sub-block is exactly 0.
def _cancel_triples():
    out = {}
    for p in range(-2, 3):
        ts = []
        for sc in range(1, 64):
            for q in range(0, 16):
                for m in range(0, 64):
                    if sc * q * 4 == m * int(4 * 2.0 ** p):
                        ts.append((sc, q, m))
        out[p] = ts
    return out


CANCEL = _cancel_triples()


def cancelling_q4k(N, K, rng, frac=1.0, near=0, wide_q=False, width=4):
    """N x K k-quant weights (width 4: Q4K, 5: Q5K) whose sub-blocks cancel: with probability
    `frac` a sub-block has q == q* throughout (exact zeros, or with `near` != 0 dmin moved by
    `near` units in the last place: tiny constant weights; with wide_q, q in q* - 1 .. q* + 1),
    otherwise random quants.  d is a random normal fp16 per super-block."""
    blocks = []
    qmax = 15 if width == 4 else 31
    for _ in range(N * (K // 256)):
        p = int(rng.integers(-2, 3))
        e = int(rng.integers(-8, 5))
        d = float(rng.integers(1024, 2048)) * 2.0 ** (e - 10)
        d_bits = h16(d)
        dmin_bits = next16(h16(d * 2.0 ** p), near)
        sc, m, q = [], [], []
        for j in range(8):
            s_, q_, m_ = CANCEL[p][int(rng.integers(len(CANCEL[p])))]
            sc.append(s_)
            m.append(m_)
            if rng.random() < frac:
                if wide_q:
                    q += [int(np.clip(q_ + rng.integers(-1, 2), 0, qmax)) for _ in range(32)]
                else:
                    q += [q_] * 32
            else:
                q += [int(v) for v in rng.integers(0, qmax + 1, 32)]
        blocks.append(make_block(d_bits, dmin_bits, sc, m, q) if width == 4 else q5k_block(d_bits, dmin_bits, sc, m, q))
    return np.frombuffer(b"".join(blocks), dtype=np.uint8)


def random_blocks(nblocks, nbytes, rng):
    """Random bytes with finite binary16 d and dmin (a non-finite one is redrawn)."""
    raw = rng.integers(0, 256, size=(nblocks, nbytes), dtype=np.uint8)
    for b in range(nblocks):
        while True:
            hdr = raw[b, :4].view(np.float16)
            if np.isfinite(hdr).all():
                break
            raw[b, :4] = rng.integers(0, 256, 4, dtype=np.uint8)
    return raw.reshape(-1)


M_LIST = [1, 3, 8, 9, 16, 17, 32]


# ------------------------------------------------------------------ the min term ----------

@pytest.mark.parametrize("variant", [FMA, TC])
def test_exact_cancellation_gives_exact_zero(qmm, oracle_lib, variant):
    """d = dmin = 1, sc = 1, m = 3, q = 3 everywhere: every weight is exactly 0, so S = 0 and
    Y must be exactly 0 for any activations."""
    N, K = 130, 2048
    blk = make_block(h16(1.0), h16(1.0), [1] * 8, [3] * 8, [3] * 256)
    Wq = np.frombuffer(blk * (N * K // 256), dtype=np.uint8)
    assert not oracle_lib.dequant(Wq, N, K).any()
    for M in M_LIST:
        X = inputs.activations_bf16_bits(M, K, 900 + M)
        Y = run(qmm, "q4k", Wq, N, K, X, variant)
        assert np.all(Y == 0.0), (M, np.abs(Y).max())


@pytest.mark.parametrize("fmt,variant", [("q4k", FMA), ("q4k", TC), ("q5k", 0)])
def test_cancelling_fields_random(qmm, oracle_lib, fmt, variant):
    """Random cancelling triples (sc, q*, m) with dmin = d 2^p: rows that cancel throughout
    give exact zeros; rows with some random sub-blocks stay within the bound."""
    ofmt = oracle_lib.FORMATS[fmt]
    width = 4 if fmt == "q4k" else 5
    rng = np.random.default_rng(11)
    N, K = 257, 2304
    for frac in (1.0, 0.75):
        Wq = cancelling_q4k(N, K, rng, frac=frac, width=width)
        for M in (1, 8, 13, 32):
            X = inputs.activations_bf16_bits(M, K, 70 + M)
            Yref, S = oracle_lib.fmt_matmul(ofmt, Wq, N, K, X)
            if frac == 1.0:
                assert not S.any()
            assert_within(run(qmm, fmt, Wq, N, K, X, variant), Yref, S, f"{fmt} frac={frac} M={M}")


@pytest.mark.parametrize("fmt,variant", [("q4k", FMA), ("q4k", TC), ("q5k", 0)])
@pytest.mark.parametrize("near,wide_q", [(1, False), (-1, False), (3, True)])
def test_near_cancelling_fields(qmm, oracle_lib, fmt, variant, near, wide_q):
    """dmin one or a few units in the last place away from cancelling: tiny weights, or tiny
    ones mixed with weights one quant step away."""
    ofmt = oracle_lib.FORMATS[fmt]
    width = 4 if fmt == "q4k" else 5
    rng = np.random.default_rng(20 + near)
    N, K = 130, 1280
    Wq = cancelling_q4k(N, K, rng, near=near, wide_q=wide_q, width=width)
    for M in (1, 7, 16, 24):
        X = inputs.activations_bf16_bits(M, K, 80 + M)
        Yref, S = oracle_lib.fmt_matmul(ofmt, Wq, N, K, X)
        assert_within(run(qmm, fmt, Wq, N, K, X, variant), Yref, S, f"{fmt} near={near} M={M}")


@pytest.mark.parametrize("fmt,variant", [("q4k", FMA), ("q4k", TC), ("q5k", 0)])
def test_random_field_bytes_through_the_product(qmm, oracle_lib, fmt, variant):
    """Random bytes (finite d, dmin): every d/dmin ratio from 2^-40 to 2^40, every field."""
    ofmt = oracle_lib.FORMATS[fmt]
    nbytes = 144 if fmt == "q4k" else 176
    rng = np.random.default_rng(31)
    N, K = 257, 2304
    Wq = random_blocks(N * K // 256, nbytes, rng)
    for M in (1, 5, 8, 13, 32):
        X = inputs.activations_bf16_bits(M, K, 90 + M)
        Yref, S = oracle_lib.fmt_matmul(ofmt, Wq, N, K, X)
        assert_within(run(qmm, fmt, Wq, N, K, X, variant), Yref, S, f"{fmt} random bytes M={M}")


# ------------------------------------------------------------------ activation range ------

def _zero_first_sub_block(W):
    """Weights whose first 32 columns of every 256 are 0 (every format packs them to exact
    zeros: a k-quant sub-block or NVFP4 block of zeros gets scale 0, INT4 and Q6K quantize 0 to
    the code of 0)."""
    W = W.copy()
    W.reshape(W.shape[0], -1, 256)[:, :, :32] = 0.0
    return W


def _wide_tokens(K, seed):
    """Activation rows (bf16 bits) whose range inside a super-block is far beyond fp16's:
    positions 0..31 of every 256 (paired with zero weights) hold values near 1 (or 2^100), the
    rest much smaller values, so S is made of the small products only."""
    rng = np.random.default_rng(seed)
    big = rng.standard_normal((1, K)).astype(np.float32)
    first = (np.arange(K) % 256) < 32
    rows = []
    for scale_big, scale_small in [(1.0, 2.0 ** -40), (1.0, 2.0 ** -100), (1.0, 1.0), (2.0 ** 100, 1.0),
                                   (2.0 ** -120, 2.0 ** -120), (1.0, 2.0 ** -20), (1.0, 2.0 ** -30)]:
        r = rng.standard_normal(K).astype(np.float64) * scale_small
        r[first] = big[0, first] * scale_big
        rows.append(r)
    X = inputs.bf16_bits_from_f32(np.array(rows, dtype=np.float32))
    # a row of bf16 subnormals (random patterns 0x0001..0x007f, random signs) after large values
    sub = rng.integers(1, 128, K).astype(np.uint16) | (rng.integers(0, 2, K).astype(np.uint16) << 15)
    sub[first] = X[0, first]
    return np.vstack([X, sub[None, :]])


@pytest.mark.parametrize("fmt", ["q4k", "q5k", "q6k", "nvfp4", "int4"])
def test_activation_range_beyond_fp16(qmm, oracle_lib, fmt):
    ofmt = oracle_lib.FORMATS[fmt]
    N, K = 300, 2304
    W = _zero_first_sub_block(inputs.weights_f32(N, K, 41) * 50.0)
    Wq = oracle_lib.fmt_pack(ofmt, W)
    Xall = _wide_tokens(K, 5)
    variants = [FMA, TC] if fmt == "q4k" else [0]
    for M in (Xall.shape[0], 16, 32):
        X = Xall[np.arange(M) % Xall.shape[0]]
        Yref, S = oracle_lib.fmt_matmul(ofmt, Wq, N, K, X)
        assert (S > 0).all()
        for v in variants:
            assert_within(run(qmm, fmt, Wq, N, K, X, v), Yref, S, f"{fmt} wide X M={M} variant={v}")


@pytest.mark.parametrize("variant", [FMA, TC])
@pytest.mark.parametrize("k", [10, 17, 19, 20, 21, 22, 25, 40])
def test_small_subblock_sums_next_to_large_activations(qmm, oracle_lib, variant, k):
    """Sub-block 0: cancelling weights (exact zeros) under activations near 1; sub-block 1: a
    constant tiny weight (dmin one unit off) under activations near 2^-k; zeros elsewhere.  S is
    then |w| sum |x| of sub-block 1 alone, and the min term carries the whole result: its
    activation sums must keep their precision (or the token must take the exact path)."""
    N, K, M = 70, 512, 4
    rng = np.random.default_rng(k)
    zero = make_block(h16(1.0), h16(1.0), [0] * 8, [0] * 8, [0] * 256)
    blocks = []
    for _ in range(N):
        # super-block 1: sub-block 0 zero (sc = m = 0), sub-block 1 the weight 3 - 3 dmin
        near = make_block(h16(1.0), h16(1.0) + int(rng.integers(1, 3)), [0, 1] + [0] * 6, [0, 3] + [0] * 6,
                          [0] * 32 + [3] * 32 + [0] * 192)
        blocks += [zero, near]
    Wq = np.frombuffer(b"".join(blocks), dtype=np.uint8)
    X = np.zeros((M, K), np.float32)
    X[:, :32] = rng.standard_normal((M, 32))
    X[:, 256:288] = rng.standard_normal((M, 32))                       # large, under zero weights
    X[:, 288:320] = rng.standard_normal((M, 32)) * 2.0 ** -k            # small, under the tiny weight
    Xb = inputs.bf16_bits_from_f32(X)
    Yref, S = oracle_lib.matmul(Wq, N, K, Xb)
    assert (S > 0).all()
    assert_within(run(qmm, "q4k", Wq, N, K, Xb, variant), Yref, S, f"k={k}")


@pytest.mark.parametrize("fmt", ["q4k", "nvfp4"])
def test_row_independence_with_wide_tokens(qmm, oracle_lib, fmt):
    """Each token's staging is its own: an M-row product equals the M one-row products bit for
    bit, also when some rows take the exact CUDA-core path (tensor-core family)."""
    ofmt = oracle_lib.FORMATS[fmt]
    N, K = 400, 2304
    Wq = oracle_lib.fmt_pack(ofmt, _zero_first_sub_block(inputs.weights_f32(N, K, 43)))
    X = _wide_tokens(K, 6)[[0, 2, 1, 7, 3]]
    variant = TC if fmt == "q4k" else 0
    Yall = run(qmm, fmt, Wq, N, K, X, variant)
    for i in range(X.shape[0]):
        Yi = run(qmm, fmt, Wq, N, K, X[i:i + 1], variant)
        assert np.array_equal(Yi[0].view(np.uint32), Yall[i].view(np.uint32)), i
