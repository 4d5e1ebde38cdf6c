"""Pins of the oracle to things other than itself (CPU only).

* number formats against numpy's binary16 and torch's bf16 (library conversions);
* the byte layout against a hand-encoded super-block (tests/golden/q4k_handbuilt_block.txt)
  whose weights have a closed form;
* dequantization against exact rational arithmetic (Python integers / Fractions);
* the product against exact big-integer dot products, within the fp64 summation bound;
* closed forms (constant weights, one-hot activations), invariants (row independence, row
  permutation) and the packer's round trip on grid-exact weights.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from bit_quantized_skinny_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U53 = 2.0 ** -53


def gamma(n):
    return n * U53 / (1 - n * U53)


# ---------------------------------------------------------------- helpers (layout spec) ----

def make_block(d_bits, dmin_bits, sc, m, q):
    """Encode one super-block from its fields, following the written layout."""
    F = 0
    for j in range(8):
        F |= (sc[j] & 63) << (12 * j)
        F |= (m[j] & 63) << (12 * j + 6)
    Q = 0
    for t in range(256):
        Q |= (q[t] & 15) << (4 * t)
    return (d_bits.to_bytes(2, "little") + dmin_bits.to_bytes(2, "little")
            + F.to_bytes(12, "little") + Q.to_bytes(128, "little"))


def half_fraction(bits):
    v = np.array([bits], dtype=np.uint16).view(np.float16)[0]
    return Fraction(float(v))


def exact_weights(block):
    """Exact weights of a super-block (integer arithmetic), as (value, negative_zero) pairs.

    A zero weight is -0 exactly when d*sc*q is -0 and dmin*m is +0 (IEEE sign rule of a
    difference of zeros; a zero product takes the sign of d or dmin since sc, q, m >= 0)."""
    d_bits = int.from_bytes(block[0:2], "little")
    m_bits = int.from_bytes(block[2:4], "little")
    d, dmin = half_fraction(d_bits), half_fraction(m_bits)
    d_neg, dmin_neg = bool(d_bits >> 15), bool(m_bits >> 15)
    F = int.from_bytes(block[4:16], "little")
    Q = int.from_bytes(block[16:144], "little")
    out = []
    for t in range(256):
        j = t // 32
        sc = (F >> (12 * j)) & 63
        m = (F >> (12 * j + 6)) & 63
        q = (Q >> (4 * t)) & 15
        a, b = d * sc * q, dmin * m
        negzero = a == 0 and b == 0 and d_neg and not dmin_neg
        out.append((a - b, negzero))
    return out


def to_f32(item):
    """Round an exact rational with <= 53 significant bits to fp32 (one rounding)."""
    fr, negzero = item
    f = float(fr)
    assert Fraction(f) == fr, "value not exact in binary64"
    return np.float32(-0.0) if negzero else np.float32(f)


def read_golden_block():
    rows = []
    with open(os.path.join(GOLDEN, "q4k_handbuilt_block.txt")) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.extend(int(h, 16) for h in line.split())
    assert len(rows) == 144
    return bytes(rows)


# ---------------------------------------------------------------- number formats --------

def test_half_value_matches_numpy(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle_lib.half_value(int(p)) for p in pats])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(ref[~np.isnan(ref)]))


def test_bf16_value_matches_torch(oracle_lib):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([oracle_lib.bf16_value(int(p)) for p in pats])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_half_from_float_matches_numpy(oracle_lib):
    rng = np.random.default_rng(7)
    vals = [0.0, -0.0, 1.0, 65504.0, 65519.0, 65519.996, 2.0 ** -24, 2.0 ** -25,
            2.0 ** -25 * 1.0000001, 3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12)]
    # exact ties between neighbouring binary16 numbers (normal and subnormal)
    h = rng.integers(1, 0x7BFF, 2000, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    vals += list(((lo + hi) / 2).astype(np.float32))
    vals += list((rng.standard_normal(3000) * np.exp(rng.uniform(-20, 11, 3000))).astype(np.float32))
    for v in vals:
        v = np.float32(v)
        bits, ovf = oracle_lib.half_from_float(float(v))
        assert ovf == (abs(float(v)) >= 65520.0), v
        if ovf:
            continue
        ref = np.array([v], dtype=np.float32).astype(np.float16).view(np.uint16)[0]
        assert bits == ref, (v, hex(bits), hex(ref))
    for v in [65520.0, 70000.0, 1e30, -65520.0]:
        assert oracle_lib.half_from_float(v)[1]


# ---------------------------------------------------------------- dequantization --------

def test_golden_block_closed_form(oracle_lib):
    blk = read_golden_block()
    w = oracle_lib.dequant(np.frombuffer(blk, dtype=np.uint8), 1, 256)[0]
    expect = np.array([(t // 32 + 1) * (t % 16) - (t // 32) for t in range(256)], dtype=np.float32)
    assert np.array_equal(w, expect)
    # the independent encoder produces the same bytes as the hand-written file
    assert make_block(0x3C00, 0x3800, [j + 1 for j in range(8)], [2 * j for j in range(8)],
                      [t % 16 for t in range(256)]) == blk


EXTREME_BLOCKS = [
    # d, dmin, sc, m, q
    (0x3C00, 0x3C00, [63] * 8, [63] * 8, [15] * 256),
    (0x3C00, 0x3C00, [63] * 8, [63] * 8, [0] * 256),
    (0x7BFF, 0x7BFF, [63] * 8, [63] * 8, [15] * 256),            # largest d: rounding of 26-bit values
    (0x7BFF, 0x0001, [63, 1, 2, 3, 4, 5, 6, 7], [1] * 8, [(7 * t) % 16 for t in range(256)]),
    (0x0001, 0x0001, [63] * 8, [63] * 8, [(t * 5) % 16 for t in range(256)]),   # subnormal d, dmin
    (0x0000, 0x3555, [9] * 8, list(range(8)), [t % 16 for t in range(256)]),    # d = 0
    (0x8000, 0x0000, [5] * 8, [5] * 8, [3] * 256),                              # -0 scales
    (0xBC00, 0x3C00, [1, 2, 3, 4, 5, 6, 7, 8], [8, 7, 6, 5, 4, 3, 2, 1],        # negative d
     [(3 * t + 1) % 16 for t in range(256)]),
    (0x2E66, 0x2A3D, [17, 0, 63, 33, 1, 48, 2, 60], [0, 63, 12, 3, 41, 7, 63, 1],
     [(11 * t + t // 7) % 16 for t in range(256)]),
]


@pytest.mark.parametrize("case", range(len(EXTREME_BLOCKS)))
def test_dequant_extreme_blocks_exact(oracle_lib, case):
    d, dm, sc, m, q = EXTREME_BLOCKS[case]
    blk = make_block(d, dm, sc, m, q)
    got = oracle_lib.dequant(np.frombuffer(blk, dtype=np.uint8), 1, 256)[0]
    ref = np.array([to_f32(v) for v in exact_weights(blk)], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_dequant_tiny_config_bit_exact(oracle_lib):
    N, K = 256, 512
    W = inputs.weights_f32(N, K, inputs.seed_for(1))
    Wq = oracle_lib.pack(W)
    got = oracle_lib.dequant(Wq, N, K)
    raw = Wq.tobytes()
    for blk_index in range(N * K // 256):
        blk = raw[blk_index * 144:(blk_index + 1) * 144]
        ref = np.array([to_f32(v) for v in exact_weights(blk)], dtype=np.float32)
        n, b = divmod(blk_index, K // 256)
        assert np.array_equal(got[n, b * 256:(b + 1) * 256].view(np.uint32), ref.view(np.uint32))


# ---------------------------------------------------------------- the product ------------

def _exact_products(w_row, x_row):
    """Exact sum of w*x and of |w*x| as Fractions (big-integer arithmetic)."""
    wn = [Fraction(float(v)) for v in w_row]
    xn = [Fraction(float(v)) for v in x_row]
    y = sum(a * b for a, b in zip(wn, xn))
    s = sum(abs(a * b) for a, b in zip(wn, xn))
    return y, s


@pytest.mark.parametrize("M", [1, 4])
def test_matmul_tiny_config_vs_exact(oracle_lib, M):
    N, K = 256, 512
    W = inputs.weights_f32(N, K, inputs.seed_for(1))
    Wq = oracle_lib.pack(W)
    X = inputs.activations_bf16_bits(M, K, inputs.seed_for(1))
    Y, S = oracle_lib.matmul(Wq, N, K, X)
    w = oracle_lib.dequant(Wq, N, K)
    x = torch.from_numpy(X.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    rows = range(N) if M == 1 else range(0, N, 5)
    for i in range(M):
        for n in rows:
            y_ex, s_ex = _exact_products(w[n], x[i])
            assert abs(Fraction(Y[i, n]) - y_ex) <= Fraction(gamma(K)) * s_ex
            assert abs(Fraction(S[i, n]) - s_ex) <= Fraction(gamma(K)) * s_ex


def test_matmul_constant_block_closed_form(oracle_lib):
    # every weight equals w0 = d*sc*q - dmin*m = 0.25*3*5 - 0.125*7 = 2.875; with integer x the
    # fp64 sums are exact, so Y = w0 * sum_k x exactly.
    N, K = 3, 768
    blk = make_block(0x3400, 0x3000, [3] * 8, [7] * 8, [5] * 256)
    Wq = np.frombuffer(blk * (N * K // 256), dtype=np.uint8)
    rng = np.random.default_rng(3)
    xi = rng.integers(-20, 21, size=(2, K)).astype(np.float32)
    X = inputs.bf16_bits_from_f32(xi)
    Y, S = oracle_lib.matmul(Wq, N, K, X)
    for i in range(2):
        assert np.all(Y[i] == 2.875 * xi[i].sum())
        assert np.all(S[i] == 2.875 * np.abs(xi[i]).sum())
    ones = inputs.bf16_bits_from_f32(np.ones((1, K), np.float32))
    Y1, _ = oracle_lib.matmul(Wq, N, K, ones)
    assert np.all(Y1 == 2.875 * K)          # x = 1 gives the row sums


def test_matmul_one_hot_reproduces_dequant(oracle_lib):
    N, K = 64, 512
    Wq = oracle_lib.pack(inputs.weights_f32(N, K, 11))
    w = oracle_lib.dequant(Wq, N, K)
    ks = [0, 1, 31, 32, 255, 256, 300, 511]
    eye = np.zeros((len(ks), K), np.float32)
    for r, k in enumerate(ks):
        eye[r, k] = 1.0
    Y, _ = oracle_lib.matmul(Wq, N, K, inputs.bf16_bits_from_f32(eye))
    for r, k in enumerate(ks):
        assert np.array_equal(Y[r], w[:, k].astype(np.float64))


def test_matmul_row_independence_and_permutation(oracle_lib):
    N, K, M = 40, 1024, 5
    Wq = oracle_lib.pack(inputs.weights_f32(N, K, 21))
    X = inputs.activations_bf16_bits(M, K, 22)
    Y, S = oracle_lib.matmul(Wq, N, K, X)
    for i in range(M):
        Yi, Si = oracle_lib.matmul(Wq, N, K, X[i:i + 1])
        assert np.array_equal(Yi[0], Y[i]) and np.array_equal(Si[0], S[i])
    perm = np.random.default_rng(1).permutation(N)
    rowbytes = (K // 256) * 144
    Wp = Wq.reshape(N, rowbytes)[perm].reshape(-1)
    Yp, _ = oracle_lib.matmul(Wp, N, K, X)
    assert np.array_equal(Yp, Y[:, perm])
    Yr, _ = oracle_lib.matmul(Wq, N, K, X, rows=perm[:7])
    assert np.array_equal(Yr, Y[:, perm[:7]])


# ---------------------------------------------------------------- the packer -------------

def _grid_exact_block(rng):
    """Fields whose weights the min/max rule must recover exactly (see test docstring)."""
    d = 2.0 ** int(rng.integers(-10, -5)) * (1 + int(rng.integers(0, 8)) / 8)
    dmin = d * 2.0 ** int(rng.integers(-2, 2)) * (1 + int(rng.integers(0, 8)) / 8)
    sc = [int(v) for v in rng.integers(0, 64, 8)]
    m = [int(v) for v in rng.integers(0, 64, 8)]
    sc[int(rng.integers(0, 8))] = 63
    m[int(rng.integers(0, 8))] = 63
    q = [int(v) for v in rng.integers(0, 16, 256)]
    for j in range(8):
        if sc[j] == 0:
            q[32 * j:32 * j + 32] = [0] * 32
        else:
            pos = rng.permutation(32)[:2]
            q[32 * j + pos[0]] = 0
            q[32 * j + pos[1]] = 15
    d_bits = int(np.array([d], np.float16).view(np.uint16)[0])
    m_bits = int(np.array([dmin], np.float16).view(np.uint16)[0])
    return make_block(d_bits, m_bits, sc, m, q)


def test_pack_round_trips_grid_exact_blocks(oracle_lib):
    """For weights that lie on the grid of some block whose largest scale and min are 63 and
    whose sub-blocks each use q = 0 and q = 15, the min/max rule finds exactly that block:
    lo_j = -dmin*m_j, hi_j = d*sc_j*15 - dmin*m_j, so scale_j = d*sc_j, d = max scale / 63, and
    every division in the rule is exact."""
    rng = np.random.default_rng(5)
    for _ in range(200):
        blk = _grid_exact_block(rng)
        w = oracle_lib.dequant(np.frombuffer(blk, dtype=np.uint8), 1, 256)
        assert oracle_lib.pack(w).tobytes() == blk


def test_pack_constant_and_zero_weights(oracle_lib):
    W = np.full((2, 256), 0.037, np.float32)
    blk = oracle_lib.pack(W).tobytes()[:144]
    F = int.from_bytes(blk[4:16], "little")
    Q = int.from_bytes(blk[16:], "little")
    assert all(((F >> (12 * j + 6)) & 63) == 0 for j in range(8))          # m = 0
    assert all(((Q >> (4 * t)) & 15) == 15 for t in range(256))             # q = 15
    assert abs(oracle_lib.dequant(np.frombuffer(blk, np.uint8), 1, 256) - 0.037).max() < 0.037 / 63
    Wn = np.full((1, 256), -0.5, np.float32)
    wn = oracle_lib.dequant(oracle_lib.pack(Wn), 1, 256)
    assert np.abs(wn + 0.5).max() <= 0.5 / 63                               # only the min term
    assert not oracle_lib.pack(np.zeros((3, 512), np.float32)).any()


def test_pack_error_bounds(oracle_lib):
    N, K = 64, 1024
    W = inputs.weights_f32(N, K, 31)
    Wq = oracle_lib.pack(W)
    w = oracle_lib.dequant(Wq, N, K)
    raw = Wq.reshape(N, K // 256, 144)
    err = np.abs(w - W).reshape(N, K // 256, 8, 32)
    steps = []
    for n in range(N):
        for b in range(K // 256):
            blk = raw[n, b].tobytes()
            d = float(half_fraction(int.from_bytes(blk[0:2], "little")))
            dm = float(half_fraction(int.from_bytes(blk[2:4], "little")))
            F = int.from_bytes(blk[4:16], "little")
            for j in range(8):
                sc = (F >> (12 * j)) & 63
                step = d * sc
                steps.append(step)
                # half a step of rounding plus the slack of rounding sc and m to integers
                assert err[n, b, j].max() <= 0.5 * step + 0.5 * dm + 7.5 * d + 1e-7
    rms = float(np.sqrt(np.mean((w - W) ** 2)))
    expect = float(np.sqrt(np.mean(np.square(steps)) / 12))
    assert 0.8 * expect < rms < 1.25 * expect


def test_pack_rejects_nonfinite_and_overflow(oracle_lib):
    W = np.zeros((1, 256), np.float32)
    W[0, 7] = np.nan
    with pytest.raises(ValueError):
        oracle_lib.pack(W)
    W[0, 7] = np.inf
    with pytest.raises(ValueError):
        oracle_lib.pack(W)
    W = np.zeros((1, 256), np.float32)
    W[0, 0] = 1e8                       # scale / 63 above the largest binary16
    with pytest.raises(ValueError):
        oracle_lib.pack(W)


# ---------------------------------------------------------------- the pages' unit -------

def test_pages_bandwidth_unit():
    """The pages' GB/s figures are packed weight bytes / time at 0.5625 B per weight."""
    with open(os.path.join(GOLDEN, "pages_bandwidth.txt")) as fh:
        rows = [ln.split() for ln in fh if ln.strip() and not ln.startswith("#")]
    assert rows
    for kind, name, N, K, ms, printed, unit in rows:
        N, K, ms, printed = int(N), int(K), float(ms), float(printed)
        if kind == "floor":
            assert abs(printed * 1e9 / 273e9 * 1e3 - ms) < 0.5
            continue
        gbps = N * (K // 256) * 144 / (ms * 1e-3) / 1e9
        if kind == "gbps":
            assert abs(gbps - printed) <= 0.1, (name, gbps, printed)
        else:
            assert abs(100 * gbps / 273 - printed) <= 0.06, (name, gbps, printed)


# ------------------------------------------------------------------ feed-forward step --------

def test_bf16_round_matches_torch_on_fp32_values():
    """The oracle's bf16 rounding (from the format's definition) equals torch's fp32 -> bf16
    conversion (round to nearest even) on random, tie and edge values."""
    import torch
    rng = np.random.default_rng(5)
    f = np.concatenate([rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
                        (rng.standard_normal(2000) * 1e-38).astype(np.float32),   # subnormal range
                        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 1e-45, 65504.0], np.float32)])
    # exact ties: values with 9 significant bits whose last bit is 1
    ties = (np.arange(1, 512, 2, dtype=np.float32) + np.float32(256.0)) * np.float32(2.0 ** -8)
    f = np.concatenate([f, ties, -ties])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle_mod().bf16_round(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_swiglu_matches_torch_silu_in_fp64():
    import torch
    rng = np.random.default_rng(6)
    F = 64
    G = rng.standard_normal((3, 2 * F)) * 4.0
    G[0, :4] = [0.0, -40.0, 40.0, -800.0]
    ref = (torch.nn.functional.silu(torch.from_numpy(G[:, :F])) * torch.from_numpy(G[:, F:])).numpy()
    got = oracle_mod().swiglu(G, F)
    assert np.allclose(got, ref, rtol=1e-15, atol=0.0)
    assert got[0, 0] == 0.0 and abs(got[0, 3]) < 1e-300   # silu(0) = 0, silu(-800) underflows to 0


def oracle_mod():
    import oracle
    return oracle
