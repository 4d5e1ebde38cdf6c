"""Pins of the oracle of the other weight formats (Q5K, Q6K, NVFP4, INT4 with one scale per 128
columns) to things other than itself (CPU only).

* E4M3 values and rounding against torch's float8_e4m3fn (a library conversion); E2M1 values
  against the format's value table; E2M1 rounding against a brute-force nearest search;
* the byte layouts against blocks encoded here from the written layouts, whose weights have a
  closed form;
* dequantization against exact rational arithmetic on packed random weights;
* the product against exact big-integer sums within the fp64 summation bound, one-hot
  activations, row independence;
* the packers' rounding: every code is a nearest one (brute force) and the error bounds hold.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from bit_quantized_skinny_gb300 import inputs

U53 = 2.0 ** -53
# The E2M1 values of codes 0..7 (OCP microscaling formats: 1 sign, 2 exponent, 1 fraction bit).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def gamma(n):
    return n * U53 / (1 - n * U53)


def half_fraction(bits):
    return Fraction(float(np.array([bits], dtype=np.uint16).view(np.float16)[0]))


# ---------------------------------------------------------------- number formats --------

def test_e2m1_values_table(oracle_lib):
    for c in range(16):
        v = oracle_lib.e2m1_value(c)
        ref = E2M1_TABLE[c & 7]
        assert v == (-ref if c & 8 else ref)
        assert np.signbit(v) == bool(c & 8)


def test_e4m3_values_match_torch(oracle_lib):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().double().numpy()
    for c in range(256):
        v = oracle_lib.e4m3_value(c)
        if np.isnan(ref[c]):
            assert np.isnan(v), c
        else:
            assert v == ref[c] and np.signbit(v) == np.signbit(ref[c]), c
    assert oracle_lib.e4m3_value(0x7E) == 448.0 and oracle_lib.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_rounding_matches_torch(oracle_lib):
    rng = np.random.default_rng(5)
    vals = list(np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 3000)).astype(np.float32))
    # every midpoint between neighbouring codes (ties go to the even code) and its neighbours
    for c in range(126):
        lo, hi = oracle_lib.e4m3_value(c), oracle_lib.e4m3_value(c + 1)
        mid = np.float32((lo + hi) / 2)
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(1e9))]
    vals += [np.float32(0.0), np.float32(448.0)]
    t = torch.tensor(np.array(vals, dtype=np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, ref in zip(vals, t):
        assert oracle_lib.e4m3_from_float(float(v)) == int(ref), v
    assert oracle_lib.e4m3_from_float(1e6) == 0x7E      # clamped to 448


def _e2m1_brute(x):
    a = abs(float(x))
    best = min(range(8), key=lambda c: (abs(a - E2M1_TABLE[c]), c % 2))   # nearest, then even
    return best | (8 if np.signbit(x) else 0)


def test_e2m1_rounding_brute_force(oracle_lib):
    rng = np.random.default_rng(6)
    vals = list(rng.uniform(-8, 8, 4000).astype(np.float32))
    vals += [np.float32(v) for v in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.0, 7.0, 100.0, -0.0, 0.0)]
    for v in vals:
        assert oracle_lib.e2m1_from_float(float(v)) == _e2m1_brute(v), v
    # the ties by hand: 0.25 -> 0, 0.75 -> 1.0, 1.25 -> 1.0, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4
    assert [oracle_lib.e2m1_from_float(v) for v in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)] == [0, 2, 2, 4, 4, 6, 6]


def test_packed_bytes(oracle_lib):
    assert oracle_lib.fmt_packed_bytes(oracle_lib.FMT_Q5K, 3, 512) == 3 * 2 * 176
    assert oracle_lib.fmt_packed_bytes(oracle_lib.FMT_NVFP4, 3, 512) == 3 * 2 * 144 + 16
    assert oracle_lib.fmt_packed_bytes(oracle_lib.FMT_INT4, 3, 512) == 3 * 256 + 3 * 4 * 2
    assert oracle_lib.fmt_packed_bytes(oracle_lib.FMT_Q6K, 3, 512) == 3 * 2 * 208 + 3 * 2 * 2


# ---------------------------------------------------------------- layouts by hand ---------

def q5k_block(d_bits, dmin_bits, sc, m, q):
    """One Q5K super-block from its fields, following the written layout."""
    F = 0
    for j in range(8):
        F |= (sc[j] & 63) << (12 * j) | (m[j] & 63) << (12 * j + 6)
    H = [0] * 8
    L = 0
    for t in range(256):
        j, c, i = t // 32, (t % 32) // 8, t % 8
        H[j] |= ((q[t] >> 4) & 1) << (4 * i + c)
        L |= (q[t] & 15) << (4 * t)
    return (d_bits.to_bytes(2, "little") + dmin_bits.to_bytes(2, "little") + F.to_bytes(12, "little")
            + b"".join(h.to_bytes(4, "little") for h in H) + L.to_bytes(128, "little"))


def q5k_exact(block):
    d, dmin = half_fraction(int.from_bytes(block[0:2], "little")), half_fraction(int.from_bytes(block[2:4], "little"))
    F = int.from_bytes(block[4:16], "little")
    H = [int.from_bytes(block[16 + 4 * j:20 + 4 * j], "little") for j in range(8)]
    L = int.from_bytes(block[48:176], "little")
    out = []
    for t in range(256):
        j, c, i = t // 32, (t % 32) // 8, t % 8
        q = ((L >> (4 * t)) & 15) + 16 * ((H[j] >> (4 * i + c)) & 1)
        out.append(d * ((F >> (12 * j)) & 63) * q - dmin * ((F >> (12 * j + 6)) & 63))
    return out


def test_q5k_handbuilt_block_closed_form(oracle_lib):
    # d = 1, dmin = 0.5, sc_j = j + 1, m_j = 2j, q_t = t mod 32: w_t = (j + 1)(t mod 32) - j
    blk = q5k_block(0x3C00, 0x3800, [j + 1 for j in range(8)], [2 * j for j in range(8)],
                    [t % 32 for t in range(256)])
    got = oracle_lib.fmt_dequant(oracle_lib.FMT_Q5K, np.frombuffer(blk, np.uint8), 1, 256)[0]
    ref = np.array([(t // 32 + 1) * (t % 32) - t // 32 for t in range(256)], np.float32)
    assert np.array_equal(got, ref)


def test_q5k_high_bit_positions(oracle_lib):
    # one high bit at a time: weight t = 32j + 8c + i reads bit 4i + c of word j
    for t in (0, 1, 7, 8, 9, 31, 32, 77, 200, 255):
        q = [0] * 256
        q[t] = 16
        blk = q5k_block(0x3C00, 0x0000, [1] * 8, [0] * 8, q)
        got = oracle_lib.fmt_dequant(oracle_lib.FMT_Q5K, np.frombuffer(blk, np.uint8), 1, 256)[0]
        ref = np.zeros(256, np.float32)
        ref[t] = 16.0
        assert np.array_equal(got, ref), t


def q6k_matrix(u, q, d_bits):
    """A 1 x 256 Q6K matrix (one block and its d) from its fields, following the written layout."""
    L = 0
    H = [0] * 16
    for t in range(256):
        m, a, i = t // 16, (t % 16) // 8, t % 8
        L |= (q[t] & 15) << (4 * t)
        H[m] |= ((q[t] >> 4) & 3) << (8 * a + 16 * (i >= 4) + 2 * (i % 4))
    return bytes(u) + L.to_bytes(128, "little") + b"".join(h.to_bytes(4, "little") for h in H) + \
        d_bits.to_bytes(2, "little")


def test_q6k_handbuilt_block_closed_form(oracle_lib):
    # d = 0.5, u_j = 64 + j + 1 (sc_j = j + 1), q_t = t mod 64: w_t = 0.5 (j + 1)((t mod 64) - 32)
    blk = q6k_matrix([65 + j for j in range(16)], [t % 64 for t in range(256)], 0x3800)
    got = oracle_lib.fmt_dequant(oracle_lib.FMT_Q6K, np.frombuffer(blk, np.uint8), 1, 256)[0]
    ref = np.array([0.5 * (t // 16 + 1) * ((t % 64) - 32) for t in range(256)], np.float32)
    assert np.array_equal(got, ref)


def test_q6k_fields(oracle_lib):
    # one weight at a time with both high bits set (q = 48: w = d sc 16); bit 7 of a scale byte
    # is not used; u = 0 is sc = -64, u = 63 is sc = -1
    for t in (0, 3, 4, 7, 8, 11, 12, 15, 16, 100, 255):
        for qt, wt in ((48, 16.0), (16, -16.0), (31, -1.0)):   # high part 3, 1 and 1 with low 15
            q = [32] * 256
            q[t] = qt
            blk = q6k_matrix([65] * 16, q, 0x3C00)
            got = oracle_lib.fmt_dequant(oracle_lib.FMT_Q6K, np.frombuffer(blk, np.uint8), 1, 256)[0]
            ref = np.zeros(256, np.float32)
            ref[t] = wt
            assert np.array_equal(got, ref), (t, qt)
    q = [63] * 256
    for u, sc in ((0, -64), (63, -1), (64 + 128, 0), (127 + 128, 63), (5 + 128, -59)):
        blk = q6k_matrix([u] * 16, q, 0x3C00)
        got = oracle_lib.fmt_dequant(oracle_lib.FMT_Q6K, np.frombuffer(blk, np.uint8), 1, 256)[0]
        assert np.all(got == np.float32(sc * 31)), u


def nvfp4_matrix(scales, codes, g):
    """A 1 x 256 NVFP4 matrix (one block and the trailer) from its fields."""
    Q = 0
    for t in range(256):
        Q |= (codes[t] & 15) << (4 * t)
    return bytes(scales) + Q.to_bytes(128, "little") + np.float32(g).tobytes() + bytes(12)


def test_nvfp4_handbuilt_block_closed_form(oracle_lib):
    # s_b has exponent field b (value 2^(b-7), s_0 = 0), code t mod 16, g = 0.5:
    # w_t = 0.5 * 2^(b-7) * E2M1[t mod 16] with b = t div 16
    scales = [b << 3 for b in range(16)]
    blk = nvfp4_matrix(scales, [t % 16 for t in range(256)], 0.5)
    got = oracle_lib.fmt_dequant(oracle_lib.FMT_NVFP4, np.frombuffer(blk, np.uint8), 1, 256)[0]
    ref = []
    for t in range(256):
        b, c = t // 16, t % 16
        s = 0.0 if b == 0 else 2.0 ** (b - 7)
        v = E2M1_TABLE[c & 7] * (-1 if c & 8 else 1)
        ref.append(0.5 * s * v)
    assert np.array_equal(got, np.array(ref, np.float32))


def int4_matrix(N, K, q, scale_bits):
    """An INT4 matrix from signed quants q[N][K] and binary16 scale bits [N][K/128]."""
    plane = bytearray(N * K // 2)
    for n in range(N):
        for k in range(K):
            plane[n * K // 2 + k // 2] |= (q[n][k] & 15) << (4 * (k % 2))
    sc = b"".join(int(s).to_bytes(2, "little") for row in scale_bits for s in row)
    return bytes(plane) + sc


def test_int4_handbuilt_closed_form(oracle_lib):
    # q = (k mod 16) - 8, scale of group g of row n = 2^(g - n) (binary16 exponent field 15+g-n)
    N, K = 2, 512
    q = [[(k % 16) - 8 for k in range(K)] for _ in range(N)]
    sb = [[(15 + g - n) << 10 for g in range(K // 128)] for n in range(N)]
    Wq = np.frombuffer(int4_matrix(N, K, q, sb), np.uint8)
    got = oracle_lib.fmt_dequant(oracle_lib.FMT_INT4, Wq, N, K)
    ref = np.array([[2.0 ** (k // 128 - n) * ((k % 16) - 8) for k in range(K)] for n in range(N)], np.float32)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- exact dequantization ----

def _exact_rows(fmt, raw, N, K, oracle_lib):
    """Exact weights of every row, decoded here from the written layouts (Fractions)."""
    nb = K // 256
    rows = []
    for n in range(N):
        row = []
        if fmt == oracle_lib.FMT_Q5K:
            for b in range(nb):
                row += q5k_exact(raw[(n * nb + b) * 176:(n * nb + b + 1) * 176])
        elif fmt == oracle_lib.FMT_NVFP4:
            g = Fraction(float(np.frombuffer(raw[N * nb * 144:N * nb * 144 + 4], np.float32)[0]))
            for b in range(nb):
                blk = raw[(n * nb + b) * 144:(n * nb + b + 1) * 144]
                Q = int.from_bytes(blk[16:], "little")
                for t in range(256):
                    s = Fraction(float(oracle_lib.e4m3_value(blk[t // 16])))
                    c = (Q >> (4 * t)) & 15
                    v = Fraction(E2M1_TABLE[c & 7]) * (-1 if c & 8 else 1)
                    row.append(g * s * v)
        elif fmt == oracle_lib.FMT_Q6K:
            for b in range(nb):
                blk = raw[(n * nb + b) * 208:(n * nb + b + 1) * 208]
                do = N * nb * 208 + (n * nb + b) * 2
                d = half_fraction(int.from_bytes(raw[do:do + 2], "little"))
                L = int.from_bytes(blk[16:144], "little")
                H = [int.from_bytes(blk[144 + 4 * m:148 + 4 * m], "little") for m in range(16)]
                for t in range(256):
                    m, a, i = t // 16, (t % 16) // 8, t % 8
                    q = ((L >> (4 * t)) & 15) + 16 * ((H[m] >> (8 * a + 16 * (i >= 4) + 2 * (i % 4))) & 3)
                    row.append(d * ((blk[t // 16] & 127) - 64) * (q - 32))
        else:
            plane = int.from_bytes(raw[n * K // 2:(n + 1) * K // 2], "little")
            so = N * K // 2 + n * (K // 128) * 2
            for k in range(K):
                u = (plane >> (4 * k)) & 15
                s = half_fraction(int.from_bytes(raw[so + 2 * (k // 128):so + 2 * (k // 128) + 2], "little"))
                row.append(s * (u - 16 if u >= 8 else u))
        rows.append(row)
    return rows


@pytest.mark.parametrize("fmt_name", ["q5k", "q6k", "nvfp4", "int4"])
def test_dequant_bit_exact_vs_rationals(oracle_lib, fmt_name):
    fmt = oracle_lib.FORMATS[fmt_name]
    N, K = 6, 512
    W = inputs.weights_f32(N, K, 77)
    Wq = oracle_lib.fmt_pack(fmt, W)
    got = oracle_lib.fmt_dequant(fmt, Wq, N, K)
    exact = _exact_rows(fmt, Wq.tobytes(), N, K, oracle_lib)
    for n in range(N):
        for k in range(K):
            f = float(exact[n][k])
            assert Fraction(f) == exact[n][k]           # the exact value fits binary64
            assert got[n, k] == np.float32(f), (n, k)   # and the oracle rounds it once


# ---------------------------------------------------------------- the product ------------

@pytest.mark.parametrize("fmt_name", ["q5k", "q6k", "nvfp4", "int4"])
def test_matmul_vs_exact_and_one_hot(oracle_lib, fmt_name):
    fmt = oracle_lib.FORMATS[fmt_name]
    N, K, M = 8, 768, 3
    Wq = oracle_lib.fmt_pack(fmt, inputs.weights_f32(N, K, 13))
    X = inputs.activations_bf16_bits(M, K, 14)
    Y, S = oracle_lib.fmt_matmul(fmt, Wq, N, K, X)
    w = oracle_lib.fmt_dequant(fmt, Wq, N, K)
    x = torch.from_numpy(X.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for i in range(M):
        for n in range(N):
            wn = [Fraction(float(v)) for v in w[n]]
            xn = [Fraction(float(v)) for v in x[i]]
            y = sum(a * b for a, b in zip(wn, xn))
            s = sum(abs(a * b) for a, b in zip(wn, xn))
            assert abs(Fraction(Y[i, n]) - y) <= Fraction(gamma(K)) * s
            assert abs(Fraction(S[i, n]) - s) <= Fraction(gamma(K)) * s
    ks = [0, 15, 16, 127, 128, 255, 256, 767]
    eye = np.zeros((len(ks), K), np.float32)
    for r, k in enumerate(ks):
        eye[r, k] = 1.0
    Y1, _ = oracle_lib.fmt_matmul(fmt, Wq, N, K, inputs.bf16_bits_from_f32(eye))
    for r, k in enumerate(ks):
        assert np.array_equal(Y1[r], w[:, k].astype(np.float64))
    # each activation row alone gives the same result, and selected rows equal the full product
    for i in range(M):
        Yi, _ = oracle_lib.fmt_matmul(fmt, Wq, N, K, X[i:i + 1])
        assert np.array_equal(Yi[0], Y[i])
    Yr, _ = oracle_lib.fmt_matmul(fmt, Wq, N, K, X, rows=[5, 0, 7])
    assert np.array_equal(Yr, Y[:, [5, 0, 7]])


# ---------------------------------------------------------------- packers ----------------

def test_q5k_pack_bounds(oracle_lib):
    N, K = 16, 1024
    W = inputs.weights_f32(N, K, 21)
    Wq = oracle_lib.fmt_pack(oracle_lib.FMT_Q5K, W)
    w = oracle_lib.fmt_dequant(oracle_lib.FMT_Q5K, Wq, N, K)
    raw = Wq.tobytes()
    for n in range(N):
        for b in range(K // 256):
            blk = raw[(n * (K // 256) + b) * 176:][:176]
            d = float(half_fraction(int.from_bytes(blk[0:2], "little")))
            F = int.from_bytes(blk[4:16], "little")
            for j in range(8):
                step = d * ((F >> (12 * j)) & 63)
                seg = slice(b * 256 + 32 * j, b * 256 + 32 * j + 32)
                # within half a step, plus the slack of the 6-bit step and offset
                err = np.abs(W[n, seg].astype(np.float64) - w[n, seg])
                assert err.max() <= 0.5 * step + 0.04 * (W[n, seg].max() - min(0, W[n, seg].min())) + 1e-9
    rms = float(np.sqrt(np.mean((w.astype(np.float64) - W) ** 2)))
    assert rms < 1.0e-3   # about half the Q4K error (31 levels instead of 15)


def test_nvfp4_pack_is_nearest(oracle_lib):
    N, K = 4, 512
    W = inputs.weights_f32(N, K, 22)
    Wq = oracle_lib.fmt_pack(oracle_lib.FMT_NVFP4, W).tobytes()
    nb = K // 256
    g = float(np.frombuffer(Wq[N * nb * 144:][:4], np.float32)[0])
    assert g == float(np.float32(np.abs(W).max()) / np.float32(2688.0))
    for n in range(N):
        for b in range(nb):
            blk = Wq[(n * nb + b) * 144:][:144]
            Q = int.from_bytes(blk[16:], "little")
            for sb in range(16):
                seg = W[n, b * 256 + 16 * sb:b * 256 + 16 * sb + 16]
                a = np.float32(np.abs(seg).max())
                s = blk[sb]
                assert s == oracle_lib.e4m3_from_float(float(np.float32(a / np.float32(6.0)) / np.float32(g)))
                S = np.float32(oracle_lib.e4m3_value(s)) * np.float32(g)
                for t in range(16):
                    c = (Q >> (4 * (16 * sb + t))) & 15
                    assert c == (_e2m1_brute(seg[t] / S) if S > 0 else 0)


def test_int4_pack_bounds_and_scales(oracle_lib):
    N, K = 8, 1024
    W = inputs.weights_f32(N, K, 23)
    Wq = oracle_lib.fmt_pack(oracle_lib.FMT_INT4, W)
    w = oracle_lib.fmt_dequant(oracle_lib.FMT_INT4, Wq, N, K)
    sc = Wq[N * K // 2:].view(np.float16).reshape(N, K // 128).astype(np.float64)
    amax = np.abs(W.reshape(N, K // 128, 128)).max(axis=2)
    assert np.array_equal(sc.astype(np.float16), (amax / np.float32(7.0)).astype(np.float32).astype(np.float16))
    err = np.abs(W.astype(np.float64) - w).reshape(N, K // 128, 128)
    assert np.all(err <= 0.5 * sc[:, :, None] + 0.5 * np.abs(amax - 7 * sc)[:, :, None] + 1e-12)


def test_q6k_pack_bounds(oracle_lib):
    N, K = 8, 1024
    W = inputs.weights_f32(N, K, 24)
    Wq = oracle_lib.fmt_pack(oracle_lib.FMT_Q6K, W)
    w = oracle_lib.fmt_dequant(oracle_lib.FMT_Q6K, Wq, N, K)
    raw = Wq.tobytes()
    nb = K // 256
    for n in range(N):
        for b in range(nb):
            blk = raw[(n * nb + b) * 208:][:208]
            do = N * nb * 208 + (n * nb + b) * 2
            d = float(half_fraction(int.from_bytes(raw[do:do + 2], "little")))
            for j in range(16):
                sc = (blk[j] & 127) - 64
                seg = slice(b * 256 + 16 * j, b * 256 + 16 * j + 16)
                a = np.abs(W[n, seg]).max()
                # within half a step, plus the slack of the 6-bit sub-block scale
                err = np.abs(W[n, seg].astype(np.float64) - w[n, seg])
                assert 0 <= sc <= 63
                assert err.max() <= 0.5 * d * sc + 0.04 * a + 1e-12
    rms = float(np.sqrt(np.mean((w.astype(np.float64) - W) ** 2)))
    assert rms < 5e-4


def test_packers_reject_nonfinite(oracle_lib):
    W = np.zeros((2, 256), np.float32)
    W[1, 3] = np.inf
    for fmt in (oracle_lib.FMT_Q5K, oracle_lib.FMT_Q6K, oracle_lib.FMT_NVFP4, oracle_lib.FMT_INT4):
        with pytest.raises(oracle_lib.OraclePackError):
            oracle_lib.fmt_pack(fmt, W)
    Z = np.zeros((2, 256), np.float32)
    for fmt in (oracle_lib.FMT_Q5K, oracle_lib.FMT_Q6K, oracle_lib.FMT_NVFP4, oracle_lib.FMT_INT4):
        assert np.all(oracle_lib.fmt_dequant(fmt, oracle_lib.fmt_pack(fmt, Z), 2, 256) == 0)
