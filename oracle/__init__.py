"""The oracle: a plain fp64 CPU statement of the skinny Q4K x bf16 product.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  The product library never calls it, and it
shares no code with the library: ``q4k_oracle.c`` decodes the byte format from its written
definition.  The computation is the quantized matrix product that the pages' verify-pass
profile singles out ("sixi-asi 0.9", section "What I got wrong in 0.8").

Functions (all on host numpy arrays):
  pack(W)                   -> packed bytes, by the asymmetric min/max rule
  dequant(Wq, N, K)         -> fp32 weights, the single rounding of d*sc*q - dmin*m
  matmul(Wq, N, K, X, rows) -> (Y, S) in fp64: Y = sum_k w*x, S = sum_k |w*x|
  half_value, half_from_float, bf16_value: the number formats, from their definitions
  bf16_round(v)             -> bf16 bits of fp64 values, round to nearest even (definition)
  fmt_pack / fmt_dequant / fmt_matmul(fmt, ...): the same for the other weight formats of
                               formats_oracle.c (Q5K, Q6K, NVFP4, INT4 with one scale per 128 columns;
                               fmt 0 is Q4K and goes to the functions above)
  e4m3_value, e2m1_value, e4m3_from_float, e2m1_from_float: the 8- and 4-bit float formats
  swiglu(G, F)              -> silu(G[:, :F]) * G[:, F:] in fp64, the step between the gate/up
                               and down products of one feed-forward block (gate+up products
                               are what FlashRT issue #153 times; the SiLU gating between them is
                               the plainest reading: the pages do not print it)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4k_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "formats_oracle.c")]
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle's C files with gcc (OpenMP, no FMA contraction, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or any(os.path.getmtime(_LIB_PATH) < os.path.getmtime(f) for f in _SRCS):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp] + _SRCS + ["-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            lib.oracle_half_value.argtypes = [ctypes.c_uint16]
            lib.oracle_half_value.restype = ctypes.c_double
            lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_value.restype = ctypes.c_double
            lib.oracle_half_from_float.argtypes = [ctypes.c_float, ctypes.POINTER(ctypes.c_uint16)]
            lib.oracle_half_from_float.restype = i32
            lib.oracle_dequant.argtypes = [vp, i64, i64, vp]
            lib.oracle_dequant.restype = None
            lib.oracle_matmul.argtypes = [vp, i64, i64, vp, i32, vp, i64, vp, vp, i32]
            lib.oracle_matmul.restype = None
            lib.oracle_pack.argtypes = [vp, i64, i64, vp]
            lib.oracle_pack.restype = i32
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_value.restype = ctypes.c_double
            lib.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
            lib.oracle_e2m1_from_float.argtypes = [ctypes.c_float]
            lib.oracle_e2m1_from_float.restype = ctypes.c_uint8
            lib.oracle_fmt_packed_bytes.argtypes = [i32, i64, i64]
            lib.oracle_fmt_packed_bytes.restype = i64
            lib.oracle_fmt_dequant.argtypes = [i32, vp, i64, i64, vp, i64, vp]
            lib.oracle_fmt_dequant.restype = None
            lib.oracle_fmt_matmul.argtypes = [i32, vp, i64, i64, vp, i32, vp, i64, vp, vp, i32]
            lib.oracle_fmt_matmul.restype = None
            lib.oracle_fmt_pack.argtypes = [i32, vp, i64, i64, vp]
            lib.oracle_fmt_pack.restype = i32
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def packed_bytes(N: int, K: int) -> int:
    return N * (K // 256) * 144


def half_value(h: int) -> float:
    return _load().oracle_half_value(h)


def bf16_value(b: int) -> float:
    return _load().oracle_bf16_value(b)


def half_from_float(f: float):
    """(bits, overflow) of the round-to-nearest-even binary16 of a float32 value."""
    out = ctypes.c_uint16(0)
    rc = _load().oracle_half_from_float(ctypes.c_float(f), ctypes.byref(out))
    return out.value, bool(rc)


class OraclePackError(ValueError):
    pass


def pack(W: np.ndarray) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    if K % 256 != 0 or K == 0 or N == 0:
        raise ValueError("K must be a positive multiple of 256 and N >= 1")
    out = np.zeros(packed_bytes(N, K), dtype=np.uint8)
    rc = _load().oracle_pack(_ptr(W), N, K, _ptr(out))
    if rc != 0:
        raise OraclePackError(f"oracle_pack failed with status {rc} (non-finite weight or fp16 overflow)")
    return out


def dequant(Wq: np.ndarray, N: int, K: int) -> np.ndarray:
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    assert Wq.size == packed_bytes(N, K)
    out = np.empty((N, K), dtype=np.float32)
    _load().oracle_dequant(_ptr(Wq), N, K, _ptr(out))
    return out


def matmul(Wq: np.ndarray, N: int, K: int, X_bits: np.ndarray, rows=None, threads: int = 0):
    """Y, S (both float64, shape M x len(rows)) for weight rows `rows` (None: all N rows).

    X_bits is M x K uint16 (bf16 bit patterns)."""
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    assert Wq.size == packed_bytes(N, K)
    X_bits = np.ascontiguousarray(X_bits, dtype=np.uint16)
    if X_bits.ndim == 1:
        X_bits = X_bits[None, :]
    M = X_bits.shape[0]
    assert X_bits.shape[1] == K
    if rows is None:
        nrows, rp = N, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        assert rows.ndim == 1 and (rows.size == 0 or (rows.min() >= 0 and rows.max() < N))
        nrows, rp = rows.size, _ptr(rows)
    Y = np.empty((M, nrows), dtype=np.float64)
    S = np.empty((M, nrows), dtype=np.float64)
    if nrows:
        _load().oracle_matmul(_ptr(Wq), N, K, _ptr(X_bits), M, rp, nrows, _ptr(Y), _ptr(S), threads)
    return Y, S


def max_threads() -> int:
    return _load().oracle_max_threads()


def bf16_round(v) -> np.ndarray:
    """bf16 bit patterns (uint16) of fp64 values, rounded to nearest even: 8 significant bits,
    exponent range of fp32 (normal down to 2^-126, subnormal steps of 2^-133), overflow to
    infinity, signs kept (also on zero)."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                                     # v = m * 2^e, 0.5 <= |m| < 1
    e = np.where(v == 0, -1000, e)
    normal = e - 1 >= -126
    r = np.where(normal, np.ldexp(np.rint(m * 256.0), e - 8),       # 8 significant bits
                 np.ldexp(np.rint(np.ldexp(v, 133)), -133))          # subnormal grid 2^-133
    r = np.where(np.abs(r) > 3.3895313892515355e38, np.copysign(np.inf, v), r)   # past max bf16
    r = np.where(v == 0, v, r)
    bits32 = r.astype(np.float32).view(np.uint32)          # r has <= 8 significant bits: exact
    return (bits32 >> 16).astype(np.uint16)


def swiglu(G: np.ndarray, F: int) -> np.ndarray:
    """silu(G[:, f]) * G[:, F + f] for f < F, in fp64, silu(g) = g / (1 + e^-g)."""
    G = np.asarray(G, dtype=np.float64)
    assert G.shape[1] == 2 * F
    g, u = G[:, :F], G[:, F:]
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g)) * u


# ---- the other weight formats (formats_oracle.c) -------------------------------------------
FMT_Q4K, FMT_Q5K, FMT_NVFP4, FMT_INT4, FMT_Q6K = 0, 1, 2, 3, 4
FORMATS = {"q4k": FMT_Q4K, "q5k": FMT_Q5K, "nvfp4": FMT_NVFP4, "int4": FMT_INT4, "q6k": FMT_Q6K}


def e4m3_value(c: int) -> float:
    return _load().oracle_e4m3_value(c)


def e2m1_value(c: int) -> float:
    return _load().oracle_e2m1_value(c)


def e4m3_from_float(x: float) -> int:
    """E4M3 code of a non-negative value: nearest, ties to even, clamped to 448."""
    return _load().oracle_e4m3_from_float(ctypes.c_float(x))


def e2m1_from_float(x: float) -> int:
    """E2M1 code of a value: nearest magnitude, ties to even, clamped to 6, sign kept."""
    return _load().oracle_e2m1_from_float(ctypes.c_float(x))


def fmt_packed_bytes(fmt: int, N: int, K: int) -> int:
    if fmt == FMT_Q4K:
        return packed_bytes(N, K)
    return int(_load().oracle_fmt_packed_bytes(fmt, N, K))


def fmt_pack(fmt: int, W: np.ndarray) -> np.ndarray:
    if fmt == FMT_Q4K:
        return pack(W)
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    if K % 256 != 0 or K == 0 or N == 0:
        raise ValueError("K must be a positive multiple of 256 and N >= 1")
    out = np.zeros(fmt_packed_bytes(fmt, N, K), dtype=np.uint8)
    rc = _load().oracle_fmt_pack(fmt, _ptr(W), N, K, _ptr(out))
    if rc != 0:
        raise OraclePackError(f"oracle_fmt_pack failed with status {rc}")
    return out


def fmt_dequant(fmt: int, Wq: np.ndarray, N: int, K: int, rows=None) -> np.ndarray:
    """fp32 weights of rows `rows` (None: all N rows) of a packed matrix."""
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    assert Wq.size == fmt_packed_bytes(fmt, N, K)
    if fmt == FMT_Q4K:
        full = dequant(Wq, N, K)
        return full if rows is None else full[np.asarray(rows)]
    if rows is None:
        nrows, rp = N, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        nrows, rp = rows.size, _ptr(rows)
    out = np.empty((nrows, K), dtype=np.float32)
    if nrows:
        _load().oracle_fmt_dequant(fmt, _ptr(Wq), N, K, rp, nrows, _ptr(out))
    return out


def fmt_matmul(fmt: int, Wq: np.ndarray, N: int, K: int, X_bits: np.ndarray, rows=None, threads: int = 0):
    """Y, S (float64, M x len(rows)) of the product in format `fmt`, as matmul() for Q4K."""
    if fmt == FMT_Q4K:
        return matmul(Wq, N, K, X_bits, rows, threads)
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    assert Wq.size == fmt_packed_bytes(fmt, N, K)
    X_bits = np.ascontiguousarray(X_bits, dtype=np.uint16)
    if X_bits.ndim == 1:
        X_bits = X_bits[None, :]
    M = X_bits.shape[0]
    assert X_bits.shape[1] == K
    if rows is None:
        nrows, rp = N, None
    else:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        assert rows.ndim == 1 and (rows.size == 0 or (rows.min() >= 0 and rows.max() < N))
        nrows, rp = rows.size, _ptr(rows)
    Y = np.empty((M, nrows), dtype=np.float64)
    S = np.empty((M, nrows), dtype=np.float64)
    if nrows:
        _load().oracle_fmt_matmul(fmt, _ptr(Wq), N, K, _ptr(X_bits), M, rp, nrows, _ptr(Y), _ptr(S), threads)
    return Y, S
