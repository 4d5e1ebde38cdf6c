"""ctypes binding of libqmm.so (include/qmm.h): argument marshalling only.

Every step of the product runs in the library's CUDA kernels; this module passes device
pointers (``tensor.data_ptr()``), sizes and the caller's current CUDA stream.  There is no
fallback: if the library is missing or cannot load, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmm.so")

QMM_QK = 256
QMM_BLOCK_BYTES = 144
QMM_MAX_M = 32
QMM_MAX_BATCH = 512

VARIANT_AUTO, VARIANT_FMA, VARIANT_TC = 0, 1, 2
VARIANT_NAMES = {VARIANT_FMA: "fma", VARIANT_TC: "tc"}

STATUS = {0: "QMM_OK", 1: "QMM_ERR_NULL", 2: "QMM_ERR_SHAPE", 3: "QMM_ERR_M_RANGE",
          4: "QMM_ERR_ALIGN", 5: "QMM_ERR_BUFSIZE", 6: "QMM_ERR_NONFINITE", 7: "QMM_ERR_CUDA",
          8: "QMM_ERR_COUNT", 9: "QMM_ERR_VARIANT", 10: "QMM_ERR_SCRATCH", 11: "QMM_ERR_FORMAT"}

FMT_Q4K, FMT_Q5K, FMT_NVFP4, FMT_INT4, FMT_Q6K = 0, 1, 2, 3, 4
FORMATS = {"q4k": FMT_Q4K, "q5k": FMT_Q5K, "q6k": FMT_Q6K, "nvfp4": FMT_NVFP4, "int4": FMT_INT4}

# Every symbol include/qmm.h declares.
EXPORTS = ["qmm_packed_bytes", "qmm_pack", "qmm_run", "qmm_run_batched", "qmm_dequant",
           "qmm_run_variant", "qmm_select_variant", "qmm_device_status", "qmm_strerror",
           "qmm_last_cuda_error", "qmm_run_noalloc", "qmm_select_variant_batched",
           "qmm_ffn_workspace_bytes", "qmm_run_ffn", "qmm_indexed_workspace_bytes", "qmm_run_indexed",
           "qmm_fmt_packed_bytes", "qmm_fmt_pack", "qmm_fmt_run", "qmm_fmt_dequant", "qmm_fmt_run_batched",
           "qmm_ffn_fused_workspace_bytes", "qmm_run_ffn_fused", "qmm_release", "qmm_workspace_bytes_held",
           "qmm_stream_read", "qmm_stream_read_sink_words", "qmm_set_wait_limit", "qmm_pack_dev"]
NOALLOC_SCRATCH_BYTES = 4 << 20


class QmmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        lib = _lib
        text = lib.qmm_strerror(status).decode() if lib is not None else STATUS.get(status, "?")
        if status == 7 and lib is not None:
            text += ": " + lib.qmm_last_cuda_error().decode()
        super().__init__(f"{what}: {STATUS.get(status, status)} ({text})")


class _Entry(ctypes.Structure):
    _fields_ = [("Wq", ctypes.c_void_p), ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class _FmtEntry(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("Wq", ctypes.c_void_p), ("X", ctypes.c_void_p), ("Y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


_lib = None


def load(path: str | None = None):
    """Load libqmm.so (raises if it is missing: build it with build_lib.build())."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libqmm.so not found at {p}: run bit_quantized_skinny_gb300.build_lib.build()")
    lib = ctypes.CDLL(p)
    vp, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint
    lib.qmm_packed_bytes.argtypes = [i64, i64]
    lib.qmm_packed_bytes.restype = ctypes.c_size_t
    lib.qmm_pack.argtypes = [vp, i64, i64, vp, ctypes.c_size_t, i32]
    lib.qmm_pack.restype = i32
    lib.qmm_pack_dev.argtypes = [vp, i64, i64, vp, ctypes.c_size_t, vp]
    lib.qmm_pack_dev.restype = i32
    lib.qmm_run.argtypes = [vp, i64, i64, vp, vp, i32, vp]
    lib.qmm_run.restype = i32
    lib.qmm_run_variant.argtypes = [vp, i64, i64, vp, vp, i32, i32, vp]
    lib.qmm_run_variant.restype = i32
    lib.qmm_run_noalloc.argtypes = [vp, i64, i64, vp, vp, i32, vp]
    lib.qmm_run_noalloc.restype = i32
    lib.qmm_stream_read.argtypes = [vp, ctypes.c_size_t, vp, vp]
    lib.qmm_stream_read.restype = i32
    lib.qmm_stream_read_sink_words.argtypes = []
    lib.qmm_stream_read_sink_words.restype = ctypes.c_size_t
    lib.qmm_set_wait_limit.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
    lib.qmm_set_wait_limit.restype = None
    lib.qmm_release.argtypes = []
    lib.qmm_release.restype = i32
    lib.qmm_workspace_bytes_held.argtypes = []
    lib.qmm_workspace_bytes_held.restype = ctypes.c_size_t
    lib.qmm_run_batched.argtypes = [ctypes.POINTER(_Entry), i32, i32, vp]
    lib.qmm_run_batched.restype = i32
    lib.qmm_dequant.argtypes = [vp, i64, i64, vp, vp]
    lib.qmm_dequant.restype = i32
    lib.qmm_select_variant.argtypes = [i32, i64, i64]
    lib.qmm_select_variant.restype = i32
    lib.qmm_select_variant_batched.argtypes = [ctypes.POINTER(_Entry), i32, i32]
    lib.qmm_select_variant_batched.restype = i32
    lib.qmm_ffn_workspace_bytes.argtypes = [i32, i64]
    lib.qmm_ffn_workspace_bytes.restype = ctypes.c_size_t
    lib.qmm_run_ffn.argtypes = [vp, vp, i64, i64, vp, vp, i32, vp, ctypes.c_size_t, vp]
    lib.qmm_run_ffn.restype = i32
    lib.qmm_ffn_fused_workspace_bytes.argtypes = [i32, i64]
    lib.qmm_ffn_fused_workspace_bytes.restype = ctypes.c_size_t
    lib.qmm_run_ffn_fused.argtypes = [vp, vp, i64, i64, vp, vp, i32, vp, ctypes.c_size_t, vp]
    lib.qmm_run_ffn_fused.restype = i32
    lib.qmm_indexed_workspace_bytes.argtypes = [i32, i64, i64]
    lib.qmm_indexed_workspace_bytes.restype = ctypes.c_size_t
    lib.qmm_run_indexed.argtypes = [ctypes.POINTER(vp), i32, i64, i64, ctypes.POINTER(ctypes.c_int32), vp, vp, i32,
                                    vp, ctypes.c_size_t, vp]
    lib.qmm_run_indexed.restype = i32
    lib.qmm_fmt_packed_bytes.argtypes = [i32, i64, i64]
    lib.qmm_fmt_packed_bytes.restype = ctypes.c_size_t
    lib.qmm_fmt_pack.argtypes = [i32, vp, i64, i64, vp, ctypes.c_size_t, i32]
    lib.qmm_fmt_pack.restype = i32
    lib.qmm_fmt_run.argtypes = [i32, vp, i64, i64, vp, vp, i32, vp]
    lib.qmm_fmt_run.restype = i32
    lib.qmm_fmt_run_batched.argtypes = [ctypes.POINTER(_FmtEntry), i32, i32, vp]
    lib.qmm_fmt_run_batched.restype = i32
    lib.qmm_fmt_dequant.argtypes = [i32, vp, i64, i64, vp, vp]
    lib.qmm_fmt_dequant.restype = i32
    lib.qmm_device_status.argtypes = [ctypes.POINTER(u32)]
    lib.qmm_device_status.restype = i32
    lib.qmm_strerror.argtypes = [i32]
    lib.qmm_strerror.restype = ctypes.c_char_p
    lib.qmm_last_cuda_error.argtypes = []
    lib.qmm_last_cuda_error.restype = ctypes.c_char_p
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        raise QmmError(status, what)


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def packed_bytes(N: int, K: int) -> int:
    return load().qmm_packed_bytes(N, K)


def pack(W: np.ndarray, threads: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """Pack an N x K fp32 host array into Q4K bytes (host, multi-threaded)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    nbytes = packed_bytes(N, K)
    if nbytes == 0:
        raise QmmError(2, "qmm_pack")
    if out is None:
        out = np.empty(nbytes, dtype=np.uint8)
    _check(load().qmm_pack(W.ctypes.data_as(ctypes.c_void_p), N, K, out.ctypes.data_as(ctypes.c_void_p),
                           out.nbytes, threads), "qmm_pack")
    return out


def pack_dev(W, out=None, stream=None):
    """qmm_pack_dev: pack an N x K fp32 CUDA tensor into Q4K bytes on the GPU (a uint8 CUDA
    tensor of packed_bytes(N, K) bytes, allocated when `out` is None), asynchronous on `stream`
    (default: torch's current stream).  Non-finite super-blocks come out as zeros and set bit 1
    of device_status()."""
    import torch
    N, K = W.shape
    nbytes = packed_bytes(N, K)
    if nbytes == 0:
        raise QmmError(2, "qmm_pack_dev")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    _check(load().qmm_pack_dev(ctypes.c_void_p(W.data_ptr()), N, K, ctypes.c_void_p(out.data_ptr()),
                               out.numel() * out.element_size(), _stream_handle(stream)), "qmm_pack_dev")
    return out


def run(Wq, N: int, K: int, X, Y, M: int | None = None, variant: int = VARIANT_AUTO, stream=None):
    """Y[M x N] = X[M x K] * dequant(Wq)^T on the GPU (torch CUDA tensors: uint8/any Wq,
    bf16 or int16 X, fp32 Y).  Asynchronous on `stream` (default: torch's current stream)."""
    if M is None:
        M = X.shape[0]
    st = load().qmm_run_variant(ctypes.c_void_p(Wq.data_ptr()), N, K, ctypes.c_void_p(X.data_ptr()),
                                ctypes.c_void_p(Y.data_ptr()), M, variant, _stream_handle(stream))
    _check(st, "qmm_run")


def run_noalloc(Wq, N: int, K: int, X, Y, M: int | None = None, stream=None):
    """qmm_run_noalloc: the tensor-core product without any device allocation (fixed 4 MiB
    library buffer for the prepared activations; see include/qmm.h for its limits)."""
    if M is None:
        M = X.shape[0]
    st = load().qmm_run_noalloc(ctypes.c_void_p(Wq.data_ptr()), N, K, ctypes.c_void_p(X.data_ptr()),
                                ctypes.c_void_p(Y.data_ptr()), M, _stream_handle(stream))
    _check(st, "qmm_run_noalloc")


def run_raw(wq_ptr: int, N: int, K: int, x_ptr: int, y_ptr: int, M: int, variant: int = VARIANT_AUTO,
            stream_handle: int = 0) -> int:
    """Unchecked call on raw device pointers; returns the status code."""
    return load().qmm_run_variant(ctypes.c_void_p(wq_ptr), N, K, ctypes.c_void_p(x_ptr),
                                  ctypes.c_void_p(y_ptr), M, variant, ctypes.c_void_p(stream_handle))


def make_entries(items):
    """items: sequence of (Wq, X, Y, N, K) with torch tensors or raw int pointers."""
    arr = (_Entry * len(items))()
    for k, (Wq, X, Y, N, K) in enumerate(items):
        ptr = lambda t: t if isinstance(t, int) else t.data_ptr()
        arr[k] = _Entry(ptr(Wq), ptr(X), ptr(Y), N, K)
    return arr


def run_batched(entries, M: int, stream=None):
    """One call over independent products sharing M (one product launch per 160 products).
    `entries` from make_entries()."""
    st = load().qmm_run_batched(entries, len(entries), M, _stream_handle(stream))
    _check(st, "qmm_run_batched")


def ffn_workspace_bytes(M: int, F: int) -> int:
    return load().qmm_ffn_workspace_bytes(M, F)


def run_ffn(Wgu, Wdown, F: int, K: int, X, Y, workspace, M: int | None = None, stream=None):
    """One feed-forward block: Y = (silu(X Wg^T) * (X Wu^T) as bf16) Wdown^T, all on the GPU.
    `workspace`: a device tensor of >= ffn_workspace_bytes(M, F) bytes (holds G and H)."""
    if M is None:
        M = X.shape[0]
    nbytes = workspace.numel() * workspace.element_size()
    st = load().qmm_run_ffn(ctypes.c_void_p(Wgu.data_ptr()), ctypes.c_void_p(Wdown.data_ptr()), F, K,
                            ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(Y.data_ptr()), M,
                            ctypes.c_void_p(workspace.data_ptr()), nbytes, _stream_handle(stream))
    _check(st, "qmm_run_ffn")


def ffn_fused_workspace_bytes(M: int, F: int) -> int:
    return load().qmm_ffn_fused_workspace_bytes(M, F)


def run_ffn_fused(Wgu_interleaved, Wdown, F: int, K: int, X, Y, workspace, M: int | None = None, stream=None):
    """The feed-forward block with the gating in the gate/up product's epilogue.  Wgu_interleaved:
    packed (2F) x K weights with row 2f = gate row f and row 2f+1 = up row f.  `workspace`: a
    device tensor of >= ffn_fused_workspace_bytes(M, F) bytes (holds H)."""
    if M is None:
        M = X.shape[0]
    nbytes = workspace.numel() * workspace.element_size()
    st = load().qmm_run_ffn_fused(ctypes.c_void_p(Wgu_interleaved.data_ptr()), ctypes.c_void_p(Wdown.data_ptr()),
                                  F, K, ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(Y.data_ptr()), M,
                                  ctypes.c_void_p(workspace.data_ptr()), nbytes, _stream_handle(stream))
    _check(st, "qmm_run_ffn_fused")


def indexed_workspace_bytes(M: int, N: int, K: int) -> int:
    return load().qmm_indexed_workspace_bytes(M, N, K)


def run_indexed(experts, N: int, K: int, ids, X, Y, workspace, stream=None):
    """Y[i] = X[i] * dequant(experts[ids[i]])^T for every row i, on the GPU.  `experts`: device
    tensors (packed N x K each); `ids`: host sequence of M expert indices; `workspace`: a device
    tensor of >= indexed_workspace_bytes(M, N, K) bytes."""
    M = len(ids)
    ptrs = (ctypes.c_void_p * len(experts))(*[w.data_ptr() for w in experts])
    idv = (ctypes.c_int32 * M)(*[int(v) for v in ids])
    nbytes = workspace.numel() * workspace.element_size()
    st = load().qmm_run_indexed(ptrs, len(experts), N, K, idv, ctypes.c_void_p(X.data_ptr()),
                                ctypes.c_void_p(Y.data_ptr()), M, ctypes.c_void_p(workspace.data_ptr()), nbytes,
                                _stream_handle(stream))
    _check(st, "qmm_run_indexed")


def dequant(Wq, N: int, K: int, out, stream=None):
    _check(load().qmm_dequant(ctypes.c_void_p(Wq.data_ptr()), N, K, ctypes.c_void_p(out.data_ptr()),
                              _stream_handle(stream)), "qmm_dequant")


def fmt_packed_bytes(fmt: int, N: int, K: int) -> int:
    return load().qmm_fmt_packed_bytes(fmt, N, K)


def fmt_pack(fmt: int, W: np.ndarray, threads: int = 0) -> np.ndarray:
    """Pack an N x K fp32 host array into weight format `fmt` (host, multi-threaded)."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    nbytes = fmt_packed_bytes(fmt, N, K)
    if nbytes == 0:
        raise QmmError(2, "qmm_fmt_pack")
    out = np.empty(nbytes, dtype=np.uint8)
    _check(load().qmm_fmt_pack(fmt, W.ctypes.data_as(ctypes.c_void_p), N, K, out.ctypes.data_as(ctypes.c_void_p),
                               out.nbytes, threads), "qmm_fmt_pack")
    return out


def fmt_run(fmt: int, Wq, N: int, K: int, X, Y, M: int | None = None, stream=None):
    """Y[M x N] = X[M x K] * dequant(Wq)^T for weights in format `fmt`, on the GPU."""
    if M is None:
        M = X.shape[0]
    st = load().qmm_fmt_run(fmt, ctypes.c_void_p(Wq.data_ptr()), N, K, ctypes.c_void_p(X.data_ptr()),
                            ctypes.c_void_p(Y.data_ptr()), M, _stream_handle(stream))
    _check(st, "qmm_fmt_run")


def make_fmt_entries(items):
    """items: sequence of (fmt, Wq, X, Y, N, K) with torch tensors or raw int pointers."""
    arr = (_FmtEntry * len(items))()
    for k, (fmt, Wq, X, Y, N, K) in enumerate(items):
        ptr = lambda t: t if isinstance(t, int) else t.data_ptr()
        arr[k] = _FmtEntry(fmt, ptr(Wq), ptr(X), ptr(Y), N, K)
    return arr


def fmt_run_batched(entries, M: int, stream=None):
    """Independent products sharing M, weights in any formats: each format's entries run as one
    batched call."""
    _check(load().qmm_fmt_run_batched(entries, len(entries), M, _stream_handle(stream)), "qmm_fmt_run_batched")


def fmt_dequant(fmt: int, Wq, N: int, K: int, out, stream=None):
    _check(load().qmm_fmt_dequant(fmt, ctypes.c_void_p(Wq.data_ptr()), N, K, ctypes.c_void_p(out.data_ptr()),
                                  _stream_handle(stream)), "qmm_fmt_dequant")


def select_variant(M: int, N: int, K: int) -> int:
    return load().qmm_select_variant(M, N, K)


def select_variant_batched(entries, M: int) -> int:
    return load().qmm_select_variant_batched(entries, len(entries), M)


def stream_read(buf, sink, stream=None) -> None:
    """qmm_stream_read: read every byte of the device tensor `buf` once (the read-bandwidth probe);
    `sink` is a device uint32 tensor of at least qmm_stream_read_sink_words() words."""
    st = load().qmm_stream_read(ctypes.c_void_p(buf.data_ptr()), buf.numel() * buf.element_size(),
                                ctypes.c_void_p(sink.data_ptr()), _stream_handle(stream))
    _check(st, "qmm_stream_read")


def stream_read_sink_words() -> int:
    return int(load().qmm_stream_read_sink_words())


def set_wait_limit(polls: int = 0, suspend_ns: int = 0) -> None:
    """qmm_set_wait_limit: the tensor-core kernel's wait bound for later launches (0, 0: default)."""
    load().qmm_set_wait_limit(polls, suspend_ns)


def release() -> None:
    """qmm_release: free every tensor-core workspace the library holds (synchronous)."""
    _check(load().qmm_release(), "qmm_release")


def workspace_bytes_held() -> int:
    """qmm_workspace_bytes_held: device bytes the tensor-core workspaces hold now."""
    return int(load().qmm_workspace_bytes_held())


def device_status() -> int:
    v = ctypes.c_uint(0)
    _check(load().qmm_device_status(ctypes.byref(v)), "qmm_device_status")
    return v.value
