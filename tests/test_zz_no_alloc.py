"""qmm_run_noalloc: the product for callers that cannot allocate device memory when they call
in (a stream being captured into a CUDA graph, a decode loop that must not touch the device
allocator, a host that owns a fixed device-memory budget).  It runs the tensor-core kernel with
its prepared activations in the library's fixed 4 MiB device buffer.

This file is collected last on purpose, so that a run stopping at the first failure has run
every other test before it.  It must pass on its own in a fresh process as well as after the
rest of the suite.
"""
import ctypes

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


def _dev(host_u8):
    return torch.from_numpy(np.ascontiguousarray(host_u8).copy()).cuda()


def _dev_x(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).cuda().view(torch.bfloat16)


def test_noalloc_matches_qmm_run_on_two_calls_in_a_row(qmm, oracle_lib):
    """Two different problems back to back through the C ABI: each result must agree with the
    existing entry point (qmm_run) and with the oracle within 1e-4 * sum|w*x|; the second call
    must not be disturbed by what the first one left in the shared buffer."""
    lib = qmm.load()
    stream = torch.cuda.current_stream().cuda_stream
    for (N, K, M, seed) in [(1001, 2304, 20, 3), (777, 5120, 5, 4)]:
        Wq = oracle_lib.pack(inputs.weights_f32(N, K, seed))
        X = inputs.activations_bf16_bits(M, K, seed + 100)
        Wd, Xd = _dev(Wq), _dev_x(X)
        Y_new = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
        Y_old = torch.full((M, N), -7.0, dtype=torch.float32, device="cuda")
        st = lib.qmm_run_noalloc(ctypes.c_void_p(Wd.data_ptr()), N, K, ctypes.c_void_p(Xd.data_ptr()),
                                 ctypes.c_void_p(Y_new.data_ptr()), M, ctypes.c_void_p(stream))
        assert st == 0, qmm.QmmError(st, "qmm_run_noalloc")
        st = lib.qmm_run(ctypes.c_void_p(Wd.data_ptr()), N, K, ctypes.c_void_p(Xd.data_ptr()),
                         ctypes.c_void_p(Y_old.data_ptr()), M, ctypes.c_void_p(stream))
        assert st == 0
        torch.cuda.synchronize()
        assert qmm.device_status() == 0
        Yref, S = oracle_lib.matmul(Wq, N, K, X)
        y_new = Y_new.cpu().numpy().astype(np.float64)
        y_old = Y_old.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(y_new - y_old) <= TOL * S)
        assert np.all(np.abs(y_new - Yref) <= TOL * S)


def _limit_k(tw):
    """Largest K the fixed buffer takes: (K/256) prepared blocks of tw * 580 + 16 bytes (tw: the
    token columns a block stores, 8 for M <= 8, 16 for M <= 16, 32 above)."""
    return (4 << 20) // (tw * 580 + 16) * 256


def test_noalloc_rejects_problems_larger_than_its_buffer(qmm):
    lib = qmm.load()
    p = ctypes.c_void_p(256)   # never dereferenced: the size check comes before any GPU work
    assert lib.qmm_run_noalloc(p, 8, _limit_k(32) + 256, p, p, 32, None) == 10   # one super-block too many, Mpad 32
    assert lib.qmm_run_noalloc(p, 8, _limit_k(16) + 256, p, p, 16, None) == 10   # and at Mpad 16
    assert lib.qmm_run_noalloc(p, 8, _limit_k(8) + 256, p, p, 8, None) == 10     # and with 8 token columns
    assert lib.qmm_strerror(10).startswith(b"qmm_run_noalloc")


@pytest.mark.parametrize("M", [32, 16, 8])
def test_noalloc_accepts_the_largest_problem_its_buffer_holds(qmm, oracle_lib, M):
    """At exactly the limit the call runs, and agrees with qmm_run within the tolerance."""
    lib = qmm.load()
    stream = torch.cuda.current_stream().cuda_stream
    N, K = 40, _limit_k(32 if M > 16 else (16 if M > 8 else 8))
    Wq = oracle_lib.pack(inputs.weights_f32(N, K, 71))
    X = inputs.activations_bf16_bits(M, K, 72)
    Wd, Xd = _dev(Wq), _dev_x(X)
    Y_new = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    Y_old = torch.full((M, N), -7.0, dtype=torch.float32, device="cuda")
    st = lib.qmm_run_noalloc(ctypes.c_void_p(Wd.data_ptr()), N, K, ctypes.c_void_p(Xd.data_ptr()),
                             ctypes.c_void_p(Y_new.data_ptr()), M, ctypes.c_void_p(stream))
    assert st == 0, qmm.QmmError(st, "qmm_run_noalloc")
    st = lib.qmm_run(ctypes.c_void_p(Wd.data_ptr()), N, K, ctypes.c_void_p(Xd.data_ptr()),
                     ctypes.c_void_p(Y_old.data_ptr()), M, ctypes.c_void_p(stream))
    assert st == 0
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    Yref, S = oracle_lib.matmul(Wq, N, K, X)
    y_new = Y_new.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y_new - Y_old.cpu().numpy().astype(np.float64)) <= TOL * S)
    assert np.all(np.abs(y_new - Yref) <= TOL * S)
