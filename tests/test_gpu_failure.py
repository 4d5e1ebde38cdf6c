"""Failure detection of the tensor-core kernel, made to happen without a GPU fault.

Every wait of the kernel is bounded.  qmm_set_wait_limit lowers the bound for later launches; at
two polls of at most 50 ns the kernel's first wait for its weight copies runs out (a copy takes a
memory access's latency, far longer).  The kernel must then record bit 0 of the device status
word, stop its other warps, wait for what it already issued and return, leaving the context
usable: the next call, with the default bound, computes the product correctly.
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


@pytest.mark.parametrize("N,K,M", [(2048, 17408, 8), (4096, 5120, 24)])
def test_wait_bound_runs_out_and_the_kernel_returns(qmm, oracle_lib, N, K, M):
    Wq = oracle_lib.pack(inputs.weights_f32(N, K, 31))
    X = inputs.activations_bf16_bits(M, K, 32)
    Wd = torch.from_numpy(Wq.copy()).cuda()
    Xd = torch.from_numpy(X.view(np.int16).copy()).cuda().view(torch.bfloat16)
    assert qmm.device_status() == 0
    Y = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    qmm.set_wait_limit(2, 50)
    try:
        qmm.run(Wd, N, K, Xd, Y, M=M, variant=qmm.VARIANT_TC)
    finally:
        qmm.set_wait_limit(0, 0)
    torch.cuda.synchronize()              # the kernel gave up and ended
    assert qmm.device_status() & 1        # ... and said so
    assert qmm.device_status() == 0       # reading cleared it
    Y2 = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    qmm.run(Wd, N, K, Xd, Y2, M=M, variant=qmm.VARIANT_TC)
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    rows = np.arange(0, N, 37)
    Yref, S = oracle_lib.matmul(Wq, N, K, X, rows=rows)
    assert np.all(np.abs(Y2.cpu().numpy()[:, rows].astype(np.float64) - Yref) <= TOL * S)
