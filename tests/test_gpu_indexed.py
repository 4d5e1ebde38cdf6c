"""GPU parity of the indexed-expert product (qmm_run_indexed): row i of X times expert ids[i],
through the C ABI, against the oracle row by row (each within 1e-4 * sum|w x|)."""
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


def _dev_x(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).cuda().view(torch.bfloat16)


@pytest.fixture(scope="module")
def experts(oracle_lib):
    N, K, E = 384, 512, 6
    packed = [oracle_lib.pack(inputs.weights_f32(N, K, 1100 + e)) for e in range(E)]
    return N, K, packed, [torch.from_numpy(p).cuda() for p in packed]


@pytest.mark.parametrize("ids", [[3], [0, 0, 0, 0, 0], [5, 1, 5, 2, 1, 5, 0, 4],
                                 list(range(6)) * 2 + [2, 2, 2, 2], [1] * 32,
                                 [i % 6 for i in range(32)], [4, 4, 4, 4, 4, 4, 4, 4, 4, 0]])
def test_indexed_rows_match_their_experts(qmm, oracle_lib, experts, ids):
    N, K, packed, dev = experts
    M = len(ids)
    X = inputs.activations_bf16_bits(M, K, 1200 + M)
    Y = torch.full((M, N), 5.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(qmm.indexed_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    ws.fill_(0xFF)   # garbage (NaN patterns) in the workspace must not leak into any result
    qmm.run_indexed(dev, N, K, ids, _dev_x(X), Y, ws)
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    got = Y.cpu().numpy()
    for i, e in enumerate(ids):
        Yref, S = oracle_lib.matmul(packed[e], N, K, X[i:i + 1])
        err = np.abs(got[i].astype(np.float64) - Yref[0])
        assert np.all(err <= TOL * S[0]), f"row {i} (expert {e}): max err {err.max()}"


def test_indexed_argument_errors(qmm, experts):
    N, K, _, dev = experts
    X = torch.zeros((2, K), dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros((2, N), device="cuda")
    ws = torch.empty(qmm.indexed_workspace_bytes(2, N, K), dtype=torch.uint8, device="cuda")
    with pytest.raises(qmm.QmmError) as ei:
        qmm.run_indexed(dev, N, K, [0, 6], X, Y, ws)          # id out of range
    assert ei.value.status == 2
    with pytest.raises(qmm.QmmError) as ei:
        qmm.run_indexed(dev, N, K, [0, 1], X, Y, ws[:-16])    # workspace too small
    assert ei.value.status == 5
