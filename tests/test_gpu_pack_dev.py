"""The device-side packer (qmm_pack_dev) against the oracle's packer: byte for byte on the same
weights, including sub-blocks of zeros, of one repeated value, of extreme magnitudes and tiny
values; non-finite weights and fp16 scale overflow give zero super-blocks and status bit 1."""
import numpy as np
import pytest
import torch

from bit_quantized_skinny_gb300 import build_lib, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def qmm():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    build_lib.build()
    from bit_quantized_skinny_gb300 import qmm as q
    q.load()
    return q


def awkward(N, K, seed):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * np.exp(rng.uniform(-14, 8, (N, 1)))).astype(np.float32)
    W[0, :256] = 0.0
    W[1, :256] = -0.0
    W[2, :256] = 3.0
    W[3, :256] = -3.0
    W[4, 0:32] = np.linspace(-1, 1, 32, dtype=np.float32)
    W[5, :] = np.float32(1e-30)
    W[6, :] = np.float32(-7e-39)            # fp32 subnormals
    W[7, :] = rng.uniform(0.5, 1.0, K).astype(np.float32)   # no negative weight: offset 0
    W[8, :] = -rng.uniform(0.5, 1.0, K).astype(np.float32)
    W[9, 32:64] = np.float32(60000.0)
    return W


@pytest.mark.parametrize("N,K,seed", [(256, 512, 1), (37, 2304, 2), (300, 5120, 3), (1, 256, 4)])
def test_pack_dev_equals_oracle_pack(qmm, oracle_lib, N, K, seed):
    W = inputs.weights_f32(N, K, seed)
    out = qmm.pack_dev(torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    assert np.array_equal(out.cpu().numpy(), oracle_lib.pack(W))


def test_pack_dev_equals_oracle_on_awkward_values(qmm, oracle_lib):
    W = awkward(48, 768, 9)
    out = qmm.pack_dev(torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    ref = oracle_lib.pack(W)
    assert np.array_equal(out.cpu().numpy(), ref)
    assert np.array_equal(ref, qmm.pack(W))


def test_pack_dev_on_a_stream_into_a_given_buffer(qmm, oracle_lib):
    N, K = 64, 1024
    W = inputs.weights_f32(N, K, 21)
    buf = torch.full((qmm.packed_bytes(N, K) + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    Wd = torch.from_numpy(W).cuda()
    torch.cuda.current_stream().synchronize()
    qmm.pack_dev(Wd, out=buf, stream=s)
    s.synchronize()
    host = buf.cpu().numpy()
    assert np.array_equal(host[:qmm.packed_bytes(N, K)], oracle_lib.pack(W))
    assert np.all(host[qmm.packed_bytes(N, K):] == 0xA5)   # nothing written past the packed bytes


def test_pack_dev_marks_bad_super_blocks(qmm, oracle_lib):
    N, K = 6, 512
    W = inputs.weights_f32(N, K, 33)
    W[1, 300] = np.nan                      # super-block 1 of row 1
    W[3, 5] = np.inf                        # super-block 0 of row 3
    W[4, 256:288] = np.float32(3e38)        # step / 63 overflows binary16: super-block 1 of row 4
    out = qmm.pack_dev(torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    assert qmm.device_status() & 2
    assert qmm.device_status() == 0          # reading cleared it
    got = out.cpu().numpy().reshape(N, 2, 144)
    bad = {(1, 1), (3, 0), (4, 1)}
    good = W.copy()
    for (n, b) in bad:
        good[n, 256 * b:256 * b + 256] = 0.0
    ref = oracle_lib.pack(good).reshape(N, 2, 144)
    for n in range(N):
        for b in range(2):
            if (n, b) in bad:
                assert np.all(got[n, b] == 0), (n, b)
            else:
                assert np.array_equal(got[n, b], ref[n, b]), (n, b)
