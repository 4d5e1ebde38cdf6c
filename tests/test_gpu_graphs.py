"""The C ABI under CUDA-graph capture: a call made while its stream is being captured records its
launches (with their programmatic dependencies) into the graph, and replaying the graph gives
the eager call's bits.  The calls that keep a workspace are made once before capture (it is
sized then; capture cannot allocate).
"""
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


def dev_bytes(host_u8):
    a = np.ascontiguousarray(host_u8)
    return torch.from_numpy(a if a.flags.writeable else a.copy()).cuda()


def dev_x(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy()).cuda().view(torch.bfloat16)


def capture_and_compare(qmm, call, outputs, replays=3):
    """Eager call on a side stream -> reference bits (and the stream's workspace sized); then
    capture `call` on that stream, replay it `replays` times (outputs poisoned before each
    replay) and compare bit for bit."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    assert qmm.device_status() == 0
    ref = [o.clone() for o in outputs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(replays):
        for o in outputs:
            o.fill_(np.nan)
        g.replay()
        torch.cuda.synchronize()
        assert qmm.device_status() == 0
        for o, r in zip(outputs, ref):
            assert torch.equal(o.view(torch.int32), r.view(torch.int32))
    return g


def test_batched_pass_in_a_graph(qmm, oracle_lib):
    M = 8
    shapes = [(5120, 5120), (1024, 5120), (4096, 5120), (5120, 4608)]
    X = {K: dev_x(inputs.activations_bf16_bits(M, K, 10 + K % 7)) for _, K in shapes}
    items, ys = [], []
    for i, (N, K) in enumerate(shapes * 3):
        rows = oracle_lib.pack(inputs.weights_f32(min(N, 512), K, 20 + i))
        W = dev_bytes(np.tile(rows, N // min(N, 512)))   # the packed rows repeated down to row N
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        items.append((W, X[K], Y, N, K))
        ys.append(Y)
    entries = qmm.make_entries(items)
    capture_and_compare(qmm, lambda: qmm.run_batched(entries, M), ys)


def test_mixed_format_batch_in_a_graph(qmm, oracle_lib):
    M = 13
    N, K = 640, 2560
    X = dev_x(inputs.activations_bf16_bits(M, K, 31))
    items, ys = [], []
    for fmt in (qmm.FMT_Q4K, qmm.FMT_Q5K, qmm.FMT_Q6K, qmm.FMT_NVFP4, qmm.FMT_INT4, qmm.FMT_NVFP4):
        W = dev_bytes(oracle_lib.fmt_pack(fmt, inputs.weights_f32(N, K, 40 + fmt)))
        Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        items.append((fmt, W, X, Y, N, K))
        ys.append(Y)
    entries = qmm.make_fmt_entries(items)
    capture_and_compare(qmm, lambda: qmm.fmt_run_batched(entries, M), ys)


@pytest.mark.parametrize("M", [1, 8])
def test_ffn_chain_in_a_graph(qmm, oracle_lib, M):
    F, K = 1536, 1024
    Wgu = dev_bytes(oracle_lib.pack(inputs.weights_f32(2 * F, K, 51)))
    Wdn = dev_bytes(oracle_lib.pack(inputs.weights_f32(K, F, 52)))
    X = dev_x(inputs.activations_bf16_bits(M, K, 53))
    Y = torch.empty((M, K), dtype=torch.float32, device="cuda")
    ws = torch.empty(qmm.ffn_workspace_bytes(M, F), dtype=torch.uint8, device="cuda")
    capture_and_compare(qmm, lambda: qmm.run_ffn(Wgu, Wdn, F, K, X, Y, ws, M=M), [Y])
