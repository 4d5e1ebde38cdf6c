"""CPU tests of the C-ABI library: it loads, exports every symbol of include/qmm.h, validates
arguments before touching the GPU, and its host packer equals the oracle's packer byte for byte."""
import ctypes
import os
import re

import numpy as np
import pytest

from bit_quantized_skinny_gb300 import build_lib, inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qmm():
    build_lib.build()
    from bit_quantized_skinny_gb300 import qmm as q
    q.load()
    return q


def header_functions():
    text = open(os.path.join(ROOT, "include", "qmm.h")).read()
    return sorted(set(re.findall(r"^\s*(?:[\w\s\*]+?)\b(qmm_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(qmm):
    declared = header_functions()
    assert "qmm_run" in declared and "qmm_pack" in declared and "qmm_run_batched" in declared
    lib = qmm.load()
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(declared) == sorted(qmm.EXPORTS)


def test_packed_bytes(qmm):
    assert qmm.packed_bytes(34816, 5120) == 100_270_080
    assert qmm.packed_bytes(248320, 5120) == 715_161_600
    assert qmm.packed_bytes(5120, 17408) == 50_135_040
    assert qmm.packed_bytes(1, 255) == 0
    assert qmm.packed_bytes(0, 256) == 0


def test_argument_errors_need_no_gpu(qmm):
    lib = qmm.load()
    p = ctypes.c_void_p(16)   # never dereferenced: every call below fails validation first
    assert lib.qmm_run(None, 4, 256, p, p, 1, None) == 1
    assert lib.qmm_run(p, 4, 255, p, p, 1, None) == 2
    assert lib.qmm_run(p, 0, 256, p, p, 1, None) == 2
    assert lib.qmm_run(p, 4, 256, p, p, 0, None) == 3
    assert lib.qmm_run(p, 4, 256, p, p, 33, None) == 3
    assert lib.qmm_run(ctypes.c_void_p(24), 4, 256, p, p, 1, None) == 4
    assert lib.qmm_run(p, 4, 256, ctypes.c_void_p(8), p, 1, None) == 4
    assert lib.qmm_run(p, 4, 256, p, ctypes.c_void_p(18), 1, None) == 4
    assert lib.qmm_run_batched(None, 1, 1, None) == 1
    ents = qmm.make_entries([(16, 16, 16, 4, 256)])
    assert lib.qmm_run_batched(ents, 0, 1, None) == 8
    assert lib.qmm_run_batched(ents, 513, 1, None) == 8
    assert lib.qmm_dequant(p, 4, 100, p, None) == 2
    assert lib.qmm_strerror(3) == b"M must be in [1, 32]"
    # the device packer validates on the host before anything is enqueued
    assert lib.qmm_pack_dev(None, 4, 256, p, 4 * 144, None) == 1
    assert lib.qmm_pack_dev(p, 4, 255, p, 4 * 144, None) == 2
    assert lib.qmm_pack_dev(p, 4, 256, p, 4 * 144 - 1, None) == 5
    assert lib.qmm_pack_dev(ctypes.c_void_p(24), 4, 256, p, 4 * 144, None) == 4
    assert lib.qmm_pack_dev(p, 4, 256, ctypes.c_void_p(40), 4 * 144, None) == 4


@pytest.mark.parametrize("shape", [(256, 512), (37, 2304), (5, 256), (64, 5120)])
def test_pack_equals_oracle_pack(qmm, oracle_lib, shape):
    N, K = shape
    W = inputs.weights_f32(N, K, 100 + N)
    assert np.array_equal(qmm.pack(W), oracle_lib.pack(W))
    assert np.array_equal(qmm.pack(W, threads=3), oracle_lib.pack(W))


def test_pack_equals_oracle_on_awkward_values(qmm, oracle_lib):
    rng = np.random.default_rng(9)
    W = (rng.standard_normal((48, 768)) * np.exp(rng.uniform(-12, 6, (48, 1)))).astype(np.float32)
    W[0, :256] = 0.0
    W[1, :256] = -0.0
    W[2, :256] = 3.0
    W[3, :256] = -3.0
    W[4, 0:32] = np.linspace(-1, 1, 32, dtype=np.float32)
    W[5, :] = np.float32(1e-30)
    W[6, :] = np.float32(-7e-6)
    assert np.array_equal(qmm.pack(W), oracle_lib.pack(W))


def test_pack_errors(qmm):
    W = np.zeros((2, 256), np.float32)
    W[1, 3] = np.nan
    with pytest.raises(qmm.QmmError) as e:
        qmm.pack(W)
    assert e.value.status == 6
    W[1, 3] = 1e9
    with pytest.raises(qmm.QmmError):
        qmm.pack(W)
    lib = qmm.load()
    small = np.zeros(10, np.uint8)
    assert lib.qmm_pack(W.ctypes.data_as(ctypes.c_void_p), 2, 256,
                        small.ctypes.data_as(ctypes.c_void_p), small.nbytes, 1) == 5


# ---------------------------------------------------------------- other weight formats ----

FMTS = ["q5k", "q6k", "nvfp4", "int4"]


def test_fmt_packed_bytes(qmm):
    assert qmm.fmt_packed_bytes(qmm.FMT_Q4K, 34816, 5120) == 100_270_080
    assert qmm.fmt_packed_bytes(qmm.FMT_Q5K, 34816, 5120) == 34816 * 20 * 176
    assert qmm.fmt_packed_bytes(qmm.FMT_NVFP4, 34816, 5120) == 100_270_080 + 16
    assert qmm.fmt_packed_bytes(qmm.FMT_INT4, 34816, 5120) == 34816 * 2560 + 34816 * 40 * 2
    assert qmm.fmt_packed_bytes(qmm.FMT_Q6K, 34816, 5120) == 34816 * 20 * 210
    assert qmm.fmt_packed_bytes(9, 4, 256) == 0
    assert qmm.fmt_packed_bytes(qmm.FMT_INT4, 4, 255) == 0


@pytest.mark.parametrize("fmt_name", FMTS)
@pytest.mark.parametrize("shape", [(37, 2304), (5, 256), (64, 5120)])
def test_fmt_pack_equals_oracle_pack(qmm, oracle_lib, fmt_name, shape):
    N, K = shape
    fmt = qmm.FORMATS[fmt_name]
    W = inputs.weights_f32(N, K, 200 + N)
    ref = oracle_lib.fmt_pack(oracle_lib.FORMATS[fmt_name], W)
    assert np.array_equal(qmm.fmt_pack(fmt, W), ref)
    assert np.array_equal(qmm.fmt_pack(fmt, W, threads=3), ref)


@pytest.mark.parametrize("fmt_name", FMTS)
def test_fmt_pack_equals_oracle_on_awkward_values(qmm, oracle_lib, fmt_name):
    rng = np.random.default_rng(19)
    W = (rng.standard_normal((24, 768)) * np.exp(rng.uniform(-12, 6, (24, 1)))).astype(np.float32)
    W[0, :256] = 0.0
    W[1, :256] = -0.0
    W[2, :256] = 3.0
    W[3, :256] = -3.0
    W[4, 0:32] = np.linspace(-1, 1, 32, dtype=np.float32)
    W[5, :] = np.float32(1e-30)
    W[6, :] = np.float32(-7e-6)
    W[7, :] = np.float32(6e4)
    for sub in (W, W[:1] * 0):    # also an all-zero matrix (NVFP4 tensor scale 1)
        ref = oracle_lib.fmt_pack(oracle_lib.FORMATS[fmt_name], sub)
        assert np.array_equal(qmm.fmt_pack(qmm.FORMATS[fmt_name], sub), ref)


def test_fmt_argument_errors_need_no_gpu(qmm):
    lib = qmm.load()
    p = ctypes.c_void_p(16)
    assert lib.qmm_fmt_run(7, p, 4, 256, p, p, 1, None) == 11
    assert lib.qmm_fmt_run(-1, p, 4, 256, p, p, 1, None) == 11
    assert lib.qmm_fmt_run(qmm.FMT_NVFP4, None, 4, 256, p, p, 1, None) == 1
    assert lib.qmm_fmt_run(qmm.FMT_INT4, p, 4, 255, p, p, 1, None) == 2
    assert lib.qmm_fmt_run(qmm.FMT_Q5K, p, 4, 256, p, p, 33, None) == 3
    assert lib.qmm_fmt_run(qmm.FMT_Q5K, ctypes.c_void_p(24), 4, 256, p, p, 1, None) == 4
    assert lib.qmm_fmt_dequant(9, p, 4, 256, p, None) == 11
    assert lib.qmm_fmt_dequant(qmm.FMT_INT4, p, 4, 100, p, None) == 2
    W = np.zeros((2, 256), np.float32)
    W[0, 1] = np.inf
    for fmt in (qmm.FMT_Q5K, qmm.FMT_Q6K, qmm.FMT_NVFP4, qmm.FMT_INT4):
        with pytest.raises(qmm.QmmError) as e:
            qmm.fmt_pack(fmt, W)
        assert e.value.status == 6
    small = np.zeros(10, np.uint8)
    W[0, 1] = 0
    assert lib.qmm_fmt_pack(qmm.FMT_INT4, W.ctypes.data_as(ctypes.c_void_p), 2, 256,
                            small.ctypes.data_as(ctypes.c_void_p), small.nbytes, 1) == 5
    assert lib.qmm_fmt_pack(5, W.ctypes.data_as(ctypes.c_void_p), 2, 256,
                            small.ctypes.data_as(ctypes.c_void_p), small.nbytes, 1) == 11
    assert lib.qmm_strerror(11) == b"unknown weight format code"


def test_fmt_batched_argument_errors_need_no_gpu(qmm):
    lib = qmm.load()
    ok = (qmm.FMT_NVFP4, 16, 16, 16, 4, 256)
    assert lib.qmm_fmt_run_batched(None, 1, 1, None) == 1
    ents = qmm.make_fmt_entries([ok])
    assert lib.qmm_fmt_run_batched(ents, 0, 1, None) == 8
    assert lib.qmm_fmt_run_batched(ents, 1, 0, None) == 3
    assert lib.qmm_fmt_run_batched(qmm.make_fmt_entries([ok, (7, 16, 16, 16, 4, 256)]), 2, 1, None) == 11
    assert lib.qmm_fmt_run_batched(qmm.make_fmt_entries([ok, (qmm.FMT_Q6K, 16, 16, 16, 4, 300)]), 2, 1, None) == 2
    assert lib.qmm_fmt_run_batched(qmm.make_fmt_entries([ok, (qmm.FMT_Q5K, 24, 16, 16, 4, 256)]), 2, 1, None) == 4


def test_force_variant_environment_override(qmm):
    """QMM_FORCE_VARIANT=fma|tc overrides the automatic choice (read once per process, so each
    setting runs in a fresh interpreter; no GPU needed to ask for the choice)."""
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, %r); from bit_quantized_skinny_gb300 import qmm; "
            "print(qmm.select_variant(8, 248320, 5120), qmm.select_variant(1, 1024, 5120))") % ROOT
    picks = {}
    for val in (None, "fma", "tc", "bogus"):
        env = dict(os.environ)
        env.pop("QMM_FORCE_VARIANT", None)
        if val:
            env["QMM_FORCE_VARIANT"] = val
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
        picks[val] = tuple(int(v) for v in out.stdout.split())
    assert picks["fma"] == (qmm.VARIANT_FMA, qmm.VARIANT_FMA)
    assert picks["tc"] == (qmm.VARIANT_TC, qmm.VARIANT_TC)
    assert picks["bogus"] == picks[None]


@pytest.mark.parametrize("fmt_name", ["q4k", "q5k", "q6k", "nvfp4", "int4"])
def test_packed_weights_fmt_replicates_rows(qmm, fmt_name):
    """The benchmark's timing buffers: the first chunk of rows packed by the library and repeated
    down to row N, each plane of the format repeated on its own (host memory, no GPU)."""
    from bit_quantized_skinny_gb300 import workloads
    fmt = qmm.FORMATS[fmt_name]
    N, K = inputs.ROWS_PER_CHUNK * 2 + 5, 512
    out = workloads.packed_weights_fmt(fmt, N, K, 7, device="cpu").numpy()
    chunk = qmm.fmt_pack(fmt, inputs.weights_f32(inputs.ROWS_PER_CHUNK, K, 7))
    R = inputs.ROWS_PER_CHUNK
    idx = np.arange(N) % R
    if fmt == qmm.FMT_INT4:
        planes = [(K // 2, 0, 0), (K // 64, N * K // 2, R * K // 2)]
    elif fmt == qmm.FMT_Q6K:
        planes = [((K // 256) * 208, 0, 0), ((K // 256) * 2, N * (K // 256) * 208, R * (K // 256) * 208)]
    else:
        planes = [((K // 256) * (176 if fmt == qmm.FMT_Q5K else 144), 0, 0)]
    for rb, off, coff in planes:
        got = out[off:off + N * rb].reshape(N, rb)
        ref = chunk[coff:coff + R * rb].reshape(R, rb)[idx]
        assert np.array_equal(got, ref)
    if fmt == qmm.FMT_NVFP4:
        assert np.array_equal(out[-16:], chunk[-16:])
    assert out.size == qmm.fmt_packed_bytes(fmt, N, K)


def test_release_without_workspaces_needs_no_gpu(qmm):
    """qmm_release with nothing allocated touches no device; nothing is held afterwards."""
    assert qmm.load().qmm_release() == 0
    assert qmm.workspace_bytes_held() == 0
