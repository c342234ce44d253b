"""The C-ABI library without a GPU: it loads, exports every function that
include/qgemv.h declares, and rejects bad arguments with status codes before
it touches CUDA. No compute call runs here."""
import ctypes
import os
import re

import pytest

import ggml_block_quantized_gb300 as qg
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")

OK, ERR_TYPE, ERR_SHAPE, ERR_ALIGN, ERR_NULL, ERR_PAIR, ERR_CUDA, ERR_WS = 0, -1, -2, -3, -4, -5, -6, -7


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    return qg.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)))


def test_header_declarations_are_exported(L):
    names = declared_functions()
    assert len(names) == 23
    assert sorted(qg.EXPORTED_SYMBOLS) == names
    for n in names:
        assert hasattr(L, n), n
    # they are real dynamic symbols of the library
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", qg.library_path()], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert set(names) <= exported


def test_type_table_matches_the_oracle(L):
    for t in (qg.F32, qg.F16, qg.Q4_0, qg.Q4_1, qg.Q5_0, qg.Q8_0, qg.Q8_1, qg.Q2_K, qg.Q3_K, qg.Q4_K,
              qg.Q5_K, qg.Q6_K, qg.Q8_K):
        assert qg.qtype_block(t) == oracle.type_info(t)
        for n in (0, 256, 4096, 11008, 32 * 7, 100):
            assert qg.qtype_nbytes(t, n) == oracle.type_nbytes(t, n)
    with pytest.raises(qg.QGError):
        qg.qtype_block(7)
    assert qg.qtype_nbytes(99, 256) == -1
    assert qg.qtype_nbytes(qg.Q8_0, -32) == -1


def test_pairing(L):
    assert qg.qtype_act_type(qg.Q4_0) == qg.Q8_0
    assert qg.qtype_act_type(qg.Q8_0) == qg.Q8_0
    assert qg.qtype_act_type(qg.Q4_K) == qg.Q8_K
    assert qg.qtype_act_type(qg.Q6_K) == qg.Q8_K
    assert qg.qtype_act_type(qg.Q5_0) == qg.Q8_0
    assert qg.qtype_act_type(qg.Q4_1) == qg.Q8_1
    for t in (qg.Q2_K, qg.Q3_K, qg.Q5_K):
        assert qg.qtype_act_type(t) == qg.Q8_K
    for t in (qg.F32, qg.F16, qg.Q8_K, qg.Q8_1, 7, 99):
        assert qg.qtype_act_type(t) == ERR_PAIR


def test_workspace_bytes(L):
    assert qg.qgemv_workspace_bytes(qg.Q4_K, 4096, 1) == 16 * 292
    assert qg.qgemv_workspace_bytes(qg.Q6_K, 11008, 8) == 8 * 43 * 292
    assert qg.qgemv_workspace_bytes(qg.Q4_0, 4096, 2) == 2 * 128 * 34
    assert qg.qgemv_workspace_bytes(qg.Q4_0, 100, 1) == 0
    assert qg.qgemv_workspace_bytes(qg.Q4_0, 4096, 9) == 0
    assert qg.qgemv_workspace_bytes(qg.Q8_K, 4096, 1) == 0
    assert qg.qgemv_workspace_bytes(qg.Q4_1, 4096, 2) == 2 * 128 * 36
    assert qg.qgemv_workspace_bytes(qg.Q5_0, 4096, 3) == 3 * 128 * 34


def test_status_strings(L):
    for s in range(-8, 1):
        assert L.qg_status_string(s)


# fake device addresses: validation must reject before any CUDA call
A = ctypes.c_void_p(0x10000)
A2 = ctypes.c_void_p(0x20000)
A3 = ctypes.c_void_p(0x30000)
MIS = ctypes.c_void_p(0x10008)
NUL = None


def test_qgemv_validation(L):
    ws = ctypes.c_size_t(1 << 20)
    g = lambda *a: L.qgemv(*a)
    assert g(99, A, A2, A3, 16, 256, 1, A, ws, NUL) == ERR_TYPE
    assert g(qg.Q8_K, A, A2, A3, 16, 256, 1, A, ws, NUL) == ERR_PAIR
    assert g(qg.F32, A, A2, A3, 16, 256, 1, A, ws, NUL) == ERR_PAIR
    assert g(qg.Q4_K, A, A2, A3, 16, 250, 1, A, ws, NUL) == ERR_SHAPE
    assert g(qg.Q4_0, A, A2, A3, 16, 100, 1, A, ws, NUL) == ERR_SHAPE  # a row of 100 is rejected
    assert g(qg.Q4_K, A, A2, A3, 16, 256, 0, A, ws, NUL) == ERR_SHAPE
    assert g(qg.Q4_K, A, A2, A3, 16, 256, 9, A, ws, NUL) == ERR_SHAPE
    assert g(qg.Q4_K, A, A2, A3, -1, 256, 1, A, ws, NUL) == ERR_SHAPE
    assert g(qg.Q4_K, NUL, A2, A3, 16, 256, 1, A, ws, NUL) == ERR_NULL
    assert g(qg.Q4_K, A, NUL, A3, 16, 256, 1, A, ws, NUL) == ERR_NULL
    assert g(qg.Q4_K, A, A2, NUL, 16, 256, 1, A, ws, NUL) == ERR_NULL
    assert g(qg.Q4_K, MIS, A2, A3, 16, 256, 1, A, ws, NUL) == ERR_ALIGN
    assert g(qg.Q4_K, A, MIS, A3, 16, 256, 1, A, ws, NUL) == ERR_ALIGN
    assert g(qg.Q4_K, A, A2, MIS, 16, 256, 1, A, ws, NUL) == ERR_ALIGN
    assert g(qg.Q4_K, A, A2, A3, 16, 256, 1, NUL, ws, NUL) == ERR_WS
    assert g(qg.Q4_K, A, A2, A3, 16, 256, 1, A, ctypes.c_size_t(291), NUL) == ERR_WS
    assert g(qg.Q4_K, A, A2, A3, 16, 256, 1, MIS, ws, NUL) == ERR_ALIGN
    # empty output: nothing to do, nothing enqueued
    assert g(qg.Q4_K, A, A2, A3, 0, 256, 1, A, ws, NUL) == OK


def test_prefill_validation(L):
    """qgemm / qgemm_f16 reject bad arguments before any CUDA call."""
    need = L.qgemm_workspace_bytes(qg.Q4_K, 64, 512, 10)
    assert need == (2 * 64 * 512 + 255) // 256 * 256 + (2 * 10 * 512 + 255) // 256 * 256
    assert L.qgemm_workspace_bytes(qg.Q4_K, 64, 500, 10) == 0
    assert L.qgemm_workspace_bytes(99, 64, 512, 10) == 0
    ws = ctypes.c_size_t(need)
    g = lambda *a: L.qgemm(*a)
    assert g(99, A, A2, A3, 64, 512, 10, A, ws, NUL) == ERR_TYPE
    assert g(qg.Q8_K, A, A2, A3, 64, 512, 10, A, ws, NUL) == ERR_PAIR
    assert g(qg.Q4_K, A, A2, A3, 64, 500, 10, A, ws, NUL) == ERR_SHAPE
    assert g(qg.Q4_K, A, A2, A3, -1, 512, 10, A, ws, NUL) == ERR_SHAPE
    assert g(qg.Q4_K, A, A2, A3, 64, 512, -1, A, ws, NUL) == ERR_SHAPE
    assert g(qg.Q4_K, NUL, A2, A3, 64, 512, 10, A, ws, NUL) == ERR_NULL
    assert g(qg.Q4_K, A, A2, NUL, 64, 512, 10, A, ws, NUL) == ERR_NULL
    assert g(qg.Q4_K, A, A2, A3, 64, 512, 10, NUL, ws, NUL) == ERR_NULL
    assert g(qg.Q4_K, MIS, A2, A3, 64, 512, 10, A, ws, NUL) == ERR_ALIGN
    assert g(qg.Q4_K, A, A2, MIS, 64, 512, 10, A, ws, NUL) == ERR_ALIGN
    assert g(qg.Q4_K, A, A2, A3, 64, 512, 10, A, ctypes.c_size_t(need - 1), NUL) == ERR_WS
    assert g(qg.Q4_K, A, A2, A3, 0, 512, 10, A, ws, NUL) == OK  # nothing to do
    assert g(qg.Q4_K, A, A2, A3, 64, 512, 0, A, ws, NUL) == OK
    f = lambda *a: L.qgemm_f16(*a)
    assert f(A, A2, A3, 64, 10, 500, NUL) == ERR_SHAPE  # K not a multiple of 8
    assert f(A, A2, A3, -1, 10, 512, NUL) == ERR_SHAPE
    assert f(NUL, A2, A3, 64, 10, 512, NUL) == ERR_NULL
    assert f(A, A2, NUL, 64, 10, 512, NUL) == ERR_NULL
    assert f(A, MIS, A3, 64, 10, 512, NUL) == ERR_ALIGN
    assert f(A, A2, A3, 0, 10, 512, NUL) == OK


def test_other_entry_points_validate(L):
    assert L.quantize_act(qg.Q4_0, A, A2, 256, 1, NUL) == ERR_TYPE
    assert L.quantize_act(qg.Q8_K, A, A2, 100, 1, NUL) == ERR_SHAPE
    assert L.quantize_act(qg.Q8_0, NUL, A2, 64, 1, NUL) == ERR_NULL
    assert L.quantize_act(qg.Q8_0, MIS, A2, 64, 1, NUL) == ERR_ALIGN
    assert L.quantize_act(qg.Q8_0, A, A2, 0, 1, NUL) == OK
    assert L.quantize_rows(qg.Q4_K, A, A2, 1, 256, NUL) == ERR_TYPE
    assert L.quantize_rows(qg.Q4_0, A, A2, 1, 33, NUL) == ERR_SHAPE
    assert L.quantize_rows(qg.Q8_1, A, A2, 1, 32, NUL) == ERR_TYPE   # activations only
    assert L.quantize_act(qg.Q4_1, A, A2, 32, 1, NUL) == ERR_TYPE
    assert L.quantize_act(qg.Q8_1, A, A2, 33, 1, NUL) == ERR_SHAPE
    assert L.quantize_rows(qg.Q5_0, A, A2, 1, 48, NUL) == ERR_SHAPE
    assert L.dequantize_rows(qg.F32, A, A2, 1, 256, NUL) == ERR_TYPE
    assert L.dequantize_rows(qg.Q6_K, A, A2, 1, 255, NUL) == ERR_SHAPE
    assert L.dequantize_rows(qg.Q6_K, A, MIS, 1, 256, NUL) == ERR_ALIGN
    assert L.qgemv_xq(qg.Q6_K, A, NUL, A3, 4, 256, 1, NUL) == ERR_NULL
    assert L.qgemv_block_isums(qg.Q6_K, A, A2, NUL, 4, 256, 1, NUL) == ERR_NULL
    assert L.qgemv_block_isums(qg.Q4_0, A, A2, A3, 4, 256, 0, NUL) == ERR_SHAPE
    assert L.qg_device_error(None) == ERR_NULL
    # bad arguments give an empty description before any CUDA call
    assert L.qgemv_kernel_info(qg.Q8_K, 16, 256, 1, 1) == b""
    assert L.qgemv_kernel_info(qg.Q4_K, 16, 250, 1, 1) == b""
    assert L.qgemv_kernel_info(qg.Q4_K, 16, 256, 9, 1) == b""
    assert L.qgemv_kernel_info(qg.Q4_K, 16, 256, 1, 0) == b""
    assert L.qgemm_kernel_info(qg.Q8_K, 16, 256, 4) == b""
    assert L.qgemm_kernel_info(qg.Q4_K, 16, 250, 4) == b""
    assert L.qgemm_kernel_info(qg.Q4_K, 0, 256, 4) == b""
    assert L.qgemm_kernel_info(qg.Q4_K, 16, 256, 0) == b""


def test_tune_knobs(L):
    """qg_tune sets a knob for the process, returns the old value, clamps to
    the knob's range and rejects unknown names (no CUDA call involved)."""
    prev = ctypes.c_int32(-1)
    assert L.qg_tune(None, 1, None) == ERR_NULL
    assert L.qg_tune(b"QG_NO_SUCH_KNOB", 1, None) == ERR_TYPE
    assert L.qg_tune(b"QG_TC", 1, ctypes.byref(prev)) == OK
    old = prev.value
    assert old in (0, 1)
    assert L.qg_tune(b"QG_TC", 7, ctypes.byref(prev)) == OK and prev.value == 1
    assert L.qg_tune(b"QG_TC", old, ctypes.byref(prev)) == OK and prev.value == 1  # clamped to 1
    assert qg.tune("QG_MMA_MIN_NVEC", 3) in range(1, 10)
    old = qg.tune("QG_FUSED_GEMM", 9)  # 0, 1 or 2 (the default: fused up to 512 tokens)
    assert old in (0, 1, 2)
    assert qg.tune("QG_FUSED_GEMM", old) == 2  # clamped to 2
    old = qg.tune("QG_GEMM_KSPLIT", 0)  # 1 .. 8 parts (the default: at most 8)
    assert old == 8 and qg.tune("QG_GEMM_KSPLIT", old) == 1  # clamped to 1


def test_batched_validation(L):
    Mat = qg.GemvMat
    ws = ctypes.c_size_t(1 << 20)
    one = (Mat * 1)(Mat(0x10000, 0x20000, 0x30000, 16))
    assert L.qgemv_batched(99, one, 1, 256, 1, A, ws, NUL) == ERR_TYPE
    assert L.qgemv_batched(qg.Q8_K, one, 1, 256, 1, A, ws, NUL) == ERR_PAIR
    assert L.qgemv_batched(qg.Q4_K, None, 1, 256, 1, A, ws, NUL) == ERR_NULL
    assert L.qgemv_batched(qg.Q4_K, one, 0, 256, 1, A, ws, NUL) == ERR_SHAPE
    assert L.qgemv_batched(qg.Q4_K, one, 257, 256, 1, A, ws, NUL) == ERR_SHAPE
    assert L.qgemv_batched(qg.Q4_K, one, 1, 250, 1, A, ws, NUL) == ERR_SHAPE
    bad = (Mat * 2)(Mat(0x10000, 0x20000, 0x30000, 16), Mat(0x10000, 0x20008, 0x30000, 16))
    assert L.qgemv_batched(qg.Q4_K, bad, 2, 256, 1, A, ws, NUL) == ERR_ALIGN
    nul = (Mat * 2)(Mat(0x10000, 0x20000, 0x30000, 16), Mat(0x10000, 0, 0x30000, 16))
    assert L.qgemv_batched(qg.Q4_K, nul, 2, 256, 1, A, ws, NUL) == ERR_NULL
    # large activations need the quantized copies in the workspace
    assert qg.qgemv_batched_workspace_bytes(qg.Q4_K, 4096, 8, 3) == 3 * 8 * 16 * 292
    assert qg.qgemv_batched_workspace_bytes(qg.Q4_K, 4096, 1, 3) == 16
    assert qg.qgemv_batched_workspace_bytes(qg.Q4_K, 4096, 1, 0) == 0
    big = (Mat * 2)(Mat(0x10000, 0x20000, 0x30000, 16), Mat(0x10000, 0x20000, 0x30000, 16))
    assert L.qgemv_batched(qg.Q4_K, big, 2, 4096, 8, A, ctypes.c_size_t(100), NUL) == ERR_WS


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(qg, "_lib", None)
    monkeypatch.setattr(qg, "library_path", lambda: "/nonexistent/libqgemv.so")
    with pytest.raises(ImportError):
        qg.lib()
