"""GB300 block-quantized matrix-vector product: thin Python binding.

The work happens in the CUDA library libqgemv.so (the C ABI of
include/qgemv.h); this module only marshals arguments: it checks dtypes,
devices and sizes of torch tensors, allocates outputs with torch when the
caller passes none, and calls the C entry points with raw device pointers and
the current CUDA stream. There is no fallback: if the library is missing,
importing this module raises.

Element types are the ggml ids (Q4_0=2, Q4_1=3, Q5_0=6, Q8_0=8, Q8_1=9,
Q2_K=10, Q3_K=11, Q4_K=12, Q5_K=13, Q6_K=14, Q8_K=15).
"""
import ctypes
import os

__all__ = [
    "F32", "F16", "Q4_0", "Q4_1", "Q5_0", "Q8_0", "Q8_1", "Q2_K", "Q3_K", "Q4_K", "Q5_K", "Q6_K", "Q8_K",
    "MAX_NVEC", "QGError",
    "library_path", "lib", "qtype_nbytes", "qtype_block", "qtype_act_type",
    "quantize_act", "quantize_rows", "dequantize_rows", "qgemv_workspace_bytes",
    "qgemv", "qgemv_xq", "qgemv_block_isums", "qgemv_noalloc", "qgemv_batched",
    "qgemv_batched_workspace_bytes", "BatchPlan", "device_error", "kernel_info", "EXPORTED_SYMBOLS",
    "MAX_BATCH", "tune", "qgemm_workspace_bytes", "qgemm", "qgemm_f16", "selftest_bounded_wait",
    "gemm_kernel_info",
]

F32, F16, Q4_0, Q4_1, Q5_0, Q8_0, Q8_1 = 0, 1, 2, 3, 6, 8, 9
Q2_K, Q3_K, Q4_K, Q5_K, Q6_K, Q8_K = 10, 11, 12, 13, 14, 15
MAX_NVEC = 8
TYPE_NAMES = {F32: "F32", F16: "F16", Q4_0: "Q4_0", Q4_1: "Q4_1", Q5_0: "Q5_0", Q8_0: "Q8_0",
              Q8_1: "Q8_1", Q2_K: "Q2_K", Q3_K: "Q3_K", Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K",
              Q8_K: "Q8_K"}

# every function declared in include/qgemv.h
EXPORTED_SYMBOLS = (
    "qtype_nbytes", "qtype_block", "qtype_act_type", "qg_status_string", "qg_last_cuda_error",
    "quantize_act", "quantize_rows", "dequantize_rows", "qgemv_workspace_bytes", "qgemv",
    "qgemv_xq", "qgemv_block_isums", "qg_device_error", "qgemv_noalloc",
    "qgemv_batched_workspace_bytes", "qgemv_batched", "qgemv_kernel_info", "qg_tune",
    "qgemm_workspace_bytes", "qgemm", "qgemm_f16", "qg_selftest_bounded_wait", "qgemm_kernel_info",
)
MAX_BATCH = 256


class GemvMat(ctypes.Structure):
    """qg_gemv_mat: one matrix of a batched call."""
    _fields_ = [("W", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p), ("n_out", ctypes.c_int64)]

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "_build", "libqgemv.so")


class QGError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().qg_status_string(status).decode()
        if status == -6:
            msg += ": " + lib().qg_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


_lib = None


def lib():
    """The loaded C library (built by build.py; raises if it is missing)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise ImportError(f"libqgemv.so not built ({path}); run ggml_block_quantized_gb300/build.py")
        L = ctypes.CDLL(path)
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        L.qtype_nbytes.argtypes, L.qtype_nbytes.restype = [i32, i64], i64
        L.qtype_block.argtypes, L.qtype_block.restype = [i32, ctypes.POINTER(i32), ctypes.POINTER(i32)], i32
        L.qtype_act_type.argtypes, L.qtype_act_type.restype = [i32], i32
        L.qg_status_string.argtypes, L.qg_status_string.restype = [i32], ctypes.c_char_p
        L.qg_last_cuda_error.argtypes, L.qg_last_cuda_error.restype = [], ctypes.c_char_p
        L.quantize_act.argtypes, L.quantize_act.restype = [i32, vp, vp, i64, i64, vp], i32
        L.quantize_rows.argtypes, L.quantize_rows.restype = [i32, vp, vp, i64, i64, vp], i32
        L.dequantize_rows.argtypes, L.dequantize_rows.restype = [i32, vp, vp, i64, i64, vp], i32
        L.qgemv_workspace_bytes.argtypes, L.qgemv_workspace_bytes.restype = [i32, i64, i64], sz
        L.qgemv.argtypes, L.qgemv.restype = [i32, vp, vp, vp, i64, i64, i64, vp, sz, vp], i32
        L.qgemv_xq.argtypes, L.qgemv_xq.restype = [i32, vp, vp, vp, i64, i64, i64, vp], i32
        L.qgemv_block_isums.argtypes, L.qgemv_block_isums.restype = [i32, vp, vp, vp, i64, i64, i64, vp], i32
        L.qg_device_error.argtypes, L.qg_device_error.restype = [ctypes.POINTER(ctypes.c_int32)], i32
        L.qgemv_noalloc.argtypes, L.qgemv_noalloc.restype = [i32, vp, vp, vp, i64, i64, i64, vp], i32
        L.qgemv_batched_workspace_bytes.argtypes = [i32, i64, i64, i32]
        L.qgemv_batched_workspace_bytes.restype = sz
        L.qgemv_batched.argtypes = [i32, ctypes.POINTER(GemvMat), i32, i64, i64, vp, sz, vp]
        L.qgemv_batched.restype = i32
        L.qgemv_kernel_info.argtypes = [i32, i64, i64, i64, i32]
        L.qgemv_kernel_info.restype = ctypes.c_char_p
        L.qgemm_kernel_info.argtypes = [i32, i64, i64, i64]
        L.qgemm_kernel_info.restype = ctypes.c_char_p
        L.qg_tune.argtypes, L.qg_tune.restype = [ctypes.c_char_p, i32, ctypes.POINTER(i32)], i32
        L.qgemm_workspace_bytes.argtypes, L.qgemm_workspace_bytes.restype = [i32, i64, i64, i64], sz
        L.qgemm.argtypes, L.qgemm.restype = [i32, vp, vp, vp, i64, i64, i64, vp, sz, vp], i32
        L.qgemm_f16.argtypes, L.qgemm_f16.restype = [vp, vp, vp, i64, i64, i64, vp], i32
        L.qg_selftest_bounded_wait.argtypes, L.qg_selftest_bounded_wait.restype = [vp], i32
        _lib = L
    return _lib


# ------------------------------------------------------------ type table
def qtype_nbytes(t: int, n: int) -> int:
    return int(lib().qtype_nbytes(t, n))


def qtype_block(t: int):
    e, b = ctypes.c_int(), ctypes.c_int()
    st = lib().qtype_block(t, ctypes.byref(e), ctypes.byref(b))
    if st != 0:
        raise QGError(st, "qtype_block")
    return e.value, b.value


def qtype_act_type(t: int) -> int:
    return int(lib().qtype_act_type(t))


# ------------------------------------------------------------ helpers
def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check(st: int, where: str):
    if st != 0:
        raise QGError(st, where)


def _dev_tensor(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _need(t, nbytes, name):
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, needs {nbytes}")


# ------------------------------------------------------------ quantizers
def quantize_act(act_type: int, x, n_vec: int = 1, out=None, stream=None):
    """x: f32 CUDA tensor of n_vec * n_in values -> uint8 blocks of act_type."""
    torch = _torch()
    _dev_tensor(x, torch.float32, "x")
    n_in = x.numel() // n_vec
    nbytes = qtype_nbytes(act_type, n_in)
    if nbytes < 0 or n_in * n_vec != x.numel():
        raise ValueError("x is not n_vec rows of whole blocks")
    if out is None:
        out = torch.empty(nbytes * n_vec, dtype=torch.uint8, device=x.device)
    _dev_tensor(out, torch.uint8, "out")
    _need(out, nbytes * n_vec, "out")
    _check(lib().quantize_act(act_type, _ptr(x), _ptr(out), n_in, n_vec, _stream(stream)), "quantize_act")
    return out


def quantize_rows(t: int, x, n_rows: int, out=None, stream=None):
    """Weights x (f32, n_rows * n_in) -> Q8_0, Q4_0, Q4_1 or Q5_0 blocks."""
    torch = _torch()
    _dev_tensor(x, torch.float32, "x")
    n_in = x.numel() // n_rows
    nbytes = qtype_nbytes(t, n_in)
    if nbytes < 0 or n_in * n_rows != x.numel():
        raise ValueError("x is not n_rows rows of whole blocks")
    if out is None:
        out = torch.empty(nbytes * n_rows, dtype=torch.uint8, device=x.device)
    _dev_tensor(out, torch.uint8, "out")
    _need(out, nbytes * n_rows, "out")
    _check(lib().quantize_rows(t, _ptr(x), _ptr(out), n_rows, n_in, _stream(stream)), "quantize_rows")
    return out


def dequantize_rows(t: int, W, n_rows: int, n_in: int, out=None, stream=None):
    torch = _torch()
    _dev_tensor(W, torch.uint8, "W")
    nbytes = qtype_nbytes(t, n_in)
    if nbytes < 0:
        raise ValueError("n_in is not whole blocks")
    _need(W, nbytes * n_rows, "W")
    if out is None:
        out = torch.empty((n_rows, n_in), dtype=torch.float32, device=W.device)
    _dev_tensor(out, torch.float32, "out")
    _need(out, 4 * n_rows * n_in, "out")
    _check(lib().dequantize_rows(t, _ptr(W), _ptr(out), n_rows, n_in, _stream(stream)), "dequantize_rows")
    return out


# ------------------------------------------------------------ product
def qgemv_workspace_bytes(t: int, n_in: int, n_vec: int = 1) -> int:
    return int(lib().qgemv_workspace_bytes(t, n_in, n_vec))


def qgemv(t: int, W, x, n_out: int, n_in: int, n_vec: int = 1, y=None, workspace=None, stream=None):
    """y[n_vec, n_out] = W . x for W in blocks of type t, x f32 [n_vec, n_in]."""
    torch = _torch()
    _dev_tensor(W, torch.uint8, "W")
    _dev_tensor(x, torch.float32, "x")
    _need(x, 4 * n_vec * n_in, "x")
    if y is None:
        y = torch.empty((n_vec, n_out), dtype=torch.float32, device=x.device)
    _dev_tensor(y, torch.float32, "y")
    _need(y, 4 * n_vec * n_out, "y")
    need = qgemv_workspace_bytes(t, n_in, n_vec)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _dev_tensor(workspace, torch.uint8, "workspace")
    _check(lib().qgemv(t, _ptr(W), _ptr(x), _ptr(y), n_out, n_in, n_vec, _ptr(workspace),
                       workspace.numel(), _stream(stream)), "qgemv")
    return y


def qgemv_xq(t: int, W, xq, n_out: int, n_in: int, n_vec: int = 1, y=None, stream=None):
    """y = W . x with x already quantized (quantize_act of the paired type)."""
    torch = _torch()
    _dev_tensor(W, torch.uint8, "W")
    _dev_tensor(xq, torch.uint8, "xq")
    if y is None:
        y = torch.empty((n_vec, n_out), dtype=torch.float32, device=W.device)
    _dev_tensor(y, torch.float32, "y")
    _need(y, 4 * n_vec * n_out, "y")
    _check(lib().qgemv_xq(t, _ptr(W), _ptr(xq), _ptr(y), n_out, n_in, n_vec, _stream(stream)), "qgemv_xq")
    return y


def qgemv_block_isums(t: int, W, xq, n_out: int, n_in: int, n_vec: int = 1, out=None, stream=None):
    """Exact per-block int32 sums, shape [n_vec, n_out, nb, k] (k = 2 for Q2_K, Q4_K, Q5_K)."""
    torch = _torch()
    _dev_tensor(W, torch.uint8, "W")
    _dev_tensor(xq, torch.uint8, "xq")
    elems, _ = qtype_block(t)
    k = 2 if t in (Q2_K, Q4_K, Q5_K) else 1
    shape = (n_vec, n_out, n_in // elems, k)
    if out is None:
        out = torch.empty(shape, dtype=torch.int32, device=W.device)
    _dev_tensor(out, torch.int32, "out")
    _check(lib().qgemv_block_isums(t, _ptr(W), _ptr(xq), _ptr(out), n_out, n_in, n_vec, _stream(stream)),
           "qgemv_block_isums")
    return out


def qgemv_noalloc(t: int, W, x, n_out: int, n_in: int, n_vec: int = 1, y=None, stream=None):
    """qgemv without a workspace: the library keeps the quantized activations
    in its own fixed device array (256 KiB), for callers that cannot allocate
    device memory where they run the product. Calls that may overlap on the
    GPU share that array and must not run concurrently. Pass y to allocate
    nothing from Python either."""
    torch = _torch()
    _dev_tensor(W, torch.uint8, "W")
    _dev_tensor(x, torch.float32, "x")
    _need(x, 4 * n_vec * n_in, "x")
    if x.device.index != torch.cuda.current_device():
        # the C call plans for and takes the array of the current device
        raise ValueError("qgemv_noalloc: x is not on the current CUDA device")
    if y is None:
        y = torch.empty((n_vec, n_out), dtype=torch.float32, device=x.device)
    _dev_tensor(y, torch.float32, "y")
    _need(y, 4 * n_vec * n_out, "y")
    _check(lib().qgemv_noalloc(t, _ptr(W), _ptr(x), _ptr(y), n_out, n_in, n_vec, _stream(stream)),
           "qgemv_noalloc")
    return y


def qgemv_batched_workspace_bytes(t: int, n_in: int, n_vec: int, n_mats: int) -> int:
    return int(lib().qgemv_batched_workspace_bytes(t, n_in, n_vec, n_mats))


class BatchPlan:
    """A prepared batched call: the matrix table is built once from tensors
    (W uint8, x f32 [n_vec, n_in], y f32 [n_vec, n_out]) and reused; run()
    only issues the C call."""

    def __init__(self, t: int, mats, n_in: int, n_vec: int = 1, workspace=None):
        torch = _torch()
        if not 1 <= len(mats) <= MAX_BATCH:
            raise ValueError(f"1..{MAX_BATCH} matrices per batch")
        self.t, self.n_in, self.n_vec = t, n_in, n_vec
        self.keep = []
        self.table = (GemvMat * len(mats))()
        for i, (W, x, y, n_out) in enumerate(mats):
            _dev_tensor(W, torch.uint8, "W")
            _dev_tensor(x, torch.float32, "x")
            _dev_tensor(y, torch.float32, "y")
            _need(x, 4 * n_vec * n_in, "x")
            _need(y, 4 * n_vec * n_out, "y")
            self.table[i] = GemvMat(W.data_ptr(), x.data_ptr(), y.data_ptr(), n_out)
            self.keep += [W, x, y]
        need = qgemv_batched_workspace_bytes(t, n_in, n_vec, len(mats))
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=mats[0][0].device)
        _dev_tensor(workspace, torch.uint8, "workspace")
        self.workspace = workspace

    def run(self, stream=None):
        _check(lib().qgemv_batched(self.t, self.table, len(self.table), self.n_in, self.n_vec,
                                   _ptr(self.workspace), self.workspace.numel(), _stream(stream)), "qgemv_batched")


def qgemv_batched(t: int, mats, n_in: int, n_vec: int = 1, workspace=None, stream=None):
    """y_i = W_i . x_i for independent matrices [(W, x, y, n_out), ...] of one
    type, row length and vector count, in one launch."""
    BatchPlan(t, mats, n_in, n_vec, workspace).run(stream)


def qgemm_workspace_bytes(t: int, n_out: int, n_in: int, n_tok: int) -> int:
    return lib().qgemm_workspace_bytes(t, n_out, n_in, n_tok)


def qgemm(t: int, W, x, n_out: int, n_in: int, n_tok: int, y=None, workspace=None, stream=None):
    """Prefill product y[n_tok, n_out] = x . W^T for W in blocks of type t and
    f32 x [n_tok, n_in]: W dequantized and x rounded to f16, one tensor-core
    GEMM with f32 accumulation."""
    torch = _torch()
    _dev_tensor(W, torch.uint8, "W")
    _dev_tensor(x, torch.float32, "x")
    _need(x, 4 * n_tok * n_in, "x")
    if y is None:
        y = torch.empty((n_tok, n_out), dtype=torch.float32, device=x.device)
    _dev_tensor(y, torch.float32, "y")
    _need(y, 4 * n_tok * n_out, "y")
    need = qgemm_workspace_bytes(t, n_out, n_in, n_tok)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _dev_tensor(workspace, torch.uint8, "workspace")
    _check(lib().qgemm(t, _ptr(W), _ptr(x), _ptr(y), n_out, n_in, n_tok, _ptr(workspace), workspace.numel(),
                       _stream(stream)), "qgemm")
    return y


def qgemm_f16(A, B, n_out: int, n_tok: int, K: int, y=None, stream=None):
    """Dense GEMM y[n_tok, n_out] = B . A^T for f16 A [n_out, K] and B
    [n_tok, K] (torch.float16 tensors, or uint8 views of f16 bytes), f32 out."""
    torch = _torch()
    for name, t_ in (("A", A), ("B", B)):
        if t_.dtype not in (torch.float16, torch.uint8) or not t_.is_cuda or not t_.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA float16 (or uint8) tensor")
    _need(A, 2 * n_out * K, "A")
    _need(B, 2 * n_tok * K, "B")
    if y is None:
        y = torch.empty((n_tok, n_out), dtype=torch.float32, device=A.device)
    _dev_tensor(y, torch.float32, "y")
    _need(y, 4 * n_tok * n_out, "y")
    _check(lib().qgemm_f16(_ptr(A), _ptr(B), _ptr(y), n_out, n_tok, K, _stream(stream)), "qgemm_f16")
    return y


def kernel_info(t: int, total_rows: int, n_in: int, n_vec: int = 1, n_mats: int = 1) -> str:
    """Which kernel and plan a product would use on the current device."""
    return lib().qgemv_kernel_info(t, total_rows, n_in, n_vec, n_mats).decode()


def gemm_kernel_info(t: int, n_out: int, n_in: int, n_tok: int) -> str:
    """Which GEMM kernel, tiles and launches qgemm would use on the current device."""
    return lib().qgemm_kernel_info(t, n_out, n_in, n_tok).decode()


def tune(name: str, value: int) -> int:
    """Set a tuning knob (an environment variable name such as "QG_TC") for
    the rest of the process; returns its previous value."""
    prev = ctypes.c_int32(0)
    _check(lib().qg_tune(name.encode(), int(value), ctypes.byref(prev)), "qg_tune")
    return prev.value


def selftest_bounded_wait(stream=None):
    """Enqueue the bounded-wait self-test kernel (a wait that runs out after
    about one second); read its code with device_error()."""
    _check(lib().qg_selftest_bounded_wait(_stream(stream)), "qg_selftest_bounded_wait")


def device_error() -> int:
    """Synchronize, read and clear the kernels' bounded-wait error word."""
    v = ctypes.c_int32(0)
    _check(lib().qg_device_error(ctypes.byref(v)), "qg_device_error")
    return v.value
