"""The oracle: a plain, slow, scalar CPU implementation of the ggml/GGUF
block-quantized matrix-vector product, written in C (qoracle.c) and wrapped
here with ctypes and numpy.

TEST INFRASTRUCTURE ONLY. Only tests/, the smoke check in __graft_entry__
and the CPU-baseline leg of bench.py may import this package. The product
library (ggml_block_quantized_gb300) never imports, links or calls it, and
the two share no code.

Every function follows a passage of the reference pages; the citations sit
beside each C function in qoracle.c. The Q6_K element mapping, the Q8_K
activation rule, the s field of Q8_1 and the Q2_K/Q3_K/Q5_K layouts are
readings of the pages (they do not define them) and are "parity unpinned"
against ggml itself: they are pinned only by structural invariants in the
tests.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32, F16, Q4_0, Q4_1, Q5_0, Q8_0, Q8_1 = 0, 1, 2, 3, 6, 8, 9
Q2_K, Q3_K, Q4_K, Q5_K, Q6_K, Q8_K = 10, 11, 12, 13, 14, 15
TYPE_NAMES = {F32: "F32", F16: "F16", Q4_0: "Q4_0", Q4_1: "Q4_1", Q5_0: "Q5_0",
              Q8_0: "Q8_0", Q8_1: "Q8_1", Q2_K: "Q2_K", Q3_K: "Q3_K", Q4_K: "Q4_K",
              Q5_K: "Q5_K", Q6_K: "Q6_K", Q8_K: "Q8_K"}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, i32, u16, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_uint16, ctypes.c_float
        vp = ctypes.c_void_p
        L.or_type_info.argtypes = [i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        L.or_type_info.restype = i32
        L.or_type_nbytes.argtypes = [i32, i64]
        L.or_type_nbytes.restype = i64
        L.or_f16_to_f32.argtypes = [u16]
        L.or_f16_to_f32.restype = f32
        L.or_f32_to_f16.argtypes = [f32]
        L.or_f32_to_f16.restype = u16
        for name in ("or_quantize_q8_0", "or_quantize_q4_0", "or_quantize_q8_k",
                     "or_quantize_q4_1", "or_quantize_q5_0", "or_quantize_q8_1"):
            getattr(L, name).argtypes = [vp, vp, i64]
            getattr(L, name).restype = None
        L.or_dequantize.argtypes = [i32, vp, vp, i64]
        L.or_dequantize.restype = i32
        L.or_act_type.argtypes = [i32]
        L.or_act_type.restype = i32
        L.or_isums_per_block.argtypes = [i32]
        L.or_isums_per_block.restype = i32
        L.or_block_isums.argtypes = [i32, vp, vp, vp, i64, i64, i64]
        L.or_block_isums.restype = i32
        L.or_gemv.argtypes = [i32, vp, vp, vp, i64, i64, i64, i64, i64]
        L.or_gemv.restype = i32
        L.or_gemv_dequant.argtypes = [i32, vp, vp, vp, i64, i64, i64]
        L.or_gemv_dequant.restype = i32
        L.or_host_is_little_endian.argtypes = []
        L.or_host_is_little_endian.restype = i32
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def type_info(t: int):
    e, b = ctypes.c_int(), ctypes.c_int()
    if lib().or_type_info(t, ctypes.byref(e), ctypes.byref(b)) != 0:
        return None
    return e.value, b.value


def type_nbytes(t: int, n: int) -> int:
    return int(lib().or_type_nbytes(t, n))


def act_type(wtype: int) -> int:
    return int(lib().or_act_type(wtype))


def isums_per_block(wtype: int) -> int:
    return int(lib().or_isums_per_block(wtype))


def f16_to_f32(bits: int) -> np.float32:
    return np.float32(lib().or_f16_to_f32(bits & 0xFFFF))


def f32_to_f16(x) -> int:
    return int(lib().or_f32_to_f16(float(np.float32(x))))


def quantize(t: int, x: np.ndarray) -> np.ndarray:
    """Quantize a float32 array (length a whole number of blocks) to the
    byte-exact blocks of type t (Q8_0, Q4_0, Q4_1, Q5_0, Q8_1 or Q8_K).
    Returns uint8 bytes."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    nbytes = type_nbytes(t, x.size)
    if nbytes < 0:
        raise ValueError(f"length {x.size} is not whole blocks of type {t}")
    out = np.zeros(nbytes, dtype=np.uint8)
    fn = {Q8_0: lib().or_quantize_q8_0, Q4_0: lib().or_quantize_q4_0,
          Q4_1: lib().or_quantize_q4_1, Q5_0: lib().or_quantize_q5_0,
          Q8_1: lib().or_quantize_q8_1, Q8_K: lib().or_quantize_q8_k}.get(t)
    if fn is None:
        raise ValueError(f"the oracle has no quantizer for type {t}")
    fn(_ptr(x), _ptr(out), x.size)
    return out


def dequantize(t: int, data: np.ndarray, n: int) -> np.ndarray:
    """Dequantize n elements of type t from raw block bytes to float32."""
    data = np.ascontiguousarray(data, dtype=np.uint8).reshape(-1)
    if type_nbytes(t, n) < 0 or data.size < type_nbytes(t, n):
        raise ValueError("bad length")
    out = np.zeros(n, dtype=np.float32)
    if lib().or_dequantize(t, _ptr(data), _ptr(out), n) != 0:
        raise ValueError(f"cannot dequantize type {t}")
    return out


def block_isums(wtype: int, W: np.ndarray, xq: np.ndarray, n_out: int, n_in: int,
                n_vec: int) -> np.ndarray:
    """Per-(vector, row, block) exact int32 sums; shape [n_vec, n_out, nb, k]
    with k = 2 (S_q, S_m) for Q2_K, Q4_K and Q5_K and 1 otherwise."""
    elems, _ = type_info(wtype)
    nb = n_in // elems
    k = isums_per_block(wtype)
    out = np.zeros((n_vec, n_out, nb, k), dtype=np.int32)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    if lib().or_block_isums(wtype, _ptr(W), _ptr(xq), _ptr(out), n_out, n_in, n_vec) != 0:
        raise ValueError("bad type or shape")
    return out


def gemv(wtype: int, W: np.ndarray, xq: np.ndarray, n_out: int, n_in: int, n_vec: int,
         rows=None, out: np.ndarray = None) -> np.ndarray:
    """y[v, o] accumulated in f64 from exact per-block sums; shape [n_vec, n_out].
    `rows` = (row0, row1) restricts the rows computed (others stay 0)."""
    row0, row1 = (0, n_out) if rows is None else rows
    if out is None:
        out = np.zeros((n_vec, n_out), dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    if lib().or_gemv(wtype, _ptr(W), _ptr(xq), _ptr(out), n_out, n_in, n_vec, row0, row1) != 0:
        raise ValueError("bad type or shape")
    return out


def gemv_dequant(wtype: int, W: np.ndarray, xq: np.ndarray, n_out: int, n_in: int,
                 n_vec: int) -> np.ndarray:
    """Brute-force form: exact dequantized W and activations, plain f64 dot."""
    out = np.zeros((n_vec, n_out), dtype=np.float64)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    if lib().or_gemv_dequant(wtype, _ptr(W), _ptr(xq), _ptr(out), n_out, n_in, n_vec) != 0:
        raise ValueError("bad type or shape")
    return out


def gemm_float(wtype: int, W: np.ndarray, x: np.ndarray, n_out: int, n_in: int, n_tok: int) -> np.ndarray:
    """The float product of [sipllm] "The fused matmul" (matmul_quant):
    each row of W dequantized to f32 (the exact values of dequantize), dotted
    with the f32 activations, here in f64 (numpy's matmul as the dot).
    x is f32 [n_tok, n_in] (not quantized); returns y [n_tok, n_out]."""
    w = dequantize(wtype, W, n_out * n_in).reshape(n_out, n_in).astype(np.float64)
    xs = np.asarray(x, dtype=np.float32).reshape(n_tok, n_in).astype(np.float64)
    return xs @ w.T


def host_is_little_endian() -> bool:
    return bool(lib().or_host_is_little_endian())
