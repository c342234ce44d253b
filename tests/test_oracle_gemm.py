"""Pins for the oracle's float product (the prefill reference): y = x . W^T
with W dequantized exactly and x in f32, accumulated in f64 ([sipllm] The
fused matmul).

It is tied to the pinned block-quantized product: when x holds exactly the
values of quantized activations, the float product equals the block form
(exact int32 sums times block scales) to f64 rounding. A transposed operand,
a wrong row stride or a dropped block would break that, and a one-hot x
must pick out one dequantized column exactly.
"""
import numpy as np
import pytest

import oracle
from ggml_block_quantized_gb300 import synth

W_TYPES = [oracle.Q8_0, oracle.Q4_0, oracle.Q4_1, oracle.Q5_0, oracle.Q2_K, oracle.Q3_K, oracle.Q4_K,
           oracle.Q5_K, oracle.Q6_K]


def weights(t, n_out, n_in, rng):
    if t in (oracle.Q8_0, oracle.Q4_0, oracle.Q4_1, oracle.Q5_0):
        return oracle.quantize(t, synth.f32_normal(rng, n_out * n_in, 0.02))
    return synth.k_blocks(t, n_out * n_in // 256, rng)


@pytest.mark.parametrize("t", W_TYPES)
def test_float_product_equals_block_form_on_quantized_activations(t):
    rng = np.random.default_rng(7100 + t)
    n_out, n_in, n_tok = 9, 512, 3
    W = weights(t, n_out, n_in, rng)
    at = oracle.act_type(t)
    # activations whose block scale is exactly 2^-7 (every block holds a
    # +-127 * 2^-7), so code * d is exact in f32 for the f32 scale of Q8_K too
    codes = rng.integers(-127, 128, size=n_tok * n_in)
    codes[::32] = 127 * np.where(rng.random(n_tok * n_in // 32) < 0.5, 1, -1)
    x = (codes * 2.0 ** -7).astype(np.float32)
    xq = oracle.quantize(at, x)
    assert np.array_equal(oracle.dequantize(at, xq, n_tok * n_in), x)
    y = oracle.gemm_float(t, W, x, n_out, n_in, n_tok)
    ref = oracle.gemv(t, W, xq, n_out, n_in, n_tok)
    if t == oracle.Q4_1:
        # the block form uses the stored f16 s of Q8_1 for the min term;
        # compare with the brute-force dot of the same exact values instead
        ref = oracle.gemv_dequant(t, W, xq, n_out, n_in, n_tok)
    # the float product uses the f32 dequantized weights (one rounding of at
    # most 2^-24 relative where the exact value needs more than 24 bits, as
    # Q4_K/Q5_K's d*sc*q - dmin*m can); the block form is exact
    wd = np.abs(oracle.dequantize(t, W, n_out * n_in).reshape(n_out, n_in).astype(np.float64))
    bound = 2.0 ** -24 * (np.abs(x.reshape(n_tok, n_in).astype(np.float64)) @ wd.T) + 1e-12 * np.abs(ref)
    assert np.all(np.abs(y - ref) <= bound)


@pytest.mark.parametrize("t", [oracle.Q8_0, oracle.Q4_K, oracle.Q6_K])
def test_one_hot_activation_picks_a_column(t):
    rng = np.random.default_rng(7200 + t)
    n_out, n_in = 5, 256
    W = weights(t, n_out, n_in, rng)
    wd = oracle.dequantize(t, W, n_out * n_in).reshape(n_out, n_in).astype(np.float64)
    for i in (0, 1, 37, 255):
        x = np.zeros((2, n_in), np.float32)
        x[0, i] = 1.0
        x[1, i] = -2.0
        y = oracle.gemm_float(t, W, x, n_out, n_in, 2)
        assert np.array_equal(y[0], wd[:, i])
        assert np.array_equal(y[1], -2.0 * wd[:, i])
