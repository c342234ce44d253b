"""The prefill product qgemm (W dequantized and x rounded to f16, one tcgen05
tensor-core GEMM with f32 accumulation) against the oracle's float product
(exact dequantized W, f32 x, f64 accumulation), through the C ABI.

The bound comes from the arithmetic: each weight and each activation is
rounded to f16 once (at most 2^-11 relative each, so a product is off by at
most ~2^-10 relative) and the f32 accumulation over n_in terms adds at most
n_in * 2^-24 relative of the sum of |products|:
|y - y_ref| <= (2^-10 + n_in * 2^-24) * sum_i |W[o][i] x[t][i]|.
Shapes cover one output, ragged row and token tiles (not multiples of 128),
k not a multiple of the 64-element k-block, several tiles per CTA, and every
weight type.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import ggml_block_quantized_gb300 as qg  # noqa: E402
import oracle  # noqa: E402
from ggml_block_quantized_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

TYPES = [qg.Q8_0, qg.Q4_0, qg.Q4_1, qg.Q5_0, qg.Q2_K, qg.Q3_K, qg.Q4_K, qg.Q5_K, qg.Q6_K]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def weights(t, n_out, n_in, rng):
    if t in (qg.Q8_0, qg.Q4_0, qg.Q4_1, qg.Q5_0):
        return oracle.quantize(t, synth.f32_normal(rng, n_out * n_in, 0.02))
    return synth.k_blocks(t, n_out * n_in // 256, rng)


def check(t, W, x, y, n_out, n_in, n_tok):
    ref = oracle.gemm_float(t, W, x, n_out, n_in, n_tok)
    wd = np.abs(oracle.dequantize(t, W, n_out * n_in).reshape(n_out, n_in).astype(np.float64))
    mag = np.abs(x.reshape(n_tok, n_in).astype(np.float64)) @ wd.T
    bound = (2.0 ** -10 + n_in * 2.0 ** -24) * mag + 1e-30
    err = np.abs(y.reshape(n_tok, n_out).astype(np.float64) - ref)
    bad = err > bound
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside the bound; worst ratio {(err / bound).max():.3f}"


@pytest.mark.parametrize("t", TYPES)
def test_gemm_small_shapes(t):
    rng = np.random.default_rng(7300 + t)
    blk = 256 if t in (qg.Q2_K, qg.Q3_K, qg.Q4_K, qg.Q5_K, qg.Q6_K) else 32
    for n_out, n_in, n_tok in [(1, blk, 1), (100, 2 * blk, 37), (129, 4 * blk, 130)]:
        W = weights(t, n_out, n_in, rng)
        x = synth.f32_normal(rng, n_tok * n_in)
        y = host(qg.qgemm(t, dev(W), dev(x), n_out, n_in, n_tok))
        check(t, W, x, y, n_out, n_in, n_tok)


@pytest.mark.parametrize("t", [qg.Q4_K, qg.Q6_K, qg.Q8_0])
def test_gemm_several_tiles_per_cta(t):
    """More 128 x 128 tiles than SMs (each CTA walks several, its two
    accumulators alternate), k of 11008 for Q6_K (172 k-blocks, not a
    multiple of 64 for Q8_0's 32-element blocks at 4128)."""
    rng = np.random.default_rng(7400 + t)
    n_out, n_in, n_tok = (4096, 11008, 520) if t == qg.Q6_K else ((3000, 4128, 700) if t == qg.Q8_0 else (4352, 4096, 640))
    W = weights(t, n_out, n_in, rng)
    x = synth.f32_normal(rng, n_tok * n_in)
    y = host(qg.qgemm(t, dev(W), dev(x), n_out, n_in, n_tok))
    # sampled rows and tokens against the oracle (the full product is large)
    rows = np.unique(np.concatenate([rng.integers(0, n_out, 40), [0, n_out - 1, 127, 128]]))
    toks = np.unique(np.concatenate([rng.integers(0, n_tok, 12), [0, n_tok - 1, 127, 128]]))
    Wr = W.reshape(n_out, -1)[rows].reshape(-1)
    xs = x.reshape(n_tok, n_in)[toks].reshape(-1)
    check(t, Wr, xs, y[np.ix_(toks, rows)], len(rows), n_in, len(toks))
    assert qg.device_error() == 0


def test_gemm_wide_token_tiles():
    """Enough tokens that 256-token tiles still give every SM a tile (the
    wide-tile kernel: N = 256 mmas, 512 tensor-memory columns), with a
    ragged last token tile."""
    rng = np.random.default_rng(7600)
    t, n_out, n_in, n_tok = qg.Q4_K, 4096, 2048, 1300
    W = weights(t, n_out, n_in, rng)
    x = synth.f32_normal(rng, n_tok * n_in)
    y = host(qg.qgemm(t, dev(W), dev(x), n_out, n_in, n_tok))
    rows = np.unique(np.concatenate([rng.integers(0, n_out, 40), [0, n_out - 1]]))
    toks = np.unique(np.concatenate([rng.integers(0, n_tok, 12), [0, 255, 256, 1279, 1280, n_tok - 1]]))
    Wr = W.reshape(n_out, -1)[rows].reshape(-1)
    xs = x.reshape(n_tok, n_in)[toks].reshape(-1)
    check(t, Wr, xs, y[np.ix_(toks, rows)], len(rows), n_in, len(toks))
    assert qg.device_error() == 0


@pytest.mark.parametrize("shape", [(1, 256, 1), (100, 512, 37), (129, 1024, 130), (4352, 4096, 640),
                                   (4096, 2048, 1300), (300, 11008, 257), (4096, 4096, 64), (4096, 11008, 200),
                                   (4096, 4096, 384)])
def test_fused_q4_k_equals_the_f16_copy_path(shape):
    """Q4_K blocks expanded to f16 inside the GEMM (into tensor memory, where
    the mma reads its A operand) give the same bits as dequantizing W to an
    f16 copy first (the same f16 values, the same mma order): ragged row
    tiles (rows past the matrix are zeros), ragged token tiles, 128- and
    256-token tiles (both also with a k split), long rows. With the k-blocks split into parts (few tiles)
    only the f32 additions differ: each part's sum, then the parts in order,
    so the two agree within n_in 2^-23 of sum_i |W[o][i] x[t][i]|."""
    n_out, n_in, n_tok = shape
    rng = np.random.default_rng(7700 + n_out + n_tok)
    W = weights(qg.Q4_K, n_out, n_in, rng)
    x = synth.f32_normal(rng, n_tok * n_in)
    Wd, xd = dev(W), dev(x)
    old = qg.tune("QG_FUSED_GEMM", 1)
    old_ks = qg.tune("QG_GEMM_KSPLIT", 1)
    try:
        fused = host(qg.qgemm(qg.Q4_K, Wd, xd, n_out, n_in, n_tok))
        qg.tune("QG_GEMM_KSPLIT", old_ks)
        split = host(qg.qgemm(qg.Q4_K, Wd, xd, n_out, n_in, n_tok))
        qg.tune("QG_FUSED_GEMM", 0)
        copy = host(qg.qgemm(qg.Q4_K, Wd, xd, n_out, n_in, n_tok))
    finally:
        qg.tune("QG_FUSED_GEMM", old)
        qg.tune("QG_GEMM_KSPLIT", old_ks)
    assert np.array_equal(fused.view(np.uint32), copy.view(np.uint32))
    wd = np.abs(oracle.dequantize(qg.Q4_K, W, n_out * n_in).reshape(n_out, n_in).astype(np.float64))
    mag = np.abs(x.reshape(n_tok, n_in).astype(np.float64)) @ wd.T
    err = np.abs(split.astype(np.float64) - copy.astype(np.float64)).reshape(n_tok, n_out)
    assert np.all(err <= n_in * 2.0 ** -23 * mag)
    assert qg.device_error() == 0


def test_gemm_plans():
    """The plan qgemm reports: Q4_K fused with a k split when its tiles are
    few, 256-token tiles when they pay, the f16-copy GEMM for the other types
    and past two fused tiles per SM; a split adds the sum launch."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    info = qg.gemm_kernel_info(qg.Q4_K, 4096, 4096, 64)
    assert info.startswith("gemm_q4k_tmem_kernel<128>") and "launches=3" in info and "ksplit=1 " not in info
    assert qg.gemm_kernel_info(qg.Q4_K, 4096, 4096, 1024).startswith("gemm_q4k_tmem_kernel<256>")
    big = qg.gemm_kernel_info(qg.Q4_K, 4096, 4096, 256 * (2 * sms // 32 + 1))
    assert big.startswith("gemm_f16_tc_kernel<256>") and big.endswith("launches=3")
    assert qg.gemm_kernel_info(qg.Q6_K, 4096, 4096, 64).startswith("gemm_f16_tc_kernel<128>")
    old = qg.tune("QG_GEMM_KSPLIT", 1)
    try:
        assert qg.gemm_kernel_info(qg.Q4_K, 4096, 4096, 64).endswith("ksplit=1 launches=2")
    finally:
        qg.tune("QG_GEMM_KSPLIT", old)


def test_gemm_is_deterministic_and_edges():
    rng = np.random.default_rng(7500)
    t, n_out, n_in, n_tok = qg.Q4_K, 300, 1024, 200
    Wd = dev(weights(t, n_out, n_in, rng))
    xd = dev(synth.f32_normal(rng, n_tok * n_in))
    a = host(qg.qgemm(t, Wd, xd, n_out, n_in, n_tok))
    b = host(qg.qgemm(t, Wd, xd, n_out, n_in, n_tok))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    # n_in == 0: zeros; n_tok == 0 / n_out == 0: nothing to do
    y = torch.full((3, 5), np.nan, device="cuda")
    qg.qgemm(t, torch.zeros(16, dtype=torch.uint8, device="cuda"), torch.zeros(16, device="cuda"), 5, 0, 3, y=y)
    assert np.all(host(y) == 0)
    qg.qgemm(t, Wd, xd, n_out, n_in, 0)
    qg.qgemm(t, Wd, xd, 0, n_in, n_tok)
    assert qg.device_error() == 0
