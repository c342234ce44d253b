"""Parity of the CUDA path (through the C ABI) with the oracle.

Bit-exact: activation blocks, weight blocks, dequantized f32 values and the
per-block int32 sums. Tolerance on y (the float step per block is not fixed
by the pages): |y - y_oracle| <= 1e-5 |y_oracle| + 1e-6 ||x_v|| ||w_o||, with
y_oracle accumulated in f64 and w_o the dequantized row.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import ggml_block_quantized_gb300 as qg  # noqa: E402
import oracle  # noqa: E402
from ggml_block_quantized_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

REL, ABS = 1e-5, 1e-6
WTYPES = [qg.Q8_0, qg.Q4_0, qg.Q4_1, qg.Q5_0, qg.Q2_K, qg.Q3_K, qg.Q4_K, qg.Q5_K, qg.Q6_K]
LEGACY = (qg.Q8_0, qg.Q4_0, qg.Q4_1, qg.Q5_0)  # 32-element blocks


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert qg.device_error() == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def weights(t, n_out, n_in, rng):
    """Host weight blocks: 32-element types from the oracle's quantizer (Q4_1
    from off-centre values), K types random."""
    if t in LEGACY:
        w = synth.f32_normal(rng, n_out * n_in, 0.02)
        if t == qg.Q4_1:
            w += np.float32(0.01)
        return oracle.quantize(t, w)
    return synth.k_blocks(t, n_out * n_in // 256, rng)


def row_norms(t, W, rows, n_in):
    rb = oracle.type_nbytes(t, n_in)
    return np.array([np.linalg.norm(oracle.dequantize(t, W[r * rb:(r + 1) * rb], n_in).astype(np.float64))
                     for r in rows])


def check_y(t, W, x, y_gpu, n_out, n_in, n_vec, rows=None):
    """y_gpu [n_vec, n_out] against the oracle on `rows` (all rows if None)."""
    at = oracle.act_type(t)
    xq = oracle.quantize(at, x)
    rows = list(range(n_out)) if rows is None else sorted(set(rows))
    y_ref = np.zeros((n_vec, n_out))
    if len(rows) == n_out:
        y_ref = oracle.gemv(t, W, xq, n_out, n_in, n_vec)
    else:
        for r in rows:
            oracle.gemv(t, W, xq, n_out, n_in, n_vec, rows=(r, r + 1), out=y_ref)
    wn = row_norms(t, W, rows, n_in)
    xn = np.linalg.norm(x.reshape(n_vec, n_in).astype(np.float64), axis=1)
    got = y_gpu[:, rows].astype(np.float64)
    ref = y_ref[:, rows]
    tol = REL * np.abs(ref) + ABS * xn[:, None] * wn[None, :]
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (f"type {t}: {bad.sum()} of {bad.size} outside tolerance; worst "
                           f"{np.max(np.abs(got - ref) / np.maximum(tol, 1e-30)):.3g} x tol")


def sample_rows(n_out, rng, k=48):
    base = [0, 1, n_out // 2, n_out - 2, n_out - 1]
    return [r for r in base if 0 <= r < n_out] + list(rng.choice(n_out, size=min(k, n_out), replace=False))


# ----------------------------------------------------------- quantizers
SPECIAL = {
    "zeros": lambda n: np.zeros(n, np.float32),
    "neg_zero": lambda n: np.full(n, -0.0, np.float32),
    "ties": lambda n: np.tile(np.concatenate([[127.0], np.arange(31) - 15 + 0.5]).astype(np.float32), n // 32),
    "tiny": lambda n: (np.float32(3e-6) * np.arange(n, dtype=np.float32) / np.float32(31)),
    "subnormal_d": lambda n: (np.float32(8e-6) * (np.arange(n) % 32).astype(np.float32) / np.float32(31)),
    "huge": lambda n: (np.float32(9e6) * (np.arange(n) % 32).astype(np.float32) / np.float32(31)),
    "equal_magnitudes": lambda n: np.tile(np.array([1.0, -1.0] * 16, np.float32), n // 32),
}


@pytest.mark.parametrize("at", [qg.Q8_0, qg.Q8_1, qg.Q8_K])
def test_quantize_act_bit_exact(at):
    rng = np.random.default_rng(100 + at)
    for n_in, n_vec in ((256, 1), (512, 3), (4096, 8), (11008, 2), (256 * 40, 5)):
        x = synth.f32_normal(rng, n_in * n_vec) * np.float32(rng.uniform(0.01, 100))
        got = host(qg.quantize_act(at, dev(x), n_vec))
        assert np.array_equal(got, oracle.quantize(at, x)), (n_in, n_vec)
    for name, fn in SPECIAL.items():
        x = fn(512)
        assert np.array_equal(host(qg.quantize_act(at, dev(x), 1)), oracle.quantize(at, x)), name
    # NaN and inf elements (candle's special-value rows): NaN -> code 0, inf -> inf scale
    for bad in (np.nan, np.inf, -np.inf):
        x = synth.f32_normal(rng, 512)
        x[[3, 300]] = bad
        assert np.array_equal(host(qg.quantize_act(at, dev(x), 1)), oracle.quantize(at, x)), bad


@pytest.mark.parametrize("t", LEGACY)
def test_quantize_rows_bit_exact(t):
    rng = np.random.default_rng(200 + t)
    # the lesson's fixed block with the 9.5 outlier, then random rows at the
    # 4096 x 4096 workload size, then blocks with repeated extreme magnitudes
    i = np.arange(64)
    x = (((i * 7919) % 1001) - 500).astype(np.float32) / np.float32(337)
    x[40] = np.float32(9.5)
    assert np.array_equal(host(qg.quantize_rows(t, dev(x), 1)), oracle.quantize(t, x))
    w = synth.single_matrix("q4_0_4096")["w_f32"]
    assert np.array_equal(host(qg.quantize_rows(t, dev(w), 4096)), oracle.quantize(t, w))
    for name, fn in SPECIAL.items():
        x = fn(1024)
        assert np.array_equal(host(qg.quantize_rows(t, dev(x), 4)), oracle.quantize(t, x)), name
    # many exact halves: x * id + 8.5 lands on integers for a power-of-two max
    x = (rng.integers(-16, 16, 32 * 64) / 2.0).astype(np.float32)
    x[::32] = -8.0
    assert np.array_equal(host(qg.quantize_rows(t, dev(x), 64)), oracle.quantize(t, x))
    if t in (qg.Q4_1, qg.Q5_0):
        # off-centre blocks (Q4_1's min at work)
        x = synth.f32_normal(rng, 32 * 64) + np.float32(3)
        assert np.array_equal(host(qg.quantize_rows(t, dev(x), 64)), oracle.quantize(t, x))
    # NaN / inf elements, which both sides define (NaN is skipped by the max
    # or min/max and gets code 0; the cast is Java's)
    for bad in (np.nan, np.inf, -np.inf):
        x = synth.f32_normal(rng, 32 * 8)
        x[[3, 100, 101]] = bad
        assert np.array_equal(host(qg.quantize_rows(t, dev(x), 8)), oracle.quantize(t, x)), bad
    # subnormal blocks: for the smallest maxima d is tiny or 0 and 1/d may
    # overflow to infinity (codes from +-inf and NaN through the Java cast)
    k = np.arange(32 * 40)
    x = (rng.integers(-12, 13, k.size) * np.exp2(-149.0 + (k // 32) % 20)).astype(np.float32)
    x[::97] = np.nan
    assert np.array_equal(host(qg.quantize_rows(t, dev(x), 40)), oracle.quantize(t, x))


# ------------------------------------------------------------- dequantize
@pytest.mark.parametrize("t", [qg.Q8_0, qg.Q4_0, qg.Q4_1, qg.Q5_0, qg.Q8_1, qg.Q2_K, qg.Q3_K, qg.Q4_K,
                               qg.Q5_K, qg.Q6_K, qg.Q8_K])
def test_dequantize_bit_exact(t):
    rng = np.random.default_rng(300 + t)
    elems, nbytes = oracle.type_info(t)
    for n_rows, n_in in ((1, elems), (3, 5 * elems), (37, 4096), (129, 11008 if elems == 256 else 1024)):
        if t in synth.K_TYPES:
            W = synth.k_blocks(t, n_rows * n_in // 256, rng)
        else:
            W = synth.random_bytes(rng, n_rows * n_in // elems * nbytes).reshape(-1, nbytes)
            if t == qg.Q8_K:
                W[:, 0:4] = np.abs(rng.standard_normal((W.shape[0], 1))).astype(np.float32).view(np.uint8)
            else:
                W[:, 0:2] = rng.standard_normal((W.shape[0], 1)).astype(np.float16).view(np.uint8)
            if t == qg.Q4_1:  # the min: finite f16 (random bytes could be NaN)
                W[:, 2:4] = rng.standard_normal((W.shape[0], 1)).astype(np.float16).view(np.uint8)
            W = W.reshape(-1)
        got = host(qg.dequantize_rows(t, dev(W), n_rows, n_in))
        want = oracle.dequantize(t, W, n_rows * n_in).reshape(n_rows, n_in)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), (n_rows, n_in)


def test_dequantize_q4_k_workload_size():
    m = synth.single_matrix("q4_k_4096")
    got = host(qg.dequantize_rows(qg.Q4_K, dev(m["w_blocks"]), 4096, 4096))
    want = oracle.dequantize(qg.Q4_K, m["w_blocks"], 4096 * 4096).reshape(4096, 4096)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


# ------------------------------------------------------- exact block sums
SHAPES = {  # (n_out, n_in): one block; ragged rows; several stages and ring wrap-around
    qg.Q8_0: [(1, 32), (37, 96), (300, 1024), (5000, 4096)],
    qg.Q4_0: [(1, 32), (37, 96), (300, 1024), (5000, 4096)],
    qg.Q4_1: [(1, 32), (37, 96), (300, 1024), (5000, 4096)],
    qg.Q5_0: [(1, 32), (37, 96), (300, 1024), (5000, 4096)],
    qg.Q4_K: [(1, 256), (37, 768), (300, 11008), (5000, 4096)],
    qg.Q2_K: [(1, 256), (37, 768), (300, 11008), (5000, 4096)],
    qg.Q3_K: [(1, 256), (37, 768), (300, 11008), (3000, 4096)],
    qg.Q5_K: [(1, 256), (37, 768), (300, 11008), (5000, 4096)],
    qg.Q6_K: [(1, 256), (37, 768), (300, 11008), (3000, 4096)],
}


@pytest.mark.parametrize("t", WTYPES)
def test_block_isums_bit_exact(t):
    rng = np.random.default_rng(400 + t)
    at = oracle.act_type(t)
    for n_out, n_in in SHAPES[t]:
        W = weights(t, n_out, n_in, rng)
        Wd = dev(W)
        for n_vec in ((1, 2, 5, 8) if n_out * n_in <= 300 * 11008 else (1, 8)):
            x = synth.f32_normal(rng, n_vec * n_in)
            xq = oracle.quantize(at, x)
            got = host(qg.qgemv_block_isums(t, Wd, dev(xq), n_out, n_in, n_vec))
            want = oracle.block_isums(t, W, xq, n_out, n_in, n_vec)
            assert np.array_equal(got, want), (n_out, n_in, n_vec)


@pytest.mark.parametrize("t", [qg.Q4_1, qg.Q5_0])
def test_every_code_and_bit_pattern(t):
    """Blocks of uniform random bytes (every nibble, every fifth bit, d of
    either sign, Q4_1's min of either sign): exact sums bit for bit and y
    within tolerance, all rows."""
    rng = np.random.default_rng(450 + t)
    at = oracle.act_type(t)
    for n_out, n_in in ((5, 32), (67, 1024), (1000, 4096)):
        W = synth.legacy_blocks(t, n_out * n_in // 32, rng)
        for n_vec in (1, 2, 3, 8):
            x = synth.f32_normal(rng, n_vec * n_in)
            xq = oracle.quantize(at, x)
            got = host(qg.qgemv_block_isums(t, dev(W), dev(xq), n_out, n_in, n_vec))
            assert np.array_equal(got, oracle.block_isums(t, W, xq, n_out, n_in, n_vec)), (n_out, n_in, n_vec)
            y = host(qg.qgemv(t, dev(W), dev(x), n_out, n_in, n_vec))
            check_y(t, W, x, y, n_out, n_in, n_vec)


def test_block_isums_at_extreme_codes():
    # Q6_K scales at -128 and every q = 0 (-32) against activations of -127:
    # the largest magnitudes the int32 sums see
    rng = np.random.default_rng(5)
    n_out, n_in = 9, 512
    W = synth.k_blocks(qg.Q6_K, n_out * 2, rng).reshape(-1, 210)
    W[:, :192] = 0
    W[:, 192:208] = np.uint8(0x80)
    W = W.reshape(-1)
    x = np.full(n_in, -1.0, np.float32)
    xq = oracle.quantize(qg.Q8_K, x)
    got = host(qg.qgemv_block_isums(qg.Q6_K, dev(W), dev(xq), n_out, n_in, 1))
    assert np.array_equal(got, oracle.block_isums(qg.Q6_K, W, xq, n_out, n_in, 1))
    assert got[0, 0, 0, 0] == 16 * (-128) * 16 * (-32) * (-127)
    # Q4_K with every scale/min byte 0xFF and every nibble 15
    W = synth.k_blocks(qg.Q4_K, n_out * 2, rng).reshape(-1, 144)
    W[:, 4:] = 0xFF
    W = W.reshape(-1)
    xq = oracle.quantize(qg.Q8_K, np.full(n_in, 1.0, np.float32))
    got = host(qg.qgemv_block_isums(qg.Q4_K, dev(W), dev(xq), n_out, n_in, 1))
    assert np.array_equal(got, oracle.block_isums(qg.Q4_K, W, xq, n_out, n_in, 1))


# ------------------------------------------------------------ y tolerance
@pytest.mark.parametrize("t", WTYPES)
def test_qgemv_small_shapes_all_rows(t):
    rng = np.random.default_rng(500 + t)
    for n_out, n_in in SHAPES[t][:3]:
        W = weights(t, n_out, n_in, rng)
        for n_vec in (1, 3, 8):
            x = synth.f32_normal(rng, n_vec * n_in)
            y = host(qg.qgemv(t, dev(W), dev(x), n_out, n_in, n_vec))
            check_y(t, W, x, y, n_out, n_in, n_vec)


@pytest.mark.parametrize("name", ["q8_0_256x1024", "q4_0_4096", "q4_k_4096", "q6_k_32000", "q4_1_32000",
                                  "q5_0_32000", "q2_k_32000", "q3_k_32000", "q5_k_32000"])
@pytest.mark.parametrize("n_vec", [1, 8])
def test_qgemv_workloads_full_size(name, n_vec):
    m = synth.single_matrix(name, n_vec=n_vec)
    t, n_out, n_in = m["type"], m["n_out"], m["n_in"]
    rng = np.random.default_rng(600)
    if "w_f32" in m:
        Wd = qg.quantize_rows(t, dev(m["w_f32"]), n_out)
        W = oracle.quantize(t, m["w_f32"])
        assert np.array_equal(host(Wd), W)
    else:
        W = m["w_blocks"]
        Wd = dev(W)
    y = host(qg.qgemv(t, Wd, dev(m["x"]), n_out, n_in, n_vec))
    rows = None if n_out * n_in * n_vec <= 4096 * 4096 else sample_rows(n_out, rng, 96)
    check_y(t, W, m["x"], y, n_out, n_in, n_vec, rows)


@pytest.mark.parametrize("m", range(len(synth.LAYER_MATRICES)))
@pytest.mark.parametrize("n_vec", [1, 8])
def test_qgemv_layer_stack_matrices(m, n_vec):
    mat = synth.layer_matrix(0, m, n_vec)
    t, n_out, n_in = mat["type"], mat["n_out"], mat["n_in"]
    y = host(qg.qgemv(t, dev(mat["w_blocks"]), dev(mat["x"]), n_out, n_in, n_vec))
    check_y(t, mat["w_blocks"], mat["x"], y, n_out, n_in, n_vec,
            sample_rows(n_out, np.random.default_rng(m), 64))


@pytest.mark.parametrize("t", WTYPES)
def test_qgemv_xq_equals_qgemv(t):
    """x quantized inside the GEMV's prologue (each warp quantizing two
    blocks at a time, with a ragged last pair) gives the same bits as the
    separate quantization launch: on normal x and on the quantizer's special
    patterns, at block counts that leave warps with one block or none."""
    rng = np.random.default_rng(8)
    cases = [(333, 1024, 2), (70, 1280, 3), (19, 256, 8), (40, 2560, 1)]
    for n_out, n_in, n_vec in cases:
        W = dev(weights(t, n_out, n_in, rng))
        xs = [synth.f32_normal(rng, n_vec * n_in)] + [f(n_vec * n_in) for f in SPECIAL.values()]
        for xh in xs:
            x = dev(xh)
            y1 = qg.qgemv(t, W, x, n_out, n_in, n_vec)
            y2 = qg.qgemv_xq(t, W, qg.quantize_act(oracle.act_type(t), x, n_vec), n_out, n_in, n_vec)
            assert torch.equal(y1.view(torch.int32), y2.view(torch.int32)), (n_out, n_in, n_vec)


def test_fused_limit_knob_keeps_results():
    """QG_FUSED_MAX_MIB moves a single call between in-kernel quantization and
    the separate launch; the product is the same bits either way."""
    t, n_out, n_in = qg.Q4_K, 3000, 4096
    rng = np.random.default_rng(81)
    W = dev(weights(t, n_out, n_in, rng))
    x = dev(synth.f32_normal(rng, n_in))
    assert "fused-quantize" in qg.kernel_info(t, n_out, n_in, 1)
    y1 = qg.qgemv(t, W, x, n_out, n_in, 1)
    prev = qg.tune("QG_FUSED_MAX_MIB", 0)
    try:
        assert "fused-quantize" not in qg.kernel_info(t, n_out, n_in, 1)
        y2 = qg.qgemv(t, W, x, n_out, n_in, 1)
    finally:
        qg.tune("QG_FUSED_MAX_MIB", prev)
    assert torch.equal(y1, y2)


# ---------------------------------------------------------------- edges
def test_edges_empty_and_tails():
    rng = np.random.default_rng(9)
    # n_in = 0: the empty sum
    y = torch.full((2, 5), 7.0, device="cuda")
    qg.qgemv(qg.Q4_K, torch.zeros(16, dtype=torch.uint8, device="cuda"),
             torch.zeros(16, dtype=torch.float32, device="cuda"), 5, 0, 2, y=y)
    assert host(y).tolist() == [[0.0] * 5] * 2
    # n_out = 0: nothing to do
    qg.qgemv(qg.Q4_K, torch.zeros(16, dtype=torch.uint8, device="cuda"),
             dev(synth.f32_normal(rng, 256)), 0, 256, 1, y=torch.zeros(4, device="cuda"))
    # W byte lengths that end inside a 16-byte chunk (34, 630, 18*3 bytes)
    for t, n_out, n_in in ((qg.Q8_0, 1, 32), (qg.Q6_K, 3, 256), (qg.Q4_0, 3, 32), (qg.Q6_K, 7, 2304),
                           (qg.Q4_1, 1, 32), (qg.Q5_0, 3, 32), (qg.Q5_0, 5, 96), (qg.Q3_K, 1, 256),
                           (qg.Q3_K, 3, 768), (qg.Q2_K, 1, 256)):
        W = weights(t, n_out, n_in, rng)
        assert W.size % 16 != 0
        for n_vec in (1, 4):
            x = synth.f32_normal(rng, n_vec * n_in)
            y = host(qg.qgemv(t, dev(W), dev(x), n_out, n_in, n_vec))
            check_y(t, W, x, y, n_out, n_in, n_vec)


def test_shape_limit_is_reported_not_launched():
    # activations of 8 vectors x 65536 Q8_0 values cannot sit in one SM's shared memory
    W = torch.zeros(16, dtype=torch.uint8, device="cuda")
    x = torch.zeros(8 * 65536 * 2, dtype=torch.float32, device="cuda")
    with pytest.raises(qg.QGError) as e:
        qg.qgemv(qg.Q8_0, W, x, 1, 65536 * 2, 8)
    assert e.value.status == -2


# ----------------------------------------------- ordering, chaining, graphs
def test_chained_calls_keep_stream_order():
    """y of one call is x of the next; with programmatic dependent launch the
    next call may start early, so compare with calls separated by syncs."""
    rng = np.random.default_rng(10)
    n = 4096
    Ws = [dev(synth.k_blocks(qg.Q4_K, n * n // 256, rng)) for _ in range(6)]
    x0 = dev(synth.f32_normal(rng, n))

    def run(sync):
        x = x0
        ys = []
        for W in Ws:
            y = qg.qgemv(qg.Q4_K, W, x, n, n, 1)
            y = y / (y.abs().max() + 1e-30)  # keep values O(1); an ordinary kernel in between
            if sync:
                torch.cuda.synchronize()
            ys.append(y)
            x = y.reshape(-1)
        return torch.stack(ys)

    a = run(False)
    b = run(True)
    assert torch.equal(a, b)

    # back-to-back qgemv calls with nothing in between (x fixed, y reused as
    # the next x without a separate kernel)
    def run2(sync):
        x = x0
        outs = []
        for W in Ws:
            y = qg.qgemv(qg.Q4_K, W, x, n, n, 1)
            if sync:
                torch.cuda.synchronize()
            outs.append(y)
            x = y.reshape(-1)
        return torch.stack(outs)

    assert torch.equal(run2(False), run2(True))


@pytest.mark.parametrize("t", LEGACY)
def test_quantize_rows_then_product_without_sync(t):
    """quantize_rows writes W and the product that streams W is enqueued
    directly behind it, with no sync in between (the product starts reading
    W before the kernel ahead of it has finished): it must read the new
    weights, not the bytes the buffer held before. One matrix of 32000 x 4096
    with one vector (x quantized in the product's prologue) and with eight
    (a separate activation launch in between), then a batched call over
    three freshly written matrices."""
    rng = np.random.default_rng(910 + t)
    n_out, n_in = 32000, 4096
    w = synth.f32_normal(rng, n_out * n_in, 0.02)
    W_host = oracle.quantize(t, w)
    wd = dev(w)
    for n_vec in (1, 8):
        x = synth.f32_normal(rng, n_vec * n_in)
        xd = dev(x)
        Wd = torch.full((W_host.size,), 0x7B, dtype=torch.uint8, device="cuda")  # stale bytes
        torch.cuda.synchronize()
        qg.quantize_rows(t, wd, n_out, out=Wd)
        y = qg.qgemv(t, Wd, xd, n_out, n_in, n_vec)
        torch.cuda.synchronize()
        assert torch.equal(y, qg.qgemv(t, Wd, xd, n_out, n_in, n_vec)), n_vec
        assert np.array_equal(host(Wd), W_host)
        check_y(t, W_host, x, host(y), n_out, n_in, n_vec, sample_rows(n_out, rng, 64))
    # batched: three matrices, each written by its own quantize_rows call
    n_outs = [4096, 11008, 4096]
    ws = [synth.f32_normal(rng, n * n_in, 0.02) for n in n_outs]
    xs = [dev(synth.f32_normal(rng, n_in)) for _ in n_outs]
    Wds = [torch.full((oracle.type_nbytes(t, n_in) * n,), 0x7B, dtype=torch.uint8, device="cuda")
           for n in n_outs]
    ys = [torch.full((1, n), np.nan, device="cuda") for n in n_outs]
    wds = [dev(a) for a in ws]
    torch.cuda.synchronize()
    for wdm, Wd, n in zip(wds, Wds, n_outs):
        qg.quantize_rows(t, wdm, n, out=Wd)
    qg.qgemv_batched(t, list(zip(Wds, xs, ys, n_outs)), n_in, 1)
    torch.cuda.synchronize()
    for Wd, xd, y, n in zip(Wds, xs, ys, n_outs):
        assert torch.equal(y, qg.qgemv(t, Wd, xd, n, n_in, 1))


def test_graph_capture_replay_matches_eager():
    rng = np.random.default_rng(11)
    mats = [synth.layer_matrix(1, m, 1) for m in range(len(synth.LAYER_MATRICES))]
    Ws = [dev(m["w_blocks"]) for m in mats]
    xs = [dev(m["x"]) for m in mats]
    ys = [torch.empty(m["n_out"], device="cuda") for m in mats]
    wss = [torch.empty(qg.qgemv_workspace_bytes(m["type"], m["n_in"], 1), dtype=torch.uint8, device="cuda")
           for m in mats]
    s = torch.cuda.Stream()

    def step():
        for m, W, x, y, ws in zip(mats, Ws, xs, ys, wss):
            qg.qgemv(m["type"], W, x, m["n_out"], m["n_in"], 1, y=y, workspace=ws, stream=s)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    eager = [y.clone() for y in ys]
    for y in ys:
        y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, ys):
        assert torch.equal(a, b)
    del rng


# ------------------------------------------------------------- batched calls
def batch_inputs(t, n_outs, n_in, n_vec, rng):
    mats, host_w, host_x = [], [], []
    for n_out in n_outs:
        W = weights(t, n_out, n_in, rng) if n_out else np.zeros(16, np.uint8)
        x = synth.f32_normal(rng, n_vec * n_in)
        mats.append((dev(W), dev(x), torch.full((n_vec, max(n_out, 1)), np.nan, device="cuda"), n_out))
        host_w.append(W)
        host_x.append(x)
    return mats, host_w, host_x


@pytest.mark.parametrize("t", WTYPES)
@pytest.mark.parametrize("n_vec", [1, 3, 8])
def test_batched_equals_single_calls(t, n_vec):
    """One launch over several independent matrices gives, per matrix, the
    same bits as one qgemv call each (n_vec 8 takes the path that quantizes
    all activations into the workspace first)."""
    rng = np.random.default_rng(900 + t + n_vec)
    n_in = 4096 if n_vec == 8 else (1024 if t in LEGACY else 2048)
    n_outs = [300, 0, 1, 2000, 77, 513]
    mats, host_w, host_x = batch_inputs(t, n_outs, n_in, n_vec, rng)
    qg.qgemv_batched(t, mats, n_in, n_vec)
    for (W, x, y, n_out), Wh, xh in zip(mats, host_w, host_x):
        if n_out == 0:
            continue
        ref = qg.qgemv(t, W, x, n_out, n_in, n_vec)
        assert torch.equal(y[:, :n_out], ref), n_out
    # and against the oracle on one matrix
    W, x, y, n_out = mats[3]
    check_y(t, host_w[3], host_x[3], host(y), n_out, n_in, n_vec, sample_rows(n_out, rng, 64))


def test_batched_layer_and_many_small_matrices():
    rng = np.random.default_rng(901)
    # the Q4_K matrices of one decoder layer
    mats = []
    ref = []
    for m in range(6):
        mat = synth.layer_matrix(2, m, 1)
        W, x = dev(mat["w_blocks"]), dev(mat["x"])
        y = torch.empty((1, mat["n_out"]), device="cuda")
        mats.append((W, x, y, mat["n_out"]))
        ref.append(qg.qgemv(qg.Q4_K, W, x, mat["n_out"], 4096, 1))
    qg.qgemv_batched(qg.Q4_K, mats, 4096, 1)
    for (W, x, y, n), r in zip(mats, ref):
        assert torch.equal(y, r)
    # 256 tiny matrices: every CTA crosses many matrix boundaries
    mats, host_w, host_x = batch_inputs(qg.Q6_K, [int(v) for v in rng.integers(1, 7, 256)], 512, 2, rng)
    qg.qgemv_batched(qg.Q6_K, mats, 512, 2)
    for (W, x, y, n_out), Wh, xh in zip(mats, host_w, host_x):
        check_y(qg.Q6_K, Wh, xh, host(y)[:, :n_out], n_out, 512, 2)


def test_batched_graph_capture():
    rng = np.random.default_rng(902)
    mats, _, _ = batch_inputs(qg.Q4_K, [4096, 4096, 11008], 4096, 1, rng)
    plan = qg.BatchPlan(qg.Q4_K, mats, 4096, 1)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        plan.run(s)
    torch.cuda.synchronize()
    eager = [y.clone() for (_, _, y, _) in mats]
    for (_, _, y, _) in mats:
        y.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.run(s)
    g.replay()
    torch.cuda.synchronize()
    for a, (_, _, y, _) in zip(eager, mats):
        assert torch.equal(a, y)
