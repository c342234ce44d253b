"""The tcgen05 Q4_K GEMV (three or more vectors; 16-row tiles of whole rows;
weights unpacked into tensor memory with eight blocks of a row side by side
on the mma's M dimension; activations as a swizzled f16 panel; the minimum
term in dp2a) against the oracle, through the C ABI.

The kernel is off by default (the mma.sync kernel measured faster on GB300)
and is switched on here with the QG_TC knob, then exercised on: a ragged last tile (rows past n_out are not copied and never
stored), both row lengths it takes (8 and 16 blocks: one or two block
groups), a batch whose matrices switch inside a CTA's tile range (the panel
is rebuilt), every vector count from 3 to 8, and extreme codes where the
exact block sum exceeds 2^24. The bar is the parity tolerance of the
other product tests, |y - y_oracle| <= 1e-5 |y_oracle| + 1e-6 ||x_v|| ||w_o||.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import ggml_block_quantized_gb300 as qg  # noqa: E402
import oracle  # noqa: E402
from ggml_block_quantized_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

T = qg.Q4_K


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


@pytest.fixture()
def forced():
    prev = qg.tune("QG_TC", 1)
    yield
    qg.tune("QG_TC", prev)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def check_y(W, x, y, n_out, n_in, n_vec):
    xq = oracle.quantize(oracle.act_type(T), x)
    ref = oracle.gemv(T, W, xq, n_out, n_in, n_vec)
    wn = np.linalg.norm(oracle.dequantize(T, W, n_out * n_in).reshape(n_out, n_in).astype(np.float64), axis=1)
    xn = np.linalg.norm(x.reshape(n_vec, n_in).astype(np.float64), axis=1)
    got = y.reshape(n_vec, n_out).astype(np.float64)
    tol = 1e-5 * np.abs(ref) + 1e-6 * xn[:, None] * wn[None, :]
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; worst {np.abs(got - ref).max()}"


SHAPES = [(1, 2048), (15, 2048), (16, 2048), (17, 4096), (300, 4096), (257, 2048), (1000, 4096)]


def test_tc_kernel_is_planned(forced):
    assert qg.kernel_info(T, 300, 2048, 8).startswith("gemv_tc_kernel<Q4_K,tcgen05>")
    assert qg.kernel_info(T, 300, 4096, 3).startswith("gemv_tc_kernel<Q4_K,tcgen05>")
    assert qg.kernel_info(T, 300, 4096, 2).startswith("gemv_kernel<Q4_K,NV=2>")
    assert qg.kernel_info(qg.Q6_K, 300, 4096, 8).startswith("gemv_mma_kernel<")
    # rows the kernel does not take (other than 8 or 16 blocks) go to the
    # mma.sync kernel
    for n_in in (256, 1024, 3072, 5120):
        assert qg.kernel_info(T, 300, n_in, 8).startswith("gemv_mma_kernel<Q4_K"), n_in


def test_tc_fallback_shapes_still_match(forced):
    rng = np.random.default_rng(4605)
    for n_out, n_in in [(70, 256), (40, 1280), (33, 3072), (20, 5120)]:
        W = synth.k_blocks(T, n_out * n_in // 256, rng)
        x = synth.f32_normal(rng, 8 * n_in)
        y = host(qg.qgemv(T, dev(W), dev(x), n_out, n_in, 8))
        check_y(W, x, y, n_out, n_in, 8)


def test_tc_kernel_is_off_by_default():
    """With the knob at its default the 32-layer stack's Q4_K launch takes the
    mma.sync kernel."""
    prev = qg.tune("QG_TC", 0)
    try:
        rows = 32 * (4 * 4096 + 2 * 11008)
        assert qg.kernel_info(T, rows, 4096, 8, 192).startswith("gemv_mma_kernel<Q4_K")
    finally:
        qg.tune("QG_TC", prev)


def test_tc_shapes_all_rows(forced):
    rng = np.random.default_rng(4600)
    for n_out, n_in in SHAPES:
        W = synth.k_blocks(T, n_out * n_in // 256, rng)
        for n_vec in (3, 5, 8):
            x = synth.f32_normal(rng, n_vec * n_in)
            y = host(qg.qgemv(T, dev(W), dev(x), n_out, n_in, n_vec))
            check_y(W, x, y, n_out, n_in, n_vec)
    assert qg.device_error() == 0


def test_tc_every_vector_count(forced):
    rng = np.random.default_rng(4601)
    n_out, n_in = 200, 2048
    W = synth.k_blocks(T, n_out * n_in // 256, rng)
    for n_vec in range(3, 9):
        x = synth.f32_normal(rng, n_vec * n_in)
        y = host(qg.qgemv(T, dev(W), dev(x), n_out, n_in, n_vec))
        check_y(W, x, y, n_out, n_in, n_vec)


def test_tc_extreme_codes(forced):
    """Every code 15, every 6-bit scale and min 63, x constant: the exact
    S_q = 8 * 63 * 32 * 15 * 127 exceeds 2^24, where the f32 accumulator may
    round once (2^-24 relative)."""
    n_out, n_in, n_vec = 130, 2048, 8
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.frombuffer(np.float16(1e-3).tobytes(), np.uint8)
    blk[2:4] = np.frombuffer(np.float16(2e-3).tobytes(), np.uint8)
    blk[4:16] = 0xFF
    blk[16:] = 0xFF
    W = np.tile(blk, n_out * n_in // 256)
    x = np.ones(n_vec * n_in, np.float32)
    x[n_in:] = -2.5
    y = host(qg.qgemv(T, dev(W), dev(x), n_out, n_in, n_vec))
    check_y(W, x, y, n_out, n_in, n_vec)


def test_tc_is_deterministic(forced):
    rng = np.random.default_rng(4602)
    n_out, n_in, n_vec = 1000, 4096, 8
    Wd = dev(synth.k_blocks(T, n_out * n_in // 256, rng))
    xd = dev(synth.f32_normal(rng, n_vec * n_in))
    a = host(qg.qgemv(T, Wd, xd, n_out, n_in, n_vec))
    b = host(qg.qgemv(T, Wd, xd, n_out, n_in, n_vec))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_tc_batched(forced):
    """A batch of ragged matrices in one launch: each matches the oracle and
    equals its single call bit for bit (a tile's sum is formed by one CTA in
    block order, whichever CTA that is)."""
    rng = np.random.default_rng(4603)
    n_in, n_vec = 2048, 8
    n_outs = [1, 15, 16, 17, 700, 64, 3000]
    mats, hw, hx = [], [], []
    for n_out in n_outs:
        W = synth.k_blocks(T, n_out * n_in // 256, rng)
        x = synth.f32_normal(rng, n_vec * n_in)
        hw.append(W)
        hx.append(x)
        mats.append((dev(W), dev(x), torch.full((n_vec, n_out), np.nan, device="cuda"), n_out))
    assert qg.kernel_info(T, sum(n_outs), n_in, n_vec, len(n_outs)).startswith("gemv_tc_kernel")
    qg.qgemv_batched(T, mats, n_in, n_vec)
    torch.cuda.synchronize()
    for (W, x, y, n_out), w_host, x_host in zip(mats, hw, hx):
        got = host(y)
        check_y(w_host, x_host, got, n_out, n_in, n_vec)
        ref = qg.qgemv(T, W, x, n_out, n_in, n_vec)
        assert np.array_equal(got.view(np.uint32), host(ref).view(np.uint32)), n_out
    assert qg.device_error() == 0


def test_tc_graph_replay_equals_eager(forced):
    rng = np.random.default_rng(4604)
    n_out, n_in, n_vec = 640, 4096, 6
    Wd = dev(synth.k_blocks(T, n_out * n_in // 256, rng))
    xd = dev(synth.f32_normal(rng, n_vec * n_in))
    ws = torch.empty(qg.qgemv_workspace_bytes(T, n_in, n_vec), dtype=torch.uint8, device="cuda")
    y_eager = host(qg.qgemv(T, Wd, xd, n_out, n_in, n_vec, workspace=ws))
    y = torch.full((n_vec, n_out), np.nan, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qg.qgemv(T, Wd, xd, n_out, n_in, n_vec, y=y, workspace=ws, stream=s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        qg.qgemv(T, Wd, xd, n_out, n_in, n_vec, y=y, workspace=ws, stream=s)
    y.fill_(np.nan)
    g.replay()
    assert np.array_equal(host(y).view(np.uint32), y_eager.view(np.uint32))
