"""The tensor-core GEMV (the K-quant weight types, and Q4_0 / Q4_1 / Q5_0 /
Q8_0 taken eight blocks at a time; three or more vectors) against the oracle,
through the C ABI. The 32-element types take that kernel by default only for
matrices of enough elements; here QG_MMA_GROUP_MELEM = 0 routes every
product of whole 8-block groups to it.

The kernel tiles 16 rows and streams each tile as chunks of whole blocks, so
the shapes here cover a ragged last tile (n_out not a multiple of 16), rows of
one block, chunks that do not divide the row (Q6_K with 43 blocks per row),
W whose end is not 16-byte aligned (Q6_K rows of 9030 bytes: the last bytes
come through plain loads), both activation-panel formats (f16 when it fits in
shared memory, biased int8 for long rows) and every vector count from 3 to 8.
The bar is the parity tolerance of the other product tests,
|y - y_oracle| <= 1e-5 |y_oracle| + 1e-6 ||x_v|| ||w_o||.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import ggml_block_quantized_gb300 as qg  # noqa: E402
import oracle  # noqa: E402
from ggml_block_quantized_gb300 import synth  # noqa: E402

pytestmark = pytest.mark.gpu

GROUPED = (qg.Q4_0, qg.Q4_1, qg.Q5_0, qg.Q8_0)  # 32-element blocks, eight to a panel block
K_TYPES = [qg.Q2_K, qg.Q3_K, qg.Q4_K, qg.Q5_K, qg.Q6_K, *GROUPED]
_GROUP_MELEM = {}  # the knob's value outside this module


def wblocks(t, n_out, n_in, rng):
    """Random weight blocks: K-quant super-blocks, or 32-element blocks of
    uniform bytes with an f16 d of either sign (every code pattern)."""
    if t in GROUPED:
        return synth.legacy_blocks(t, n_out * n_in // 32, rng)
    return synth.k_blocks(t, n_out * n_in // 256, rng)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    _GROUP_MELEM["v"] = qg.tune("QG_MMA_GROUP_MELEM", 0)
    yield
    qg.tune("QG_MMA_GROUP_MELEM", _GROUP_MELEM["v"])


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def check_y(t, W, x, y, n_out, n_in, n_vec, rows=None):
    xq = oracle.quantize(oracle.act_type(t), x)
    if rows is None:
        ref = oracle.gemv(t, W, xq, n_out, n_in, n_vec)
        rows = np.arange(n_out)
    else:
        ref = np.zeros((n_vec, n_out))
        for r in rows:
            oracle.gemv(t, W, xq, n_out, n_in, n_vec, rows=(int(r), int(r) + 1), out=ref)
    wn = np.linalg.norm(oracle.dequantize(t, W, n_out * n_in).reshape(n_out, n_in).astype(np.float64), axis=1)
    xn = np.linalg.norm(x.reshape(n_vec, n_in).astype(np.float64), axis=1)
    got = y.reshape(n_vec, n_out)[:, rows].astype(np.float64)
    want = ref[:, rows]
    tol = 1e-5 * np.abs(want) + 1e-6 * xn[:, None] * wn[None, rows]
    bad = np.abs(got - want) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance; worst {np.abs(got - want).max()}"


# (n_out, n_in): ragged tiles, one-block rows, multi-chunk rows, unaligned W end
SHAPES = [(33, 256), (40, 768), (100, 2816), (16, 4096), (257, 4096), (17, 11008), (31, 11008)]


@pytest.mark.parametrize("t", K_TYPES)
def test_mma_shapes_all_rows(t):
    rng = np.random.default_rng(4100 + t)
    for n_out, n_in in SHAPES:
        W = wblocks(t, n_out, n_in, rng)
        for n_vec in (3, 5, 8):
            x = synth.f32_normal(rng, n_vec * n_in)
            y = host(qg.qgemv(t, dev(W), dev(x), n_out, n_in, n_vec))
            check_y(t, W, x, y, n_out, n_in, n_vec)


@pytest.mark.parametrize("t", K_TYPES)
def test_mma_every_vector_count(t):
    rng = np.random.default_rng(4200 + t)
    n_out, n_in = 48, 2048
    W = wblocks(t, n_out, n_in, rng)
    for n_vec in range(3, 9):
        x = synth.f32_normal(rng, n_vec * n_in)
        y = host(qg.qgemv(t, dev(W), dev(x), n_out, n_in, n_vec))
        check_y(t, W, x, y, n_out, n_in, n_vec)


@pytest.mark.parametrize("t", K_TYPES)
def test_mma_is_deterministic(t):
    rng = np.random.default_rng(4300 + t)
    n_out, n_in, n_vec = 1000, 11008 if t == qg.Q6_K else 4096, 8
    Wd = dev(wblocks(t, n_out, n_in, rng))
    xd = dev(synth.f32_normal(rng, n_vec * n_in))
    a = host(qg.qgemv(t, Wd, xd, n_out, n_in, n_vec))
    b = host(qg.qgemv(t, Wd, xd, n_out, n_in, n_vec))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("t", K_TYPES)
def test_mma_batched_equals_single_calls(t):
    """A batch of matrices of ragged sizes in one launch gives, per matrix,
    the same bits as one call each (a tile's sum does not depend on which
    CTA computes it)."""
    rng = np.random.default_rng(4400 + t)
    n_in, n_vec = (11008, 8) if t == qg.Q6_K else (4096, 8)
    n_outs = [1, 15, 16, 17, 100, 700, 4096]
    mats, hw, hx = [], [], []
    for n_out in n_outs:
        W = wblocks(t, n_out, n_in, rng)
        x = synth.f32_normal(rng, n_vec * n_in)
        hw.append(W)
        hx.append(x)
        mats.append((dev(W), dev(x), torch.full((n_vec, n_out), np.nan, device="cuda"), n_out))
    qg.qgemv_batched(t, mats, n_in, n_vec)
    torch.cuda.synchronize()
    for (W, x, y, n_out), w_host, x_host in zip(mats, hw, hx):
        ref = qg.qgemv(t, W, x, n_out, n_in, n_vec)
        got = host(y)
        assert np.array_equal(got.view(np.uint32), host(ref).view(np.uint32)), n_out
    W, x, y, n_out = mats[-2]
    check_y(t, hw[-2], hx[-2], host(y), n_out, n_in, n_vec)
    assert qg.device_error() == 0


@pytest.mark.parametrize("t", K_TYPES)
def test_mma_forced_plans(t):
    """Plans the automatic choice does not take for these shapes, forced with
    the QG_MMA_PANEL / QG_MMA_KB knobs: the f16 and the int8 panel for short
    rows, and 43-block rows in chunks of at most 12, 11, 10, 8 and 4 blocks
    (rings of 2 to 8 stages, plain and doubled partial-output buffers). All
    rows against the oracle."""
    rng = np.random.default_rng(4500 + t)
    cases = [(1, 0, 40, 768), (8, 0, 40, 768), (1, 0, 33, 4096), (8, 0, 33, 4096),
             (0, 12, 31, 11008), (0, 11, 31, 11008), (0, 10, 47, 11008), (0, 8, 31, 11008), (0, 4, 17, 11008)]
    for panel, kb, n_out, n_in in cases:
        p0 = qg.tune("QG_MMA_PANEL", panel)
        k0 = qg.tune("QG_MMA_KB", kb)
        try:
            info = qg.kernel_info(t, n_out, n_in, 8)
            assert info.startswith("gemv_mma_kernel<"), info
            if panel == 8:
                assert ",panel8," in info, info
            elif panel == 1:
                assert ",panel" in info, info
            if kb:
                assert int(info.split(" kb=")[1].split()[0]) <= kb, info
            W = wblocks(t, n_out, n_in, rng)
            for n_vec in (3, 8):
                x = synth.f32_normal(rng, n_vec * n_in)
                y = host(qg.qgemv(t, dev(W), dev(x), n_out, n_in, n_vec))
                check_y(t, W, x, y, n_out, n_in, n_vec)
        finally:
            qg.tune("QG_MMA_PANEL", p0)
            qg.tune("QG_MMA_KB", k0)
    assert qg.device_error() == 0


@pytest.mark.parametrize("t,nbytes,dpos,fill", [(qg.Q5_K, 176, (0, 2), 0xFF), (qg.Q2_K, 84, (80, 82), 0xFF),
                                                (qg.Q3_K, 110, (108,), 0xFF), (qg.Q4_0, 18, (0,), 0xFF),
                                                (qg.Q4_1, 20, (0, 2), 0xFF), (qg.Q5_0, 22, (0,), 0xFF),
                                                (qg.Q8_0, 34, (0,), 0x80)])
def test_mma_extreme_codes(t, nbytes, dpos, fill):
    """Every code at its largest (Q5_K 31: nibbles 15 and every fifth bit set;
    Q2_K 3; Q3_K 3 with every hmask bit set; Q4_0 / Q4_1 15; Q5_0 31; Q8_0
    -128), every scale and min at its largest, activations at the int8
    extreme 127: the exact block sums stay exact in the f32 accumulators."""
    rng = np.random.default_rng(4600 + t)
    n_out, n_in = 40, 4096
    W = np.full((n_out * n_in // (32 if t in GROUPED else 256), nbytes), fill, np.uint8)
    for p in dpos:  # d, dmin: f16 of |N(0,1)| * 1e-3
        W[:, p:p + 2] = (np.abs(rng.standard_normal((W.shape[0], 1))) * 1e-3).astype(np.float16).view(np.uint8)
    W = W.reshape(-1)
    for n_vec in (3, 8):
        x = np.full(n_vec * n_in, 2.5, np.float32)
        x[::7] = -2.5
        y = host(qg.qgemv(t, dev(W), dev(x), n_out, n_in, n_vec))
        check_y(t, W, x, y, n_out, n_in, n_vec)


def test_kernel_choice_is_reported():
    """The tensor-core kernel is the one planned for the K-quant types from 3
    vectors, the __dp4a kernel below that; the 32-element types take it by
    default for large launches with several vectors only."""
    qg.tune("QG_MMA_GROUP_MELEM", _GROUP_MELEM["v"])
    try:
        _kernel_choice()
    finally:
        qg.tune("QG_MMA_GROUP_MELEM", 0)


def _kernel_choice():
    assert qg.kernel_info(qg.Q4_K, 4096, 4096, 8).startswith("gemv_mma_kernel<Q4_K,regs,8w>")
    assert qg.kernel_info(qg.Q6_K, 4096, 11008, 8).startswith("gemv_mma_kernel<Q6_K,panel8,16w>")
    assert qg.kernel_info(qg.Q4_K, 4096, 4096, 3).startswith("gemv_mma_kernel<")
    assert qg.kernel_info(qg.Q5_K, 32000, 4096, 8).startswith("gemv_mma_kernel<Q5_K,")
    assert qg.kernel_info(qg.Q5_K, 32000, 4096, 2).startswith("gemv_kernel<Q5_K,NV=2>")
    assert qg.kernel_info(qg.Q2_K, 32000, 4096, 8).startswith("gemv_mma_kernel<Q2_K,")
    assert qg.kernel_info(qg.Q3_K, 32000, 4096, 8).startswith("gemv_mma_kernel<Q3_K,")
    assert qg.kernel_info(qg.Q4_K, 4096, 4096, 2).startswith("gemv_kernel<Q4_K,NV=2>")
    for t in GROUPED:
        assert qg.kernel_info(t, 32000, 4096, 8).startswith("gemv_mma_kernel<"), t
        assert qg.kernel_info(t, 11008, 4096, 4).startswith("gemv_mma_kernel<"), t
        assert qg.kernel_info(t, 4096, 4096, 6).startswith("gemv_mma_kernel<"), t
        assert qg.kernel_info(t, 4096, 4096, 5).startswith("gemv_kernel<"), t
        assert qg.kernel_info(t, 4096, 96, 8).startswith("gemv_kernel<"), t  # not whole groups
    # the __dp4a kernel's two Q6_K items: two lanes per block where their
    # 16-block iterations fill (16 blocks a row), four where they would not
    # (43 blocks a row); the parity tests cover both row lengths
    assert "lanes_per_block=2" in qg.kernel_info(qg.Q6_K, 32000, 4096, 1)
    assert "lanes_per_block=4" in qg.kernel_info(qg.Q6_K, 4096, 11008, 1, 32)


@pytest.mark.parametrize("t", GROUPED)
def test_batch_split_by_routing(t):
    """With the default size rule a batch whose matrices fall on both sides
    of it runs as two launches (tensor cores for the large matrix, __dp4a for
    the small ones); every matrix gives the bits of its own single call, and
    the large one matches the oracle on sampled rows."""
    prev = qg.tune("QG_MMA_GROUP_MELEM", _GROUP_MELEM["v"])
    try:
        rng = np.random.default_rng(4700 + t)
        n_in, n_vec = 4096, 8
        n_outs = [100, 11008, 17, 513]
        kinds = [qg.kernel_info(t, n, n_in, n_vec).split("<")[0] for n in n_outs]
        assert kinds == ["gemv_kernel", "gemv_mma_kernel", "gemv_kernel", "gemv_kernel"], kinds
        mats, hw, hx = [], [], []
        for n_out in n_outs:
            W = wblocks(t, n_out, n_in, rng)
            x = synth.f32_normal(rng, n_vec * n_in)
            hw.append(W)
            hx.append(x)
            mats.append((dev(W), dev(x), torch.full((n_vec, n_out), np.nan, device="cuda"), n_out))
        qg.qgemv_batched(t, mats, n_in, n_vec)
        torch.cuda.synchronize()
        for W, x, y, n_out in mats:
            ref = qg.qgemv(t, W, x, n_out, n_in, n_vec)
            assert np.array_equal(host(y).view(np.uint32), host(ref).view(np.uint32)), n_out
        rows = np.random.default_rng(1).choice(n_outs[1], 48, replace=False)
        check_y(t, hw[1], hx[1], host(mats[1][2]), n_outs[1], n_in, n_vec, rows=rows)
        assert qg.device_error() == 0
    finally:
        qg.tune("QG_MMA_GROUP_MELEM", prev)
