"""Pins of the oracle against values the reference pages print.

Each test reads a fixture under tests/golden/ (the fixture names the page
and section) and checks the oracle reproduces it. Nothing here touches the
CUDA library.
"""
import math

import numpy as np
import pytest

import oracle
from goldens import floats, hexbytes, ints, keyvals, rows
from javarand import JavaRandom

ORACLE_TYPES = {"Q4_0": oracle.Q4_0, "Q4_1": oracle.Q4_1, "Q5_0": oracle.Q5_0,
                "Q8_0": oracle.Q8_0, "Q2_K": oracle.Q2_K, "Q3_K": oracle.Q3_K,
                "Q4_K": oracle.Q4_K, "Q5_K": oracle.Q5_K, "Q6_K": oracle.Q6_K,
                "Q8_K": oracle.Q8_K}


def lesson_block():
    """x_i = (float)(((i * 7919) % 1001) - 500) / 337f, i = 0..31."""
    i = np.arange(32)
    return (((i * 7919) % 1001) - 500).astype(np.float32) / np.float32(337)


def d_of(block: bytes) -> float:
    return float(oracle.f16_to_f32(block[0] | (block[1] << 8)))


# ---------------------------------------------------------------- type table
def test_type_table():
    seen = 0
    for name, elems, nbytes, bpw in rows("type_table.txt"):
        elems, nbytes, bpw = int(elems), int(nbytes), float(bpw)
        assert nbytes * 8 / elems == pytest.approx(bpw, abs=5e-5)
        if name in ORACLE_TYPES:
            assert oracle.type_info(ORACLE_TYPES[name]) == (elems, nbytes)
            assert oracle.type_nbytes(ORACLE_TYPES[name], 4096) == 4096 // elems * nbytes
            seen += 1
    assert seen == 10
    assert oracle.type_info(99) is None


def test_activation_pairing_follows_the_vec_dot_type_table():
    # "量化格式" (candle), the VecDotType table: Q4_0/Q5_0/Q8_0 pair with
    # Q8_0, Q4_1 with Q8_1, the K-quants with Q8K.
    assert oracle.act_type(oracle.Q4_0) == oracle.Q8_0
    assert oracle.act_type(oracle.Q5_0) == oracle.Q8_0
    assert oracle.act_type(oracle.Q8_0) == oracle.Q8_0
    assert oracle.act_type(oracle.Q4_1) == oracle.Q8_1
    for t in (oracle.Q2_K, oracle.Q3_K, oracle.Q4_K, oracle.Q5_K, oracle.Q6_K):
        assert oracle.act_type(t) == oracle.Q8_K


def test_row_length_must_be_whole_blocks():
    # "Building Q8_0 and Q4_0 Like ggml", Example 15: a row of 100 is rejected.
    assert oracle.type_nbytes(oracle.Q4_0, 100) == -1
    assert oracle.type_nbytes(oracle.Q4_K, 4096 + 32) == -1


def test_tensor_sizes_example9():
    g = keyvals("lesson21_seeded_examples.txt")
    assert oracle.type_nbytes(oracle.Q8_0, 64 * 4096) == int(g["ex9_q8_0_bytes"])
    assert oracle.type_nbytes(oracle.Q4_0, 64 * 4096) == int(g["ex9_q4_0_bytes"])
    assert oracle.type_nbytes(oracle.Q8_0, 4096) == int(g["ex9_q8_0_stride"])
    assert oracle.type_nbytes(oracle.Q4_0, 4096) == int(g["ex9_q4_0_stride"])


# ------------------------------------------------------- candle Q8_0 block
def test_candle_q8_0_block():
    g = keyvals("candle_q8_0_block.txt")
    x = (np.arange(32).astype(np.float32) - np.float32(15.5)) / np.float32(10)
    b = oracle.quantize(oracle.Q8_0, x).tobytes()
    assert b[:2] == hexbytes(g["d_bytes_hex"])
    assert d_of(b) == pytest.approx(float(g["d"]), rel=1e-7)
    assert list(np.frombuffer(b[2:], np.int8)) == ints(g["qs"])
    back = oracle.dequantize(oracle.Q8_0, np.frombuffer(b, np.uint8), 32)
    for got, want in zip(back[:4], floats(g["back_0_3"])):
        assert float(got) == pytest.approx(want, rel=1e-7)


# --------------------------------------------------- candle special values
def test_candle_special_values():
    for name, a, repl, shown_in, shown_out in rows("candle_special_values.txt", sep="|"):
        i = np.arange(32).astype(np.float32)
        x = np.float32(float(a)) * i / np.float32(31)
        if repl != "-":
            x[1] = np.float32(float(repl))
        want_in = [float(t) for t in shown_in.split()]
        for got, want in zip(x[:3], want_in):
            if math.isnan(want) or math.isinf(want):
                assert (math.isnan(got) and math.isnan(want)) or got == want
            else:
                assert float(got) == pytest.approx(want, rel=1e-6, abs=0), name
        q = oracle.quantize(oracle.Q8_0, x)
        out = oracle.dequantize(oracle.Q8_0, q, 32)
        for got, want in zip(out[:3], [float(t) for t in shown_out.split()]):
            if math.isnan(want):
                assert math.isnan(got), name
            elif math.isinf(want):
                assert got == want, name
            else:
                assert float(got) == pytest.approx(want, rel=1e-7, abs=0), name


# ------------------------------------------------------------ rml Q4_0 block
def test_rml_q4_0_block():
    g = keyvals("rml_q4_0_block.txt")
    x = np.zeros(32, np.float32)
    x[:4] = np.array(floats(g["x_0_3"]), np.float32)
    b = oracle.quantize(oracle.Q4_0, x).tobytes()
    want = hexbytes(g["first_bytes_hex"])
    assert b[:len(want)] == want
    back = oracle.dequantize(oracle.Q4_0, np.frombuffer(b, np.uint8), 32)
    assert float(back[2]) == float(g["decoded_element_2"])
    assert float(back[0]) == -2.0


# ---------------------------------------------------- lesson 21 fixed blocks
def test_lesson21_example2_q8_0():
    g = keyvals("lesson21_fixed_blocks.txt")
    x = lesson_block()
    amax = float(np.max(np.abs(x)))
    assert f"{amax:.6f}" == g["ex2_amax"]
    b = oracle.quantize(oracle.Q8_0, x).tobytes()
    bits = b[0] | (b[1] << 8)
    assert f"{bits:04X}" == g["ex2_d_f16_bits"]
    assert f"{d_of(b):.9f}" == g["ex2_d_f16"]
    assert list(np.frombuffer(b[2:], np.int8)) == ints(g["ex2_qs"])


def test_lesson21_example3_and_4():
    g = keyvals("lesson21_fixed_blocks.txt")
    x = lesson_block()
    b = oracle.quantize(oracle.Q8_0, x)
    assert b[:2].tobytes().hex() == g["ex4_d_hex"]
    assert b[2:].tobytes().hex() == g["ex4_qs_hex"]
    y = oracle.dequantize(oracle.Q8_0, b, 32)
    assert float(y[0]) == pytest.approx(float(g["ex4_y0"]), rel=1e-7)
    err = np.abs(y.astype(np.float64) - x)
    assert f"{err.max():.6f}" == g["ex3_max_err_f16_d"]
    rmse = 100 * math.sqrt(np.sum((y - x).astype(np.float64) ** 2) / np.sum(x.astype(np.float64) ** 2))
    assert f"{rmse:.4f}" == g["ex3_rel_rmse_pct"]
    # fixed point: quantizing the dequantized values reproduces the bytes
    assert np.array_equal(oracle.quantize(oracle.Q8_0, y), b)


def test_lesson21_example6_q4_0_vs_q8_0():
    g = keyvals("lesson21_fixed_blocks.txt")
    x = lesson_block()
    y4 = oracle.dequantize(oracle.Q4_0, oracle.quantize(oracle.Q4_0, x), 32)
    y8 = oracle.dequantize(oracle.Q8_0, oracle.quantize(oracle.Q8_0, x), 32)
    assert [f"{v:.4f}" for v in y4[:4]] == g["ex6_q4_0_0_3"].split()
    assert [f"{v:.4f}" for v in y8[:4]] == g["ex6_q8_0_0_3"].split()
    for y, tag in ((y4, "q4_0"), (y8, "q8_0")):
        e = (y.astype(np.float64) - x)
        assert f"{np.abs(e).max():.4f}" == g[f"ex6_{tag}_max_err"]
        rmse = 100 * math.sqrt(np.sum(e ** 2) / np.sum(x.astype(np.float64) ** 2))
        assert f"{rmse:.3f}" == g[f"ex6_{tag}_rel_rmse_pct"]


def test_lesson21_example14_hex():
    g = keyvals("lesson21_fixed_blocks.txt")
    i = np.arange(64)
    x = (((i * 7919) % 1001) - 500).astype(np.float32) / np.float32(337)
    x[40] = np.float32(9.5)
    for blk in range(2):
        xb = x[32 * blk:32 * blk + 32]
        assert oracle.quantize(oracle.Q8_0, xb).tobytes().hex() == g[f"ex14_block{blk}_q8_0"]
        assert oracle.quantize(oracle.Q4_0, xb).tobytes().hex() == g[f"ex14_block{blk}_q4_0"]
        assert oracle.quantize(oracle.Q4_1, xb).tobytes().hex() == g[f"ex14_block{blk}_q4_1"]
        assert oracle.quantize(oracle.Q5_0, xb).tobytes().hex() == g[f"ex14_block{blk}_q5_0"]


def page_rel_rmse_pct(y, x):
    """The lesson's error measure: the difference taken in f32, squared and
    summed in f64, over the f32 squares of x summed in f64."""
    e = (y.astype(np.float32) - x.astype(np.float32)).astype(np.float64)
    p = (x.astype(np.float32) * x.astype(np.float32)).astype(np.float64)
    return 100 * math.sqrt(np.sum(e ** 2) / np.sum(p))


def test_lesson21_example7_q4_1():
    g = keyvals("lesson21_fixed_blocks.txt")
    centered = lesson_block()
    shifted = np.float32(2) + np.abs(centered)
    for x, tag in ((centered, "centered"), (shifted, "shifted")):
        lo, hi = float(x.min()), float(x.max())
        assert [f"{lo:.3f}", f"{hi:.3f}"] == g[f"ex7_{tag}_range"].split()
        q = oracle.quantize(oracle.Q4_1, x).tobytes()
        # the printed d and m are the f32 values before f16 storage
        d = np.float32(np.float32(hi) - np.float32(lo)) / np.float32(15)
        assert f"{d:.4f}" == g[f"ex7_{tag}_d"]
        assert f"{lo:.4f}" == g[f"ex7_{tag}_m"]
        assert q[0] | (q[1] << 8) == oracle.f32_to_f16(d)
        assert q[2] | (q[3] << 8) == oracle.f32_to_f16(lo)
        y = oracle.dequantize(oracle.Q4_1, np.frombuffer(q, np.uint8), 32)
        assert f"{page_rel_rmse_pct(y, x):.3f}" == g[f"ex7_{tag}_rmse_pct"]


def test_lesson21_example8_q5_0():
    g = keyvals("lesson21_fixed_blocks.txt")
    x = lesson_block()
    q = oracle.quantize(oracle.Q5_0, x).tobytes()
    assert len(q) == 22
    mx = x[np.argmax(np.abs(x))]                   # first of largest magnitude
    assert f"{mx:.4f}" == g["ex8_max"]
    assert f"{mx / np.float32(-16):.5f}" == g["ex8_d"]
    qh = int.from_bytes(q[2:6], "little")
    assert format(qh, "032b") == g["ex8_qh_bits"]
    y = oracle.dequantize(oracle.Q5_0, np.frombuffer(q, np.uint8), 32)
    assert f"{page_rel_rmse_pct(y, x):.3f}" == g["ex8_rmse_pct"]
    # the same block is the first Q5_0 line of Example 14
    assert q.hex() == g["ex14_block0_q5_0"]


def test_lesson21_example5_q4_0_signed_max_and_nibbles():
    g = keyvals("lesson21_fixed_blocks.txt")
    a = (np.arange(32).astype(np.float32) - np.float32(12)) / np.float32(4)
    for x, tag in ((a, "a"), (-a, "b")):
        q = oracle.quantize(oracle.Q4_0, x).tobytes()
        assert f"{d_of(q):.4f}" == g[f"ex5_{tag}_d"]
        assert f"{q[2]:02X}" == g["ex5_byte0"]
        assert f"{q[3]:02X}" == g["ex5_byte1"]
        assert q[2] & 0xF == int(g["ex5_code_0"])
        assert q[2] >> 4 == int(g["ex5_code_16"])
        back = oracle.dequantize(oracle.Q4_0, np.frombuffer(q, np.uint8), 32)
        # the extreme value maps to code 0 (-8) and is stored up to f16 rounding of d
        assert float(back[31]) == pytest.approx(float(g[f"ex5_{tag}_max"]), rel=1e-3)


def test_q4_0_nan_and_overflowing_inverse_follow_the_java_cast():
    """Lesson 21's Q4_0 quantizer (Example 5) is Java: its (int) cast truncates,
    gives 0 for NaN and saturates at the int range; a NaN element is skipped
    by the signed max (the comparison is false) and gets code 0, as candle's
    special-value table ("一些边界值") also has it. Bytes derived by hand."""
    # NaN first, then 1.0, then zeros: max = 1.0, d = -0.125 (f16 0xB000),
    # id = -8; NaN -> 0, 1.0 -> (int)0.5 = 0, 0.0 -> (int)8.5 = 8.
    x = np.zeros(32, np.float32)
    x[0], x[1] = np.nan, 1.0
    q = oracle.quantize(oracle.Q4_0, x).tobytes()
    assert q == bytes([0x00, 0xB0, 0x80, 0x80] + [0x88] * 14)
    # max = 2^-146 (a subnormal): d = -2^-149, 1/d overflows to -inf, so
    # 2^-146 * id = -inf -> int minimum -> low nibble 0; -2^-147 * id = +inf
    # -> int maximum -> min(15, .) = 15; 0 * id = NaN -> 0. d rounds to f16 -0.
    x = np.zeros(32, np.float32)
    x[0], x[1] = np.float32(2.0 ** -146), np.float32(-(2.0 ** -147))
    q = oracle.quantize(oracle.Q4_0, x).tobytes()
    assert q == bytes([0x00, 0x80, 0x00, 0x0F] + [0x00] * 14)


def test_q4_1_nan_element_gets_code_0():
    """Lesson 21's Q4_1 (Example 7, Java): NaN fails both the min and the max
    comparison, so min = 0 and max = 1 here; its code is (int)NaN = 0."""
    x = np.zeros(32, np.float32)
    x[0], x[1] = np.nan, 1.0
    q = oracle.quantize(oracle.Q4_1, x).tobytes()
    d = np.float32(1.0) / np.float32(15.0)
    assert q[0:2] == np.float16(d).tobytes() and q[2:4] == bytes(2)
    # 1.0: (1 - 0) * id + 0.5 rounds to 15.5 -> 15; zeros: 0.5 -> 0
    assert q[4] == 0x00 and q[5] == 0x0F and q[6:] == bytes(14)


# --------------------------------------------- lesson 21 seeded Java examples
def java_pairs(seed, n, scale_a=0.02):
    r = JavaRandom(seed)
    a = np.zeros(n, np.float32)
    b = np.zeros(n, np.float32)
    for i in range(n):
        a[i] = np.float32(r.next_gaussian()) * np.float32(scale_a)
        b[i] = np.float32(r.next_gaussian())
    return a, b


def java_outlier_weights(r, n):
    w = np.zeros(n, np.float32)
    for i in range(n):
        g = np.float32(r.next_gaussian()) * np.float32(0.02)
        w[i] = g * np.float32(10 if r.next_int(500) == 0 else 1)
    return w


def java_gaussians(r, n):
    return np.array([np.float32(r.next_gaussian()) for _ in range(n)], np.float32)


def f16_field(blocks: np.ndarray, nbytes: int, nblocks: int) -> np.ndarray:
    raw = blocks.reshape(nblocks, nbytes)[:, :2].copy().view(np.uint16).reshape(-1)
    return np.array([oracle.f16_to_f32(int(h)) for h in raw], np.float32)


def test_lesson21_example10_q8_0_dot():
    g = keyvals("lesson21_seeded_examples.txt")
    n = 4096
    a, b = java_pairs(22, n)
    assert f"{np.dot(a.astype(np.float64), b.astype(np.float64)):.6f}" == g["ex10_exact"]
    qa, qb = oracle.quantize(oracle.Q8_0, a), oracle.quantize(oracle.Q8_0, b)
    s = oracle.block_isums(oracle.Q8_0, qa, qb, 1, n, 1).reshape(-1)
    da, db = f16_field(qa, 34, n // 32), f16_field(qb, 34, n // 32)
    # the page's float loop: sumf += sumi * (dx * dy), all in f32
    sumf = np.float32(0)
    for ib in range(n // 32):
        sumf = np.float32(sumf + np.float32(np.float32(s[ib]) * np.float32(da[ib] * db[ib])))
    assert f"{sumf:.6f}" == g["ex10_q8_0_dot"]
    y = oracle.gemv(oracle.Q8_0, qa, qb, 1, n, 1)[0, 0]
    assert y == pytest.approx(float(g["ex10_q8_0_dot"]), abs=5e-6)


def test_lesson21_example11_q4_0_q8_0_dot():
    g = keyvals("lesson21_seeded_examples.txt")
    n = 4096
    w, x = java_pairs(23, n)
    assert f"{np.dot(w.astype(np.float64), x.astype(np.float64)):.6f}" == g["ex11_exact"]
    qw, qx = oracle.quantize(oracle.Q4_0, w), oracle.quantize(oracle.Q8_0, x)
    wdeq = oracle.dequantize(oracle.Q4_0, qw, n)
    assert f"{np.dot(wdeq.astype(np.float64), x.astype(np.float64)):.6f}" == g["ex11_weight_only"]
    s = oracle.block_isums(oracle.Q4_0, qw, qx, 1, n, 1).reshape(-1)
    dw, dx = f16_field(qw, 18, n // 32), f16_field(qx, 34, n // 32)
    sumf = np.float32(0)
    for ib in range(n // 32):  # (sumi0 + sumi1) * dw * dx, left to right in f32
        sumf = np.float32(sumf + np.float32(np.float32(np.float32(s[ib]) * dw[ib]) * dx[ib]))
    assert f"{sumf:.6f}" == g["ex11_kernel"]
    y = oracle.gemv(oracle.Q4_0, qw, qx, 1, n, 1)[0, 0]
    assert y == pytest.approx(float(g["ex11_kernel"]), abs=5e-6)


def rel_rmse_pct(y, x):
    e = y.astype(np.float64) - x.astype(np.float64)
    return 100 * math.sqrt(np.sum(e ** 2) / np.sum(x.astype(np.float64) ** 2))


def test_lesson21_example12_error_table():
    g = keyvals("lesson21_seeded_examples.txt")
    x = java_outlier_weights(JavaRandom(24), 65536)
    f16 = np.array([oracle.f16_to_f32(oracle.f32_to_f16(v)) for v in x], np.float32)
    assert f"{rel_rmse_pct(f16, x):.4f}" == g["ex12_f16_rmse_pct"]
    for t, key in ((oracle.Q8_0, "ex12_q8_0_rmse_pct"), (oracle.Q4_0, "ex12_q4_0_rmse_pct"),
                   (oracle.Q5_0, "ex12_q5_0_rmse_pct"), (oracle.Q4_1, "ex12_q4_1_rmse_pct")):
        y = oracle.dequantize(t, oracle.quantize(t, x), x.size)
        assert f"{rel_rmse_pct(y, x):.4f}" == g[key]
    for t, key in ((oracle.Q5_0, "ex12_q5_0_snr_db"), (oracle.Q4_1, "ex12_q4_1_snr_db")):
        y = oracle.dequantize(t, oracle.quantize(t, x), x.size)
        e = np.sum((y.astype(np.float64) - x) ** 2)
        assert f"{10 * math.log10(np.sum(x.astype(np.float64) ** 2) / e):.2f}" == g[key]


@pytest.mark.slow
def test_lesson21_example13_output_error():
    g = keyvals("lesson21_seeded_examples.txt")
    rows_, cols = 256, 4096
    r = JavaRandom(25)
    w = java_outlier_weights(r, rows_ * cols)
    x = java_gaussians(r, cols)
    ref = w.reshape(rows_, cols).astype(np.float64) @ x.astype(np.float64)
    qx = oracle.quantize(oracle.Q8_0, x)
    for t, key in ((oracle.Q8_0, "ex13_q8_0_out_err_pct"), (oracle.Q4_0, "ex13_q4_0_out_err_pct")):
        qw = oracle.quantize(t, w)
        y = oracle.gemv(t, qw, qx, rows_, cols, 1)[0]
        err = 100 * math.sqrt(np.sum((y - ref) ** 2) / np.sum(ref ** 2))
        assert f"{err:.4f}" == g[key]


@pytest.mark.slow
def test_lesson21_example15_quantizer_report():
    g = keyvals("lesson21_seeded_examples.txt")
    rows_, cols = 512, 2048
    r = JavaRandom(26)
    w = java_outlier_weights(r, rows_ * cols)
    x = java_gaussians(r, cols)
    W = w.reshape(rows_, cols).astype(np.float64)
    ref = W @ x.astype(np.float64)
    for t, tag in ((oracle.Q8_0, "q8_0"), (oracle.Q4_0, "q4_0")):
        q = oracle.quantize(t, w)
        assert q.size == int(g[f"ex15_{tag}_bytes"])
        wq = oracle.dequantize(t, q, w.size)
        assert f"{rel_rmse_pct(wq, w):.3f}" == g[f"ex15_{tag}_weight_rmse_pct"]
        yq = wq.reshape(rows_, cols).astype(np.float64) @ x.astype(np.float64)
        err = 100 * math.sqrt(np.sum((yq - ref) ** 2) / np.sum(ref ** 2))
        assert f"{err:.3f}" == g[f"ex15_{tag}_output_err_pct"]
        # "stable": re-quantizing the dequantized tensor gives the same bytes
        assert np.array_equal(oracle.quantize(t, wq), q)


# ------------------------------------------------------- rml Q4_K trace
def test_rml_q4_k_element_200_trace():
    g = keyvals("rml_q4_k_trace.txt")
    e = int(g["element"])
    rng = np.random.default_rng(7)
    blk = bytearray(rng.integers(0, 256, 144, dtype=np.uint8).tobytes())
    d, dmin = 0.5, 0.25
    blk[0:2] = np.float16(d).tobytes()
    blk[2:4] = np.float16(dmin).tobytes()
    s = blk[4:16]
    qs = blk[16:144]
    sc = (s[int(g["scale_low_byte"])] & 0xF) | ((s[int(g["scale_high_byte"])] >> 6) << 4)
    mn = (s[int(g["min_low_byte"])] >> 4) | ((s[int(g["min_high_byte"])] >> 6) << 4)
    q = qs[int(g["qs_byte"])] & 0xF
    assert g["qs_nibble"] == "low" and e // 32 == int(g["sub_block"])
    vals = oracle.dequantize(oracle.Q4_K, np.frombuffer(bytes(blk), np.uint8), 256)
    assert float(vals[e]) == np.float32(d * sc * q - dmin * mn)
    # changing any byte the trace does not name leaves element 200 unchanged
    named = {0, 1, 2, 3, 4 + 10, 4 + 2, 4 + 6, 16 + 104}
    for pos in range(144):
        if pos in named:
            continue
        b2 = bytearray(blk)
        b2[pos] ^= 0xFF
        v2 = oracle.dequantize(oracle.Q4_K, np.frombuffer(bytes(b2), np.uint8), 256)
        assert v2[e] == vals[e], pos
