"""Pins of the oracle against closed forms, library routines, brute force and
structural invariants of the block formats (no GPU).

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign, index or shift, a transposed operand) fails at least one.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(12345)


# ------------------------------------------------------------- f16 codec
def test_f16_decode_matches_numpy_for_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits], np.float32)
    same = (got.view(np.uint32) == want.view(np.uint32)) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def test_f16_encode_matches_numpy_round_to_nearest_even():
    edge = [0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e9, -1e9,
            2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 3 * 2.0 ** -25, 2.0 ** -14,
            2.0 ** -14 * (1 - 2.0 ** -11), 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
            0.012204724, 1.0 / 127, float("inf"), float("-inf")]
    rnd = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32),
        (RNG.standard_normal(20000) * 1e-5).astype(np.float32),
        (RNG.standard_normal(20000) * 3e4).astype(np.float32),
        # exact ties between two f16 values in the normal and subnormal ranges
        (np.arange(1, 2000) * 2.0 ** -25).astype(np.float32),
        ((1024 + np.arange(0, 1024) + 0.5) * 2.0 ** -10).astype(np.float32),
    ])
    xs = np.concatenate([np.array(edge, np.float32), rnd])
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16(v) for v in xs], np.uint16)
    assert np.array_equal(got, want)
    assert oracle.f32_to_f16(float("nan")) & 0x7C00 == 0x7C00
    assert oracle.f32_to_f16(float("nan")) & 0x3FF != 0


# ------------------------------------------- exactness of dequantization
def f32_round(fr: Fraction) -> float:
    """Round an exact rational to the nearest f32 (ties to even), written
    from the binary32 format (24-bit significand, normal range only)."""
    if fr == 0:
        return 0.0
    sign = -1 if fr < 0 else 1
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    scaled = a / Fraction(2) ** (e - 23)          # in [2^23, 2^24)
    fl = scaled.numerator // scaled.denominator
    rem = scaled - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * float(fl * Fraction(2) ** (e - 23))


def random_k_block(t):
    b = bytearray(RNG.integers(0, 256, oracle.type_info(t)[1], dtype=np.uint8).tobytes())
    d = np.float16(abs(RNG.standard_normal()) * 1e-3)
    if t == oracle.Q4_K:
        b[0:2] = d.tobytes()
        b[2:4] = np.float16(abs(RNG.standard_normal()) * 1e-3).tobytes()
    else:
        b[208:210] = d.tobytes()
    return bytes(b)


def half(raw: bytes, off: int) -> Fraction:
    return Fraction(float(np.frombuffer(raw[off:off + 2], np.float16)[0]))


def test_dequant_is_the_correctly_rounded_exact_value():
    # Q4_K: d*sc*q and dmin*m are exact in f32, so the value is the exact
    # rational d*sc*q - dmin*m rounded once. The test decodes through the
    # element-200 rule for every sub-block of the upper half and checks the
    # lower half through the 6-bit low fields named by the candle page.
    for _ in range(20):
        raw = random_k_block(oracle.Q4_K)
        vals = oracle.dequantize(oracle.Q4_K, np.frombuffer(raw, np.uint8), 256)
        d, dmin, s, qs = half(raw, 0), half(raw, 2), raw[4:16], raw[16:]
        for e in range(256):
            j = e // 32
            if j < 4:
                sc, m = s[j] & 63, s[j + 4] & 63
            else:
                sc = (s[j + 4] & 0xF) | ((s[j - 4] >> 6) << 4)
                m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4)
            p = e % 64
            q = qs[32 * (e // 64) + p] & 0xF if p < 32 else qs[32 * (e // 64) + p - 32] >> 4
            exact = d * sc * q - dmin * m
            assert float(vals[e]) == f32_round(exact)
    # Q6_K, Q8_0, Q4_0: every product is exact, so dequantized values are
    # exactly d * integer.
    for _ in range(20):
        raw = random_k_block(oracle.Q6_K)
        vals = oracle.dequantize(oracle.Q6_K, np.frombuffer(raw, np.uint8), 256)
        d = half(raw, 208)
        sc = np.frombuffer(raw[192:208], np.int8)
        for e in range(256):
            ratio = Fraction(float(vals[e])) / (d * int(sc[e // 16])) if sc[e // 16] and d else None
            if ratio is not None:
                assert ratio.denominator == 1 and -32 <= ratio <= 31
    for t, nbytes in ((oracle.Q8_0, 34), (oracle.Q4_0, 18)):
        raw = bytearray(RNG.integers(0, 256, nbytes * 8, dtype=np.uint8).tobytes())
        for b in range(8):
            raw[nbytes * b:nbytes * b + 2] = np.float16(RNG.standard_normal()).tobytes()
        vals = oracle.dequantize(t, np.frombuffer(bytes(raw), np.uint8), 256)
        for b in range(8):
            d = half(bytes(raw), nbytes * b)
            for e in range(32):
                r = Fraction(float(vals[32 * b + e])) / d
                assert r.denominator == 1
                assert (-128 <= r <= 127) if t == oracle.Q8_0 else (-8 <= r <= 7)
    # Q5_0 and Q8_1: d times an integer in [-16, 15] / [-128, 127];
    # Q4_1: code * d is exact in f32 (15 bits), so the value is the exact
    # code * d + m rounded once.
    for t, nbytes in ((oracle.Q5_0, 22), (oracle.Q8_1, 36), (oracle.Q4_1, 20)):
        raw = bytearray(RNG.integers(0, 256, nbytes * 8, dtype=np.uint8).tobytes())
        for b in range(8):
            raw[nbytes * b:nbytes * b + 2] = np.float16(RNG.standard_normal()).tobytes()
            if t == oracle.Q4_1:
                raw[nbytes * b + 2:nbytes * b + 4] = np.float16(RNG.standard_normal()).tobytes()
        raw = bytes(raw)
        vals = oracle.dequantize(t, np.frombuffer(raw, np.uint8), 256)
        for b in range(8):
            blk = raw[nbytes * b:nbytes * (b + 1)]
            d = half(blk, 0)
            for e in range(32):
                if t == oracle.Q4_1:
                    byte = blk[4 + e % 16]
                    code = byte & 0xF if e < 16 else byte >> 4
                    assert float(vals[32 * b + e]) == f32_round(code * d + half(blk, 2))
                    continue
                r = Fraction(float(vals[32 * b + e])) / d
                assert r.denominator == 1
                assert (-16 <= r <= 15) if t == oracle.Q5_0 else (-128 <= r <= 127)


def test_q5_0_every_bit_is_one_bit_of_one_element():
    # "Building Q8_0 and Q4_0 Like ggml", Example 8: bit j of the 32-bit qh
    # word is bit 4 of code j; the low 4 bits sit in nibbles as in Q4_0
    # (byte j: element j low, element j + 16 high). Setting one bit of a zero
    # block (codes 0, value -16 d) raises exactly one element by its weight.
    base = bytearray(22)
    base[0:2] = np.float16(1.0).tobytes()
    v0 = oracle.dequantize(oracle.Q5_0, np.frombuffer(bytes(base), np.uint8), 32)
    assert np.all(v0 == -16.0)
    for bit in range(8 * 20):
        raw = bytearray(base)
        raw[2 + bit // 8] |= 1 << (bit % 8)
        v = oracle.dequantize(oracle.Q5_0, np.frombuffer(bytes(raw), np.uint8), 32) - v0
        hit = np.nonzero(v)[0]
        assert hit.size == 1
        if bit < 32:                                   # qh, little-endian word
            assert hit[0] == bit and v[hit[0]] == 16
        else:
            j, k = divmod(bit - 32, 8)
            assert hit[0] == (j if k < 4 else j + 16)
            assert v[hit[0]] == 1 << (k % 4)


def test_q8_1_is_q8_0_plus_the_scaled_code_sum():
    # "量化格式" (candle): Q8_1 is the activation format of the _1 types and
    # carries the block's sum beside Q8_0's d and codes. The codes and d must
    # be Q8_0's bytes, and s the f16 of d times the code sum.
    x = RNG.standard_normal(32 * 64).astype(np.float32)
    x[::97] *= 50
    q1 = oracle.quantize(oracle.Q8_1, x).reshape(64, 36)
    q0 = oracle.quantize(oracle.Q8_0, x).reshape(64, 34)
    assert np.array_equal(q1[:, 0:2], q0[:, 0:2])
    assert np.array_equal(q1[:, 4:], q0[:, 2:])
    for b in range(64):
        d = float(np.frombuffer(q0[b, 0:2].tobytes(), np.float16)[0])
        s = float(np.frombuffer(q1[b, 2:4].tobytes(), np.float16)[0])
        tot = int(q1[b, 4:].view(np.int8).astype(np.int64).sum())
        # s was rounded from the f32 d, which is within 2^-11 of the f16 d
        assert abs(s - d * tot) <= (2.0 ** -10) * abs(d * tot) + 1e-7
    assert np.array_equal(oracle.dequantize(oracle.Q8_1, q1.reshape(-1), x.size),
                          oracle.dequantize(oracle.Q8_0, q0.reshape(-1), x.size))
    # a block holding inf: d = inf, every code 0, s = 0 * inf stored as the
    # one quiet NaN 0x7E00, whatever sign the host gives that NaN
    x = np.ones(32, np.float32)
    x[5] = np.inf
    q = oracle.quantize(oracle.Q8_1, x).tobytes()
    assert q[0:4] == bytes([0x00, 0x7C, 0x00, 0x7E]) and not any(q[4:])


# ----------------------------------------------- Q4_K packing structure
def q4k_fields(raw):
    """(scale[8], min[8]) observed through the oracle: d = 1, dmin = 0 gives
    sc*q; d = 0, dmin = -1 gives +m; all nibbles 1."""
    b = bytearray(raw)
    b[16:] = bytes([0x11]) * 128
    b[0:2] = np.float16(1).tobytes()
    b[2:4] = np.float16(0).tobytes()
    v = oracle.dequantize(oracle.Q4_K, np.frombuffer(bytes(b), np.uint8), 256)
    sc = [int(v[32 * j]) for j in range(8)]
    assert all((v[32 * j:32 * j + 32] == v[32 * j]).all() for j in range(8))
    b[0:2] = np.float16(0).tobytes()
    b[2:4] = np.float16(-1).tobytes()
    v = oracle.dequantize(oracle.Q4_K, np.frombuffer(bytes(b), np.uint8), 256)
    mn = [int(v[32 * j]) for j in range(8)]
    return sc, mn


def test_q4_k_scales_use_every_bit_once():
    base = bytes(144)
    sc0, mn0 = q4k_fields(base)
    assert sc0 == [0] * 8 and mn0 == [0] * 8
    hits = {}
    for byte in range(12):
        for bit in range(8):
            b = bytearray(base)
            b[4 + byte] = 1 << bit
            sc, mn = q4k_fields(bytes(b))
            changed = [("sc", j, v) for j, v in enumerate(sc) if v] + \
                      [("m", j, v) for j, v in enumerate(mn) if v]
            assert len(changed) == 1, (byte, bit, changed)
            kind, j, v = changed[0]
            assert v & (v - 1) == 0  # a single bit of a 6-bit field
            hits[(kind, j, v.bit_length() - 1)] = (byte, bit)
            # candle: sub-blocks 0..3 sit in the low 6 bits of bytes 0..7;
            # sub-blocks 4..7 keep low 4 bits in bytes 8..11 and borrow the
            # top 2 bits of bytes 0..7
            if j < 4:
                assert byte < 8 and bit < 6
            elif v.bit_length() - 1 < 4:
                assert byte >= 8
            else:
                assert byte < 8 and bit >= 6
    assert len(hits) == 96  # 16 fields x 6 bits, each reached by one bit


def test_q4_k_nibbles_are_a_bijection_in_element_order():
    base = bytearray(144)
    base[0:2] = np.float16(1).tobytes()
    base[4:16] = bytes([1, 1, 1, 1, 0, 0, 0, 0, 0x01, 0x01, 0x01, 0x01])  # all scales 1, mins 0
    seen = {}
    for byte in range(128):
        for hi in (0, 1):
            b = bytearray(base)
            b[16 + byte] = 0x10 if hi else 0x01
            v = oracle.dequantize(oracle.Q4_K, np.frombuffer(bytes(b), np.uint8), 256)
            nz = np.nonzero(v)[0]
            assert len(nz) == 1 and v[nz[0]] == 1.0
            seen[int(nz[0])] = (byte, hi)
    assert sorted(seen) == list(range(256))
    # element order inside a 64-element chunk: low nibbles of the chunk's 32
    # bytes first, then high nibbles (the element-200 trace generalised)
    assert seen[200] == (104, 0) and seen[232] == (104, 1) and seen[0] == (0, 0)


# ----------------------------------------------- Q6_K packing structure
def q6k_block(d=1.0, scales=None, ql=None, qh=None):
    b = bytearray(210)
    if ql is not None:
        b[0:128] = ql
    if qh is not None:
        b[128:192] = qh
    b[192:208] = np.array(scales if scales is not None else [1] * 16, np.int8).tobytes()
    b[208:210] = np.float16(d).tobytes()
    return np.frombuffer(bytes(b), np.uint8)


def test_q6_k_every_bit_is_one_bit_of_one_element():
    zero = oracle.dequantize(oracle.Q6_K, q6k_block(), 256)
    assert (zero == -32).all()  # q = 0 means -32
    owner = {}
    for byte in range(192):
        for bit in range(8):
            raw = bytearray(192)
            raw[byte] = 1 << bit
            v = oracle.dequantize(oracle.Q6_K, q6k_block(ql=raw[:128], qh=raw[128:]), 256)
            nz = np.nonzero(v != -32)[0]
            assert len(nz) == 1, (byte, bit)
            delta = int(v[nz[0]] + 32)
            assert delta & (delta - 1) == 0
            # ql gives the low 4 bits, qh the high 2 bits of q
            assert (delta < 16) == (byte < 128)
            owner.setdefault(int(nz[0]), set()).add(delta)
    assert sorted(owner) == list(range(256))
    assert all(s == {1, 2, 4, 8, 16, 32} for s in owner.values())


def test_q6_k_scale_index_is_element_over_16_and_d_is_last():
    for j in range(16):
        sc = [0] * 16
        sc[j] = -3
        v = oracle.dequantize(oracle.Q6_K, q6k_block(d=0.5, scales=sc), 256)
        nz = np.nonzero(v)[0]
        assert list(nz) == list(range(16 * j, 16 * j + 16))
        assert (v[nz] == np.float32(0.5 * -3 * -32)).all()


# ------------------------------------------------------- Q8_K reading
def test_q8_k_rule_and_bsums():
    x = (RNG.standard_normal(256 * 6) * np.array([1, 1e-3, 50, 1, 1, 1]).repeat(256)).astype(np.float32)
    x[256 * 4:256 * 5] = 0  # an all-zero block
    q = oracle.quantize(oracle.Q8_K, x).reshape(6, 292)
    for b in range(6):
        xb = x[256 * b:256 * b + 256]
        d = q[b, 0:4].copy().view(np.float32)[0]
        qs = q[b, 4:260].copy().view(np.int8).astype(np.int32)
        bs = q[b, 260:292].copy().view(np.int16).astype(np.int32)
        amax = np.float32(np.max(np.abs(xb)))
        assert d == amax / np.float32(127)            # f32 d, not rounded to f16
        assert np.array_equal(bs, qs.reshape(16, 16).sum(axis=1))
        if amax == 0:
            assert (qs == 0).all()
            continue
        assert abs(qs[np.argmax(np.abs(xb))]) == 127
        assert np.abs(qs).max() <= 127
        # every code is the nearest integer to x/d up to the rounding of id
        assert np.all(np.abs(qs - xb.astype(np.float64) / float(d)) <= 0.5 + 1e-4)


def test_q8_0_codes_round_half_away_from_zero():
    # x = k + 0.5 steps with d exactly 1: amax = 127 gives d = 1, id = 1
    x = np.zeros(32, np.float32)
    x[0] = 127
    x[1:6] = [2.5, -2.5, 0.5, -0.5, 126.5]
    q = oracle.quantize(oracle.Q8_0, x)
    codes = q[2:].view(np.int8)
    assert list(codes[:6]) == [127, 3, -3, 1, -1, 127]


def test_zero_block_gives_zero():
    # rml tests: ZeroActivationsGiveZero -- an all-zero row has d = 0, id = 0
    for t in (oracle.Q8_0, oracle.Q8_K):
        q = oracle.quantize(t, np.zeros(256, np.float32))
        assert not q.any()
    # Q4_0: d = 0 / -8 = -0.0 (f16 0x8000) and every code is 8, meaning 0
    q = oracle.quantize(oracle.Q4_0, np.zeros(32, np.float32))
    assert q.tobytes() == bytes([0x00, 0x80]) + bytes([0x88]) * 16
    assert not oracle.dequantize(oracle.Q4_0, q, 32).any()
    W = oracle.quantize(oracle.Q8_0, RNG.standard_normal(256).astype(np.float32))
    xq = oracle.quantize(oracle.Q8_0, np.zeros(256, np.float32))
    assert oracle.gemv(oracle.Q8_0, W, xq, 1, 256, 1)[0, 0] == 0.0
    # Q5_0: d = -0.0, every code 16 (all fifth bits set, nibbles 0)
    q = oracle.quantize(oracle.Q5_0, np.zeros(32, np.float32))
    assert q.tobytes() == bytes([0x00, 0x80]) + bytes([0xFF]) * 4 + bytes(16)
    assert not oracle.dequantize(oracle.Q5_0, q, 32).any()
    # Q4_1: d = 0, m = 0, codes 0; a constant block keeps its value in m
    assert not oracle.quantize(oracle.Q4_1, np.zeros(32, np.float32)).any()
    q = oracle.quantize(oracle.Q4_1, np.full(32, 0.75, np.float32))
    assert np.all(oracle.dequantize(oracle.Q4_1, q, 32) == 0.75)
    assert not oracle.quantize(oracle.Q8_1, np.zeros(32, np.float32)).any()


# -------------------------------------------------- brute force on tiny inputs
def random_weights(t, n_out, n_in):
    if t in (oracle.Q8_0, oracle.Q4_0, oracle.Q5_0, oracle.Q4_1):
        return oracle.quantize(t, (RNG.standard_normal(n_out * n_in) * 0.02).astype(np.float32))
    nb = n_out * n_in // 256
    if t in (oracle.Q2_K, oracle.Q3_K, oracle.Q5_K):
        from ggml_block_quantized_gb300 import synth
        return synth.k_blocks(t, nb, RNG)
    return np.frombuffer(b"".join(random_k_block(t) for _ in range(nb)), np.uint8).copy()


@pytest.mark.parametrize("t", [oracle.Q8_0, oracle.Q4_0, oracle.Q5_0, oracle.Q2_K, oracle.Q3_K,
                               oracle.Q4_K, oracle.Q5_K, oracle.Q6_K])
def test_block_form_equals_dequantize_then_f64_dot(t):
    for n_out, n_in, n_vec in ((1, 256, 1), (3, 512, 2), (8, 512, 3)):
        W = random_weights(t, n_out, n_in)
        x = RNG.standard_normal(n_vec * n_in).astype(np.float32)
        xq = oracle.quantize(oracle.act_type(t), x)
        y = oracle.gemv(t, W, xq, n_out, n_in, n_vec)
        yb = oracle.gemv_dequant(t, W, xq, n_out, n_in, n_vec)
        # scale for the bound: sum of |w_i * a_i|
        wd = oracle.dequantize(t, W, n_out * n_in).reshape(n_out, n_in).astype(np.float64)
        ad = oracle.dequantize(oracle.act_type(t), xq, n_vec * n_in).reshape(n_vec, n_in)
        mag = np.abs(ad.astype(np.float64)) @ np.abs(wd).T
        assert np.all(np.abs(y - yb) <= 1e-12 * mag + 1e-300)


def test_q4_1_block_form_differs_only_by_the_rounded_activation_sum():
    # Q4_1 against Q8_1: each block's dot splits into d_w d_x sum(code q)
    # plus m_w times the activation sum; the block form takes that sum as the
    # stored f16 s. So block form minus the exact f64 dot is, per block,
    # m_w (s - d_x sum q), and |s - d_x sum q| <= 2^-10 |d_x sum q| (f16
    # rounding of a value computed from the f32 d).
    n_out, n_in, n_vec = 5, 512, 3
    W = random_weights(oracle.Q4_1, n_out, n_in)
    x = (RNG.standard_normal(n_vec * n_in) + 0.3).astype(np.float32)
    xq = oracle.quantize(oracle.Q8_1, x)
    y = oracle.gemv(oracle.Q4_1, W, xq, n_out, n_in, n_vec)
    yb = oracle.gemv_dequant(oracle.Q4_1, W, xq, n_out, n_in, n_vec)
    nb = n_in // 32
    Wb = W.reshape(n_out, nb, 20)
    Xb = xq.reshape(n_vec, nb, 36)
    m = np.frombuffer(Wb[:, :, 2:4].tobytes(), np.float16).astype(np.float64).reshape(n_out, nb)
    dx = np.frombuffer(Xb[:, :, 0:2].tobytes(), np.float16).astype(np.float64).reshape(n_vec, nb)
    sx = np.frombuffer(Xb[:, :, 2:4].tobytes(), np.float16).astype(np.float64).reshape(n_vec, nb)
    cs = Xb[:, :, 4:].view(np.int8).astype(np.float64).sum(axis=2)
    corr = (sx - dx * cs) @ m.T                                    # [n_vec, n_out]
    assert np.allclose(y, yb + corr, rtol=1e-12, atol=1e-12)
    bound = (2.0 ** -10) * (np.abs(dx * cs) @ np.abs(m).T)
    assert np.all(np.abs(y - yb) <= bound + 1e-12)
    assert np.any(corr != 0)


def test_block_isums_by_hand_for_one_q8_0_and_q4_0_block():
    w = np.arange(-16, 16).astype(np.float32)     # Q8_0: d = 16/127
    x = np.linspace(-1, 1, 32).astype(np.float32)
    for t in (oracle.Q8_0, oracle.Q4_0):
        qw, qx = oracle.quantize(t, w), oracle.quantize(oracle.Q8_0, x)
        s = int(oracle.block_isums(t, qw, qx, 1, 32, 1)[0, 0, 0, 0])
        cx = qx[2:].view(np.int8).astype(np.int64)
        if t == oracle.Q8_0:
            cw = qw[2:].view(np.int8).astype(np.int64)
        else:
            nib = np.concatenate([qw[2:] & 0xF, qw[2:] >> 4]).astype(np.int64)
            cw = nib - 8
        assert s == int(np.dot(cw, cx))
    # Q5_0 codes minus 16 against Q8_0; Q4_1 raw codes against Q8_1
    qw, qx = oracle.quantize(oracle.Q5_0, w), oracle.quantize(oracle.Q8_0, x)
    qh = int.from_bytes(qw[2:6].tobytes(), "little")
    nib = np.concatenate([qw[6:] & 0xF, qw[6:] >> 4]).astype(np.int64)
    cw = nib + 16 * np.array([(qh >> j) & 1 for j in range(32)]) - 16
    assert int(oracle.block_isums(oracle.Q5_0, qw, qx, 1, 32, 1)[0, 0, 0, 0]) == int(np.dot(cw, qx[2:].view(np.int8)))
    qw, qx = oracle.quantize(oracle.Q4_1, w), oracle.quantize(oracle.Q8_1, x)
    nib = np.concatenate([qw[4:] & 0xF, qw[4:] >> 4]).astype(np.int64)
    assert int(oracle.block_isums(oracle.Q4_1, qw, qx, 1, 32, 1)[0, 0, 0, 0]) == int(np.dot(nib, qx[4:].view(np.int8)))


def test_q4_k_min_term_equals_bsum_pairs():
    # rml: the sub-block min term is min * sum(a), and sum(a) over 32
    # activations is two of the stored 16-sums
    W = random_weights(oracle.Q4_K, 2, 512)
    xq = oracle.quantize(oracle.Q8_K, RNG.standard_normal(512).astype(np.float32))
    sums = oracle.block_isums(oracle.Q4_K, W, xq, 2, 512, 1)
    for o in range(2):
        for b in range(2):
            blk = W[(o * 2 + b) * 144:(o * 2 + b + 1) * 144].tobytes()
            s = blk[4:16]
            mins = [s[j + 4] & 63 if j < 4 else (s[j + 4] >> 4) | ((s[j] >> 6) << 4) for j in range(8)]
            bs = xq[b * 292 + 260:b * 292 + 292].copy().view(np.int16).astype(np.int64)
            assert sums[0, o, b, 1] == sum(mins[j] * (bs[2 * j] + bs[2 * j + 1]) for j in range(8))


def test_int32_sums_stay_in_range_at_extremes():
    # all codes at their extremes: Q6_K q = 0 (-32), scales -128, a = -127
    W = q6k_block(d=1.0, scales=[-128] * 16)
    xq = oracle.quantize(oracle.Q8_K, np.full(256, -1.0, np.float32))
    s = oracle.block_isums(oracle.Q6_K, W, xq, 1, 256, 1)[0, 0, 0, 0]
    assert s == 16 * (-128) * 16 * (-32) * (-127)


# ------------------------------------------------------ sanity (unpinned)
def test_round_trip_rmse_near_candle_table():
    # candle's round-trip table on 262144 N(0,1) values: Q8_0 0.5365%,
    # Q8K 0.6948%. Different random draws, so a loose statistical check.
    x = RNG.standard_normal(262144).astype(np.float32)
    for t, want in ((oracle.Q8_0, 0.5365), (oracle.Q8_K, 0.6948)):
        y = oracle.dequantize(t, oracle.quantize(t, x), x.size)
        e = (y.astype(np.float64) - x)
        got = 100 * math.sqrt(np.sum(e ** 2) / np.sum(x.astype(np.float64) ** 2))
        assert got == pytest.approx(want, rel=0.01)


# ------------------------------------------- Q2_K / Q3_K / Q5_K structure
# The pages give these types' sizes (and, for Q5_K, that it carries dmin and
# Q4_K's packed scales); the element layouts are readings. They are pinned
# here by structure: every bit is one bit of one element or one field, the
# scale of an element is that of its 16- or 32-element sub-block, Q5_K
# reduces to the pinned Q4_K, and the block form equals brute force.
def k_block(t, d=1.0, dmin=0.0):
    raw = bytearray(oracle.type_info(t)[1])
    if t == oracle.Q2_K:
        raw[80:82] = np.float16(d).tobytes()
        raw[82:84] = np.float16(dmin).tobytes()
    elif t == oracle.Q3_K:
        raw[108:110] = np.float16(d).tobytes()
    elif t == oracle.Q5_K:
        raw[0:2] = np.float16(d).tobytes()
        raw[2:4] = np.float16(dmin).tobytes()
    return raw


def deq(t, raw):
    return oracle.dequantize(t, np.frombuffer(bytes(raw), np.uint8), 256).astype(np.float64)


def test_q5_k_reduces_to_q4_k():
    # qh all zero: the same d, dmin, scales and qs decode exactly as Q4_K
    # (whose element-200 trace the rml page prints); a set qh bit adds
    # exactly 16 * d * sc of the element's 32-element sub-block
    for _ in range(10):
        q4 = bytearray(RNG.integers(0, 256, 144, dtype=np.uint8).tobytes())
        q4[0:2] = np.float16(abs(RNG.standard_normal()) * 1e-2).tobytes()
        q4[2:4] = np.float16(abs(RNG.standard_normal()) * 1e-2).tobytes()
        q5 = bytearray(176)
        q5[0:16] = q4[0:16]
        q5[48:176] = q4[16:144]
        v4 = oracle.dequantize(oracle.Q4_K, np.frombuffer(bytes(q4), np.uint8), 256)
        assert np.array_equal(oracle.dequantize(oracle.Q5_K, np.frombuffer(bytes(q5), np.uint8), 256), v4)
    blk = k_block(oracle.Q5_K, d=1.0)
    blk[4:16] = bytes([5, 6, 7, 8, 0, 0, 0, 0, 0x21, 0x43, 0x65, 0x87])  # sub-block scales 5..8, then 1..7 and 8 low nibbles
    base = deq(oracle.Q5_K, blk)
    seen = set()
    for byte in range(32):
        for bit in range(8):
            raw = bytearray(blk)
            raw[16 + byte] |= 1 << bit
            dv = deq(oracle.Q5_K, raw) - base
            hit = np.nonzero(dv)[0]
            assert hit.size == 1
            e = int(hit[0])
            seen.add(e)
            sc = [5, 6, 7, 8, 1, 3, 5, 7][e // 32]
            assert dv[e] == 16 * sc
    assert seen == set(range(256))


@pytest.mark.parametrize("t", [oracle.Q2_K, oracle.Q3_K])
def test_q2_k_q3_k_every_code_bit_is_one_bit_of_one_element(t):
    blk = k_block(t, d=1.0, dmin=0.0)
    if t == oracle.Q2_K:
        blk[0:16] = bytes([1] * 16)      # every scale 1, every min 0
        qs_off, qs_len = 16, 64
    else:
        blk[96:104] = bytes([0x11] * 8)  # low 4 bits 1 for every scale
        blk[104:108] = bytes([0xAA] * 4)  # high 2 bits 2: biased 33, i.e. scale 1
        qs_off, qs_len = 32, 64
    base = deq(t, blk)
    weight_of = {}
    for byte in range(qs_len):
        for bit in range(8):
            raw = bytearray(blk)
            raw[qs_off + byte] ^= 1 << bit
            dv = deq(t, raw) - base
            hit = np.nonzero(dv)[0]
            assert hit.size == 1, (byte, bit)
            e = int(hit[0])
            assert abs(dv[e]) == (1 << (bit % 2)), (byte, bit)  # bits come in 2-bit fields
            weight_of.setdefault(e, []).append(bit % 2)
    assert sorted(weight_of) == list(range(256))
    assert all(sorted(v) == [0, 1] for v in weight_of.values())
    if t == oracle.Q3_K:
        # the 256 hmask bits: one per element, each moving it by 4
        hit_all = set()
        for byte in range(32):
            for bit in range(8):
                raw = bytearray(blk)
                raw[byte] ^= 1 << bit
                dv = deq(t, raw) - base
                hit = np.nonzero(dv)[0]
                assert hit.size == 1 and abs(dv[hit[0]]) == 4
                hit_all.add(int(hit[0]))
        assert hit_all == set(range(256))
        # all code bits and hmask bits clear: -4 times the scale everywhere
        assert np.all(base == -4.0)


@pytest.mark.parametrize("t", [oracle.Q2_K, oracle.Q3_K])
def test_q2_k_q3_k_scales_cover_16_element_sub_blocks(t):
    # every code 1 (Q3_K: 2-bit value 1 with its hmask bit set), d = 1; each
    # scale bit then moves exactly the 16 elements of one sub-block, and the
    # sub-blocks are 16 consecutive elements each
    blk = k_block(t, d=1.0, dmin=0.5)
    if t == oracle.Q2_K:
        blk[16:80] = bytes([0x55] * 64)
        scale_bytes = range(0, 16)
    else:
        blk[32:96] = bytes([0x55] * 64)
        blk[0:32] = bytes([0xFF] * 32)
        scale_bytes = range(96, 108)
    base = deq(t, blk)
    owners = {}
    for byte in scale_bytes:
        for bit in range(8):
            raw = bytearray(blk)
            raw[byte] ^= 1 << bit
            dv = deq(t, raw) - base
            hit = np.nonzero(dv)[0]
            assert hit.size == 16, (byte, bit)
            j = int(hit[0]) // 16
            assert list(hit) == list(range(16 * j, 16 * j + 16))
            assert np.all(dv[hit] == dv[hit[0]])
            owners.setdefault(j, []).append(abs(dv[hit[0]]))
    assert sorted(owners) == list(range(16))
    if t == oracle.Q2_K:   # 4 scale bits (x code 1) and 4 min bits (x dmin 0.5) per sub-block
        assert all(sorted(v) == [0.5, 1, 1, 2, 2, 4, 4, 8] for v in owners.values())
    else:                  # 6 scale bits per sub-block, code 1
        assert all(sorted(v) == [1, 2, 4, 8, 16, 32] for v in owners.values())


@pytest.mark.parametrize("t", [oracle.Q2_K, oracle.Q3_K, oracle.Q5_K])
def test_new_k_types_dequant_rounds_once(t):
    # every product is exact in f32, so values are the exact rationals rounded
    # once: compare with the brute-force form's exact doubles through f32
    W = random_weights(t, 4, 512)
    xq = oracle.quantize(oracle.Q8_K, np.zeros(512, np.float32))
    vals = oracle.dequantize(t, W, 4 * 512)
    # the exact value of each element is the brute-force form's dot with a
    # one-hot activation: build it through gemv_dequant on unit activations
    unit = np.zeros(256, np.float32)
    unit[0] = 127.0                    # Q8_K: d = 1, code 127 -> a_0 = 127 exactly
    xu = oracle.quantize(oracle.Q8_K, unit)
    for blk in range(8):
        w = W[blk * oracle.type_info(t)[1]:(blk + 1) * oracle.type_info(t)[1]]
        exact = oracle.gemv_dequant(t, w, xu, 1, 256, 1)[0, 0] / 127.0
        assert float(vals[blk * 256]) == f32_round(Fraction(exact))
    del xq


def test_q3_k_int32_extremes():
    blk = k_block(oracle.Q3_K, d=1.0)
    blk[96:108] = bytes(12)                 # every biased scale 0 -> -32
    # codes: 2-bit value 0 with hmask clear -> -4 everywhere
    xq = oracle.quantize(oracle.Q8_K, np.full(256, -1.0, np.float32))
    s = oracle.block_isums(oracle.Q3_K, np.frombuffer(bytes(blk), np.uint8), xq, 1, 256, 1)[0, 0, 0, 0]
    assert s == 16 * (-32) * 16 * (-4) * (-127)
