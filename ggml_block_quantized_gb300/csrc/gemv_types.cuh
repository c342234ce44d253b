// gemv_types.cuh - per-type policies of the streaming GEMV kernel: how the
// paired activation blocks are laid out in shared memory (filled either from
// byte-exact Q8_0/Q8_K blocks or by quantizing f32 x in the kernel's
// prologue), and how a group of lanes forms one weight block's exact int32
// sums and float terms.
//
// Block formats ("量化格式" (candle), block structure table; "Building Q8_0
// and Q4_0 Like ggml", Examples 1 and 5; "Quantization" (rml), Unpacking the
// packed fields):
//   Q8_0  34 B: f16 d, int8 qs[32]                          value q * d
//   Q4_0  18 B: f16 d, qs[16]; byte j = elem j | elem j+16 << 4, value (c - 8) * d
//   Q4_1  20 B: f16 d, f16 m, qs[16] as Q4_0; value c * d + m
//   Q5_0  22 B: f16 d, u32 qh (LE), qs[16] as Q4_0 for the low 4 bits; bit j of
//               qh is bit 4 of code j; value (c - 16) * d
//   Q8_1  36 B: f16 d, f16 s = f16(d * sum of codes), int8 qs[32] (activations)
//   Q4_K 144 B: f16 d, f16 dmin, scales[12] (8 x 6-bit scale, 8 x 6-bit min),
//               qs[128]; elem e in chunk e/64: low nibble of qs[32(e/64) + e%64]
//               for e%64 < 32, else high nibble of qs[32(e/64) + e%64 - 32];
//               value d * sc_j * q - dmin * m_j, j = e / 32
//   Q6_K 210 B: ql[128], qh[64], int8 scales[16], f16 d (last); for
//               e = 128h + 32k + l: low 4 bits from ql[64h + 32(k&1) + l]
//               (low nibble for k < 2, high for k >= 2), high 2 bits from
//               (qh[32h + l] >> 2k) & 3; value d * scales[e/16] * (q - 32)
//   Q8_K 292 B: f32 d, int8 qs[256], int16 bsums[16] (activations only)
//
// Exact block sums (the int32 part of every product):
//   Q8_0: S = sum qw * qx
//   Q4_0: S = sum c * qx - 8 * sum qx
//   Q5_0: S = sum c * qx - 16 * sum qx
//   Q4_1: S = sum c * qx  (the min enters as m_w * s_x)
//   Q4_K: S_q = sum_j sc_j * sum_{i in j} q_i a_i ; S_m = sum_j m_j (bsum_2j + bsum_2j+1)
//   Q6_K: S = sum_j sc_j * sum_{i in j} q_i a_i - 32 * sum_j sc_j * bsum_j
// Float step: Q8_0, Q4_0, Q5_0, Q6_K: S * (d_w * d_x); Q4_1: S * (d_w * d_x)
// + m_w * s_x; Q4_K: d_x * (d_w * S_q - dmin * S_m). In the product, a block's lanes each apply the float step to
// their own exact partial sums (no cross-lane sum per block); the
// diagnostic mode adds the partials across the block's lanes first and
// writes the whole-block sums.
//
// Activation quantization in the prologue follows the rule of quantize.cu
// exactly (amax over the block, d = amax / 127 with IEEE division, id = 1/d
// or 0, code = roundf(x * id)), so the codes are the bytes quantize_act
// writes.
#pragma once

#include "qg_common.cuh"

namespace qg {

// Sum of a 32-bit int over aligned groups of G lanes (G = 1, 2, 4, 8).
template <int G>
__device__ __forceinline__ int group_sum(int v) {
#pragma unroll
    for (int m = 1; m < G; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int m = 1; m < G; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}

// Eight consecutive f32 values of x from global memory (16-byte aligned),
// cached in L2 only: x may have been written by the kernel this one waited
// for.
__device__ __forceinline__ void load8g(const float *p, float (&v)[8]) {
    const float4 a = __ldcg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldcg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Codes of 8 values with the inverse scale id, packed 4 per word; returns
// their sum.
__device__ __forceinline__ int codes8(const float (&v)[8], float id, int lo, int hi, uint32_t (&w)[2]) {
    w[0] = w[1] = 0u;
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q = code_from_rounded(roundf(__fmul_rn(v[i], id)), lo, hi);
        sum += q;
        w[i >> 2] |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * (i & 3));
    }
    return sum;
}

__device__ __forceinline__ uint32_t pack16(int lo, int hi) {
    return (static_cast<uint32_t>(lo) & 0xFFFFu) | (static_cast<uint32_t>(hi) << 16);
}

// Q8_0-rule quantization of 32-value blocks 0..count-1 of f32 x (global
// memory) inside the GEMV prologue: 4 lanes per block (lane l takes values
// 8(l%4)..+7 of block base + l/4), 8 blocks per warp step, two steps at a
// time so that their load round trips and reduction chains overlap.
// emit(i, ok, part, w, sum, d) stores one lane's part of block i (ok: i < count);
// loaded() runs once per warp, when its first loads have arrived.
template <int LO, class Emit, class Loaded>
__device__ __forceinline__ void stage_x_q8_0(const float *x, int count, int warp, int nwarps, int lane, Emit emit,
                                             Loaded loaded) {
    const int part = lane & 3;
    for (int base = warp * 8; base < count; base += 2 * nwarps * 8) {
        int idx[2];
        bool ok[2];
        float v[2][8];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            idx[n] = base + n * nwarps * 8 + (lane >> 2);
            ok[n] = idx[n] < count;
            if (ok[n]) {
                load8g(x + 32 * static_cast<size_t>(idx[n]) + 8 * part, v[n]);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) v[n][k] = 0.0f;
            }
        }
        float a[2];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            a[n] = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) a[n] = fmaxf(a[n], fabsf(v[n][k]));
        }
        if (base == warp * 8 && a[0] >= 0.0f) loaded();  // (a >= 0 always: waits for the loads)
#pragma unroll
        for (int m = 1; m < 4; m <<= 1)
#pragma unroll
            for (int n = 0; n < 2; ++n) a[n] = fmaxf(a[n], __shfl_xor_sync(0xffffffffu, a[n], m));
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const float d = a[n] / 127.0f;
            const float id = d != 0.0f ? 1.0f / d : 0.0f;
            uint32_t w[2];
            const int sum = group_sum<4>(codes8(v[n], id, LO, 127, w));
            emit(idx[n], ok[n], part, w, sum, d);
        }
    }
}

// Q8_K quantization of 256-value blocks 0..count-1 of f32 x (global memory):
// one warp per block, lane l owning values 8l..8l+7, two blocks at a time.
// emit(i, w, sum16, d) stores block i's part of lane l: its codes (2 words),
// the 16-value sum of lanes (2k, 2k+1) (in both lanes of the pair) and d.
// emit is called by all lanes of the warp together (it may shuffle);
// loaded() runs once per warp, when its first loads have arrived.
template <class Emit, class Loaded>
__device__ __forceinline__ void stage_x_q8_k(const float *x, int count, int warp, int nwarps, int lane, Emit emit,
                                             Loaded loaded) {
    for (int i = warp; i < count; i += 2 * nwarps) {
        const int j = i + nwarps;
        const bool two = j < count;  // warp-uniform
        float v[2][8];
        load8g(x + 256 * static_cast<size_t>(i) + 8 * lane, v[0]);
        if (two) {
            load8g(x + 256 * static_cast<size_t>(j) + 8 * lane, v[1]);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) v[1][k] = 0.0f;
        }
        float a[2];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            a[n] = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) a[n] = fmaxf(a[n], fabsf(v[n][k]));
        }
        if (i == warp && a[0] >= 0.0f) loaded();  // (a >= 0 always: waits for the loads)
#pragma unroll
        for (int m = 1; m < 32; m <<= 1)
#pragma unroll
            for (int n = 0; n < 2; ++n) a[n] = fmaxf(a[n], __shfl_xor_sync(0xffffffffu, a[n], m));
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const float d = a[n] / 127.0f;
            const float id = d != 0.0f ? 1.0f / d : 0.0f;
            uint32_t w[2];
            const int s = codes8(v[n], id, -127, 127, w);
            const int sum16 = s + __shfl_xor_sync(0xffffffffu, s, 1);
            if (n == 0 || two) emit(n == 0 ? i : j, w, sum16, d);
        }
    }
}

// ========================================================================
// Staging interfaces shared by all types:
//   stage_act(xq, act, nb, nv, tid, nthr): records from byte-exact blocks.
//   stage_x(x, act, count, warp, nwarps, lane, loaded): records for
//     activation blocks 0 .. count-1 (block index g = v * nb + b) quantized
//     from their f32 values in global memory (x = value 0 of block 0);
//     loaded() is called once per warp that loads anything, when its first
//     loads have arrived.
// Item interface: item<NV, ISUMS>(rowa, b, sub, active, acta, nb, acc,
//   isum_row, isum_vstride) adds the block's float terms of one weight row
//   (shared address rowa) to acc[v], or writes its exact sums.
// ========================================================================

// ------------------------------------------------------------------------
// Q8_0-paired types (Q8_0, Q4_0): activations staged as 48-byte records
// per (vector, block): qs[32] | f32 d_x | int32 sum(qs) | 8 pad bytes.
// Record stride 48 B makes 8 consecutive blocks' 128-bit loads hit 8
// disjoint bank quads.
// ------------------------------------------------------------------------
struct ActQ8_0 {
    static constexpr int kRecord = 48;
    static constexpr int kValues = 32;  // f32 values per activation block
    static size_t bytes(int nb, int nv) { return static_cast<size_t>(nv) * nb * kRecord; }

    // From byte-exact Q8_0 blocks: xq [nv][nb] x 34 B (2-byte aligned each).
    __device__ static void stage(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        const int n = nb * nv;
        for (int i = tid; i < n; i += nthr) {
            const uint16_t *blk = reinterpret_cast<const uint16_t *>(xq + static_cast<size_t>(i) * 34);
            uint32_t w[8];
            int asum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                w[j] = static_cast<uint32_t>(__ldg(blk + 1 + 2 * j)) |
                       (static_cast<uint32_t>(__ldg(blk + 2 + 2 * j)) << 16);
                asum = dp4a(w[j], 0x01010101u, asum);
            }
            uint8_t *rec = act + static_cast<size_t>(i) * kRecord;
            reinterpret_cast<uint4 *>(rec)[0] = make_uint4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<uint4 *>(rec)[1] = make_uint4(w[4], w[5], w[6], w[7]);
            const float dx = f16_bits_to_f32(__ldg(blk));
            reinterpret_cast<uint4 *>(rec)[2] =
                make_uint4(__float_as_uint(dx), static_cast<uint32_t>(asum), 0u, 0u);
        }
    }

    // From f32 x: 4 lanes per 32-value block (the Q8_0 rule).
    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        stage_x_q8_0<-128>(x, count, warp, nwarps, lane,
                           [&](int i, bool ok, int part, const uint32_t (&w)[2], int sum, float d) {
                               if (!ok) return;
                               uint8_t *rec = act + static_cast<size_t>(i) * kRecord;
                               reinterpret_cast<uint2 *>(rec)[part] = make_uint2(w[0], w[1]);
                               if (part == 0) {
                                   const float dx = __half2float(__float2half_rn(d));  // the stored f16 scale
                                   reinterpret_cast<uint4 *>(rec)[2] =
                                       make_uint4(__float_as_uint(dx), static_cast<uint32_t>(sum), 0u, 0u);
                               }
                           },
                           loaded);
    }
};

struct TypeQ8_0 {
    static constexpr int kBlockElems = 32, kBlockBytes = 34, kLanesPerBlock = 1, kSums = 1;
    static constexpr int kActValues = ActQ8_0::kValues;
    static size_t act_bytes(int nb, int nv) { return ActQ8_0::bytes(nb, nv); }
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        ActQ8_0::stage(xq, act, nb, nv, tid, nthr);
    }
    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        ActQ8_0::stage_x(x, act, count, warp, nwarps, lane, loaded);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int /*sub*/, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;
        const float dw = f16_bits_to_f32(ld_s16(blk));
        uint32_t w[8];
        ld_words_a2<8>(blk + 2, w);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + (static_cast<uint32_t>(v) * nb + b) * ActQ8_0::kRecord;
            const uint4 a0 = ld_s128(rec), a1 = ld_s128(rec + 16);
            const float dx = __uint_as_float(ld_s32(rec + 32));
            int s = dp4a(w[0], a0.x, 0);
            s = dp4a(w[1], a0.y, s);
            s = dp4a(w[2], a0.z, s);
            s = dp4a(w[3], a0.w, s);
            s = dp4a(w[4], a1.x, s);
            s = dp4a(w[5], a1.y, s);
            s = dp4a(w[6], a1.z, s);
            s = dp4a(w[7], a1.w, s);
            if (ISUMS) {
                if (active) isum_row[v * isum_vstride + b] = s;
            } else if (active) {
                acc[v] = fmaf(static_cast<float>(s), dw * dx, acc[v]);
            }
        }
    }
};

struct TypeQ4_0 {
    static constexpr int kBlockElems = 32, kBlockBytes = 18, kLanesPerBlock = 1, kSums = 1;
    static constexpr int kActValues = ActQ8_0::kValues;
    static size_t act_bytes(int nb, int nv) { return ActQ8_0::bytes(nb, nv); }
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        ActQ8_0::stage(xq, act, nb, nv, tid, nthr);
    }
    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        ActQ8_0::stage_x(x, act, count, warp, nwarps, lane, loaded);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int /*sub*/, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;
        const float dw = f16_bits_to_f32(ld_s16(blk));
        uint32_t q[4];
        ld_words_a2<4>(blk + 2, q);
        uint32_t lo[4], hi[4];  // codes of elements 4i.. and 16+4i..
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = q[i] & 0x0F0F0F0Fu;
            hi[i] = (q[i] >> 4) & 0x0F0F0F0Fu;
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + (static_cast<uint32_t>(v) * nb + b) * ActQ8_0::kRecord;
            const uint4 a0 = ld_s128(rec), a1 = ld_s128(rec + 16), ex = ld_s128(rec + 32);
            int s = dp4a(lo[0], a0.x, 0);
            s = dp4a(lo[1], a0.y, s);
            s = dp4a(lo[2], a0.z, s);
            s = dp4a(lo[3], a0.w, s);
            s = dp4a(hi[0], a1.x, s);
            s = dp4a(hi[1], a1.y, s);
            s = dp4a(hi[2], a1.z, s);
            s = dp4a(hi[3], a1.w, s);
            s -= 8 * static_cast<int>(ex.y);
            if (ISUMS) {
                if (active) isum_row[v * isum_vstride + b] = s;
            } else if (active) {
                acc[v] = fmaf(static_cast<float>(s), dw * __uint_as_float(ex.x), acc[v]);
            }
        }
    }
};

// Bit 4 of each byte of a word from 4 consecutive bits of x (x < 16): the
// multiplier places bit k at bit 8k + 4 (the shifted copies 7 bits apart
// never overlap, so nothing carries).
__device__ __forceinline__ uint32_t fifth_bits(uint32_t x4) { return (x4 * 0x02040810u) & 0x10101010u; }

// Q5_0 (weights, paired with Q8_0): 22-byte blocks, 2-byte aligned.
struct TypeQ5_0 {
    static constexpr int kBlockElems = 32, kBlockBytes = 22, kLanesPerBlock = 1, kSums = 1;
    static constexpr int kActValues = ActQ8_0::kValues;
    static size_t act_bytes(int nb, int nv) { return ActQ8_0::bytes(nb, nv); }
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        ActQ8_0::stage(xq, act, nb, nv, tid, nthr);
    }
    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        ActQ8_0::stage_x(x, act, count, warp, nwarps, lane, loaded);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int /*sub*/, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;
        const float dw = f16_bits_to_f32(ld_s16(blk));
        uint32_t w[5];  // qh, then the 16 nibble bytes
        ld_words_a2<5>(blk + 2, w);
        const uint32_t qh = w[0];
        uint32_t lo[4], hi[4];  // 5-bit codes of elements 4i.. and 16+4i..
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = (w[1 + i] & 0x0F0F0F0Fu) | fifth_bits((qh >> (4 * i)) & 0xFu);
            hi[i] = ((w[1 + i] >> 4) & 0x0F0F0F0Fu) | fifth_bits((qh >> (16 + 4 * i)) & 0xFu);
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + (static_cast<uint32_t>(v) * nb + b) * ActQ8_0::kRecord;
            const uint4 a0 = ld_s128(rec), a1 = ld_s128(rec + 16), ex = ld_s128(rec + 32);
            int s = dp4a(lo[0], a0.x, 0);
            s = dp4a(lo[1], a0.y, s);
            s = dp4a(lo[2], a0.z, s);
            s = dp4a(lo[3], a0.w, s);
            s = dp4a(hi[0], a1.x, s);
            s = dp4a(hi[1], a1.y, s);
            s = dp4a(hi[2], a1.z, s);
            s = dp4a(hi[3], a1.w, s);
            s -= 16 * static_cast<int>(ex.y);
            if (ISUMS) {
                if (active) isum_row[v * isum_vstride + b] = s;
            } else if (active) {
                acc[v] = fmaf(static_cast<float>(s), dw * __uint_as_float(ex.x), acc[v]);
            }
        }
    }
};

// ------------------------------------------------------------------------
// Q8_1-paired type (Q4_1): the Q8_0 record with s_x in the third word of its
// tail: qs[32] | f32 d_x | int32 sum(qs) | f32 s_x | 4 pad bytes.
// ------------------------------------------------------------------------
struct ActQ8_1 {
    static constexpr int kRecord = ActQ8_0::kRecord;
    static constexpr int kValues = 32;
    static size_t bytes(int nb, int nv) { return static_cast<size_t>(nv) * nb * kRecord; }

    // From byte-exact Q8_1 blocks: xq [nv][nb] x 36 B (4-byte aligned each).
    __device__ static void stage(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        const int n = nb * nv;
        for (int i = tid; i < n; i += nthr) {
            const uint32_t *blk = reinterpret_cast<const uint32_t *>(xq + static_cast<size_t>(i) * 36);
            const uint32_t ds = __ldg(blk);
            uint32_t w[8];
            int asum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                w[j] = __ldg(blk + 1 + j);
                asum = dp4a(w[j], 0x01010101u, asum);
            }
            uint8_t *rec = act + static_cast<size_t>(i) * kRecord;
            reinterpret_cast<uint4 *>(rec)[0] = make_uint4(w[0], w[1], w[2], w[3]);
            reinterpret_cast<uint4 *>(rec)[1] = make_uint4(w[4], w[5], w[6], w[7]);
            reinterpret_cast<uint4 *>(rec)[2] =
                make_uint4(__float_as_uint(f16_bits_to_f32(ds)), static_cast<uint32_t>(asum),
                           __float_as_uint(f16_bits_to_f32(ds >> 16)), 0u);
        }
    }

    // From f32 x (the Q8_0 rule, then s = f16(sum * d) from the f32 d): 4
    // lanes per block.
    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        stage_x_q8_0<-128>(x, count, warp, nwarps, lane,
                           [&](int i, bool ok, int part, const uint32_t (&w)[2], int sum, float d) {
                               if (!ok) return;
                               uint8_t *rec = act + static_cast<size_t>(i) * kRecord;
                               reinterpret_cast<uint2 *>(rec)[part] = make_uint2(w[0], w[1]);
                               if (part == 0) {
                                   const float dx = __half2float(__float2half_rn(d));
                                   const float sx =
                                       __half2float(__float2half_rn(__fmul_rn(static_cast<float>(sum), d)));
                                   reinterpret_cast<uint4 *>(rec)[2] = make_uint4(
                                       __float_as_uint(dx), static_cast<uint32_t>(sum), __float_as_uint(sx), 0u);
                               }
                           },
                           loaded);
    }
};

// Q4_1 (weights, paired with Q8_1): 20-byte blocks. Rows start at multiples
// of 20 bytes from a 16-byte aligned W and stages keep the address modulo
// 16, so every block is 4-byte aligned in shared memory.
struct TypeQ4_1 {
    static constexpr int kBlockElems = 32, kBlockBytes = 20, kLanesPerBlock = 1, kSums = 1;
    static constexpr int kActValues = ActQ8_1::kValues;
    static size_t act_bytes(int nb, int nv) { return ActQ8_1::bytes(nb, nv); }
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        ActQ8_1::stage(xq, act, nb, nv, tid, nthr);
    }
    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        ActQ8_1::stage_x(x, act, count, warp, nwarps, lane, loaded);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int /*sub*/, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;
        const uint32_t dm = ld_s32(blk);
        const float dw = f16_bits_to_f32(dm), mw = f16_bits_to_f32(dm >> 16);
        uint32_t qw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qw[i] = ld_s32(blk + 4 + 4 * i);
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = qw[i] & 0x0F0F0F0Fu;
            hi[i] = (qw[i] >> 4) & 0x0F0F0F0Fu;
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + (static_cast<uint32_t>(v) * nb + b) * ActQ8_1::kRecord;
            const uint4 a0 = ld_s128(rec), a1 = ld_s128(rec + 16), ex = ld_s128(rec + 32);
            int s = dp4a(lo[0], a0.x, 0);
            s = dp4a(lo[1], a0.y, s);
            s = dp4a(lo[2], a0.z, s);
            s = dp4a(lo[3], a0.w, s);
            s = dp4a(hi[0], a1.x, s);
            s = dp4a(hi[1], a1.y, s);
            s = dp4a(hi[2], a1.z, s);
            s = dp4a(hi[3], a1.w, s);
            if (ISUMS) {
                if (active) isum_row[v * isum_vstride + b] = s;
            } else if (active) {
                acc[v] = fmaf(static_cast<float>(s), dw * __uint_as_float(ex.x), acc[v]);
                acc[v] = fmaf(mw, __uint_as_float(ex.z), acc[v]);
            }
        }
    }
};


// ------------------------------------------------------------------------
// Q4_K. Two lanes per block: lane h takes half h (values 128h..128h+127,
// sub-blocks 4h..4h+3, qs bytes 64h..64h+63). Activations staged per
// (vector, block, half) as a 144-byte record:
//   codes[128] | int16 bsum32[4] (sub-blocks 4h..4h+3) | f32 d_x | pad
// where bsum32(j) = bsums[2j] + bsums[2j+1]. A 144-byte stride (36 words)
// puts 8 consecutive records' 128-bit loads in 8 disjoint bank quads.
// ------------------------------------------------------------------------
struct TypeQ4_K {
    static constexpr int kBlockElems = 256, kBlockBytes = 144, kLanesPerBlock = 2, kSums = 2;
    static constexpr int kActValues = 256;
    static constexpr int kRecord = 144;
    static size_t act_bytes(int nb, int nv) { return static_cast<size_t>(nv) * nb * 2 * kRecord; }

    // From byte-exact Q8_K blocks (292 B, 4-byte aligned): 9 16-byte units per record.
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        const int n = nb * nv * 2 * 9;
        for (int u = tid; u < n; u += nthr) {
            const int r = u / 9, part = u % 9;
            const int blk = r >> 1, h = r & 1;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + static_cast<size_t>(blk) * 292);
            uint4 *rec = reinterpret_cast<uint4 *>(act + static_cast<size_t>(r) * kRecord);
            if (part < 8) {
                const int w = 1 + 32 * h + 4 * part;  // codes start at byte 4
                rec[part] = make_uint4(__ldg(src + w), __ldg(src + w + 1), __ldg(src + w + 2), __ldg(src + w + 3));
            } else {
                // bsums (int16) at byte 260 = word 65; sub-block 4h+t needs bsums[8h+2t], [8h+2t+1]
                int s[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const uint32_t pr = __ldg(src + 65 + 4 * h + t);
                    s[t] = static_cast<int>(static_cast<int16_t>(pr & 0xFFFFu)) +
                           static_cast<int>(static_cast<int16_t>(pr >> 16));
                }
                rec[8] = make_uint4(pack16(s[0], s[1]), pack16(s[2], s[3]), __ldg(src), 0u);
            }
        }
    }

    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        const int h = lane >> 4;
        stage_x_q8_k(x, count, warp, nwarps, lane, [&](int i, const uint32_t (&w)[2], int s16, float d) {
            const int s32 = s16 + __shfl_xor_sync(0xffffffffu, s16, 2);  // sub-block lane/4
            uint8_t *rec = act + (static_cast<size_t>(i) * 2 + h) * kRecord;
            reinterpret_cast<uint2 *>(rec)[lane & 15] = make_uint2(w[0], w[1]);
            if ((lane & 3) == 0) reinterpret_cast<int16_t *>(rec + 128)[(lane >> 2) & 3] = static_cast<int16_t>(s32);
            if ((lane & 15) == 0) reinterpret_cast<uint2 *>(rec + 136)[0] = make_uint2(__float_as_uint(d), 0u);
        }, loaded);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int h, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;  // 16-byte aligned
        const uint4 hdr = ld_s128(blk);
        const float dw = f16_bits_to_f32(hdr.x);
        const float dmin = f16_bits_to_f32(hdr.x >> 16);
        // 6-bit scales and mins of sub-blocks 4h..4h+3, one per byte.
        // scales[0..3] = hdr.y, [4..7] = hdr.z, [8..11] = hdr.w. Half 0: sc = s[j] & 63,
        // m = s[j+4] & 63. Half 1 (j = 4 + t): sc = (s[8+t] & 15) | (s[t] >> 6) << 4,
        // m = (s[8+t] >> 4) | (s[4+t] >> 6) << 4.
        const uint32_t SC = h == 0 ? (hdr.y & 0x3F3F3F3Fu)
                                   : ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u));
        const uint32_t M = h == 0 ? (hdr.z & 0x3F3F3F3Fu)
                                  : (((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u));
        uint32_t q[16];
        const uint32_t qa = blk + 16u + 64u * h;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 t = ld_s128(qa + 16u * j);
            q[4 * j] = t.x; q[4 * j + 1] = t.y; q[4 * j + 2] = t.z; q[4 * j + 3] = t.w;
        }
        const int sc0 = SC & 0xFF, sc1 = (SC >> 8) & 0xFF, sc2 = (SC >> 16) & 0xFF, sc3 = SC >> 24;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + ((static_cast<uint32_t>(v) * nb + b) * 2 + h) * kRecord;
            uint32_t a[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint4 t = ld_s128(rec + 16u * j);
                a[4 * j] = t.x; a[4 * j + 1] = t.y; a[4 * j + 2] = t.z; a[4 * j + 3] = t.w;
            }
            const uint4 ex = ld_s128(rec + 128);
            int d0 = 0, d1 = 0, d2 = 0, d3 = 0;  // d1, d3 carry a factor 16
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                d0 = dp4a(q[i] & 0x0F0F0F0Fu, a[i], d0);
                d1 = dp4a_us(q[i] & 0xF0F0F0F0u, a[8 + i], d1);
                d2 = dp4a(q[8 + i] & 0x0F0F0F0Fu, a[16 + i], d2);
                d3 = dp4a_us(q[8 + i] & 0xF0F0F0F0u, a[24 + i], d3);
            }
            int sq = ((sc0 * d0 + sc2 * d2) * 16 + sc1 * d1 + sc3 * d3) >> 4;  // exact: divisible by 16
            int sm = dp2a_hi_su(ex.y, M, dp2a_lo_su(ex.x, M, 0));
            if (ISUMS) {
                sq = group_sum<2>(sq);
                sm = group_sum<2>(sm);
                if (active && h == 0) {
                    isum_row[v * isum_vstride + 2 * b] = sq;
                    isum_row[v * isum_vstride + 2 * b + 1] = sm;
                }
            } else if (active) {
                const float dx = __uint_as_float(ex.z);
                acc[v] = fmaf(dx * dw, static_cast<float>(sq), acc[v]);
                acc[v] = fmaf(-(dx * dmin), static_cast<float>(sm), acc[v]);
            }
        }
    }
};

// ------------------------------------------------------------------------
// Q6_K. Two lanes per block: lane sub = h takes half h, i.e. the four
// 32-value rows k of ql[64h..64h+63] / qh[32h..32h+31] and the 16-value
// sub-blocks j = 8h + 2k + m (m = 0, 1). Its ql and qh runs are contiguous,
// so the 2-byte aligned block costs one extra word load and one funnel shift
// per word of the run. Activations staged per (vector, block, half) as a
// 176-byte record (codes 128h.. in order | int16 bsums 8h..8h+7 | f32 d_x).
// The -32 offset of q is applied through the bsums.
// ------------------------------------------------------------------------
struct TypeQ6_K {
    static constexpr int kBlockElems = 256, kBlockBytes = 210, kLanesPerBlock = 2, kSums = 1;
    static constexpr int kActValues = 256;
    // 176-byte records (44 words): 8 consecutive records' 128-bit loads fall
    // in 8 disjoint bank quads. Layout: codes 128h..128h+127 of the block in
    // order | bsums 8h..8h+7 (int16) at +128 | f32 d at +144.
    static constexpr int kRecord = 176;
    static size_t act_bytes(int nb, int nv) { return static_cast<size_t>(nv) * nb * 2 * kRecord; }

    // From byte-exact Q8_K blocks (292 B, 4-byte aligned): 8 16-byte units of
    // codes, then the bsums with d.
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        const int n = nb * nv * 2 * 9;
        for (int u = tid; u < n; u += nthr) {
            const int r = u / 9, part = u % 9;
            const int blk = r >> 1, h = r & 1;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + static_cast<size_t>(blk) * 292);
            uint4 *rec = reinterpret_cast<uint4 *>(act + static_cast<size_t>(r) * kRecord);
            if (part < 8) {
                const int w = 1 + 32 * h + 4 * part;  // codes start at byte 4
                rec[part] = make_uint4(__ldg(src + w), __ldg(src + w + 1), __ldg(src + w + 2), __ldg(src + w + 3));
            } else {
                const int w = 65 + 4 * h;  // bsums (int16) start at byte 260
                rec[8] = make_uint4(__ldg(src + w), __ldg(src + w + 1), __ldg(src + w + 2), __ldg(src + w + 3));
                reinterpret_cast<uint32_t *>(rec + 9)[0] = __ldg(src);
            }
        }
    }

    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        // lane l holds values 8l..8l+7: half h = l/16
        const int h = lane >> 4;
        stage_x_q8_k(x, count, warp, nwarps, lane, [&](int i, const uint32_t (&w)[2], int s16, float d) {
            uint8_t *rec = act + (static_cast<size_t>(i) * 2 + h) * kRecord;
            reinterpret_cast<uint2 *>(rec)[lane & 15] = make_uint2(w[0], w[1]);
            if ((lane & 1) == 0) reinterpret_cast<int16_t *>(rec + 128)[(lane & 15) >> 1] = static_cast<int16_t>(s16);
            if ((lane & 15) == 0) reinterpret_cast<float *>(rec + 144)[0] = d;
        }, loaded);
    }

    // Lane part h: element e = 128h + 32k + 16m + lam (sub-block j = 8h + 2k + m)
    // takes its low 4 bits from nibble k>>1 of ql[64h + 32(k&1) + 16m + lam] and
    // its high 2 bits from bits 2k of qh[32h + 16m + lam].
    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int sub, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;  // 2-byte aligned
        const uint32_t h = static_cast<uint32_t>(sub);
        uint32_t ql[16], qh[8], scw[2];
        ld_words_a2<16>(blk + 64u * h, ql);         // words 0..7: k = 0, 2; words 8..15: k = 1, 3
        ld_words_a2<8>(blk + 128u + 32u * h, qh);   // bits 2k..2k+1 of each byte: k
        ld_words_a2<2>(blk + 192u + 8u * h, scw);   // scales 8h..8h+7: byte 2k + m of the pair
        const float dw = f16_bits_to_f32(ld_s16(blk + 208u));
        uint32_t q[4][8];  // codes 0..63 of row k, words w = 0..7 (m = w / 4)
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            q[0][w] = (ql[w] & 0x0F0F0F0Fu) | ((qh[w] << 4) & 0x30303030u);
            q[1][w] = (ql[8 + w] & 0x0F0F0F0Fu) | ((qh[w] << 2) & 0x30303030u);
            q[2][w] = ((ql[w] >> 4) & 0x0F0F0F0Fu) | (qh[w] & 0x30303030u);
            q[3][w] = ((ql[8 + w] >> 4) & 0x0F0F0F0Fu) | ((qh[w] >> 2) & 0x30303030u);
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + ((static_cast<uint32_t>(v) * nb + b) * 2 + h) * kRecord;
            int s = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 a0 = ld_s128(rec + 32u * k), a1 = ld_s128(rec + 32u * k + 16u);
                const int d0 = dp4a(q[k][3], a0.w, dp4a(q[k][2], a0.z, dp4a(q[k][1], a0.y, dp4a(q[k][0], a0.x, 0))));
                const int d1 = dp4a(q[k][7], a1.w, dp4a(q[k][6], a1.z, dp4a(q[k][5], a1.y, dp4a(q[k][4], a1.x, 0))));
                s += sbyte(scw[k >> 1], 2 * (k & 1)) * d0 + sbyte(scw[k >> 1], 2 * (k & 1) + 1) * d1;
            }
            // the q - 32 offset: 32 * sum_j sc_j * bsum_j (int16 pairs times scale byte pairs)
            const uint4 bs = ld_s128(rec + 128u);
            int t = dp2a_lo_ss(bs.x, scw[0], 0);
            t = dp2a_hi_ss(bs.y, scw[0], t);
            t = dp2a_lo_ss(bs.z, scw[1], t);
            t = dp2a_hi_ss(bs.w, scw[1], t);
            s -= 32 * t;
            if (ISUMS) {
                s = group_sum<2>(s);
                if (active && h == 0) isum_row[v * isum_vstride + b] = s;
            } else if (active) {
                acc[v] = fmaf(static_cast<float>(s), dw * __uint_as_float(ld_s32(rec + 144u)), acc[v]);
            }
        }
    }
};

// ------------------------------------------------------------------------
// Q6_K, four lanes per block (for rows whose block count leaves the
// two-lane item's 16-block iterations partly empty): lane sub = 2h + p takes
// half h and the 16 positions l = 16p..16p+15 of each of the four 32-value
// rows k, i.e. the
// 16-value sub-blocks j_k = 8h + 2k + p (k = 0..3). Activations staged per
// (vector, block, sub) as an 80-byte record:
//   codes[64] (k-th 16 bytes = values 128h + 32k + 16p ..) |
//   int16 bsums[j_0..j_3] | f32 d_x | pad
// An 80-byte stride (20 words) puts 8 consecutive records' 128-bit loads in
// 8 disjoint bank quads. The -32 offset of q is applied through the bsums.
// ------------------------------------------------------------------------
struct TypeQ6_K4 {
    static constexpr int kBlockElems = 256, kBlockBytes = 210, kLanesPerBlock = 4, kSums = 1;
    static constexpr int kActValues = 256;
    static constexpr int kRecord = 80;
    static size_t act_bytes(int nb, int nv) { return static_cast<size_t>(nv) * nb * 4 * kRecord; }

    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        const int n = nb * nv * 4 * 5;
        for (int u = tid; u < n; u += nthr) {
            const int r = u / 5, part = u % 5;
            const int blk = r >> 2, sub = r & 3, h = sub >> 1, p = sub & 1;
            const uint8_t *src = xq + static_cast<size_t>(blk) * 292;
            uint4 *rec = reinterpret_cast<uint4 *>(act + static_cast<size_t>(r) * kRecord);
            if (part < 4) {
                const uint32_t *w = reinterpret_cast<const uint32_t *>(src + 4 + 128 * h + 32 * part + 16 * p);
                rec[part] = make_uint4(__ldg(w), __ldg(w + 1), __ldg(w + 2), __ldg(w + 3));
            } else {
                const int16_t *bs = reinterpret_cast<const int16_t *>(src + 260);
                int s[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) s[k] = __ldg(bs + 8 * h + 2 * k + p);
                rec[4] = make_uint4(pack16(s[0], s[1]), pack16(s[2], s[3]),
                                    __ldg(reinterpret_cast<const uint32_t *>(src)), 0u);
            }
        }
    }

    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        // lane l holds values 8l..8l+7: h = l/16, k = (l%16)/4, p = (l%4)/2
        const int h = lane >> 4, k = (lane >> 2) & 3, p = (lane >> 1) & 1;
        const int sub = 2 * h + p;
        stage_x_q8_k(x, count, warp, nwarps, lane, [&](int i, const uint32_t (&w)[2], int s16, float d) {
            uint8_t *rec = act + (static_cast<size_t>(i) * 4 + sub) * kRecord;
            reinterpret_cast<uint2 *>(rec + 16 * k)[lane & 1] = make_uint2(w[0], w[1]);
            if ((lane & 1) == 0) reinterpret_cast<int16_t *>(rec + 64)[k] = static_cast<int16_t>(s16);
            if (k == 0 && (lane & 1) == 0) reinterpret_cast<uint2 *>(rec + 72)[0] = make_uint2(__float_as_uint(d), 0u);
        }, loaded);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int sub, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;  // 2-byte aligned
        const uint32_t h = static_cast<uint32_t>(sub) >> 1, p = static_cast<uint32_t>(sub) & 1u;
        uint32_t ql0[4], ql1[4], qh[4], scw[2];
        ld_words_a2<4>(blk + 64u * h + 16u * p, ql0);
        ld_words_a2<4>(blk + 64u * h + 32u + 16u * p, ql1);
        ld_words_a2<4>(blk + 128u + 32u * h + 16u * p, qh);
        ld_words_a2<2>(blk + 192u + 8u * h, scw);  // scales[8h .. 8h+7]
        const float dw = f16_bits_to_f32(ld_s16(blk + 208u));
        // scales of sub-blocks 8h + 2k + p, k = 0..3, as 4 signed bytes
        const uint32_t SC = __byte_perm(scw[0], scw[1], p ? 0x7531u : 0x6420u);
        const int sc0 = sbyte(SC, 0), sc1 = sbyte(SC, 1), sc2 = sbyte(SC, 2), sc3 = sbyte(SC, 3);
        uint32_t qv[4][4];  // q (0..63) of the lane's 16 values of row k, 4 per word
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            qv[0][i] = (ql0[i] & 0x0F0F0F0Fu) | ((qh[i] << 4) & 0x30303030u);
            qv[1][i] = (ql1[i] & 0x0F0F0F0Fu) | ((qh[i] << 2) & 0x30303030u);
            qv[2][i] = ((ql0[i] >> 4) & 0x0F0F0F0Fu) | (qh[i] & 0x30303030u);
            qv[3][i] = ((ql1[i] >> 4) & 0x0F0F0F0Fu) | ((qh[i] >> 2) & 0x30303030u);
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + ((static_cast<uint32_t>(v) * nb + b) * 4 + sub) * kRecord;
            int dk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 a = ld_s128(rec + 16u * k);
                int s = dp4a(qv[k][0], a.x, 0);
                s = dp4a(qv[k][1], a.y, s);
                s = dp4a(qv[k][2], a.z, s);
                dk[k] = dp4a(qv[k][3], a.w, s);
            }
            const uint4 ex = ld_s128(rec + 64u);
            int s = sc0 * dk[0] + sc1 * dk[1] + sc2 * dk[2] + sc3 * dk[3];
            s -= 32 * dp2a_hi_ss(ex.y, SC, dp2a_lo_ss(ex.x, SC, 0));
            if (ISUMS) {
                s = group_sum<4>(s);
                if (active && sub == 0) isum_row[v * isum_vstride + b] = s;
            } else if (active) {
                acc[v] = fmaf(static_cast<float>(s), dw * __uint_as_float(ex.z), acc[v]);
            }
        }
    }
};

// ------------------------------------------------------------------------
// Q5_K (176-byte blocks, 16-byte aligned: f16 d, f16 dmin, scales[12] as
// Q4_K, qh[32], qs[128]). Two lanes per block as Q4_K, same activation
// record. The fifth bit of value l of sub-block j is bit j of qh[l]; it is
// merged into bit 4 of the code bytes (low- and high-nibble sub-blocks
// alike, so no factor 16 here).
// ------------------------------------------------------------------------
struct TypeQ5_K {
    static constexpr int kBlockElems = 256, kBlockBytes = 176, kLanesPerBlock = 2, kSums = 2;
    static constexpr int kActValues = 256;
    static constexpr int kRecord = TypeQ4_K::kRecord;
    static size_t act_bytes(int nb, int nv) { return TypeQ4_K::act_bytes(nb, nv); }
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        TypeQ4_K::stage_act(xq, act, nb, nv, tid, nthr);
    }
    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        TypeQ4_K::stage_x(x, act, count, warp, nwarps, lane, loaded);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int h, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;  // 16-byte aligned
        const uint4 hdr = ld_s128(blk);
        const float dw = f16_bits_to_f32(hdr.x);
        const float dmin = f16_bits_to_f32(hdr.x >> 16);
        const uint32_t SC = h == 0 ? (hdr.y & 0x3F3F3F3Fu)
                                   : ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u));
        const uint32_t M = h == 0 ? (hdr.z & 0x3F3F3F3Fu)
                                  : (((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u));
        // fifth bits of sub-blocks 4h..4h+3: bits 0..3 of each qh byte after the shift
        uint32_t qh[8];
        {
            const uint4 t0 = ld_s128(blk + 16u), t1 = ld_s128(blk + 32u);
            const uint32_t w[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) qh[i] = (w[i] >> (4 * h)) & 0x0F0F0F0Fu;
        }
        uint32_t c[4][8];  // 5-bit codes of sub-block 4h + s, 4 per word
        const uint32_t qa = blk + 48u + 64u * h;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 t = ld_s128(qa + 16u * j);
            const uint32_t q[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = 4 * (j & 1) + u;      // word of the 32-value run
                const int s0 = 2 * (j >> 1);        // low-nibble sub-block of this run
                c[s0][i] = (q[u] & 0x0F0F0F0Fu) | ((qh[i] << (4 - s0)) & 0x10101010u);
                c[s0 + 1][i] = ((q[u] >> 4) & 0x0F0F0F0Fu) | ((qh[i] << (3 - s0)) & 0x10101010u);
            }
        }
        const int sc0 = SC & 0xFF, sc1 = (SC >> 8) & 0xFF, sc2 = (SC >> 16) & 0xFF, sc3 = SC >> 24;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + ((static_cast<uint32_t>(v) * nb + b) * 2 + h) * kRecord;
            int d[4] = {0, 0, 0, 0};
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const uint4 a0 = ld_s128(rec + 32u * s), a1 = ld_s128(rec + 32u * s + 16u);
                int t = dp4a(c[s][0], a0.x, 0);
                t = dp4a(c[s][1], a0.y, t);
                t = dp4a(c[s][2], a0.z, t);
                t = dp4a(c[s][3], a0.w, t);
                t = dp4a(c[s][4], a1.x, t);
                t = dp4a(c[s][5], a1.y, t);
                t = dp4a(c[s][6], a1.z, t);
                d[s] = dp4a(c[s][7], a1.w, t);
            }
            const uint4 ex = ld_s128(rec + 128);
            int sq = sc0 * d[0] + sc1 * d[1] + sc2 * d[2] + sc3 * d[3];
            int sm = dp2a_hi_su(ex.y, M, dp2a_lo_su(ex.x, M, 0));
            if (ISUMS) {
                sq = group_sum<2>(sq);
                sm = group_sum<2>(sm);
                if (active && h == 0) {
                    isum_row[v * isum_vstride + 2 * b] = sq;
                    isum_row[v * isum_vstride + 2 * b + 1] = sm;
                }
            } else if (active) {
                const float dx = __uint_as_float(ex.z);
                acc[v] = fmaf(dx * dw, static_cast<float>(sq), acc[v]);
                acc[v] = fmaf(-(dx * dmin), static_cast<float>(sm), acc[v]);
            }
        }
    }
};

// ------------------------------------------------------------------------
// Q2_K (84-byte blocks, 4-byte aligned: scales[16] (scale | min << 4),
// qs[64], f16 d, f16 dmin). Two lanes per block: lane h takes values
// 128h..128h+127, i.e. qs[32h..32h+31] and the 16-value sub-blocks 8h..8h+7.
// Value 32j + 16hh + l of the half is bits 2j..2j+1 of byte 16hh + l of the
// lane's qs run, so word i of the run (hh = i / 4) holds, at shift 2j, the
// four codes that meet activation word 8j + i of the Q6_K-style record.
// ------------------------------------------------------------------------
struct TypeQ2_K {
    static constexpr int kBlockElems = 256, kBlockBytes = 84, kLanesPerBlock = 2, kSums = 2;
    static constexpr int kActValues = 256;
    static constexpr int kRecord = TypeQ6_K::kRecord;
    static size_t act_bytes(int nb, int nv) { return TypeQ6_K::act_bytes(nb, nv); }
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        TypeQ6_K::stage_act(xq, act, nb, nv, tid, nthr);
    }
    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        TypeQ6_K::stage_x(x, act, count, warp, nwarps, lane, loaded);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int h, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;  // 4-byte aligned
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = ld_s32(blk + 16u + 32u * h + 4u * i);
        const uint32_t sw0 = ld_s32(blk + 8u * h), sw1 = ld_s32(blk + 8u * h + 4u);
        const uint32_t dd = ld_s32(blk + 80u);
        const float dw = f16_bits_to_f32(dd), dmin = f16_bits_to_f32(dd >> 16);
        const uint32_t M0 = (sw0 >> 4) & 0x0F0F0F0Fu, M1 = (sw1 >> 4) & 0x0F0F0F0Fu;
        const uint32_t S0 = sw0 & 0x0F0F0F0Fu, S1 = sw1 & 0x0F0F0F0Fu;
        int sc[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            sc[k] = (S0 >> (8 * k)) & 0xFF;
            sc[4 + k] = (S1 >> (8 * k)) & 0xFF;
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + ((static_cast<uint32_t>(v) * nb + b) * 2 + h) * kRecord;
            int sq = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 a0 = ld_s128(rec + 32u * j), a1 = ld_s128(rec + 32u * j + 16u);
                // sub-blocks 2j (words 0..3) and 2j + 1 (words 4..7)
                int t0 = dp4a((q[0] >> (2 * j)) & 0x03030303u, a0.x, 0);
                t0 = dp4a((q[1] >> (2 * j)) & 0x03030303u, a0.y, t0);
                t0 = dp4a((q[2] >> (2 * j)) & 0x03030303u, a0.z, t0);
                t0 = dp4a((q[3] >> (2 * j)) & 0x03030303u, a0.w, t0);
                int t1 = dp4a((q[4] >> (2 * j)) & 0x03030303u, a1.x, 0);
                t1 = dp4a((q[5] >> (2 * j)) & 0x03030303u, a1.y, t1);
                t1 = dp4a((q[6] >> (2 * j)) & 0x03030303u, a1.z, t1);
                t1 = dp4a((q[7] >> (2 * j)) & 0x03030303u, a1.w, t1);
                sq += sc[2 * j] * t0 + sc[2 * j + 1] * t1;
            }
            // min term: sum over the 8 sub-blocks of m * bsum16
            const uint4 ex = ld_s128(rec + 128u);
            int sm = dp2a_lo_su(ex.x, M0, 0);
            sm = dp2a_hi_su(ex.y, M0, sm);
            sm = dp2a_lo_su(ex.z, M1, sm);
            sm = dp2a_hi_su(ex.w, M1, sm);
            if (ISUMS) {
                sq = group_sum<2>(sq);
                sm = group_sum<2>(sm);
                if (active && h == 0) {
                    isum_row[v * isum_vstride + 2 * b] = sq;
                    isum_row[v * isum_vstride + 2 * b + 1] = sm;
                }
            } else if (active) {
                const float dx = __uint_as_float(ld_s32(rec + 144u));
                acc[v] = fmaf(dx * dw, static_cast<float>(sq), acc[v]);
                acc[v] = fmaf(-(dx * dmin), static_cast<float>(sm), acc[v]);
            }
        }
    }
};

// Six-bit fields of each byte (0..63) minus 32, as signed bytes: b ^ 32
// flips the field's top bit, then that bit is copied into bits 6..7 (the
// product with 6 stays inside its byte).
__device__ __forceinline__ uint32_t bias32_to_s8x4(uint32_t b) {
    const uint32_t x = b ^ 0x20202020u;
    return x | ((x & 0x20202020u) * 6u);
}

// ------------------------------------------------------------------------
// Q3_K (110-byte blocks, 2-byte aligned: hmask[32], qs[64], scales[12],
// f16 d). Two lanes per block: lane h takes values 128h..128h+127 (qs bytes
// 32h.., bit 4h + j of hmask, sub-blocks 8h..8h+7). Codes enter as
// c = q2 + 4 * hbit in 0..7 (value c - 4); the -4 goes through the bsums.
// Sub-block scale = 6-bit field - 32: low 4 bits in nibble h of bytes
// 0..7, high 2 bits at bits 4h + 2(sb / 4) of byte 8 + sb % 4.
// ------------------------------------------------------------------------
struct TypeQ3_K {
    static constexpr int kBlockElems = 256, kBlockBytes = 110, kLanesPerBlock = 2, kSums = 1;
    static constexpr int kActValues = 256;
    static constexpr int kRecord = TypeQ6_K::kRecord;
    static size_t act_bytes(int nb, int nv) { return TypeQ6_K::act_bytes(nb, nv); }
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        TypeQ6_K::stage_act(xq, act, nb, nv, tid, nthr);
    }
    template <class Loaded>
    __device__ static void stage_x(const float *x, uint8_t *act, int count, int warp, int nwarps, int lane,
                                   Loaded loaded) {
        TypeQ6_K::stage_x(x, act, count, warp, nwarps, lane, loaded);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(uint32_t rowa, int b, int h, bool active, uint32_t acta, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint32_t blk = rowa + static_cast<uint32_t>(b) * kBlockBytes;  // 2-byte aligned
        uint32_t hm[8], q[8], sw[3];
        ld_words_a2<8>(blk, hm);
        ld_words_a2<8>(blk + 32u + 32u * h, q);
        ld_words_a2<3>(blk + 96u, sw);
        const float dw = f16_bits_to_f32(ld_s16(blk + 108u));
#pragma unroll
        for (int i = 0; i < 8; ++i) hm[i] = (hm[i] >> (4 * h)) & 0x0F0F0F0Fu;  // bit j: row j of this half
        // biased 6-bit scales of sub-blocks 8h..8h+3 and 8h+4..8h+7
        const uint32_t lo0 = (sw[0] >> (4 * h)) & 0x0F0F0F0Fu, lo1 = (sw[1] >> (4 * h)) & 0x0F0F0F0Fu;
        const uint32_t B0 = lo0 | (((sw[2] >> (4 * h)) & 0x03030303u) << 4);
        const uint32_t B1 = lo1 | (((sw[2] >> (4 * h + 2)) & 0x03030303u) << 4);
        const uint32_t SC0 = bias32_to_s8x4(B0), SC1 = bias32_to_s8x4(B1);
        int sc[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            sc[k] = sbyte(SC0, k);
            sc[4 + k] = sbyte(SC1, k);
        }
        uint32_t c[4][8];  // codes q2 + 4 hbit of row j, word i
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i)
                c[j][i] = ((q[i] >> (2 * j)) & 0x03030303u) | (j <= 2 ? ((hm[i] << (2 - j)) & 0x04040404u)
                                                                      : ((hm[i] >> 1) & 0x04040404u));
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint32_t rec = acta + ((static_cast<uint32_t>(v) * nb + b) * 2 + h) * kRecord;
            int s = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 a0 = ld_s128(rec + 32u * j), a1 = ld_s128(rec + 32u * j + 16u);
                int t0 = dp4a(c[j][0], a0.x, 0);
                t0 = dp4a(c[j][1], a0.y, t0);
                t0 = dp4a(c[j][2], a0.z, t0);
                t0 = dp4a(c[j][3], a0.w, t0);
                int t1 = dp4a(c[j][4], a1.x, 0);
                t1 = dp4a(c[j][5], a1.y, t1);
                t1 = dp4a(c[j][6], a1.z, t1);
                t1 = dp4a(c[j][7], a1.w, t1);
                s += sc[2 * j] * t0 + sc[2 * j + 1] * t1;
            }
            // the -4 offset: 4 * sum over sub-blocks of sc * bsum16
            const uint4 ex = ld_s128(rec + 128u);
            int t = dp2a_lo_ss(ex.x, SC0, 0);
            t = dp2a_hi_ss(ex.y, SC0, t);
            t = dp2a_lo_ss(ex.z, SC1, t);
            t = dp2a_hi_ss(ex.w, SC1, t);
            s -= 4 * t;
            if (ISUMS) {
                s = group_sum<2>(s);
                if (active && h == 0) isum_row[v * isum_vstride + b] = s;
            } else if (active) {
                acc[v] = fmaf(static_cast<float>(s), dw * __uint_as_float(ld_s32(rec + 144u)), acc[v]);
            }
        }
    }
};


}  // namespace qg
