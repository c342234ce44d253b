// gemv_types.cuh - per-type policies of the streaming GEMV kernel: how the
// paired activation blocks are laid out in shared memory, and how a group of
// lanes forms one weight block's exact int32 sums and float term.
//
// Block formats ("量化格式" (candle), block structure table; "Building Q8_0
// and Q4_0 Like ggml", Examples 1 and 5; "Quantization" (rml), Unpacking the
// packed fields):
//   Q8_0  34 B: f16 d, int8 qs[32]                          value q * d
//   Q4_0  18 B: f16 d, qs[16]; byte j = elem j | elem j+16 << 4, value (c - 8) * d
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
//   Q4_K: S_q = sum_j sc_j * sum_{i in j} q_i a_i ; S_m = sum_j m_j (bsum_2j + bsum_2j+1)
//   Q6_K: S = sum_j sc_j * sum_{i in j} q_i a_i - 32 * sum_j sc_j * bsum_j
// Float step per block: Q8_0, Q4_0, Q6_K: S * (d_w * d_x); Q4_K:
// d_x * (d_w * S_q - dmin * S_m).
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

// ========================================================================
// Q8_0-paired types (Q8_0, Q4_0): activations staged as 48-byte records
// per (vector, block): qs[32] | f32 d_x | int32 sum(qs) | 8 pad bytes.
// Record stride 48 B makes 8 consecutive blocks' 128-bit loads hit 8
// disjoint bank quads.
// ========================================================================
struct ActQ8_0 {
    static constexpr int kRecord = 48;
    static size_t bytes(int nb, int nv) { return static_cast<size_t>(nv) * nb * kRecord; }

    // xq: [nv][nb] byte-exact Q8_0 blocks (34 B, 2-byte aligned each).
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
};

struct TypeQ8_0 {
    static constexpr int kBlockElems = 32, kBlockBytes = 34, kLanesPerBlock = 1, kSums = 1;
    static size_t act_bytes(int nb, int nv) { return ActQ8_0::bytes(nb, nv); }
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        ActQ8_0::stage(xq, act, nb, nv, tid, nthr);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(const uint8_t *rowp, int b, int /*sub*/, bool active, const uint8_t *act,
                                int nb, float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint8_t *blk = rowp + b * kBlockBytes;
        const float dw = f16_bits_to_f32(lds_u16(blk));
        uint32_t w[8];
        lds_words_a2<8>(blk + 2, w);
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint8_t *rec = act + (static_cast<size_t>(v) * nb + b) * ActQ8_0::kRecord;
            const uint4 a0 = reinterpret_cast<const uint4 *>(rec)[0];
            const uint4 a1 = reinterpret_cast<const uint4 *>(rec)[1];
            const float dx = reinterpret_cast<const float *>(rec)[8];
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
                acc[v] += static_cast<float>(s) * (dw * dx);
            }
        }
    }
};

struct TypeQ4_0 {
    static constexpr int kBlockElems = 32, kBlockBytes = 18, kLanesPerBlock = 1, kSums = 1;
    static size_t act_bytes(int nb, int nv) { return ActQ8_0::bytes(nb, nv); }
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        ActQ8_0::stage(xq, act, nb, nv, tid, nthr);
    }

    template <int NV, bool ISUMS>
    __device__ static void item(const uint8_t *rowp, int b, int /*sub*/, bool active, const uint8_t *act,
                                int nb, float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint8_t *blk = rowp + b * kBlockBytes;
        const float dw = f16_bits_to_f32(lds_u16(blk));
        uint32_t q[4];
        lds_words_a2<4>(blk + 2, q);
        uint32_t lo[4], hi[4];  // codes of elements 4i.. and 16+4i..
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = q[i] & 0x0F0F0F0Fu;
            hi[i] = (q[i] >> 4) & 0x0F0F0F0Fu;
        }
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint8_t *rec = act + (static_cast<size_t>(v) * nb + b) * ActQ8_0::kRecord;
            const uint4 a0 = reinterpret_cast<const uint4 *>(rec)[0];
            const uint4 a1 = reinterpret_cast<const uint4 *>(rec)[1];
            const uint4 ex = reinterpret_cast<const uint4 *>(rec)[2];
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
                acc[v] += static_cast<float>(s) * (dw * __uint_as_float(ex.x));
            }
        }
    }
};

// ========================================================================
// Q4_K. Four lanes per block, lane c takes the 64-element chunk c: the 32
// bytes qs[32c..32c+31] hold sub-block 2c in their low nibbles and 2c+1 in
// their high nibbles. Activations staged per (vector, block, chunk) as an
// 80-byte record: a[64] | bsum(2c) | bsum(2c+1) | f32 d_x | pad, where
// bsum(j) = bsums[2j] + bsums[2j+1] is the sum of sub-block j's 32 codes.
// ========================================================================
struct TypeQ4_K {
    static constexpr int kBlockElems = 256, kBlockBytes = 144, kLanesPerBlock = 4, kSums = 2;
    static constexpr int kRecord = 80;
    static size_t act_bytes(int nb, int nv) { return static_cast<size_t>(nv) * nb * 4 * kRecord; }

    // xq: [nv][nb] byte-exact Q8_K blocks (292 B, 4-byte aligned).
    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        const int n = nb * nv * 4;
        for (int i = tid; i < n; i += nthr) {
            const int blk = i >> 2, c = i & 3;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + static_cast<size_t>(blk) * 292);
            uint4 *rec = reinterpret_cast<uint4 *>(act + static_cast<size_t>(i) * kRecord);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int w = 1 + 16 * c + 4 * j;  // qs start at byte 4
                rec[j] = make_uint4(__ldg(src + w), __ldg(src + w + 1), __ldg(src + w + 2), __ldg(src + w + 3));
            }
            // bsums (int16) at byte 260 = word 65: sub-blocks 2c, 2c+1 need bsums[4c..4c+3]
            const uint32_t p0 = __ldg(src + 65 + 2 * c), p1 = __ldg(src + 66 + 2 * c);
            const int bs0 = static_cast<int>(static_cast<int16_t>(p0 & 0xFFFFu)) +
                            static_cast<int>(static_cast<int16_t>(p0 >> 16));
            const int bs1 = static_cast<int>(static_cast<int16_t>(p1 & 0xFFFFu)) +
                            static_cast<int>(static_cast<int16_t>(p1 >> 16));
            rec[4] = make_uint4(static_cast<uint32_t>(bs0), static_cast<uint32_t>(bs1), __ldg(src), 0u);
        }
    }

    template <int NV, bool ISUMS>
    __device__ static void item(const uint8_t *rowp, int b, int c, bool active, const uint8_t *act, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint8_t *blk = rowp + b * kBlockBytes;  // 16-byte aligned (144 = 9 x 16)
        const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
        const float dw = f16_bits_to_f32(hdr.x);
        const float dmin = f16_bits_to_f32(hdr.x >> 16);
        // scales[0..3] = hdr.y, scales[4..7] = hdr.z, scales[8..11] = hdr.w.
        // Sub-block j < 4: sc = s[j] & 63, m = s[j+4] & 63. j >= 4 (jj = j-4):
        // sc = (s[j+4] & 15) | (s[jj] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4.
        int sc[2], mn[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = 2 * c + h;
            const int jj = j & 3;
            const uint32_t y8 = (hdr.y >> (8 * jj)) & 0xFFu;
            const uint32_t z8 = (hdr.z >> (8 * jj)) & 0xFFu;
            const uint32_t w8 = (hdr.w >> (8 * jj)) & 0xFFu;
            if (j < 4) {
                sc[h] = static_cast<int>(y8 & 63u);
                mn[h] = static_cast<int>(z8 & 63u);
            } else {
                sc[h] = static_cast<int>((w8 & 15u) | ((y8 >> 6) << 4));
                mn[h] = static_cast<int>((w8 >> 4) | ((z8 >> 6) << 4));
            }
        }
        const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
        const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
        const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint4 *rec = reinterpret_cast<const uint4 *>(
                act + ((static_cast<size_t>(v) * nb + b) * 4 + c) * kRecord);
            const uint4 a0 = rec[0], a1 = rec[1], a2 = rec[2], a3 = rec[3], ex = rec[4];
            const uint32_t a[16] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w,
                                    a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
            int lo = 0, hi = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                lo = dp4a(q[i] & 0x0F0F0F0Fu, a[i], lo);
                hi = dp4a((q[i] >> 4) & 0x0F0F0F0Fu, a[8 + i], hi);
            }
            int sq = sc[0] * lo + sc[1] * hi;
            int sm = mn[0] * static_cast<int>(ex.x) + mn[1] * static_cast<int>(ex.y);
            sq = group_sum<4>(sq);
            sm = group_sum<4>(sm);
            if (ISUMS) {
                if (active && c == 0) {
                    isum_row[v * isum_vstride + 2 * b] = sq;
                    isum_row[v * isum_vstride + 2 * b + 1] = sm;
                }
            } else if (active && c == 0) {
                const float dx = __uint_as_float(ex.z);
                acc[v] += dx * (dw * static_cast<float>(sq) - dmin * static_cast<float>(sm));
            }
        }
    }
};

// ========================================================================
// Q6_K. Eight lanes per block: lane (h, lq) = (sub >> 2, sub & 3) takes
// l = 8lq..8lq+7 of half h for all four k, i.e. 8 elements of each of the
// sub-blocks j_k = 8h + 2k + (lq >> 1). Activations staged as
//   qs records [nv][nb] x 320 B: segment s = 4h + k (elements 128h + 32k ..
//     +31) at 40 s, so a lane's 8-byte loads are conflict free;
//   extras [nv][nb] x 48 B: int16 bsums permuted so that position
//     8h + 4p + k holds bsums[8h + 2k + p], then f32 d_x at byte 32.
// The -32 offset of q is applied through the bsums: lanes with even lq
// subtract 32 * sum_k sc_k * bsum(j_k) for their four sub-blocks.
// ========================================================================
struct TypeQ6_K {
    static constexpr int kBlockElems = 256, kBlockBytes = 210, kLanesPerBlock = 8, kSums = 1;
    static constexpr int kQsRecord = 320, kExRecord = 48;
    static size_t act_bytes(int nb, int nv) {
        return static_cast<size_t>(nv) * nb * (kQsRecord + kExRecord);
    }

    __device__ static void stage_act(const uint8_t *xq, uint8_t *act, int nb, int nv, int tid, int nthr) {
        const int nblk = nb * nv;
        uint8_t *ex = act + static_cast<size_t>(nblk) * kQsRecord;
        for (int i = tid; i < nblk * 9; i += nthr) {
            const int blk = i / 9, s = i % 9;
            const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + static_cast<size_t>(blk) * 292);
            if (s < 8) {
                uint2 *dst = reinterpret_cast<uint2 *>(act + static_cast<size_t>(blk) * kQsRecord + 40 * s);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_uint2(__ldg(src + 1 + 8 * s + 2 * j), __ldg(src + 2 + 8 * s + 2 * j));
            } else {
                const int16_t *bs = reinterpret_cast<const int16_t *>(xq + static_cast<size_t>(blk) * 292 + 260);
                int16_t *dst = reinterpret_cast<int16_t *>(ex + static_cast<size_t>(blk) * kExRecord);
                for (int h = 0; h < 2; ++h)
                    for (int par = 0; par < 2; ++par)
                        for (int k = 0; k < 4; ++k) dst[8 * h + 4 * par + k] = __ldg(bs + 8 * h + 2 * k + par);
                reinterpret_cast<uint32_t *>(dst)[8] = __ldg(src);  // d_x
                reinterpret_cast<uint32_t *>(dst)[9] = 0u;
                reinterpret_cast<uint2 *>(dst)[5] = make_uint2(0u, 0u);
            }
        }
    }

    template <int NV, bool ISUMS>
    __device__ static void item(const uint8_t *rowp, int b, int sub, bool active, const uint8_t *act, int nb,
                                float (&acc)[NV], int32_t *isum_row, int64_t isum_vstride) {
        const uint8_t *blk = rowp + b * kBlockBytes;  // 2-byte aligned
        const int h = sub >> 2, lq = sub & 3, par = lq >> 1;
        uint32_t ql0[2], ql1[2], qh[2], scw[2];
        lds_words_a2<2>(blk + 64 * h + 8 * lq, ql0);
        lds_words_a2<2>(blk + 64 * h + 32 + 8 * lq, ql1);
        lds_words_a2<2>(blk + 128 + 32 * h + 8 * lq, qh);
        lds_words_a2<2>(blk + 192 + 8 * h, scw);  // scales[8h .. 8h+7]
        const float dw = f16_bits_to_f32(lds_u16(blk + 208));
        int sc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) sc[k] = sbyte(scw[k >> 1], 2 * (k & 1) + par);
        // q (0..63) of the lane's 8 elements for each k, 4 per word
        uint32_t qv[4][2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            qv[0][i] = (ql0[i] & 0x0F0F0F0Fu) | ((qh[i] << 4) & 0x30303030u);
            qv[1][i] = (ql1[i] & 0x0F0F0F0Fu) | ((qh[i] << 2) & 0x30303030u);
            qv[2][i] = ((ql0[i] >> 4) & 0x0F0F0F0Fu) | (qh[i] & 0x30303030u);
            qv[3][i] = ((ql1[i] >> 4) & 0x0F0F0F0Fu) | ((qh[i] >> 2) & 0x30303030u);
        }
        const uint8_t *exbase = act + static_cast<size_t>(NV) * nb * kQsRecord;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const size_t r = static_cast<size_t>(v) * nb + b;
            const uint8_t *rq = act + r * kQsRecord + 8 * lq;
            int part = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint2 a = *reinterpret_cast<const uint2 *>(rq + 40 * (4 * h + k));
                const int dk = dp4a(qv[k][1], a.y, dp4a(qv[k][0], a.x, 0));
                part += sc[k] * dk;
            }
            const uint8_t *re = exbase + r * kExRecord;
            if ((lq & 1) == 0) {
                const uint2 bw = *reinterpret_cast<const uint2 *>(re + 8 * (2 * h + par));
                const int bsum = sc[0] * static_cast<int>(static_cast<int16_t>(bw.x & 0xFFFFu)) +
                                 sc[1] * static_cast<int>(static_cast<int16_t>(bw.x >> 16)) +
                                 sc[2] * static_cast<int>(static_cast<int16_t>(bw.y & 0xFFFFu)) +
                                 sc[3] * static_cast<int>(static_cast<int16_t>(bw.y >> 16));
                part -= 32 * bsum;
            }
            part = group_sum<8>(part);
            if (ISUMS) {
                if (active && sub == 0) isum_row[v * isum_vstride + b] = part;
            } else if (active && sub == 0) {
                const float dx = *reinterpret_cast<const float *>(re + 32);
                acc[v] += static_cast<float>(part) * (dw * dx);
            }
        }
    }
};

}  // namespace qg
