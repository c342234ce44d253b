// gemv_mma.cuh - the block-quantized GEMV for several vectors on the tensor
// cores: Y[v][o] = sum over the blocks of row o of (exact sub-block sums) x
// (block scales), for the K-quant weights (Q2_K .. Q6_K) with Q8_K
// activations and the 32-element types (Q4_0, Q4_1, Q5_0, Q8_0) with Q8_0 /
// Q8_1 activations, the latter eight blocks at a time ("Quantization" (rml),
// Quantized dot products, K-quants; "How to Read ggml/GGUF" (sh), block
// layouts).
//
// Why tensor cores here. With n_vec vectors every weight code meets n_vec
// activation codes: the product is the dense contraction
// [16 rows x n_in] x [n_in x 8 vectors] per tile of rows, and the __dp4a form
// spends n_vec multiply instructions and activation loads per weight word.
// mma.sync m16n8k16 (f16 in, f32 accumulate) takes 16 rows x 16 codes x 8
// vectors per instruction. It stays exact:
//  * a weight code q (4 or 6 bits, unsigned) enters as the f16 whose bit
//    pattern is q -- the subnormal q * 2^-24 -- built from the block bytes
//    by one mask (Q4_K's high nibbles give 16q * 2^-24);
//  * an activation code (-127..127) is an exact f16;
//  * every product and every partial sum of one sub-block is an integer
//    times 2^-24 below 2^0, exact in the f32 accumulator;
// so the accumulator of a sub-block (32 codes for Q4_K, 16 for Q6_K, one
// block of a 32-element type) is its exact int32 sum times 2^-24 (times 16
// for Q4_K odd sub-blocks). The
// sub-block scales are then applied in f32 (an exact small integer times the
// accumulator), the minimum / offset terms come from one more small mma over
// the Q8_K block sums (bsums), and only d_w, dmin_w and d_x are inexact
// floats -- the same arithmetic as the scalar definition up to f32 rounding.
//
// Structure (one CTA = NW consumer warps + 1 or 2 producer warps, one CTA per SM):
//  * Work unit: a tile of 16 consecutive rows of one matrix. A CTA owns a
//    balanced contiguous range of the launch's tiles (matrices of a batch
//    numbered consecutively). Each tile is streamed as one or more chunks of
//    kb blocks of its 16 rows ("stages").
//  * The producer warp copies each stage into a ring slot with 1-D bulk
//    async copies (TMA engine, non-tensor form). A slot holds 4 groups of 4
//    stage rows, group q at q * gpitch, row j of a group at j * rpitch. When
//    a stage spans whole rows, a group's 4 rows are contiguous in W and
//    travel as one copy (4 requests a stage; each bulk request costs the
//    issuing thread on the order of 100 cycles); otherwise each row segment
//    is its own copy (16 requests: panel modes split them over two
//    producer warps). gpitch is 32 modulo 128 bytes and the mma rows are
//    mapped to stage rows so that the 4 rows read by one 16-lane phase of a
//    64-bit load lie in 4 different groups: their banks are distinct. A copy
//    takes the 16-byte aligned window covering its bytes; bytes of W past its
//    last 16-byte boundary are copied with plain loads.
//  * Activations: at the start of each matrix the consumers rebuild a panel
//    in shared memory from the Q8_K blocks -- per block the B fragments of
//    every mma in lane order (f16, or biased int8 when f16 does not fit),
//    the bsums operands of the correction mma, d_x and the block sums.
//  * Consumers (NW warps): warp w takes blocks w, w+NW, ... of each stage's
//    chunk for all 16 rows and accumulates the tile's partial outputs in
//    registers across the chunks. After the tile's last chunk every warp
//    stores its partials to the stage's partial buffer before releasing the
//    ring slot.
//  * Register mode (8 consumer warps, one chunk per tile): a reducer warp
//    waits for each stage's release (the consumers' partials are in), adds
//    the tile's NW partials in a fixed warp order (deterministic), writes y
//    and then frees the slot for the producer on a second mbarrier. Because
//    the producer refills a slot only after the reducer has seen its
//    previous release, no waiter can miss an mbarrier phase. The CTA's final
//    tile is added up by the last consumer warp to store its partials (same
//    warp order), so the end of a short launch waits for no other warp.
//  * Panel modes (16 consumer warps and 2 producer warps; a 19th warp would
//    leave too few registers): the last consumer warp to store its partials adds up every
//    tile. With the partial buffers doubled it first releases the ring slot,
//    so the refill does not wait.
//  * Full/empty mbarriers with bounded waits (about 1 s), as in the __dp4a
//    kernel; programmatic dependent launch: the producer streams W while the
//    previous kernel finishes, the consumers wait for it before reading the
//    activations.
#pragma once

#include "qg_common.cuh"

namespace qg {

// Where a warp's activation (B) fragments come from: a panel in shared
// memory built per matrix (f16, or biased int8 when f16 does not fit), or
// registers -- when every stage spans whole rows of at most 2 * NW blocks,
// warp w always takes blocks w and w + NW, so it loads their fragments once
// per matrix and shared memory holds only the ring.
enum MmaBMode : int { kMmaPanel16 = 0, kMmaPanel8 = 1, kMmaRegs = 2 };
constexpr int kMmaTileRows = 16;
constexpr int kMmaMaxStages = 8;
// mbarriers full[8], empty[8] | partial-buffer counters (64 bytes) | mbarriers reduced[8] | pad
constexpr int kMmaHeaderBytes = 2 * 8 * kMmaMaxStages + 4 * 2 * kMmaMaxStages + 8 * 2 * kMmaMaxStages;
constexpr int kMmaRecords = 8;              // fragment records per block
constexpr int kMmaTailBytes = 256 + 32 + 32;  // per block: correction operands, d_x[8], block sums[8]
// Bytes of one partial-output buffer: every consumer lane's 4 partial outputs.
__host__ __device__ constexpr int mma_red_bytes(int nw) { return nw * 32 * 16; }
constexpr int kMmaNvec = 8;                 // vectors per mma (the n of m16n8k16)

// Panel bytes per weight block: fragment records (lane order, 16 bytes a lane
// in f16, 8 in biased int8) then the tail.
__host__ __device__ constexpr int mma_rec_bytes(bool b16) { return kMmaRecords * 32 * (b16 ? 16 : 8) + kMmaTailBytes; }
__host__ __device__ constexpr int mma_frag_bytes(bool b16) { return kMmaRecords * 32 * (b16 ? 16 : 8); }

struct MmaMat {
    const uint8_t *W;   // [n_out][row_bytes], 16-byte aligned
    const uint8_t *xq;  // byte-exact Q8_K blocks [n_vec][nb]
    float *y;           // [n_vec][n_out]
    int64_t tile_base;  // launch-wide index of this matrix's first tile
    int n_out;
    int pad;
};

template <int MAXB>
struct MmaBatch {
    MmaMat m[MAXB];
};

struct MmaParams {
    int32_t *err;         // device error word
    int64_t row_bytes;    // bytes of one row
    int64_t total_tiles;  // tiles of all matrices
    int n_mats;
    int nb;               // blocks per row
    int nv;               // vectors (1..8)
    int kb;               // blocks per chunk
    int n_chunks;         // chunks per row: ceil(nb / kb)
    int rpitch;           // bytes between the rows of a group in a slot
    int gpitch;           // bytes between the 4 row groups of a slot (32 mod 128)
    int contig;           // 1: a stage spans whole rows (one copy per group)
    int stage_bytes;      // 4 * gpitch
    int n_stages;         // ring depth (2..kMmaMaxStages)
    int red_slots;        // partial-output buffers: n_stages, or 2 * n_stages (then the
                          // warp that adds a tile's partials releases the slot first)
    int rec_bytes;        // panel bytes per block
    int panel_bytes;      // nb * rec_bytes
};

struct MmaStage {
    int mat, tile, kc;
    bool last;  // the tile's last chunk
};

// Stage row of mma row r (0..15): rows r and r+4... of one 16-lane load
// phase (r = 0..3, 4..7, 8..11, 12..15) fall in the 4 different groups.
__device__ __forceinline__ int mma_stage_row(int r) { return 4 * (r & 3) + ((r >> 2) & 1) + 2 * (r >> 3); }

// Walks a CTA's tiles, each as n_chunks stages. Producer and consumers run
// the same walk.
struct MmaWalk {
    int64_t t, t1;
    int m, kc;
    int64_t base, next_base;  // tile_base of matrices m and m+1 (cached: the table is kernel parameters)

    template <int MAXB>
    __device__ __forceinline__ bool next(const MmaBatch<MAXB> &b, const MmaParams &p, MmaStage &s) {
        if (t >= t1) return false;
        while (t >= next_base) {
            ++m;
            base = next_base;
            next_base = m + 1 < p.n_mats ? b.m[m + 1].tile_base : INT64_MAX;
        }
        s.mat = m;
        s.tile = static_cast<int>(t - base);
        s.kc = kc;
        s.last = kc == p.n_chunks - 1;
        if (++kc == p.n_chunks) {
            kc = 0;
            ++t;
        }
        return true;
    }
};

template <int MAXB>
__device__ __forceinline__ MmaWalk mma_cta_walk(const MmaParams &p, const MmaBatch<MAXB> &b) {
    MmaWalk w;
    w.t = static_cast<int64_t>(blockIdx.x) * p.total_tiles / gridDim.x;
    w.t1 = static_cast<int64_t>(blockIdx.x + 1) * p.total_tiles / gridDim.x;
    w.m = 0;
    w.kc = 0;
    w.base = 0;
    w.next_base = p.n_mats > 1 ? b.m[1].tile_base : INT64_MAX;
    return w;
}

// ------------------------------------------------------------ mma wrappers
// D += A (16x16, rows g and g+8 of lane 4g+t hold columns 2t,2t+1 and
// 2t+8,2t+9) x B (16x8, column g holds rows 2t,2t+1 and 2t+8,2t+9), f16 in,
// f32 accumulate; d[0..3] = D[g][2t], D[g][2t+1], D[g+8][2t], D[g+8][2t+1].
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// D = A x B + C with C given apart from D.
__device__ __forceinline__ void mma_16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                            uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}
// The k = 8 form: a0/a1 = rows g/g+8, columns 2t,2t+1; b0 = rows 2t,2t+1 of column g.
__device__ __forceinline__ void mma_1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(b0));
}

// Two f16 lanes minus the two f16 lanes of c.
__device__ __forceinline__ uint32_t hsub2c(uint32_t h, uint32_t c) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(c));
    return r;
}

// Two f16 lanes minus 1152 each (exact for the integers used here).
__device__ __forceinline__ uint32_t hsub1152(uint32_t h) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}

// The B fragments of record r for this lane: b[0], b[1] for the record's
// first mma, b[2], b[3] for its second (HI: the second run divided by 16).
template <bool B16, bool HI = false>
__device__ __forceinline__ void mma_load_b(uint32_t rec, int r, int lane, uint32_t (&b)[4]) {
    if (B16) {
        const uint4 v = ld_s128(rec + static_cast<uint32_t>((r * 32 + lane) * 16));
        b[0] = v.x;
        b[1] = v.y;
        b[2] = v.z;
        b[3] = v.w;
    } else {
        // biased bytes c = a + 128 -> f16 (1024 + c) by placing 0x64 above
        // each byte, then subtract 1152
        const uint2 v = ld_s64(rec + static_cast<uint32_t>((r * 32 + lane) * 8));
        b[0] = hsub1152(__byte_perm(v.x, 0x64646464u, 0x4140));
        b[1] = hsub1152(__byte_perm(v.x, 0x64646464u, 0x4342));
        if constexpr (HI) {
            // under 0x54 a byte c is the f16 64 + c/16 (steps of 1/16 in
            // [64, 128)); minus 72 gives (c - 128)/16
            b[2] = hsub2c(__byte_perm(v.y, 0x54545454u, 0x4140), 0x54805480u);
            b[3] = hsub2c(__byte_perm(v.y, 0x54545454u, 0x4342), 0x54805480u);
        } else {
            b[2] = hsub1152(__byte_perm(v.y, 0x64646464u, 0x4140));
            b[3] = hsub1152(__byte_perm(v.y, 0x64646464u, 0x4342));
        }
    }
}

__device__ __forceinline__ uint32_t mma_pack(unsigned short lo, unsigned short hi) {
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// A warp's B operands for one weight block: the fragments of record r
// (b(r, .)), the correction operand of the lane and d_x / block sums of
// vectors 2t, 2t+1 -- read from the shared-memory panel ...
template <bool B16, bool HI = false>
struct MmaSmemB {
    uint32_t rec;
    int lane;
    __device__ __forceinline__ void b(int r, uint32_t (&bf)[4]) const { mma_load_b<B16, HI>(rec, r, lane, bf); }
    __device__ __forceinline__ uint32_t corr32() const { return ld_s32(rec + mma_frag_bytes(B16) + 8 * lane); }
    __device__ __forceinline__ uint2 corr64() const { return ld_s64(rec + mma_frag_bytes(B16) + 8 * lane); }
    __device__ __forceinline__ uint2 dxw(int t) const { return ld_s64(rec + mma_frag_bytes(B16) + 256 + 8 * t); }
    __device__ __forceinline__ uint2 bsw(int t) const { return ld_s64(rec + mma_frag_bytes(B16) + 288 + 8 * t); }
    // groups of 32-element blocks: the tail float4 of record r and lane t
    __device__ __forceinline__ uint4 tail(int r, int t) const {
        return ld_s128(rec + mma_frag_bytes(B16) + static_cast<uint32_t>(64 * r + 16 * t));
    }
};

// ... or held in registers (f16 fragments).
struct MmaRegB {
    const uint32_t (&r)[kMmaRecords][4];
    uint2 corr, dx, bs;
    __device__ __forceinline__ void b(int i, uint32_t (&bf)[4]) const {
        bf[0] = r[i][0];
        bf[1] = r[i][1];
        bf[2] = r[i][2];
        bf[3] = r[i][3];
    }
    __device__ __forceinline__ uint32_t corr32() const { return corr.x; }
    __device__ __forceinline__ uint2 corr64() const { return corr; }
    __device__ __forceinline__ uint2 dxw(int) const { return dx; }
    __device__ __forceinline__ uint2 bsw(int) const { return bs; }
};

// ------------------------------------------------------------------ Q4_K
// Block: f16 d, f16 dmin, 12 bytes of packed 6-bit scales and mins, 128 bytes
// of nibbles (element 64c + l: low nibble of qs[32c + l], element 64c+32+l:
// high nibble). Sub-block j = 2c + n (n = nibble) has scale sc_j, min m_j.
// Lane (g, t) reads 8 bytes qs[32c + 8t ..] of rows g and g+8; mma (j, u)
// takes its words u: f16 lanes of bytes 0,2 (k-slots 2t, 2t+1) and 1,3
// (slots 2t+8, 2t+9). The panel's record j holds the matching activation
// codes 32j + 8t + {0,2,1,3, 4,6,5,7} of vector g.
struct MmaQ4_K {
    static constexpr int kBlockBytes = 144;
    static constexpr int kActBytes = 0;  // activations: Q8_K blocks (the panel's bsums tail)
    static constexpr bool kHiScaled = false;

    // Element offsets (within the block) of the two 4-code runs of record r
    // for lane t; the run is permuted to slots {0,2,1,3}.
    __device__ static int run0(int r, int t) { return 32 * r + 8 * t; }
    __device__ static int run1(int r, int t) { return 32 * r + 8 * t + 4; }

    // Correction operand of lane (g, t): the 32-code sums of sub-blocks 2t
    // and 2t+1 of vector g (k = 8 mma over the 8 sub-blocks).
    __device__ static void corr(const int16_t *bs, int t, float (&c)[4]) {
        c[0] = static_cast<float>(bs[4 * t] + bs[4 * t + 1]);
        c[1] = static_cast<float>(bs[4 * t + 2] + bs[4 * t + 3]);
        c[2] = 0.0f;
        c[3] = 0.0f;
    }

    template <class BS>
    __device__ __forceinline__ static void tile_block(uint32_t ra, uint32_t rb, const BS &B, int lane,
                                                      float (&acc)[4]) {
        const int t = lane & 3;
        const uint4 ha = ld_s128(ra), hb = ld_s128(rb);
        // scales (bytes 0..3: sub-blocks 0..3, 4..7: sub-blocks 4..7) and mins
        const uint32_t sca0 = ha.y & 0x3F3F3F3Fu, sca1 = (ha.w & 0x0F0F0F0Fu) | ((ha.y >> 2) & 0x30303030u);
        const uint32_t scb0 = hb.y & 0x3F3F3F3Fu, scb1 = (hb.w & 0x0F0F0F0Fu) | ((hb.y >> 2) & 0x30303030u);
        const uint32_t ma0 = ha.z & 0x3F3F3F3Fu, ma1 = ((ha.w >> 4) & 0x0F0F0F0Fu) | ((ha.z >> 2) & 0x30303030u);
        const uint32_t mb0 = hb.z & 0x3F3F3F3Fu, mb1 = ((hb.w >> 4) & 0x0F0F0F0Fu) | ((hb.z >> 2) & 0x30303030u);
        // min term: sum_j m_j * bsum32_j (m as subnormal f16 bits: m * 2^-24)
        const uint32_t msel = (t & 1) ? 0x4342u : 0x4140u;
        float m2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_1688(m2, __byte_perm(t < 2 ? ma0 : ma1, 0u, msel), __byte_perm(t < 2 ? mb0 : mb1, 0u, msel), B.corr32());
        float2 Ta = make_float2(0.0f, 0.0f), Tb = make_float2(0.0f, 0.0f);  // rows g, g+8
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const uint2 wa = ld_s64(ra + 16 + 32 * c + 8 * t), wb = ld_s64(rb + 16 + 32 * c + 8 * t);
            const uint32_t sa0 = wa.x >> 8, sa1 = wa.y >> 8, sb0 = wb.x >> 8, sb1 = wb.y >> 8;
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int j = 2 * c + n;
                const uint32_t M = n ? 0x00F000F0u : 0x000F000Fu;
                uint32_t bf[4];
                B.b(j, bf);
                float C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                mma_16816(C, wa.x & M, wb.x & M, sa0 & M, sb0 & M, bf[0], bf[1]);
                mma_16816(C, wa.y & M, wb.y & M, sa1 & M, sb1 & M, bf[2], bf[3]);
                // the two rows' scales of sub-block j: byte j&3 placed in the
                // mantissa of 2^23 (even j) or 2^19 (odd j: the high nibbles
                // carry a factor 16), then the power of two subtracted
                const uint32_t swa = j < 4 ? sca0 : sca1, swb = j < 4 ? scb0 : scb1;
                const uint32_t hi = n ? 0x49000000u : 0x4B000000u;
                const float off = n ? -524288.0f : -8388608.0f;
                const float2 f = fadd2(make_float2(__uint_as_float(__byte_perm(swa, hi, 0x7540u | (j & 3))),
                                                   __uint_as_float(__byte_perm(swb, hi, 0x7540u | (j & 3)))),
                                       make_float2(off, off));
                Ta = ffma2(make_float2(f.x, f.x), make_float2(C[0], C[1]), Ta);
                Tb = ffma2(make_float2(f.y, f.y), make_float2(C[2], C[3]), Tb);
            }
        }
        // block value = d_x * 2^24 * (d * T - dmin * m2)
        const float da = f16_bits_to_f32(ha.x) * 16777216.0f, dma = f16_bits_to_f32(ha.x >> 16) * -16777216.0f;
        const float db = f16_bits_to_f32(hb.x) * 16777216.0f, dmb = f16_bits_to_f32(hb.x >> 16) * -16777216.0f;
        const uint2 dxw = B.dxw(t);
        const float2 dx = make_float2(__uint_as_float(dxw.x), __uint_as_float(dxw.y));
        const float2 ua = ffma2(make_float2(da, da), Ta, make_float2(dma * m2[0], dma * m2[1]));
        const float2 ub = ffma2(make_float2(db, db), Tb, make_float2(dmb * m2[2], dmb * m2[3]));
        float2 acc01 = ffma2(dx, ua, make_float2(acc[0], acc[1]));
        float2 acc23 = ffma2(dx, ub, make_float2(acc[2], acc[3]));
        acc[0] = acc01.x;
        acc[1] = acc01.y;
        acc[2] = acc23.x;
        acc[3] = acc23.y;
    }
};

// ------------------------------------------------------------------ Q5_K
// Block: f16 d, f16 dmin, Q4_K's 12 scale/min bytes, qh[32], then Q4_K's 128
// bytes of nibbles (176 bytes, 16-byte aligned). The fifth bit of element
// e = 64c + 32n + l (sub-block j = 2c + n) is bit j of qh[l] ("量化格式"
// (candle), block structure table: Q5_K carries Q4_K's fields plus qh).
// Lane (g, t) reads the nibbles of Q4_K's lane and qh[8t .. 8t + 7], the
// fifth bits of the same positions, so the activation panel, its runs and
// the min term are Q4_K's. Both nibbles become plain 5-bit codes (the high
// nibble shifted down, the fifth bit moved to bit 4 of each byte), so every
// sub-block's scale takes the factor 2^23 and the sums stay exact: 32 codes
// below 32 times activations of at most 127 is below 2^17 units of 2^-24.
struct MmaQ5_K : MmaQ4_K {
    static constexpr int kBlockBytes = 176;

    // Bit j of each byte of w, moved to bit 4 of the byte.
    template <int J>
    __device__ __forceinline__ static uint32_t fifth(uint32_t w) {
        return (J <= 4 ? (w << (4 - J)) : (w >> (J - 4))) & 0x10101010u;
    }

    template <int C, int N, class BS>
    __device__ __forceinline__ static void sub_block(uint2 wa, uint2 wb, uint2 qa, uint2 qb, uint32_t swa,
                                                     uint32_t swb, const BS &B, float2 &Ta, float2 &Tb) {
        constexpr int J = 2 * C + N;
        // 5-bit codes, one a byte: nibble N of each qs byte | fifth bit J of the qh byte
        const uint32_t ca0 = ((N ? wa.x >> 4 : wa.x) & 0x0F0F0F0Fu) | fifth<J>(qa.x);
        const uint32_t ca1 = ((N ? wa.y >> 4 : wa.y) & 0x0F0F0F0Fu) | fifth<J>(qa.y);
        const uint32_t cb0 = ((N ? wb.x >> 4 : wb.x) & 0x0F0F0F0Fu) | fifth<J>(qb.x);
        const uint32_t cb1 = ((N ? wb.y >> 4 : wb.y) & 0x0F0F0F0Fu) | fifth<J>(qb.y);
        uint32_t bf[4];
        B.b(J, bf);
        float C4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        // bytes 0,2 and bytes 1,3 of each word as the f16 subnormal bits of two lanes
        mma_16816(C4, ca0 & 0x00FF00FFu, cb0 & 0x00FF00FFu, __byte_perm(ca0, 0u, 0x4341u),
                  __byte_perm(cb0, 0u, 0x4341u), bf[0], bf[1]);
        mma_16816(C4, ca1 & 0x00FF00FFu, cb1 & 0x00FF00FFu, __byte_perm(ca1, 0u, 0x4341u),
                  __byte_perm(cb1, 0u, 0x4341u), bf[2], bf[3]);
        // the two rows' scales of sub-block J: byte J&3 in the mantissa of 2^23
        const float2 f = fadd2(make_float2(__uint_as_float(__byte_perm(swa, 0x4B000000u, 0x7540u | (J & 3))),
                                           __uint_as_float(__byte_perm(swb, 0x4B000000u, 0x7540u | (J & 3)))),
                               make_float2(-8388608.0f, -8388608.0f));
        Ta = ffma2(make_float2(f.x, f.x), make_float2(C4[0], C4[1]), Ta);
        Tb = ffma2(make_float2(f.y, f.y), make_float2(C4[2], C4[3]), Tb);
    }

    template <int C, class BS>
    __device__ __forceinline__ static void chunk(uint32_t ra, uint32_t rb, int t, uint2 qa, uint2 qb, uint32_t sca0,
                                                 uint32_t sca1, uint32_t scb0, uint32_t scb1, const BS &B, float2 &Ta,
                                                 float2 &Tb) {
        const uint2 wa = ld_s64(ra + 48 + 32 * C + 8 * t), wb = ld_s64(rb + 48 + 32 * C + 8 * t);
        sub_block<C, 0>(wa, wb, qa, qb, C < 2 ? sca0 : sca1, C < 2 ? scb0 : scb1, B, Ta, Tb);
        sub_block<C, 1>(wa, wb, qa, qb, C < 2 ? sca0 : sca1, C < 2 ? scb0 : scb1, B, Ta, Tb);
    }

    template <class BS>
    __device__ __forceinline__ static void tile_block(uint32_t ra, uint32_t rb, const BS &B, int lane,
                                                      float (&acc)[4]) {
        const int t = lane & 3;
        const uint4 ha = ld_s128(ra), hb = ld_s128(rb);
        // scales and mins exactly as Q4_K
        const uint32_t sca0 = ha.y & 0x3F3F3F3Fu, sca1 = (ha.w & 0x0F0F0F0Fu) | ((ha.y >> 2) & 0x30303030u);
        const uint32_t scb0 = hb.y & 0x3F3F3F3Fu, scb1 = (hb.w & 0x0F0F0F0Fu) | ((hb.y >> 2) & 0x30303030u);
        const uint32_t ma0 = ha.z & 0x3F3F3F3Fu, ma1 = ((ha.w >> 4) & 0x0F0F0F0Fu) | ((ha.z >> 2) & 0x30303030u);
        const uint32_t mb0 = hb.z & 0x3F3F3F3Fu, mb1 = ((hb.w >> 4) & 0x0F0F0F0Fu) | ((hb.z >> 2) & 0x30303030u);
        const uint32_t msel = (t & 1) ? 0x4342u : 0x4140u;
        float m2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_1688(m2, __byte_perm(t < 2 ? ma0 : ma1, 0u, msel), __byte_perm(t < 2 ? mb0 : mb1, 0u, msel), B.corr32());
        const uint2 qa = ld_s64(ra + 16 + 8 * t), qb = ld_s64(rb + 16 + 8 * t);  // qh[8t .. 8t + 7]
        float2 Ta = make_float2(0.0f, 0.0f), Tb = make_float2(0.0f, 0.0f);  // rows g, g+8
        chunk<0>(ra, rb, t, qa, qb, sca0, sca1, scb0, scb1, B, Ta, Tb);
        chunk<1>(ra, rb, t, qa, qb, sca0, sca1, scb0, scb1, B, Ta, Tb);
        chunk<2>(ra, rb, t, qa, qb, sca0, sca1, scb0, scb1, B, Ta, Tb);
        chunk<3>(ra, rb, t, qa, qb, sca0, sca1, scb0, scb1, B, Ta, Tb);
        // block value = d_x * 2^24 * (d * T - dmin * m2)
        const float da = f16_bits_to_f32(ha.x) * 16777216.0f, dma = f16_bits_to_f32(ha.x >> 16) * -16777216.0f;
        const float db = f16_bits_to_f32(hb.x) * 16777216.0f, dmb = f16_bits_to_f32(hb.x >> 16) * -16777216.0f;
        const uint2 dxw = B.dxw(t);
        const float2 dx = make_float2(__uint_as_float(dxw.x), __uint_as_float(dxw.y));
        const float2 ua = ffma2(make_float2(da, da), Ta, make_float2(dma * m2[0], dma * m2[1]));
        const float2 ub = ffma2(make_float2(db, db), Tb, make_float2(dmb * m2[2], dmb * m2[3]));
        float2 acc01 = ffma2(dx, ua, make_float2(acc[0], acc[1]));
        float2 acc23 = ffma2(dx, ub, make_float2(acc[2], acc[3]));
        acc[0] = acc01.x;
        acc[1] = acc01.y;
        acc[2] = acc23.x;
        acc[3] = acc23.y;
    }
};

// ------------------------------------------------------------------ Q6_K
// Block: ql[128], qh[64], int8 scales[16], f16 d (the 210 bytes start
// 2-byte aligned). Element e = 128h + 32k + 16m + lam (sub-block
// j = 8h + 2k + m = e / 16): low 4 bits from nibble k>>1 of
// ql[64h + 32(k&1) + 16m + lam], high 2 bits from bits 2k of
// qh[32h + 16m + lam]; value d * sc_j * (q - 32). Lane (g, t) takes
// lam = 4t..4t+3 of every sub-block: bytes 0,2 -> k-slots 2t, 2t+1, bytes
// 1,3 -> slots 2t+8, 2t+9. Record i of the panel holds activation codes
// 32i + 4t + {0,2,1,3} (sub-block 2i) and 32i + 16 + 4t + {0,2,1,3}
// (sub-block 2i+1) of vector g.
struct MmaQ6_K {
    static constexpr int kBlockBytes = 210;
    static constexpr int kActBytes = 0;  // activations: Q8_K blocks (the panel's bsums tail)
    static constexpr bool kHiScaled = false;

    __device__ static int run0(int r, int t) { return 32 * r + 4 * t; }
    __device__ static int run1(int r, int t) { return 32 * r + 16 + 4 * t; }

    // Correction operand of lane (g, t): bsums 2t, 2t+1, 2t+8, 2t+9 of
    // vector g (k = 16 mma over the 16 sub-blocks).
    __device__ static void corr(const int16_t *bs, int t, float (&c)[4]) {
        c[0] = static_cast<float>(bs[2 * t]);
        c[1] = static_cast<float>(bs[2 * t + 1]);
        c[2] = static_cast<float>(bs[2 * t + 8]);
        c[3] = static_cast<float>(bs[2 * t + 9]);
    }

    // The 4 codes q = low nibble | 2 high bits << 4 of one word (one code a
    // byte); the mma operands take bytes 0,2 and bytes 1,3 of it as the
    // f16 subnormal bits of two lanes.
    __device__ __forceinline__ static uint32_t codes(uint32_t ql, uint32_t qh, int k) {
        const uint32_t lo = (ql >> (4 * (k >> 1))) & 0x0F0F0F0Fu;
        const uint32_t hi = k < 2 ? qh << (4 - 2 * k) : qh >> (2 * k - 4);  // bits 2k, 2k+1 to 4, 5
        return lo | (hi & 0x30303030u);
    }
    __device__ __forceinline__ static uint32_t even(uint32_t c) { return c & 0x00FF00FFu; }
    __device__ __forceinline__ static uint32_t odd(uint32_t c) { return __byte_perm(c, 0u, 0x4341u); }

    template <class BS>
    __device__ __forceinline__ static void tile_block(uint32_t ra, uint32_t rb, const BS &B, int lane,
                                                      float (&acc)[4]) {
        const int t = lane & 3;
        // scales as biased bytes sc + 128
        uint32_t swa[4], swb[4];
        ld_words_a2<4>(ra + 192, swa);
        ld_words_a2<4>(rb + 192, swb);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            swa[i] ^= 0x80808080u;
            swb[i] ^= 0x80808080u;
        }
        // offset term: sum_j (sc_j + 128) * bsum16_j (subnormal bits)
        const uint32_t ssel = (t & 1) ? 0x4342u : 0x4140u;
        const uint2 cw = B.corr64();
        float mq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_16816(mq, __byte_perm(t < 2 ? swa[0] : swa[1], 0u, ssel), __byte_perm(t < 2 ? swb[0] : swb[1], 0u, ssel),
                  __byte_perm(t < 2 ? swa[2] : swa[3], 0u, ssel), __byte_perm(t < 2 ? swb[2] : swb[3], 0u, ssel),
                  cw.x, cw.y);
        float2 Ta = make_float2(0.0f, 0.0f), Tb = make_float2(0.0f, 0.0f);  // rows g, g+8
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t qla[2][2], qlb[2][2], qha[2], qhb[2];  // [m][k & 1], [m]
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                uint32_t w[1];
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    ld_words_a2<1>(ra + 64 * h + 32 * kk + 16 * m + 4 * t, w);
                    qla[m][kk] = w[0];
                    ld_words_a2<1>(rb + 64 * h + 32 * kk + 16 * m + 4 * t, w);
                    qlb[m][kk] = w[0];
                }
                ld_words_a2<1>(ra + 128 + 32 * h + 16 * m + 4 * t, w);
                qha[m] = w[0];
                ld_words_a2<1>(rb + 128 + 32 * h + 16 * m + 4 * t, w);
                qhb[m] = w[0];
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t bf[4];
                B.b(4 * h + k, bf);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int j = 8 * h + 2 * k + m;
                    const uint32_t ca = codes(qla[m][k & 1], qha[m], k), cb = codes(qlb[m][k & 1], qhb[m], k);
                    float C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    mma_16816(C, even(ca), even(cb), odd(ca), odd(cb), bf[2 * m], bf[2 * m + 1]);
                    const float2 f = fadd2(
                        make_float2(__uint_as_float(__byte_perm(swa[j >> 2], 0x4B000000u, 0x7540u | (j & 3))),
                                    __uint_as_float(__byte_perm(swb[j >> 2], 0x4B000000u, 0x7540u | (j & 3)))),
                        make_float2(-8388736.0f, -8388736.0f));
                    Ta = ffma2(make_float2(f.x, f.x), make_float2(C[0], C[1]), Ta);
                    Tb = ffma2(make_float2(f.y, f.y), make_float2(C[2], C[3]), Tb);
                }
            }
        }
        // block value = d * d_x * 2^24 * (T - 32 mq + 2^-12 * block sum)
        const float da = f16_bits_to_f32(ld_s16(ra + 208)) * 16777216.0f;
        const float db = f16_bits_to_f32(ld_s16(rb + 208)) * 16777216.0f;
        const uint2 dxw = B.dxw(t);
        const uint2 bsw = B.bsw(t);
        const float dx0 = __uint_as_float(dxw.x), dx1 = __uint_as_float(dxw.y);
        const float2 bs = make_float2(__uint_as_float(bsw.x), __uint_as_float(bsw.y));
        const float2 q4 = make_float2(0.000244140625f, 0.000244140625f), m32 = make_float2(-32.0f, -32.0f);
        const float2 ea = ffma2(q4, bs, ffma2(m32, make_float2(mq[0], mq[1]), Ta));
        const float2 eb = ffma2(q4, bs, ffma2(m32, make_float2(mq[2], mq[3]), Tb));
        const float2 acc01 = ffma2(make_float2(da * dx0, da * dx1), ea, make_float2(acc[0], acc[1]));
        const float2 acc23 = ffma2(make_float2(db * dx0, db * dx1), eb, make_float2(acc[2], acc[3]));
        acc[0] = acc01.x;
        acc[1] = acc01.y;
        acc[2] = acc23.x;
        acc[3] = acc23.y;
    }
};

// ------------------------------------------------------------------ Q2_K
// Block: scales[16] (sub-block s: scale in the low nibble of byte s, min in
// the high one), qs[64], f16 d, f16 dmin (84 bytes, 4-byte aligned). Element
// e = 128n + 32j + 16h + l takes bits 2j, 2j+1 of qs[32n + 16h + l] and lies
// in the 16-element sub-block s = 8n + 2j + h = e / 16; its value is
// d sc_s q - dmin m_s ("量化格式" (candle), block structure table; the
// library's reading of the ggml layout). The 16-element sub-blocks line up
// with Q6_K's, so the activation panel, its runs and the correction operand
// (bsums of the 16 sub-blocks) are Q6_K's: lane (g, t) takes positions
// l = 4t..4t+3 of every sub-block, i.e. the word qs[32n + 16h + 4t ..] of
// each row, whose bit pair 2j gives sub-block 8n + 2j + h. The min term
// sum_s m_s bsum_s is one k = 16 mma over the mins; the codes (0..3) and
// the sums (16 codes times activations of at most 127) stay exact.
struct MmaQ2_K : MmaQ6_K {
    static constexpr int kBlockBytes = 84;

    template <class BS>
    __device__ __forceinline__ static void tile_block(uint32_t ra, uint32_t rb, const BS &B, int lane,
                                                      float (&acc)[4]) {
        const int t = lane & 3;
        uint32_t swa[4], swb[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            swa[i] = ld_s32(ra + 4 * i);
            swb[i] = ld_s32(rb + 4 * i);
        }
        // min term: sum_s m_s * bsum16_s (mins as subnormal f16 bits: m * 2^-24)
        const uint32_t ssel = (t & 1) ? 0x4342u : 0x4140u;
        auto mins = [](uint32_t w) { return (w >> 4) & 0x0F0F0F0Fu; };
        const uint2 cw = B.corr64();
        float mq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_16816(mq, __byte_perm(mins(t < 2 ? swa[0] : swa[1]), 0u, ssel),
                  __byte_perm(mins(t < 2 ? swb[0] : swb[1]), 0u, ssel),
                  __byte_perm(mins(t < 2 ? swa[2] : swa[3]), 0u, ssel),
                  __byte_perm(mins(t < 2 ? swb[2] : swb[3]), 0u, ssel), cw.x, cw.y);
        float2 Ta = make_float2(0.0f, 0.0f), Tb = make_float2(0.0f, 0.0f);  // rows g, g+8
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            uint32_t qa[2], qb[2];  // [h]: qs[32n + 16h + 4t ..]
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                qa[h] = ld_s32(ra + 16 + 32 * n + 16 * h + 4 * t);
                qb[h] = ld_s32(rb + 16 + 32 * n + 16 * h + 4 * t);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t bf[4];
                B.b(4 * n + j, bf);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int sb = 8 * n + 2 * j + h;
                    const uint32_t ca = (qa[h] >> (2 * j)) & 0x03030303u, cb = (qb[h] >> (2 * j)) & 0x03030303u;
                    float C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    mma_16816(C, ca & 0x00FF00FFu, cb & 0x00FF00FFu, __byte_perm(ca, 0u, 0x4341u),
                              __byte_perm(cb, 0u, 0x4341u), bf[2 * h], bf[2 * h + 1]);
                    // the two rows' scales of sub-block sb: the low nibble of byte
                    // sb placed in the mantissa of 2^23, then 2^23 subtracted
                    const float2 f = fadd2(
                        make_float2(__uint_as_float(__byte_perm(swa[sb >> 2] & 0x0F0F0F0Fu, 0x4B000000u,
                                                                0x7540u | (sb & 3))),
                                    __uint_as_float(__byte_perm(swb[sb >> 2] & 0x0F0F0F0Fu, 0x4B000000u,
                                                                0x7540u | (sb & 3)))),
                        make_float2(-8388608.0f, -8388608.0f));
                    Ta = ffma2(make_float2(f.x, f.x), make_float2(C[0], C[1]), Ta);
                    Tb = ffma2(make_float2(f.y, f.y), make_float2(C[2], C[3]), Tb);
                }
            }
        }
        // block value = d_x * 2^24 * (d * T - dmin * mq)
        const uint32_t dda = ld_s32(ra + 80), ddb = ld_s32(rb + 80);
        const float da = f16_bits_to_f32(dda) * 16777216.0f, dma = f16_bits_to_f32(dda >> 16) * -16777216.0f;
        const float db = f16_bits_to_f32(ddb) * 16777216.0f, dmb = f16_bits_to_f32(ddb >> 16) * -16777216.0f;
        const uint2 dxw = B.dxw(t);
        const float2 dx = make_float2(__uint_as_float(dxw.x), __uint_as_float(dxw.y));
        const float2 ua = ffma2(make_float2(da, da), Ta, make_float2(dma * mq[0], dma * mq[1]));
        const float2 ub = ffma2(make_float2(db, db), Tb, make_float2(dmb * mq[2], dmb * mq[3]));
        float2 acc01 = ffma2(dx, ua, make_float2(acc[0], acc[1]));
        float2 acc23 = ffma2(dx, ub, make_float2(acc[2], acc[3]));
        acc[0] = acc01.x;
        acc[1] = acc01.y;
        acc[2] = acc23.x;
        acc[3] = acc23.y;
    }
};

// ------------------------------------------------------------------ Q3_K
// Block: hmask[32], qs[64], 12 bytes of packed 6-bit scales, f16 d (110
// bytes, 2-byte aligned). Element e = 128n + 32j + 16h + l: 2-bit value from
// bits 2j, 2j+1 of qs[32n + 16h + l], third bit from bit 4n + j of
// hmask[16h + l], q = value + 4 * bit - 4 (-4..3); sub-block s = 8n + 2j + h
// with scale sc_s = v_s - 32, v_s 6 bits (low 4 in the nibbles of bytes
// 0..7, high 2 in bytes 8..11) (the library's reading of the ggml layout).
// As for Q2_K, the activation panel, runs and correction operand are Q6_K's.
// The mma takes the unsigned codes c = q + 4 (0..7) and the scales biased by
// 32, so S = sum_s sc_s sum c a - 4 sum_s sc_s bsum_s, with
// sum_s sc_s bsum_s = sum_s v_s bsum_s - 32 (block sum): one k = 16 mma over
// the biased scales gives sum_s v_s bsum_s.
struct MmaQ3_K : MmaQ6_K {
    static constexpr int kBlockBytes = 110;

    template <class BS>
    __device__ __forceinline__ static void tile_block(uint32_t ra, uint32_t rb, const BS &B, int lane,
                                                      float (&acc)[4]) {
        const int t = lane & 3;
        // biased 6-bit scales v_s, one a byte: word k holds s = 4k .. 4k+3
        uint32_t sa[3], sb[3];
        ld_words_a2<3>(ra + 96, sa);
        ld_words_a2<3>(rb + 96, sb);
        uint32_t va[4], vb[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            va[k] = (((k & 2) ? sa[k & 1] >> 4 : sa[k & 1]) & 0x0F0F0F0Fu) | (((sa[2] >> (2 * k)) & 0x03030303u) << 4);
            vb[k] = (((k & 2) ? sb[k & 1] >> 4 : sb[k & 1]) & 0x0F0F0F0Fu) | (((sb[2] >> (2 * k)) & 0x03030303u) << 4);
        }
        const uint32_t ssel = (t & 1) ? 0x4342u : 0x4140u;
        const uint2 cw = B.corr64();
        float mq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_16816(mq, __byte_perm(t < 2 ? va[0] : va[1], 0u, ssel), __byte_perm(t < 2 ? vb[0] : vb[1], 0u, ssel),
                  __byte_perm(t < 2 ? va[2] : va[3], 0u, ssel), __byte_perm(t < 2 ? vb[2] : vb[3], 0u, ssel), cw.x,
                  cw.y);
        uint32_t hma[2], hmb[2];  // [h]: hmask[16h + 4t ..]
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w[1];
            ld_words_a2<1>(ra + 16 * h + 4 * t, w);
            hma[h] = w[0];
            ld_words_a2<1>(rb + 16 * h + 4 * t, w);
            hmb[h] = w[0];
        }
        float2 Ta = make_float2(0.0f, 0.0f), Tb = make_float2(0.0f, 0.0f);  // rows g, g+8
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            uint32_t qa[2], qb[2];  // [h]: qs[32n + 16h + 4t ..]
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t w[1];
                ld_words_a2<1>(ra + 32 + 32 * n + 16 * h + 4 * t, w);
                qa[h] = w[0];
                ld_words_a2<1>(rb + 32 + 32 * n + 16 * h + 4 * t, w);
                qb[h] = w[0];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t bf[4];
                B.b(4 * n + j, bf);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int sb = 8 * n + 2 * j + h;
                    const int hb = 4 * n + j;  // the hmask bit, moved to bit 2 of each byte
                    const uint32_t ha3 = (hb >= 2 ? hma[h] >> (hb - 2) : hma[h] << (2 - hb)) & 0x04040404u;
                    const uint32_t hb3 = (hb >= 2 ? hmb[h] >> (hb - 2) : hmb[h] << (2 - hb)) & 0x04040404u;
                    const uint32_t ca = ((qa[h] >> (2 * j)) & 0x03030303u) | ha3;
                    const uint32_t cb = ((qb[h] >> (2 * j)) & 0x03030303u) | hb3;
                    float C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    mma_16816(C, ca & 0x00FF00FFu, cb & 0x00FF00FFu, __byte_perm(ca, 0u, 0x4341u),
                              __byte_perm(cb, 0u, 0x4341u), bf[2 * h], bf[2 * h + 1]);
                    // sc_s = v_s - 32: byte s of the biased words in the mantissa
                    // of 2^23, then 2^23 + 32 subtracted
                    const float2 f = fadd2(
                        make_float2(__uint_as_float(__byte_perm(va[sb >> 2], 0x4B000000u, 0x7540u | (sb & 3))),
                                    __uint_as_float(__byte_perm(vb[sb >> 2], 0x4B000000u, 0x7540u | (sb & 3)))),
                        make_float2(-8388640.0f, -8388640.0f));
                    Ta = ffma2(make_float2(f.x, f.x), make_float2(C[0], C[1]), Ta);
                    Tb = ffma2(make_float2(f.y, f.y), make_float2(C[2], C[3]), Tb);
                }
            }
        }
        // block value = d * d_x * 2^24 * (T - 4 mq + 2^-17 * block sum)
        const float da = f16_bits_to_f32(ld_s16(ra + 108)) * 16777216.0f;
        const float db = f16_bits_to_f32(ld_s16(rb + 108)) * 16777216.0f;
        const uint2 dxw = B.dxw(t);
        const uint2 bsw = B.bsw(t);
        const float dx0 = __uint_as_float(dxw.x), dx1 = __uint_as_float(dxw.y);
        const float2 bs = make_float2(__uint_as_float(bsw.x), __uint_as_float(bsw.y));
        const float2 q17 = make_float2(0.00000762939453125f, 0.00000762939453125f), m4 = make_float2(-4.0f, -4.0f);
        const float2 ea = ffma2(q17, bs, ffma2(m4, make_float2(mq[0], mq[1]), Ta));
        const float2 eb = ffma2(q17, bs, ffma2(m4, make_float2(mq[2], mq[3]), Tb));
        const float2 acc01 = ffma2(make_float2(da * dx0, da * dx1), ea, make_float2(acc[0], acc[1]));
        const float2 acc23 = ffma2(make_float2(db * dx0, db * dx1), eb, make_float2(acc[2], acc[3]));
        acc[0] = acc01.x;
        acc[1] = acc01.y;
        acc[2] = acc23.x;
        acc[3] = acc23.y;
    }
};

// ------------------------------------------------------- 32-element blocks
// Q4_0, Q5_0, Q4_1 and Q8_0 rows are taken eight blocks (256 elements) at a
// time: one panel block per group, record r = block r of the group
// ("Building Q8_0 and Q4_0 Like ggml", Examples 1, 5, 7 and 8; "量化格式"
// (candle), block structure table). Lane (g, t) takes elements 4t..4t+3 (the
// record's first run: the block's first mma) and 16 + 4t..16 + 4t + 3 (the
// second run: its second mma) of each block of rows g and g + 8.
//  * Codes enter unsigned, as f16 subnormal bit patterns cut from the block
//    bytes by one mask: code c (Q8_0: q + 128) is c 2^-24. Where a code's
//    low bits sit at bits 4..7 of a byte (the second run of Q4_0, Q4_1 and
//    Q5_0) the mask leaves them there, giving 16 c 2^-24, and the panel holds
//    that run's activations divided by 16 (exact in f16): every product is
//    c a 2^-24 exactly.
//  * The offset of the signed types (value (c - bias) d) is the mma
//    accumulator's initial value -bias S 2^-24, S = the block's activation
//    code sum, which the panel holds per block and vector. The block's
//    exact sum of (c - bias) a, times 2^-24, is then the mma's result (every
//    partial sum an integer times 2^-24 of magnitude below 1: exact in f32).
//  * A group's rows start 16-byte aligned in the ring (eight blocks are a
//    multiple of 16 bytes and so is every row and chunk offset), so the
//    alignment of each field is fixed by its block index; a 2-byte aligned
//    word is read as its two aligned neighbours, whose bytes one permute per
//    operand sorts into even and odd bytes.
// The panel's tail holds per record r and lane t the float4 {d_x 2^24 of
// vectors 2t, 2t+1; the accumulator's initial value for the same vectors
// (Q4_1: s_x)}.

// The 4-byte word at base + 4t + OFF (base 16-byte aligned, OFF a constant)
// as E = its bytes 0 and 2 in the low byte of each 16-bit lane and O = its
// bytes 1 and 3 likewise; the high byte of each lane is unspecified.
template <int OFF>
__device__ __forceinline__ void mma_eo(uint32_t base_t, uint32_t &E, uint32_t &O) {
    if constexpr (OFF % 4 == 0) {
        E = ld_s32(base_t + OFF);
        O = E >> 8;
    } else {
        static_assert(OFF % 4 == 2, "block fields are 2-byte aligned");
        const uint32_t w0 = ld_s32(base_t + OFF - 2), w1 = ld_s32(base_t + OFF + 2);
        E = __byte_perm(w0, w1, 0x0402);
        O = __byte_perm(w0, w1, 0x0503);
    }
}

// The 4 bytes at base + OFF (same alignment rule), as one word.
template <int OFF>
__device__ __forceinline__ uint32_t mma_word(uint32_t base) {
    if constexpr (OFF % 4 == 0) {
        return ld_s32(base + OFF);
    } else {
        static_assert(OFF % 4 == 2, "block fields are 2-byte aligned");
        return __byte_perm(ld_s32(base + OFF - 2), ld_s32(base + OFF + 2), 0x5432);
    }
}

// Packed two-lane f32 product (one instruction for both lanes).
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// The first mma of a block, its accumulator starting from the tail's
// initial values (rows g, g+8; vectors 2t, 2t+1).
__device__ __forceinline__ void mma_group_first(float (&C)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                uint32_t b0, uint32_t b1, uint4 tl) {
    const float c0 = __uint_as_float(tl.z), c1 = __uint_as_float(tl.w);
    mma_16816_c(C, a0, a1, a2, a3, b0, b1, c0, c1, c0, c1);
}

// acc += d_w (d_x 2^24) C for rows g, g+8 and vectors 2t, 2t+1.
__device__ __forceinline__ void mma_group_step(const float (&C)[4], float dwa, float dwb, uint4 tl, float (&acc)[4]) {
    const float2 dx = make_float2(__uint_as_float(tl.x), __uint_as_float(tl.y));
    const float2 a01 = ffma2(fmul2(make_float2(dwa, dwa), dx), make_float2(C[0], C[1]), make_float2(acc[0], acc[1]));
    const float2 a23 = ffma2(fmul2(make_float2(dwb, dwb), dx), make_float2(C[2], C[3]), make_float2(acc[2], acc[3]));
    acc[0] = a01.x;
    acc[1] = a01.y;
    acc[2] = a23.x;
    acc[3] = a23.y;
}

// The eight blocks of a group, unrolled (each block's field offsets, and so
// their alignment, are constants).
template <class T, class BS, int R = 0>
__device__ __forceinline__ void mma_group_blocks(uint32_t ra, uint32_t rb, const BS &B, int t, float (&acc)[4]) {
    T::template block<R>(ra, rb, B, t, acc);
    if constexpr (R + 1 < kMmaRecords) mma_group_blocks<T, BS, R + 1>(ra, rb, B, t, acc);
}

// Q4_0: 18-byte blocks (f16 d, qs[16]: byte k = code k | code k+16 << 4),
// value (code - 8) d, paired with Q8_0 activations.
struct MmaQ4_0 {
    static constexpr int kBlockBytes = 8 * 18;
    static constexpr int kActBytes = 34;
    static constexpr int kBias = 8;
    static constexpr bool kHiScaled = true;

    template <int R, class BS>
    __device__ __forceinline__ static void block(uint32_t ra, uint32_t rb, const BS &B, int t, float (&acc)[4]) {
        uint32_t Ea, Oa, Eb, Ob;
        mma_eo<18 * R + 2>(ra + 4 * t, Ea, Oa);  // qs[4t..4t+3]
        mma_eo<18 * R + 2>(rb + 4 * t, Eb, Ob);
        const float dwa = f16_bits_to_f32(ld_s16(ra + 18 * R)), dwb = f16_bits_to_f32(ld_s16(rb + 18 * R));
        uint32_t bf[4];
        B.b(R, bf);
        const uint4 tl = B.tail(R, t);
        float C[4];
        mma_group_first(C, Ea & 0x000F000Fu, Eb & 0x000F000Fu, Oa & 0x000F000Fu, Ob & 0x000F000Fu, bf[0], bf[1], tl);
        mma_16816(C, Ea & 0x00F000F0u, Eb & 0x00F000F0u, Oa & 0x00F000F0u, Ob & 0x00F000F0u, bf[2], bf[3]);
        mma_group_step(C, dwa, dwb, tl, acc);
    }
    template <class BS>
    __device__ __forceinline__ static void tile_block(uint32_t ra, uint32_t rb, const BS &B, int lane,
                                                      float (&acc)[4]) {
        mma_group_blocks<MmaQ4_0>(ra, rb, B, lane & 3, acc);
    }
};

// Q8_0: 34-byte blocks (f16 d, 32 int8 codes), value q d, paired with Q8_0
// activations; the mma takes q + 128.
struct MmaQ8_0 {
    static constexpr int kBlockBytes = 8 * 34;
    static constexpr int kActBytes = 34;
    static constexpr int kBias = 128;
    static constexpr bool kHiScaled = false;

    __device__ __forceinline__ static uint32_t u(uint32_t e) { return (e ^ 0x00800080u) & 0x00FF00FFu; }

    template <int R, class BS>
    __device__ __forceinline__ static void block(uint32_t ra, uint32_t rb, const BS &B, int t, float (&acc)[4]) {
        uint32_t Ea, Oa, Eb, Ob, Fa, Pa, Fb, Pb;
        mma_eo<34 * R + 2>(ra + 4 * t, Ea, Oa);  // codes 4t..4t+3
        mma_eo<34 * R + 2>(rb + 4 * t, Eb, Ob);
        mma_eo<34 * R + 18>(ra + 4 * t, Fa, Pa);  // codes 16 + 4t..
        mma_eo<34 * R + 18>(rb + 4 * t, Fb, Pb);
        const float dwa = f16_bits_to_f32(ld_s16(ra + 34 * R)), dwb = f16_bits_to_f32(ld_s16(rb + 34 * R));
        uint32_t bf[4];
        B.b(R, bf);
        const uint4 tl = B.tail(R, t);
        float C[4];
        mma_group_first(C, u(Ea), u(Eb), u(Oa), u(Ob), bf[0], bf[1], tl);
        mma_16816(C, u(Fa), u(Fb), u(Pa), u(Pb), bf[2], bf[3]);
        mma_group_step(C, dwa, dwb, tl, acc);
    }
    template <class BS>
    __device__ __forceinline__ static void tile_block(uint32_t ra, uint32_t rb, const BS &B, int lane,
                                                      float (&acc)[4]) {
        mma_group_blocks<MmaQ8_0>(ra, rb, B, lane & 3, acc);
    }
};

// Q5_0: 22-byte blocks (f16 d, u32 qh: bit j = fifth bit of code j, qs[16]
// as in Q4_0), value (code - 16) d, paired with Q8_0 activations. A lane's
// nibble n of qh (the fifth bits of its 4 codes of one run) is spread to
// bits 0, 8, 16, 24 by one multiply (the four shifted copies of n do not
// overlap), then each pair is shifted under its code: bits 4 and 20 in the
// first run, 8 and 24 in the second (where the code is 16 c).
struct MmaQ5_0 {
    static constexpr int kBlockBytes = 8 * 22;
    static constexpr int kActBytes = 34;
    static constexpr int kBias = 16;
    static constexpr bool kHiScaled = true;

    __device__ __forceinline__ static void ops(uint32_t E, uint32_t O, uint32_t n0, uint32_t n1, uint32_t (&a)[4]) {
        const uint32_t x0 = ((n0 & 15u) * 0x00204081u) & 0x01010101u;
        const uint32_t x1 = ((n1 & 15u) * 0x00204081u) & 0x01010101u;
        a[0] = (E & 0x000F000Fu) | ((x0 << 4) & 0x00100010u);
        a[1] = (O & 0x000F000Fu) | ((x0 >> 4) & 0x00100010u);
        a[2] = (E & 0x00F000F0u) | ((x1 << 8) & 0x01000100u);
        a[3] = (O & 0x00F000F0u) | (x1 & 0x01000100u);
    }

    template <int R, class BS>
    __device__ __forceinline__ static void block(uint32_t ra, uint32_t rb, const BS &B, int t, float (&acc)[4]) {
        uint32_t Ea, Oa, Eb, Ob;
        mma_eo<22 * R + 6>(ra + 4 * t, Ea, Oa);  // qs[4t..4t+3]
        mma_eo<22 * R + 6>(rb + 4 * t, Eb, Ob);
        const uint32_t qa = mma_word<22 * R + 2>(ra), qb = mma_word<22 * R + 2>(rb);
        const float dwa = f16_bits_to_f32(ld_s16(ra + 22 * R)), dwb = f16_bits_to_f32(ld_s16(rb + 22 * R));
        uint32_t xa[4], xb[4];
        ops(Ea, Oa, qa >> (4 * t), qa >> (16 + 4 * t), xa);
        ops(Eb, Ob, qb >> (4 * t), qb >> (16 + 4 * t), xb);
        uint32_t bf[4];
        B.b(R, bf);
        const uint4 tl = B.tail(R, t);
        float C[4];
        mma_group_first(C, xa[0], xb[0], xa[1], xb[1], bf[0], bf[1], tl);
        mma_16816(C, xa[2], xb[2], xa[3], xb[3], bf[2], bf[3]);
        mma_group_step(C, dwa, dwb, tl, acc);
    }
    template <class BS>
    __device__ __forceinline__ static void tile_block(uint32_t ra, uint32_t rb, const BS &B, int lane,
                                                      float (&acc)[4]) {
        mma_group_blocks<MmaQ5_0>(ra, rb, B, lane & 3, acc);
    }
};

// Q4_1: 20-byte blocks (f16 d, f16 m, qs[16] as in Q4_0), value code d + m,
// paired with Q8_1 activations (d_x, s = d_x sum q): per block
// d d_x sum(code q) + m s.
struct MmaQ4_1 {
    static constexpr int kBlockBytes = 8 * 20;
    static constexpr int kActBytes = 36;
    static constexpr int kBias = 0;
    static constexpr bool kHiScaled = true;

    template <int R, class BS>
    __device__ __forceinline__ static void block(uint32_t ra, uint32_t rb, const BS &B, int t, float (&acc)[4]) {
        uint32_t Ea, Oa, Eb, Ob;
        mma_eo<20 * R + 4>(ra + 4 * t, Ea, Oa);
        mma_eo<20 * R + 4>(rb + 4 * t, Eb, Ob);
        const uint32_t ha = ld_s32(ra + 20 * R), hb = ld_s32(rb + 20 * R);  // d | m << 16
        const float dwa = f16_bits_to_f32(ha & 0xFFFFu), dwb = f16_bits_to_f32(hb & 0xFFFFu);
        const float ma = f16_bits_to_f32(ha >> 16), mb = f16_bits_to_f32(hb >> 16);
        uint32_t bf[4];
        B.b(R, bf);
        const uint4 tl = B.tail(R, t);
        float C[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_16816(C, Ea & 0x000F000Fu, Eb & 0x000F000Fu, Oa & 0x000F000Fu, Ob & 0x000F000Fu, bf[0], bf[1]);
        mma_16816(C, Ea & 0x00F000F0u, Eb & 0x00F000F0u, Oa & 0x00F000F0u, Ob & 0x00F000F0u, bf[2], bf[3]);
        const float2 sx = make_float2(__uint_as_float(tl.z), __uint_as_float(tl.w));
        const float2 m01 = ffma2(make_float2(ma, ma), sx, make_float2(acc[0], acc[1]));
        const float2 m23 = ffma2(make_float2(mb, mb), sx, make_float2(acc[2], acc[3]));
        float m4[4] = {m01.x, m01.y, m23.x, m23.y};
        mma_group_step(C, dwa, dwb, tl, m4);
        acc[0] = m4[0];
        acc[1] = m4[1];
        acc[2] = m4[2];
        acc[3] = m4[3];
    }
    template <class BS>
    __device__ __forceinline__ static void tile_block(uint32_t ra, uint32_t rb, const BS &B, int lane,
                                                      float (&acc)[4]) {
        mma_group_blocks<MmaQ4_1>(ra, rb, B, lane & 3, acc);
    }
};

// ------------------------------------------------------------------ panel
// Activations of one matrix (Q8_K blocks [nv][nb] at xq) into the panel:
// per block, fragment record r of lane (g, t) = codes of vector g at the
// type's two 4-code runs, each permuted to slots {0,2,1,3}; then per lane
// the correction operand (f16), d_x[8] and the block sums[8] (f32). Vectors
// g >= nv are zero. All consumer threads take part.
template <class T, bool B16>
__device__ __forceinline__ void mma_build_panel(const MmaParams &p, const uint8_t *xq, uint8_t *pan, int tid,
                                                int nthr) {
    const int nb = p.nb, nv = p.nv;
    const int n_rec = nb * kMmaRecords * 32;
    constexpr int kBatch = 8;  // records whose loads are in flight together
    for (int u0 = tid; u0 < n_rec; u0 += kBatch * nthr) {
        uint32_t w0[kBatch], w1[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int u = u0 + i * nthr;
            const int b = u / (kMmaRecords * 32), r = (u / 32) % kMmaRecords, L = u % 32;
            const int g = L >> 2, t = L & 3;
            w0[i] = w1[i] = 0u;
            if (u < n_rec && g < nv) {
                const uint8_t *qs = xq + (static_cast<size_t>(g) * nb + b) * 292 + 4;
                w0[i] = __ldg(reinterpret_cast<const uint32_t *>(qs + T::run0(r, t)));
                w1[i] = __ldg(reinterpret_cast<const uint32_t *>(qs + T::run1(r, t)));
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int u = u0 + i * nthr;
            if (u >= n_rec) break;
            const int b = u / (kMmaRecords * 32), r = (u / 32) % kMmaRecords, L = u % 32;
            const uint32_t x0 = __byte_perm(w0[i], 0u, 0x3120), x1 = __byte_perm(w1[i], 0u, 0x3120);
            uint8_t *dst = pan + static_cast<size_t>(b) * p.rec_bytes;
            if (B16) {
                uint4 o;
                o.x = mma_pack(__half_as_ushort(__int2half_rn(sbyte(x0, 0))), __half_as_ushort(__int2half_rn(sbyte(x0, 1))));
                o.y = mma_pack(__half_as_ushort(__int2half_rn(sbyte(x0, 2))), __half_as_ushort(__int2half_rn(sbyte(x0, 3))));
                o.z = mma_pack(__half_as_ushort(__int2half_rn(sbyte(x1, 0))), __half_as_ushort(__int2half_rn(sbyte(x1, 1))));
                o.w = mma_pack(__half_as_ushort(__int2half_rn(sbyte(x1, 2))), __half_as_ushort(__int2half_rn(sbyte(x1, 3))));
                reinterpret_cast<uint4 *>(dst)[r * 32 + L] = o;
            } else {
                reinterpret_cast<uint2 *>(dst)[r * 32 + L] = make_uint2(x0 ^ 0x80808080u, x1 ^ 0x80808080u);
            }
        }
    }
    // per (block, vector): the correction operands of the vector's 4 lanes,
    // d_x and the block sum
    for (int u = tid; u < nb * kMmaNvec; u += nthr) {
        const int b = u / kMmaNvec, v = u % kMmaNvec;
        int16_t bs[16];
        float dx = 0.0f;
        if (v < nv) {
            const uint8_t *blk = xq + (static_cast<size_t>(v) * nb + b) * 292;
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i] = __ldg(reinterpret_cast<const uint32_t *>(blk + 260) + i);
            dx = __ldg(reinterpret_cast<const float *>(blk));
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                bs[2 * i] = static_cast<int16_t>(w[i] & 0xFFFFu);
                bs[2 * i + 1] = static_cast<int16_t>(w[i] >> 16);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) bs[i] = 0;
        }
        uint8_t *tail = pan + static_cast<size_t>(b) * p.rec_bytes + mma_frag_bytes(B16);
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) sum += bs[i];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            float c[4];
            T::corr(bs, t, c);
            reinterpret_cast<uint2 *>(tail)[4 * v + t] =
                make_uint2(mma_pack(__half_as_ushort(__float2half_rn(c[0])), __half_as_ushort(__float2half_rn(c[1]))),
                           mma_pack(__half_as_ushort(__float2half_rn(c[2])), __half_as_ushort(__float2half_rn(c[3]))));
        }
        reinterpret_cast<float *>(tail + 256)[v] = dx;
        reinterpret_cast<float *>(tail + 288)[v] = static_cast<float>(sum);
    }
}

// Activations of one matrix from Q8_0 (34-byte) or Q8_1 (36-byte) blocks
// [nv][8 nb] into the panel, for weights in groups of eight 32-element blocks
// (one panel block per group): record r = activation block r of the group,
// its two 4-code runs at codes 4t and 16 + 4t permuted to slots {0,2,1,3}
// (the layout of the Q6_K records; the second run divided by 16 in the f16
// panel when T::kHiScaled); then per record and lane t the float4 {d_x 2^24,
// d_x 2^24, c, c} of vectors 2t, 2t+1, c = -T::kBias * (sum of the block's
// codes) * 2^-24 (Q8_1: its s). Vectors g >= nv are zero.
template <class T, bool B16>
__device__ __forceinline__ void mma_build_panel_q8(const MmaParams &p, const uint8_t *xq, uint8_t *pan, int tid,
                                                   int nthr) {
    constexpr int AB = T::kActBytes, CO = AB - 32;  // block bytes; offset of the codes
    const int nb = p.nb, nv = p.nv, nb32 = 8 * nb;
    const int n_rec = nb * kMmaRecords * 32;
    auto ld4 = [](const uint8_t *a) {  // 4 bytes at a 2-byte aligned address
        const uint16_t *h = reinterpret_cast<const uint16_t *>(a);
        return static_cast<uint32_t>(__ldg(h)) | (static_cast<uint32_t>(__ldg(h + 1)) << 16);
    };
    constexpr int kBatch = 8;
    for (int u0 = tid; u0 < n_rec; u0 += kBatch * nthr) {
        uint32_t w0[kBatch], w1[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int u = u0 + i * nthr;
            const int b = u / (kMmaRecords * 32), r = (u / 32) % kMmaRecords, L = u % 32;
            const int g = L >> 2, t = L & 3;
            w0[i] = w1[i] = 0u;
            if (u < n_rec && g < nv) {
                const uint8_t *qs = xq + (static_cast<size_t>(g) * nb32 + 8 * b + r) * AB + CO;
                w0[i] = ld4(qs + 4 * t);
                w1[i] = ld4(qs + 16 + 4 * t);
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int u = u0 + i * nthr;
            if (u >= n_rec) break;
            const int b = u / (kMmaRecords * 32), r = (u / 32) % kMmaRecords, L = u % 32;
            const uint32_t x0 = __byte_perm(w0[i], 0u, 0x3120), x1 = __byte_perm(w1[i], 0u, 0x3120);
            uint8_t *dst = pan + static_cast<size_t>(b) * p.rec_bytes;
            if constexpr (T::kBias != 0) {
                // the block's code sum S: the 4 lanes t of vector g hold its
                // 32 codes (lanes 4g..4g+3 of this warp, the same u / 32);
                // lane t = 0 stores the accumulator's start -bias S 2^-24
                // (exact: |bias S| < 2^24)
                int sum = __dp4a(static_cast<int>(w0[i]), 0x01010101, __dp4a(static_cast<int>(w1[i]), 0x01010101, 0));
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if ((L & 3) == 0) {
                    const int g = L >> 2;
                    reinterpret_cast<float *>(dst + mma_frag_bytes(B16))[16 * r + 4 * (g >> 1) + 2 + (g & 1)] =
                        static_cast<float>(-T::kBias * sum) * 5.9604644775390625e-8f;
                }
            }
            if (B16) {
                uint4 o;
                o.x = mma_pack(__half_as_ushort(__int2half_rn(sbyte(x0, 0))), __half_as_ushort(__int2half_rn(sbyte(x0, 1))));
                o.y = mma_pack(__half_as_ushort(__int2half_rn(sbyte(x0, 2))), __half_as_ushort(__int2half_rn(sbyte(x0, 3))));
                constexpr float hs = T::kHiScaled ? 0.0625f : 1.0f;  // exact: a power of two
                o.z = mma_pack(__half_as_ushort(__float2half_rn(hs * sbyte(x1, 0))),
                               __half_as_ushort(__float2half_rn(hs * sbyte(x1, 1))));
                o.w = mma_pack(__half_as_ushort(__float2half_rn(hs * sbyte(x1, 2))),
                               __half_as_ushort(__float2half_rn(hs * sbyte(x1, 3))));
                reinterpret_cast<uint4 *>(dst)[r * 32 + L] = o;
            } else {
                reinterpret_cast<uint2 *>(dst)[r * 32 + L] = make_uint2(x0 ^ 0x80808080u, x1 ^ 0x80808080u);
            }
        }
    }
    // per (group, record, vector): d_x 2^24 and (Q8_1) s
    for (int u = tid; u < nb * kMmaRecords * kMmaNvec; u += nthr) {
        const int b = u / (kMmaRecords * kMmaNvec), r = (u / kMmaNvec) % kMmaRecords, v = u % kMmaNvec;
        float dx = 0.0f, sx = 0.0f;
        if (v < nv) {
            const uint8_t *blk = xq + (static_cast<size_t>(v) * nb32 + 8 * b + r) * AB;
            dx = f16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t *>(blk))) * 16777216.0f;
            if constexpr (AB == 36) sx = f16_bits_to_f32(__ldg(reinterpret_cast<const uint16_t *>(blk + 2)));
        }
        float *tail = reinterpret_cast<float *>(pan + static_cast<size_t>(b) * p.rec_bytes + mma_frag_bytes(B16));
        tail[16 * r + 4 * (v >> 1) + (v & 1)] = dx;
        if constexpr (T::kBias == 0) tail[16 * r + 4 * (v >> 1) + 2 + (v & 1)] = sx;
    }
}

// The B operands of one weight block `blk` of the matrix whose activations
// are xq, into registers (the panel's contents for this lane: fragments as
// f16, the correction operand, d_x and block sums of vectors 2t, 2t+1).
template <class T>
__device__ __forceinline__ void mma_load_regs(const uint8_t *xq, int nb, int nv, int blk, int lane,
                                              uint32_t (&r)[kMmaRecords][4], uint2 &corr, uint2 &dx, uint2 &bs) {
    const int g = lane >> 2, t = lane & 3;
    uint32_t w0[kMmaRecords], w1[kMmaRecords];
    const uint8_t *qs = xq + (static_cast<size_t>(g) * nb + blk) * 292 + 4;
#pragma unroll
    for (int i = 0; i < kMmaRecords; ++i) {
        w0[i] = g < nv ? __ldg(reinterpret_cast<const uint32_t *>(qs + T::run0(i, t))) : 0u;
        w1[i] = g < nv ? __ldg(reinterpret_cast<const uint32_t *>(qs + T::run1(i, t))) : 0u;
    }
    int16_t bsv[16];
    if (g < nv) {
        const uint32_t *bw = reinterpret_cast<const uint32_t *>(xq + (static_cast<size_t>(g) * nb + blk) * 292 + 260);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w = __ldg(bw + i);
            bsv[2 * i] = static_cast<int16_t>(w & 0xFFFFu);
            bsv[2 * i + 1] = static_cast<int16_t>(w >> 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) bsv[i] = 0;
    }
    float dxv[2] = {0.0f, 0.0f}, bsum[2] = {0.0f, 0.0f};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int v = 2 * t + u;
        if (v < nv) {
            const uint8_t *vb = xq + (static_cast<size_t>(v) * nb + blk) * 292;
            dxv[u] = __ldg(reinterpret_cast<const float *>(vb));
            int sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(vb + 260) + i);
                sum += static_cast<int16_t>(w & 0xFFFFu) + static_cast<int16_t>(w >> 16);
            }
            bsum[u] = static_cast<float>(sum);
        }
    }
#pragma unroll
    for (int i = 0; i < kMmaRecords; ++i) {
        // slots {0,2,1,3} of each run, biased bytes -> f16 (1024 + c) -> minus 1152
        const uint32_t x0 = __byte_perm(w0[i], 0u, 0x3120) ^ 0x80808080u;
        const uint32_t x1 = __byte_perm(w1[i], 0u, 0x3120) ^ 0x80808080u;
        r[i][0] = hsub1152(__byte_perm(x0, 0x64646464u, 0x4140));
        r[i][1] = hsub1152(__byte_perm(x0, 0x64646464u, 0x4342));
        r[i][2] = hsub1152(__byte_perm(x1, 0x64646464u, 0x4140));
        r[i][3] = hsub1152(__byte_perm(x1, 0x64646464u, 0x4342));
    }
    float c[4];
    T::corr(bsv, t, c);
    corr = make_uint2(mma_pack(__half_as_ushort(__float2half_rn(c[0])), __half_as_ushort(__float2half_rn(c[1]))),
                      mma_pack(__half_as_ushort(__float2half_rn(c[2])), __half_as_ushort(__float2half_rn(c[3]))));
    dx = make_uint2(__float_as_uint(dxv[0]), __float_as_uint(dxv[1]));
    bs = make_uint2(__float_as_uint(bsum[0]), __float_as_uint(bsum[1]));
}

// ------------------------------------------------------------------ producer
// The tile's output: the NW warps' partials of buffer ri added in warp
// order, stored to y (lane (g, t) holds rows g and g+8, vectors 2t, 2t+1 of
// the mma tile, i.e. stage rows mma_stage_row(g), mma_stage_row(g + 8)).
template <int NW>
__device__ __forceinline__ void mma_finish_tile(const MmaParams &p, const float4 *red, int ri, float *y, int n_out,
                                                int tile, int lane) {
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        const float4 v = red[(ri * NW + w) * 32 + lane];
        s[0] += v.x;
        s[1] += v.y;
        s[2] += v.z;
        s[3] += v.w;
    }
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int row = tile * kMmaTileRows + mma_stage_row(g + (q >= 2 ? 8 : 0));
        const int v = 2 * t + (q & 1);
        if (row < n_out && v < p.nv) y[static_cast<int64_t>(v) * n_out + row] = s[q];
    }
}

// One stage's copies, shared by the NP producer warps: copy i = lane * NP + pw
// of producer warp pw is row group i (whole rows) or row segment i. Each
// bulk request costs its issuing thread on the order of 100 cycles, so with
// 16 row segments a stage two warps issue in parallel. mma_plan_copy works
// out this lane's window (it does not touch the slot, so it runs before the
// slot is free); mma_issue_copy stores the bytes past W's last 16-byte
// boundary, announces the warp's bytes on the stage's barrier (one arrival
// per producer warp) and issues the copy.
struct MmaCopy {
    int64_t a0, a1, e;  // window [a0, a1) of W by bulk copy, [a1, e) by plain loads
    uint32_t dst;       // slot offset of the window
    uint32_t total;     // bytes by bulk copy, this warp's part of the stage (every lane)
};

template <class T, int NP>
__device__ __forceinline__ MmaCopy mma_plan_copy(const MmaParams &p, int n_out, const MmaStage &st, int lane,
                                                 int pw) {
    const int rows = min(kMmaTileRows, n_out - st.tile * kMmaTileRows);
    const int64_t row0 = static_cast<int64_t>(st.tile) * kMmaTileRows;
    const int i = lane * NP + pw;
    MmaCopy c;
    int64_t s;
    bool mine;
    if (p.contig) {
        mine = 4 * i < rows;
        s = (row0 + 4 * i) * p.row_bytes;
        c.e = s + static_cast<int64_t>(min(4, rows - 4 * i)) * p.row_bytes;
        c.dst = static_cast<uint32_t>(i * p.gpitch);
    } else {
        mine = i < rows;
        const int kbt = min(p.kb, p.nb - st.kc * p.kb);
        s = (row0 + i) * p.row_bytes + static_cast<int64_t>(st.kc) * p.kb * T::kBlockBytes;
        c.e = s + static_cast<int64_t>(kbt) * T::kBlockBytes;
        c.dst = static_cast<uint32_t>((i >> 2) * p.gpitch + (i & 3) * p.rpitch);
    }
    c.a0 = c.a1 = c.e = mine ? c.e : 0;
    if (mine) {
        const int64_t lim = (static_cast<int64_t>(n_out) * p.row_bytes) & ~int64_t(15);
        c.a0 = s & ~int64_t(15);
        c.a1 = (c.e + 15) & ~int64_t(15);
        if (c.a1 > lim) c.a1 = lim;
        if (c.a1 < c.a0) c.a1 = c.a0;
    }
    uint32_t total = static_cast<uint32_t>(c.a1 - c.a0);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
    c.total = total;
    return c;
}

__device__ __forceinline__ void mma_issue_copy(const MmaCopy &c, const uint8_t *W, uint8_t *buf, uint32_t bar,
                                               uint64_t policy, int lane) {
    uint8_t *dst = buf + c.dst;
    for (int64_t x = c.a1; x < c.e; ++x) dst[x - c.a0] = __ldg(W + x);  // rare: W's last < 16 bytes
    __syncwarp();  // the plain stores come before the arrival that publishes the stage
    if (lane == 0) mbar_arrive_expect_tx(bar, c.total);
    __syncwarp();
    if (c.a1 > c.a0) bulk_copy_g2s(smem_addr(dst), W + c.a0, static_cast<uint32_t>(c.a1 - c.a0), bar, policy);
}

// One producer warp (pw of NP): lane 0 waits for free slots (with a reducer:
// slots the reducer has freed) and the warp issues its copies. A producer
// cannot get a phase ahead of another: a slot is released only after its
// stage's full barrier has all NP arrivals.
template <class T, bool RED, int NP, int MAXB>
__device__ __forceinline__ void mma_producer(const MmaParams &p, const MmaBatch<MAXB> &b, uint8_t *ring,
                                             uint32_t full0, uint32_t empty0, uint32_t reduced0, int lane, int pw) {
    const uint64_t policy = l2_evict_first_policy();
    const int S = p.n_stages;
    const uint32_t free0 = RED ? reduced0 : empty0;  // where a slot's release is announced
    int cur = -1;
    const uint8_t *W = nullptr;
    int n_out = 0;
    MmaWalk walk = mma_cta_walk(p, b);
    MmaStage st;
    int issued = 0;
    // slot = k mod S and phase = (k / S) & 1, kept incrementally
    int slot = 0;
    uint32_t phase = 0;
    for (int k = 0; walk.next(b, p, st); ++k) {
        if (st.mat != cur) {  // the matrix's fields, read from the parameter table once
            cur = st.mat;
            W = b.m[MAXB == 1 ? 0 : cur].W;
            n_out = b.m[MAXB == 1 ? 0 : cur].n_out;
        }
        const MmaCopy cp = mma_plan_copy<T, NP>(p, n_out, st, lane, pw);  // before the slot is free
        if (k >= S) {
            bool got = true;
            if (lane == 0) got = mbar_wait_bounded(free0 + 8 * slot, phase ^ 1u);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                if (lane == 0) record_error(p.err, kErrProducerWait);
                break;
            }
        }
        mma_issue_copy(cp, W, ring + static_cast<size_t>(slot) * p.stage_bytes, full0 + 8 * slot, policy, lane);
        ++issued;
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
    }
    // Leave no copy in flight into this CTA's shared memory.
    for (int k = max(0, issued - S); k < issued; ++k) {
        const int sk = k % S;
        bool got = true;
        if (lane == 0) got = mbar_wait_bounded(full0 + 8 * sk, static_cast<uint32_t>((k / S) & 1));
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
            if (lane == 0) record_error(p.err, kErrDrainWait);
            return;
        }
    }
}

// The reducer warp: for each stage but the CTA's final one, once the
// consumers have released it, the tile's outputs; then the slot (and its
// partial buffer) is marked free for the producer.
template <int NW, int MAXB>
__device__ __forceinline__ void mma_reducer(const MmaParams &p, const MmaBatch<MAXB> &b, const float4 *red,
                                            uint32_t empty0, uint32_t reduced0, int lane) {
    const int S = p.n_stages, R = p.red_slots;
    MmaWalk walk = mma_cta_walk(p, b);
    MmaStage st;
    int slot = 0, ri = 0;
    uint32_t phase = 0;
    while (walk.next(b, p, st)) {
        if (st.last && walk.t >= walk.t1) break;  // the final stage: the consumers add it up
        bool got = true;
        if (lane == 0) got = mbar_wait_bounded(empty0 + 8 * slot, phase);
        got = __shfl_sync(0xffffffffu, got, 0);
        __syncwarp();  // the partials, released with the slot, are seen by every lane
        if (!got) {
            if (lane == 0) record_error(p.err, kErrConsumerWait);
            return;
        }
        if (st.last) {
            const MmaMat &m = b.m[MAXB == 1 ? 0 : st.mat];
            mma_finish_tile<NW>(p, red, ri, m.y, m.n_out, st.tile, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(reduced0 + 8 * slot);
        if (++ri == R) ri = 0;
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
    }
}

// ------------------------------------------------------------------ kernel
// Shared memory: mbarriers | panel | partial outputs [red_slots][warps][32]
// float4 | ring of n_stages stages.
// Warps of a launch: NW consumers, then the producers (one in register mode,
// two with a panel) and, in register mode, the reducer.
__host__ __device__ constexpr int mma_producers(int bmode) { return bmode == kMmaRegs ? 1 : 2; }
__host__ __device__ constexpr int mma_warps(int bmode, int nw) { return nw + mma_producers(bmode) + (bmode == kMmaRegs ? 1 : 0); }

template <class T, int BMODE, int NW, int MAXB>
__global__ void __launch_bounds__(mma_warps(BMODE, NW) * 32, 1) gemv_mma_kernel(const MmaParams p, const MmaBatch<MAXB> b) {
    constexpr bool B16 = BMODE == kMmaPanel16;
    constexpr bool REGS = BMODE == kMmaRegs;
    constexpr bool RED = REGS;  // a reducer warp
    constexpr int NP = mma_producers(BMODE);
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t full0 = smem_addr(smem);
    const uint32_t empty0 = full0 + 8 * kMmaMaxStages;
    const uint32_t reduced0 = full0 + 2 * 8 * kMmaMaxStages + 4 * 2 * kMmaMaxStages;
    uint8_t *pan = smem + kMmaHeaderBytes;
    float4 *red = reinterpret_cast<float4 *>(pan + p.panel_bytes);
    uint8_t *ring = pan + p.panel_bytes + p.red_slots * mma_red_bytes(NW);
    // warps done with the tile of each partial buffer (without a reducer), or with the final tile ([0])
    int *red_count = reinterpret_cast<int *>(smem + 2 * 8 * kMmaMaxStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = p.n_stages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, NP);
            mbar_init(empty0 + 8 * s, NW);
        }
        for (int r = 0; r < p.red_slots; ++r) red_count[r] = 0;
        for (int r = 0; r < S; ++r) mbar_init(reduced0 + 8 * r, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_allow_dependents();

    if (warp >= NW && warp < NW + NP) {
        mma_producer<T, RED, NP, MAXB>(p, b, ring, full0, empty0, reduced0, lane, warp - NW);
        return;
    }
    if (RED && warp == NW + NP) {
        mma_reducer<NW, MAXB>(p, b, red, empty0, reduced0, lane);
        return;
    }

    // ---- consumers ----
    pdl_wait_prior_grids();  // the activations may come from the previous kernel
    const int g = lane >> 2;
    const int sra = mma_stage_row(g), srb = mma_stage_row(g + 8);
    const uint32_t pan_a = smem_addr(pan), ring_a = smem_addr(ring);
    bool failed = false;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    MmaWalk walk = mma_cta_walk(p, b);
    MmaStage st;
    int cur = -1;
    MmaStage fin = {};
    int fin_ri = -1;  // partial buffer of the CTA's final tile
    constexpr int RB = 2;  // REGS: blocks a warp keeps (warp, warp + NW)
    uint32_t breg[RB][kMmaRecords][4];
    uint2 bcorr[RB], bdx[RB], bbs[RB];
    // slot = k mod S, its phase (k / S) & 1 and the partial buffer k mod red_slots, kept incrementally
    int slot = 0, ri = 0;
    uint32_t phase = 0;
    for (int k = 0; walk.next(b, p, st); ++k) {
        if (st.mat != cur) {  // a new matrix: its activations
            if constexpr (REGS) {
#pragma unroll
                for (int i = 0; i < RB; ++i)
                    if (warp + i * NW < p.nb)
                        mma_load_regs<T>(b.m[MAXB == 1 ? 0 : st.mat].xq, p.nb, p.nv, warp + i * NW, lane, breg[i],
                                         bcorr[i], bdx[i], bbs[i]);
            } else {
                if (cur >= 0) named_barrier(1, NW * 32);
                if constexpr (T::kActBytes == 0)
                    mma_build_panel<T, B16>(p, b.m[MAXB == 1 ? 0 : st.mat].xq, pan, threadIdx.x, NW * 32);
                else
                    mma_build_panel_q8<T, B16>(p, b.m[MAXB == 1 ? 0 : st.mat].xq, pan, threadIdx.x, NW * 32);
                named_barrier(1, NW * 32);
            }
            cur = st.mat;
        }
        if (!failed) {
            // every lane waits (each needs the acquire); the warp agrees on
            // the outcome, since mma.sync needs all 32 lanes
            const bool got = mbar_wait_bounded(full0 + 8 * slot, phase);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) record_error(p.err, kErrConsumerWait);
                failed = true;
            }
        }
        if (!failed) {
            const uint32_t sb = ring_a + static_cast<uint32_t>(slot * p.stage_bytes);
            // row sr of the stage: group sr/4 at sr/4 * gpitch, row sr%4 of it at
            // (sr%4) * rpitch, plus the copy's offset from its 16-byte window
            // only the offset modulo 16 is needed, so 32-bit (wrapping) products suffice
            const uint32_t row0 = static_cast<uint32_t>(st.tile) * kMmaTileRows;
            const uint32_t rbytes = static_cast<uint32_t>(p.row_bytes);
            const uint32_t koff = static_cast<uint32_t>(st.kc * p.kb * T::kBlockBytes);
            const uint32_t ca = (p.contig ? row0 + (sra & ~3) : row0 + sra) * rbytes + koff;
            const uint32_t cb = (p.contig ? row0 + (srb & ~3) : row0 + srb) * rbytes + koff;
            const uint32_t ra = sb + static_cast<uint32_t>((sra >> 2) * p.gpitch + (sra & 3) * p.rpitch) + (ca & 15u);
            const uint32_t rb = sb + static_cast<uint32_t>((srb >> 2) * p.gpitch + (srb & 3) * p.rpitch) + (cb & 15u);
            const int kbt = min(p.kb, p.nb - st.kc * p.kb);
            const uint32_t rec0 = pan_a + static_cast<uint32_t>(st.kc * p.kb * p.rec_bytes);
            if constexpr (REGS) {
                // both blocks in one straight-line sequence when the warp has
                // two, so the scheduler can interleave their dependency chains
                const uint32_t o0 = static_cast<uint32_t>(warp * T::kBlockBytes);
                const uint32_t o1 = static_cast<uint32_t>((warp + NW) * T::kBlockBytes);
                if (warp + NW < kbt) {
                    T::tile_block(ra + o0, rb + o0, MmaRegB{breg[0], bcorr[0], bdx[0], bbs[0]}, lane, acc);
                    T::tile_block(ra + o1, rb + o1, MmaRegB{breg[1], bcorr[1], bdx[1], bbs[1]}, lane, acc);
                } else if (warp < kbt) {
                    T::tile_block(ra + o0, rb + o0, MmaRegB{breg[0], bcorr[0], bdx[0], bbs[0]}, lane, acc);
                }
            } else {
                for (int kb = warp; kb < kbt; kb += NW)
                    T::tile_block(ra + kb * T::kBlockBytes, rb + kb * T::kBlockBytes,
                                  MmaSmemB<B16, T::kHiScaled>{rec0 + static_cast<uint32_t>(kb * p.rec_bytes), lane},
                                  lane, acc);
            }
        }
        bool last_warp = false;
        if (st.last) {
            // this warp's share of the tile, added up by the reducer warp (the
            // CTA's final tile: by the last consumer warp, after the loop) or,
            // without a reducer, by the last warp to get here
            red[(ri * NW + warp) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
            if (RED) {
                if (walk.t >= walk.t1) {
                    fin = st;
                    fin_ri = ri;
                }
            } else {
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    __threadfence_block();
                    last = atomicAdd(red_count + ri, 1) == NW - 1;
                }
                last_warp = __shfl_sync(0xffffffffu, last, 0);
                __syncwarp();  // orders lane 0's observation before every lane's reads
                if (last_warp) {
                    __threadfence_block();
                    const bool doubled = p.red_slots > S;
                    if (doubled && lane == 0) mbar_arrive(empty0 + 8 * slot);  // the slot is free already
                    const MmaMat &m = b.m[MAXB == 1 ? 0 : st.mat];
                    if (!failed) mma_finish_tile<NW>(p, red, ri, m.y, m.n_out, st.tile, lane);
                    __syncwarp();
                    if (lane == 0) {
                        red_count[ri] = 0;
                        if (!doubled) mbar_arrive(empty0 + 8 * slot);
                    }
                }
            }
        }
        if (!last_warp) {
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * slot);  // releases the slot (and the partials)
        }
        if (++ri == p.red_slots) ri = 0;
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (RED && fin_ri >= 0) {  // the last warp to get here adds up the final tile
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(red_count, 1) == NW - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();  // orders lane 0's observation before every lane's reads
        if (last) {
            __threadfence_block();
            const MmaMat &m = b.m[MAXB == 1 ? 0 : fin.mat];
            mma_finish_tile<NW>(p, red, fin_ri, m.y, m.n_out, fin.tile, lane);
        }
    }
}

}  // namespace qg

namespace qg {

// Host side: grid, shared memory and instance of one launch.
struct MmaLaunch {
    int grid;
    int smem;
    int smem_optin;  // the device's opt-in shared-memory limit per CTA
    int mode;        // MmaBMode
    int warps;       // consumer warps (8 with registers, 16 with a panel)
};

}  // namespace qg
