// gemv_tc.cuh - the Q4_K GEMV for several vectors on the 5th-generation tensor
// cores (tcgen05): Y[v][o] = sum over the blocks of row o of
// d_x * (d_w * S_q - dmin_w * S_m), with S_q = sum_j sc_j sum_i q_i a_i and
// S_m = sum_j m_j (bsum_2j + bsum_2j+1) ("Quantization" (rml), Quantized dot
// products and K-quants; "量化格式" (candle), the Q4K and Q8K block tables).
//
// Why tcgen05 here. With 3..8 vectors every weight code meets up to 8
// activation codes: a dense contraction. The legacy mma.sync form keeps every
// weight code in a register fragment of the warp that issues the mma and
// applies the sub-block scales to f32 accumulators afterwards; its warps are
// bound by that integer work and by latency. Here tcgen05.mma.kind::f16
// (M = 128, N = 64, K = 16) takes
//  * A (the weights) from tensor memory: lane m holds one (row, block) pair
//    of a 16-row tile -- 16 rows x 8 consecutive blocks per block group.
//    Converter threads own one lane each, unpack four codes per instruction
//    and fold the sub-block scale into the f16 operand with one f16x2
//    multiply;
//  * B (the activations) from a 128-byte-swizzled K-major f16 panel in shared
//    memory, built once per matrix from the Q8_K blocks: column n = 8 j + v
//    holds vector v's codes of block j of the group. So D[m][8 j(m) + v] is
//    the lane's block sum for vector v; the other 56 columns of a lane pair
//    it with the wrong block and are not read. An mma costs about the same
//    for N = 16..64, so the unread columns are nearly free, and a tile's rows
//    arrive as whole rows: the weights stream in large contiguous bulk
//    copies, 37 KB a stage, four stages in flight;
//  * D in tensor memory: k-steps 0..7 and 8..15 go to two accumulators (one
//    per issuing warp), added when read back.
// Exactness: a code q enters as the f16 subnormal q * 2^-24 (bit pattern q),
// times the scale sc (an exact f16 integer; sc / 16 for high nibbles, which
// are masked in place as 16 q) -- sc * q * 2^-24 <= 945 * 2^-24, an exact
// subnormal. Activation codes (-127..127) are exact f16 integers. Every
// partial sum of a block is an integer times 2^-24, so the f32 accumulators
// hold S_q * 2^-24 exactly while |S_q| < 2^24 (random blocks stay far below;
// at the extreme one rounding of 2^-24 relative). The minimum term S_m is a
// small integer sum formed with dp2a from the 6-bit mins and the activation
// block's 32-element sums.
//
// Structure (one CTA per SM, 11 warps):
//  * warps 0..7: converters. Warp w owns tensor-memory lanes 32 (w % 4) ..
//    +31; lane l of it takes row 4 (l % 4) + l / 8 and block 2 (w % 4) +
//    (l / 4) % 2 of each group, and half h = w / 4 of that block's codes
//    (chunks 2h, 2h+1: sub-blocks 4h..4h+3). Half 0 reads D back; half 1
//    forms the minimum term. Both keep y partial sums, added in a fixed order
//    at the end of each tile.
//  * warps 8, 9: lane 0 of warp 8 + h issues the 8 mmas of half h of every
//    group as soon as the four half-h converters are done, and commits them
//    to the group's mbarrier. Warp 8 also allocates tensor memory.
//  * warp 10: the producer. A stage is one 16-row tile of whole rows, copied
//    as 4 bulk copies of 4 contiguous rows into groups at a pitch of 32
//    modulo 128 bytes; the lane-to-(row, block) map above puts the 8 lanes of
//    each 128-bit load phase on 8 different bank groups.
//  * A CTA owns a balanced contiguous range of the launch's 16-row tiles
//    (matrices of a batch numbered consecutively).
//  * All waits are bounded (about 1 s) and also give up when another thread
//    of the CTA has recorded an error; tensor memory is freed on every path.
//
// Measured on GB300 against the mma.sync kernel on the 32-layer stack's
// 192 Q4_K matrices (8 vectors): 3.0-3.9 TB/s for the variants of this
// design against 4.5 TB/s, so it is off by default (QG_TC). What bounds it:
// an mma instruction holds its issuing warp for 45-77 cycles and the SM takes
// about one every 32 cycles, a 128-row-block group needs 16 of them, and the
// 512 tensor-memory columns hold only three A buffers and two D buffers, so
// the chain commit -> read-back -> conversion of the buffer's next group
// leaves the converters waiting for the mmas of the group before last.
#pragma once

#include "tc_common.cuh"

namespace qg {

constexpr int kTcRows = 16;          // rows of a tile (one stage)
constexpr int kTcGroupBlocks = 8;    // blocks of a row per mma group
constexpr int kTcM = 128;            // M of the mma = tensor-memory lanes = 16 rows x 8 blocks
constexpr int kTcN = 64;             // N of the mma = 8 blocks x 8 vectors
constexpr int kTcConvWarps = 8;      // converter warps
constexpr int kTcIssuers = 2;        // mma-issuing warps (groups alternate between them)
constexpr int kTcThreads = (kTcConvWarps + kTcIssuers + 1) * 32;
constexpr int kTcABufs = 3;          // A buffers in tensor memory
constexpr int kTcDBufs = 2;          // D buffers in tensor memory
constexpr int kTcTmemCols = 512;
constexpr int kTcMaxStages = 8;
constexpr int kTcMaxBatch = 256;     // matrices per launch (their table is a kernel parameter)
constexpr int kTcBlockBytes = 144;   // Q4_K block
constexpr int kTcMaxBlocks = 16;     // blocks per row (whole rows travel per stage)
constexpr int kTcAtom = 1024;        // 8 rows x 128 bytes of the swizzled panel

// Tensor-memory columns: A buffer b (128 columns: 256 f16 codes), D buffer d
// (64 f32 columns).
__host__ __device__ constexpr uint32_t tc_col_a(int b) { return 128u * static_cast<uint32_t>(b); }
__host__ __device__ constexpr uint32_t tc_col_d(int d) { return 384u + 64u * static_cast<uint32_t>(d); }

// Shared-memory layout, offsets from a 1024-aligned base: header (barriers,
// tensor-memory address, abort flag), y partial sums, the d_x table, the
// 32-element bsums table, the activation panel (block group g: atom
// 32 g + 8 kk + j for k-atom kk and block j) and the ring of stages.
constexpr int kTcHdrBytes = 1024;
constexpr int kTcRedBytes = 2 * kTcConvWarps * kTcRows * 8 * 4;  // 2 buffers x 8 warps x 16 rows x 8 vectors
__host__ __device__ constexpr int tc_dx_bytes(int nb) { return (nb * 32 + kTcAtom - 1) / kTcAtom * kTcAtom; }
__host__ __device__ constexpr int tc_bs_bytes(int nb) { return (nb * 8 * 16 + kTcAtom - 1) / kTcAtom * kTcAtom; }
__host__ __device__ constexpr int tc_groups(int nb) { return nb / kTcGroupBlocks; }
__host__ __device__ constexpr int tc_panel_bytes(int nb) { return 32 * tc_groups(nb) * kTcAtom; }
// A stage: 4 groups of 4 rows at a pitch of 32 modulo 128 bytes.
__host__ __device__ constexpr int tc_gpitch(int nb) { return (4 * nb * kTcBlockBytes + 127) / 128 * 128 + 32; }
__host__ __device__ constexpr int tc_stage_bytes(int nb) { return (4 * tc_gpitch(nb) + 127) / 128 * 128; }
__host__ __device__ constexpr int tc_smem_bytes(int nb, int stages) {
    return kTcAtom /* base alignment */ + kTcHdrBytes + kTcRedBytes + tc_dx_bytes(nb) + tc_bs_bytes(nb) +
           tc_panel_bytes(nb) + stages * tc_stage_bytes(nb);
}

struct TcMat {
    const uint8_t *W;   // [n_out][nb * 144], 16-byte aligned
    const uint8_t *xq;  // byte-exact Q8_K blocks [n_vec][nb]
    float *y;           // [n_vec][n_out]
    int64_t tile_base;  // launch-wide index of the matrix's first 16-row tile
    int n_out;
    int pad;
};

template <int MAXB>
struct TcBatch {
    TcMat m[MAXB];
};

struct TcParams {
    int32_t *err;
    int64_t total_tiles;
    int n_mats;
    int nb;        // blocks per row (8 or 16)
    int nv;        // vectors (1..8)
    int n_stages;  // ring depth (2..kTcMaxStages)
};

// Eight mmas over consecutive k-steps s = 0..7 into one accumulator: A at
// a_t + 8 s columns, B at descriptor b0 (steps 0..3) or b4 (steps 4..7),
// advanced by 32 bytes a step within a 128-byte swizzle row; the first step
// overwrites D unless acc_first. All operands are formed inside one asm statement, so the
// issuing thread spends its time in the mma instructions (each holds the
// issuing warp for tens of cycles), not in dependent arithmetic between them.
__device__ __forceinline__ void tc_mma_k8(uint32_t d_t, uint32_t a_t, uint64_t b0, uint64_t b4, uint32_t idesc,
                                          uint32_t acc_first) {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b64 b1, b2, b3, b5, b6, b7;\n\t"
        ".reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
        "setp.ne.u32 pf, %5, 0;\n\tsetp.eq.u32 pt, %4, %4;\n\t"
        "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
        "add.s64 b5, %3, 2;\n\tadd.s64 b6, %3, 4;\n\tadd.s64 b7, %3, 6;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\tadd.u32 a4, %1, 32;\n\t"
        "add.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\tadd.u32 a7, %1, 56;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, pf;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], %3, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %4, pt;\n\t}" ::"r"(d_t),
        "r"(a_t), "l"(b0), "l"(b4), "r"(idesc), "r"(acc_first)
        : "memory");
}

// 32 lanes x 16 columns into registers, waited for in the same statement.
__device__ __forceinline__ void tc_ld16_wait(uint32_t ta, uint32_t (&a)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
          "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15])
        : "r"(ta)
        : "memory");
}
__device__ __forceinline__ void tc_ld16x2_wait(uint32_t ta, uint32_t tb, uint32_t (&a)[16], uint32_t (&b)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3]), "=r"(a[4]), "=r"(a[5]), "=r"(a[6]), "=r"(a[7]),
          "=r"(a[8]), "=r"(a[9]), "=r"(a[10]), "=r"(a[11]), "=r"(a[12]), "=r"(a[13]), "=r"(a[14]), "=r"(a[15]),
          "=r"(b[0]), "=r"(b[1]), "=r"(b[2]), "=r"(b[3]), "=r"(b[4]), "=r"(b[5]), "=r"(b[6]), "=r"(b[7]),
          "=r"(b[8]), "=r"(b[9]), "=r"(b[10]), "=r"(b[11]), "=r"(b[12]), "=r"(b[13]), "=r"(b[14]), "=r"(b[15])
        : "r"(ta), "r"(tb)
        : "memory");
}

// Instruction descriptor: N = 64, M = 128.
constexpr uint32_t kTcIdesc = tc_idesc_f16(kTcM, kTcN);

// Walks a CTA's tiles. Every role runs the same walk.
struct TcWalk {
    int64_t t, t1;
    int m;
    int64_t next_base;

    template <int MAXB>
    __device__ __forceinline__ void init(const TcParams &p, const TcBatch<MAXB> &b) {
        t = static_cast<int64_t>(blockIdx.x) * p.total_tiles / gridDim.x;
        t1 = static_cast<int64_t>(blockIdx.x + 1) * p.total_tiles / gridDim.x;
        m = 0;
        next_base = p.n_mats > 1 ? b.m[1].tile_base : INT64_MAX;
    }
    // The next tile: matrix and tile within the matrix.
    template <int MAXB>
    __device__ __forceinline__ bool next(const TcParams &p, const TcBatch<MAXB> &b, int &mat, int &tile) {
        if (t >= t1) return false;
        while (t >= next_base) {
            ++m;
            next_base = m + 1 < p.n_mats ? b.m[m + 1].tile_base : INT64_MAX;
        }
        mat = m;
        tile = static_cast<int>(t - b.m[m].tile_base);
        ++t;
        return true;
    }
};

// Lane l of a converter warp: tile row 4 (l % 4) + l / 8 (copy group l % 4,
// row l / 8 of it) and block 2 q + (l / 4) % 2 of the group, q the warp's
// lane quarter.
__device__ __forceinline__ int tc_lane_row(int l) { return 4 * (l & 3) + (l >> 3); }
__device__ __forceinline__ int tc_lane_jb(int l) { return (l >> 2) & 1; }

// The activation panel of one matrix from its Q8_K blocks (all 256 converter
// threads). For block group g, atom 32 g + 8 kk + j holds, in row v
// (vector), the 64 codes of chunk kk of block 8 g + j in the mma's k order:
// 16-byte chunk p is codes 64 kk + 4p + {0,2,1,3} then
// 64 kk + 32 + 4p + {0,2,1,3} (the order in which the converters emit the low
// and high nibbles of weight word p), at (p ^ v) * 16 in the row (128-byte
// swizzle). Rows of vectors >= nv are zero. Also the tables d_x[b][v] and
// bs32[b][v][j] (the 32-element sums of sub-block j, as int16).
__device__ __forceinline__ void tc_build_panel(const TcParams &p, const uint8_t *xq, uint8_t *pan, float *dx,
                                               uint4 *bs32, int tid) {
    const int nb = p.nb, nv = p.nv;
    constexpr int kThreads = kTcConvWarps * 32;
    const int n_chunks = nb * 4 * 8 * 8;  // blocks x chunks kk x vectors v x 16-byte chunks p
    for (int u = tid; u < n_chunks; u += kThreads) {
        const int pp = u & 7, v = (u >> 3) & 7, kk = (u >> 6) & 3, b = u >> 8;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (v < nv) {
            const uint8_t *qs = xq + (static_cast<size_t>(v) * nb + b) * 292 + 4;
            const uint32_t wl = __ldg(reinterpret_cast<const uint32_t *>(qs + 64 * kk + 4 * pp));
            const uint32_t wh = __ldg(reinterpret_cast<const uint32_t *>(qs + 64 * kk + 32 + 4 * pp));
            const uint32_t xl = __byte_perm(wl, 0u, 0x3120) ^ 0x80808080u;
            const uint32_t xh = __byte_perm(wh, 0u, 0x3120) ^ 0x80808080u;
            // biased byte c -> f16 (1024 + c) -> minus 1152
            o.x = hsub2(__byte_perm(xl, 0x64646464u, 0x4140), 0x64806480u);
            o.y = hsub2(__byte_perm(xl, 0x64646464u, 0x4342), 0x64806480u);
            o.z = hsub2(__byte_perm(xh, 0x64646464u, 0x4140), 0x64806480u);
            o.w = hsub2(__byte_perm(xh, 0x64646464u, 0x4342), 0x64806480u);
        }
        const int g = b / kTcGroupBlocks, j = b % kTcGroupBlocks;
        uint8_t *atom = pan + static_cast<size_t>(32 * g + 8 * kk + j) * kTcAtom;
        *reinterpret_cast<uint4 *>(atom + v * 128 + ((pp ^ v) << 4)) = o;
    }
    for (int u = tid; u < nb * 8; u += kThreads) {
        const int b = u >> 3, v = u & 7;
        float d = 0.0f;
        uint32_t s[4] = {0u, 0u, 0u, 0u};
        if (v < nv) {
            const uint8_t *blk = xq + (static_cast<size_t>(v) * nb + b) * 292;
            d = __ldg(reinterpret_cast<const float *>(blk));
            const uint32_t *bw = reinterpret_cast<const uint32_t *>(blk + 260);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t w0 = __ldg(bw + 2 * i), w1 = __ldg(bw + 2 * i + 1);
                const int s0 = static_cast<int16_t>(w0 & 0xFFFFu) + static_cast<int16_t>(w0 >> 16);
                const int s1 = static_cast<int16_t>(w1 & 0xFFFFu) + static_cast<int16_t>(w1 >> 16);
                s[i] = (static_cast<uint32_t>(s0) & 0xFFFFu) | (static_cast<uint32_t>(s1) << 16);
            }
        }
        dx[u] = d;
        bs32[u] = make_uint4(s[0], s[1], s[2], s[3]);
    }
}

// One converter thread's half h of a block (its bytes at `blkp`): columns
// 64h .. 64h + 63 of the A buffer at a_t (chunk c at a_t + 32 c). Returns the
// block's first 16 bytes (d, dmin, packed scales and mins).
__device__ __forceinline__ uint4 tc_convert_half(uint32_t blkp, int h, uint32_t a_t) {
    const uint4 hd = ld_s128(blkp);
    // 6-bit scales of sub-blocks 4h..4h+3, one per byte
    const uint32_t scw = h == 0 ? (hd.y & 0x3F3F3F3Fu) : ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u));
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * h + cc;
        // f16 pairs (sc, sc) for the low nibbles and (sc / 16, sc / 16) for the
        // high ones: bytes -> 1024 + sc -> exact arithmetic
        const uint32_t ke = static_cast<uint32_t>(2 * cc), ko = ke + 1;
        const uint32_t me = hsub2(__byte_perm(scw, 0x64u, ke | 0x40u | (ke << 8) | 0x4000u), 0x64006400u);
        const uint32_t mo = hfma2(__byte_perm(scw, 0x64u, ko | 0x40u | (ko << 8) | 0x4000u), 0x2C002C00u, 0xD400D400u);
        const uint4 q0 = ld_s128(blkp + 16 + 32 * c), q1 = ld_s128(blkp + 32 + 32 * c);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        uint32_t v[32];
#pragma unroll
        for (int pp = 0; pp < 8; ++pp) {
            const uint32_t t = w[pp] >> 8;
            v[4 * pp + 0] = hmul2(w[pp] & 0x000F000Fu, me);
            v[4 * pp + 1] = hmul2(t & 0x000F000Fu, me);
            v[4 * pp + 2] = hmul2(w[pp] & 0x00F000F0u, mo);
            v[4 * pp + 3] = hmul2(t & 0x00F000F0u, mo);
        }
        tc_st32(a_t + 32u * static_cast<uint32_t>(c), v);
    }
    return hd;
}

// ------------------------------------------------------------------ kernel
template <int MAXB>
__global__ void __launch_bounds__(kTcThreads, 1) gemv_tc_q4_k_kernel(const TcParams p, const __grid_constant__ TcBatch<MAXB> b) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_a = smem_addr(smem_raw);
    const uint32_t base_a = (raw_a + kTcAtom - 1) & ~static_cast<uint32_t>(kTcAtom - 1);
    uint8_t *base = smem_raw + (base_a - raw_a);
    const int nb = p.nb, S = p.n_stages, G = tc_groups(nb);
    // header: full[8] | empty[8] | afull[3] | mdone[3] | dfree[2] | mfinal | tmem address | abort flag
    const uint32_t full0 = base_a, empty0 = base_a + 64, afull0 = base_a + 128, mdone0 = base_a + 152;
    const uint32_t dfree0 = base_a + 176, mfinal = base_a + 192;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + 200);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + 204);
    float *red = reinterpret_cast<float *>(base + kTcHdrBytes);  // [2][8 warps][16 rows][8 vectors]
    float *dx = reinterpret_cast<float *>(base + kTcHdrBytes + kTcRedBytes);
    uint4 *bs32 = reinterpret_cast<uint4 *>(base + kTcHdrBytes + kTcRedBytes + tc_dx_bytes(nb));
    uint8_t *pan = base + kTcHdrBytes + kTcRedBytes + tc_dx_bytes(nb) + tc_bs_bytes(nb);
    const uint32_t pan_a = smem_addr(pan);
    const uint32_t ring_a = pan_a + static_cast<uint32_t>(tc_panel_bytes(nb));
    const int gpitch = tc_gpitch(nb), stage_bytes = tc_stage_bytes(nb);
    const int64_t row_bytes = static_cast<int64_t>(nb) * kTcBlockBytes;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kTcConvWarps);
        }
        for (int i = 0; i < kTcABufs; ++i) {
            mbar_init(afull0 + 8 * i, kTcConvWarps);
            mbar_init(mdone0 + 8 * i, 1);
        }
        for (int i = 0; i < kTcDBufs; ++i) mbar_init(dfree0 + 8 * i, kTcConvWarps / 2);
        mbar_init(mfinal, kTcIssuers);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcConvWarps) {
        tc_alloc(smem_addr(tmem_slot), kTcTmemCols);
        tc_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_allow_dependents();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTcConvWarps + kTcIssuers) {
        // ---------------- producer: one stage per 16-row tile, 4 copies of 4 rows
        const uint64_t policy = l2_evict_first_policy();
        TcWalk walk;
        walk.init(p, b);
        int mat, tile, slot = 0;
        uint32_t phase = 0;
        int64_t issued = 0;
        while (walk.next(p, b, mat, tile)) {
            const TcMat &mm = b.m[mat];
            const int rows = min(kTcRows, mm.n_out - tile * kTcRows);
            const int mine = lane < 4 ? max(0, min(4, rows - 4 * lane)) : 0;  // rows of copy group `lane`
            const uint32_t bytes = static_cast<uint32_t>(mine * row_bytes);
            uint32_t total = bytes;
#pragma unroll
            for (int o = 2; o >= 1; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
            bool got = true;
            if (issued >= S && lane == 0) got = tc_wait(empty0 + 8 * slot, phase ^ 1u, abort_flag);
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                if (lane == 0) {
                    record_error(p.err, kErrProducerWait);
                    *abort_flag = 1;
                }
                break;
            }
            if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * slot, total);
            __syncwarp();
            if (bytes > 0)
                bulk_copy_g2s(ring_a + static_cast<uint32_t>(slot * stage_bytes + lane * gpitch),
                              mm.W + (static_cast<int64_t>(tile) * kTcRows + 4 * lane) * row_bytes, bytes,
                              full0 + 8 * slot, policy);
            ++issued;
            if (++slot == S) {
                slot = 0;
                phase ^= 1u;
            }
        }
        // leave no copy in flight into this CTA's shared memory
        if (lane == 0) {
            for (int64_t k = issued > S ? issued - S : 0; k < issued; ++k) {
                const int sl = static_cast<int>(k % S);
                if (!mbar_wait_bounded(full0 + 8 * sl, static_cast<uint32_t>((k / S) & 1))) {
                    record_error(p.err, kErrDrainWait);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp >= kTcConvWarps) {
        // ---------------- mma issuers: warp kTcConvWarps + k takes groups i = k mod 2
        if (lane == 0) {
            const int k = warp - kTcConvWarps;
            TcWalk walk;
            walk.init(p, b);
            int mat, tile;
            int64_t i = 0;
            int a = 0, d = 0;  // i mod 3, i mod 2
            bool ok = true;
            const uint32_t idesc = kTcIdesc;
            while (ok && walk.next(p, b, mat, tile)) {
                for (int g = 0; g < G; ++g, ++i) {
                    if ((i & 1) == k) {
                        // A of group i written; D buffer free (group i - 2 read back)
                        if (!tc_wait(afull0 + 8 * a, static_cast<uint32_t>((i / kTcABufs) & 1), abort_flag) ||
                            (i >= kTcDBufs &&
                             !tc_wait(dfree0 + 8 * d, static_cast<uint32_t>(((i - kTcDBufs) / kTcDBufs) & 1), abort_flag))) {
                            record_error(p.err, kErrConsumerWait);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        // k-steps 0..15: k-atom s / 4 of group g (8 atoms apart), 32 bytes per step
                        const uint64_t d0 = tc_smem_desc(pan_a + static_cast<uint32_t>(32 * g * kTcAtom), kTcAtom);
                        const uint64_t atom8 = static_cast<uint64_t>((8 * kTcAtom) >> 4);
                        const uint32_t dt = tmem + tc_col_d(d), at = tmem + tc_col_a(a);
                        tc_mma_k8(dt, at, d0, d0 + atom8, idesc, 0u);
                        tc_mma_k8(dt, at + 64u, d0 + 2 * atom8, d0 + 3 * atom8, idesc, 1u);
                        tc_commit(mdone0 + 8 * a);
                    }
                    if (++a == kTcABufs) a = 0;
                    d ^= 1;
                }
            }
            // every mma of this warp complete before tensor memory is freed
            tc_commit(mfinal);
            if (!mbar_wait_bounded(mfinal, 0u)) record_error(p.err, kErrDrainWait);
        }
        __syncwarp();
    } else {
        // ---------------- converters
        // A warp that fails a wait keeps walking without waiting or working,
        // so that every converter reaches the same named barriers.
        const int q = warp & 3, h = warp >> 2;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);  // this warp's lanes
        const int lrow = tc_lane_row(lane), jb = tc_lane_jb(lane);
        const int lblk = 2 * q + jb;  // block of the group
        const uint32_t lane_off = static_cast<uint32_t>((lane & 3) * gpitch + (lane >> 3) * row_bytes + lblk * kTcBlockBytes);
        TcWalk walk;
        walk.init(p, b);
        int mat, tile, cur = -1;
        int slot = 0, a = 0, rg = 0, rred = 0;
        uint32_t sphase = 0;
        int64_t i = 0, rb = 0;        // groups converted / read back
        int rb_mat = 0, rb_tile = 0;  // tile of the group being read back
        // per A buffer: the block header words the read-back needs (half 0:
        // d; half 1: dmin and the packed mins)
        uint32_t hq0[kTcABufs] = {0u, 0u, 0u}, hq1[kTcABufs] = {0u, 0u, 0u}, hq2[kTcABufs] = {0u, 0u, 0u};
        float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
        bool ok = true;
        // tile of each group read back: the conversion walk's history by tile
        // number mod 4 (read-back lags conversion by at most two groups)
        int hist_mat[4] = {0, 0, 0, 0}, hist_tile[4] = {0, 0, 0, 0};
        int64_t ctile = 0, rtile = 0;  // tiles started by conversion / by read-back
        // Read back group rb once its mmas are complete (which also frees its A
        // buffer): half 0 adds d_x d 2^24 D to its y partials and frees the D
        // buffer, half 1 adds -d_x dmin S_m. At the tile's last group every
        // converter stores its partials, and after a barrier 128 threads add
        // the 16 partials of each (row, vector) in a fixed order and store y.
        auto read_back = [&]() {
            const int ra = static_cast<int>(rb % kTcABufs), rd = static_cast<int>(rb & 1);
            if (ok && !tc_wait(mdone0 + 8 * ra, static_cast<uint32_t>((rb / kTcABufs) & 1), abort_flag)) {
                if (lane == 0) {
                    record_error(p.err, kErrConsumerWait);
                    *abort_flag = 1;
                }
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);
            tc_fence_after();
            if (rg == 0) {
                rb_mat = hist_mat[rtile & 3];
                rb_tile = hist_tile[rtile & 3];
                ++rtile;
            }
            const int blk = kTcGroupBlocks * rg + lblk;
            const float4 x0 = reinterpret_cast<const float4 *>(dx)[2 * blk];
            const float4 x1 = reinterpret_cast<const float4 *>(dx)[2 * blk + 1];
            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const uint32_t hx = ra == 0 ? hq0[0] : (ra == 1 ? hq0[1] : hq0[2]);
            if (ok && h == 0) {
                uint32_t d0[16];
                tc_ld16_wait(tl + tc_col_d(rd) + 16u * static_cast<uint32_t>(q), d0);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dfree0 + 8 * rd);
                const float dw = f16_bits_to_f32(hx) * 16777216.0f;
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[v] = fmaf(xv[v] * dw, __uint_as_float(jb ? d0[8 + v] : d0[v]), acc[v]);
            } else if (ok) {
                // S_m[v] = sum_j m_j bs32_j[v], exact in integers (dp2a: two
                // int16 sums times two unsigned mins each)
                const uint32_t hz = ra == 0 ? hq1[0] : (ra == 1 ? hq1[1] : hq1[2]);
                const uint32_t hw = ra == 0 ? hq2[0] : (ra == 1 ? hq2[1] : hq2[2]);
                const float dmn = f16_bits_to_f32(hx >> 16);
                const uint32_t m03 = hz & 0x3F3F3F3Fu;
                const uint32_t m47 = ((hw >> 4) & 0x0F0F0F0Fu) | ((hz >> 2) & 0x30303030u);
                const uint4 *bsb = bs32 + blk * 8;
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    const uint4 sv = bsb[v];
                    int sm = dp2a_lo_su(sv.x, m03, 0);
                    sm = dp2a_hi_su(sv.y, m03, sm);
                    sm = dp2a_lo_su(sv.z, m47, sm);
                    sm = dp2a_hi_su(sv.w, m47, sm);
                    acc[v] = fmaf(-xv[v] * dmn, static_cast<float>(sm), acc[v]);
                }
            }
            if (rg == G - 1) {
                // the tile's partial sums: fold the two blocks of the warp that
                // share a row (lanes l and l ^ 4), store, barrier, add in order
                float *rr = red + rred * (kTcConvWarps * kTcRows * 8);
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[v] += __shfl_xor_sync(0xffffffffu, acc[v], 4);
                if (ok && jb == 0) {
                    float4 *dst = reinterpret_cast<float4 *>(rr + (warp * kTcRows + lrow) * 8);
                    dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
                    dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
                }
                named_barrier(1, kTcConvWarps * 32);
                if (ok && threadIdx.x < kTcRows * 8) {
                    const TcMat &mm = b.m[rb_mat];
                    const int row = threadIdx.x & (kTcRows - 1), v = threadIdx.x >> 4;
                    float sum = 0.0f;
#pragma unroll
                    for (int w8 = 0; w8 < kTcConvWarps; ++w8) sum += rr[(w8 * kTcRows + row) * 8 + v];
                    const int orow = rb_tile * kTcRows + row;
                    if (v < p.nv && orow < mm.n_out) mm.y[static_cast<int64_t>(v) * mm.n_out + orow] = sum;
                }
                rred ^= 1;
#pragma unroll
                for (int v = 0; v < 8; ++v) acc[v] = 0.0f;
            }
            ++rb;
            if (++rg == G) rg = 0;
        };
        while (walk.next(p, b, mat, tile)) {
            if (mat != cur) {
                // a new matrix: finish every group of the previous one (its
                // mmas read the panel), then rebuild the panel
                while (rb < i) read_back();
                if (cur < 0) pdl_wait_prior_grids();  // the activations may come from the previous kernel
                named_barrier(1, kTcConvWarps * 32);
                if (!*abort_flag) tc_build_panel(p, b.m[mat].xq, pan, dx, bs32, threadIdx.x);
                fence_proxy_async_smem();
                named_barrier(1, kTcConvWarps * 32);
                cur = mat;
            }
            hist_mat[ctile & 3] = mat;
            hist_tile[ctile & 3] = tile;
            ++ctile;
            if (ok && !tc_wait(full0 + 8 * slot, sphase, abort_flag)) {
                if (lane == 0) {
                    record_error(p.err, kErrConsumerWait);
                    *abort_flag = 1;
                }
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);
            const uint32_t rowp = ring_a + static_cast<uint32_t>(slot * stage_bytes) + lane_off;
            for (int g = 0; g < G; ++g) {
                // A buffer i mod 3 is free: group i - 3 was read back (its mmas
                // complete) before group i - 1 was converted
                if (ok) {
                    const uint4 hd = tc_convert_half(rowp + static_cast<uint32_t>(g * kTcGroupBlocks * kTcBlockBytes), h,
                                                     tl + tc_col_a(a));
                    if (a == 0) {
                        hq0[0] = hd.x;
                        hq1[0] = hd.z;
                        hq2[0] = hd.w;
                    } else if (a == 1) {
                        hq0[1] = hd.x;
                        hq1[1] = hd.z;
                        hq2[1] = hd.w;
                    } else {
                        hq0[2] = hd.x;
                        hq1[2] = hd.z;
                        hq2[2] = hd.w;
                    }
                    tc_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(afull0 + 8 * a);
                }
                ++i;
                if (++a == kTcABufs) a = 0;
                // read back the group two behind the one just converted
                if (rb + 2 <= i - 1) read_back();
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(empty0 + 8 * slot);
            if (++slot == S) {
                slot = 0;
                sphase ^= 1u;
            }
        }
        while (rb < i) read_back();
    }
    // free tensor memory once every role is done with it
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTcConvWarps) tc_dealloc(tmem, kTcTmemCols);
}

}  // namespace qg
