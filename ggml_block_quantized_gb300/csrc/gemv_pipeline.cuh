// gemv_pipeline.cuh - the streaming block-quantized GEMV kernel.
//
// y[v][o] = sum over the blocks b of row o of (exact int32 block sum) x
// (block scales), for W in GGUF blocks and activations in the paired Q8_0 /
// Q8_K blocks ("Quantization" (rml), Quantized dot products; "Building Q8_0
// and Q4_0 Like ggml", Examples 10-11).
//
// Design (one CTA = 1 producer warp + 8 consumer warps):
//  * A launch covers one matrix or a batch of independent matrices with the
//    same type, row length and vector count; their rows are numbered
//    consecutively ("global rows"). Each CTA owns a balanced contiguous range
//    of global rows; within one matrix that is one contiguous byte range of
//    its W. The producer's lane 0 streams it into a ring of shared-memory
//    stages with 1-D bulk async copies (the TMA engine's non-tensor form),
//    each stage a whole number of rows of one matrix. A stage copies the 16-byte aligned
//    window that covers its rows, so rows of any byte length (Q6_K rows of
//    9030 bytes start 2-byte aligned) need no special case; the last < 16
//    bytes of W, which no aligned window may cover without reading past the
//    buffer, are copied with plain loads.
//  * Full/empty mbarriers hand stages between producer and consumers; every
//    wait is bounded (about 1 s) and reports through the device error word.
//  * The producer starts before the previous kernel on the stream has
//    finished (programmatic dependent launch): W does not depend on it. The
//    consumers wait for the previous grid before reading the activations.
//  * Consumers first stage the activations (every vector, the whole row
//    length) into shared memory in a per-type padded layout that makes the
//    hot loop's 128-bit shared loads bank-conflict free -- either copied from
//    byte-exact Q8_0/Q8_K blocks or, for small activations, quantized from
//    f32 x right there (the same rule, so the same bytes; it saves a
//    dependent launch per call) -- then for each
//    stage take kRowsPerWarp rows per `split` warps, interleaved. When a
//    CTA's stages move on to the next matrix of a batch, the consumers
//    stage that matrix's activations. Lanes are grouped per block
//    (kLanesPerBlock lanes share one block); each group forms the block's
//    exact int32 sums with __dp4a, combines them with warp shuffles, and the
//    group leader applies the block's float scales.
#pragma once

#include "qg_common.cuh"

namespace qg {

constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 16;
constexpr int kRowsPerWarp = 2;  // most rows a warp group takes per stage (its items are flattened over them)
// Vector counts whose two-row straight-line form fits the registers (no spills).
constexpr int kStraightNv = 1;
constexpr int kMaxBatch = 256;   // matrices per batched launch (their table is a kernel parameter)
// The producer issues only the first stages (GemvParams::pre_x, about 56 KiB)
// before the consumers' first activation loads have arrived: behind a deep
// queue of weight copies those loads wait for microseconds.
// Shared memory: header (kMaxStages full + kMaxStages empty mbarriers, the
// activations-arrived mbarrier, 8 bytes of padding) |
// staged activations | cross-warp partial sums (split > 1:
// [2 * n_stages][kConsumerWarps][kRowsPerWarp][NV] floats) | ring of stages.
constexpr int kHeaderBytes = 2 * 8 * kMaxStages + 16;

// One matrix of a launch.
struct GemvMat {
    const uint8_t *W;    // [n_out][row_bytes], 16-byte aligned
    const float *x;      // f32 activations [n_vec][n_in], quantized in the kernel; or null and
    const uint8_t *xq;   // byte-exact activation blocks [n_vec][nb] (Q8_0 or Q8_K)
    float *y;            // [n_vec][n_out]
    int32_t *isums;      // [n_vec][n_out][nb][kSums] (diagnostic mode only)
    int64_t row_base;    // global row of this matrix's row 0
    int n_out;
    int pad;
};

template <int MAXB>
struct GemvBatch {
    GemvMat m[MAXB];
};

// Geometry shared by every matrix of a launch.
struct GemvParams {
    int32_t *err;        // device error word
    int64_t row_bytes;   // bytes of one row (n_in / block elems * block bytes)
    int64_t total_rows;  // sum of n_out over the matrices
    int64_t rows_q;      // total_rows / gridDim.x and total_rows % gridDim.x: CTA b starts at global
    int rows_r;          // row b * rows_q + b * rows_r / gridDim.x (no 64-bit division in the kernel)
    int n_mats;
    int nb;              // blocks per row
    int rows_per_stage;  // (kConsumerWarps / split) * (1 or kRowsPerWarp)
    int split;           // consumer warps per row: 1, 2, 4 or 8
    int split_log2;      // log2(split)
    int n_stages;        // ring depth (2..kMaxStages)
    int stage_bytes;     // bytes per ring slot, multiple of 16
    int act_bytes;       // bytes of staged activations, multiple of 16
    int red_bytes;       // bytes of the cross-warp partial sums (split > 1), else 0
    int pre_x;           // stages issued before the consumers' first activation loads arrive (>= 1)
};

// Walks a CTA's global rows [g, g1) as stages of at most R rows that never
// cross a matrix boundary. Producer and consumers run the same walk.
struct StageWalk {
    int64_t g, g1;
    int m;
    int n_out;                // rows of matrix m
    int64_t base, next_base;  // row_base of matrices m and m+1 (cached: the table is kernel parameters)

    template <int MAXB>
    __device__ __forceinline__ bool next(const GemvBatch<MAXB> &b, int n_mats, int R, int &mat, int &r, int &rows) {
        if (g >= g1) return false;
        while (MAXB > 1 && g >= next_base) {  // (one matrix: a constant index, no local copy of the table)
            ++m;
            base = next_base;
            n_out = b.m[m].n_out;
            next_base = m + 1 < n_mats ? b.m[m + 1].row_base : INT64_MAX;
        }
        mat = m;
        r = static_cast<int>(g - base);
        int64_t left = n_out - r;
        if (g1 - g < left) left = g1 - g;
        rows = static_cast<int>(left < R ? left : R);
        g += rows;
        return true;
    }
};

// CTA b's rows: [floor(b * total / grid), floor((b + 1) * total / grid)),
// formed as b * q + floor(b * r / grid) with total = q * grid + r.
__device__ __forceinline__ int64_t cta_row_start(const GemvParams &p, unsigned b) {
    return static_cast<int64_t>(b) * p.rows_q + (b * static_cast<unsigned>(p.rows_r)) / gridDim.x;
}

template <int MAXB>
__device__ __forceinline__ StageWalk cta_rows(const GemvParams &p, const GemvBatch<MAXB> &b) {
    StageWalk w;
    w.g = cta_row_start(p, blockIdx.x);
    w.g1 = cta_row_start(p, blockIdx.x + 1);
    w.m = 0;
    w.n_out = b.m[0].n_out;
    w.base = 0;
    w.next_base = MAXB > 1 && p.n_mats > 1 ? b.m[MAXB > 1 ? 1 : 0].row_base : INT64_MAX;
    return w;
}

// ------------------------------------------------------------------------
// Producer: the last warp. Lane 0 waits for free slots and streams the
// stages. Besides that the warp finishes rows split across consumer warps
// (split > 1): once a stage is consumed its lanes add the warps' partial sums
// of each row in a fixed order and write y, so the consumer warps of a row
// never wait for one another. The partial sums are double-buffered (buffer
// k mod 2S for stage k), so the warp adds them up after issuing the copy
// that refills the slot: the refill does not wait for the additions. With
// no split rows to finish, lane 0 runs alone.
// ------------------------------------------------------------------------
struct StageInfo {
    float *y;
    int n_out, r, rows;
};

template <int NV>
__device__ __forceinline__ void finish_split_rows(const GemvParams &p, const float *red, int ri, const StageInfo &st,
                                                  int lane) {
    const int split = p.split;
    const int gshift = 3 - p.split_log2;  // log2(kConsumerWarps / split)
    for (int o = lane; o < st.rows * NV; o += 32) {
        const int ris = o / NV, v = o % NV;
        const int grp = ris & ((1 << gshift) - 1), i = ris >> gshift;
        float sum = 0.0f;
        for (int q = 0; q < split; ++q) sum += red[((ri * kConsumerWarps + grp * split + q) * kRowsPerWarp + i) * NV + v];
        st.y[static_cast<int64_t>(v) * st.n_out + st.r + ris] = sum;
    }
}

template <int MAXB, int NV, bool ISUMS>
__device__ __forceinline__ void gemv_producer(const GemvParams &p, const GemvBatch<MAXB> &b, uint8_t *ring,
                                              const float *red, uint32_t bar_full0, uint32_t bar_empty0,
                                              uint32_t bar_x, int lane) {
    const uint64_t policy = l2_evict_first_policy();
    const int S = p.n_stages;
    const bool reduce = !ISUMS && p.split > 1;
    // without split rows to finish, lane 0 alone runs the loop
    if (!reduce && lane != 0) return;
    const unsigned lanes = reduce ? 0xffffffffu : 1u;
    StageInfo info[kMaxStages];
    StageWalk walk = cta_rows(p, b);
    int mat, r, rows;
    int issued = 0;
    bool ok = true;
    // slot = k mod S, phase = (k / S) & 1 and rprev = (k - S) mod 2S (the partial-sum
    // buffer of the stage the slot held before), kept incrementally
    int slot = 0, rprev = 0;
    uint32_t phase = 0;
    int cur = -1;
    const uint8_t *W = nullptr;
    float *y = nullptr;
    int n_out = 0;
    int64_t lim = 0;
    for (int k = 0; walk.next(b, p.n_mats, p.rows_per_stage, mat, r, rows); ++k) {
        if (k == p.pre_x) {  // the rest after the consumers' first activation loads
            bool got = true;
            if (lane == 0) got = mbar_wait_bounded(bar_x, 0);
            got = __shfl_sync(lanes, got, 0);
            if (!got) {
                if (lane == 0) record_error(p.err, kErrProducerWait);
                ok = false;
                break;
            }
        }
        if (k >= S) {
            const uint32_t parity = phase ^ 1u;
            bool got = true;
            if (lane == 0) got = mbar_wait_bounded(bar_empty0 + 8 * slot, parity);
            got = __shfl_sync(lanes, got, 0);
            __syncwarp(lanes);
            if (!got) {
                if (lane == 0) record_error(p.err, kErrProducerWait);
                ok = false;
                break;
            }
        }
        if (mat != cur) {  // the matrix's fields, read from the parameter table once
            cur = mat;
            const GemvMat &mt = b.m[MAXB == 1 ? 0 : mat];
            W = mt.W;
            y = mt.y;
            n_out = mt.n_out;
            lim = (static_cast<int64_t>(n_out) * p.row_bytes) & ~int64_t(15);
        }
        // the stage info is kept (in local memory) only when split rows need it
        StageInfo prev = {};
        if (reduce) {
            prev = info[slot];
            info[slot] = StageInfo{y, n_out, r, rows};
        }
        if (lane == 0) {
            const int64_t start = static_cast<int64_t>(r) * p.row_bytes;
            const int64_t end = start + static_cast<int64_t>(rows) * p.row_bytes;
            const int64_t a0 = start & ~int64_t(15);
            int64_t a1 = (end + 15) & ~int64_t(15);
            if (a1 > lim) a1 = lim;
            const uint32_t bulk = a1 > a0 ? static_cast<uint32_t>(a1 - a0) : 0u;
            uint8_t *buf = ring + static_cast<size_t>(slot) * p.stage_bytes;
            // bytes past the last 16-byte boundary of W: plain loads
            for (int64_t i = a0 + bulk; i < end; ++i) buf[i - a0] = __ldg(W + i);
            mbar_arrive_expect_tx(bar_full0 + 8 * slot, bulk);
            if (bulk) bulk_copy_g2s(smem_addr(buf), W + a0, bulk, bar_full0 + 8 * slot, policy);
        }
        // the partial sums of stage k - S (buffer (k - S) mod 2S; stage k uses k mod 2S)
        if (reduce && k >= S) {
            finish_split_rows<NV>(p, red, rprev, prev, lane);
            if (++rprev == 2 * S) rprev = 0;
        }
        ++issued;
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
    }
    // Do not leave while copies into this CTA's shared memory are in flight,
    // then finish the last stages' split rows once they are consumed.
    for (int k = max(0, issued - S); k < issued; ++k) {
        const int slot = k % S;
        bool got = true;
        if (lane == 0) got = mbar_wait_bounded(bar_full0 + 8 * slot, static_cast<uint32_t>((k / S) & 1));
        got = __shfl_sync(lanes, got, 0);
        if (!got) {
            if (lane == 0) record_error(p.err, kErrDrainWait);
            return;
        }
    }
    if (!reduce || !ok) return;
    for (int k = max(0, issued - S); k < issued; ++k) {
        const int slot = k % S;
        bool got = true;
        if (lane == 0) got = mbar_wait_bounded(bar_empty0 + 8 * slot, static_cast<uint32_t>((k / S) & 1));
        got = __shfl_sync(lanes, got, 0);
        __syncwarp(lanes);
        if (!got) {
            if (lane == 0) record_error(p.err, kErrDrainWait);
            return;
        }
        finish_split_rows<NV>(p, red, k % (2 * S), info[slot], lane);
    }
}

// Sum over the 32 lanes of a warp (butterfly: every lane gets the total).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// Activations of one matrix into shared memory (all consumer threads): f32
// x quantized straight from global memory (each warp loads the blocks it
// quantizes, two at a time), or records copied from byte-exact blocks.
// With bar_x != 0 each consumer warp arrives on it once its first loads have
// arrived (or at once when it has none), which lets the producer issue its
// further stages.
template <class T, int NV>
__device__ __forceinline__ void stage_activations(const GemvParams &p, const GemvMat &mt, uint8_t *act, int warp,
                                                  int lane, uint32_t bar_x) {
    bool told = bar_x == 0;
    auto loaded = [&]() {
        if (!told && lane == 0) mbar_arrive(bar_x);
        told = true;
    };
    if (mt.x) {
        T::stage_x(mt.x, act, p.nb * NV, warp, kConsumerWarps, lane, loaded);
    } else {
        T::stage_act(mt.xq, act, p.nb, NV, threadIdx.x, kConsumerWarps * 32);
    }
    loaded();
    named_barrier(1, kConsumerWarps * 32);
}

// ------------------------------------------------------------------------
// The kernel. T is the per-type policy (gemv_types.cuh), NV the number of
// vectors, ISUMS selects the diagnostic output of the exact block sums,
// MAXB the capacity of the matrix table.
// ------------------------------------------------------------------------
template <class T, int NV, bool ISUMS, int MAXB>
__global__ void __launch_bounds__(kGemvThreads, NV <= 2 ? 2 : 1)
    gemv_kernel(const GemvParams p, const GemvBatch<MAXB> b) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t bar_full0 = smem_addr(smem);
    const uint32_t bar_empty0 = bar_full0 + 8 * kMaxStages;
    const uint32_t bar_x = bar_full0 + 16 * kMaxStages;
    uint8_t *act = smem + kHeaderBytes;
    float *red = reinterpret_cast<float *>(act + p.act_bytes);
    uint8_t *ring = act + p.act_bytes + p.red_bytes;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int R = p.rows_per_stage;
    const int S = p.n_stages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full0 + 8 * s, 1);
            mbar_init(bar_empty0 + 8 * s, kConsumerWarps);
        }
        mbar_init(bar_x, kConsumerWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Let the next kernel on the stream start its own prologue early.
    pdl_allow_dependents();

    if (warp == kConsumerWarps) {
        gemv_producer<MAXB, NV, ISUMS>(p, b, ring, red, bar_full0, bar_empty0, bar_x, lane);
        return;
    }

    // ---- consumers ----
    // Everything up to the first activation read is independent of the
    // previous kernel and runs before waiting for it.
    bool failed = false;

    const int split = p.split;
    const int groups = kConsumerWarps >> p.split_log2;
    const int grp = warp >> p.split_log2;
    const int part = warp & (split - 1);
    const int b0 = (part * p.nb) >> p.split_log2;
    const int b1 = ((part + 1) * p.nb) >> p.split_log2;
    const int nbw = b1 - b0;  // blocks of each of this warp's rows
    constexpr int kBlocksPerIter = 32 / T::kLanesPerBlock;
    const int sub = lane % T::kLanesPerBlock;  // the lane's part of a block
    const int lane_blk = lane / T::kLanesPerBlock;
    const uint32_t acta = smem_addr(act);

    StageWalk walk = cta_rows(p, b);
    int cur = -1;
    int mat, r, rows;
    float *y = nullptr;          // the current matrix's fields, read from the parameter table once
    int32_t *isums = nullptr;
    int n_out = 0;
    // slot = k mod S, its phase (k / S) & 1 and the partial-sum buffer k mod 2S, kept incrementally
    int slot = 0, ri = 0;
    uint32_t phase = 0;
    for (int k = 0; walk.next(b, p.n_mats, R, mat, r, rows); ++k) {
        if (mat != cur) {  // this CTA reaches a new matrix: stage its activations
            if (cur >= 0) named_barrier(1, kConsumerWarps * 32);
            else pdl_wait_prior_grids();  // activations may come from the previous kernel
            stage_activations<T, NV>(p, b.m[MAXB == 1 ? 0 : mat], act, warp, lane, cur < 0 ? bar_x : 0u);
            cur = mat;
            const GemvMat &mt = b.m[MAXB == 1 ? 0 : mat];  // constant index: no local copy of the table
            y = mt.y;
            isums = mt.isums;
            n_out = mt.n_out;
        }
        if (!failed && !mbar_wait_bounded(bar_full0 + 8 * slot, phase)) {
            record_error(p.err, kErrConsumerWait);
            failed = true;
        }
        const int64_t start = static_cast<int64_t>(r) * p.row_bytes;
        const uint8_t *stage = ring + static_cast<size_t>(slot) * p.stage_bytes + (start & 15);
        const int64_t isum_vstride = static_cast<int64_t>(n_out) * p.nb * T::kSums;
        // this warp group's rows in the stage: grp + groups * i
        const uint8_t *rowp[kRowsPerWarp];
        bool has[kRowsPerWarp];
        int32_t *isum_row[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
            const int ris = grp + groups * i;
            has[i] = ris < rows;
            rowp[i] = stage + static_cast<int64_t>(has[i] ? ris : 0) * p.row_bytes;
            isum_row[i] = ISUMS ? isums + static_cast<int64_t>(r + (has[i] ? ris : 0)) * p.nb * T::kSums
                                : nullptr;
        }
        float acc[kRowsPerWarp][NV];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
            for (int v = 0; v < NV; ++v) acc[i][v] = 0.0f;
        if (NV <= kStraightNv && !failed && has[0] && nbw == kBlocksPerIter) {
            // One iteration per row (K-quant rows of 4096 elements): the
            // warp's two rows as one straight-line sequence, so the scheduler
            // can interleave their loads and dependency chains. Each row's
            // block sum is formed from zero and then added, as in the loop at
            // the end, so the result does not depend on which form ran.
            const int blk = b0 + lane_blk;
            float part0[NV], part1[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v) part0[v] = part1[v] = 0.0f;
            T::template item<NV, ISUMS>(smem_addr(rowp[0]), blk, sub, true, acta, p.nb, part0, isum_row[0],
                                        isum_vstride);
            if (has[1])
                T::template item<NV, ISUMS>(smem_addr(rowp[1]), blk, sub, true, acta, p.nb, part1, isum_row[1],
                                            isum_vstride);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                acc[0][v] += part0[v];
                acc[1][v] += part1[v];
            }
        } else if (NV <= kStraightNv && !failed && has[0] && nbw % kBlocksPerIter == 0) {
            // Several whole iterations per row (32-element rows of 4096
            // elements): the same pairing of the two rows per iteration, each
            // iteration's sum added to its row in the loop's order.
            const uint32_t ra0 = smem_addr(rowp[0]), ra1 = smem_addr(rowp[1]);
            for (int vb = lane_blk; vb < nbw; vb += kBlocksPerIter) {
                const int blk = b0 + vb;
                float part0[NV], part1[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v) part0[v] = part1[v] = 0.0f;
                T::template item<NV, ISUMS>(ra0, blk, sub, true, acta, p.nb, part0, isum_row[0], isum_vstride);
                if (has[1])
                    T::template item<NV, ISUMS>(ra1, blk, sub, true, acta, p.nb, part1, isum_row[1], isum_vstride);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    acc[0][v] += part0[v];
                    acc[1][v] += part1[v];
                }
            }
        } else if (!failed && has[0] && !has[1]) {
            // One row for this warp in the stage (rows split over warps, or
            // the stage's last rows): its blocks in 32 / lanes-per-block
            // steps, lanes past the row's end inactive.
            const uint32_t rowa0 = smem_addr(rowp[0]);
            const int lim = (nbw + kBlocksPerIter - 1) / kBlocksPerIter * kBlocksPerIter;
            for (int vb = lane_blk; vb < lim; vb += kBlocksPerIter) {
                const bool active = vb < nbw;
                float part[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v) part[v] = 0.0f;
                T::template item<NV, ISUMS>(rowa0, b0 + (active ? vb : 0), sub, active, acta, p.nb, part, isum_row[0],
                                            isum_vstride);
#pragma unroll
                for (int v = 0; v < NV; ++v) acc[0][v] += part[v];
            }
        } else if (!failed && has[0]) {
            // The warp's blocks over its rows, flattened (virtual block vb:
            // row vb / nbw, block vb % nbw), so the lanes stay busy whatever
            // the row length. A lane always takes the same part `sub` of its
            // blocks (32 is a multiple of the lanes per block).
            const int tot = nbw * (has[1] ? 2 : 1);
            const int lim = (tot + kBlocksPerIter - 1) / kBlocksPerIter * kBlocksPerIter;
            const uint32_t rowa0 = smem_addr(rowp[0]), rowa1 = smem_addr(rowp[1]);
            for (int vb = lane_blk; vb < lim; vb += kBlocksPerIter) {
                const bool active = vb < tot;
                const bool second = active && vb >= nbw;
                const int blk = b0 + (active ? (second ? vb - nbw : vb) : 0);
                float part[NV];
#pragma unroll
                for (int v = 0; v < NV; ++v) part[v] = 0.0f;
                T::template item<NV, ISUMS>(second ? rowa1 : rowa0, blk, sub, active, acta, p.nb, part,
                                            second ? isum_row[1] : isum_row[0], isum_vstride);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    acc[0][v] += second ? 0.0f : part[v];
                    acc[1][v] += second ? part[v] : 0.0f;
                }
            }
        }
        if (!ISUMS && has[0]) {
#pragma unroll
            for (int i = 0; i < kRowsPerWarp; ++i)
                if (i == 0 || has[i]) {  // warp-uniform: stages of one row per warp group leave row 1 empty
#pragma unroll
                    for (int v = 0; v < NV; ++v) acc[i][v] = warp_sum(acc[i][v]);
                }
            if (split == 1) {
                if (lane == 0 && !failed) {
#pragma unroll
                    for (int i = 0; i < kRowsPerWarp; ++i) {
                        if (!has[i]) continue;
                        const int row = r + grp + groups * i;
#pragma unroll
                        for (int v = 0; v < NV; ++v) y[static_cast<int64_t>(v) * n_out + row] = acc[i][v];
                    }
                }
            } else if (lane == 0) {
                // partial sums of this warp's part of its rows; the producer adds them up
                float *rp = red + ((ri * kConsumerWarps + warp) * kRowsPerWarp) * NV;
#pragma unroll
                for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
                    for (int v = 0; v < NV; ++v) rp[i * NV + v] = acc[i][v];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty0 + 8 * slot);
        if (++ri == 2 * S) ri = 0;
        if (++slot == S) {
            slot = 0;
            phase ^= 1u;
        }
    }
}

}  // namespace qg
