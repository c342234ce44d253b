// gemv_pipeline.cuh - the streaming block-quantized GEMV kernel.
//
// y[v][o] = sum over the blocks b of row o of (exact int32 block sum) x
// (block scales), for W in GGUF blocks and activations in the paired Q8_0 /
// Q8_K blocks ("Quantization" (rml), Quantized dot products; "Building Q8_0
// and Q4_0 Like ggml", Examples 10-11).
//
// Design (one CTA = 1 producer warp + 8 consumer warps):
//  * Each CTA owns a contiguous range of rows, i.e. one contiguous byte range
//    of W. The producer's lane 0 streams it into a ring of shared-memory
//    stages with 1-D bulk async copies (the TMA engine's non-tensor form),
//    each stage a whole number of rows. A stage copies the 16-byte aligned
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
//    stage take one row per `split` warps. Lanes are grouped per block
//    (kLanesPerBlock lanes share one block); each group forms the block's
//    exact int32 sums with __dp4a, combines them with warp shuffles, and the
//    group leader applies the block's float scales.
#pragma once

#include "qg_common.cuh"

namespace qg {

constexpr int kConsumerWarps = 8;
constexpr int kGemvThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxStages = 16;
// Shared-memory header: 2 x kMaxStages mbarriers (256 B), then the
// cross-warp partial sums [2][kConsumerWarps][kMaxNvec] floats (512 B).
constexpr int kRedOffset = 2 * 8 * kMaxStages;
constexpr int kHeaderBytes = kRedOffset + 2 * kConsumerWarps * kMaxNvec * 4;

struct GemvParams {
    const uint8_t *W;    // [n_out][row_bytes], 16-byte aligned
    const uint8_t *xq;   // [n_vec][nb] activation blocks (byte-exact GGUF), or
    const float *x;      // f32 activations [n_vec][n_in], quantized in the prologue when non-null
    float *y;            // [n_vec][n_out]
    int32_t *isums;      // [n_vec][n_out][nb][kSums] (diagnostic mode only)
    int32_t *err;        // device error word
    int64_t row_bytes;
    int64_t w_total;     // n_out * row_bytes
    int n_out;
    int nb;              // blocks per row
    int rows_per_stage;  // kConsumerWarps / split
    int split;           // consumer warps per row: 1, 2, 4 or 8
    int n_stages;        // ring depth (2..kMaxStages)
    int stage_bytes;     // bytes per ring slot, multiple of 16
    int act_bytes;       // bytes of staged activations, multiple of 16
};

// ------------------------------------------------------------------------
// Producer: lane 0 of the last warp.
// ------------------------------------------------------------------------
__device__ __forceinline__ void gemv_producer(const GemvParams &p, uint8_t *ring, uint32_t bar_full0,
                                              uint32_t bar_empty0, int r0, int r1, int n_iter) {
    const uint64_t policy = l2_evict_first_policy();
    const int R = p.rows_per_stage;
    const int S = p.n_stages;
    const int64_t lim = p.w_total & ~int64_t(15);
    int issued = 0;
    for (int k = 0; k < n_iter; ++k) {
        const int slot = k % S;
        if (k >= S) {
            const uint32_t parity = static_cast<uint32_t>((k / S) & 1) ^ 1u;
            if (!mbar_wait_bounded(bar_empty0 + 8 * slot, parity)) {
                record_error(p.err, kErrProducerWait);
                break;
            }
        }
        const int row = r0 + k * R;
        const int rows = min(R, r1 - row);
        const int64_t start = static_cast<int64_t>(row) * p.row_bytes;
        const int64_t end = start + static_cast<int64_t>(rows) * p.row_bytes;
        const int64_t a0 = start & ~int64_t(15);
        int64_t a1 = (end + 15) & ~int64_t(15);
        if (a1 > lim) a1 = lim;
        const uint32_t bulk = a1 > a0 ? static_cast<uint32_t>(a1 - a0) : 0u;
        uint8_t *buf = ring + static_cast<size_t>(slot) * p.stage_bytes;
        // bytes past the last 16-byte boundary of W: plain loads
        for (int64_t i = a0 + bulk; i < end; ++i) buf[i - a0] = __ldg(p.W + i);
        mbar_arrive_expect_tx(bar_full0 + 8 * slot, bulk);
        if (bulk) bulk_copy_g2s(smem_addr(buf), p.W + a0, bulk, bar_full0 + 8 * slot, policy);
        ++issued;
    }
    // Do not leave while copies into this CTA's shared memory are in flight.
    for (int k = max(0, issued - S); k < issued; ++k) {
        const int slot = k % S;
        if (!mbar_wait_bounded(bar_full0 + 8 * slot, static_cast<uint32_t>((k / S) & 1))) {
            record_error(p.err, kErrDrainWait);
            break;
        }
    }
}

// Sum over the 32 lanes of a warp (butterfly: every lane gets the total).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

// ------------------------------------------------------------------------
// The kernel. T is the per-type policy (gemv_types.cuh), NV the number of
// vectors, ISUMS selects the diagnostic output of the exact block sums.
// ------------------------------------------------------------------------
template <class T, int NV, bool ISUMS>
__global__ void __launch_bounds__(kGemvThreads, 1) gemv_kernel(const GemvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t bar_full0 = smem_addr(smem);
    const uint32_t bar_empty0 = bar_full0 + 8 * kMaxStages;
    uint8_t *act = smem + kHeaderBytes;
    uint8_t *ring = act + p.act_bytes;
    float *red = reinterpret_cast<float *>(smem + kRedOffset);  // [2][8][NV] partials (split > 1)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int r0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.n_out / gridDim.x);
    const int r1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.n_out / gridDim.x);
    const int R = p.rows_per_stage;
    const int S = p.n_stages;
    const int n_iter = (r1 - r0 + R - 1) / R;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_full0 + 8 * s, 1);
            mbar_init(bar_empty0 + 8 * s, kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Let the next kernel on the stream start its own prologue early.
    pdl_allow_dependents();

    if (warp == kConsumerWarps) {
        if (lane == 0) gemv_producer(p, ring, bar_full0, bar_empty0, r0, r1, n_iter);
        return;
    }

    // ---- consumers ----
    pdl_wait_prior_grids();  // activations may come from the previous kernel
    if (p.x)
        T::stage_x(p.x, act, p.nb, NV, warp, kConsumerWarps, lane);
    else
        T::stage_act(p.xq, act, p.nb, NV, threadIdx.x, kConsumerWarps * 32);
    named_barrier(1, kConsumerWarps * 32);

    const int split = p.split;
    const int row_in_stage = warp / split;
    const int part = warp % split;
    const int b0 = part * p.nb / split;
    const int b1 = (part + 1) * p.nb / split;
    const int items = (b1 - b0) * T::kLanesPerBlock;
    const int64_t isum_vstride = static_cast<int64_t>(p.n_out) * p.nb * T::kSums;
    bool failed = false;

    for (int k = 0; k < n_iter; ++k) {
        const int slot = k % S;
        if (!failed && !mbar_wait_bounded(bar_full0 + 8 * slot, static_cast<uint32_t>((k / S) & 1))) {
            record_error(p.err, kErrConsumerWait);
            failed = true;
        }
        const int row_first = r0 + k * R;
        const int rows = min(R, r1 - row_first);
        if (row_in_stage < rows) {
            const int row = row_first + row_in_stage;
            const int64_t start = static_cast<int64_t>(row_first) * p.row_bytes;
            const uint8_t *rowp = ring + static_cast<size_t>(slot) * p.stage_bytes + (start & 15) +
                                  static_cast<int64_t>(row_in_stage) * p.row_bytes;
            float acc[NV];
#pragma unroll
            for (int v = 0; v < NV; ++v) acc[v] = 0.0f;
            int32_t *isum_row = ISUMS ? p.isums + static_cast<int64_t>(row) * p.nb * T::kSums : nullptr;
            if (!failed) {
                for (int it = lane; it < ((items + 31) & ~31); it += 32) {
                    const bool active = it < items;
                    const int b = active ? b0 + it / T::kLanesPerBlock : b1 - 1;
                    const int sub = it % T::kLanesPerBlock;
                    T::template item<NV, ISUMS>(rowp, b, sub, active, act, p.nb, acc, isum_row,
                                                isum_vstride);
                }
            }
            if (!ISUMS) {
#pragma unroll
                for (int v = 0; v < NV; ++v) acc[v] = warp_sum(acc[v]);
                if (split == 1) {
                    if (lane == 0 && !failed) {
#pragma unroll
                        for (int v = 0; v < NV; ++v) p.y[static_cast<int64_t>(v) * p.n_out + row] = acc[v];
                    }
                } else {
                    float *r = red + ((k & 1) * kConsumerWarps + warp) * NV;
                    if (lane == 0) {
#pragma unroll
                        for (int v = 0; v < NV; ++v) r[v] = acc[v];
                    }
                    named_barrier(2 + row_in_stage, split * 32);
                    if (part == 0 && lane == 0 && !failed) {
                        const float *g = red + ((k & 1) * kConsumerWarps + warp) * NV;
#pragma unroll
                        for (int v = 0; v < NV; ++v) {
                            float s = 0.0f;
                            for (int q = 0; q < split; ++q) s += g[q * NV + v];
                            p.y[static_cast<int64_t>(v) * p.n_out + row] = s;
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty0 + 8 * slot);
    }
}

}  // namespace qg
