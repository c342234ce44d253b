// gemm_tc.cu - the prefill product for many tokens: Y[t][o] = sum_i W[o][i]
// X[t][i] with W dequantized to f16 and X rounded to f16 ("Quantization"
// (sipllm), The fused matmul: dequantize a row, then a float dot product;
// here a whole dense GEMM on the 5th-generation tensor cores, f32
// accumulation).
//
// One persistent CTA per SM walks 128 x BN output tiles (rows of W x
// tokens; BN = 128 or 256), M fastest so that consecutive CTAs share a token
// tile.
//  * warp 0, lane 0: TMA producer. Per 64-element k-block it loads the A tile
//    (128 rows of W, 128 bytes each) and the B tile (128 tokens) with 2-D
//    tensor maps and 128-byte swizzle into a ring of stages, completion on an
//    mbarrier; rows and k past the matrix read as zeros.
//  * warp 1: allocates 2 BN tensor-memory columns (two 128 x BN f32
//    accumulators); lane 0 issues tcgen05.mma (M = 128, N = BN, K = 16, A
//    and B from shared memory), four per k-block, commits each k-block to
//    the stage's empty barrier and each tile to its accumulator's barrier.
//  * warps 2..5: epilogue. Each reads its 32 tensor-memory lanes (rows) of
//    the finished accumulator, 32 columns (tokens) at a time, writes them to
//    a 4 KB shared-memory buffer as [token][row] and sends the buffer to Y
//    with one TMA tensor store (two buffers per warp, so the next chunk is
//    written while the store reads the last). Plain stores replace them when
//    Y is not 16-byte aligned or n_out is not a multiple of 4: measured, the
//    32 scalar stores of a chunk took about 0.65 us, a 128 x 128 tile about
//    3 us, at the end of every CTA's last tile.
// All waits are bounded and give up when another thread has recorded an
// error; tensor memory is freed on every path.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "gemm_tc.cuh"
#include "tc_common.cuh"

namespace qg {

constexpr int kGemmBM = 128, kGemmBK = 64;
constexpr int kGemmThreads = 6 * 32;
constexpr int kGemmTileBytes = kGemmBM * kGemmBK * 2;  // the A tile, f16
constexpr int kGemmHdrBytes = 1024;
// Epilogue staging: two 4 KB buffers (32 tokens x 32 rows of f32) for each of
// the four epilogue warps, after the ring.
constexpr int kEpiBytes = 4 * 2 * 4096;
// Per token-tile width BN (128 or 256): B tile bytes, stage bytes, ring
// depth (what fits next to the header), shared memory, tensor-memory columns
// (two accumulators).
template <int BN> struct GemmShape {
    static constexpr int kBTile = BN * kGemmBK * 2;
    static constexpr int kStage = kGemmTileBytes + kBTile;
    static constexpr int kStages = BN == 128 ? 6 : 4;
    static constexpr int kSmem = 1024 /* base alignment */ + kGemmHdrBytes + kStages * kStage + kEpiBytes;
    static constexpr int kTmemCols = 2 * BN;
    static_assert(kSmem <= 232448, "shared memory");
};

struct GemmParams {
    float *y;  // [n_tok][n_out]
    int32_t *err;
    int n_out, n_tok, K;
    int tiles_m, tiles_n;
    // k split (tensor-memory prefill kernel): each tile's k-blocks in ksplit
    // parts, run as separate work items; part 0 writes y, part k > 0 writes the
    // same layout at part + (k - 1) n_tok n_out, and gemm_ksum adds them after
    int ksplit;
    float *part;
    // 1: tiles leave through shared memory and TMA tensor stores (the output
    // maps); 0: plain stores (y not 16-byte aligned or n_out not a multiple of 4)
    int tma_out;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *tm, int c0, int c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// D (tensor memory) = A (shared memory) x B (shared memory) (+ D).
__device__ __forceinline__ void tc_mma_ss(uint32_t d_t, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_t),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void tc_ld32_wait(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
        "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

// TMA tensor store of a shared-memory box into a 3-D f32 tensor, in the
// issuing thread's bulk group; the parts of the box past the tensor's extent
// are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *tm, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most one of this thread's bulk groups still reads shared memory.
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Wait until this thread's bulk groups are complete (their writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_b32(uint32_t a, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}

// Epilogue of one warp's 32 rows of an accumulator tile: tensor-memory
// columns tcol .. tcol + BN (this warp's lanes) to out[z][tok0 + c][row0 + r].
// Each 32-column chunk goes from registers into one of the warp's two 4 KB
// buffers as [token][row] (for one token the 32 lanes write 128 consecutive
// bytes, no bank conflict) and leaves with one TMA tensor store, which clips
// rows and tokens past the tensor. Lane 0 issues the stores; a buffer is
// rewritten only after the store from it two chunks earlier has read it.
template <int BN>
__device__ __forceinline__ void epilogue_tma(uint32_t tcol, const CUtensorMap *out, int row0, int tok0, int z,
                                             uint32_t buf, int lane) {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tc_ld32_wait(tcol + static_cast<uint32_t>(c0), v);
        const uint32_t b = buf + static_cast<uint32_t>((c0 >> 5) & 1) * 4096u;
        if (lane == 0) bulk_wait_read1();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 32; ++j) st_shared_b32(b + 128u * j + 4u * lane, v[j]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(out, b, row0, tok0 + c0, z);
            bulk_commit();
        }
    }
}

// The same with plain stores to out[tok][n_out] (row = this lane's row).
template <int BN>
__device__ __forceinline__ void epilogue_plain(uint32_t tcol, float *out, int n_out, int n_tok, int row, int tok0) {
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tc_ld32_wait(tcol + static_cast<uint32_t>(c0), v);
        if (row < n_out) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (tok0 + c0 + j < n_tok) out[static_cast<int64_t>(tok0 + c0 + j) * n_out + row] = __uint_as_float(v[j]);
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_f16_tc_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                       const __grid_constant__ CUtensorMap tma_y, const GemmParams p) {
    using Sh = GemmShape<BN>;
    constexpr int kGemmStages = Sh::kStages, kGemmStageBytes = Sh::kStage, kGemmTmemCols = Sh::kTmemCols;
    constexpr int kGemmBN = BN;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_a = smem_addr(smem_raw);
    const uint32_t base_a = (raw_a + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_a - raw_a);
    // header: full[stages] | empty[stages] | tfull[2] | tempty[2] | mfinal | tmem address | abort flag
    const uint32_t full0 = base_a, empty0 = base_a + 64, tfull0 = base_a + 128, tempty0 = base_a + 144;
    const uint32_t mfinal = base_a + 160;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + 168);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + 172);
    const uint32_t stages_a = base_a + kGemmHdrBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total = p.tiles_m * p.tiles_n;
    const int nk = (p.K + kGemmBK - 1) / kGemmBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(tfull0 + 8 * d, 1);
            mbar_init(tempty0 + 8 * d, 4);
        }
        mbar_init(mfinal, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tc_alloc(smem_addr(tmem_slot), kGemmTmemCols);
        tc_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_allow_dependents();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            pdl_wait_prior_grids();  // A and B are written by the kernels before this one
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            for (int t = blockIdx.x; t < total; t += gridDim.x) {
                const int tm = t % p.tiles_m, tn = t / p.tiles_m;
                bool ok = true;
                for (int kb = 0; kb < nk; ++kb) {
                    if (issued >= kGemmStages && !tc_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) {
                        record_error(p.err, kErrProducerWait);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    const uint32_t sa = stages_a + static_cast<uint32_t>(s * kGemmStageBytes);
                    mbar_arrive_expect_tx(full0 + 8 * s, static_cast<uint32_t>(kGemmStageBytes));
                    tma_load_2d(sa, &tma_a, kb * kGemmBK, tm * kGemmBM, full0 + 8 * s);
                    tma_load_2d(sa + kGemmTileBytes, &tma_b, kb * kGemmBK, tn * kGemmBN, full0 + 8 * s);
                    ++issued;
                    if (++s == kGemmStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
            }
            // leave no copy in flight into this CTA's shared memory
            for (int64_t k = issued > kGemmStages ? issued - kGemmStages : 0; k < issued; ++k) {
                if (!mbar_wait_bounded(full0 + 8 * static_cast<int>(k % kGemmStages),
                                       static_cast<uint32_t>((k / kGemmStages) & 1))) {
                    record_error(p.err, kErrDrainWait);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- mma issuer
        if (lane == 0) {
            const uint32_t idesc = tc_idesc_f16(kGemmBM, kGemmBN);
            int s = 0, it = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++it) {
                const int d = it & 1;
                if (it >= 2 && !tc_wait(tempty0 + 8 * d, static_cast<uint32_t>(((it - 2) >> 1) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem + static_cast<uint32_t>(d * kGemmBN);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!tc_wait(full0 + 8 * s, ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = stages_a + static_cast<uint32_t>(s * kGemmStageBytes);
                    const uint64_t da = tc_smem_desc(sa, 1024), db = tc_smem_desc(sa + kGemmTileBytes, 1024);
#pragma unroll
                    for (int k = 0; k < kGemmBK / 16; ++k)
                        tc_mma_ss(dt, da + static_cast<uint64_t>(2 * k), db + static_cast<uint64_t>(2 * k), idesc,
                                  (kb | k) != 0 ? 1u : 0u);
                    tc_commit(empty0 + 8 * s);  // the stage is free once these mmas are done
                    if (++s == kGemmStages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) tc_commit(tfull0 + 8 * d);
            }
            if (!ok) {
                record_error(p.err, kErrConsumerWait);
                *abort_flag = 1;
            }
            // every mma complete before tensor memory is freed
            tc_commit(mfinal);
            if (!mbar_wait_bounded(mfinal, 0u)) record_error(p.err, kErrDrainWait);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: warp w reads tensor-memory lanes 32 (w % 4) ..
        const int q = warp & 3;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
        const uint32_t epi_buf = stages_a + static_cast<uint32_t>(kGemmStages * kGemmStageBytes + q * 8192);
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const int tm = t % p.tiles_m, tn = t / p.tiles_m, d = it & 1;
            if (ok && !tc_wait(tfull0 + 8 * d, static_cast<uint32_t>((it >> 1) & 1), abort_flag)) {
                if (lane == 0) {
                    record_error(p.err, kErrConsumerWait);
                    *abort_flag = 1;
                }
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tcol = tl + static_cast<uint32_t>(d * kGemmBN);
            if (p.tma_out)
                epilogue_tma<kGemmBN>(tcol, &tma_y, tm * kGemmBM + 32 * q, tn * kGemmBN, 0, epi_buf, lane);
            else
                epilogue_plain<kGemmBN>(tcol, p.y, p.n_out, p.n_tok, tm * kGemmBM + 32 * q + lane, tn * kGemmBN);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * d);
        }
        if (lane == 0) bulk_wait_all();  // the stores have read shared memory and written y
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tc_dealloc(tmem, kGemmTmemCols);
}

constexpr int kQ4kBlockBytes = 144;
constexpr int kRawHdr = kGemmBM * 16, kRawCodes = kGemmBM * 32;  // raw bytes of one k-block

// 6-bit scale and min of Q4_K sub-block j from the 12 scale bytes (words
// s0 = bytes 0..3, s1 = 4..7, s2 = 8..11) ("Quantization" (rml), Unpacking
// the packed fields; "量化格式" (candle), block structure table).
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j, int &sc, int &m) {
    auto byte = [&](int k) {
        const uint32_t w = k < 4 ? s0 : (k < 8 ? s1 : s2);
        return static_cast<int>((w >> (8 * (k & 3))) & 0xFFu);
    };
    if (j < 4) {
        sc = byte(j) & 63;
        m = byte(j + 4) & 63;
    } else {
        sc = (byte(j + 4) & 0xF) | ((byte(j - 4) >> 6) << 4);
        m = (byte(j + 4) >> 4) | ((byte(j) >> 6) << 4);
    }
}

// Two f32 values to one f16x2 word (round to nearest even), lo first.
__device__ __forceinline__ uint32_t pack_f16x2(float2 v) {
    const __half2 h = __floats2half2_rn(v.x, v.y);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// ---------------------------------------------------------------------------
// The prefill product for Q4_K weights with the dequantization fused into the
// GEMM: no f16 copy of W in memory. Same tiles, mma issue and epilogue as
// gemm_f16_tc_kernel, but tcgen05.mma reads its A operand (the dequantized
// weights) from tensor memory: lane m = row m of the tile, two f16 per
// 32-bit column, the even k in the low half.
//  * warp 0, lane 0: per 64-element k-block three 2-D tensor loads into a
//    ring stage: the B tile as in gemm_f16_tc_kernel, and the raw bytes the
//    k-block needs for each of the tile's 128 rows -- the 16-byte header of
//    its Q4_K block (d, dmin, 12 scale bytes; box 16 bytes x 128 rows) and
//    the 32 bytes of codes (box 32 x 128; k-block q of a block uses
//    qs[32 q .. 32 q + 31], low nibbles for its first 32 elements, high
//    nibbles for the other 32);
//  * tensor memory: kND accumulators of BN columns (one when BN = 256, so
//    the mma waits for the epilogue to drain it before a tile's first mma),
//    then one 32-column A slot per ring stage;
//  * warps 6..13 (converters): warp w serves tensor-memory lanes 32 (w % 4)
//    .. (the only lanes it may access) and half (w - 6) / 4 of each k-block,
//    i.e. thread = (row, one 32-element sub-block j = 2 q + half): value
//    d sc_j q - dmin m_j in f32 (the product d sc_j q is exact; the
//    subtraction rounds once), rounded to f16 -- the values dequantize_rows
//    gives, rounded as the f16-copy path rounds them -- 16 columns with one
//    tcgen05.st; then tcgen05.wait::st and the before-thread-sync fence, and
//    the warp arrives on the stage's A-full barrier; the mma waits for that
//    barrier and the stage's full barrier;
//  * the A slot of stage s is rewritten only after the producer has reused
//    stage s, i.e. after the mmas that read it completed (their commit to the
//    stage's empty barrier).
// Writing A to tensor memory leaves shared memory to the tensor loads and
// the mma's B reads: the ring holds only the B tile and the raw bytes.
// ---------------------------------------------------------------------------
constexpr int kTmemConvWarps = 8;
constexpr int kTmemThreads = (6 + kTmemConvWarps) * 32;

template <int BN> struct TmemFuseShape {
    static constexpr int kBTile = BN * kGemmBK * 2;
    static constexpr int kStage = kBTile + kRawHdr + kRawCodes;  // a multiple of 1024
    static constexpr int kND = BN == 256 ? 1 : 2;                 // accumulators
    static constexpr int kStages = BN == 256 ? 5 : 8;
    static constexpr int kACol0 = kND * BN;                       // first A column
    static constexpr int kSmem = 1024 + kGemmHdrBytes + kStages * kStage + kEpiBytes;
    static constexpr int kTmemCols = 512;
    static_assert(kStage % 1024 == 0, "swizzled B tiles start 1024-byte aligned");
    static_assert(kACol0 + 32 * kStages <= kTmemCols, "tensor-memory columns");
    static_assert(kSmem <= 232448, "shared memory");
};

// D (tensor memory) = A (tensor memory) x B (shared memory) (+ D).
__device__ __forceinline__ void tc_mma_ts(uint32_t d_t, uint32_t a_t, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_t),
        "r"(a_t), "l"(b_desc), "r"(idesc), "r"(acc)
        : "memory");
}

// 32 lanes x 16 columns from this warp's 16 registers each.
__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

template <int BN>
__global__ void __launch_bounds__(kTmemThreads, 1)
    gemm_q4k_tmem_kernel(const __grid_constant__ CUtensorMap tma_hdr, const __grid_constant__ CUtensorMap tma_codes,
                         const __grid_constant__ CUtensorMap tma_b, const __grid_constant__ CUtensorMap tma_y,
                         const __grid_constant__ CUtensorMap tma_part, const GemmParams p) {
    using Sh = TmemFuseShape<BN>;
    constexpr int S = Sh::kStages, ND = Sh::kND;
    constexpr int kOffHdr = Sh::kBTile, kOffCodes = kOffHdr + kRawHdr;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_a = smem_addr(smem_raw);
    const uint32_t base_a = (raw_a + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (base_a - raw_a);
    // header: full[S] | afull[S] | empty[S] | tfull[2] | tempty[2] | mfinal | tmem | abort
    const uint32_t full0 = base_a, afull0 = base_a + 64, empty0 = base_a + 128;
    const uint32_t tfull0 = base_a + 192, tempty0 = base_a + 208, mfinal = base_a + 224;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base + 232);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(base + 236);
    const uint32_t stages_a = base_a + kGemmHdrBytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = p.tiles_m * p.tiles_n;
    const int total = tiles * p.ksplit;  // work items: (tile, k part), the tile fastest
    const int nk = p.K / kGemmBK;
    // item t: tile t % tiles, k-blocks [kb0, kb1) of part t / tiles
    auto kb_range = [&](int t, int &kb0, int &kb1) {
        const int ks = t / tiles;
        kb0 = ks * nk / p.ksplit;
        kb1 = (ks + 1) * nk / p.ksplit;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(afull0 + 8 * s, kTmemConvWarps);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(tfull0 + 8 * d, 1);
            mbar_init(tempty0 + 8 * d, 4);
        }
        mbar_init(mfinal, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tc_alloc(smem_addr(tmem_slot), Sh::kTmemCols);
        tc_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_allow_dependents();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer: per k-block the B tile and the raw bytes
        if (lane == 0) {
            pdl_wait_prior_grids();  // B is written by the kernel before this one
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
                const int tile = t % tiles, tm = tile % p.tiles_m, tn = tile / p.tiles_m;
                int kb0, kb1;
                kb_range(t, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (issued >= S && !tc_wait(empty0 + 8 * s, ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = stages_a + static_cast<uint32_t>(s * Sh::kStage);
                    const int x0 = (kb >> 2) * kQ4kBlockBytes;  // the block column's first byte in a row
                    mbar_arrive_expect_tx(full0 + 8 * s, static_cast<uint32_t>(Sh::kStage));
                    tma_load_2d(st, &tma_b, kb * kGemmBK, tn * BN, full0 + 8 * s);
                    tma_load_2d(st + kOffHdr, &tma_hdr, x0, tm * kGemmBM, full0 + 8 * s);
                    tma_load_2d(st + kOffCodes, &tma_codes, x0 + 16 + 32 * (kb & 3), tm * kGemmBM, full0 + 8 * s);
                    ++issued;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                record_error(p.err, kErrProducerWait);
                *abort_flag = 1;
            }
            // leave no copy in flight into this CTA's shared memory
            for (int64_t k = issued > S ? issued - S : 0; k < issued; ++k) {
                if (!mbar_wait_bounded(full0 + 8 * static_cast<int>(k % S), static_cast<uint32_t>((k / S) & 1))) {
                    record_error(p.err, kErrDrainWait);
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- mma issuer
        if (lane == 0) {
            const uint32_t idesc = tc_idesc_f16(kGemmBM, BN);
            int s = 0, it = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++it) {
                const int d = it % ND;
                if (it >= ND && !tc_wait(tempty0 + 8 * d, static_cast<uint32_t>(((it - ND) / ND) & 1), abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dt = tmem + static_cast<uint32_t>(d * BN);
                int kb0, kb1;
                kb_range(t, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!tc_wait(full0 + 8 * s, ph, abort_flag) || !tc_wait(afull0 + 8 * s, ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = stages_a + static_cast<uint32_t>(s * Sh::kStage);
                    const uint64_t db = tc_smem_desc(st, 1024);
                    const uint32_t at = tmem + static_cast<uint32_t>(Sh::kACol0 + 32 * s);
#pragma unroll
                    for (int k = 0; k < kGemmBK / 16; ++k)
                        tc_mma_ts(dt, at + static_cast<uint32_t>(8 * k), db + static_cast<uint64_t>(2 * k), idesc,
                                  (kb != kb0 || k != 0) ? 1u : 0u);
                    tc_commit(empty0 + 8 * s);  // stage s and its A slot are free once these mmas are done
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) tc_commit(tfull0 + 8 * d);
            }
            if (!ok) {
                record_error(p.err, kErrConsumerWait);
                *abort_flag = 1;
            }
            tc_commit(mfinal);
            if (!mbar_wait_bounded(mfinal, 0u)) record_error(p.err, kErrDrainWait);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ---------------- epilogue: warp w reads tensor-memory lanes 32 (w % 4) ..
        const int q = warp & 3;
        const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
        const uint32_t epi_buf = stages_a + static_cast<uint32_t>(S * Sh::kStage + q * 8192);
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const int tile = t % tiles, tm = tile % p.tiles_m, tn = tile / p.tiles_m, d = it % ND;
            if (ok && !tc_wait(tfull0 + 8 * d, static_cast<uint32_t>((it / ND) & 1), abort_flag)) {
                if (lane == 0) {
                    record_error(p.err, kErrConsumerWait);
                    *abort_flag = 1;
                }
                ok = false;
            }
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            const int ks = t / tiles;
            const uint32_t tcol = tl + static_cast<uint32_t>(d * BN);
            if (p.tma_out) {
                epilogue_tma<BN>(tcol, ks == 0 ? &tma_y : &tma_part, tm * kGemmBM + 32 * q, tn * BN,
                                 ks == 0 ? 0 : ks - 1, epi_buf, lane);
            } else {
                float *out = ks == 0 ? p.y : p.part + static_cast<int64_t>(ks - 1) * p.n_tok * p.n_out;
                epilogue_plain<BN>(tcol, out, p.n_out, p.n_tok, tm * kGemmBM + 32 * q + lane, tn * BN);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * d);
        }
        if (lane == 0) bulk_wait_all();  // the stores have read shared memory and written their tensor
        __syncwarp();
    } else {
        // ---------------- converters: lanes 32 q .. of tensor memory, sub-block `half` of each k-block
        const int q = warp & 3, half = (warp - 6) >> 2;
        const int row = 32 * q + lane;
        const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(Sh::kACol0 + 16 * half);
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
            int kb0, kb1;
            kb_range(t, kb0, kb1);
            for (int kb = kb0; kb < kb1; ++kb) {
                // the tensor-memory store below is warp-collective: the warp goes on or stops as one
                if (!__all_sync(0xffffffffu, tc_wait(full0 + 8 * s, ph, abort_flag))) {
                    ok = false;
                    break;
                }
                const uint32_t st = stages_a + static_cast<uint32_t>(s * Sh::kStage);
                const uint4 hdr = ld_s128(st + kOffHdr + 16u * row);  // d | dmin | scales[0..11]
                const uint4 w0 = ld_s128(st + kOffCodes + 32u * row), w1 = ld_s128(st + kOffCodes + 32u * row + 16u);
                int sc, m;
                q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * (kb & 3) + half, sc, m);
                const float dsc = __fmul_rn(f16_bits_to_f32(hdr.x), static_cast<float>(sc));
                const float off = __fmul_rn(f16_bits_to_f32(hdr.x >> 16), static_cast<float>(m));
                // Code q in the low byte of the float 2^23 (one byte permute
                // after the word's nibbles are masked): the float is 2^23 + q
                // exactly, and fma(d sc, 2^23 + q, -d sc 2^23) = d sc q is exact
                // (d sc has at most 17 significant bits, q 4). The subtraction
                // of dmin m then rounds once, as d sc q - dmin m does in
                // dequantize_rows.
                const float2 s2 = make_float2(dsc, dsc), c2 = make_float2(-dsc * 8388608.0f, -dsc * 8388608.0f);
                const float2 off2 = make_float2(-off, -off);
                const uint32_t qw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                uint32_t o[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t nib = (half ? qw[i] >> 4 : qw[i]) & 0x0F0F0F0Fu;
#pragma unroll
                    for (int b = 0; b < 4; b += 2) {
                        const float2 mg = make_float2(__uint_as_float(__byte_perm(nib, 0x4B000000u, 0x7650u | b)),
                                                      __uint_as_float(__byte_perm(nib, 0x4B000000u, 0x7651u | b)));
                        o[2 * i + (b >> 1)] = pack_f16x2(fadd2(ffma2(s2, mg, c2), off2));
                    }
                }
                tc_st16(ta + static_cast<uint32_t>(32 * s), o);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull0 + 8 * s);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok) {
            if (lane == 0) record_error(p.err, kErrConsumerWait);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tc_dealloc(tmem, Sh::kTmemCols);
}

// f32 -> f16 (round to nearest even), 8 elements per thread.
__global__ void f32_to_f16_kernel(const float *__restrict__ x, __half *__restrict__ out, int64_t groups) {
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups;
         g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(x) + 2 * g);
        const float4 b = __ldg(reinterpret_cast<const float4 *>(x) + 2 * g + 1);
        uint4 o;
        o.x = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(a.x))) | (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(a.y))) << 16);
        o.y = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(a.z))) | (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(a.w))) << 16);
        o.z = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(b.x))) | (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(b.y))) << 16);
        o.w = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(b.z))) | (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(b.w))) << 16);
        reinterpret_cast<uint4 *>(out)[g] = o;
    }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// A row-major f16 matrix [rows][K] as a 2-D tensor, box {64, box_rows},
// 128-byte swizzle (the mma's K-major operand layout); out-of-range rows and
// k read as zeros.
bool encode_f16_map(CUtensorMap *tm, const void *base, int64_t rows, int64_t K, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kGemmBK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The raw Q4_K blocks of W as a 2-D byte tensor [n_out][row_bytes] with a
// box of `box_bytes` x 128 rows; rows past the matrix read as zeros.
bool encode_q4k_map(CUtensorMap *tm, const void *W, int64_t n_out, int64_t row_bytes, int box_bytes) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(n_out)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes), static_cast<cuuint32_t>(kGemmBM)};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An f32 output [depth][n_tok][n_out] as a 3-D tensor with a box of 32 rows x
// 32 tokens x 1 (the epilogue's TMA stores). Needs base 16-byte aligned and
// n_out a multiple of 4 (16-byte row pitch).
bool encode_out_map(CUtensorMap *tm, void *base, int64_t n_out, int64_t n_tok, int64_t depth) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(n_out), static_cast<cuuint64_t>(n_tok),
                                static_cast<cuuint64_t>(depth)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(n_out) * 4, static_cast<cuuint64_t>(n_out * n_tok) * 4};
    const cuuint32_t box[3] = {32u, 32u, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Whether y (and the k-split partials) can leave through TMA stores.
bool out_tma_ok(const float *y, int64_t n_out) {
    return (reinterpret_cast<uintptr_t>(y) & 15u) == 0 && n_out % 4 == 0;
}

}  // namespace

cudaError_t launch_f32_to_f16(const float *x, __half *out, int64_t n, int sms, cudaStream_t s) {
    const int64_t groups = n / 8;
    if (groups == 0) return cudaSuccess;
    int64_t grid = (groups + 255) / 256;
    if (grid > static_cast<int64_t>(sms) * 16) grid = static_cast<int64_t>(sms) * 16;
    f32_to_f16_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(x, out, groups);
    return cudaGetLastError();
}

// y[i] += part[0][i] + ... + part[n_parts - 1][i], added in that order (part k
// at part + k n), after the GEMM that wrote them has finished.
__global__ void gemm_ksum_kernel(float *__restrict__ y, const float *__restrict__ part, int64_t n, int n_parts) {
    pdl_wait_prior_grids();
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float v[7];
#pragma unroll
        for (int k = 0; k < 7; ++k) v[k] = k < n_parts ? __ldcg(part + k * n + i) : 0.0f;
        float acc = y[i];
#pragma unroll
        for (int k = 0; k < 7; ++k)
            if (k < n_parts) acc += v[k];
        y[i] = acc;
    }
}

template <int BN>
cudaError_t launch_gemm_bn(const __half *A, const __half *B, float *y, int64_t n_out, int64_t n_tok, int64_t K,
                           int32_t *err, int sms, int device, cudaStream_t s) {
    CUtensorMap ta, tb, ty;
    const bool tma_out = out_tma_ok(y, n_out);
    if (!encode_f16_map(&ta, A, n_out, K, kGemmBM) || !encode_f16_map(&tb, B, n_tok, K, BN) ||
        (tma_out && !encode_out_map(&ty, y, n_out, n_tok, 1))) {
        g_launch_step = "cuTensorMapEncodeTiled";
        return cudaErrorInvalidValue;
    }
    if (!tma_out) ty = tb;  // unused
    GemmParams p = {};
    p.y = y;
    p.tma_out = tma_out ? 1 : 0;
    p.err = err;
    p.n_out = static_cast<int>(n_out);
    p.n_tok = static_cast<int>(n_tok);
    p.K = static_cast<int>(K);
    p.tiles_m = static_cast<int>((n_out + kGemmBM - 1) / kGemmBM);
    p.tiles_n = static_cast<int>((n_tok + BN - 1) / BN);
    const int64_t total = static_cast<int64_t>(p.tiles_m) * p.tiles_n;
    const int grid = static_cast<int>(total < sms ? total : sms);
    static std::atomic<uint64_t> done{0};
    const uint64_t bit = 1ull << (device & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
        g_launch_step = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)";
        cudaError_t e = cudaFuncSetAttribute(gemm_f16_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             GemmShape<BN>::kSmem);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit, std::memory_order_acq_rel);
    }
    return launch_pdl(gemm_f16_tc_kernel<BN>, grid, kGemmThreads, GemmShape<BN>::kSmem, s, ta, tb, ty, p);
}

template <int BN>
cudaError_t launch_tmem_bn(const uint8_t *W, const __half *B, float *y, int64_t n_out, int64_t n_tok, int64_t K,
                           int ksplit, float *part, int32_t *err, int sms, int device, cudaStream_t s) {
    CUtensorMap th, tc, tb, ty, tp;
    const int64_t row_bytes = K / 256 * kQ4kBlockBytes;
    const bool tma_out = out_tma_ok(y, n_out);
    if (!encode_q4k_map(&th, W, n_out, row_bytes, 16) || !encode_q4k_map(&tc, W, n_out, row_bytes, 32) ||
        !encode_f16_map(&tb, B, n_tok, K, BN) || (tma_out && !encode_out_map(&ty, y, n_out, n_tok, 1)) ||
        (tma_out && ksplit > 1 && !encode_out_map(&tp, part, n_out, n_tok, ksplit - 1))) {
        g_launch_step = "cuTensorMapEncodeTiled";
        return cudaErrorInvalidValue;
    }
    if (!tma_out) ty = tb;  // unused
    if (!tma_out || ksplit == 1) tp = ty;
    GemmParams p = {};
    p.y = y;
    p.tma_out = tma_out ? 1 : 0;
    p.err = err;
    p.n_out = static_cast<int>(n_out);
    p.n_tok = static_cast<int>(n_tok);
    p.K = static_cast<int>(K);
    p.tiles_m = static_cast<int>((n_out + kGemmBM - 1) / kGemmBM);
    p.tiles_n = static_cast<int>((n_tok + BN - 1) / BN);
    p.ksplit = ksplit;
    p.part = part;
    const int64_t total = static_cast<int64_t>(p.tiles_m) * p.tiles_n * ksplit;
    const int grid = static_cast<int>(total < sms ? total : sms);
    static std::atomic<uint64_t> done{0};
    const uint64_t bit = 1ull << (device & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
        g_launch_step = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)";
        cudaError_t e = cudaFuncSetAttribute(gemm_q4k_tmem_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             TmemFuseShape<BN>::kSmem);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit, std::memory_order_acq_rel);
    }
    return launch_pdl(gemm_q4k_tmem_kernel<BN>, grid, kTmemThreads, TmemFuseShape<BN>::kSmem, s, th, tc, tb, ty, tp,
                      p);
}

// Y[n_tok][n_out] = dequant(W)[n_out][K] . B[n_tok][K]^T for Q4_K W (K a
// multiple of 256, rows 16-byte aligned) and f16 B, the dequantization done
// on the way into tensor memory, with the tile width and k split of `plan`
// (gemm_q4k_tmem_plan); a split's partials go to `part`.
cudaError_t launch_gemm_q4k_tmem(const uint8_t *W, const __half *B, float *y, int64_t n_out, int64_t n_tok,
                                 int64_t K, GemmPlan plan, float *part, int32_t *err, int sms, int device,
                                 cudaStream_t s) {
    cudaError_t e = plan.bn == 256 ? launch_tmem_bn<256>(W, B, y, n_out, n_tok, K, plan.ks, part, err, sms, device, s)
                                   : launch_tmem_bn<128>(W, B, y, n_out, n_tok, K, plan.ks, part, err, sms, device, s);
    if (e != cudaSuccess || plan.ks == 1) return e;
    g_launch_step = "k-split sum";
    const int64_t n = n_out * n_tok;
    const int64_t grid = std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(sms) * 8);
    return launch_pdl(gemm_ksum_kernel, static_cast<int>(grid), 256, 0, s, y, static_cast<const float *>(part), n,
                      plan.ks - 1);
}

// Token-tile width and k split for a GEMM of these sizes: the pair that
// minimizes the busiest CTA's time, ceil(tiles ks / sms) ceil(nk / ks)
// k-blocks at 10 units each with 128-token tiles and unit256 with 256-token
// tiles, plus the split's own cost: about 4 k-blocks for the sum launch and one
// per 2^19 partial values it reads. Splits keep at least 4 k-blocks a part, at
// most max_parts (and 8) parts, the parts after the first (f32 [n_tok][n_out]
// each) within scratch_bytes, and with 256-token tiles at most one item per
// CTA. Ties keep the narrower tile and fewer parts.
GemmPlan gemm_plan(int64_t n_out, int64_t n_tok, int64_t K, int sms, int max_parts, size_t scratch_bytes,
                   int unit256) {
    GemmPlan best = {128, 1};
    const int64_t tm = (n_out + kGemmBM - 1) / kGemmBM, nk = (K + kGemmBK - 1) / kGemmBK;
    if (tm == 0 || n_tok == 0 || nk == 0 || sms < 1) return best;
    int64_t best_cost = -1;
    for (int bn : {128, 256}) {
        const int64_t tiles = tm * ((n_tok + bn - 1) / bn), unit = bn == 256 ? unit256 : 10;
        for (int ks = 1; ks <= std::min(max_parts, 8); ++ks) {
            if (ks > 1 && (nk / ks < 4 || static_cast<size_t>(ks - 1) * n_tok * n_out * 4 > scratch_bytes)) break;
            if (bn == 256 && ks > 1 && tiles * ks > sms) break;
            int64_t cost = ((tiles * ks + sms - 1) / sms) * ((nk + ks - 1) / ks) * unit;
            if (ks > 1) cost += 10 * (4 + ((ks - 1) * n_tok * n_out >> 19));
            if (best_cost < 0 || cost < best_cost) {
                best = {bn, ks};
                best_cost = cost;
            }
        }
    }
    return best;
}

// The fused Q4_K GEMM's plan: measured 0.39 us a k-block with 128-token tiles
// and about 0.5 with 256 (five ring stages instead of eight, one accumulator,
// an mma twice as large), so 13 units.
GemmPlan gemm_q4k_tmem_plan(int64_t n_out, int64_t n_tok, int64_t K, int sms, int max_parts, size_t scratch_bytes) {
    return gemm_plan(n_out, n_tok, K, sms, max_parts, scratch_bytes, 13);
}

// The f16 GEMM's plan (no split: qgemm_f16 has no scratch): measured 0.37 us
// a k-block with 128-token tiles and 0.38 with 256, so 11 units.
GemmPlan gemm_f16_plan(int64_t n_out, int64_t n_tok, int64_t K, int sms) {
    return gemm_plan(n_out, n_tok, K, sms, 1, 0, 11);
}

// Y[n_tok][n_out] = A[n_out][K] . B[n_tok][K]^T for f16 A, B (16-byte
// aligned, K a multiple of 8), token tiles as gemm_f16_plan chooses them.
cudaError_t launch_gemm_f16_tc(const __half *A, const __half *B, float *y, int64_t n_out, int64_t n_tok, int64_t K,
                               int32_t *err, int sms, int device, cudaStream_t s) {
    if (gemm_f16_plan(n_out, n_tok, K, sms).bn == 256)
        return launch_gemm_bn<256>(A, B, y, n_out, n_tok, K, err, sms, device, s);
    return launch_gemm_bn<128>(A, B, y, n_out, n_tok, K, err, sms, device, s);
}

}  // namespace qg
