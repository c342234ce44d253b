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
//    the finished accumulator, 32 columns (tokens) at a time, and stores
//    them: for one token, 32 lanes write 32 consecutive rows of Y.
// All waits are bounded and give up when another thread has recorded an
// error; tensor memory is freed on every path.
#include <cudaTypedefs.h>

#include <atomic>

#include "tc_common.cuh"

namespace qg {

constexpr int kGemmBM = 128, kGemmBK = 64;
constexpr int kGemmThreads = 6 * 32;
constexpr int kGemmTileBytes = kGemmBM * kGemmBK * 2;  // the A tile, f16
constexpr int kGemmHdrBytes = 1024;
// Per token-tile width BN (128 or 256): B tile bytes, stage bytes, ring
// depth (what fits next to the header), shared memory, tensor-memory columns
// (two accumulators).
template <int BN> struct GemmShape {
    static constexpr int kBTile = BN * kGemmBK * 2;
    static constexpr int kStage = kGemmTileBytes + kBTile;
    static constexpr int kStages = BN == 128 ? 6 : 4;
    static constexpr int kSmem = 1024 /* base alignment */ + kGemmHdrBytes + kStages * kStage;
    static constexpr int kTmemCols = 2 * BN;
};

struct GemmParams {
    float *y;  // [n_tok][n_out]
    int32_t *err;
    int n_out, n_tok, K;
    int tiles_m, tiles_n;
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

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_f16_tc_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                       const GemmParams p) {
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
            const int row = tm * kGemmBM + 32 * q + lane;
#pragma unroll 1
            for (int c0 = 0; c0 < kGemmBN; c0 += 32) {
                uint32_t v[32];
                tc_ld32_wait(tl + static_cast<uint32_t>(d * kGemmBN + c0), v);
                const int tok0 = tn * kGemmBN + c0;
                if (row < p.n_out) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (tok0 + j < p.n_tok)
                            p.y[static_cast<int64_t>(tok0 + j) * p.n_out + row] = __uint_as_float(v[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty0 + 8 * d);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tc_dealloc(tmem, kGemmTmemCols);
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

}  // namespace

cudaError_t launch_f32_to_f16(const float *x, __half *out, int64_t n, int sms, cudaStream_t s) {
    const int64_t groups = n / 8;
    if (groups == 0) return cudaSuccess;
    int64_t grid = (groups + 255) / 256;
    if (grid > static_cast<int64_t>(sms) * 16) grid = static_cast<int64_t>(sms) * 16;
    f32_to_f16_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(x, out, groups);
    return cudaGetLastError();
}

template <int BN>
cudaError_t launch_gemm_bn(const __half *A, const __half *B, float *y, int64_t n_out, int64_t n_tok, int64_t K,
                           int32_t *err, int sms, int device, cudaStream_t s) {
    CUtensorMap ta, tb;
    if (!encode_f16_map(&ta, A, n_out, K, kGemmBM) || !encode_f16_map(&tb, B, n_tok, K, BN)) {
        g_launch_step = "cuTensorMapEncodeTiled";
        return cudaErrorInvalidValue;
    }
    GemmParams p = {};
    p.y = y;
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
    return launch_pdl(gemm_f16_tc_kernel<BN>, grid, kGemmThreads, GemmShape<BN>::kSmem, s, ta, tb, p);
}

// Y[n_tok][n_out] = A[n_out][K] . B[n_tok][K]^T for f16 A, B (16-byte
// aligned, K a multiple of 8). Token tiles of 256 (an mma of N = 256 does
// twice the work of N = 128 for about 1.35 times the cycles) when they still
// give every SM a tile, else 128.
cudaError_t launch_gemm_f16_tc(const __half *A, const __half *B, float *y, int64_t n_out, int64_t n_tok, int64_t K,
                               int32_t *err, int sms, int device, cudaStream_t s) {
    const int64_t tiles256 = ((n_out + kGemmBM - 1) / kGemmBM) * ((n_tok + 255) / 256);
    if (tiles256 >= sms) return launch_gemm_bn<256>(A, B, y, n_out, n_tok, K, err, sms, device, s);
    return launch_gemm_bn<128>(A, B, y, n_out, n_tok, K, err, sms, device, s);
}

}  // namespace qg
