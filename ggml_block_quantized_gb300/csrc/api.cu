// api.cu - the C ABI declared in include/qgemv.h: argument validation,
// launch planning and kernel launches. Nothing here allocates device memory
// or synchronizes (except qg_device_error, which says so).
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <atomic>

#include "gemm_tc.cuh"
#include "gemv_launch.cuh"
#include "gemv_tc.cuh"

namespace qg {

cudaError_t launch_quantize_kernel(int type, int grid, int block, cudaStream_t s, const float *x, uint8_t *out,
                                   int64_t n_blocks);
cudaError_t launch_quantize_batched_kernel(int type, int grid, int block, cudaStream_t s, const QuantTable &t,
                                           uint8_t *out, int n_mats, int64_t blocks_per_mat);
// dequant.cu: every element of `groups` 8-element groups of the block stream
// w to O (f32 for dequantize_rows, f16 for the prefill GEMM's operand).
template <class O>
cudaError_t launch_dequant(int type, const uint8_t *w, O *out, int64_t groups, unsigned grid, int threads,
                           cudaStream_t s);
cudaError_t launch_gemv_tc_q4_k(const TcParams &p, const TcMat *mats, int n, int grid, int smem, int smem_optin,
                                int device, cudaStream_t s);

__device__ int32_t g_device_error = 0;

// One thread waits, with the product kernels' bounded wait, on an mbarrier
// that nothing arrives on; the wait gives up after about one second and the
// kernel records the consumer-wait code and returns.
__global__ void selftest_wait_kernel(int32_t *err) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_addr(&bar);
    mbar_init(b, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!mbar_wait_bounded(b, 0u)) record_error(err, kErrConsumerWait);
}

// Does nothing. quantize_rows launches it after the weight quantizer without
// programmatic dependent launch, so it starts only once the weights are
// written and visible; a product enqueued next, which may start streaming W
// while the kernel before it finishes, then reads finished weights.
__global__ void stream_order_kernel() {}

namespace {

thread_local char g_last_cuda_error[256] = "";

int cuda_fail(cudaError_t e, const char *where = "") {
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s (%s)", cudaGetErrorName(e),
                  cudaGetErrorString(e), where);
    return QG_ERR_CUDA;
}

bool block_info(int type, int *elems, int *bytes) {
    switch (type) {
    case QG_F32: *elems = 1; *bytes = 4; return true;
    case QG_F16: *elems = 1; *bytes = 2; return true;
    case QG_Q4_0: *elems = 32; *bytes = 18; return true;
    case QG_Q4_1: *elems = 32; *bytes = 20; return true;
    case QG_Q5_0: *elems = 32; *bytes = 22; return true;
    case QG_Q8_0: *elems = 32; *bytes = 34; return true;
    case QG_Q8_1: *elems = 32; *bytes = 36; return true;
    case QG_Q2_K: *elems = 256; *bytes = 84; return true;
    case QG_Q3_K: *elems = 256; *bytes = 110; return true;
    case QG_Q4_K: *elems = 256; *bytes = 144; return true;
    case QG_Q5_K: *elems = 256; *bytes = 176; return true;
    case QG_Q6_K: *elems = 256; *bytes = 210; return true;
    case QG_Q8_K: *elems = 256; *bytes = 292; return true;
    default: return false;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DeviceInfo {
    int device;
    int sms;
    int smem_optin;  // opt-in dynamic shared memory per CTA (bytes)
    int32_t *err;    // device address of g_device_error on this device
};

int current_device(DeviceInfo *info) {
    static int sm_count[64] = {0};
    static int optin[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int sms = (dev >= 0 && dev < 64) ? __atomic_load_n(&sm_count[dev], __ATOMIC_RELAXED) : 0;
    int smem = (dev >= 0 && dev < 64) ? __atomic_load_n(&optin[dev], __ATOMIC_RELAXED) : 0;
    if (sms == 0 || smem == 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(MultiProcessorCount)");
        e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(MaxSharedMemoryPerBlockOptin)");
        if (smem > kSmemLimit) smem = kSmemLimit;
        if (dev >= 0 && dev < 64) {
            __atomic_store_n(&sm_count[dev], sms, __ATOMIC_RELAXED);
            __atomic_store_n(&optin[dev], smem, __ATOMIC_RELAXED);
        }
    }
    static int32_t *err_addr[64] = {nullptr};
    int32_t *err = (dev >= 0 && dev < 64) ? __atomic_load_n(&err_addr[dev], __ATOMIC_ACQUIRE) : nullptr;
    if (!err) {
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&err), g_device_error);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_device_error)");
        if (dev >= 0 && dev < 64) __atomic_store_n(&err_addr[dev], err, __ATOMIC_RELEASE);
    }
    info->device = dev;
    info->sms = sms;
    info->smem_optin = smem;
    info->err = err;
    return QG_OK;
}

int env_int(const char *name, int dflt, int lo, int hi) {
    const char *s = std::getenv(name);
    if (!s || !*s) return dflt;
    int v = std::atoi(s);
    return v < lo ? lo : (v > hi ? hi : v);
}

// Tuning knobs. Each is read once from the environment variable of the same
// name (defaults are the measured best) and can be set for the rest of the
// process with qg_tune():
//  QG_CTAS_PER_SM, QG_RING_KIB: CTAs per SM the __dp4a GEMV grid aims at, and
//    its shared-memory ring budget per CTA in KiB;
//  QG_MMA_MIN_NVEC: vectors from which K-quant (Q2_K .. Q6_K) products run on the
//    tensor cores;
//  QG_MMA_GROUP_MELEM: the 32-element types (Q4_0, Q4_1, Q5_0, Q8_0) take the
//    tensor cores from QG_MMA_MIN_NVEC vectors when a matrix's elements
//    n_out * n_in times (vectors - 3) reach this many Mi (2^20): the __dp4a
//    kernel's time grows with the vectors, the tensor-core kernel's barely,
//    but the latter pays a fixed activation-panel prologue. Measured on this
//    GPU, all four types win at 32000 x 4096 and 11008 x 4096 from 4 vectors
//    (Q5_0 at 11008 ties), at 4096 x 4096 from 5 to 7 depending on the type
//    (the default, 40, takes the tensor cores from 6 there: within 8% of
//    the faster kernel for every type);
//  QG_MMA_PANEL, QG_MMA_KB: mma.sync plan overrides (activation source: 0
//    automatic, 1 a shared-memory panel, 8 the biased-int8 panel; an upper
//    bound on blocks per chunk, 0 none);
//  QG_FUSED_QUANT_KIB: f32 activations up to this size are quantized inside
//    the GEMV's prologue;
//  QG_FUSED_MAX_MIB: ... for a single matrix of at most this many MiB of
//    blocks (larger ones take the separate quantization launch; the default
//    sets no limit: in-kernel quantization measured faster at every size);
//  QG_TC: the tcgen05 Q4_K kernel for three or more vectors -- 0 never (the
//    default: the mma.sync kernel measured faster on this GPU), 1 whenever its
//    shared memory fits (rows of 8 or 16 blocks);
//  QG_FUSED_GEMM: qgemm on Q4_K weights dequantizes into an f16 copy in the
//    workspace first (0) or inside the GEMM, into tensor memory (1: no f16
//    copy of W); 2, the default, fuses while the fused GEMM has at most two
//    256-token tiles per SM (fused_gemm_default: measured as fast or faster
//    from 16 to 2048 tokens on 4096 x 4096, 10% slower at 4096 tokens);
//  QG_GEMM_KSPLIT: the fused GEMM splits each tile's k-blocks into at most this
//    many parts when its tiles leave SMs idle (1: no split).
enum KnobId {
    kKnobCtasPerSm,
    kKnobRingKib,
    kKnobMmaMinNvec,
    kKnobMmaPanel,
    kKnobMmaKb,
    kKnobFusedQuantKib,
    kKnobTc,
    kKnobFusedMaxMib,
    kKnobFusedGemm,
    kKnobMmaGroupMelem,
    kKnobGemmKsplit,
    kKnobCount
};
struct KnobDef {
    const char *name;
    int dflt, lo, hi;
};
constexpr KnobDef kKnobs[kKnobCount] = {
    {"QG_CTAS_PER_SM", 2, 1, 4},          {"QG_RING_KIB", 96, 16, 200}, {"QG_MMA_MIN_NVEC", 3, 1, QG_MAX_NVEC + 1},
    {"QG_MMA_PANEL", 0, 0, 16},           {"QG_MMA_KB", 0, 0, 4096},    {"QG_FUSED_QUANT_KIB", 16, 0, 1024},
    {"QG_TC", 0, 0, 1},                   {"QG_FUSED_MAX_MIB", 1 << 20, 0, 1 << 20},
    {"QG_FUSED_GEMM", 2, 0, 2},           {"QG_MMA_GROUP_MELEM", 40, 0, 1 << 20},
    {"QG_GEMM_KSPLIT", 8, 1, 8}};
std::atomic<int> g_knob_val[kKnobCount];  // value + 1; 0 = not read yet

int knob(KnobId k) {
    int v = g_knob_val[k].load(std::memory_order_relaxed);
    if (v == 0) {
        int expected = 0;
        const int env = env_int(kKnobs[k].name, kKnobs[k].dflt, kKnobs[k].lo, kKnobs[k].hi) + 1;
        g_knob_val[k].compare_exchange_strong(expected, env, std::memory_order_relaxed);
        v = g_knob_val[k].load(std::memory_order_relaxed);
    }
    return v - 1;
}

int tune_ctas_per_sm() { return knob(kKnobCtasPerSm); }
int tune_ring_kib() { return knob(kKnobRingKib); }
int tune_mma_min_nvec() { return knob(kKnobMmaMinNvec); }
int tune_mma_panel() { return knob(kKnobMmaPanel); }
int tune_mma_kb() { return knob(kKnobMmaKb); }
int tune_tc() { return knob(kKnobTc); }

// The weight types with a tensor-core item: every K-quant type, and the
// 32-element types taken eight blocks at a time (rows of whole groups).
bool mma_grouped(int type) { return type == QG_Q4_0 || type == QG_Q4_1 || type == QG_Q5_0 || type == QG_Q8_0; }
bool mma_type(int type) { return (type >= QG_Q2_K && type <= QG_Q6_K) || mma_grouped(type); }

// Whether a product (not the exact-block-sum diagnostic) may take the
// tensor-core kernel; it reads activations from the workspace, so such calls
// never quantize x inside the GEMV prologue.
bool mma_preferred(int type, int64_t n_vec) { return mma_type(type) && n_vec >= tune_mma_min_nvec(); }

// ... and whether it does, for a matrix of n_out x n_in.
bool mma_wins(int type, int64_t n_vec, int64_t n_out, int64_t n_in) {
    if (!mma_preferred(type, n_vec)) return false;
    return !mma_grouped(type) || n_out * n_in * (n_vec - 3) >= (static_cast<int64_t>(knob(kKnobMmaGroupMelem)) << 20);
}

size_t act_smem_bytes(int type, int lpb, int nb, int nv) {
    switch (type) {
    case QG_Q8_0: return TypeQ8_0::act_bytes(nb, nv);
    case QG_Q4_0: return TypeQ4_0::act_bytes(nb, nv);
    case QG_Q4_1: return TypeQ4_1::act_bytes(nb, nv);
    case QG_Q5_0: return TypeQ5_0::act_bytes(nb, nv);
    case QG_Q4_K: return TypeQ4_K::act_bytes(nb, nv);
    case QG_Q5_K: return TypeQ5_K::act_bytes(nb, nv);
    case QG_Q2_K: return TypeQ2_K::act_bytes(nb, nv);
    case QG_Q3_K: return TypeQ3_K::act_bytes(nb, nv);
    case QG_Q6_K: return lpb == TypeQ6_K4::kLanesPerBlock ? TypeQ6_K4::act_bytes(nb, nv) : TypeQ6_K::act_bytes(nb, nv);
    default: return 0;
    }
}

size_t round16(size_t v) { return (v + 15) & ~size_t(15); }

constexpr int kSmemTailPad = 16;  // unaligned word reads may touch up to 4 bytes past a stage

// The item variants a type offers (lanes per weight block); Q6_K has a
// two-lane item (fewer instructions per code) and a four-lane one (its
// 8-block iterations fill better for some row lengths).
int item_lpbs(int type, int (&out)[2]) {
    switch (type) {
    case QG_Q4_K: out[0] = TypeQ4_K::kLanesPerBlock; return 1;
    case QG_Q5_K: out[0] = TypeQ5_K::kLanesPerBlock; return 1;
    case QG_Q2_K: out[0] = TypeQ2_K::kLanesPerBlock; return 1;
    case QG_Q3_K: out[0] = TypeQ3_K::kLanesPerBlock; return 1;
    case QG_Q6_K: out[0] = TypeQ6_K::kLanesPerBlock; out[1] = TypeQ6_K4::kLanesPerBlock; return 2;
    default: out[0] = 1; return 1;
    }
}

// Stage geometry and grid of one GEMV launch. Among the configurations whose
// shared memory lets the tuned number of CTAs share an SM (more resident
// warps hide more latency), the plan keeps the lanes of each warp's item
// loop fullest, then the larger ring. (In-kernel quantization of f32 x needs
// no shared memory of its own: each warp loads the blocks it quantizes.)
// Returns QG_ERR_SHAPE when the activations do not fit next to two stages
// even with one CTA per SM.
int plan_gemv(int type, int64_t total_rows, int64_t n_in, int nv, int sms, int smem_limit, GemvParams *p,
              GemvLaunch *l) {
    int elems, bytes;
    if (!block_info(type, &elems, &bytes)) return QG_ERR_TYPE;
    const int64_t nb = n_in / elems;
    const int64_t row_bytes = nb * bytes;
    const size_t ring_target = static_cast<size_t>(tune_ring_kib()) * 1024;
    const size_t sm_smem = 228 * 1024, cta_reserve = 1024;  // per-SM shared memory, per-CTA driver share
    int lpbs[2] = {1, 1};
    const int n_lpb = item_lpbs(type, lpbs);
    for (int per_sm = tune_ctas_per_sm(); per_sm >= 1; --per_sm) {
        size_t budget = sm_smem / per_sm - cta_reserve;
        if (budget > static_cast<size_t>(smem_limit)) budget = static_cast<size_t>(smem_limit);
        bool found = false;
        double best_score = -1.0;
        GemvParams bp = {};
        size_t best_smem = 0;
        int best_lpb = lpbs[0];
        for (int li = 0; li < n_lpb; ++li) {
        const int lpb = lpbs[li];
        const size_t act = round16(act_smem_bytes(type, lpb, static_cast<int>(nb), nv));
        {
            const size_t fixed0 = kHeaderBytes + act + kSmemTailPad;
            for (int split = 1; split <= kConsumerWarps; split *= 2) {
            for (int rpw = kRowsPerWarp; rpw >= 1; --rpw) {  // rows a warp group takes per stage
                const int R = (kConsumerWarps / split) * rpw;
                const size_t stage = round16(static_cast<size_t>(R) * row_bytes + 15);
                if (split < kConsumerWarps && stage > 40960) continue;  // stages of <= 40 KiB
                // partial sums of split rows, double-buffered: [2S][warps][rows per warp][nv] floats
                auto red_bytes = [&](int S) {
                    return split > 1 ? round16(static_cast<size_t>(2 * S) * kConsumerWarps * kRowsPerWarp * nv * 4) : 0;
                };
                if (fixed0 + red_bytes(2) + 2 * stage > budget) continue;
                int S = static_cast<int>(ring_target / stage);
                S = S < 2 ? 2 : (S > kMaxStages ? kMaxStages : S);
                while (S > 2 && fixed0 + red_bytes(S) + S * stage > budget) --S;
                // lane use of the busiest warp's flattened item loop (two rows)
                const int64_t items = (nb + split - 1) / split * lpb * rpw;
                const double eff = static_cast<double>(nb * lpb * rpw) / split /
                                   (32.0 * static_cast<double>((items + 31) / 32));
                // fuller lanes first; then fewer warps per row (each stage does
                // more work per warp, and no partial sums to add up); then two
                // rows per warp group over one (the per-stage work is shared by
                // more blocks); then the item with fewer lanes per block (fewer
                // instructions per code); then the larger ring
                const double score = static_cast<int>(eff * 20.0 + 0.5) * 100.0 - split * 10.0 -
                                     (kRowsPerWarp - rpw) * 3.0 - li * 6.0 +
                                     static_cast<double>(S * stage) / (4.0 * 1024 * 1024);
                if (score > best_score) {
                    best_score = score;
                    found = true;
                    best_lpb = lpb;
                    bp.row_bytes = row_bytes;
                    bp.total_rows = total_rows;
                    bp.nb = static_cast<int>(nb);
                    bp.rows_per_stage = R;
                    bp.split = split;
                    bp.split_log2 = split == 1 ? 0 : split == 2 ? 1 : split == 4 ? 2 : 3;
                    bp.n_stages = S;
                    bp.stage_bytes = static_cast<int>(stage);
                    bp.act_bytes = static_cast<int>(act);
                    bp.red_bytes = static_cast<int>(red_bytes(S));
                    // stages in flight while the consumers' first activation
                    // loads travel: about 56 KiB (measured best for rows of
                    // 1.3-3.4 KB)
                    bp.pre_x = static_cast<int>(57344 / stage);
                    bp.pre_x = bp.pre_x < 1 ? 1 : (bp.pre_x > S ? S : bp.pre_x);
                    best_smem = fixed0 + red_bytes(S) + S * stage;
                }
            }
            }
        }
        }
        if (!found) continue;
        *p = bp;
        const int64_t tiles = (total_rows + bp.rows_per_stage - 1) / bp.rows_per_stage;
        const int64_t cap = static_cast<int64_t>(sms) * per_sm;
        l->grid = static_cast<int>(tiles < cap ? tiles : cap);
        l->smem = static_cast<int>(best_smem);
        l->smem_optin = smem_limit;
        l->sms = sms;
        l->lpb = best_lpb;
        return QG_OK;
    }
    return QG_ERR_SHAPE;
}

// Geometry of a tensor-core launch. A stage is 16 rows in 4 groups of 4
// whose starts are 32 modulo 128 bytes apart (one bulk copy per group when
// the stage spans whole rows). When a whole row has at most 16 blocks, it is
// one stage and 8 consumer warps keep their activation fragments in
// registers (nothing but the ring in shared memory). Otherwise 16 warps read
// them from a shared-memory panel (f16 when it fits, else biased int8), the
// row is split into chunks of kb blocks, and among the shapes that fit the
// plan keeps the warps busiest, then a ring of at least 3 stages, then the
// f16 panel, then the longer chunk. Partial-output buffers are doubled when
// that keeps the ring as deep. Returns QG_ERR_SHAPE when nothing fits (the
// caller then uses the __dp4a kernel).
namespace {

// Slot layout for kb blocks per chunk of a row of nb blocks of `bytes` each.
void mma_slot_layout(int nb, int kb, int bytes, int *rpitch, int *gpitch, bool apart = false) {
    if (apart) {
        // one copy per row, rows 16 mod 128 bytes apart and groups 32 mod
        // 128: the 8 rows a 32-bit warp load touches (2 in each group) start
        // on 8 different 4-bank sets
        *rpitch = static_cast<int>((static_cast<int64_t>(kb) * bytes + 32 + 111) / 128 * 128 + 16);
        *gpitch = (4 * *rpitch + 95) / 128 * 128 + 32;
        return;
    }
    const bool contig = kb == nb;
    const int64_t row = static_cast<int64_t>(nb) * bytes;
    *rpitch = contig ? static_cast<int>(row) : static_cast<int>(round16(static_cast<size_t>(kb) * bytes + 32));
    int gp = contig ? static_cast<int>(round16(static_cast<size_t>(4 * row + 32))) : 4 * *rpitch;
    *gpitch = (gp + 95) / 128 * 128 + 32;  // the smallest value >= gp that is 32 mod 128
}

// Ring depth and partial-buffer count for `stage` bytes per slot next to
// `fixed` bytes; false when not even two stages fit.
bool mma_ring(int64_t smem_limit, int64_t fixed, int64_t stage, int nw, int *S, int *red_slots) {
    const int64_t red = mma_red_bytes(nw);
    if (fixed + 2 * (stage + red) > smem_limit) return false;
    int64_t s1 = (smem_limit - fixed) / (stage + red);
    int64_t s2 = (smem_limit - fixed) / (stage + 2 * red);
    if (s1 > kMmaMaxStages) s1 = kMmaMaxStages;
    if (s2 > kMmaMaxStages) s2 = kMmaMaxStages;
    const bool dbl = s2 >= 2 && s2 >= (s1 < 3 ? s1 : 3);
    *S = static_cast<int>(dbl ? s2 : s1);
    *red_slots = dbl ? 2 * *S : *S;
    return true;
}

}  // namespace

int plan_gemv_mma(int type, int64_t total_tiles, int64_t n_in, int nv, int sms, int smem_limit, MmaParams *p,
                  MmaLaunch *l) {
    int elems, bytes;
    if (!block_info(type, &elems, &bytes)) return QG_ERR_TYPE;
    const bool grouped = mma_grouped(type);
    // rows of 32-bit lane loads: one copy per row, pitches that spread a warp
    // load's 8 rows over the banks (the K-quant items' loads measured no
    // faster with it)
    const bool apart = grouped;
    if (grouped) {  // eight 32-element blocks per panel block: rows of whole groups only
        if (n_in % 256 != 0) return QG_ERR_SHAPE;
        elems = 256;
        bytes *= 8;
    }
    const int64_t nb64 = n_in / elems;
    if (nb64 < 1 || nb64 > 4096 || total_tiles < 1) return QG_ERR_SHAPE;
    const int nb = static_cast<int>(nb64);
    MmaParams bp = {};
    MmaLaunch bl = {};
    bp.row_bytes = nb64 * bytes;
    bp.total_tiles = total_tiles;
    bp.nb = nb;
    bp.nv = nv;
    bool found = false;
    const int force = tune_mma_panel();  // 0 automatic, 1 a panel, 8 the int8 panel
    constexpr int rw = 8;  // consumer warps of the register kernel: blocks w and w + 8 each
    if (force == 0 && nb <= 2 * rw && !grouped) {
        int rp, gp, S, R;
        mma_slot_layout(nb, nb, bytes, &rp, &gp);
        if (mma_ring(smem_limit, kMmaHeaderBytes, 4 * static_cast<int64_t>(gp), rw, &S, &R)) {
            bp.kb = nb;
            bp.n_chunks = 1;
            bp.rpitch = rp;
            bp.gpitch = gp;
            bp.contig = 1;
            bp.stage_bytes = 4 * gp;
            bp.n_stages = S;
            bp.red_slots = R;
            bp.rec_bytes = 0;
            bp.panel_bytes = 0;
            bl.smem = kMmaHeaderBytes + S * bp.stage_bytes + R * mma_red_bytes(rw);
            bl.mode = kMmaRegs;
            bl.warps = rw;
            found = true;
        }
    }
    if (!found) {
        constexpr int W = 16;
        long best = -1;
        constexpr int kCands = 9;
        const int cands[kCands] = {nb, 32, 24, 16, 12, 11, 10, 8, 4};
        for (int f = 0; f < 2; ++f) {
            const bool b16 = f == 0;
            if (b16 && force == 8) continue;
            // grouped types: per record and lane a float4 (512 bytes) in place of the Q8_K tail
            const int rec = mma_rec_bytes(b16) + (grouped ? 512 - kMmaTailBytes : 0);
            const int64_t panel = static_cast<int64_t>(nb) * rec;
            for (int ci = 0; ci < kCands; ++ci) {
                const int kb = cands[ci];
                if (kb > nb || (ci > 0 && kb == nb)) continue;
                if (tune_mma_kb() > 0 && kb > tune_mma_kb()) continue;
                int rp, gp, S, R;
                mma_slot_layout(nb, kb, bytes, &rp, &gp, apart);
                const int64_t stage = 4 * static_cast<int64_t>(gp);
                const int64_t fixed = kMmaHeaderBytes + panel;
                if (!mma_ring(smem_limit, fixed, stage, W, &S, &R)) continue;
                const int n_chunks = (nb + kb - 1) / kb;
                const int last = nb - (n_chunks - 1) * kb;
                const int64_t slots = static_cast<int64_t>(n_chunks - 1) * ((kb + W - 1) / W * W) + (last + W - 1) / W * W;
                const long eff = static_cast<long>(50.0 * nb / slots + 0.5);
                const long score = eff * 100000 + (S >= 3 ? 10000 : 0) + (b16 ? 1000 : 0) + kb;
                if (score <= best) continue;
                best = score;
                bp.kb = kb;
                bp.n_chunks = n_chunks;
                bp.rpitch = rp;
                bp.gpitch = gp;
                bp.contig = kb == nb && !apart ? 1 : 0;
                bp.stage_bytes = static_cast<int>(stage);
                bp.n_stages = S;
                bp.red_slots = R;
                bp.rec_bytes = rec;
                bp.panel_bytes = static_cast<int>(panel);
                bl.smem = static_cast<int>(fixed + S * stage + static_cast<int64_t>(R) * mma_red_bytes(W));
                bl.mode = b16 ? kMmaPanel16 : kMmaPanel8;
                bl.warps = W;
                found = true;
            }
        }
    }
    if (!found) return QG_ERR_SHAPE;
    *p = bp;
    bl.grid = static_cast<int>(total_tiles < sms ? total_tiles : sms);
    bl.smem_optin = smem_limit;
    *l = bl;
    return QG_OK;
}

// Plan of the tcgen05 Q4_K kernel: ring depth next to the activation panel,
// grid. False when the knob is off or the shapes rule it out: rows of 8 or 16
// blocks only (whole rows travel per stage; blocks go to the mma in groups of
// eight), or fewer than two stages of shared memory.
bool plan_gemv_tc(int type, int64_t tiles, int64_t n_in, int nv, int n_mats, int sms, int smem_limit, TcParams *p,
                  int *grid, int *smem) {
    const int mode = tune_tc();
    if (type != QG_Q4_K || mode == 0 || n_mats < 1 || n_mats > kTcMaxBatch || tiles < 1) return false;
    const int64_t nb = n_in / 256;
    if (nb != kTcGroupBlocks && nb != 2 * kTcGroupBlocks) return false;
    const int64_t fixed = tc_smem_bytes(static_cast<int>(nb), 0);
    int64_t S = (smem_limit - fixed) / tc_stage_bytes(static_cast<int>(nb));
    if (S > kTcMaxStages) S = kTcMaxStages;
    if (S < 2) return false;
    *p = TcParams{};
    p->total_tiles = tiles;
    p->n_mats = n_mats;
    p->nb = static_cast<int>(nb);
    p->nv = nv;
    p->n_stages = static_cast<int>(S);
    *grid = static_cast<int>(tiles < sms ? tiles : sms);
    *smem = tc_smem_bytes(static_cast<int>(nb), static_cast<int>(S));
    return true;
}

cudaError_t launch_gemv(int type, const GemvParams &p, const GemvMat *mats, int n, int nv, bool isums,
                        const GemvLaunch &l, int device, cudaStream_t s) {
    switch (type) {
    case QG_Q8_0: return launch_gemv_q8_0(p, mats, n, nv, isums, l, device, s);
    case QG_Q4_0: return launch_gemv_q4_0(p, mats, n, nv, isums, l, device, s);
    case QG_Q4_1: return launch_gemv_q4_1(p, mats, n, nv, isums, l, device, s);
    case QG_Q5_0: return launch_gemv_q5_0(p, mats, n, nv, isums, l, device, s);
    case QG_Q4_K: return launch_gemv_q4_k(p, mats, n, nv, isums, l, device, s);
    case QG_Q5_K: return launch_gemv_q5_k(p, mats, n, nv, isums, l, device, s);
    case QG_Q2_K: return launch_gemv_q2_k(p, mats, n, nv, isums, l, device, s);
    case QG_Q3_K: return launch_gemv_q3_k(p, mats, n, nv, isums, l, device, s);
    case QG_Q6_K: return launch_gemv_q6_k(p, mats, n, nv, isums, l, device, s);
    default: return cudaErrorInvalidValue;
    }
}

// Weight-type checks shared by the product entry points.
int check_weight_type(int type) {
    int e, b;
    if (!block_info(type, &e, &b)) return QG_ERR_TYPE;
    if (qtype_act_type(type) < 0) return QG_ERR_PAIR;
    return QG_OK;
}

int check_gemv_shape(int type, int64_t n_out, int64_t n_in, int64_t n_vec) {
    int elems, bytes;
    if (!block_info(type, &elems, &bytes)) return QG_ERR_TYPE;
    if (n_out < 0 || n_in < 0 || n_out > INT32_MAX) return QG_ERR_SHAPE;
    if (n_vec < 1 || n_vec > QG_MAX_NVEC) return QG_ERR_SHAPE;
    if (n_in % elems != 0 || n_in / elems > INT32_MAX / 4) return QG_ERR_SHAPE;
    return QG_OK;
}

int launch_quantize(int act_type, const float *x, void *xq, int64_t n_blocks, int sms, cudaStream_t s) {
    if (n_blocks == 0) return QG_OK;
    const int warps_per_cta = 8;
    int64_t grid = (n_blocks + warps_per_cta - 1) / warps_per_cta;
    if (grid > static_cast<int64_t>(sms) * 16) grid = static_cast<int64_t>(sms) * 16;
    uint8_t *out = static_cast<uint8_t *>(xq);
    const int g = static_cast<int>(grid), blk = 32 * warps_per_cta;
    const cudaError_t e = launch_quantize_kernel(act_type, g, blk, s, x, out, n_blocks);
    return e == cudaSuccess ? QG_OK : cuda_fail(e, "quantize launch");
}

// Activations of n matrices (xs[m], blocks_per_mat blocks each) into xq.
int launch_quantize_batched(int act_type, const QuantTable &t, int n, void *xq, int64_t blocks_per_mat, int sms,
                            cudaStream_t s) {
    const int64_t n_blocks = blocks_per_mat * n;
    if (n_blocks == 0) return QG_OK;
    const int warps_per_cta = 8;
    int64_t grid = (n_blocks + warps_per_cta - 1) / warps_per_cta;
    if (grid > static_cast<int64_t>(sms) * 16) grid = static_cast<int64_t>(sms) * 16;
    uint8_t *out = static_cast<uint8_t *>(xq);
    const int g = static_cast<int>(grid), blk = 32 * warps_per_cta;
    const cudaError_t e = launch_quantize_batched_kernel(act_type, g, blk, s, t, out, n, blocks_per_mat);
    return e == cudaSuccess ? QG_OK : cuda_fail(e, "batched quantize launch");
}

// Activations of at most this many f32 bytes per call (QG_FUSED_QUANT_KIB,
// default 16 KiB) are quantized inside the GEMV's prologue (every CTA
// quantizes all of x); larger ones go through the separate quantization
// launch into the workspace. Every CTA's share of that prologue grows with
// the blocks of x: measured on this GPU, a 4096-element x (16 KiB) is
// faster quantized in the prologue, an 11008-element one (43 KiB) or two
// vectors of 4096 (32 KiB) through the separate launch.
int64_t fused_quant_max_bytes() { return static_cast<int64_t>(knob(kKnobFusedQuantKib)) * 1024; }

bool fused_quantization(int64_t n_in, int64_t n_vec) { return 4 * n_in * n_vec <= fused_quant_max_bytes(); }

// A single product quantizes x inside the GEMV when its matrix is at most
// QG_FUSED_MAX_MIB of blocks (by default any matrix); above that the separate
// quantization launch, overlapped with the GEMV's weight prefetch, is taken.
bool fused_single(int type, int64_t n_out, int64_t n_in, int64_t n_vec) {
    return fused_quantization(n_in, n_vec) && !mma_wins(type, n_vec, n_out, n_in) &&
           qtype_nbytes(type, n_in) * n_out <= (static_cast<int64_t>(knob(kKnobFusedMaxMib)) << 20);
}

// The product over `n` matrices of one type, row length and vector count
// (activations from mats[i].x quantized in the kernel when x_bytes > 0, else
// from mats[i].xq). Arguments are already validated.
int run_gemv_mats(int type, GemvMat *mats, int n, int64_t n_in, int64_t n_vec, size_t x_bytes, bool isums,
                  const DeviceInfo &dev, cudaStream_t s) {
    int64_t total = 0;
    for (int i = 0; i < n; ++i) {
        mats[i].row_base = total;
        total += mats[i].n_out;
    }
    if (total == 0) return QG_OK;
    bool use_mma = !isums && x_bytes == 0 && mma_preferred(type, n_vec);
    if (use_mma && mma_grouped(type)) {
        // each matrix takes the kernel a call on it alone would take (the
        // choice depends on its size), so a batch gives the same bits as
        // single calls: the matrices the tensor cores win on in one launch,
        // the others in a second
        GemvMat win[QG_MAX_BATCH], rest[QG_MAX_BATCH];
        int nw = 0, nr = 0;
        for (int i = 0; i < n; ++i) {
            if (mma_wins(type, n_vec, mats[i].n_out, n_in))
                win[nw++] = mats[i];
            else
                rest[nr++] = mats[i];
        }
        if (nw > 0 && nr > 0) {
            int st = run_gemv_mats(type, win, nw, n_in, n_vec, x_bytes, isums, dev, s);
            return st != QG_OK ? st : run_gemv_mats(type, rest, nr, n_in, n_vec, x_bytes, isums, dev, s);
        }
        use_mma = nw > 0;
    }
    if (use_mma) {
        // several vectors: the tcgen05 kernel (Q4_K, launches of many 16-row
        // tiles), else the mma.sync kernel, when their shapes fit
        int64_t tiles16 = 0;
        for (int i = 0; i < n; ++i) tiles16 += (mats[i].n_out + kTcRows - 1) / kTcRows;
        TcParams tp = {};
        int tgrid = 0, tsmem = 0;
        if (plan_gemv_tc(type, tiles16, n_in, static_cast<int>(n_vec), n, dev.sms, dev.smem_optin, &tp, &tgrid,
                         &tsmem)) {
            TcMat tm[kTcMaxBatch];
            int64_t base = 0;
            for (int i = 0; i < n; ++i) {
                tm[i] = TcMat{};
                tm[i].W = mats[i].W;
                tm[i].xq = mats[i].xq;
                tm[i].y = mats[i].y;
                tm[i].n_out = mats[i].n_out;
                tm[i].tile_base = base;
                base += (mats[i].n_out + kTcRows - 1) / kTcRows;
            }
            tp.err = dev.err;
            cudaError_t e = launch_gemv_tc_q4_k(tp, tm, n, tgrid, tsmem, dev.smem_optin, dev.device, s);
            if (e != cudaSuccess) {
                char where[160];
                std::snprintf(where, sizeof where, "%s; tcgen05 grid %d block %d smem %d stages %d", g_launch_step,
                              tgrid, kTcThreads, tsmem, tp.n_stages);
                return cuda_fail(e, where);
            }
            return QG_OK;
        }
        MmaMat mm[QG_MAX_BATCH];
        int64_t tiles = 0;
        for (int i = 0; i < n; ++i) {
            mm[i] = MmaMat{};
            mm[i].W = mats[i].W;
            mm[i].xq = mats[i].xq;
            mm[i].y = mats[i].y;
            mm[i].n_out = mats[i].n_out;
            mm[i].tile_base = tiles;
            tiles += (mats[i].n_out + kMmaTileRows - 1) / kMmaTileRows;
        }
        MmaParams mp = {};
        MmaLaunch ml = {};
        if (plan_gemv_mma(type, tiles, n_in, static_cast<int>(n_vec), dev.sms, dev.smem_optin, &mp, &ml) == QG_OK) {
            mp.err = dev.err;
            mp.n_mats = n;
            cudaError_t e = launch_gemv_mma(type, mp, mm, n, ml, dev.device, s);
            if (e != cudaSuccess) {
                char where[160];
                std::snprintf(where, sizeof where, "%s; tensor-core grid %d block %d smem %d stages %d", g_launch_step,
                              ml.grid, mma_warps(ml.mode, ml.warps) * 32, ml.smem, mp.n_stages);
                return cuda_fail(e, where);
            }
            return QG_OK;
        }
    }
    GemvParams p = {};
    GemvLaunch l = {};
    int st = plan_gemv(type, total, n_in, static_cast<int>(n_vec), dev.sms, dev.smem_optin, &p, &l);
    if (st != QG_OK) return st;
    p.err = dev.err;
    p.n_mats = n;
    cudaError_t e = launch_gemv(type, p, mats, n, static_cast<int>(n_vec), isums, l, dev.device, s);
    if (e != cudaSuccess) {
        char where[160];
        std::snprintf(where, sizeof where, "%s; grid %d block %d smem %d stages %d stage_bytes %d", g_launch_step,
                      l.grid, kGemvThreads, l.smem, p.n_stages, p.stage_bytes);
        return cuda_fail(e, where);
    }
    return QG_OK;
}

// One matrix: activations from xq, or from f32 x quantized in the kernel when
// x is non-null (shared by qgemv, qgemv_xq, qgemv_noalloc and
// qgemv_block_isums).
int run_gemv(int type, const void *W, const void *xq, float *y, int32_t *isums, int64_t n_out, int64_t n_in,
             int64_t n_vec, const DeviceInfo &dev, cudaStream_t s, const float *x = nullptr) {
    GemvMat m = {};
    m.W = static_cast<const uint8_t *>(W);
    m.x = x;
    m.xq = static_cast<const uint8_t *>(xq);
    m.y = y;
    m.isums = isums;
    m.n_out = static_cast<int>(n_out);
    const size_t x_bytes = x ? static_cast<size_t>(4 * n_in * n_vec) : 0;
    return run_gemv_mats(type, &m, 1, n_in, n_vec, x_bytes, isums != nullptr, dev, s);
}

// Validation shared by qgemv_xq and qgemv_block_isums.
int check_gemv_args(int type, const void *W, const void *xq, const void *out, int64_t n_out, int64_t n_in,
                    int64_t n_vec) {
    int st = check_weight_type(type);
    if (st != QG_OK) return st;
    st = check_gemv_shape(type, n_out, n_in, n_vec);
    if (st != QG_OK) return st;
    if (n_out > 0 && (!W || !out)) return QG_ERR_NULL;
    if (n_out > 0 && n_in > 0 && !xq) return QG_ERR_NULL;
    if ((W && !aligned16(W)) || (xq && !aligned16(xq)) || (out && !aligned16(out))) return QG_ERR_ALIGN;
    return QG_OK;
}

}  // namespace
}  // namespace qg

using namespace qg;

extern "C" {

int64_t qtype_nbytes(int type, int64_t n) {
    int elems, bytes;
    if (!block_info(type, &elems, &bytes)) return -1;
    if (n < 0 || n % elems != 0) return -1;
    return n / elems * bytes;
}

int qtype_block(int type, int *elems, int *bytes) {
    int e, b;
    if (!block_info(type, &e, &b)) return QG_ERR_TYPE;
    if (!elems || !bytes) return QG_ERR_NULL;
    *elems = e;
    *bytes = b;
    return QG_OK;
}

int qtype_act_type(int weight_type) {
    switch (weight_type) {
    case QG_Q4_0:
    case QG_Q5_0:
    case QG_Q8_0: return QG_Q8_0;
    case QG_Q4_1: return QG_Q8_1;
    case QG_Q2_K:
    case QG_Q3_K:
    case QG_Q4_K:
    case QG_Q5_K:
    case QG_Q6_K: return QG_Q8_K;
    default: return QG_ERR_PAIR;
    }
}

const char *qg_status_string(int status) {
    switch (status) {
    case QG_OK: return "ok";
    case QG_ERR_TYPE: return "unknown or unsupported type";
    case QG_ERR_SHAPE: return "bad shape (not whole blocks, or a size out of range)";
    case QG_ERR_ALIGN: return "device pointer not 16-byte aligned";
    case QG_ERR_NULL: return "required pointer is NULL";
    case QG_ERR_PAIR: return "weight type has no activation pairing";
    case QG_ERR_CUDA: return "CUDA error";
    case QG_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

const char *qg_last_cuda_error(void) { return g_last_cuda_error; }

int qg_tune(const char *name, int value, int *previous) {
    if (!name) return QG_ERR_NULL;
    for (int k = 0; k < kKnobCount; ++k) {
        if (std::strcmp(name, kKnobs[k].name) != 0) continue;
        const int old = knob(static_cast<KnobId>(k));
        const int v = value < kKnobs[k].lo ? kKnobs[k].lo : (value > kKnobs[k].hi ? kKnobs[k].hi : value);
        g_knob_val[k].store(v + 1, std::memory_order_relaxed);
        if (previous) *previous = old;
        return QG_OK;
    }
    return QG_ERR_TYPE;
}

int quantize_act(int act_type, const float *x, void *xq, int64_t n_in, int64_t n_vec, qg_stream_t stream) {
    int elems, bytes;
    if (!block_info(act_type, &elems, &bytes)) return QG_ERR_TYPE;
    if (act_type != QG_Q8_0 && act_type != QG_Q8_1 && act_type != QG_Q8_K) return QG_ERR_TYPE;
    if (n_in < 0 || n_vec < 0 || n_in % elems != 0) return QG_ERR_SHAPE;
    const int64_t n_blocks = n_in / elems * n_vec;
    if (n_blocks == 0) return QG_OK;
    if (!x || !xq) return QG_ERR_NULL;
    if (!aligned16(x) || !aligned16(xq)) return QG_ERR_ALIGN;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st != QG_OK) return st;
    return launch_quantize(act_type, x, xq, n_blocks, dev.sms, reinterpret_cast<cudaStream_t>(stream));
}

int quantize_rows(int type, const float *x, void *out, int64_t n_rows, int64_t n_in, qg_stream_t stream) {
    int elems, bytes;
    if (!block_info(type, &elems, &bytes)) return QG_ERR_TYPE;
    if (type != QG_Q8_0 && type != QG_Q4_0 && type != QG_Q4_1 && type != QG_Q5_0) return QG_ERR_TYPE;
    if (n_in < 0 || n_rows < 0 || n_in % elems != 0) return QG_ERR_SHAPE;
    const int64_t n_blocks = n_in / elems * n_rows;
    if (n_blocks == 0) return QG_OK;
    if (!x || !out) return QG_ERR_NULL;
    if (!aligned16(x) || !aligned16(out)) return QG_ERR_ALIGN;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st != QG_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = launch_quantize(type, x, out, n_blocks, dev.sms, s);
    if (st != QG_OK) return st;
    // the products read W before waiting for the kernel ahead of them: end
    // with a kernel that starts only after the weights are complete
    stream_order_kernel<<<1, 32, 0, s>>>();
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e, "stream-order launch");
}

int dequantize_rows(int type, const void *W, float *out, int64_t n_rows, int64_t n_in, qg_stream_t stream) {
    int elems, bytes;
    if (!block_info(type, &elems, &bytes)) return QG_ERR_TYPE;
    if (type == QG_F32 || type == QG_F16) return QG_ERR_TYPE;
    if (n_in < 0 || n_rows < 0 || n_in % elems != 0) return QG_ERR_SHAPE;
    const int64_t groups = n_in / 8 * n_rows;
    if (groups == 0) return QG_OK;
    if (!W || !out) return QG_ERR_NULL;
    if (!aligned16(W) || !aligned16(out)) return QG_ERR_ALIGN;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st != QG_OK) return st;
    const int threads = 256;
    int64_t grid = (groups + threads - 1) / threads;
    // 32 CTAs of 256 threads per SM (two waves of resident CTAs; measured
    // faster than 16 for the write-bound Q4_K 4096 x 4096 case)
    if (grid > static_cast<int64_t>(dev.sms) * 32) grid = static_cast<int64_t>(dev.sms) * 32;
    const uint8_t *w = static_cast<const uint8_t *>(W);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const unsigned g = static_cast<unsigned>(grid);
    cudaError_t e = launch_dequant(type, w, out, groups, g, threads, s);
    return e == cudaSuccess ? QG_OK : cuda_fail(e, "dequantize launch");
}

size_t qgemv_workspace_bytes(int type, int64_t n_in, int64_t n_vec) {
    if (check_weight_type(type) != QG_OK) return 0;
    if (check_gemv_shape(type, 0, n_in, n_vec) != QG_OK) return 0;
    const int64_t nb = qtype_nbytes(qtype_act_type(type), n_in);
    return nb < 0 ? 0 : static_cast<size_t>(nb * n_vec);
}

int qgemv_xq(int type, const void *W, const void *xq, float *y, int64_t n_out, int64_t n_in, int64_t n_vec,
             qg_stream_t stream) {
    int st = check_gemv_args(type, W, xq, y, n_out, n_in, n_vec);
    if (st != QG_OK) return st;
    if (n_out == 0) return QG_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n_in == 0) {  // the empty sum
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(n_out * n_vec) * sizeof(float), s);
        return e == cudaSuccess ? QG_OK : cuda_fail(e);
    }
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != QG_OK) return st;
    return run_gemv(type, W, xq, y, nullptr, n_out, n_in, n_vec, dev, s);
}

int qgemv_block_isums(int type, const void *W, const void *xq, int32_t *isums, int64_t n_out, int64_t n_in,
                      int64_t n_vec, qg_stream_t stream) {
    int st = check_gemv_args(type, W, xq, isums, n_out, n_in, n_vec);
    if (st != QG_OK) return st;
    if (n_out == 0 || n_in == 0) return QG_OK;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != QG_OK) return st;
    return run_gemv(type, W, xq, nullptr, isums, n_out, n_in, n_vec, dev,
                    reinterpret_cast<cudaStream_t>(stream));
}

int qgemv(int type, const void *W, const float *x, float *y, int64_t n_out, int64_t n_in, int64_t n_vec,
          void *workspace, size_t workspace_bytes, qg_stream_t stream) {
    int st = check_gemv_args(type, W, x, y, n_out, n_in, n_vec);
    if (st != QG_OK) return st;
    if (n_out == 0) return QG_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n_in == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(n_out * n_vec) * sizeof(float), s);
        return e == cudaSuccess ? QG_OK : cuda_fail(e);
    }
    const size_t need = qgemv_workspace_bytes(type, n_in, n_vec);
    if (!workspace || workspace_bytes < need) return QG_ERR_WORKSPACE;
    if (!aligned16(workspace)) return QG_ERR_ALIGN;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != QG_OK) return st;
    // the product's shape limits are checked before anything is enqueued
    GemvParams probe = {};
    GemvLaunch pl = {};
    const bool fused = fused_single(type, n_out, n_in, n_vec);
    st = plan_gemv(type, n_out, n_in, static_cast<int>(n_vec), dev.sms, dev.smem_optin, &probe, &pl);
    if (st != QG_OK) return st;
    if (fused)  // one launch: x quantized in the GEMV's prologue
        return run_gemv(type, W, nullptr, y, nullptr, n_out, n_in, n_vec, dev, s, x);
    const int at = qtype_act_type(type);
    int elems, bytes;
    if (!block_info(at, &elems, &bytes)) return QG_ERR_PAIR;
    st = launch_quantize(at, x, workspace, n_in / elems * n_vec, dev.sms, s);
    if (st != QG_OK) return st;
    return run_gemv(type, W, workspace, y, nullptr, n_out, n_in, n_vec, dev, s);
}

size_t qgemv_batched_workspace_bytes(int type, int64_t n_in, int64_t n_vec, int n_mats) {
    if (n_mats < 1 || n_mats > QG_MAX_BATCH) return 0;
    const size_t one = qgemv_workspace_bytes(type, n_in, n_vec);
    if (one == 0) return 0;
    return fused_quantization(n_in, n_vec) && !mma_preferred(type, n_vec) ? 16 : one * static_cast<size_t>(n_mats);
}

int qgemv_batched(int type, const qg_gemv_mat *mats, int n_mats, int64_t n_in, int64_t n_vec, void *workspace,
                  size_t workspace_bytes, qg_stream_t stream) {
    int st = check_weight_type(type);
    if (st != QG_OK) return st;
    if (!mats) return QG_ERR_NULL;
    if (n_mats < 1 || n_mats > QG_MAX_BATCH) return QG_ERR_SHAPE;
    for (int i = 0; i < n_mats; ++i) {
        st = check_gemv_args(type, mats[i].W, mats[i].x, mats[i].y, mats[i].n_out, n_in, n_vec);
        if (st != QG_OK) return st;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n_in == 0) {
        for (int i = 0; i < n_mats; ++i) {
            if (mats[i].n_out == 0) continue;
            cudaError_t e = cudaMemsetAsync(mats[i].y, 0, static_cast<size_t>(mats[i].n_out * n_vec) * sizeof(float), s);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
        }
        return QG_OK;
    }
    const bool fused = fused_quantization(n_in, n_vec) && !mma_preferred(type, n_vec);
    const size_t need = qgemv_batched_workspace_bytes(type, n_in, n_vec, n_mats);
    if (!fused && (!workspace || workspace_bytes < need)) return QG_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return QG_ERR_ALIGN;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != QG_OK) return st;
    int64_t total = 0;
    for (int i = 0; i < n_mats; ++i) total += mats[i].n_out;
    if (total == 0) return QG_OK;
    GemvParams probe = {};
    GemvLaunch pl = {};
    st = plan_gemv(type, total, n_in, static_cast<int>(n_vec), dev.sms, dev.smem_optin, &probe, &pl);
    if (st != QG_OK) return st;
    GemvMat gm[QG_MAX_BATCH];
    const int at = qtype_act_type(type);
    int elems, bytes;
    if (!block_info(at, &elems, &bytes)) return QG_ERR_PAIR;
    const int64_t blocks_per_mat = n_in / elems * n_vec;
    if (!fused) {
        QuantTable t = {};
        for (int i = 0; i < n_mats; ++i) t.x[i] = mats[i].x;
        st = launch_quantize_batched(at, t, n_mats, workspace, blocks_per_mat, dev.sms, s);
        if (st != QG_OK) return st;
    }
    for (int i = 0; i < n_mats; ++i) {
        gm[i] = GemvMat{};
        gm[i].W = static_cast<const uint8_t *>(mats[i].W);
        gm[i].x = fused ? mats[i].x : nullptr;
        gm[i].xq = fused ? nullptr : static_cast<const uint8_t *>(workspace) + i * blocks_per_mat * bytes;
        gm[i].y = mats[i].y;
        gm[i].n_out = static_cast<int>(mats[i].n_out);
    }
    return run_gemv_mats(type, gm, n_mats, n_in, n_vec, fused ? static_cast<size_t>(4 * n_in * n_vec) : 0, false,
                         dev, s);
}

size_t qgemm_workspace_bytes(int type, int64_t n_out, int64_t n_in, int64_t n_tok) {
    if (check_weight_type(type) != QG_OK) return 0;
    int elems, bytes;
    if (!block_info(type, &elems, &bytes)) return 0;
    if (n_out < 0 || n_in < 0 || n_tok < 0 || n_out > INT32_MAX || n_tok > INT32_MAX || n_in % elems != 0) return 0;
    const size_t a = (static_cast<size_t>(2 * n_out * n_in) + 255) & ~size_t(255);
    const size_t b = (static_cast<size_t>(2 * n_tok * n_in) + 255) & ~size_t(255);
    return a + b > 0 ? a + b : 16;
}

// Whether qgemm routes Q4_K weights to the fused GEMM (QG_FUSED_GEMM).
bool fused_gemm(int type, int64_t n_out, int64_t n_tok, int sms) {
    if (type != QG_Q4_K) return false;
    const int fuse = knob(kKnobFusedGemm);
    return fuse == 1 || (fuse == 2 && ((n_out + 127) / 128) * ((n_tok + 255) / 256) <= 2 * static_cast<int64_t>(sms));
}

int qgemm(int type, const void *W, const float *x, float *y, int64_t n_out, int64_t n_in, int64_t n_tok,
          void *workspace, size_t workspace_bytes, qg_stream_t stream) {
    int st = check_weight_type(type);
    if (st != QG_OK) return st;
    int elems, bytes;
    if (!block_info(type, &elems, &bytes)) return QG_ERR_TYPE;
    if (n_out < 0 || n_in < 0 || n_tok < 0 || n_out > INT32_MAX || n_tok > INT32_MAX || n_in % elems != 0 ||
        n_in > INT32_MAX)
        return QG_ERR_SHAPE;
    if (n_out == 0 || n_tok == 0) return QG_OK;
    if (!y) return QG_ERR_NULL;
    if (!aligned16(y)) return QG_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n_in == 0) {  // the empty sum
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(n_out * n_tok) * sizeof(float), s);
        return e == cudaSuccess ? QG_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (!W || !x || !workspace) return QG_ERR_NULL;
    if (!aligned16(W) || !aligned16(x) || !aligned16(workspace)) return QG_ERR_ALIGN;
    if (workspace_bytes < qgemm_workspace_bytes(type, n_out, n_in, n_tok)) return QG_ERR_WORKSPACE;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != QG_OK) return st;
    __half *A = static_cast<__half *>(workspace);
    __half *B = reinterpret_cast<__half *>(static_cast<uint8_t *>(workspace) +
                                           ((static_cast<size_t>(2 * n_out * n_in) + 255) & ~size_t(255)));
    if (fused_gemm(type, n_out, n_tok, dev.sms)) {
        // W is dequantized inside the GEMM (into tensor memory): only x is converted first.
        // With few tiles the GEMM splits k; the workspace's f16-weight part, unused
        // here, holds the partial products of the parts after the first.
        const GemmPlan plan = gemm_q4k_tmem_plan(n_out, n_tok, n_in, dev.sms, knob(kKnobGemmKsplit),
                                                 static_cast<size_t>(2 * n_out * n_in));
        cudaError_t e = launch_f32_to_f16(x, B, n_tok * n_in, dev.sms, s);
        if (e != cudaSuccess) return cuda_fail(e, "prefill: x to f16");
        e = launch_gemm_q4k_tmem(static_cast<const uint8_t *>(W), B, y, n_out, n_tok, n_in, plan,
                                 reinterpret_cast<float *>(A), dev.err, dev.sms, dev.device, s);
        if (e != cudaSuccess) return cuda_fail(e, g_launch_step);
        return QG_OK;
    }
    const int64_t groups = n_out * n_in / 8;
    int64_t grid = (groups + 255) / 256;
    if (grid > static_cast<int64_t>(dev.sms) * 32) grid = static_cast<int64_t>(dev.sms) * 32;
    cudaError_t e = launch_dequant(type, static_cast<const uint8_t *>(W), A, groups, static_cast<unsigned>(grid), 256, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill: dequantize to f16");
    e = launch_f32_to_f16(x, B, n_tok * n_in, dev.sms, s);
    if (e != cudaSuccess) return cuda_fail(e, "prefill: x to f16");
    e = launch_gemm_f16_tc(A, B, y, n_out, n_tok, n_in, dev.err, dev.sms, dev.device, s);
    if (e != cudaSuccess) return cuda_fail(e, g_launch_step);
    return QG_OK;
}

int qgemm_f16(const void *A, const void *B, float *y, int64_t n_out, int64_t n_tok, int64_t K, qg_stream_t stream) {
    if (n_out < 0 || n_tok < 0 || K < 0 || n_out > INT32_MAX || n_tok > INT32_MAX || K > INT32_MAX || K % 8 != 0)
        return QG_ERR_SHAPE;
    if (n_out == 0 || n_tok == 0) return QG_OK;
    if (!y) return QG_ERR_NULL;
    if (!aligned16(y)) return QG_ERR_ALIGN;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(n_out * n_tok) * sizeof(float), s);
        return e == cudaSuccess ? QG_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    if (!A || !B) return QG_ERR_NULL;
    if (!aligned16(A) || !aligned16(B)) return QG_ERR_ALIGN;
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st != QG_OK) return st;
    cudaError_t e = launch_gemm_f16_tc(static_cast<const __half *>(A), static_cast<const __half *>(B), y, n_out, n_tok, K,
                                       dev.err, dev.sms, dev.device, s);
    return e == cudaSuccess ? QG_OK : cuda_fail(e, g_launch_step);
}

const char *qgemv_kernel_info(int type, int64_t total_rows, int64_t n_in, int64_t n_vec, int n_mats) {
    static thread_local char buf[320];  // room for "cuda: " and a whole CUDA error string
    buf[0] = 0;
    if (check_weight_type(type) != QG_OK || check_gemv_shape(type, total_rows, n_in, n_vec) != QG_OK) return buf;
    if (n_mats < 1 || n_mats > QG_MAX_BATCH || total_rows < 1 || n_in < 1) return buf;
    DeviceInfo dev;
    if (current_device(&dev) != QG_OK) {
        std::snprintf(buf, sizeof buf, "cuda: %s", g_last_cuda_error);
        return buf;
    }
    const char *tn = type == QG_Q4_K ? "Q4_K" : type == QG_Q6_K ? "Q6_K" : type == QG_Q8_0 ? "Q8_0"
                   : type == QG_Q4_1 ? "Q4_1" : type == QG_Q5_0 ? "Q5_0" : type == QG_Q2_K ? "Q2_K"
                   : type == QG_Q3_K ? "Q3_K" : type == QG_Q5_K ? "Q5_K" : "Q4_0";
    if (mma_wins(type, n_vec, total_rows / n_mats, n_in)) {
        // tiles: a batch of equal matrices is assumed for the tile count
        const int64_t per = total_rows / n_mats;
        TcParams tp = {};
        int tgrid = 0, tsmem = 0;
        if (plan_gemv_tc(type, n_mats * ((per + kTcRows - 1) / kTcRows), n_in, static_cast<int>(n_vec), n_mats,
                         dev.sms, dev.smem_optin, &tp, &tgrid, &tsmem)) {
            std::snprintf(buf, sizeof buf, "gemv_tc_kernel<%s,tcgen05> grid=%d stages=%d tile_rows=%d smem=%d", tn,
                          tgrid, tp.n_stages, kTcRows, tsmem);
            return buf;
        }
        const int64_t tiles = n_mats * ((per + kMmaTileRows - 1) / kMmaTileRows);
        MmaParams mp = {};
        MmaLaunch ml = {};
        if (plan_gemv_mma(type, tiles, n_in, static_cast<int>(n_vec), dev.sms, dev.smem_optin, &mp, &ml) == QG_OK) {
            const char *mode = ml.mode == kMmaRegs ? "regs" : ml.mode == kMmaPanel16 ? "panel16" : "panel8";
            std::snprintf(buf, sizeof buf, "gemv_mma_kernel<%s,%s,%dw> grid=%d stages=%d kb=%d smem=%d partials=%d", tn,
                          mode, ml.warps, ml.grid, mp.n_stages, mp.kb, ml.smem, mp.red_slots);
            return buf;
        }
    }
    const bool fused = n_mats == 1 ? fused_single(type, total_rows, n_in, n_vec)
                                   : fused_quantization(n_in, n_vec) && !mma_preferred(type, n_vec);
    GemvParams gp = {};
    GemvLaunch gl = {};
    if (plan_gemv(type, total_rows, n_in, static_cast<int>(n_vec), dev.sms, dev.smem_optin, &gp, &gl) != QG_OK)
        return buf;
    std::snprintf(buf, sizeof buf, "gemv_kernel<%s,NV=%d> grid=%d stages=%d split=%d rows_per_stage=%d lanes_per_block=%d smem=%d%s",
                  tn, static_cast<int>(n_vec), gl.grid, gp.n_stages, gp.split, gp.rows_per_stage, gl.lpb, gl.smem,
                  fused ? " fused-quantize" : "");
    return buf;
}

const char *qgemm_kernel_info(int type, int64_t n_out, int64_t n_in, int64_t n_tok) {
    static thread_local char buf[320];
    buf[0] = 0;
    int elems, bytes;
    if (check_weight_type(type) != QG_OK || !block_info(type, &elems, &bytes)) return buf;
    if (n_out < 1 || n_tok < 1 || n_in < 1 || n_out > INT32_MAX || n_tok > INT32_MAX || n_in > INT32_MAX ||
        n_in % elems != 0)
        return buf;
    DeviceInfo dev;
    if (current_device(&dev) != QG_OK) {
        std::snprintf(buf, sizeof buf, "cuda: %s", g_last_cuda_error);
        return buf;
    }
    if (fused_gemm(type, n_out, n_tok, dev.sms)) {
        const GemmPlan p = gemm_q4k_tmem_plan(n_out, n_tok, n_in, dev.sms, knob(kKnobGemmKsplit),
                                              static_cast<size_t>(2 * n_out * n_in));
        const int64_t items = ((n_out + 127) / 128) * ((n_tok + p.bn - 1) / p.bn) * p.ks;
        std::snprintf(buf, sizeof buf, "gemm_q4k_tmem_kernel<%d> grid=%d ksplit=%d launches=%d", p.bn,
                      static_cast<int>(std::min<int64_t>(items, dev.sms)), p.ks, p.ks > 1 ? 3 : 2);
        return buf;
    }
    const GemmPlan p = gemm_f16_plan(n_out, n_tok, n_in, dev.sms);
    const int64_t tiles = ((n_out + 127) / 128) * ((n_tok + p.bn - 1) / p.bn);
    std::snprintf(buf, sizeof buf, "gemm_f16_tc_kernel<%d> grid=%d ksplit=1 launches=3", p.bn,
                  static_cast<int>(std::min<int64_t>(tiles, dev.sms)));
    return buf;
}

int qg_device_error(int32_t *code) {
    if (!code) return QG_ERR_NULL;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    int32_t v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
    if (e != cudaSuccess) return cuda_fail(e);
    const int32_t zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_fail(e);
    *code = v;
    return QG_OK;
}

int qg_selftest_bounded_wait(qg_stream_t stream) {
    DeviceInfo dev;
    int st = current_device(&dev);
    if (st != QG_OK) return st;
    selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(dev.err);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? QG_OK : cuda_fail(e, "self-test launch");
}

}  // extern "C"

// ---------------------------------------------------------------------------
// qgemv_noalloc: qgemv for callers that cannot hand the library a workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// product: a plugin or custom operator whose host framework owns every device
// buffer and gives it none; a decode loop that must not call cudaMalloc or
// cudaFree, because those calls can synchronize the whole device and stall
// other streams; code being recorded by CUDA stream capture, where
// allocation calls are not allowed. This entry point keeps the quantized
// activations in a fixed array in the library's own device memory instead.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes bytes;
// every GPU that loads this library holds it until the process exits. In
// host code its name is only a host-side handle, not a device address, so
// the first call on each device (with that device current) asks the runtime
// for the device address with cudaGetSymbolAddress and keeps it; later
// calls on that device reuse it.
// ---------------------------------------------------------------------------
namespace qg {
namespace {

constexpr size_t kNoAllocScratchBytes = 256 * 1024;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device.
int noalloc_scratch(int device, void **out) {
    static void *addr[64] = {nullptr};
    void *p = (device >= 0 && device < 64) ? __atomic_load_n(&addr[device], __ATOMIC_ACQUIRE) : nullptr;
    if (!p) {
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(g_noalloc_scratch)");
        if (device >= 0 && device < 64) __atomic_store_n(&addr[device], p, __ATOMIC_RELEASE);
    }
    *out = p;
    return QG_OK;
}

}  // namespace
}  // namespace qg

extern "C" int qgemv_noalloc(int type, const void *W, const float *x, float *y, int64_t n_out, int64_t n_in,
                             int64_t n_vec, qg_stream_t stream) {
    int st = check_gemv_args(type, W, x, y, n_out, n_in, n_vec);
    if (st != QG_OK) return st;
    if (n_out == 0) return QG_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n_in == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(n_out * n_vec) * sizeof(float), s);
        return e == cudaSuccess ? QG_OK : cuda_fail(e, "cudaMemsetAsync");
    }
    // the quantized activations must fit in the fixed array
    if (qgemv_workspace_bytes(type, n_in, n_vec) > kNoAllocScratchBytes) return QG_ERR_WORKSPACE;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != QG_OK) return st;
    GemvParams probe = {};
    GemvLaunch pl = {};
    st = plan_gemv(type, n_out, n_in, static_cast<int>(n_vec), dev.sms, dev.smem_optin, &probe, &pl);
    if (st != QG_OK) return st;
    // where qgemv quantizes x inside the product it needs no memory at all:
    // the same single launch, and the array is not touched
    if (fused_single(type, n_out, n_in, n_vec))
        return run_gemv(type, W, nullptr, y, nullptr, n_out, n_in, n_vec, dev, s, x);
    void *scratch = nullptr;
    st = noalloc_scratch(dev.device, &scratch);
    if (st != QG_OK) return st;
    // Every byte the product reads from the array is written by the
    // quantization launched just before it, so nothing needs clearing.
    const int at = qtype_act_type(type);
    int elems, bytes;
    if (!block_info(at, &elems, &bytes)) return QG_ERR_PAIR;
    st = launch_quantize(at, x, scratch, n_in / elems * n_vec, dev.sms, s);
    if (st != QG_OK) return st;
    return run_gemv(type, W, scratch, y, nullptr, n_out, n_in, n_vec, dev, s);
}
