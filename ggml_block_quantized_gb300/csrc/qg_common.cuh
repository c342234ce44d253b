// qg_common.cuh - device helpers shared by the kernels of the GB300
// block-quantized GEMV library: inline PTX for mbarriers, 1-D bulk async
// copies (the TMA engine's non-tensor mode), programmatic dependent launch,
// bounded waits and unaligned shared-memory word reads.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "qgemv.h"  // include/ is on the include path

namespace qg {

// ---------------------------------------------------------------- limits
constexpr int kMaxNvec = QG_MAX_NVEC;
constexpr int kQuantTableMax = 256;  // matrices per batched quantization launch

// Activation pointers of a batched quantization launch (a kernel parameter).
struct QuantTable {
    const float *x[kQuantTableMax];
};
constexpr int kSmemLimit = 227 * 1024;  // opt-in dynamic shared memory per CTA

// Device-side error word: 0 = fine; the first failing wait records its code.
enum DeviceError : int32_t {
    kErrNone = 0,
    kErrProducerWait = 1,  // producer gave up waiting for a free stage
    kErrConsumerWait = 2,  // consumer gave up waiting for a filled stage
    kErrDrainWait = 3,     // producer gave up waiting for its copies at exit
};

// The word lives in api.cu; kernels receive its address as a parameter.
__device__ __forceinline__ void record_error(int32_t *err, int32_t code) {
    atomicCAS(err, 0, code);
}

// ----------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that lets the hardware suspend the thread until the phase
// completes or about `hint_ns` pass, instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity, giving up after about
// one second (the clock is read every 16 polls) or 2^26 polls. Each poll may
// suspend the thread until the phase completes (at most 20 us). Returns
// false on timeout; the caller records the error and winds down.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kWaitLimitPolls = 1u << 26;

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1; i < kWaitLimitPolls; ++i) {
        if (mbar_try_wait_hint(bar, parity, 20000u)) return true;
        if ((i & 15u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return false;
}

// One bulk copy global -> shared (TMA engine, non-tensor form). Both
// addresses 16-byte aligned, bytes a multiple of 16. Completion is reported
// to `bar` as transaction bytes.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// The same copy with the default L2 policy.
__device__ __forceinline__ void bulk_copy_g2s_plain(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// L2 policy: weights are streamed once, so let them be evicted first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch (PDL).
__device__ __forceinline__ void pdl_wait_prior_grids() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier among `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------ shared-memory word reads
// Loads from 32-bit shared-memory addresses (no generic-address arithmetic).
__device__ __forceinline__ uint32_t ld_s32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t ld_s16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint2 ld_s64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 ld_s128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

// N consecutive 32-bit words starting at a 2-byte-aligned shared address.
template <int N>
__device__ __forceinline__ void ld_words_a2(uint32_t a, uint32_t (&out)[N]) {
    const uint32_t base = a & ~3u;
    const uint32_t sh = (a & 3u) * 8u;  // 0 or 16
    uint32_t raw[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) raw[i] = ld_s32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

// Four bytes starting at a 2-byte-aligned shared-memory address.
__device__ __forceinline__ uint32_t lds_u32_a2(const uint8_t *p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;  // 0 or 16
    return __funnelshift_r(w[0], w[1], sh);
}

// N consecutive 32-bit words starting at a 2-byte-aligned address.
template <int N>
__device__ __forceinline__ void lds_words_a2(const uint8_t *p, uint32_t (&out)[N]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
    uint32_t raw[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) raw[i] = w[i];
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(raw[i], raw[i + 1], sh);
}

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits & 0xFFFFu)));
}

__device__ __forceinline__ uint16_t lds_u16(const uint8_t *p) {
    return *reinterpret_cast<const uint16_t *>(p);
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// Unsigned bytes of a times signed bytes of b, summed into c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two signed 16-bit halves of a times bytes 0,1 (lo) or 2,3 (hi) of b.
__device__ __forceinline__ int dp2a_lo_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_lo_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp2a_hi_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Packed two-lane f32 arithmetic (one instruction for both lanes).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 ra, ra, rb, rc;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 ra, ra, rb;\n\tmov.b64 {%0, %1}, ra;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Sign-extend byte k of w.
__device__ __forceinline__ int sbyte(uint32_t w, int k) {
    return static_cast<int>(static_cast<int8_t>((w >> (8 * k)) & 0xFFu));
}

// roundf result -> code: NaN gives 0, values saturate to [lo, hi]
// (the special-value behaviour printed by candle's "一些边界值" table).
__device__ __forceinline__ int code_from_rounded(float r, int lo, int hi) {
    if (r != r) return 0;
    r = fminf(fmaxf(r, static_cast<float>(lo)), static_cast<float>(hi));
    return static_cast<int>(r);
}

// Which CUDA call of a launch failed (for the error text).
inline thread_local const char *g_launch_step = "";

// Launch with programmatic dependent launch enabled: the kernel may start
// while the previous kernel on the stream finishes; it orders itself with
// griddepcontrol.wait before touching anything that kernel may write.
template <class K, class... Args>
inline cudaError_t launch_pdl(K kernel, int grid, int block, int smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    g_launch_step = "cudaLaunchKernelEx";
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace qg
