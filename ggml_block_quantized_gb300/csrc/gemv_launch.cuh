// gemv_launch.cuh - host-side launch of the streaming GEMV kernel for one
// weight type: picks the template instance for n_vec and the output mode,
// raises its shared-memory limit once per device and launches it with
// programmatic dependent launch enabled.
#pragma once

#include <atomic>

#include "gemv_mma_launch.cuh"
#include "gemv_pipeline.cuh"
#include "gemv_types.cuh"

namespace qg {

struct GemvLaunch {
    int grid;
    int smem;
    int smem_optin;  // the device's opt-in shared-memory limit per CTA
    int sms;         // SMs of the device
    int lpb;         // lanes per weight block of the chosen item (Q6_K: 2 or 4)
};


// Shared-memory opt-in, done once per (kernel, device). The flag is keyed by
// the kernel's template arguments (every instance has the same C++ type).
template <class T, int NV, bool ISUMS, class K>
inline cudaError_t ensure_smem_attr(K kernel, int device, int bytes) {
    static std::atomic<uint64_t> done{0};
    const uint64_t bit = 1ull << (device & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    g_launch_step = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)";
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// CTAs of kernel k that one SM holds with `smem` bytes of shared memory,
// cached per (kernel, device) for the last shared-memory size asked.
template <class T, int NV, bool ISUMS, class K>
inline int resident_ctas(K kernel, int device, int smem) {
    static thread_local int cache_dev = -1, cache_smem = -1, cache_n = 0;
    if (cache_dev == device && cache_smem == smem) return cache_n;
    int n = 0;
    g_launch_step = "cudaOccupancyMaxActiveBlocksPerMultiprocessor";
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kGemvThreads, smem) != cudaSuccess) n = 1;
    cache_dev = device;
    cache_smem = smem;
    cache_n = n < 1 ? 1 : n;
    return cache_n;
}

template <class T, int NV, bool ISUMS, int MAXB>
inline cudaError_t launch_gemv_inst(const GemvParams &p, const GemvBatch<MAXB> &b, const GemvLaunch &l,
                                    int device, cudaStream_t s) {
    auto k = gemv_kernel<T, NV, ISUMS, MAXB>;
    cudaError_t e = ensure_smem_attr<T, NV, ISUMS>(k, device, l.smem_optin);
    if (e != cudaSuccess) return e;
    // never more CTAs than fit at once: every CTA streams a fixed row range
    int grid = l.grid;
    const int cap = resident_ctas<T, NV, ISUMS>(k, device, l.smem) * l.sms;
    if (grid > cap) grid = cap;
    GemvParams q = p;  // the CTAs' row ranges for the final grid
    q.rows_q = p.total_rows / grid;
    q.rows_r = static_cast<int>(p.total_rows % grid);
    return launch_pdl(k, grid, kGemvThreads, l.smem, s, q, b);
}

template <class T, int NV>
inline cudaError_t launch_gemv_nv(const GemvParams &p, const GemvMat *mats, int n, bool isums, const GemvLaunch &l,
                                  int device, cudaStream_t s) {
    if (n == 1) {
        GemvBatch<1> b;
        b.m[0] = mats[0];
        return isums ? launch_gemv_inst<T, NV, true, 1>(p, b, l, device, s)
                     : launch_gemv_inst<T, NV, false, 1>(p, b, l, device, s);
    }
    if (isums || n > kMaxBatch) return cudaErrorInvalidValue;
    GemvBatch<kMaxBatch> b = {};
    for (int i = 0; i < n; ++i) b.m[i] = mats[i];
    return launch_gemv_inst<T, NV, false, kMaxBatch>(p, b, l, device, s);
}

template <class T>
inline cudaError_t launch_gemv_type(const GemvParams &p, const GemvMat *mats, int n, int nv, bool isums,
                                    const GemvLaunch &l, int device, cudaStream_t s) {
    switch (nv) {
    case 1: return launch_gemv_nv<T, 1>(p, mats, n, isums, l, device, s);
    case 2: return launch_gemv_nv<T, 2>(p, mats, n, isums, l, device, s);
    case 3: return launch_gemv_nv<T, 3>(p, mats, n, isums, l, device, s);
    case 4: return launch_gemv_nv<T, 4>(p, mats, n, isums, l, device, s);
    case 5: return launch_gemv_nv<T, 5>(p, mats, n, isums, l, device, s);
    case 6: return launch_gemv_nv<T, 6>(p, mats, n, isums, l, device, s);
    case 7: return launch_gemv_nv<T, 7>(p, mats, n, isums, l, device, s);
    case 8: return launch_gemv_nv<T, 8>(p, mats, n, isums, l, device, s);
    default: return cudaErrorInvalidValue;
    }
}

// One definition per weight type, each in its own translation unit.
#define QG_DECLARE_GEMV_LAUNCH(name)                                                                       \
    cudaError_t name(const GemvParams &p, const GemvMat *mats, int n, int nv, bool isums, const GemvLaunch &l, \
                     int device, cudaStream_t s);
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q8_0)
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q4_0)
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q4_1)
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q5_0)
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q4_k)
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q2_k)
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q3_k)
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q5_k)
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q6_k)
QG_DECLARE_GEMV_LAUNCH(launch_gemv_q6_k4)
#undef QG_DECLARE_GEMV_LAUNCH

}  // namespace qg
