// gemv_mma_launch.cuh - host-side launch of the tensor-core GEMV for one
// weight type: picks the instance for the activation-source mode, the number
// of consumer warps and the table size, raises its shared-memory limit once
// per device and launches it with programmatic dependent launch enabled.
#pragma once

#include <atomic>

#include "gemv_mma.cuh"

namespace qg {

constexpr int kMmaMaxBatch = 256;

template <class T, int BM, int NW, int MAXB, class K>
inline cudaError_t mma_smem_attr(K kernel, int device, int bytes) {
    static std::atomic<uint64_t> done{0};
    const uint64_t bit = 1ull << (device & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    g_launch_step = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)";
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

template <class T, int BM, int NW, int MAXB>
inline cudaError_t mma_launch_inst(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                   cudaStream_t s) {
    MmaBatch<MAXB> b = {};
    for (int i = 0; i < n; ++i) b.m[i] = mats[i];
    auto k = gemv_mma_kernel<T, BM, NW, MAXB>;
    cudaError_t e = mma_smem_attr<T, BM, NW, MAXB>(k, device, l.smem_optin);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, l.grid, mma_warps(BM, NW) * 32, l.smem, s, p, b);
}

template <class T, int BM, int NW>
inline cudaError_t mma_launch_mode(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                   cudaStream_t s) {
    if (n == 1) return mma_launch_inst<T, BM, NW, 1>(p, mats, n, l, device, s);
    if (n > kMmaMaxBatch) return cudaErrorInvalidValue;
    return mma_launch_inst<T, BM, NW, kMmaMaxBatch>(p, mats, n, l, device, s);
}

template <class T>
inline cudaError_t mma_launch_type(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                   cudaStream_t s) {
    switch (l.mode) {
    case kMmaRegs:
        // activation fragments in registers: Q8_K-paired types only
        if constexpr (T::kActBytes != 0) return cudaErrorInvalidValue;
        else return l.warps == 8 ? mma_launch_mode<T, kMmaRegs, 8>(p, mats, n, l, device, s) : cudaErrorInvalidValue;
    case kMmaPanel16:
        return l.warps == 16 ? mma_launch_mode<T, kMmaPanel16, 16>(p, mats, n, l, device, s) : cudaErrorInvalidValue;
    case kMmaPanel8:
        return l.warps == 16 ? mma_launch_mode<T, kMmaPanel8, 16>(p, mats, n, l, device, s) : cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
    }
}

// One definition per weight type, each in its own translation unit.
cudaError_t launch_gemv_mma_q4_k(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s);
cudaError_t launch_gemv_mma_q4_0(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s);
cudaError_t launch_gemv_mma_q4_1(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s);
cudaError_t launch_gemv_mma_q5_0(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s);
cudaError_t launch_gemv_mma_q8_0(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s);
cudaError_t launch_gemv_mma_q2_k(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s);
cudaError_t launch_gemv_mma_q3_k(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s);
cudaError_t launch_gemv_mma_q5_k(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s);
cudaError_t launch_gemv_mma_q6_k(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s);

inline cudaError_t launch_gemv_mma(int type, const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l,
                                   int device, cudaStream_t s) {
    switch (type) {
    case QG_Q4_0: return launch_gemv_mma_q4_0(p, mats, n, l, device, s);
    case QG_Q4_1: return launch_gemv_mma_q4_1(p, mats, n, l, device, s);
    case QG_Q5_0: return launch_gemv_mma_q5_0(p, mats, n, l, device, s);
    case QG_Q8_0: return launch_gemv_mma_q8_0(p, mats, n, l, device, s);
    case QG_Q2_K: return launch_gemv_mma_q2_k(p, mats, n, l, device, s);
    case QG_Q3_K: return launch_gemv_mma_q3_k(p, mats, n, l, device, s);
    case QG_Q4_K: return launch_gemv_mma_q4_k(p, mats, n, l, device, s);
    case QG_Q5_K: return launch_gemv_mma_q5_k(p, mats, n, l, device, s);
    case QG_Q6_K: return launch_gemv_mma_q6_k(p, mats, n, l, device, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qg
