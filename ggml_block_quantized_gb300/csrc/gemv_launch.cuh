// gemv_launch.cuh - host-side launch of the streaming GEMV kernel for one
// weight type: picks the template instance for n_vec and the output mode,
// raises its shared-memory limit once per device and launches it with
// programmatic dependent launch enabled.
#pragma once

#include <atomic>

#include "gemv_pipeline.cuh"
#include "gemv_types.cuh"

namespace qg {

struct GemvLaunch {
    int grid;
    int smem;
    int smem_optin;  // the device's opt-in shared-memory limit per CTA
};

// Which CUDA call of a launch failed (for the error text).
inline thread_local const char *g_launch_step = "";

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

template <class T, int NV>
inline cudaError_t launch_gemv_nv(const GemvParams &p, bool isums, const GemvLaunch &l, int device,
                                  cudaStream_t s) {
    if (isums) {
        auto k = gemv_kernel<T, NV, true>;
        cudaError_t e = ensure_smem_attr<T, NV, true>(k, device, l.smem_optin);
        if (e != cudaSuccess) return e;
        return launch_pdl(k, l.grid, kGemvThreads, l.smem, s, p);
    }
    auto k = gemv_kernel<T, NV, false>;
    cudaError_t e = ensure_smem_attr<T, NV, false>(k, device, l.smem_optin);
    if (e != cudaSuccess) return e;
    return launch_pdl(k, l.grid, kGemvThreads, l.smem, s, p);
}

template <class T>
inline cudaError_t launch_gemv_type(const GemvParams &p, int nv, bool isums, const GemvLaunch &l, int device,
                                    cudaStream_t s) {
    switch (nv) {
    case 1: return launch_gemv_nv<T, 1>(p, isums, l, device, s);
    case 2: return launch_gemv_nv<T, 2>(p, isums, l, device, s);
    case 3: return launch_gemv_nv<T, 3>(p, isums, l, device, s);
    case 4: return launch_gemv_nv<T, 4>(p, isums, l, device, s);
    case 5: return launch_gemv_nv<T, 5>(p, isums, l, device, s);
    case 6: return launch_gemv_nv<T, 6>(p, isums, l, device, s);
    case 7: return launch_gemv_nv<T, 7>(p, isums, l, device, s);
    case 8: return launch_gemv_nv<T, 8>(p, isums, l, device, s);
    default: return cudaErrorInvalidValue;
    }
}

// One definition per weight type, each in its own translation unit.
cudaError_t launch_gemv_q8_0(const GemvParams &p, int nv, bool isums, const GemvLaunch &l, int device,
                             cudaStream_t s);
cudaError_t launch_gemv_q4_0(const GemvParams &p, int nv, bool isums, const GemvLaunch &l, int device,
                             cudaStream_t s);
cudaError_t launch_gemv_q4_k(const GemvParams &p, int nv, bool isums, const GemvLaunch &l, int device,
                             cudaStream_t s);
cudaError_t launch_gemv_q6_k(const GemvParams &p, int nv, bool isums, const GemvLaunch &l, int device,
                             cudaStream_t s);

}  // namespace qg
