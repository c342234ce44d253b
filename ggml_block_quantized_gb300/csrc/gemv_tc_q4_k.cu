// gemv_tc_q4_k.cu - host side of the tcgen05 Q4_K GEMV: the shared-memory
// opt-in and the launch, one matrix or a batch.
#include <atomic>

#include "gemv_tc.cuh"

namespace qg {

namespace {

template <int MAXB>
cudaError_t launch_inst(const TcParams &p, const TcMat *mats, int n, int grid, int smem, int smem_optin, int device,
                        cudaStream_t s) {
    TcBatch<MAXB> b = {};
    for (int i = 0; i < n; ++i) b.m[i] = mats[i];
    auto k = gemv_tc_q4_k_kernel<MAXB>;
    static std::atomic<uint64_t> done{0};
    const uint64_t bit = 1ull << (device & 63);
    if (!(done.load(std::memory_order_acquire) & bit)) {
        g_launch_step = "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)";
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
        if (e != cudaSuccess) return e;
        done.fetch_or(bit, std::memory_order_acq_rel);
    }
    return launch_pdl(k, grid, kTcThreads, smem, s, p, b);
}

}  // namespace

cudaError_t launch_gemv_tc_q4_k(const TcParams &p, const TcMat *mats, int n, int grid, int smem, int smem_optin,
                                int device, cudaStream_t s) {
    if (n < 1 || n > kTcMaxBatch) return cudaErrorInvalidValue;
    if (n == 1) return launch_inst<1>(p, mats, n, grid, smem, smem_optin, device, s);
    return launch_inst<kTcMaxBatch>(p, mats, n, grid, smem, smem_optin, device, s);
}

}  // namespace qg
