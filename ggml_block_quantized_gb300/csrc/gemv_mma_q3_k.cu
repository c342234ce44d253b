// gemv_mma_q3_k.cu - template instances of the tensor-core GEMV for Q3_K
// weights (activation fragments in registers with 8 consumer warps, or from
// an f16 / biased-int8 shared-memory panel with 16; one matrix or a batch).
#include "gemv_mma_launch.cuh"

namespace qg {

cudaError_t launch_gemv_mma_q3_k(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s) {
    return mma_launch_type<MmaQ3_K>(p, mats, n, l, device, s);
}

}  // namespace qg
