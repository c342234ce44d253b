// gemv_mma_q8_0.cu - template instances of the tensor-core GEMV for Q8_0
// weights in groups of eight blocks (activation fragments from an f16 /
// biased-int8 shared-memory panel with 16 consumer warps; one matrix or a
// batch).
#include "gemv_mma_launch.cuh"

namespace qg {

cudaError_t launch_gemv_mma_q8_0(const MmaParams &p, const MmaMat *mats, int n, const MmaLaunch &l, int device,
                                 cudaStream_t s) {
    return mma_launch_type<MmaQ8_0>(p, mats, n, l, device, s);
}

}  // namespace qg
