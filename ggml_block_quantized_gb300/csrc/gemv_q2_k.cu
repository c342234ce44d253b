// gemv_q2_k.cu - template instances of the streaming GEMV kernel for Q2_K
// weights (n_vec = 1..8; single matrix with product or exact-block-sum output, batches
// of up to kMaxBatch matrices with product output).
#include "gemv_launch.cuh"

namespace qg {

cudaError_t launch_gemv_q2_k(const GemvParams &p, const GemvMat *mats, int n, int nv, bool isums, const GemvLaunch &l,
                             int device, cudaStream_t s) {
    return launch_gemv_type<TypeQ2_K>(p, mats, n, nv, isums, l, device, s);
}

}  // namespace qg
