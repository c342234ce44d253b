// gemv_q6_k.cu - template instances of the streaming GEMV kernel for Q6_K
// weights with the two-lanes-per-block item (n_vec = 1..8; single matrix with
// product or exact-block-sum output, batches of up to kMaxBatch matrices with
// product output); plans that chose the four-lane item go to gemv_q6_k4.cu.
#include "gemv_launch.cuh"

namespace qg {

cudaError_t launch_gemv_q6_k(const GemvParams &p, const GemvMat *mats, int n, int nv, bool isums, const GemvLaunch &l,
                             int device, cudaStream_t s) {
    if (l.lpb == TypeQ6_K4::kLanesPerBlock) return launch_gemv_q6_k4(p, mats, n, nv, isums, l, device, s);
    return launch_gemv_type<TypeQ6_K>(p, mats, n, nv, isums, l, device, s);
}

}  // namespace qg
