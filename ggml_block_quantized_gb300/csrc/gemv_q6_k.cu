// gemv_q6_k.cu - template instances of the streaming GEMV kernel for Q6_K
// weights (n_vec = 1..8, product and exact-block-sum outputs).
#include "gemv_launch.cuh"

namespace qg {

cudaError_t launch_gemv_q6_k(const GemvParams &p, int nv, bool isums, const GemvLaunch &l, int device,
                             cudaStream_t s) {
    return launch_gemv_type<TypeQ6_K>(p, nv, isums, l, device, s);
}

}  // namespace qg
