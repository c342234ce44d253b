// gemv_q4_k.cu - template instances of the streaming GEMV kernel for Q4_K
// weights (n_vec = 1..8, product and exact-block-sum outputs).
#include "gemv_launch.cuh"

namespace qg {

cudaError_t launch_gemv_q4_k(const GemvParams &p, int nv, bool isums, const GemvLaunch &l, int device,
                             cudaStream_t s) {
    return launch_gemv_type<TypeQ4_K>(p, nv, isums, l, device, s);
}

}  // namespace qg
