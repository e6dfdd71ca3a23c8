// gemm_umma_tf32.cu -- the tensor-core GEMM instances for TF32 (B read MN-major from B[K, N])
// (every CTA-pair mode, K slices per stage and trace/dynamic mode).
#include "gemm_umma.cuh"

namespace gbr {

void* umma_kernel_tf32(int pair, int ksub, int mode) {
    return umma::select_kernel_kg<kUmmaTf32, false>(pair, ksub, mode);
}

}  // namespace gbr
