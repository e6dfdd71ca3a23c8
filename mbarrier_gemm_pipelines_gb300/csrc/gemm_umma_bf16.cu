// gemm_umma_bf16.cu -- the tensor-core GEMM instances for bf16 inputs, dense
// (every CTA-pair mode, K slices per stage and trace/dynamic mode).
#include "gemm_umma.cuh"

namespace gbr {

void* umma_kernel_bf16(int pair, int ksub, int mode) {
    return umma::select_kernel_kg<kUmmaBf16, false>(pair, ksub, mode);
}

}  // namespace gbr
