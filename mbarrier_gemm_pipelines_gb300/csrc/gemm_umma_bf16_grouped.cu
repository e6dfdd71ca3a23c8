// gemm_umma_bf16_grouped.cu -- the tensor-core GEMM instances for bf16 inputs, grouped (MoE)
// (every CTA-pair mode, K slices per stage and trace/dynamic mode).
#include "gemm_umma.cuh"

namespace gbr {

void* umma_kernel_bf16_grouped(int pair, int ksub, int mode) {
    return umma::select_kernel_kg<kUmmaBf16, true>(pair, ksub, mode);
}

}  // namespace gbr
