// gemm_umma.cu -- host side of the tensor-core GEMM (gemm_umma.cuh): shared
// memory sizes, per-device function attributes, the register-split check and
// the launches.  The kernels themselves are instantiated in gemm_umma_*.cu.
#include "gemm_umma.cuh"

namespace gbr {

namespace {

using umma::kThreads;
using umma::kRegsWG0;
using umma::kRegsWG1;
using umma::Pair;
using umma::UmmaParams;

// The instance for (kind, grouped, pair, 128-byte K slices per stage, mode);
// null for combinations that are not built (grouped runs bf16 only).
void* select_kernel(int kind, bool grouped, int pair, int ksub, int mode) {
    if (kind == kUmmaBf16)
        return grouped ? umma_kernel_bf16_grouped(pair, ksub, mode)
                       : umma_kernel_bf16(pair, ksub, mode);
    if (grouped) return nullptr;
    return umma_kernel_tf32(pair, ksub, mode);
}

int ksub_of(const GemmShape& s) { return s.k_sub == 2 ? 2 : 1; }

// Launches the instance for (kind, pair, k_sub); a CTA pair is a cluster of 2.
template <bool GROUPED>
cudaError_t launch_umma(int kind, int pair, const UmmaParams<GROUPED>& P, int grid, size_t smem,
                        cudaStream_t stream) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pair == 2) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = pair;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    n += unsigned(programmatic_launch_attr(attr + n));
    cfg.attrs = attr;
    cfg.numAttrs = n;
    void* args[] = {const_cast<UmmaParams<GROUPED>*>(&P)};
    const int mode = P.s.ctl.trace != nullptr ? 1 : P.s.dyn_counter != nullptr ? 2 : 0;
    return cudaLaunchKernelExC(&cfg, select_kernel(kind, GROUPED, pair, ksub_of(P.s), mode), args);
}

}  // namespace

size_t umma_ring_bytes(int stages, int pair, int k_sub) {
    const size_t stage = pair == 2 ? Pair<2>::stage_bytes : Pair<1>::stage_bytes;
    return 1024 + size_t(stages) * size_t(k_sub) * stage + kUmmaEpiBytes + kUmmaBarrierBytes +
           kUmmaBiasBytes;
}

size_t umma_smem_bytes(int stages, int pair, int k_sub) {
    const size_t need = umma_ring_bytes(stages, pair, k_sub);
    // At least half the SM's shared memory, so that two CTAs never share an
    // SM and compete for its 512 TMEM columns.
    const size_t floor_one_cta = 120 * 1024;
    return need > floor_one_cta ? need : floor_one_cta;
}
size_t umma_smem_bytes(int stages) { return umma_smem_bytes(stages, 1); }

cudaError_t umma_prepare(int kind, bool grouped, int pair, size_t smem) {
    static std::mutex mu;
    // [dev][kind][grouped][pair-1][ksub-1][mode]
    static size_t set[kMaxDeviceSlots][kUmmaKinds][2][2][2][3] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDeviceSlots) return cudaErrorInvalidDevice;
    if (select_kernel(kind, grouped, pair, 1, 0) == nullptr) return cudaErrorInvalidValue;
    std::lock_guard<std::mutex> lk(mu);
    for (int ksub = 1; ksub <= 2; ++ksub)
        for (int mode = 0; mode < 3; ++mode) {
            e = raise_smem_limit(select_kernel(kind, grouped, pair, ksub, mode), smem,
                                 &set[dev][kind][grouped ? 1 : 0][pair - 1][ksub - 1][mode]);
            if (e != cudaSuccess) return e;
        }
    return cudaSuccess;
}
cudaError_t umma_prepare(int kind, bool grouped, size_t smem) {
    return umma_prepare(kind, grouped, 1, smem);
}

cudaError_t umma_check_registers(int kind, bool grouped, int pair, int* regs) {
    cudaFuncAttributes fa;
    const long need = 128L * kRegsWG0 + 128L * kRegsWG1;
    if (select_kernel(kind, grouped, pair, 1, 0) == nullptr) return cudaErrorInvalidValue;
    for (int ksub = 1; ksub <= 2; ++ksub)
        for (int mode = 0; mode < 3; ++mode) {
            cudaError_t e =
                cudaFuncGetAttributes(&fa, select_kernel(kind, grouped, pair, ksub, mode));
            if (e != cudaSuccess) return e;
            *regs = fa.numRegs;
            if (long(fa.numRegs) * kThreads < need) return cudaErrorInvalidConfiguration;
        }
    return cudaSuccess;
}
cudaError_t umma_check_registers(int kind, bool grouped, int* regs) {
    return umma_check_registers(kind, grouped, 1, regs);
}

cudaError_t launch_gemm_umma(int kind, int pair, const CUtensorMap& mapA, const CUtensorMap& mapB,
                             const CUtensorMap& mapC, const GemmShape& s, int grid, size_t smem,
                             cudaStream_t stream) {
    UmmaParams<false> P;
    memset(&P, 0, sizeof(P));
    P.mapA = mapA;
    P.mapB = mapB;
    P.mapC[0] = mapC;
    P.s = s;
    P.bias_group_stride = 0;
    return launch_umma<false>(kind, pair, P, grid, smem, stream);
}
cudaError_t launch_gemm_umma(int kind, const CUtensorMap& mapA, const CUtensorMap& mapB,
                             const CUtensorMap& mapC, const GemmShape& s, int grid, size_t smem,
                             cudaStream_t stream) {
    return launch_gemm_umma(kind, 1, mapA, mapB, mapC, s, grid, smem, stream);
}

cudaError_t launch_gemm_umma_grouped(int pair, const CUtensorMap& mapX, const CUtensorMap& mapW,
                                     const CUtensorMap* mapsC, const GroupTable& g,
                                     const GemmShape& s, int64_t bias_group_stride, int grid,
                                     size_t smem, cudaStream_t stream) {
    UmmaParams<true> P;
    memset(&P, 0, sizeof(P));
    P.mapA = mapX;
    P.mapB = mapW;
    for (int e = 0; e < g.num_groups; ++e) P.mapC[e] = mapsC[e];
    P.s = s;
    P.g = g;
    P.bias_group_stride = bias_group_stride;
    return launch_umma<true>(kUmmaBf16, pair, P, grid, smem, stream);
}

}  // namespace gbr
