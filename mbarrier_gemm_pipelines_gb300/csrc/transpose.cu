// transpose.cu -- Bt[N, K] = B[K, N] for 32-bit elements.
//
// The sm_100-family tensor core reads TF32 operands only in K-major order
// (an N-major B operand of tcgen05.mma.kind::tf32 yields zeros), so the TF32
// GEMM first turns the row-major B[K, N] into K-major Bt[N, K].  HBM-bound:
// each 64x64 tile is read with coalesced 16-byte loads along N, staged in
// padded shared memory, and written with coalesced 16-byte stores along K.
#include "gbr_internal.h"

namespace gbr {

namespace {

constexpr int kT = 64;          // tile edge
constexpr int kThreadsX = 16;   // float4 columns per tile row
constexpr int kThreadsY = 16;

__global__ void __launch_bounds__(kThreadsX * kThreadsY)
    transpose_f32_kernel(const float* __restrict__ B, float* __restrict__ Bt, int K, int N) {
    __shared__ float tile[kT][kT + 1];
    const int n0 = blockIdx.x * kT, k0 = blockIdx.y * kT;
    const int tx = threadIdx.x, ty = threadIdx.y;
    ptx::griddep_wait();                 // B may come from the previous kernel in the stream
    ptx::griddep_launch_dependents();    // the GEMM that reads Bt may be scheduled (it waits too)
    // Load rows k0..k0+63, columns n0 + 4tx .. +3 (N is a multiple of 4).
#pragma unroll
    for (int r = ty; r < kT; r += kThreadsY) {
        const int k = k0 + r, n = n0 + 4 * tx;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < K && n < N) v = __ldg(reinterpret_cast<const float4*>(B + size_t(k) * N + n));
        tile[r][4 * tx + 0] = v.x;
        tile[r][4 * tx + 1] = v.y;
        tile[r][4 * tx + 2] = v.z;
        tile[r][4 * tx + 3] = v.w;
    }
    __syncthreads();
    // Store rows n0..n0+63 of Bt, columns k0 + 4tx .. +3 (K is a multiple of 4).
#pragma unroll
    for (int r = ty; r < kT; r += kThreadsY) {
        const int n = n0 + r, k = k0 + 4 * tx;
        if (n < N && k < K) {
            float4 v;
            v.x = tile[4 * tx + 0][r];
            v.y = tile[4 * tx + 1][r];
            v.z = tile[4 * tx + 2][r];
            v.w = tile[4 * tx + 3][r];
            *reinterpret_cast<float4*>(Bt + size_t(n) * K + k) = v;
        }
    }
}

}  // namespace

cudaError_t launch_transpose_f32(const float* B, float* Bt, int K, int N, cudaStream_t stream) {
    dim3 grid((N + kT - 1) / kT, (K + kT - 1) / kT);
    dim3 block(kThreadsX, kThreadsY);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = programmatic_launch_attr(attr);
    cfg.attrs = attr;
    return cudaLaunchKernelEx(&cfg, transpose_f32_kernel, B, Bt, K, N);
}

}  // namespace gbr
