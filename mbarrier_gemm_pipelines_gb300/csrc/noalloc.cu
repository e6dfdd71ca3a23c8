// noalloc.cu -- the TF32 GEMM + bias + ReLU for callers that cannot allocate
// device memory.
//
// The regular entry point allocates the library's per-device status block on
// first use, and may take per-call scratch from the stream-ordered allocator
// (split-tile partial sums, the dynamic tile counter).  Some callers cannot
// allow either: serving loops that must never enter an allocator (it can take
// locks or synchronise the device at unpredictable times), plug-ins whose host
// framework owns all device allocation, and processes whose device memory is
// entirely reserved by another allocator, so that a cudaMalloc or
// cudaMallocAsync from this library would fail.  This variant runs the TF32
// tensor-core GEMM kernel, one CTA per tile and never split, and takes its
// only scratch -- the status words -- from a file-scope device array that the
// CUDA driver creates when the library's module is loaded.
#include "gbr.h"
#include "gbr_internal.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace gbr {

namespace {

constexpr size_t kNoallocStatusBytes = 256;             // kStatusWords words, padded
constexpr size_t kNoallocScratchBytes = kNoallocStatusBytes;

// Held by every device that loads this library until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
struct NoallocDevice {
    bool ready = false;
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch
    int sm_count = 0;
    int smem_optin = 0;
    bool regs_ok = false;
};
NoallocDevice g_na[kMaxDev];
std::mutex g_na_mu;

PFN_cuTensorMapEncodeTiled_v12000 na_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool na_map_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
               uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto fn = na_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * 4};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(ptr), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B [K, N] fp32 as a 3-D tensor (column in a 32-column panel, K, panel), for
// N a multiple of 32: one box brings the 8 panels of a 32-row K slice of a
// 256-column tile, in the 32-byte-atom swizzle that the TF32 MMA reads.
bool na_map_b_panels(CUtensorMap* map, const void* B, uint64_t K, uint64_t N) {
    auto fn = na_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {32, K, N / 32};
    cuuint64_t strides[2] = {N * 4, 128};
    cuuint32_t box[3] = {32, 32, 8};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(B), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Once per device, with that device current: the device address of the
// scratch array (in host code the array's name is only a host-side stand-in),
// the attributes the launch needs, and the register check of the GEMM kernel.
int na_setup(NoallocDevice** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return report_error(GBR_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDev) return report_error(GBR_ERR_INVALID, "device index out of range");
    std::lock_guard<std::mutex> lk(g_na_mu);
    NoallocDevice& d = g_na[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return report_error(GBR_ERR_CUDA, "cudaDeviceGetAttribute failed");
        if (major != 10 || minor != 3)
            return report_error(GBR_ERR_UNSUPPORTED, "this library is built for sm_103a only");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return report_error(GBR_ERR_CUDA, "cudaGetSymbolAddress(no-alloc scratch) failed");
        // The array starts zeroed when the module loads; clear its status words
        // once more here, and wait, so that no launch can overtake the clear.
        if (cudaMemset(p, 0, kNoallocStatusBytes) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess)
            return report_error(GBR_ERR_CUDA, "clearing the no-alloc status words failed");
        int regs = 0;
        d.regs_ok = umma_check_registers(kUmmaTf32, false, &regs) == cudaSuccess;
        d.scratch = static_cast<unsigned char*>(p);
        d.ready = true;
    }
    *out = &d;
    return GBR_OK;
}

}  // namespace

// Reads the status words of the no-alloc scratch on the current device and,
// when a timeout is recorded there, clears them and waits for the clear (so
// that no later launch can overtake it).  The caller has synchronised the
// stream the no-alloc calls ran on.  Returns the error bits (0: nothing
// recorded, or the scratch was never set up on this device) and copies words
// [0..3] out; allocates nothing.
uint32_t noalloc_take_status(uint32_t* words4) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    unsigned char* scratch;
    {
        std::lock_guard<std::mutex> lk(g_na_mu);
        if (!g_na[dev].ready) return 0;
        scratch = g_na[dev].scratch;
    }
    uint32_t st[kStatusWords];
    if (cudaMemcpy(st, scratch, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return 0;
    if (st[0] == 0) return 0;
    cudaMemset(scratch, 0, sizeof(st));
    cudaDeviceSynchronize();
    for (int i = 0; i < 4; ++i) words4[i] = st[i];
    return st[0];
}

}  // namespace gbr

using namespace gbr;

extern "C" int gemm_bias_relu_tf32_noalloc(const float* A, const float* B, const float* bias,
                                           float* C, int64_t M, int64_t N, int64_t K, int stages,
                                           gbr_stream_t stream) {
    const int64_t lim = int64_t(1) << 31;
    if (M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim)
        return report_error(GBR_ERR_INVALID, "gemm_bias_relu_tf32_noalloc: M, N, K must be in [0, 2^31)");
    NoallocDevice* d;
    int r = na_setup(&d);
    if (r != GBR_OK) return r;
    // One CTA per 128x256 tile: as many 48 KiB stages as fit beside the
    // epilogue staging (4 on GB300).
    int smax = 0;
    while (smax < 16 && 1024 + size_t(smax + 1) * kUmmaStageBytes + kUmmaEpiBytes + kUmmaBarrierBytes +
                                kUmmaBiasBytes <=
                            size_t(d->smem_optin))
        ++smax;
    if (stages < 1 || stages > smax) {
        char msg[160];
        snprintf(msg, sizeof(msg),
                 "gemm_bias_relu_tf32_noalloc: stages=%d outside [1, %d] (one CTA per tile)",
                 stages, smax);
        return report_error(GBR_ERR_SMEM, msg);
    }
    if (M == 0 || N == 0) return GBR_OK;
    if (!C || !bias || (K > 0 && (!A || !B)))
        return report_error(GBR_ERR_INVALID, "gemm_bias_relu_tf32_noalloc: NULL buffer");
    auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!al(C) || !al(bias) || (K > 0 && (!al(A) || !al(B))) || (N % 4) || (K % 4))
        return report_error(GBR_ERR_ALIGN,
                            "gemm_bias_relu_tf32_noalloc: 16-byte aligned buffers, K and N "
                            "multiples of 4");
    auto overlap = [](const void* a, size_t an, const void* b, size_t bn) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
        return a0 < b0 + bn && b0 < a0 + an;
    };
    const size_t c_bytes = size_t(M) * size_t(N) * 4u;
    if ((K > 0 && (overlap(C, c_bytes, A, size_t(M) * size_t(K) * 4u) ||
                   overlap(C, c_bytes, B, size_t(K) * size_t(N) * 4u))) ||
        overlap(C, c_bytes, bias, size_t(N) * 4u))
        return report_error(GBR_ERR_INVALID, "gemm_bias_relu_tf32_noalloc: C overlaps an input");
    if (!d->regs_ok)
        return report_error(GBR_ERR_CUDA, "tcgen05 GEMM kernel has too few registers for its role split");

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // Status words: zero at set-up and after every read that found a timeout,
    // so a recorded timeout stays until gbr_device_status() reads it (the
    // first one recorded is the one kept).
    uint32_t* status = reinterpret_cast<uint32_t*>(d->scratch);

    GemmShape s;
    memset(&s, 0, sizeof(s));
    s.M = int32_t(M);
    s.N = int32_t(N);
    s.K = int32_t(K);
    s.stages = stages;
    s.bias = bias;
    s.C = C;
    s.ctl.status = status;
    s.ctl.timeout_ns = wait_timeout_ns();
    s.inject = injection_now();   // zero except under gbr_selftest_noalloc_skip_load
    s.m_tiles = int32_t((M + kUmmaBM - 1) / kUmmaBM);
    s.n_tiles = int32_t((N + kUmmaBN - 1) / kUmmaBN);
    s.num_kb = int32_t((K + 31) / 32);
    s.num_tiles = s.m_tiles * s.n_tiles;
    s.group_m = 16;
    CUtensorMap ma, mb, mc;
    if (!na_map_2d(&mc, C, uint64_t(N), uint64_t(M), 32, 32))
        return report_error(GBR_ERR_INVALID, "encoding the C tensor map failed");
    if (K > 0) {
        // A K-major; B as N-major panels of 32 columns x 32 K rows in the
        // 32-byte-atom swizzle that the TF32 MMA reads (one box per panel, or
        // one per K slice when N is a whole number of panels).
        s.b_panels_3d = N % 32 == 0 ? 1u : 0u;
        if (!na_map_2d(&ma, A, uint64_t(K), uint64_t(M), 32, 128) ||
            !(s.b_panels_3d ? na_map_b_panels(&mb, B, uint64_t(K), uint64_t(N))
                            : na_map_2d(&mb, B, uint64_t(N), uint64_t(K), 32, 32,
                                        CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B)))
            return report_error(GBR_ERR_INVALID, "encoding the A/B tensor maps failed");
    } else {
        ma = mc;
        mb = mc;
    }
    const size_t smem = umma_smem_bytes(stages);
    if (umma_prepare(kUmmaTf32, false, smem) != cudaSuccess)
        return report_error(GBR_ERR_CUDA, "cudaFuncSetAttribute(tcgen05 GEMM) failed");
    const int grid = int(std::min<int64_t>(s.num_tiles, d->sm_count));
    if (launch_gemm_umma(kUmmaTf32, ma, mb, mc, s, grid, smem, st) != cudaSuccess)
        return report_error(GBR_ERR_CUDA, "launching the tcgen05 GEMM failed");
    count_launch();
    return GBR_OK;
}
