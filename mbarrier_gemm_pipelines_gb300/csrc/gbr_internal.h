// gbr_internal.h -- host-side interface between the C ABI (api.cu) and the
// kernel translation units.  Not installed; not part of the public ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gbr_common.cuh"

namespace gbr {

// Raises (never lowers) a kernel's dynamic shared-memory limit on the current
// device.  The limit is one value per kernel: lowering it for a small launch
// would make a later, larger launch of the same kernel fail.  `slot` holds the
// value set so far on this device; the caller's lock makes check-and-set atomic.
inline cudaError_t raise_smem_limit(const void* fn, size_t smem, size_t* slot) {
    if (smem <= *slot) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) *slot = smem;
    return e;
}
constexpr int kMaxDeviceSlots = 64;

// Failure-detection self test: the producer of CTA `cta` registers the bytes
// of its ring item `item` with expect_tx but issues no TMA load for it, so the
// consumer's bounded wait on that stage must run out.  All zero: no injection.
struct FaultInjection {
    uint32_t enabled;
    int32_t cta;
    int32_t item;
};

__device__ __forceinline__ bool inject_skip(const FaultInjection& f, uint32_t item) {
    return f.enabled != 0 && int32_t(blockIdx.x) == f.cta && int32_t(item) == f.item;
}

// The same for kernels whose CTAs work in units that share each ring item (a
// CTA pair): `cta` names the unit, and every CTA of it skips that item's loads.
__device__ __forceinline__ bool inject_skip_unit(const FaultInjection& f, uint32_t unit,
                                                 uint32_t item) {
    return f.enabled != 0 && int32_t(unit) == f.cta && int32_t(item) == f.item;
}

// ------------------------------------------------------------ staged copy
struct CopyArgs {
    int32_t rows, cols;            // fp32 elements
    int32_t tile_rows, tile_cols;  // TMA box
    int32_t tiles_c;               // tiles per row of tiles
    int64_t num_tiles;
    int32_t stages;
    uint32_t tile_bytes;
    int32_t store_lag;             // 0: release a slot when its own store has read it
                                   // 1: release the previous slot after issuing the next store
    KernelCtl ctl;
    uint32_t l2_hint;              // 0 none, 1 loads evict_first, 2 stores evict_first, 3 both
    FaultInjection inject;         // failure-detection self test only (zeroed: none)
};

// Distance between the staged copy's ring slots: the tile's bytes rounded up
// to 128 (the alignment of a TMA copy's shared-memory address).
__host__ __device__ constexpr uint32_t copy_slot_bytes(uint32_t tile_bytes) {
    return (tile_bytes + 127u) & ~127u;
}
size_t copy_smem_bytes(int stages, uint32_t tile_bytes);
cudaError_t copy_prepare(size_t smem);                 // per-device function attributes
cudaError_t copy_occupancy(size_t smem, int* blocks_per_sm);
cudaError_t launch_staged_copy(const CUtensorMap& src, const CUtensorMap& dst, const CopyArgs& a,
                               int grid, size_t smem, cudaStream_t stream);

// ------------------------------------------------------------ GEMM common
struct GemmShape {
    int32_t M, N, K;
    int32_t m_tiles, n_tiles, num_kb;
    int32_t num_tiles;
    int32_t stages;
    int32_t group_m;
    const float* bias;
    void* C;                       // used by epilogues that store with st.global
    const void* A;                 // read directly only by the cp.async producer variant
    const void* B;
    KernelCtl ctl;
    uint32_t k_sub;                // tensor-core GEMM: 128-byte K slices per ring stage (1, 2)
    uint32_t b_panels_3d;          // dense tensor-core GEMM: 1 when mapB is 3-D (column in
                                   // panel, K, panel), one box per K slice for all of this
                                   // CTA's B panels; 0: one 2-D box per panel
    uint32_t l2_hint;              // tensor-core GEMM operand loads: 0 none, 1 A and B
                                   // evict_last, 2 A evict_first / B evict_last,
                                   // 3 A evict_last / B evict_first, 4 both evict_normal
    FaultInjection inject;         // failure-detection self test only (zeroed: none)
    // Split tail (tensor-core GEMM; all zero: off, every tile runs whole).
    // The first dp_tiles tiles (a multiple of the unit count) run whole, one
    // per unit per round; the k-blocks of the last sk_tiles tiles, taken in
    // (tile, k-block) order, are dealt out in runs of sk_iters to the units.
    // Of the units sharing a tile, all but the last to arrive add their fp32
    // part into the tile's sum in sk_sum; the last waits for them on
    // sk_count, adds the sum to its own part and runs the epilogue.
    int32_t dp_tiles;
    int32_t sk_tiles;
    int32_t sk_iters;
    float* sk_sum;                 // [sk_tiles][tile rows][256] fp32, zeroed
    uint32_t* sk_count;            // [sk_tiles][CTAs per tile][4 epilogue warps][2], zeroed
    // Dynamic tile order (tensor-core GEMM; null: the static order above).
    // The even CTA's producer takes the next tile from this zeroed counter
    // with atomicAdd and hands its id to every role through a shared-memory
    // ring; no split tail then.
    uint32_t* dyn_counter;
};

// FFMA path (strict fp32, CUDA cores): 128x128x32 tiles.
constexpr int kFfmaBM = 128, kFfmaBN = 128, kFfmaBK = 32;
constexpr uint32_t kFfmaStageBytes = (kFfmaBM + kFfmaBN) * kFfmaBK * 4;
size_t ffma_smem_bytes(int stages);
cudaError_t ffma_prepare(size_t smem);
cudaError_t ffma_occupancy(size_t smem, int* blocks_per_sm);
cudaError_t ffma_check_registers(int* regs);
// split: the launch runs the split tail of s (TMA producer only).
cudaError_t launch_gemm_ffma(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmShape& s,
                             int grid, size_t smem, cudaStream_t stream, bool cpasync = false,
                             bool split = false);
// Consumer warps of the FFMA kernels (and of the homogeneous baseline's
// micro-tile layout): 8 (default) or 16; returns 0, or -1 for other values.
int ffma_set_consumer_warps(int cw);
int ffma_consumer_warps();
// Homogeneous baseline (every thread loads, syncs, computes, syncs); one CTA
// per 128x128 tile, single-buffered, plain global loads.
cudaError_t launch_gemm_ffma_sync(const float* A, const float* B, const GemmShape& s,
                                  cudaStream_t stream);

// tcgen05 path: 128x256 output tiles, 128-byte K slices per stage.
constexpr int kUmmaBM = 128, kUmmaBN = 256;
constexpr uint32_t kUmmaAStageBytes = kUmmaBM * 128;        // 16 KiB
constexpr uint32_t kUmmaBStageBytes = kUmmaBN * 128;        // 32 KiB
constexpr uint32_t kUmmaStageBytes = kUmmaAStageBytes + kUmmaBStageBytes;
constexpr uint32_t kUmmaEpiBytes = 4 * 2 * 32 * 128;        // 4 warps x 2 buffers x 4 KiB
// Barriers and small per-CTA words after the epilogue staging: 20 S + 132
// bytes for S ring stages (S <= 6 on every kernel instance), rounded up.
constexpr uint32_t kUmmaBarrierBytes = 384;
// The tile's bias (256 fp32), staged in shared memory by a bulk copy for the
// epilogue; after the barriers.
constexpr uint32_t kUmmaBiasBytes = kUmmaBN * 4;
constexpr int kMaxGroups = 32;

// Operand types of the tensor-core GEMM; both read A K-major from A[M, K] and
// B MN-major from B[K, N].
enum UmmaKind : int { kUmmaBf16 = 0, kUmmaTf32 = 1 };
constexpr int kUmmaKinds = 2;

struct GroupTable {
    int32_t num_groups;
    int32_t row_off[kMaxGroups];       // first row of group e in X and C
    int32_t rows[kMaxGroups];          // n_e
    int32_t m_tiles[kMaxGroups];       // ceil(n_e / tile rows)
    int32_t tile_start[kMaxGroups + 1];  // prefix sum of m_tiles[e] * n_tiles
    // CTA-pair launches: rows of group e's last M-tile when that tile runs
    // transposed (a "thin" tile: C^T = W^T X^T, the tile's rows as the MMA's
    // N), or 0 when it runs as an ordinary 256-row tile.
    int32_t thin[kMaxGroups];
};

// pair = 1: one CTA per 128x256 tile; pair = 2: a two-CTA cluster per 256x256
// tile (cta_group::2).  Overloads without `pair` mean pair = 1.
size_t umma_ring_bytes(int stages, int pair, int k_sub = 1);   // shared memory the ring needs
size_t umma_smem_bytes(int stages, int pair, int k_sub = 1);   // what the launch requests
size_t umma_smem_bytes(int stages);
cudaError_t umma_prepare(int kind, bool grouped, int pair, size_t smem);
cudaError_t umma_prepare(int kind, bool grouped, size_t smem);
cudaError_t umma_check_registers(int kind, bool grouped, int pair, int* regs);
cudaError_t umma_check_registers(int kind, bool grouped, int* regs);
cudaError_t launch_gemm_umma(int kind, int pair, const CUtensorMap& mapA, const CUtensorMap& mapB,
                             const CUtensorMap& mapC, const GemmShape& s, int grid, size_t smem,
                             cudaStream_t stream);
cudaError_t launch_gemm_umma(int kind, const CUtensorMap& mapA, const CUtensorMap& mapB,
                             const CUtensorMap& mapC, const GemmShape& s, int grid, size_t smem,
                             cudaStream_t stream);
cudaError_t launch_gemm_umma_grouped(int pair, const CUtensorMap& mapX, const CUtensorMap& mapW,
                                     const CUtensorMap* mapsC, const GroupTable& g,
                                     const GemmShape& s, int64_t bias_group_stride, int grid,
                                     size_t smem, cudaStream_t stream);

// Bt[N, K] = B[K, N], 32-bit elements, K and N multiples of 4.

// ------------------------------------------------------------ no-alloc variant
// Status words of the no-alloc scratch on the current device: returns the error
// bits (0: none or never set up) and copies words [0..3] out, then clears them.
uint32_t noalloc_take_status(uint32_t* words4);

// Programmatic dependent launch (on unless gbr_launch_overlap(0)): fills
// attr[0] and returns 1, or returns 0 when it is off.  Every kernel launched
// with it runs griddep_wait() before its first global-memory access.
int programmatic_launch_attr(cudaLaunchAttribute* attr);

// ------------------------------------------------------------ api.cu services
int report_error(int code, const char* msg);   // sets gbr_last_error(), returns code
void count_launch();                           // adds one to gbr_launch_count()
uint64_t wait_timeout_ns();                    // per-wait limit of this thread's next launch
FaultInjection injection_now();                // self-test fault of this thread's next launch

// ------------------------------------------------------------ self test
cudaError_t launch_wait_selftest(KernelCtl ctl, cudaStream_t stream);

}  // namespace gbr
