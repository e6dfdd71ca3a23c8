// gemm_ffma.cu -- warp-specialized fp32 GEMM + bias + ReLU on CUDA cores.
//
// The SGEMM test bench of "pwwt.cn news/4436243", section 4.1: A[M,K] and
// B[K,N] fp32, C[M,N] = ReLU(A*B + bias), with the K loop turned into the
// ring buffer of section 3.4: a producer role moves K tiles into a stage ring
// while consumer roles compute on full stages and hand them back.
//
// Roles (one CTA = 3 warpgroups, 384 threads, "gpu_warp_specialization",
// "The architecture: every piece explained": whole warps take whole jobs,
// and the register budget moves from the producers to the consumers):
//   warpgroup 0  warp 0 lane 0 = TMA producer; the group gives up registers
//   warpgroups 1-2 (8 warps)   = FFMA consumers, one 8x8 register micro-tile
//                                 per thread of a 128x128 output tile
// Ring: S stages of { A 128x32 fp32, 128-byte swizzled rows;
//                     B 32x128 fp32 as four 32-column 128-byte swizzled panels }.
// full[s]: 1 arrival (producer's arrive.expect_tx) + 32 KiB of TMA bytes.
// empty[s]: 8 arrivals, one per consumer warp after its last read of the slot.
// Slot/parity of k-iteration i (running across this CTA's tiles):
//   slot = i % S, full parity = (i / S) & 1, empty parity = ((i / S) & 1) ^ 1.
#include "gbr_internal.h"

namespace gbr {

namespace {

constexpr int kThreads = 384;
constexpr int kConsumerWarps = 8;
constexpr uint32_t kABytes = kFfmaBM * kFfmaBK * 4;   // 16 KiB
constexpr uint32_t kBPanelBytes = kFfmaBK * 128;      // 32 rows x 128 B
constexpr uint32_t kProducerRegs = 40;
constexpr uint32_t kConsumerRegs = 232;

// One 32-deep K stage of the 128 x 128 tile for thread (tx, ty): rows
// ty + 16 r, columns 4 tx .. 4 tx + 3 and 64 + 4 tx .. 64 + 4 tx + 3.  All of
// the thread's rows share one swizzle phase (a_ph = ty % 8) per k-group, and
// all its columns one phase per k, read from the table b_sw, so every
// shared-memory load of a k-group is base + immediate offset.
//
// The accumulators are packed column pairs: acc[r][j] holds columns
// (2j, 2j + 1) of the thread's eight, and each step is one packed fp32x2 FMA
// (two IEEE fp32 FMAs, the same results as two scalar ones) of A broadcast to
// both halves and a B pair read straight from shared memory as 64 bits.  Half
// as many FMA instructions leave issue slots for the loads.
__device__ __forceinline__ void ffma_stage(uint64_t (&acc)[8][4], const uint8_t* As,
                                           const uint8_t* Bs, uint32_t a_row, uint32_t a_ph,
                                           const uint32_t (&b_sw)[8]) {
#pragma unroll
    for (uint32_t k4 = 0; k4 < kFfmaBK / 4; ++k4) {
        const uint8_t* ap = As + a_row + ((k4 ^ a_ph) << 4);   // row ty, 16-byte chunk k4
        float4 a[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) a[r] = *reinterpret_cast<const float4*>(ap + r * 16 * 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t k = 4 * k4 + kk;
            const uint8_t* bp = Bs + b_sw[k & 7u] + k * 128u;
            const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(bp);
            const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(bp + 2 * kBPanelBytes);
            uint64_t a2[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                a2[r] = ptx::f32x2_splat(kk == 0 ? a[r].x : kk == 1 ? a[r].y : kk == 2 ? a[r].z : a[r].w);
            const uint64_t bj[4] = {b0.x, b0.y, b1.x, b1.y};
            // Column pair outer, row inner: eight independent FMAs share one B
            // pair (measured 4% faster than the row-outer order).
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int r = 0; r < 8; ++r) ptx::fma_f32x2(acc[r][j], a2[r], bj[j]);
        }
    }
}

__device__ __forceinline__ void ffma_zero(uint64_t (&acc)[8][4]) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[r][j] = 0ull;
}

__device__ __forceinline__ void ffma_tables(uint32_t tx, uint32_t ty, uint32_t& a_row,
                                            uint32_t& a_ph, uint32_t (&b_sw)[8]) {
    a_row = ty * 128u;
    a_ph = ty & 7u;
#pragma unroll
    for (uint32_t j = 0; j < 8; ++j)
        b_sw[j] = (tx >> 3) * kBPanelBytes + (((tx & 7u) ^ j) << 4);  // column 4 tx, K row % 8 = j
}

// C = max(0, acc + bias) for the thread's 8 x 8 outputs of tile (mt, nt).
__device__ __forceinline__ void ffma_epilogue(const uint64_t (&acc)[8][4], const GemmShape& p,
                                              uint32_t mt, uint32_t nt, uint32_t tx, uint32_t ty) {
    float* C = static_cast<float*>(p.C);
    const int n0 = int(nt) * kFfmaBN, m0 = int(mt) * kFfmaBM;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int n = n0 + int(4 * tx) + 64 * h;
        if (n >= p.N) continue;
        const float4 bb = __ldg(reinterpret_cast<const float4*>(p.bias + n));
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int m = m0 + int(ty) + 16 * r;
            if (m >= p.M) continue;
            const uint64_t lo = acc[r][2 * h], hi = acc[r][2 * h + 1];
            float4 v;
            v.x = fmaxf(__uint_as_float(uint32_t(lo)) + bb.x, 0.f);
            v.y = fmaxf(__uint_as_float(uint32_t(lo >> 32)) + bb.y, 0.f);
            v.z = fmaxf(__uint_as_float(uint32_t(hi)) + bb.z, 0.f);
            v.w = fmaxf(__uint_as_float(uint32_t(hi >> 32)) + bb.w, 0.f);
            *reinterpret_cast<float4*>(C + size_t(m) * p.N + n) = v;
        }
    }
}

// CPASYNC = false: one TMA lane produces each stage (the default).
// CPASYNC = true: the historical producer ("gpu_warp_specialization" and
// "pwwt.cn news/4436243" section 2: Ampere cp.async): the whole producer
// warpgroup copies the stage with 16-byte cp.async per thread into the same
// swizzled layout, and each of its 128 threads arrives on full[s] with
// cp.async.mbarrier.arrive.noinc once its own copies have landed.
template <bool CPASYNC>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_ffma_kernel(const __grid_constant__ CUtensorMap mapA,
                     const __grid_constant__ CUtensorMap mapB, const GemmShape p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = align_1024(smem_raw);
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + size_t(S) * kFfmaStageBytes);
    uint64_t* empty = full + S;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + S);

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(ptx::smem_addr(full + s), CPASYNC ? 128u : 1u);
            ptx::mbar_init(ptx::smem_addr(empty + s), kConsumerWarps);
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    } else if (threadIdx.x == 32) {
        ptx::prefetch_tensormap(&mapA);
        ptx::prefetch_tensormap(&mapB);
    }
    __syncthreads();
    // The set-up above overlaps the end of the previous kernel in the stream;
    // no role touches global memory before that kernel is done.
    ptx::griddep_wait();

    const uint32_t ring_base = ptx::smem_addr(ring);
    uint32_t issued = 0;   // TMA producer lane: ring items registered on full[]

    if (warp < 4) {
        ptx::setmaxnreg_dec<kProducerRegs>();
        if (CPASYNC) {
            // ------------------------------------ cp.async producer warpgroup
            const uint32_t pt = threadIdx.x;   // 0..127
            const float* A = static_cast<const float*>(p.A);
            const float* B = static_cast<const float*>(p.B);
            uint32_t i = 0, ntr = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
                uint32_t mt, nt;
                raster_tile(t, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
                const int m0 = int(mt) * kFfmaBM, n0 = int(nt) * kFfmaBN;
                for (int kb = 0; kb < p.num_kb; ++kb, ++i) {
                    const uint32_t s = i % S, ph = (i / S) & 1u;
                    if (!mbar_wait_warp(ptx::smem_addr(empty + s), ph ^ 1u, p.ctl, abort_flag,
                                        kSiteProducerEmpty, i)) {
                        ok = false;
                        break;
                    }
                    if (pt == 0) {   // thread 0 traces for the warpgroup
                        trace_event(p.ctl, kRoleProducer, ntr, kEvWaitDone, i, s, ph ^ 1u);
                        trace_event(p.ctl, kRoleProducer, ntr, kEvIssued, i, s, 0);
                    }
                    const uint32_t st = ring_base + s * kFfmaStageBytes;
                    const int k0 = kb * kFfmaBK;
#pragma unroll
                    for (uint32_t j = 0; j < 8; ++j) {   // A: 128 rows x 8 chunks of 16 B
                        const uint32_t c = pt + 128u * j, row = c >> 3, k4 = c & 7u;
                        const int m = m0 + int(row), k = k0 + int(4 * k4);
                        const bool in = m < p.M && k < p.K;
                        ptx::cp_async_16(st + row * 128u + ((k4 ^ (row & 7u)) << 4),
                                         in ? A + size_t(m) * p.K + k : A, in ? 16u : 0u);
                    }
#pragma unroll
                    for (uint32_t j = 0; j < 8; ++j) {   // B: 32 K rows x 32 chunks of 16 B
                        const uint32_t c = pt + 128u * j, kr = c >> 5, n4 = c & 31u;
                        const int k = k0 + int(kr), n = n0 + int(4 * n4);
                        const bool in = k < p.K && n < p.N;
                        ptx::cp_async_16(st + kABytes + (n4 >> 3) * kBPanelBytes + kr * 128u +
                                             (((n4 & 7u) ^ (kr & 7u)) << 4),
                                         in ? B + size_t(k) * p.N + n : B, in ? 16u : 0u);
                    }
                    ptx::cp_async_mbar_arrive_noinc(ptx::smem_addr(full + s));
                }
            }
            if (pt == 0) trace_count(p.ctl, kRoleProducer, ntr);
            ptx::griddep_launch_dependents();
            ptx::cp_async_wait_all();   // no copy may still be writing when the CTA exits
        } else if (warp == 0 && lane == 0) {
            // ------------------------------------------------ producer
            uint32_t i = 0, ntr = 0;
            bool ok = true;
            for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
                uint32_t mt, nt;
                raster_tile(t, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
                for (int kb = 0; kb < p.num_kb; ++kb, ++i) {
                    const uint32_t s = i % S, ph = (i / S) & 1u;
                    if (!mbar_wait(ptx::smem_addr(empty + s), ph ^ 1u, p.ctl, abort_flag,
                                   kSiteProducerEmpty, i)) {
                        ok = false;
                        break;
                    }
                    trace_event(p.ctl, kRoleProducer, ntr, kEvWaitDone, i, s, ph ^ 1u);
                    const uint32_t fb = ptx::smem_addr(full + s);
                    ptx::mbar_arrive_expect_tx(fb, kFfmaStageBytes);
                    if (inject_skip(p.inject, i)) continue;   // self test: stage never fills
                    trace_event(p.ctl, kRoleProducer, ntr, kEvIssued, i, s, 0);
                    const uint32_t st = ring_base + s * kFfmaStageBytes;
                    ptx::tma_load_2d(st, &mapA, fb, kb * kFfmaBK, int(mt) * kFfmaBM);
#pragma unroll
                    for (int j = 0; j < kFfmaBN / 32; ++j)
                        ptx::tma_load_2d(st + kABytes + j * kBPanelBytes, &mapB, fb,
                                         int(nt) * kFfmaBN + 32 * j, kb * kFfmaBK);
                }
            }
            trace_count(p.ctl, kRoleProducer, ntr);
            ptx::griddep_launch_dependents();   // every load issued: the next launch may be scheduled
            issued = i;
        }
    } else {
        ptx::setmaxnreg_inc<kConsumerRegs>();
        // ---------------------------------------------------- consumers
        // Thread (tx, ty) of 16 x 16 owns rows ty + 16 r (r = 0..7) and columns
        // 4 tx .. 4 tx + 3 and 64 + 4 tx .. 64 + 4 tx + 3 of the 128 x 128 tile.
        // All its rows have the same (row % 8), so every A read of a k-group
        // uses one swizzle phase; all its columns sit at the same position
        // inside their 32-column panels, so every B read of a k uses one
        // phase too.  The phases come from two 8-entry tables and every
        // shared-memory load is base + immediate offset.
        const uint32_t ct = threadIdx.x - 128;        // 0..255
        const uint32_t tx = ct & 15u, ty = ct >> 4;
        uint32_t a_row, a_ph, b_sw[8];
        ffma_tables(tx, ty, a_row, a_ph, b_sw);

        uint32_t i = 0, ntr = 0;
        const bool tracer = p.ctl.trace != nullptr && warp == 4 && lane == 0;   // one consumer lane
        bool ok = true;
        for (int t = blockIdx.x; ok && t < p.num_tiles; t += gridDim.x) {
            uint32_t mt, nt;
            raster_tile(t, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
            uint64_t acc[8][4];
            ffma_zero(acc);

            for (int kb = 0; kb < p.num_kb; ++kb, ++i) {
                const uint32_t s = i % S, ph = (i / S) & 1u;
                if (!mbar_wait_warp(ptx::smem_addr(full + s), ph, p.ctl, abort_flag,
                                    kSiteConsumerFull, i)) {
                    ok = false;
                    break;
                }
                if (tracer) trace_event(p.ctl, kRoleConsumer, ntr, kEvWaitDone, i, s, ph);
                const uint8_t* As = ring + size_t(s) * kFfmaStageBytes;
                ffma_stage(acc, As, As + kABytes, a_row, a_ph, b_sw);
                __syncwarp();
                if (tracer) trace_event(p.ctl, kRoleConsumer, ntr, kEvReleased, i, s, 0);
                if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(empty + s));
            }
            if (!ok) break;

            ffma_epilogue(acc, p, mt, nt, tx, ty);
        }
        if (tracer) trace_count(p.ctl, kRoleConsumer, ntr);
    }
    __syncwarp();
    __syncthreads();
    // Every role has left its loop, so the abort flag is final.  After an
    // abort the TMA lane waits (bounded) for its loads still in flight -- the
    // last S items it registered, except a self test's unissued one -- before
    // the CTA may exit.  (The cp.async producers waited for their own copies.)
    if (!CPASYNC && warp == 0 && lane == 0 && *abort_flag) {
        const uint32_t n = issued < uint32_t(S) ? issued : uint32_t(S);
        for (uint32_t j = issued - n; j < issued; ++j)
            if (!inject_skip(p.inject, j))
                mbar_wait_drain(ptx::smem_addr(full + j % S), (j / S) & 1u, p.ctl.timeout_ns);
    }
    __syncthreads();
}

// The homogeneous baseline of "pwwt.cn news/4436243", section 1.1: every
// thread loads its share of the next K tile from global memory into shared
// memory, the block synchronises, every thread computes on the tile, and the
// block synchronises again before the buffer may be overwritten.  Same tile,
// same shared-memory layout and same FFMA micro-kernel as the warp-specialized
// kernel above; no roles, no ring, no mbarriers.  One CTA per output tile.
constexpr int kSyncThreads = 256;

__global__ void __launch_bounds__(kSyncThreads, 2) gemm_ffma_sync_kernel(const float* __restrict__ A,
                                                                         const float* __restrict__ B,
                                                                         const GemmShape p) {
    __shared__ __align__(1024) uint8_t tile[kFfmaStageBytes];
    uint8_t* As = tile;
    uint8_t* Bs = tile + kABytes;
    const uint32_t t = threadIdx.x;
    const uint32_t tx = t & 15u, ty = t >> 4;
    uint32_t mt, nt;
    raster_tile(blockIdx.x, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
    const int m0 = int(mt) * kFfmaBM, n0 = int(nt) * kFfmaBN;
    uint32_t a_row, a_ph, b_sw[8];
    ffma_tables(tx, ty, a_row, a_ph, b_sw);
    uint64_t acc[8][4];
    ffma_zero(acc);

    for (int kb = 0; kb < p.num_kb; ++kb) {
        const int k0 = kb * kFfmaBK;
        // load: 4 float4 of A (row idx/8, 16-byte chunk idx%8) and 4 of B
        // (K row idx/32, 16-byte chunk idx%32) per thread, zero outside the
        // matrix, stored in the same swizzled layout the TMA path produces.
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t idx = t + kSyncThreads * j;
            const uint32_t row = idx >> 3, k4 = idx & 7u;
            const int m = m0 + int(row), k = k0 + int(4 * k4);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m < p.M && k < p.K) v = __ldg(reinterpret_cast<const float4*>(A + size_t(m) * p.K + k));
            *reinterpret_cast<float4*>(As + row * 128u + ((k4 ^ (row & 7u)) << 4)) = v;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t idx = t + kSyncThreads * j;
            const uint32_t kr = idx >> 5, n4 = idx & 31u;
            const int k = k0 + int(kr), n = n0 + int(4 * n4);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < p.K && n < p.N) v = __ldg(reinterpret_cast<const float4*>(B + size_t(k) * p.N + n));
            *reinterpret_cast<float4*>(Bs + (n4 >> 3) * kBPanelBytes + kr * 128u +
                                       (((n4 & 7u) ^ (kr & 7u)) << 4)) = v;
        }
        __syncthreads();   // the whole tile has arrived
        ffma_stage(acc, As, Bs, a_row, a_ph, b_sw);
        __syncthreads();   // every thread is done with it
    }
    ffma_epilogue(acc, p, mt, nt, tx, ty);
}

}  // namespace

cudaError_t launch_gemm_ffma_sync(const float* A, const float* B, const GemmShape& s,
                                  cudaStream_t stream) {
    gemm_ffma_sync_kernel<<<s.num_tiles, kSyncThreads, 0, stream>>>(A, B, s);
    return cudaGetLastError();
}

size_t ffma_smem_bytes(int stages) {
    return 1024 + size_t(stages) * kFfmaStageBytes + size_t(2 * stages) * 8 + 16;
}

cudaError_t ffma_prepare(size_t smem) {
    static std::mutex mu;
    static size_t set[kMaxDeviceSlots][2] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDeviceSlots) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if ((e = raise_smem_limit(reinterpret_cast<const void*>(gemm_ffma_kernel<false>), smem,
                              &set[dev][0])) != cudaSuccess)
        return e;
    return raise_smem_limit(reinterpret_cast<const void*>(gemm_ffma_kernel<true>), smem, &set[dev][1]);
}

cudaError_t ffma_occupancy(size_t smem, int* blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, gemm_ffma_kernel<false>,
                                                         kThreads, smem);
}

// The register split must fit in what the CTA is launched with, or the
// consumers' setmaxnreg.inc would wait forever for registers.
cudaError_t ffma_check_registers(int* regs) {
    const long need = 128L * kProducerRegs + 256L * kConsumerRegs;
    for (const void* fn : {reinterpret_cast<const void*>(gemm_ffma_kernel<false>),
                           reinterpret_cast<const void*>(gemm_ffma_kernel<true>)}) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return e;
        *regs = fa.numRegs;
        if (long(fa.numRegs) * kThreads < need) return cudaErrorInvalidConfiguration;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm_ffma(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmShape& s,
                             int grid, size_t smem, cudaStream_t stream, bool cpasync) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = programmatic_launch_attr(attr);
    cfg.attrs = attr;
    if (cpasync) return cudaLaunchKernelEx(&cfg, gemm_ffma_kernel<true>, mapA, mapB, s);
    return cudaLaunchKernelEx(&cfg, gemm_ffma_kernel<false>, mapA, mapB, s);
}

}  // namespace gbr
