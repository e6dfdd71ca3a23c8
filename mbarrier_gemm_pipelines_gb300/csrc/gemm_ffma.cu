// gemm_ffma.cu -- warp-specialized fp32 GEMM + bias + ReLU on CUDA cores.
//
// The SGEMM test bench of "pwwt.cn news/4436243", section 4.1: A[M,K] and
// B[K,N] fp32, C[M,N] = ReLU(A*B + bias), with the K loop turned into the
// ring buffer of section 3.4: a producer role moves K tiles into a stage ring
// while consumer roles compute on full stages and hand them back.
//
// Roles ("gpu_warp_specialization", "The architecture: every piece
// explained": whole warps take whole jobs, and the register budget moves from
// the producers to the consumers):
//   warpgroup 0  warp 0 lane 0 = TMA producer; the group gives up registers
//   CW consumer warps           = FFMA consumers of a 128x128 output tile:
//     CW = 8 (default): 2 warpgroups, 384 threads per CTA, an 8x8 register
//                       micro-tile per thread, 2 consumer warps per scheduler
//     CW = 16:          4 warpgroups, 640 threads per CTA, an 8x4 micro-tile,
//                       4 consumer warps per scheduler
// A thread reads rows + columns floats from shared memory per k for
// rows x columns FMAs: 16 per 64 at 8x8, 12 per 32 at 8x4.  Measured on GB300
// the 8x4 layout keeps the FMA pipe busy 63% of active cycles against 74.5%
// at 8x8 (48.8 against 57 TFLOP/s): more warps per scheduler do not pay for
// the extra shared-memory traffic per FMA.
// Ring: S stages of { A 128x32 fp32, 128-byte swizzled rows;
//                     B 32x128 fp32 as four 32-column 128-byte swizzled panels }.
// full[s]: 1 arrival (producer's arrive.expect_tx) + 32 KiB of TMA bytes.
// empty[s]: CW arrivals, one per consumer warp after its last read of the slot.
// Slot/parity of k-iteration i (running across this CTA's tiles):
//   slot = i % S, full parity = (i / S) & 1, empty parity = ((i / S) & 1) ^ 1.
// A launch's last partial round of tiles can instead run as a split tail: the
// whole tiles in one launch of this kernel, then a second, separate instance
// (SPLIT) that deals the remaining tiles' k-blocks to every CTA and adds each
// tile's parts in a fixed order (split_plan.cuh holds the schedule).
#include "gbr_internal.h"
#include "split_plan.cuh"

namespace gbr {

namespace {

constexpr uint32_t kABytes = kFfmaBM * kFfmaBK * 4;   // 16 KiB
constexpr uint32_t kBPanelBytes = kFfmaBK * 128;      // 32 rows x 128 B

// Consumer layouts of the 128 x 128 tile.  np: packed column pairs per thread
// (8 rows x 2 np columns).  The register split (producer warpgroup + consumers)
// must fit in what the CTA is launched with: threads x launch registers.
template <int CW>
struct Cons;
template <>
struct Cons<8> {
    static constexpr int threads = 256, np = 4;
    static constexpr uint32_t regs = 232, producer_regs = 40;
};
template <>
struct Cons<16> {
    static constexpr int threads = 512, np = 2;
    static constexpr uint32_t regs = 104, producer_regs = 64;
};
template <int CW>
constexpr int kThreads = 128 + Cons<CW>::threads;

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
//
// NP = 2 (the 16-warp layout): columns 4 tx .. 4 tx + 3 only, one B pair load.
template <int NP>
__device__ __forceinline__ void ffma_stage(uint64_t (&acc)[8][NP], const uint8_t* As,
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
            uint64_t bj[NP];
            bj[0] = b0.x;
            bj[1] = b0.y;
            if (NP == 4) {
                const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(bp + 2 * kBPanelBytes);
                bj[NP > 2 ? 2 : 0] = b1.x;
                bj[NP > 2 ? 3 : 1] = b1.y;
            }
            uint64_t a2[8];
#pragma unroll
            for (int r = 0; r < 8; ++r)
                a2[r] = ptx::f32x2_splat(kk == 0 ? a[r].x : kk == 1 ? a[r].y : kk == 2 ? a[r].z : a[r].w);
            // Column pair outer, row inner: eight independent FMAs share one B
            // pair (measured 4% faster than the row-outer order).
#pragma unroll
            for (int j = 0; j < NP; ++j)
#pragma unroll
                for (int r = 0; r < 8; ++r) ptx::fma_f32x2(acc[r][j], a2[r], bj[j]);
        }
    }
}

template <int NP>
__device__ __forceinline__ void ffma_zero(uint64_t (&acc)[8][NP]) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
        for (int j = 0; j < NP; ++j) acc[r][j] = 0ull;
}

__device__ __forceinline__ void ffma_tables(uint32_t tx, uint32_t ty, uint32_t& a_row,
                                            uint32_t& a_ph, uint32_t (&b_sw)[8]) {
    a_row = ty * 128u;
    a_ph = ty & 7u;
#pragma unroll
    for (uint32_t j = 0; j < 8; ++j)
        b_sw[j] = (tx >> 3) * kBPanelBytes + (((tx & 7u) ^ j) << 4);  // column 4 tx, K row % 8 = j
}

// Thread (tx, ty) of consumer `ct` in the CW-warp layout.  CW = 8: 16 x 16
// threads, tx fastest.  CW = 16: 32 x 16 threads, each warp 8 tx x 4 ty, so
// that one warp's A reads touch 4 rows (distinct swizzle phases) and its B
// reads 8 chunks of one 128-byte panel row: one wavefront each.
template <int CW>
__device__ __forceinline__ void ffma_thread(uint32_t ct, uint32_t& tx, uint32_t& ty) {
    if (CW == 8) {
        tx = ct & 15u;
        ty = ct >> 4;
    } else {
        const uint32_t w = ct >> 5, l = ct & 31u;
        tx = 8u * (w >> 2) + (l & 7u);
        ty = 4u * (w & 3u) + (l >> 3);
    }
}

// C = max(0, acc + bias) for the thread's 8 x (2 NP) outputs of tile (mt, nt):
// rows ty + 16 r, columns 4 tx + 64 h + (0..3).
template <int NP>
__device__ __forceinline__ void ffma_epilogue(const uint64_t (&acc)[8][NP], const GemmShape& p,
                                              uint32_t mt, uint32_t nt, uint32_t tx, uint32_t ty) {
    float* C = static_cast<float*>(p.C);
    const int n0 = int(nt) * kFfmaBN, m0 = int(mt) * kFfmaBM;
#pragma unroll
    for (int h = 0; h < NP / 2; ++h) {
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

// Item j of this CTA: the whole tile blockIdx.x + j * gridDim.x of
// [0, num_tiles), or (SPLIT) the CTA's run of k-blocks of the split tail,
// which meets at most two tiles (the schedule of split_plan.cuh; the whole
// tiles before it run in a separate launch).
template <bool SPLIT>
__device__ __forceinline__ bool ffma_item(const GemmShape& p, uint32_t j, WorkItem& w) {
    if (!SPLIT) {
        w.tile = blockIdx.x + j * gridDim.x;
        w.kb0 = 0;
        w.kb1 = p.num_kb;
        w.part = 0;
        w.parts = 1;
        w.sk = 0;
        return w.tile < uint32_t(p.num_tiles);
    }
    return work_item(p, blockIdx.x, gridDim.x, j + uint32_t(p.dp_tiles) / gridDim.x, w);
}

// Tile w.tile is split along K among w.parts CTAs.  Each CTA stores its fp32
// part in its own 128 x 128 slot.  Every consumer warp owns a fixed set of the
// tile's elements in every CTA and counts its arrival on its own counter; the
// warp whose arrival completes a count adds that warp region's parts in part
// order (so the result does not depend on which CTA arrives last), then
// applies bias and ReLU.  No warp waits for another warp or CTA, so a warp
// that left its loop after a timeout cannot hold up the rest.
template <int CW, int NP>
__device__ __forceinline__ void ffma_split_epilogue(const uint64_t (&acc)[8][NP],
                                                    const GemmShape& p, const WorkItem& w,
                                                    uint32_t mt, uint32_t nt, uint32_t tx,
                                                    uint32_t ty, uint32_t ct) {
    constexpr uint32_t kSlot = kFfmaBM * kFfmaBN;
    float* slots = p.sk_sum + size_t(w.sk) * size_t(kSplitMaxParts) * kSlot;
    float* mine = slots + size_t(w.part) * kSlot;
#pragma unroll
    for (int h = 0; h < NP / 2; ++h)
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const uint64_t lo = acc[r][2 * h], hi = acc[r][2 * h + 1];
            __stcg(reinterpret_cast<float4*>(mine + (ty + 16u * r) * kFfmaBN + 4u * tx + 64u * h),
                   make_float4(__uint_as_float(uint32_t(lo)), __uint_as_float(uint32_t(lo >> 32)),
                               __uint_as_float(uint32_t(hi)), __uint_as_float(uint32_t(hi >> 32))));
        }
    __threadfence();
    __syncwarp();
    uint32_t arrived = 0;
    if ((ct & 31u) == 0)
        arrived = atomicAdd(p.sk_count + size_t(w.sk) * kFfmaMaxConsumerWarps + (ct >> 5), 1u) + 1u;
    arrived = __shfl_sync(0xffffffffu, arrived, 0);
    if (arrived != uint32_t(w.parts)) return;
    __threadfence();
    uint64_t sum[8][NP];
#pragma unroll
    for (int h = 0; h < NP / 2; ++h)
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const size_t off = (ty + 16u * r) * kFfmaBN + 4u * tx + 64u * h;
            float4 t = __ldcg(reinterpret_cast<const float4*>(slots + off));
            for (int q = 1; q < w.parts; ++q) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(slots + q * kSlot + off));
                t.x += v.x;
                t.y += v.y;
                t.z += v.z;
                t.w += v.w;
            }
            sum[r][2 * h] = uint64_t(__float_as_uint(t.x)) | (uint64_t(__float_as_uint(t.y)) << 32);
            sum[r][2 * h + 1] = uint64_t(__float_as_uint(t.z)) | (uint64_t(__float_as_uint(t.w)) << 32);
        }
    ffma_epilogue(sum, p, mt, nt, tx, ty);
}

// CPASYNC = false: one TMA lane produces each stage (the default).
// CPASYNC = true: the historical producer ("gpu_warp_specialization" and
// "pwwt.cn news/4436243" section 2: Ampere cp.async): the whole producer
// warpgroup copies the stage with 16-byte cp.async per thread into the same
// swizzled layout, and each of its 128 threads arrives on full[s] with
// cp.async.mbarrier.arrive.noinc once its own copies have landed.
// SPLIT (TMA producer only): the launch runs the split tail of the schedule
// instead of whole tiles; a separate instance, so that the whole-tile kernel
// keeps its register allocation.
template <int CW, bool CPASYNC, bool SPLIT = false>
__global__ void __launch_bounds__(kThreads<CW>, 1)
    gemm_ffma_kernel(const __grid_constant__ CUtensorMap mapA,
                     const __grid_constant__ CUtensorMap mapB, const GemmShape p) {
    using L = Cons<CW>;
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
            ptx::mbar_init(ptx::smem_addr(empty + s), CW);
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
        ptx::setmaxnreg_dec<L::producer_regs>();
        if (CPASYNC) {
            // ------------------------------------ cp.async producer warpgroup
            const uint32_t pt = threadIdx.x;   // 0..127
            const float* A = static_cast<const float*>(p.A);
            const float* B = static_cast<const float*>(p.B);
            uint32_t i = 0, ntr = 0;
            bool ok = true;
            WorkItem w;
            for (uint32_t j = 0; ok && ffma_item<SPLIT>(p, j, w); ++j) {
                uint32_t mt, nt;
                raster_tile(w.tile, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
                const int m0 = int(mt) * kFfmaBM, n0 = int(nt) * kFfmaBN;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++i) {
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
            WorkItem w;
            for (uint32_t j = 0; ok && ffma_item<SPLIT>(p, j, w); ++j) {
                uint32_t mt, nt;
                raster_tile(w.tile, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++i) {
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
        ptx::setmaxnreg_inc<L::regs>();
        // ---------------------------------------------------- consumers
        // Thread (tx, ty) owns rows ty + 16 r (r = 0..7) and columns
        // 4 tx .. 4 tx + 3 (and, at CW = 8, 64 + 4 tx .. 64 + 4 tx + 3) of the
        // 128 x 128 tile.  All its rows have the same (row % 8), so every A
        // read of a k-group uses one swizzle phase; all its columns sit at the
        // same position inside their 32-column panels, so every B read of a k
        // uses one phase too.  The phases come from two 8-entry tables and
        // every shared-memory load is base + immediate offset.
        const uint32_t ct = threadIdx.x - 128;
        uint32_t tx, ty;
        ffma_thread<CW>(ct, tx, ty);
        uint32_t a_row, a_ph, b_sw[8];
        ffma_tables(tx, ty, a_row, a_ph, b_sw);

        uint32_t i = 0, ntr = 0;
        const bool tracer = p.ctl.trace != nullptr && warp == 4 && lane == 0;   // one consumer lane
        bool ok = true;
        WorkItem w;
        for (uint32_t j = 0; ok && ffma_item<SPLIT>(p, j, w); ++j) {
            uint32_t mt, nt;
            raster_tile(w.tile, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
            uint64_t acc[8][L::np];
            ffma_zero(acc);

            for (int kb = w.kb0; kb < w.kb1; ++kb, ++i) {
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

            if (SPLIT)
                ffma_split_epilogue<CW>(acc, p, w, mt, nt, tx, ty, ct);
            else
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
// Threads per CTA: the CW consumer layout's (256: 2 CTAs per SM, 512: 1).
template <int CW>
__global__ void __launch_bounds__(Cons<CW>::threads, CW == 8 ? 2 : 1)
    gemm_ffma_sync_kernel(const float* __restrict__ A, const float* __restrict__ B,
                          const GemmShape p) {
    constexpr int kSyncThreads = Cons<CW>::threads;
    constexpr int kLoads = 1024 / kSyncThreads;   // 16-byte chunks of A (and of B) per thread
    __shared__ __align__(1024) uint8_t tile[kFfmaStageBytes];
    uint8_t* As = tile;
    uint8_t* Bs = tile + kABytes;
    const uint32_t t = threadIdx.x;
    uint32_t tx, ty;
    ffma_thread<CW>(t, tx, ty);
    uint32_t mt, nt;
    raster_tile(blockIdx.x, p.m_tiles, p.n_tiles, p.group_m, mt, nt);
    const int m0 = int(mt) * kFfmaBM, n0 = int(nt) * kFfmaBN;
    uint32_t a_row, a_ph, b_sw[8];
    ffma_tables(tx, ty, a_row, a_ph, b_sw);
    uint64_t acc[8][Cons<CW>::np];
    ffma_zero(acc);

    for (int kb = 0; kb < p.num_kb; ++kb) {
        const int k0 = kb * kFfmaBK;
        // load: kLoads float4 of A (row idx/8, 16-byte chunk idx%8) and of B
        // (K row idx/32, 16-byte chunk idx%32) per thread, zero outside the
        // matrix, stored in the same swizzled layout the TMA path produces.
#pragma unroll
        for (int j = 0; j < kLoads; ++j) {
            const uint32_t idx = t + kSyncThreads * j;
            const uint32_t row = idx >> 3, k4 = idx & 7u;
            const int m = m0 + int(row), k = k0 + int(4 * k4);
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m < p.M && k < p.K) v = __ldg(reinterpret_cast<const float4*>(A + size_t(m) * p.K + k));
            *reinterpret_cast<float4*>(As + row * 128u + ((k4 ^ (row & 7u)) << 4)) = v;
        }
#pragma unroll
        for (int j = 0; j < kLoads; ++j) {
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

int g_ffma_warps = 8;    // consumer warps of the FFMA kernels (8 or 16)
std::mutex g_ffma_mu;

int ffma_warps_now() {
    std::lock_guard<std::mutex> lk(g_ffma_mu);
    return g_ffma_warps;
}

template <int CW>
const void* ffma_fn(bool cpasync, bool split = false) {
    if (split) return reinterpret_cast<const void*>(gemm_ffma_kernel<CW, false, true>);
    return cpasync ? reinterpret_cast<const void*>(gemm_ffma_kernel<CW, true>)
                   : reinterpret_cast<const void*>(gemm_ffma_kernel<CW, false>);
}

}  // namespace

int ffma_consumer_warps() { return ffma_warps_now(); }

int ffma_set_consumer_warps(int cw) {
    if (cw != 8 && cw != 16) return -1;
    std::lock_guard<std::mutex> lk(g_ffma_mu);
    g_ffma_warps = cw;
    return 0;
}

cudaError_t launch_gemm_ffma_sync(const float* A, const float* B, const GemmShape& s,
                                  cudaStream_t stream) {
    if (ffma_warps_now() == 16)
        gemm_ffma_sync_kernel<16><<<s.num_tiles, Cons<16>::threads, 0, stream>>>(A, B, s);
    else
        gemm_ffma_sync_kernel<8><<<s.num_tiles, Cons<8>::threads, 0, stream>>>(A, B, s);
    return cudaGetLastError();
}

size_t ffma_smem_bytes(int stages) {
    return 1024 + size_t(stages) * kFfmaStageBytes + size_t(2 * stages) * 8 + 16;   // + flags
}

cudaError_t ffma_prepare(size_t smem) {
    static std::mutex mu;
    static size_t set[kMaxDeviceSlots][6] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDeviceSlots) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    const void* fns[6] = {ffma_fn<8>(false), ffma_fn<8>(true), ffma_fn<16>(false),
                          ffma_fn<16>(true), ffma_fn<8>(false, true), ffma_fn<16>(false, true)};
    for (int i = 0; i < 6; ++i)
        if ((e = raise_smem_limit(fns[i], smem, &set[dev][i])) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t ffma_occupancy(size_t smem, int* blocks_per_sm) {
    if (ffma_warps_now() == 16)
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            blocks_per_sm, gemm_ffma_kernel<16, false>, kThreads<16>, smem);
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, gemm_ffma_kernel<8, false>,
                                                         kThreads<8>, smem);
}

// The register split must fit in what the CTA is launched with, or the
// consumers' setmaxnreg.inc would wait forever for registers.
template <int CW>
cudaError_t ffma_check_registers_cw(int* regs) {
    const long need = 128L * Cons<CW>::producer_regs + long(Cons<CW>::threads) * Cons<CW>::regs;
    for (const void* fn : {ffma_fn<CW>(false), ffma_fn<CW>(true), ffma_fn<CW>(false, true)}) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, fn);
        if (e != cudaSuccess) return e;
        *regs = fa.numRegs;
        if (long(fa.numRegs) * kThreads<CW> < need) return cudaErrorInvalidConfiguration;
    }
    return cudaSuccess;
}

cudaError_t ffma_check_registers(int* regs) {
    cudaError_t e = ffma_check_registers_cw<8>(regs);
    if (e != cudaSuccess) return e;
    return ffma_check_registers_cw<16>(regs);
}

cudaError_t launch_gemm_ffma(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmShape& s,
                             int grid, size_t smem, cudaStream_t stream, bool cpasync, bool split) {
    const int cw = ffma_warps_now();
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(cw == 16 ? kThreads<16> : kThreads<8>);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = programmatic_launch_attr(attr);
    cfg.attrs = attr;
    if (split) {
        if (cw == 16) return cudaLaunchKernelEx(&cfg, gemm_ffma_kernel<16, false, true>, mapA, mapB, s);
        return cudaLaunchKernelEx(&cfg, gemm_ffma_kernel<8, false, true>, mapA, mapB, s);
    }
    if (cw == 16) {
        if (cpasync) return cudaLaunchKernelEx(&cfg, gemm_ffma_kernel<16, true>, mapA, mapB, s);
        return cudaLaunchKernelEx(&cfg, gemm_ffma_kernel<16, false>, mapA, mapB, s);
    }
    if (cpasync) return cudaLaunchKernelEx(&cfg, gemm_ffma_kernel<8, true>, mapA, mapB, s);
    return cudaLaunchKernelEx(&cfg, gemm_ffma_kernel<8, false>, mapA, mapB, s);
}

}  // namespace gbr
