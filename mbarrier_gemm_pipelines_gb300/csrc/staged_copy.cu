// staged_copy.cu -- TMA gmem -> smem -> gmem copy through an S-slot ring.
//
// "Producer-Consumer Warp Specialization for TMA Operations": a TMA load puts
// each tile into a shared-memory staging buffer and a TMA store drains it to
// HBM; every buffer has a "full" mbarrier (tripped as data flows in) and an
// "empty" mbarrier (tripped as data flows out); the buffer and the waited
// phase parity of tile i follow from i alone.  Here the ring has S slots:
//   slot        = i % S
//   full  wait  = parity (i / S) & 1          (the loader's data has landed)
//   empty wait  = parity ((i / S) & 1) ^ 1    (the previous occupant was drained;
//                                              on the first lap this names the
//                                              phase before a fresh barrier,
//                                              which counts as complete)
// One lane of warp 0 loads, one lane of warp 1 stores.  CTAs are persistent:
// CTA b copies tiles b, b + grid, b + 2 grid, ... so i is the CTA-local count.
// Slots are copy_slot_bytes() apart: a TMA copy's shared-memory address must
// be 128-byte aligned, and a tile may be any multiple of 16 bytes.
#include "gbr_internal.h"

namespace gbr {

namespace {

__global__ void __launch_bounds__(64, 1)
    staged_copy_kernel(const __grid_constant__ CUtensorMap src_map,
                       const __grid_constant__ CUtensorMap dst_map, const CopyArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* ring = align_1024(smem_raw);
    const int S = a.stages;
    const uint32_t slot_bytes = copy_slot_bytes(a.tile_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + size_t(S) * slot_bytes);
    uint64_t* empty = full + S;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + S);

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(ptx::smem_addr(full + s), 1);   // producer's arrive + tx bytes
            ptx::mbar_init(ptx::smem_addr(empty + s), 1);  // storer's release
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    } else if (threadIdx.x == 32) {
        ptx::prefetch_tensormap(&src_map);
        ptx::prefetch_tensormap(&dst_map);
    }
    __syncthreads();
    // Everything above overlaps the end of the previous kernel in the stream;
    // nothing below touches global memory before that kernel is done.
    ptx::griddep_wait();

    const uint32_t ring_base = ptx::smem_addr(ring);
    // Every byte is read once and written once: optionally tell L2 to evict
    // these lines first, so they do not push out lines that will be reused.
    const bool hint_load = (a.l2_hint & 1u) != 0, hint_store = (a.l2_hint & 2u) != 0;
    uint32_t issued = 0;   // load lane: ring items registered on full[]
    if (warp == 0 && lane == 0) {
        // ---------------- producer: wait empty -> expect_tx -> TMA load
        uint32_t i = 0, nt = 0;
        for (int64_t t = blockIdx.x; t < a.num_tiles; t += gridDim.x, ++i) {
            const uint32_t s = i % S, ph = (i / S) & 1u;
            if (!mbar_wait(ptx::smem_addr(empty + s), ph ^ 1u, a.ctl, abort_flag,
                           kSiteProducerEmpty, i))
                break;
            trace_event(a.ctl, kRoleProducer, nt, kEvWaitDone, i, s, ph ^ 1u);
            const uint32_t fb = ptx::smem_addr(full + s);
            ptx::mbar_arrive_expect_tx(fb, a.tile_bytes);
            if (inject_skip(a.inject, i)) continue;   // self test: this stage never fills
            trace_event(a.ctl, kRoleProducer, nt, kEvIssued, i, s, 0);   // before the load lands
            const int32_t tr = int32_t(t / a.tiles_c), tc = int32_t(t % a.tiles_c);
            if (hint_load)
                ptx::tma_load_2d_hint(ring_base + s * slot_bytes, &src_map, fb, tc * a.tile_cols,
                                      tr * a.tile_rows, ptx::l2_policy_evict_first());
            else
                ptx::tma_load_2d(ring_base + s * slot_bytes, &src_map, fb, tc * a.tile_cols,
                                 tr * a.tile_rows);
        }
        trace_count(a.ctl, kRoleProducer, nt);
        ptx::griddep_launch_dependents();   // every load issued: the next launch may be scheduled
        issued = i;
    } else if (warp == 1 && lane == 0) {
        // ---------------- storer: wait full -> TMA store -> release when read
        uint32_t i = 0, nt = 0;
        for (int64_t t = blockIdx.x; t < a.num_tiles; t += gridDim.x, ++i) {
            const uint32_t s = i % S, ph = (i / S) & 1u;
            if (!mbar_wait(ptx::smem_addr(full + s), ph, a.ctl, abort_flag, kSiteStorerFull, i))
                break;
            trace_event(a.ctl, kRoleConsumer, nt, kEvWaitDone, i, s, ph);
            const int32_t tr = int32_t(t / a.tiles_c), tc = int32_t(t % a.tiles_c);
            if (hint_store)
                ptx::tma_store_2d_hint(&dst_map, ring_base + s * slot_bytes, tc * a.tile_cols,
                                       tr * a.tile_rows, ptx::l2_policy_evict_first());
            else
                ptx::tma_store_2d(&dst_map, ring_base + s * slot_bytes, tc * a.tile_cols,
                                  tr * a.tile_rows);
            ptx::bulk_commit_group();
            if (a.store_lag == 0) {
                ptx::bulk_wait_group_read<0>();
                trace_event(a.ctl, kRoleConsumer, nt, kEvReleased, i, s, 0);
                ptx::mbar_arrive(ptx::smem_addr(empty + s));
            } else {
                ptx::bulk_wait_group_read<1>();
                if (i > 0) {
                    trace_event(a.ctl, kRoleConsumer, nt, kEvReleased, i - 1, (i - 1) % S, 0);
                    ptx::mbar_arrive(ptx::smem_addr(empty + (i - 1) % S));
                }
            }
        }
        trace_count(a.ctl, kRoleConsumer, nt);
        ptx::bulk_wait_group<0>();
    }
    __syncwarp();
    __syncthreads();
    // Both lanes have left their loops, so the abort flag is final.  After an
    // abort the load lane lets its own loads still in flight land (the last S
    // items it registered, except a self test's unissued one) before the CTA
    // may exit.
    if (warp == 0 && lane == 0 && *abort_flag) {
        const uint32_t n = issued < uint32_t(S) ? issued : uint32_t(S);
        for (uint32_t j = issued - n; j < issued; ++j)
            if (!inject_skip(a.inject, j))
                mbar_wait_drain(ptx::smem_addr(full + j % S), (j / S) & 1u, a.ctl.timeout_ns);
    }
    __syncthreads();
}

}  // namespace

size_t copy_smem_bytes(int stages, uint32_t tile_bytes) {
    return 1024 + size_t(stages) * copy_slot_bytes(tile_bytes) + size_t(2 * stages) * 8 + 16;
}

cudaError_t copy_prepare(size_t smem) {
    static std::mutex mu;
    static size_t set[kMaxDeviceSlots] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDeviceSlots) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    return raise_smem_limit(reinterpret_cast<const void*>(staged_copy_kernel), smem, &set[dev]);
}

cudaError_t copy_occupancy(size_t smem, int* blocks_per_sm) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, staged_copy_kernel, 64,
                                                         smem);
}

cudaError_t launch_staged_copy(const CUtensorMap& src, const CUtensorMap& dst, const CopyArgs& a,
                               int grid, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(64);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = programmatic_launch_attr(attr);
    cfg.attrs = attr;
    return cudaLaunchKernelEx(&cfg, staged_copy_kernel, src, dst, a);
}

}  // namespace gbr
