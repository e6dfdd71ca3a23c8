// gbr_common.cuh -- pieces shared by every pipeline kernel: the bounded
// mbarrier wait, the device status block and the persistent tile order.
#pragma once
#include <cstdint>
#include "gbr_ptx.cuh"

namespace gbr {

// Device status block, one per device (kStatusWords 32-bit words):
//   [0] error bits (kDevErrTimeout), [1] code of the first wait that gave up,
//   [2] its CTA index, [3] its item/iteration index.
constexpr int kStatusWords = 16;
constexpr uint32_t kDevErrTimeout = 1u;

// Wait-site codes recorded in status[1] (role << 4 | which barrier).
enum WaitSite : uint32_t {
    kSiteProducerEmpty = 0x11,
    kSiteProducerDrain = 0x12,
    kSiteProducerTile = 0x13,
    kSiteConsumerFull = 0x21,
    kSiteMmaFull = 0x31,
    kSiteMmaAccEmpty = 0x32,
    kSiteMmaDrain = 0x33,
    kSiteMmaTile = 0x34,
    kSiteEpiAccFull = 0x41,
    kSiteEpiSplitSum = 0x42,
    kSiteEpiTile = 0x43,
    kSiteEpiBias = 0x44,
    kSiteStorerFull = 0x51,
    kSiteSelfTest = 0x71,
};

// Optional event trace (null: off).  Layout of the trace buffer:
//   [kTraceMaxCtas][kTraceRoles] uint32 event counts (kTraceHeaderBytes), then
//   per (CTA, role) a region of trace_cap 16-byte records
//   { uint64 %globaltimer, uint32 item, uint8 role, event, slot, parity }.
// A role counts every event; it writes the first trace_cap of them.
constexpr uint32_t kTraceMaxCtas = 512;
constexpr uint32_t kTraceRoles = 4;
constexpr size_t kTraceHeaderBytes = size_t(kTraceMaxCtas) * kTraceRoles * 4;
enum TraceRole : uint32_t {
    kRoleProducer = 0,   // ring producer: waits on empty, issues TMA
    kRoleConsumer = 1,   // ring consumer: FFMA warp, MMA lane or copy storer
    kRoleEpilogue = 2,   // tcgen05 epilogue warp: waits on acc_full, frees acc_empty
    kRoleMmaAcc = 3,     // tcgen05 MMA lane on the accumulator ring
};
enum TraceEvent : uint32_t {
    kEvWaitDone = 0,     // a wait returned: (item, slot, parity waited on)
    kEvIssued = 1,       // producer issued the stage's loads / MMA lane committed a tile
    kEvReleased = 2,     // the slot's release is issued (arrive or commit follows)
};

struct KernelCtl {
    uint32_t* status = nullptr;      // device status block (kStatusWords words)
    uint64_t timeout_ns = 0;         // per-wait limit on %globaltimer
    uint8_t* trace = nullptr;        // event trace buffer, or null
    uint32_t trace_cap = 0;          // records per (CTA, role)
};

// Records one event of `role` (n: that role's running count in this CTA).
__device__ __forceinline__ void trace_event(const KernelCtl& c, uint32_t role, uint32_t& n,
                                            uint32_t ev, uint32_t item, uint32_t slot,
                                            uint32_t parity) {
    if (c.trace == nullptr || blockIdx.x >= kTraceMaxCtas) return;
    if (n < c.trace_cap) {
        const uint64_t t = ptx::globaltimer();
        uint4 v;
        v.x = uint32_t(t);
        v.y = uint32_t(t >> 32);
        v.z = item;
        v.w = role | (ev << 8) | ((slot & 0xFFu) << 16) | ((parity & 0xFFu) << 24);
        reinterpret_cast<uint4*>(c.trace + kTraceHeaderBytes)
            [(size_t(blockIdx.x) * kTraceRoles + role) * c.trace_cap + n] = v;
    }
    ++n;
}

// Publishes a role's event count for this CTA.
__device__ __forceinline__ void trace_count(const KernelCtl& c, uint32_t role, uint32_t n) {
    if (c.trace != nullptr && blockIdx.x < kTraceMaxCtas)
        reinterpret_cast<uint32_t*>(c.trace)[blockIdx.x * kTraceRoles + role] = n;
}

// Iteration cap of one bounded wait; the time limit normally ends it first.
constexpr uint32_t kMaxPollIters = 1u << 26;

__device__ __forceinline__ void record_timeout(const KernelCtl& ctl, uint32_t site, uint32_t item) {
    atomicOr(ctl.status + 0, kDevErrTimeout);
    if (atomicCAS(ctl.status + 1, 0u, site) == 0u) {
        ctl.status[2] = blockIdx.x;
        ctl.status[3] = item;
    }
}

// One poll of a barrier phase; CLUSTER selects cluster-scope acquire, for
// barriers that receive arrivals or commits from the other CTA of a pair.
template <bool CLUSTER>
__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {
    return CLUSTER ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
}

// Non-blocking poll (never suspends the thread).
template <bool CLUSTER>
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    return CLUSTER ? ptx::mbar_test_wait_cluster(bar, parity) : ptx::mbar_test_wait(bar, parity);
}

// Slow path of a bounded wait: polls until the phase completes, another role
// raised the CTA's abort flag, or the time/iteration limit runs out (then it
// records the site, raises the abort flag and gives up).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, const KernelCtl& ctl,
                                               volatile int* abort_flag, uint32_t site,
                                               uint32_t item) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t iter = 0; iter < kMaxPollIters; ++iter) {
        if (mbar_poll<CLUSTER>(bar, parity)) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > ctl.timeout_ns) break;
    }
    *abort_flag = 1;
    record_timeout(ctl, site, item);
    return false;
}

// Bounded wait for the phase of `bar` with the given parity to complete.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const KernelCtl& ctl,
                                          volatile int* abort_flag, uint32_t site, uint32_t item) {
    if (mbar_poll<CLUSTER>(bar, parity)) return true;
    return mbar_wait_slow<CLUSTER>(bar, parity, ctl, abort_flag, site, item);
}

// The same wait taken by all 32 lanes of a warp.  The outcome is made
// warp-uniform, so a warp never splits into lanes that carry on and lanes that
// abort (the warp-wide .sync.aligned instructions that follow need every lane).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, const KernelCtl& ctl,
                                               volatile int* abort_flag, uint32_t site,
                                               uint32_t item) {
    const bool ok = mbar_wait<CLUSTER>(bar, parity, ctl, abort_flag, site, item);
    return __all_sync(0xffffffffu, ok);
}

// Wait used only while tearing down after an abort: bounded, records nothing
// new and ignores the abort flag (it waits for this CTA's own copies in flight).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t iter = 0; iter < kMaxPollIters; ++iter) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (ptx::globaltimer() - t0 > limit_ns) return false;
    }
    return false;
}

// Bounded wait (one thread) until the global counter reaches `target`; the
// writers are CTAs of the same launch that have already started, and they
// increment the counter without waiting on anything.
__device__ __forceinline__ bool counter_wait(const uint32_t* counter, uint32_t target,
                                             const KernelCtl& ctl, volatile int* abort_flag,
                                             uint32_t site, uint32_t item) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t iter = 0; iter < kMaxPollIters; ++iter) {
        if (ptx::ld_acquire_gpu_u32(counter) >= target) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > ctl.timeout_ns) break;
        __nanosleep(100);
    }
    *abort_flag = 1;
    record_timeout(ctl, site, item);
    return false;
}

// Persistent tile order over an (m_tiles x n_tiles) grid of output tiles:
// bands of `group_m` tile rows, column-major inside a band, so that the CTAs
// running at the same time share A rows and B columns in L2.
__device__ __forceinline__ void raster_tile(uint32_t t, uint32_t m_tiles, uint32_t n_tiles,
                                            uint32_t group_m, uint32_t& mt, uint32_t& nt) {
    const uint32_t band = group_m * n_tiles;
    const uint32_t g = t / band;
    const uint32_t first_m = g * group_m;
    const uint32_t rows = min(group_m, m_tiles - first_m);
    const uint32_t r = t - g * band;
    mt = first_m + r % rows;
    nt = r / rows;
}

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace gbr
