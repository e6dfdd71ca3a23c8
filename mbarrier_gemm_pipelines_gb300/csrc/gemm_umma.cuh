// gemm_umma.cuh -- warp-specialized, persistent tensor-core GEMM + bias + ReLU
// for sm_103a (tcgen05 MMA into Tensor Memory), bf16 or TF32 inputs, one CTA
// per output tile (PAIR = 1) or a CTA pair per tile (PAIR = 2).  The kernel
// template; each gemm_umma_<kind>.cu instantiates the instances of one kind
// (so that they compile in parallel) and gemm_umma.cu holds the host side.
//
// Method ("gpu_warp_specialization", "The architecture: every piece
// explained" and "End-to-end flow"; "pwwt.cn news/4436243", sections 3.2-3.4
// and 4.1): a block owns output tiles; producer warps stream the K tiles of A
// and B into a multi-stage shared-memory ring with asynchronous copies, each
// stage guarded by a "full" and an "empty" barrier; the math role waits for a
// full stage, runs the matrix multiply-accumulate on it and marks it empty; a
// fused epilogue adds the bias and applies ReLU.
//
// What the sm_103a version keeps and changes:
//   * TMA producer: one lane of warp 0, `cp.async.bulk.tensor` with
//     expect_tx on full[s] (the copy engine completes the phase).
//   * The math role is ONE elected lane (warp 1) issuing tcgen05.mma: the
//     accumulator lives in Tensor Memory, not registers, so a single thread
//     drives the tensor core; `tcgen05.commit` arrives on empty[s] when the
//     MMAs that read stage s have finished (no consumer thread has to arrive).
//   * The accumulator is double-buffered in TMEM (2 x 256 columns): the
//     epilogue warps (warps 4-7, one TMEM lane quarter each) drain tile j
//     while the MMA lane accumulates tile j+1.  acc_full/acc_empty form a
//     second 2-slot ring with the same slot/parity rule.
//   * Epilogue: tcgen05.ld -> +bias -> ReLU -> (bf16 round-to-nearest-even)
//     -> 128-byte swizzled st.shared -> TMA store, per warp, double-buffered.
//     The tile's bias is staged in shared memory by one cp.async.bulk per
//     tile (a one-slot ring of its own, bias_full / bias_empty).
//   * Persistent CTAs walk tiles t = unit + j * units in banded order; every
//     role walks the same sequence, and the k-iteration counter runs across
//     tiles so phases carry over.
//   * Registers move from warpgroup 0 (producer / MMA / TMEM allocator) to the
//     epilogue warpgroup with setmaxnreg.
//
// PAIR = 2 (a cluster of two CTAs on the two SMs of a TPC, 256 x 256 tiles):
// each CTA loads its own 128 rows of A and its own 128 columns of B, so the
// shared-memory bytes written by TMA and read by the tensor core per SM are
// half those of a one-SM 128 x 256 tile for the same MMA work.  The even CTA
// (rank 0) owns the ring's full barriers and the accumulator's empty
// barriers: both CTAs' TMA loads complete on the even CTA's full[s] (the even
// CTA alone registers the pair's bytes with expect_tx), the even CTA's lane
// issues the M = 256 MMAs, and its commits multicast to empty[s] and
// acc_full[a] of both CTAs; the epilogue warps of both CTAs arrive on the even
// CTA's acc_empty[a] (8 arrivals).  Each CTA drains its own 128 rows of the
// accumulator from its own TMEM.
//
// Shared-memory ring stage (every kind: 128 bytes of K per row):
//   A: 128 rows (M) x 128 B, K-major, TMA 128-byte swizzle      16 KiB
//   B: 256 / PAIR columns of this CTA, N-major panels of 128 B of N read
//      straight from B[K, N] (MN-major operand):
//      bf16: 64 rows (K) x 64 columns, TMA 128-byte swizzle       8 KiB each
//      tf32: 32 rows (K) x 32 columns, TMA 128-byte swizzle with
//            32-byte atoms (the only MN-major form kind::tf32 reads)  4 KiB each
//   PAIR = 1: 48 KiB per stage, PAIR = 2: 32 KiB per stage.
// kind     BK  MMA K
// bf16     64   16
// tf32     32    8
#pragma once
#include "gbr_internal.h"
#include "split_plan.cuh"

#include <cuda_bf16.h>

namespace gbr {

namespace umma {

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kRegsWG0 = 88;
constexpr uint32_t kRegsWG1 = 224;
constexpr uint32_t kEpiBufBytes = 32 * 128;   // 32 rows x 128 B per warp buffer

// Layout field of a shared-memory matrix descriptor (see sw128_desc).
constexpr uint32_t kDescSw128 = 2, kDescSw128Atom32 = 1;

template <int KIND>
struct Kind;
template <>
struct Kind<kUmmaBf16> {
    static constexpr uint32_t esize = 2, bk = 64, mma_k = 16, panel_cols = 64;
    static constexpr uint32_t ab_format = 1;          // BF16
    static constexpr uint32_t out_chunk_cols = 64;    // 64 bf16 = 128 B per row
    // MN-major B: 128-byte swizzle, 8-row K groups 1024 B apart.
    static constexpr uint32_t b_layout = kDescSw128, b_sbo = 1024;
};
template <>
struct Kind<kUmmaTf32> {
    static constexpr uint32_t esize = 4, bk = 32, mma_k = 8, panel_cols = 32;
    static constexpr uint32_t ab_format = 2;          // TF32
    static constexpr uint32_t out_chunk_cols = 32;    // 32 fp32 = 128 B per row
    // MN-major B: 128-byte swizzle of 32-byte atoms, 4-row K groups 512 B apart.
    static constexpr uint32_t b_layout = kDescSw128Atom32, b_sbo = 512;
};

template <int PAIR>
struct Pair {
    static constexpr uint32_t tile_m = 128 * PAIR;           // rows per output tile
    static constexpr uint32_t b_cols = kUmmaBN / PAIR;       // B columns held per CTA
    static constexpr uint32_t b_bytes = b_cols * 128;        // B bytes per CTA per stage
    static constexpr uint32_t stage_bytes = kUmmaAStageBytes + b_bytes;
};

// Instruction descriptor, kind::f16 / kind::tf32: fp32 accumulator, A K-major,
// B MN-major, M = 128 * PAIR, N = 256, dense.
template <int KIND, int PAIR>
__host__ __device__ constexpr uint32_t make_idesc() {
    return (1u << 4)                                     // D format: f32
           | (Kind<KIND>::ab_format << 7)                // A format
           | (Kind<KIND>::ab_format << 10)               // B format
           | (0u << 15)                                  // A: K-major
           | (1u << 16)                                  // B: MN-major
           | ((uint32_t(kUmmaBN) >> 3) << 17)            // N / 8
           | ((Pair<PAIR>::tile_m >> 4) << 24);          // M / 16
}

// Shared-memory matrix descriptor, 128-byte rows.
//   bits  0-13 start address >> 4     bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4  bits 46-48 = 0b001 (tcgen05 version)
//   bits 49-51 base offset = 0 (atoms are 1024-byte aligned)
//   bits 61-63 layout: 2 = 128-byte swizzle (16-byte atoms),
//                      1 = 128-byte swizzle of 32-byte atoms
// K-major operand (A): rows 128 B apart, 8-row groups SBO = 1024 B apart, LBO
// unused; the k-th MMA of a stage starts k * 32 bytes into the row.
// MN-major B: each K row of a panel holds 128 B of N; K groups are SBO apart
// (bf16: 8 rows, 1024 B; tf32: 4 rows, 512 B) and 128-byte column panels LBO
// = panel bytes apart; the k-th MMA of a stage starts k * MMA-K rows into the
// panel.  kind::tf32 reads an MN-major operand only in the 32-byte-atom form
// (which TMA writes with CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B): measured on
// GB300, the same panels in the 16-byte-atom form give exact zeros, and with
// 32-byte atoms and 8-row groups the rows of each group come out permuted.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t layout = kDescSw128) {
    return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) |
           (uint64_t(layout) << 61);
}

// TMA loads of one operand box, one CTA or the CTA pair, with or without an
// L2 eviction-priority policy.
template <int PAIR>
__device__ __forceinline__ void load_box_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, bool hint, uint64_t pol) {
    if (PAIR == 2) {
        if (hint) ptx::tma_load_2d_pair_hint(dst, map, bar, c0, c1, pol);
        else ptx::tma_load_2d_pair(dst, map, bar, c0, c1);
    } else {
        if (hint) ptx::tma_load_2d_hint(dst, map, bar, c0, c1, pol);
        else ptx::tma_load_2d(dst, map, bar, c0, c1);
    }
}
template <int PAIR>
__device__ __forceinline__ void load_box_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1, int32_t c2, bool hint,
                                            uint64_t pol) {
    if (PAIR == 2) {
        if (hint) ptx::tma_load_3d_pair_hint(dst, map, bar, c0, c1, c2, pol);
        else ptx::tma_load_3d_pair(dst, map, bar, c0, c1, c2);
    } else {
        if (hint) ptx::tma_load_3d_hint(dst, map, bar, c0, c1, c2, pol);
        else ptx::tma_load_3d(dst, map, bar, c0, c1, c2);
    }
}

template <bool GROUPED>
struct UmmaParams {
    CUtensorMap mapA;
    CUtensorMap mapB;
    CUtensorMap mapC[GROUPED ? kMaxGroups : 1];
    GemmShape s;
    GroupTable g;
    int64_t bias_group_stride;
};

struct TileInfo {
    int32_t a_row;   // row coordinate of this CTA's A/X box
    int32_t c_row;   // row coordinate of this CTA's C rows in mapC[group] (thin: the tile's)
    int32_t n0;      // first output column of the tile
    int32_t group;
    int32_t thin;    // 0, or the rows of a transposed (thin) tile (its MMA N: rounded up to 16)
};

// Instruction descriptor of a thin tile (CTA pair, bf16): the MMA computes
// C^T = W^T X^T, with A = W^T (the tile's 256 weight columns, MN-major: the
// same N-major panels the ordinary tile reads as B) and B = X^T (the tile's
// rows, K-major: the same boxes the ordinary tile reads as A); M = 256,
// N = n_pad.
__device__ __forceinline__ uint32_t make_idesc_thin(uint32_t n_pad) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (0u << 16) | ((n_pad >> 3) << 17) |
           ((256u >> 4) << 24);
}

template <bool GROUPED, int PAIR>
__device__ __forceinline__ TileInfo decode_tile(const UmmaParams<GROUPED>& P, uint32_t t,
                                                uint32_t rank) {
    TileInfo ti;
    ti.thin = 0;
    uint32_t mt, nt;
    if (!GROUPED) {
        raster_tile(t, P.s.m_tiles, P.s.n_tiles, P.s.group_m, mt, nt);
        ti.c_row = int32_t(mt * Pair<PAIR>::tile_m + rank * 128);
        ti.a_row = ti.c_row;
        ti.group = 0;
    } else {
        int e = 0;
        while (e + 1 < P.g.num_groups && int32_t(t) >= P.g.tile_start[e + 1]) ++e;
        raster_tile(t - uint32_t(P.g.tile_start[e]), uint32_t(P.g.m_tiles[e]), P.s.n_tiles,
                    P.s.group_m, mt, nt);
        ti.c_row = int32_t(mt * Pair<PAIR>::tile_m + rank * 128);
        ti.a_row = P.g.row_off[e] + ti.c_row;
        ti.group = e;
        if (PAIR == 2 && P.g.thin[e] > 0 && int32_t(mt) + 1 == P.g.m_tiles[e]) {
            // Thin tile: the tile's rows are the MMA's N columns, half of them
            // (n_pad / 2 rows of X) from each CTA of the pair.
            ti.thin = P.g.thin[e];
            ti.c_row = int32_t(mt * Pair<PAIR>::tile_m);
            ti.a_row = P.g.row_off[e] + ti.c_row + int32_t(rank) * (((ti.thin + 15) & ~15) / 2);
        }
    }
    ti.n0 = int32_t(nt) * kUmmaBN;
    return ti;
}

// Sum of split tile sk, the block of epilogue warp q of CTA `rank`: its 32
// rows x 256 columns as [column / 4][lane] float4s, so that one warp
// instruction touches 512 contiguous bytes.
template <int PAIR>
__device__ __forceinline__ float4* sum_block(const GemmShape& s, int32_t sk, uint32_t rank,
                                             uint32_t q) {
    const size_t blk = (size_t(sk) * PAIR + rank) * 4u + q;
    return reinterpret_cast<float4*>(s.sk_sum) + blk * (kUmmaBN / 4u) * 32u;
}

// Adds columns [c, c + 32) of this lane's row to the tile's sum (at L2).
__device__ __forceinline__ void sum_add32(float4* blk, uint32_t c, uint32_t lane,
                                          const uint32_t (&r)[32]) {
#pragma unroll
    for (uint32_t i = 0; i < 8; ++i)
        ptx::red_add_v4_f32(blk + (c / 4u + i) * 32u + lane, __uint_as_float(r[4 * i]),
                            __uint_as_float(r[4 * i + 1]), __uint_as_float(r[4 * i + 2]),
                            __uint_as_float(r[4 * i + 3]));
}

// Adds columns [c, c + 32) of this lane's row of the tile's sum, read at L2.
__device__ __forceinline__ void sum_accum32(const float4* blk, uint32_t c, uint32_t lane,
                                            uint32_t (&r)[32]) {
#pragma unroll
    for (uint32_t i = 0; i < 8; ++i) {
        const float4 v = __ldcg(blk + (c / 4u + i) * 32u + lane);
        r[4 * i] = __float_as_uint(__uint_as_float(r[4 * i]) + v.x);
        r[4 * i + 1] = __float_as_uint(__uint_as_float(r[4 * i + 1]) + v.y);
        r[4 * i + 2] = __float_as_uint(__uint_as_float(r[4 * i + 2]) + v.z);
        r[4 * i + 3] = __float_as_uint(__uint_as_float(r[4 * i + 3]) + v.w);
    }
}

// Dynamic tile order: a ring of kTileRing tile ids in shared memory.  The
// even CTA's producer (the fetcher) takes tile ids from the global counter
// in order of request and publishes item j's id in slot j % kTileRing of both
// CTAs; every other role reads it there and arrives on the even CTA's
// tile_empty[slot] when done.  kTileEnd marks the end of the work.
constexpr uint32_t kTileRing = 4;
constexpr uint32_t kTileEnd = 0xFFFFFFFFu;

struct TileRing {
    uint64_t* full;    // [kTileRing], 1 arrival (the fetcher)
    uint64_t* empty;   // [kTileRing], one arrival per reader
    uint32_t* ids;     // [kTileRing]
};

__device__ __forceinline__ void whole_tile(const GemmShape& s, uint32_t t, WorkItem& w) {
    w.tile = t;
    w.kb0 = 0;
    w.kb1 = s.num_kb;
    w.part = 0;
    w.parts = 1;
    w.sk = 0;
}

// Fetcher: item j of this unit.  The fetcher runs kTileAhead items ahead of
// its own use, so that the atomic's round trip is not on the path from one
// tile's loads to the next: before item j it has taken items up to
// j + kTileAhead (fetched counts them; done once it published the end).
// False at the end or when a wait gave up.
constexpr uint32_t kTileAhead = kTileRing - 2;

template <int PAIR>
__device__ __forceinline__ bool dyn_fetch(const GemmShape& s, const TileRing& r, uint32_t j,
                                          volatile int* abort_flag, uint32_t& fetched, bool& done,
                                          WorkItem& w) {
    while (!done && fetched <= j + kTileAhead) {
        const uint32_t i = fetched, slot = i % kTileRing, ph = (i / kTileRing) & 1u;
        if (!mbar_wait<PAIR == 2>(ptx::smem_addr(r.empty + slot), ph ^ 1u, s.ctl, abort_flag,
                                  kSiteProducerTile, i))
            return false;
        uint32_t t = atomicAdd(s.dyn_counter, 1u);
        if (t >= uint32_t(s.num_tiles)) t = kTileEnd;
        r.ids[slot] = t;
        if (PAIR == 2) {
            ptx::st_shared_cluster_u32(ptx::mapa_shared(ptx::smem_addr(r.ids + slot), 1), t);
            ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_addr(r.full + slot), 1));
        }
        ptx::mbar_arrive(ptx::smem_addr(r.full + slot));
        done = t == kTileEnd;
        ++fetched;
    }
    const uint32_t t = r.ids[j % kTileRing];   // written by this thread above
    whole_tile(s, t, w);
    return t != kTileEnd;
}

// Reader (one thread, or a whole warp with warp = true): item j's tile id.
template <int PAIR, bool WARP>
__device__ __forceinline__ bool dyn_read(const GemmShape& s, const TileRing& r, uint32_t j,
                                         uint32_t lane, volatile int* abort_flag, uint32_t site,
                                         WorkItem& w) {
    const uint32_t slot = j % kTileRing, ph = (j / kTileRing) & 1u;
    const uint32_t fb = ptx::smem_addr(r.full + slot);
    const bool ok = WARP ? mbar_wait_warp<PAIR == 2>(fb, ph, s.ctl, abort_flag, site, j)
                         : mbar_wait<PAIR == 2>(fb, ph, s.ctl, abort_flag, site, j);
    if (!ok) return false;
    const uint32_t t = *reinterpret_cast<volatile uint32_t*>(r.ids + slot);
    if (WARP) __syncwarp();
    if (!WARP || lane == 0) {
        const uint32_t eb = ptx::smem_addr(r.empty + slot);
        if (PAIR == 2)
            ptx::mbar_arrive_cluster(ptx::mapa_shared(eb, 0));
        else
            ptx::mbar_arrive(eb);
    }
    whole_tile(s, t, w);
    return t != kTileEnd;
}

// The epilogue warp is done reading accumulator buffer `ae` belongs to.
template <int PAIR>
__device__ __forceinline__ void acc_release(uint32_t ae, uint32_t lane) {
    ptx::tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) {
        if (PAIR == 2)
            ptx::mbar_arrive_cluster(ptx::mapa_shared(ae, 0));
        else
            ptx::mbar_arrive(ae);
    }
}

// Epilogue of a thin tile (grouped, CTA pair): C^T sits in TMEM, lane =
// output column `col` of the tile (n0 + col), column j = row j of the tile.
// Each lane writes its column of the tile's rows with bias and ReLU; for a
// given row the warp's lanes write 32 consecutive columns.  The accumulator
// may be released once this returns (every tcgen05.ld has completed).
__device__ __forceinline__ void thin_epilogue(const GemmShape& s, const TileInfo& ti,
                                              const float* bias_sm, int32_t group_row0,
                                              uint32_t tcol, uint32_t col, bool zero_acc) {
    const int n = ti.n0 + int(col);
    const bool col_in = n < s.N;
    const float bv = col_in ? bias_sm[col] : 0.f;   // the tile's bias, staged in shared memory
    const size_t pitch = size_t(s.N);
    __nv_bfloat16* cp = static_cast<__nv_bfloat16*>(s.C) +
                        size_t(group_row0 + ti.c_row) * pitch + size_t(n);
    const int n_pad = (ti.thin + 15) & ~15;
#pragma unroll 1
    for (int c = 0; c < n_pad; c += 16) {
        uint32_t r[16];
        ptx::tmem_ld_32x32b_x16(tcol + uint32_t(c), r);
        ptx::tmem_ld_wait();
        const int rows = col_in ? ti.thin - c : 0;   // rows of this chunk to store
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (j < rows)
                *cp = __float2bfloat16_rn(fmaxf((zero_acc ? 0.f : __uint_as_float(r[j])) + bv, 0.f));
            cp += pitch;
        }
    }
}

// The MMAs of one ring stage (KSUB 128-byte K slices) into accumulator d_tmem.
// THIN (grouped, CTA pair, bf16): the tile is computed transposed, so the
// weight panels are the A operand and the X rows the B operand, with the thin
// instruction descriptor.  `first`: this stage starts the accumulation.
template <int KIND, int PAIR, uint32_t KSUB, bool THIN>
__device__ __forceinline__ void issue_stage(uint32_t d_tmem, uint32_t stage_base, bool first,
                                            uint32_t thin_idesc) {
    using K_ = Kind<KIND>;
    using PR = Pair<PAIR>;
    constexpr uint32_t kPanelBytes = K_::bk * 128;
    constexpr uint32_t kIdesc = make_idesc<KIND, PAIR>();
#pragma unroll
    for (uint32_t h = 0; h < KSUB; ++h) {
        const uint32_t a_base = stage_base + h * kUmmaAStageBytes;
        const uint32_t b_base = stage_base + KSUB * kUmmaAStageBytes + h * PR::b_bytes;
#pragma unroll
        for (uint32_t k = 0; k < 128 / (K_::mma_k * K_::esize); ++k) {
            const uint64_t ad = sw128_desc(a_base + k * K_::mma_k * K_::esize, 16, 1024);
            const uint64_t bd = sw128_desc(b_base + k * K_::mma_k * 128, kPanelBytes,
                                           K_::b_sbo, K_::b_layout);
            const uint32_t acc = (!first || h != 0 || k != 0) ? 1u : 0u;
            if (PAIR == 2) {
                if (KIND == kUmmaBf16) {
                    if (THIN)
                        ptx::mma_f16_pair(d_tmem, bd, ad, thin_idesc, acc);
                    else
                        ptx::mma_f16_pair(d_tmem, ad, bd, kIdesc, acc);
                } else {
                    ptx::mma_tf32_pair(d_tmem, ad, bd, kIdesc, acc);
                }
            } else {
                if (KIND == kUmmaBf16)
                    ptx::mma_f16(d_tmem, ad, bd, kIdesc, acc);
                else
                    ptx::mma_tf32(d_tmem, ad, bd, kIdesc, acc);
            }
        }
    }
}

// Teardown after an abort, by the even CTA's producer lane once every role of
// the unit has left its loop: waits (bounded) until every TMA load that this
// CTA or its peer issued has landed, so that no copy still writes shared
// memory when the CTAs exit.  This CTA registered items [0, issued) on its
// full barriers (expect_tx of the whole unit's bytes) and issued its own loads
// for them; the peer issued its loads for items [0, issued_peer); neither
// issued the injected item of a self test.  Only the last S items can be
// outstanding: item j is registered or issued only after item j - S was
// consumed, so the window's items sit on distinct slots in phase j / S.
// Registrations are evened up first: the peer's half of an item it never
// issued is counted done (complete_tx), and an item only the peer issued gets
// the arrival and expect_tx of the peer's half.
template <int PAIR>
__device__ __forceinline__ void drain_ring(uint64_t* full, uint32_t S, uint32_t issued,
                                           uint32_t issued_peer, uint32_t cta_bytes,
                                           const FaultInjection& inj, uint32_t unit,
                                           uint64_t limit_ns) {
    const uint32_t hi = issued > issued_peer ? issued : issued_peer;
    const uint32_t lo = hi > S ? hi - S : 0u;
    for (uint32_t j = lo; j < hi; ++j) {
        if (inject_skip_unit(inj, unit, j)) continue;   // no CTA issued a load for it
        const uint32_t bar = ptx::smem_addr(full + j % S);
        const bool mine = j < issued, peer = PAIR == 2 && j < issued_peer;
        if (PAIR == 2) {
            if (!mine && !peer) continue;
            if (mine && !peer) ptx::mbar_complete_tx(bar, cta_bytes);
            if (!mine && peer) ptx::mbar_arrive_expect_tx(bar, cta_bytes);
        } else if (!mine) {
            continue;
        }
        mbar_wait_drain(bar, (j / S) & 1u, limit_ns);
    }
}

// MODE 0: the static tile order only (the instances the library normally runs).
// MODE 1: event trace points, and the dynamic order when requested.
// MODE 2: the dynamic tile order, without trace points.
template <int KIND, bool GROUPED, int PAIR, int KSUB, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_umma_kernel(const __grid_constant__ UmmaParams<GROUPED> P) {
    constexpr bool kTrace = MODE == 1;
    constexpr bool kDyn = MODE != 0;
    using K_ = Kind<KIND>;
    using PR = Pair<PAIR>;
    constexpr bool kCl = PAIR == 2;                      // cluster-scope waits
    constexpr uint32_t kPanelBytes = K_::bk * 128;
    constexpr uint32_t kIdesc = make_idesc<KIND, PAIR>();
    constexpr uint32_t kChunks = kUmmaBN / K_::out_chunk_cols;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align_1024(smem_raw);
    const int S = P.s.stages;
    uint8_t* ring = base;
    constexpr uint32_t ksub = KSUB;                      // 128-byte K slices per stage
    constexpr uint32_t stage_bytes = ksub * PR::stage_bytes;  // [ksub A slices][ksub B slices]
    uint8_t* epi = ring + size_t(S) * stage_bytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(epi + kUmmaEpiBytes);
    uint64_t* empty = full + S;
    uint64_t* acc_full = empty + S;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
    TileRing tiles;
    tiles.full = drain + 2;
    tiles.empty = tiles.full + kTileRing;
    tiles.ids = reinterpret_cast<uint32_t*>(tiles.empty + kTileRing);
    uint32_t* issued_word = tiles.ids + kTileRing;   // ring items this CTA's producer issued
    // The epilogue's bias slot: bias_full (one arrive.expect_tx + the bulk
    // copy's bytes), bias_empty (the 4 epilogue warps of this CTA).
    uint64_t* bias_full = reinterpret_cast<uint64_t*>(issued_word + 2);
    uint64_t* bias_empty = bias_full + 1;
    const float* bias_sm = reinterpret_cast<const float*>(epi + kUmmaEpiBytes + kUmmaBarrierBytes);

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const uint32_t rank = PAIR == 2 ? ptx::cluster_ctarank() : 0u;
    const uint32_t unit = blockIdx.x / PAIR, units = gridDim.x / PAIR;
    const GemmShape& s = P.s;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(ptx::smem_addr(full + i), 1);    // producer arrive + TMA bytes
            ptx::mbar_init(ptx::smem_addr(empty + i), 1);   // one tcgen05.commit
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(acc_full + a), 1);                // one commit
            ptx::mbar_init(ptx::smem_addr(acc_empty + a), 4 * PAIR);        // epilogue warps
        }
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        ptx::mbar_init(ptx::smem_addr(bias_full), 1);
        ptx::mbar_init(ptx::smem_addr(bias_empty), 4);
        for (uint32_t d = 0; d < kTileRing; ++d) {
            ptx::mbar_init(ptx::smem_addr(tiles.full + d), 1);
            // readers: the MMA lane, the epilogue warps of the unit, the odd CTA's producer
            ptx::mbar_init(ptx::smem_addr(tiles.empty + d), 1 + 4 * PAIR + (PAIR == 2 ? 1 : 0));
        }
        *abort_flag = 0;
        ptx::fence_barrier_init();
    } else if (threadIdx.x == 32) {
        ptx::prefetch_tensormap(&P.mapA);
        ptx::prefetch_tensormap(&P.mapB);
    }
    if (warp == 2) {
        if (PAIR == 2) {
            ptx::tmem_alloc_pair(ptx::smem_addr(tmem_holder), kTmemCols);
            ptx::tmem_relinquish_alloc_permit_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_addr(tmem_holder), kTmemCols);
            ptx::tmem_relinquish_alloc_permit();
        }
    }
    ptx::tc_fence_before_sync();
    if (PAIR == 2)
        ptx::cluster_sync_all();   // barriers of both CTAs initialised before any remote use
    else
        __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;
    // The set-up above overlaps the end of the previous kernel in the stream;
    // no role touches global memory before that kernel is done.
    ptx::griddep_wait();
    uint32_t issued = 0;   // producer lane: ring items registered / issued

    if (warp < 4) {
        ptx::setmaxnreg_dec<kRegsWG0>();
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------- TMA producer
            const uint32_t ring_base = ptx::smem_addr(ring);
            const bool hint = s.l2_hint != 0;
            const uint64_t pol_last = ptx::l2_policy_evict_last();
            const uint64_t pol_first = ptx::l2_policy_evict_first();
            const uint64_t pol_normal = ptx::l2_policy_evict_normal();
            const uint64_t pol_a = s.l2_hint == 2 ? pol_first : s.l2_hint == 4 ? pol_normal : pol_last;
            const uint64_t pol_b = s.l2_hint == 3 ? pol_first : s.l2_hint == 4 ? pol_normal : pol_last;
            uint32_t it = 0, ntr = 0, fetched = 0;
            bool ok = true, fetch_done = false;
            const bool dyn = kDyn && s.dyn_counter != nullptr;
            WorkItem w;
            for (uint32_t j = 0;
                 ok && (!dyn ? work_item(s, unit, units, j, w)
                             : rank == 0 ? dyn_fetch<PAIR>(s, tiles, j, abort_flag, fetched,
                                                           fetch_done, w)
                                         : dyn_read<PAIR, false>(s, tiles, j, 0, abort_flag,
                                                                  kSiteProducerTile, w));
                 ++j) {
                const TileInfo ti = decode_tile<GROUPED, PAIR>(P, w.tile, rank);
                const int32_t bcol0 = ti.n0 + int32_t(rank * PR::b_cols);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const uint32_t slot = it % S, ph = (it / S) & 1u;
                    if (!mbar_wait<kCl>(ptx::smem_addr(empty + slot), ph ^ 1u, s.ctl, abort_flag,
                                        kSiteProducerEmpty, it)) {
                        ok = false;
                        break;
                    }
                    if (kTrace) trace_event(s.ctl, kRoleProducer, ntr, kEvWaitDone, it, slot, ph ^ 1u);
                    const uint32_t fb_local = ptx::smem_addr(full + slot);
                    const uint32_t fb = PAIR == 2 ? ptx::mapa_shared(fb_local, 0) : fb_local;
                    if (rank == 0) ptx::mbar_arrive_expect_tx(fb_local, PAIR * stage_bytes);
                    if (inject_skip_unit(s.inject, unit, it)) continue;   // self test
                    if (kTrace) trace_event(s.ctl, kRoleProducer, ntr, kEvIssued, it, slot, 0);
                    const uint32_t stage_base = ring_base + slot * stage_bytes;
#pragma unroll
                    for (uint32_t h = 0; h < ksub; ++h) {
                        const uint32_t a_dst = stage_base + h * kUmmaAStageBytes;
                        const uint32_t b_dst =
                            stage_base + ksub * kUmmaAStageBytes + h * PR::b_bytes;
                        const int32_t k0 = (kb * int32_t(ksub) + int32_t(h)) * int32_t(K_::bk);
                        load_box_2d<PAIR>(a_dst, &P.mapA, fb, k0, ti.a_row, hint, pol_a);
                        if (!GROUPED && s.b_panels_3d) {
                            // All of this CTA's panels of the slice in one box.
                            load_box_3d<PAIR>(b_dst, &P.mapB, fb, 0, k0,
                                              bcol0 / int32_t(K_::panel_cols), hint, pol_b);
                        } else {
#pragma unroll
                            for (uint32_t j = 0; j < PR::b_cols / K_::panel_cols; ++j) {
                                const int32_t n = bcol0 + int32_t(j * K_::panel_cols);
                                const uint32_t d = b_dst + j * kPanelBytes;
                                if (GROUPED)
                                    load_box_3d<PAIR>(d, &P.mapB, fb, n, k0, ti.group, hint,
                                                      pol_b);
                                else
                                    load_box_2d<PAIR>(d, &P.mapB, fb, n, k0, hint, pol_b);
                            }
                        }
                    }
                }
            }
            if (kTrace) trace_count(s.ctl, kRoleProducer, ntr);
            ptx::griddep_launch_dependents();   // every load issued: the next launch may be scheduled
            issued = it;
            *issued_word = it;
        } else if (warp == 1 && lane == 0 && rank == 0) {
            // ---------------------------------------------------- MMA issuer
            const uint32_t ring_base = ptx::smem_addr(ring);
            uint32_t it = 0, tl = 0, ntr = 0, nta = 0;
            bool ok = true;
            const bool dyn = kDyn && s.dyn_counter != nullptr;
            WorkItem w;
            for (; ok && (!dyn ? work_item(s, unit, units, tl, w)
                               : dyn_read<PAIR, false>(s, tiles, tl, 0, abort_flag, kSiteMmaTile, w));
                 ++tl) {
                const uint32_t a = tl & 1u, aph = (tl >> 1) & 1u;
                if (!mbar_wait<kCl>(ptx::smem_addr(acc_empty + a), aph ^ 1u, s.ctl, abort_flag,
                                    kSiteMmaAccEmpty, tl))
                    break;
                if (kTrace) trace_event(s.ctl, kRoleMmaAcc, nta, kEvWaitDone, tl, a, aph ^ 1u);
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + a * kAccCols;
                // Thin tile (grouped, CTA pair): A and B swap roles (C^T = W^T X^T).
                uint32_t thin_idesc = 0;
                if (GROUPED && PAIR == 2) {
                    const TileInfo ti = decode_tile<GROUPED, PAIR>(P, w.tile, 0);
                    if (ti.thin > 0) thin_idesc = make_idesc_thin(uint32_t(ti.thin + 15) & ~15u);
                }
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const uint32_t slot = it % S, ph = (it / S) & 1u;
                    if (!mbar_wait<kCl>(ptx::smem_addr(full + slot), ph, s.ctl, abort_flag,
                                        kSiteMmaFull, it)) {
                        ok = false;
                        break;
                    }
                    if (kTrace) trace_event(s.ctl, kRoleConsumer, ntr, kEvWaitDone, it, slot, ph);
                    ptx::tc_fence_after_sync();
                    const uint32_t stage_base = ring_base + slot * stage_bytes;
                    if (GROUPED && PAIR == 2 && KIND == kUmmaBf16 && thin_idesc != 0)
                        issue_stage<KIND, PAIR, KSUB, true>(d_tmem, stage_base, kb == w.kb0,
                                                            thin_idesc);
                    else
                        issue_stage<KIND, PAIR, KSUB, false>(d_tmem, stage_base, kb == w.kb0, 0u);
                    if (kTrace) trace_event(s.ctl, kRoleConsumer, ntr, kEvReleased, it, slot, 0);
                    if (PAIR == 2)
                        ptx::mma_commit_pair_multicast(ptx::smem_addr(empty + slot), 0x3);
                    else
                        ptx::mma_commit(ptx::smem_addr(empty + slot));
                }
                if (!ok) break;
                if (kTrace) trace_event(s.ctl, kRoleMmaAcc, nta, kEvIssued, tl, a, 0);
                if (w.kb1 > w.kb0) {
                    if (PAIR == 2)
                        ptx::mma_commit_pair_multicast(ptx::smem_addr(acc_full + a), 0x3);
                    else
                        ptx::mma_commit(ptx::smem_addr(acc_full + a));
                } else {
                    const uint32_t af = ptx::smem_addr(acc_full + a);
                    if (PAIR == 2) {
                        ptx::mbar_arrive_cluster(ptx::mapa_shared(af, 0));
                        ptx::mbar_arrive_cluster(ptx::mapa_shared(af, 1));
                    } else {
                        ptx::mbar_arrive(af);
                    }
                }
            }
            if (kTrace) trace_count(s.ctl, kRoleConsumer, ntr);
            if (kTrace) trace_count(s.ctl, kRoleMmaAcc, nta);
            // No MMA may still be running when TMEM (or the peer's smem) is released.
            if (PAIR == 2)
                ptx::mma_commit_pair_multicast(ptx::smem_addr(drain), 0x1);
            else
                ptx::mma_commit(ptx::smem_addr(drain));
            mbar_wait_drain(ptx::smem_addr(drain), 0, s.ctl.timeout_ns);
        }
    } else {
        ptx::setmaxnreg_inc<kRegsWG1>();
        // -------------------------------------------------------- epilogue
        const uint32_t q = warp & 3u;                 // TMEM lane quarter / row block
        const uint32_t lane_base = (q * 32u) << 16;
        const uint32_t stage0 = ptx::smem_addr(epi) + q * 2u * kEpiBufBytes;
        const uint32_t row_off = lane * 128u;
        const uint32_t swz = lane & 7u;
        uint32_t chunk_ctr = 0, ntr = 0;
        uint32_t bias_issued = 0;                     // warp 0: bias copies issued
        const bool tracer = kTrace && s.ctl.trace != nullptr && q == 0 && lane == 0;   // one lane
        const bool dyn = kDyn && s.dyn_counter != nullptr;
        WorkItem w;
        for (uint32_t tl = 0;
             !dyn ? work_item(s, unit, units, tl, w)
                  : dyn_read<PAIR, true>(s, tiles, tl, lane, abort_flag, kSiteEpiTile, w);
             ++tl) {
            const TileInfo ti = decode_tile<GROUPED, PAIR>(P, w.tile, rank);
            const uint32_t a = tl & 1u, aph = (tl >> 1) & 1u;
            const uint32_t ae = ptx::smem_addr(acc_empty + a);
            // Warp 0 stages this item's bias (the tile's columns that lie
            // inside N) once all 4 warps are done with the previous item's.
            // The copy lands while the item's mainloop runs.
            if (q == 0) {
                if (tl > 0 && !mbar_wait_warp(ptx::smem_addr(bias_empty), (tl - 1u) & 1u, s.ctl,
                                              abort_flag, kSiteEpiBias, tl))
                    break;
                if (lane == 0) {
                    const int32_t cols = s.N - ti.n0 < int32_t(kUmmaBN) ? s.N - ti.n0 : int32_t(kUmmaBN);
                    const uint32_t bytes = uint32_t(cols) * 4u;
                    const uint32_t bf = ptx::smem_addr(bias_full);
                    ptx::mbar_arrive_expect_tx(bf, bytes);
                    ptx::bulk_load(ptx::smem_addr(bias_sm),
                                   s.bias + (GROUPED ? P.bias_group_stride * ti.group : 0) + ti.n0,
                                   bytes, bf);
                }
                ++bias_issued;
            }
            if (!mbar_wait_warp<kCl>(ptx::smem_addr(acc_full + a), aph, s.ctl, abort_flag,
                                     kSiteEpiAccFull, tl))
                break;
            if (tracer) trace_event(s.ctl, kRoleEpilogue, ntr, kEvWaitDone, tl, a, aph);
            ptx::tc_fence_after_sync();
            const bool zero_acc = w.kb1 == w.kb0;
            // Split tile: each unit sharing it checks in on arrival.  All but
            // the last to arrive add their fp32 part of these 32 rows into the
            // tile's zeroed sum (reductions at L2), free the accumulator and
            // count themselves done.  The last to arrive waits until the
            // others are done -- they have all started, and they finish
            // without waiting on anything -- then adds the sum to its own
            // accumulator in the epilogue below.
            const float4* sum = nullptr;
            if (w.parts > 1) {
                float4* blk = sum_block<PAIR>(s, w.sk, rank, q);
                uint32_t* arrived = s.sk_count + ((uint32_t(w.sk) * PAIR + rank) * 4u + q) * 2u;
                uint32_t before = 0;
                if (lane == 0) before = atomicAdd(arrived, 1u);
                before = __shfl_sync(0xffffffffu, before, 0);
                if (before + 1u != uint32_t(w.parts)) {
                    const uint32_t acc0 = tmem_base + lane_base + a * kAccCols;
#pragma unroll 1
                    for (uint32_t c2 = 0; c2 < kAccCols; c2 += 64) {
                        uint32_t r0[32], r1[32];
                        ptx::tmem_ld_32x32b_x32(acc0 + c2, r0);
                        ptx::tmem_ld_32x32b_x32(acc0 + c2 + 32, r1);
                        ptx::tmem_ld_wait();
                        sum_add32(blk, c2, lane, r0);
                        sum_add32(blk, c2 + 32, lane, r1);
                    }
                    if (tracer) trace_event(s.ctl, kRoleEpilogue, ntr, kEvReleased, tl, a, 0);
                    acc_release<PAIR>(ae, lane);
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) atomicAdd(arrived + 1, 1u);
                    // This part runs no epilogue, but hands the bias slot on.
                    if (!mbar_wait_warp(ptx::smem_addr(bias_full), tl & 1u, s.ctl, abort_flag,
                                        kSiteEpiBias, tl))
                        break;
                    if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(bias_empty));
                    continue;
                }
                bool ok = true;
                if (lane == 0)
                    ok = counter_wait(arrived + 1, uint32_t(w.parts - 1), s.ctl, abort_flag,
                                      kSiteEpiSplitSum, tl);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
                __threadfence();
                sum = blk;
            }
            if (!mbar_wait_warp(ptx::smem_addr(bias_full), tl & 1u, s.ctl, abort_flag,
                                kSiteEpiBias, tl))
                break;
            if (GROUPED && PAIR == 2 && KIND == kUmmaBf16 && ti.thin > 0) {
                // Thin tile: the accumulator holds C^T, TMEM lane = output
                // column, column j = row j of the tile.  Each lane stores its
                // column of the tile's rows; a warp's 32 lanes write 64
                // contiguous bytes of a row.  (Thin tiles are never split.)
                thin_epilogue(s, ti, bias_sm, P.g.row_off[ti.group],
                              tmem_base + lane_base + a * kAccCols, rank * 128u + q * 32u + lane,
                              zero_acc);
                if (tracer) trace_event(s.ctl, kRoleEpilogue, ntr, kEvReleased, tl, a, 0);
                acc_release<PAIR>(ae, lane);
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(bias_empty));
                continue;
            }
            const CUtensorMap* mapC = &P.mapC[GROUPED ? ti.group : 0];
            for (uint32_t c = 0; c < kChunks; ++c, ++chunk_ctr) {
                const uint32_t col0 = c * K_::out_chunk_cols;
                const uint32_t taddr = tmem_base + lane_base + a * kAccCols + col0;
                uint32_t packed[32];
                if (KIND == kUmmaBf16) {
                    uint32_t r0[32], r1[32];
                    ptx::tmem_ld_32x32b_x32(taddr, r0);
                    ptx::tmem_ld_32x32b_x32(taddr + 32, r1);
                    ptx::tmem_ld_wait();
                    if (c + 1 == kChunks) {
                        if (tracer) trace_event(s.ctl, kRoleEpilogue, ntr, kEvReleased, tl, a, 0);
                        acc_release<PAIR>(ae, lane);
                    }
                    if (sum != nullptr) {
                        sum_accum32(sum, col0, lane, r0);
                        sum_accum32(sum, col0 + 32, lane, r1);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t* r = h == 0 ? r0 : r1;
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const int n = ti.n0 + int(col0) + 32 * h + 4 * j4;
                            float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (n < s.N) b = *reinterpret_cast<const float4*>(bias_sm + (n - ti.n0));
                            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int j = 4 * j4 + 2 * u;
                                const float x0 = zero_acc ? 0.f : __uint_as_float(r[j]);
                                const float x1 = zero_acc ? 0.f : __uint_as_float(r[j + 1]);
                                const __nv_bfloat162 v = __floats2bfloat162_rn(
                                    fmaxf(x0 + bv[2 * u], 0.f), fmaxf(x1 + bv[2 * u + 1], 0.f));
                                packed[16 * h + j / 2] = *reinterpret_cast<const uint32_t*>(&v);
                            }
                        }
                    }
                } else {
                    uint32_t r0[32];
                    ptx::tmem_ld_32x32b_x32(taddr, r0);
                    ptx::tmem_ld_wait();
                    if (c + 1 == kChunks) {
                        if (tracer) trace_event(s.ctl, kRoleEpilogue, ntr, kEvReleased, tl, a, 0);
                        acc_release<PAIR>(ae, lane);
                    }
                    if (sum != nullptr) sum_accum32(sum, col0, lane, r0);
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const int n = ti.n0 + int(col0) + 4 * j4;
                        float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (n < s.N) b = *reinterpret_cast<const float4*>(bias_sm + (n - ti.n0));
                        const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float x = zero_acc ? 0.f : __uint_as_float(r0[4 * j4 + u]);
                            packed[4 * j4 + u] = __float_as_uint(fmaxf(x + bv[u], 0.f));
                        }
                    }
                }
                // Stage the 32 x 128 B sub-tile (TMA 128-byte swizzle) and store it.
                const uint32_t buf = stage0 + (chunk_ctr & 1u) * kEpiBufBytes;
                if (chunk_ctr >= 2) {
                    if (lane == 0) ptx::bulk_wait_group_read<1>();
                    __syncwarp();
                }
#pragma unroll
                for (uint32_t j = 0; j < 8; ++j)
                    ptx::st_shared_v4(buf + row_off + ((j ^ swz) << 4), packed[4 * j],
                                      packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    ptx::tma_store_2d(mapC, buf, ti.n0 + int32_t(col0), ti.c_row + int32_t(q * 32));
                    ptx::bulk_commit_group();
                }
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(bias_empty));   // done with this bias
        }
        // The last bias copy issued has landed before the CTA may exit (it
        // has, unless an abort left its item unconsumed).
        if (q == 0 && lane == 0 && bias_issued > 0)
            mbar_wait_drain(ptx::smem_addr(bias_full), (bias_issued - 1u) & 1u, s.ctl.timeout_ns);
        if (tracer) trace_count(s.ctl, kRoleEpilogue, ntr);
        if (lane == 0) ptx::bulk_wait_group<0>();
    }

    __syncwarp();
    ptx::tc_fence_before_sync();
    if (PAIR == 2)
        ptx::cluster_sync_all();
    else
        __syncthreads();
    // Every role of the unit has left its loop, so the abort flags are final.
    // After an abort, loads may still be in flight (a stage nobody consumed):
    // the even CTA's producer lane waits for them -- its own and its peer's --
    // while every other thread of the unit waits at the barrier below.
    if (warp == 0 && lane == 0 && rank == 0) {
        bool aborted = *abort_flag != 0;
        uint32_t issued_peer = issued;
        if (PAIR == 2) {
            const uint32_t flag_addr = ptx::smem_addr(const_cast<int*>(abort_flag));
            aborted = aborted || ptx::ld_shared_cluster_u32(ptx::mapa_shared(flag_addr, 1)) != 0;
            issued_peer = ptx::ld_shared_cluster_u32(ptx::mapa_shared(ptx::smem_addr(issued_word), 1));
        }
        if (aborted)
            drain_ring<PAIR>(full, uint32_t(S), issued, issued_peer, stage_bytes, s.inject, unit,
                             s.ctl.timeout_ns);
    }
    if (PAIR == 2)
        ptx::cluster_sync_all();   // no CTA leaves while its peer may still touch its smem
    else
        __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after_sync();
        if (PAIR == 2)
            ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int KIND, bool GROUPED, int PAIR, int KSUB, int MODE>
void* kernel_ptr() {
    return reinterpret_cast<void*>(&gemm_umma_kernel<KIND, GROUPED, PAIR, KSUB, MODE>);
}

// Mode 0 runs unless a trace buffer (mode 1) or the dynamic order (mode 2) is
// requested: compiled into the plain instances, that code costs them 2-5%
// (trace points and per-item tile reads on the MMA lane, register pressure in
// the epilogue).  Calling this instantiates every (pair, k-slices, mode) of
// one (kind, grouped).
template <int KIND, bool GROUPED, int MODE>
void* select_kernel_kgm(int pair, int ksub) {
    if (pair == 2)
        return ksub == 2 ? kernel_ptr<KIND, GROUPED, 2, 2, MODE>()
                         : kernel_ptr<KIND, GROUPED, 2, 1, MODE>();
    return ksub == 2 ? kernel_ptr<KIND, GROUPED, 1, 2, MODE>()
                     : kernel_ptr<KIND, GROUPED, 1, 1, MODE>();
}

template <int KIND, bool GROUPED>
void* select_kernel_kg(int pair, int ksub, int mode) {
    return mode == 1 ? select_kernel_kgm<KIND, GROUPED, 1>(pair, ksub)
         : mode == 2 ? select_kernel_kgm<KIND, GROUPED, 2>(pair, ksub)
                     : select_kernel_kgm<KIND, GROUPED, 0>(pair, ksub);
}

}  // namespace umma

// One translation unit per (kind, grouped) instantiates its kernels.
void* umma_kernel_bf16(int pair, int ksub, int mode);
void* umma_kernel_bf16_grouped(int pair, int ksub, int mode);
void* umma_kernel_tf32(int pair, int ksub, int mode);

}  // namespace gbr
