// gemm_umma.cu -- warp-specialized, persistent tensor-core GEMM + bias + ReLU
// for sm_103a (tcgen05 MMA into Tensor Memory), bf16 or TF32 inputs.
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
//   * Persistent CTAs (one per SM) walk tiles t = blockIdx.x + j * gridDim.x
//     in banded order; every role walks the same sequence, and the
//     k-iteration counter runs across tiles so phases carry over.
//   * Registers move from warpgroup 0 (producer / MMA / TMEM allocator) to the
//     epilogue warpgroup with setmaxnreg.
//
// Shared-memory ring stage (both kinds: 128 bytes of K per row):
//   A: 128 rows (M) x 128 B, K-major, TMA 128-byte swizzle      16 KiB
//   B: BK rows (K) x 256 columns (N), N-major (B is row-major [K, N]),
//      stored as 256*esize/128 panels of BK rows x 128 B          32 KiB
// kind     BK  MMA K  panels  panel bytes
// bf16     64   16      4       8 KiB
// tf32     32    8      8       4 KiB
#include "gbr_internal.h"

#include <cuda_bf16.h>

namespace gbr {

namespace {

constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kRegsWG0 = 88;
constexpr uint32_t kRegsWG1 = 224;
constexpr uint32_t kEpiBufBytes = 32 * 128;   // 32 rows x 128 B per warp buffer

template <int KIND>
struct Kind;
template <>
struct Kind<kUmmaBf16> {
    static constexpr uint32_t esize = 2, bk = 64, mma_k = 16, panel_cols = 64, panels = 4;
    static constexpr uint32_t ab_format = 1;          // BF16
    static constexpr uint32_t out_chunk_cols = 64;    // 64 bf16 = 128 B per row
    static constexpr bool b_kmajor = false;           // B stays row-major [K, N]
};
template <>
struct Kind<kUmmaTf32> {
    static constexpr uint32_t esize = 4, bk = 32, mma_k = 8, panel_cols = 32, panels = 8;
    static constexpr uint32_t ab_format = 2;          // TF32
    static constexpr uint32_t out_chunk_cols = 32;    // 32 fp32 = 128 B per row
    static constexpr bool b_kmajor = true;            // B arrives transposed, Bt[N, K]
};

// Instruction descriptor, kind::f16 / kind::tf32: fp32 accumulator, A K-major,
// B MN-major (bf16) or K-major (tf32), M = 128, N = 256, dense, no negation.
template <int KIND>
__host__ __device__ constexpr uint32_t make_idesc() {
    return (1u << 4)                              // D format: f32
           | (Kind<KIND>::ab_format << 7)         // A format
           | (Kind<KIND>::ab_format << 10)        // B format
           | (0u << 15)                           // A: K-major
           | ((Kind<KIND>::b_kmajor ? 0u : 1u) << 16)  // B: K-major / MN-major
           | ((uint32_t(kUmmaBN) >> 3) << 17)     // N / 8
           | ((uint32_t(kUmmaBM) >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor with 128-byte swizzling.
//   bits  0-13 start address >> 4     bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4  bits 46-48 = 0b001 (tcgen05 version)
//   bits 49-51 base offset = 0 (atoms are 1024-byte aligned)
//   bits 61-63 = 2 (128-byte swizzle)
// K-major operand (A; TF32 B): rows 128 B apart, 8-row groups SBO = 1024 B
// apart, LBO unused; the k-th MMA of a stage starts k * 32 bytes into the row.
// MN-major B (bf16): 8 K-rows form a 1024-byte atom, atoms along K are
// SBO = 1024 B apart and 128-byte column panels are LBO = panel bytes apart.
// (An MN-major B operand is not usable with kind::tf32: the MMA reads zeros.)
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
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
    int32_t a_row;   // row coordinate of the A/X box
    int32_t c_row;   // row coordinate of the C box in mapC[group]
    int32_t n0;      // first output column
    int32_t group;
};

template <bool GROUPED>
__device__ __forceinline__ TileInfo decode_tile(const UmmaParams<GROUPED>& P, uint32_t t) {
    TileInfo ti;
    uint32_t mt, nt;
    if (!GROUPED) {
        raster_tile(t, P.s.m_tiles, P.s.n_tiles, P.s.group_m, mt, nt);
        ti.a_row = int32_t(mt) * kUmmaBM;
        ti.c_row = ti.a_row;
        ti.group = 0;
    } else {
        int e = 0;
        while (e + 1 < P.g.num_groups && int32_t(t) >= P.g.tile_start[e + 1]) ++e;
        raster_tile(t - uint32_t(P.g.tile_start[e]), uint32_t(P.g.m_tiles[e]), P.s.n_tiles,
                    P.s.group_m, mt, nt);
        ti.c_row = int32_t(mt) * kUmmaBM;
        ti.a_row = P.g.row_off[e] + ti.c_row;
        ti.group = e;
    }
    ti.n0 = int32_t(nt) * kUmmaBN;
    return ti;
}

template <int KIND, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_umma_kernel(const __grid_constant__ UmmaParams<GROUPED> P) {
    using K_ = Kind<KIND>;
    constexpr uint32_t kPanelBytes = K_::bk * 128;
    constexpr uint32_t kIdesc = make_idesc<KIND>();
    constexpr uint32_t kChunks = kUmmaBN / K_::out_chunk_cols;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align_1024(smem_raw);
    const int S = P.s.stages;
    uint8_t* ring = base;
    uint8_t* epi = ring + size_t(S) * kUmmaStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(epi + kUmmaEpiBytes);
    uint64_t* empty = full + S;
    uint64_t* acc_full = empty + S;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31u;
    const GemmShape& s = P.s;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(ptx::smem_addr(full + i), 1);    // producer arrive + TMA bytes
            ptx::mbar_init(ptx::smem_addr(empty + i), 1);   // one tcgen05.commit
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(ptx::smem_addr(acc_full + a), 1);   // one tcgen05.commit
            ptx::mbar_init(ptx::smem_addr(acc_empty + a), 4);  // one arrive per epilogue warp
        }
        ptx::mbar_init(ptx::smem_addr(drain), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    } else if (threadIdx.x == 32) {
        ptx::prefetch_tensormap(&P.mapA);
        ptx::prefetch_tensormap(&P.mapB);
    }
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_holder), kTmemCols);
        ptx::tmem_relinquish_alloc_permit();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;

    if (warp < 4) {
        ptx::setmaxnreg_dec<kRegsWG0>();
        if (warp == 0 && lane == 0) {
            // ---------------------------------------------------- TMA producer
            const uint32_t ring_base = ptx::smem_addr(ring);
            uint32_t it = 0;
            bool ok = true;
            for (uint32_t t = blockIdx.x; ok && t < uint32_t(s.num_tiles); t += gridDim.x) {
                const TileInfo ti = decode_tile<GROUPED>(P, t);
                for (int kb = 0; kb < s.num_kb; ++kb, ++it) {
                    const uint32_t slot = it % S, ph = (it / S) & 1u;
                    if (!mbar_wait(ptx::smem_addr(empty + slot), ph ^ 1u, s.ctl, abort_flag,
                                   kSiteProducerEmpty, it)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = ptx::smem_addr(full + slot);
                    ptx::mbar_arrive_expect_tx(fb, kUmmaStageBytes);
                    const uint32_t a_dst = ring_base + slot * kUmmaStageBytes;
                    const uint32_t b_dst = a_dst + kUmmaAStageBytes;
                    const int32_t k0 = kb * int32_t(K_::bk);
                    ptx::tma_load_2d(a_dst, &P.mapA, fb, k0, ti.a_row);
                    if (K_::b_kmajor) {
                        // Bt[N, K]: one 256-row box, 128 bytes of K per row.
                        ptx::tma_load_2d(b_dst, &P.mapB, fb, k0, ti.n0);
                    } else {
#pragma unroll
                        for (uint32_t j = 0; j < K_::panels; ++j) {
                            const int32_t n = ti.n0 + int32_t(j * K_::panel_cols);
                            if (GROUPED)
                                ptx::tma_load_3d(b_dst + j * kPanelBytes, &P.mapB, fb, n, k0,
                                                 ti.group);
                            else
                                ptx::tma_load_2d(b_dst + j * kPanelBytes, &P.mapB, fb, n, k0);
                        }
                    }
                }
            }
            if (*abort_flag) {
                const uint32_t n = it < uint32_t(S) ? it : uint32_t(S);
                for (uint32_t j = it - n; j < it; ++j)
                    mbar_wait_drain(ptx::smem_addr(full + j % S), (j / S) & 1u, s.ctl.timeout_ns);
            }
        } else if (warp == 1 && lane == 0) {
            // ---------------------------------------------------- MMA issuer
            const uint32_t ring_base = ptx::smem_addr(ring);
            uint32_t it = 0, tl = 0;
            bool ok = true;
            for (uint32_t t = blockIdx.x; ok && t < uint32_t(s.num_tiles); t += gridDim.x, ++tl) {
                const uint32_t a = tl & 1u, aph = (tl >> 1) & 1u;
                if (!mbar_wait(ptx::smem_addr(acc_empty + a), aph ^ 1u, s.ctl, abort_flag,
                               kSiteMmaAccEmpty, tl))
                    break;
                ptx::tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + a * kAccCols;
                for (int kb = 0; kb < s.num_kb; ++kb, ++it) {
                    const uint32_t slot = it % S, ph = (it / S) & 1u;
                    if (!mbar_wait(ptx::smem_addr(full + slot), ph, s.ctl, abort_flag,
                                   kSiteMmaFull, it)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after_sync();
                    const uint32_t a_base = ring_base + slot * kUmmaStageBytes;
                    const uint32_t b_base = a_base + kUmmaAStageBytes;
#pragma unroll
                    for (uint32_t k = 0; k < 128 / (K_::mma_k * K_::esize); ++k) {
                        const uint64_t ad = sw128_desc(a_base + k * K_::mma_k * K_::esize, 16, 1024);
                        const uint64_t bd =
                            K_::b_kmajor
                                ? sw128_desc(b_base + k * K_::mma_k * K_::esize, 16, 1024)
                                : sw128_desc(b_base + k * K_::mma_k * 128, kPanelBytes, 1024);
                        if (KIND == kUmmaBf16)
                            ptx::mma_f16(d_tmem, ad, bd, kIdesc, (kb | k) != 0);
                        else
                            ptx::mma_tf32(d_tmem, ad, bd, kIdesc, (kb | k) != 0);
                    }
                    ptx::mma_commit(ptx::smem_addr(empty + slot));
                }
                if (!ok) break;
                if (s.num_kb > 0)
                    ptx::mma_commit(ptx::smem_addr(acc_full + a));
                else
                    ptx::mbar_arrive(ptx::smem_addr(acc_full + a));
            }
            // No MMA may still be running when TMEM is released.
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
        const bool zero_acc = s.num_kb == 0;
        uint32_t tl = 0, chunk_ctr = 0;
        for (uint32_t t = blockIdx.x; t < uint32_t(s.num_tiles); t += gridDim.x, ++tl) {
            const TileInfo ti = decode_tile<GROUPED>(P, t);
            const uint32_t a = tl & 1u, aph = (tl >> 1) & 1u;
            if (!mbar_wait_warp(ptx::smem_addr(acc_full + a), aph, s.ctl, abort_flag,
                                kSiteEpiAccFull, tl))
                break;
            ptx::tc_fence_after_sync();
            const float* bias = s.bias + (GROUPED ? P.bias_group_stride * ti.group : 0);
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
                        ptx::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(acc_empty + a));
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t* r = h == 0 ? r0 : r1;
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4) {
                            const int n = ti.n0 + int(col0) + 32 * h + 4 * j4;
                            float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (n < s.N) b = __ldg(reinterpret_cast<const float4*>(bias + n));
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
                        ptx::tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(acc_empty + a));
                    }
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        const int n = ti.n0 + int(col0) + 4 * j4;
                        float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (n < s.N) b = __ldg(reinterpret_cast<const float4*>(bias + n));
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
        }
        if (lane == 0) ptx::bulk_wait_group<0>();
    }

    __syncwarp();
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int KIND, bool GROUPED>
void* kernel_ptr() {
    return reinterpret_cast<void*>(&gemm_umma_kernel<KIND, GROUPED>);
}

void* select_kernel(int kind, bool grouped) {
    if (kind == kUmmaBf16) return grouped ? kernel_ptr<kUmmaBf16, true>() : kernel_ptr<kUmmaBf16, false>();
    return grouped ? kernel_ptr<kUmmaTf32, true>() : kernel_ptr<kUmmaTf32, false>();
}

}  // namespace

size_t umma_smem_bytes(int stages) {
    const size_t need = 1024 + size_t(stages) * kUmmaStageBytes + kUmmaEpiBytes + 256;
    // At least half the SM's shared memory, so that two CTAs never share an
    // SM and compete for its 512 TMEM columns.
    const size_t floor_one_cta = 120 * 1024;
    return need > floor_one_cta ? need : floor_one_cta;
}

cudaError_t umma_prepare(int kind, bool grouped, size_t smem) {
    return cudaFuncSetAttribute(select_kernel(kind, grouped),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
}

cudaError_t umma_check_registers(int kind, bool grouped, int* regs) {
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, select_kernel(kind, grouped));
    if (e != cudaSuccess) return e;
    *regs = fa.numRegs;
    const long need = 128L * kRegsWG0 + 128L * kRegsWG1;
    return (long(fa.numRegs) * kThreads >= need) ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t launch_gemm_umma(int kind, const CUtensorMap& mapA, const CUtensorMap& mapB,
                             const CUtensorMap& mapC, const GemmShape& s, int grid, size_t smem,
                             cudaStream_t stream) {
    UmmaParams<false> P;
    memset(&P, 0, sizeof(P));
    P.mapA = mapA;
    P.mapB = mapB;
    P.mapC[0] = mapC;
    P.s = s;
    P.bias_group_stride = 0;
    if (kind == kUmmaBf16)
        gemm_umma_kernel<kUmmaBf16, false><<<grid, kThreads, smem, stream>>>(P);
    else
        gemm_umma_kernel<kUmmaTf32, false><<<grid, kThreads, smem, stream>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_gemm_umma_grouped(const CUtensorMap& mapX, const CUtensorMap& mapW,
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
    gemm_umma_kernel<kUmmaBf16, true><<<grid, kThreads, smem, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace gbr
