// api.cu -- the C ABI (include/gbr.h): validation, tensor-map encoding,
// launch configuration and the device status block.
#include "gbr.h"
#include "gbr_internal.h"
#include "split_plan.cuh"

#include <cudaTypedefs.h>

#include <algorithm>
#include <array>
#include <atomic>
#include <map>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

namespace gbr {
namespace {

thread_local std::string t_last_error;
// Failure-detection self test: injection and wait limit for the next launch on
// this thread (set and cleared by the gbr_selftest_* entry points only).
thread_local FaultInjection t_inject = {0, 0, 0};
thread_local uint64_t t_timeout_override = 0;
std::atomic<long long> g_launches{0};
std::mutex g_mu;
uint64_t g_timeout_ns = 0;  // 0: not yet resolved
int g_copy_store_lag = -1;
int g_copy_ctas_per_sm = -1;
int g_copy_l2_hint = -1;
int g_gemm_pair = -1;      // -1 auto, 1 one CTA per tile, 2 CTA pair per tile
int g_gemm_group_m = -1;   // -1 auto: tile rows per raster band
int g_gemm_l2_hint = -1;   // -1 auto (none): L2 policy of the operand loads
int g_gemm_k_sub = -1;     // -1 auto (1): 128-byte K slices per ring stage
int g_gemm_split = -1;     // -1 auto, 0 off, 1 on whenever some tile can be split
int g_gemm_dynamic = 0;    // 1: tensor-core GEMMs take tiles from an atomic counter
int g_gemm_thin = 1;       // 1: grouped CTA-pair launches run short last M-tiles transposed
int g_launch_overlap = 1;  // 1: kernels are launched with programmatic stream serialization
uint8_t* g_trace = nullptr;  // event trace buffer (device memory of the caller), or null
uint32_t g_trace_cap = 0;    // records per (CTA, role)

constexpr int kMaxDevices = 64;
constexpr int kHostChunks = 8;                       // M chunks of a host-buffer GEMM
constexpr int kHostEvents = 2 * kHostChunks + 2;     // fork, per chunk in/computed, join

struct DevCtx {
    bool ready = false;
    int sm_count = 0;
    int smem_optin = 0;
    uint32_t* status = nullptr;
    cudaMemPool_t pool = nullptr;   // stream-ordered scratch; keeps what it maps
    // Host-buffer GEMM: copy-in, compute and copy-out streams and their events,
    // created on first use; one enqueue sequence at a time (host_mu).
    bool host_ready = false;
    cudaStream_t host_streams[3] = {};
    cudaEvent_t host_events[kHostEvents] = {};
    std::mutex host_mu;
    bool ffma_regs_ok = false, ffma_regs_checked = false;
    bool umma_regs_ok[kUmmaKinds][2][2] = {};        // [kind][grouped][pair - 1]
    bool umma_regs_checked[kUmmaKinds][2][2] = {};
};
DevCtx g_dev[kMaxDevices];

// Per-device memo of occupancy queries (pure functions of kernel and shared
// memory size).  Key: {operator, dtype/kind, grouped, pair, smem bytes}.
using PrepKey = std::array<int64_t, 5>;
std::mutex g_prep_mu;
std::map<PrepKey, int> g_prep[kMaxDevices];

template <class F>
int prepared(int dev, const PrepKey& key, int* value, F&& prepare) {
    {
        std::lock_guard<std::mutex> lk(g_prep_mu);
        auto it = g_prep[dev].find(key);
        if (it != g_prep[dev].end()) {
            *value = it->second;
            return GBR_OK;
        }
    }
    const int r = prepare(value);
    if (r != GBR_OK) return r;
    std::lock_guard<std::mutex> lk(g_prep_mu);
    g_prep[dev][key] = *value;
    return GBR_OK;
}

enum PrepOp : int64_t { kPrepCopy = 1, kPrepFfma = 2 };

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(GBR_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

uint64_t timeout_ns() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_timeout_ns == 0) {
        const char* env = std::getenv("GBR_WAIT_TIMEOUT_NS");
        unsigned long long v = env ? std::strtoull(env, nullptr, 10) : 0ull;
        g_timeout_ns = v ? v : 2000000000ull;
    }
    return g_timeout_ns;
}

int get_ctx(DevCtx** out, int* dev_out = nullptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GBR_ERR_INVALID, "device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_mu);
    DevCtx& c = g_dev[dev];
    if (!c.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&c.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&c.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        if (major != 10 || minor != 3)
            return fail(GBR_ERR_UNSUPPORTED,
                        "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                        minor);
        if ((e = cudaMalloc(&c.status, kStatusWords * sizeof(uint32_t))) != cudaSuccess)
            return cuda_fail(e, "cudaMalloc(status block)");
        if ((e = cudaMemset(c.status, 0, kStatusWords * sizeof(uint32_t))) != cudaSuccess)
            return cuda_fail(e, "cudaMemset(status block)");
        // A pool of this library's own for per-call scratch (split-tile
        // partial sums, the dynamic tile counter): allocation and release are
        // stream-ordered, so calls on different streams never share scratch,
        // and the pool keeps the memory it has mapped for the next call.
        cudaMemPoolProps props;
        memset(&props, 0, sizeof(props));
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if ((e = cudaMemPoolCreate(&c.pool, &props)) != cudaSuccess)
            return cuda_fail(e, "cudaMemPoolCreate");
        uint64_t keep = ~0ull;
        if ((e = cudaMemPoolSetAttribute(c.pool, cudaMemPoolAttrReleaseThreshold, &keep)) !=
            cudaSuccess)
            return cuda_fail(e, "cudaMemPoolSetAttribute");
        c.ready = true;
    }
    *out = &c;
    if (dev_out) *dev_out = dev;
    return GBR_OK;
}

KernelCtl make_ctl(const DevCtx& c) {
    KernelCtl k;
    k.status = c.status;
    k.timeout_ns = t_timeout_override ? t_timeout_override : timeout_ns();
    std::lock_guard<std::mutex> lk(g_mu);
    k.trace = g_trace;
    k.trace_cap = g_trace_cap;
    return k;
}

// Runs `call` with a fault injected into the next pipeline launch of this thread.
template <class F>
int with_injection(int cta, int item, uint64_t limit_ns, F&& call) {
    if (cta < 0 || item < 0) return fail(GBR_ERR_INVALID, "self test: cta and item must be >= 0");
    if (limit_ns == 0 || limit_ns > 10000000000ull)
        return fail(GBR_ERR_INVALID, "self test: limit must be in (0, 10 s]");
    t_inject = FaultInjection{1u, cta, item};
    t_timeout_override = limit_ns;
    const int r = call();
    t_inject = FaultInjection{0u, 0, 0};
    t_timeout_override = 0;
    return r;
}

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

int encode(CUtensorMap* map, CUtensorMapDataType dt, uint32_t rank, const void* ptr,
           const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
           CUtensorMapSwizzle swz, const char* what) {
    auto fn = encode_fn();
    if (!fn) return fail(GBR_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    cuuint64_t d[5];
    cuuint64_t st[4];
    cuuint32_t b[5], es[5];
    for (uint32_t i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        es[i] = 1;
    }
    for (uint32_t i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
    CUresult r = fn(map, dt, rank, const_cast<void*>(ptr), d, st, b, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(GBR_ERR_INVALID, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", what,
                    int(r));
    return GBR_OK;
}

int encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
              uint64_t outer, uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz, const char* what) {
    const uint64_t dims[2] = {inner, outer};
    const uint64_t strides[1] = {pitch_bytes};
    const uint32_t box[2] = {box_inner, box_outer};
    return encode(map, dt, 2, ptr, dims, strides, box, swz, what);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + bn && b0 < a0 + an;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

int max_stages_for(size_t (*bytes)(int), int smem_optin) {
    int s = 0;
    while (s < 64 && bytes(s + 1) <= size_t(smem_optin)) ++s;
    return s;
}

size_t ffma_bytes_fn(int s) { return ffma_smem_bytes(s); }
// The padding that keeps one CTA per SM is not part of the ring budget.
size_t umma1_bytes_fn(int s) { return umma_ring_bytes(s, 1); }
size_t umma2_bytes_fn(int s) { return umma_ring_bytes(s, 2); }
size_t umma1k2_bytes_fn(int s) { return umma_ring_bytes(s, 1, 2); }
size_t umma2k2_bytes_fn(int s) { return umma_ring_bytes(s, 2, 2); }

int umma_max_stages(int pair, int smem_optin, int k_sub = 1) {
    if (k_sub == 2) return max_stages_for(pair == 2 ? umma2k2_bytes_fn : umma1k2_bytes_fn, smem_optin);
    return max_stages_for(pair == 2 ? umma2_bytes_fn : umma1_bytes_fn, smem_optin);
}

int pair_forced() {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_gemm_pair;
}

int k_sub_forced() {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_gemm_k_sub;
}

// 128-byte K slices per stage: forced by gbr_gemm_tuning, else two on the
// CTA pair whenever the requested ring fits (fewer full/empty handshakes per
// MMA; the handshakes, not the loads, limit the one-slice ring).
int choose_k_sub(int pair, int stages, int smem_optin) {
    const int f = k_sub_forced();
    if (f == 1 || f == 2) return f;
    return (pair == 2 && stages <= umma_max_stages(2, smem_optin, 2)) ? 2 : 1;
}

// Largest ring depth for the dtype (tcgen05: that of the CTA-pair kernel).
int gemm_max_stages(int dtype, int smem_optin) {
    if (dtype == GBR_F32_FFMA_SYNC) return 1;   // single-buffered by definition
    return dtype == GBR_F32_FFMA || dtype == GBR_F32_FFMA_CPASYNC
               ? max_stages_for(ffma_bytes_fn, smem_optin)
               : umma_max_stages(2, smem_optin);
}

// One CTA or a CTA pair per tile: forced by gbr_gemm_tuning, else the pair
// whenever there is more than one 128-row tile or the ring is deeper than the
// one-CTA kernel can hold.
int choose_pair(int64_t rows, int stages, int smem_optin, int* pair) {
    int forced;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        forced = g_gemm_pair;
    }
    const int fk = k_sub_forced();
    const int ks = fk == 2 ? 2 : 1;   // pair choice is made for the smaller stage unless forced
    const int max1 = umma_max_stages(1, smem_optin, ks);
    if (forced == 1) {
        if (stages > max1)
            return fail(GBR_ERR_SMEM, "stages=%d exceeds %d for one CTA per tile", stages, max1);
        *pair = 1;
    } else if (forced == 2) {
        *pair = 2;
    } else {
        *pair = (rows > 128 || stages > max1) ? 2 : 1;
    }
    const int max2 = umma_max_stages(2, smem_optin, ks);
    if (*pair == 2 && stages > max2)
        return fail(GBR_ERR_SMEM, "stages=%d exceeds %d for this stage size", stages, max2);
    return GBR_OK;
}

// Fills the split fields of `s` (see split_plan.cuh); returns the scratch
// bytes the launch needs (0: no split).
size_t plan_split(GemmShape& s, int64_t units, SplitScratch kind,
                  int64_t gain_div = kSplitMinGainDiv) {
    int mode;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        mode = g_gemm_split;
    }
    return plan_split_fields(s, units, mode, gain_div) ? split_scratch_bytes(s, kind) : 0;
}

// Dynamic tile order (the split tail is then off): requested, and usable?
bool dynamic_wanted(const GemmShape& s) {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_gemm_dynamic != 0 && !s.inject.enabled && s.num_tiles > 0;
}

// Its zeroed counter, from the device's pool (*ws null when not wanted).
int dynamic_scratch(const DevCtx& c, GemmShape& s, cudaStream_t st, void** ws) {
    *ws = nullptr;
    if (!dynamic_wanted(s)) return GBR_OK;
    cudaError_t e = cudaMallocFromPoolAsync(ws, 256, c.pool, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync(tile counter)");
    if ((e = cudaMemsetAsync(*ws, 0, sizeof(uint32_t), st)) != cudaSuccess) {
        cudaFreeAsync(*ws, st);
        *ws = nullptr;
        return cuda_fail(e, "cudaMemsetAsync(tile counter)");
    }
    s.dyn_counter = static_cast<uint32_t*>(*ws);
    return GBR_OK;
}

// Scratch of one split launch from the device's pool, zeroed on the stream:
// the counters, then the tiles' sums (zero_sums false: the counters only).
int split_scratch(const DevCtx& c, GemmShape& s, SplitScratch kind, size_t bytes, cudaStream_t st,
                  void** ws, bool zero_sums = true) {
    *ws = nullptr;
    if (bytes == 0) return GBR_OK;
    cudaError_t e = cudaMallocFromPoolAsync(ws, bytes, c.pool, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocFromPoolAsync(split-tile scratch)");
    if ((e = cudaMemsetAsync(*ws, 0, zero_sums ? bytes : split_count_bytes(s, kind), st)) !=
        cudaSuccess) {
        cudaFreeAsync(*ws, st);
        *ws = nullptr;
        return cuda_fail(e, "cudaMemsetAsync(split-tile scratch)");
    }
    s.sk_count = static_cast<uint32_t*>(*ws);
    s.sk_sum = reinterpret_cast<float*>(static_cast<uint8_t*>(*ws) + split_count_bytes(s, kind));
    return GBR_OK;
}

int group_m_for(int pair) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_gemm_group_m > 0) return g_gemm_group_m;
    return pair == 2 ? 8 : 16;
}

uint32_t l2_hint_now() {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_gemm_l2_hint > 0 ? uint32_t(g_gemm_l2_hint) : 0u;
}

int copy_max_stages(uint32_t tile_bytes, int smem_optin) {
    int s = 0;
    while (s < 64 && copy_smem_bytes(s + 1, tile_bytes) <= size_t(smem_optin)) ++s;
    return s;
}

int check_umma_regs(DevCtx& c, int kind, bool grouped, int pair) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!c.umma_regs_checked[kind][grouped][pair - 1]) {
        int regs = 0;
        cudaError_t e = umma_check_registers(kind, grouped, pair, &regs);
        c.umma_regs_checked[kind][grouped][pair - 1] = true;
        c.umma_regs_ok[kind][grouped][pair - 1] = (e == cudaSuccess);
        if (e != cudaSuccess && e != cudaErrorInvalidConfiguration)
            return cuda_fail(e, "cudaFuncGetAttributes(tcgen05 GEMM)");
    }
    if (!c.umma_regs_ok[kind][grouped][pair - 1])
        return fail(GBR_ERR_CUDA,
                    "tcgen05 GEMM kernel was built with too few registers for its role split");
    return GBR_OK;
}

}  // namespace

int report_error(int code, const char* msg) { return fail(code, "%s", msg); }
void count_launch() { ++g_launches; }
uint64_t wait_timeout_ns() { return t_timeout_override ? t_timeout_override : timeout_ns(); }
FaultInjection injection_now() { return t_inject; }

int programmatic_launch_attr(cudaLaunchAttribute* attr) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_launch_overlap) return 0;
    }
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
    return 1;
}

}  // namespace gbr

using namespace gbr;

extern "C" {

const char* gbr_last_error(void) { return t_last_error.c_str(); }

long long gbr_launch_count(void) { return g_launches.load(); }

int gbr_sm_count(void) {
    DevCtx* c;
    int r = get_ctx(&c);
    return r == GBR_OK ? c->sm_count : -r;
}

int gbr_set_wait_timeout_ns(uint64_t ns) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_timeout_ns = 0;
    if (ns) g_timeout_ns = ns;
    return GBR_OK;
}

int gbr_copy_tuning(int store_lag, int ctas_per_sm, int l2_hint) {
    if (store_lag < -1 || store_lag > 1 || ctas_per_sm < -1 || ctas_per_sm == 0 || l2_hint < -1 ||
        l2_hint > 3)
        return fail(GBR_ERR_INVALID,
                    "gbr_copy_tuning: store_lag in {-1,0,1}, ctas_per_sm -1 or >= 1, l2_hint -1..3");
    std::lock_guard<std::mutex> lk(g_mu);
    g_copy_store_lag = store_lag;
    g_copy_ctas_per_sm = ctas_per_sm;
    g_copy_l2_hint = l2_hint;
    return GBR_OK;
}

int gbr_gemm_tuning(int cta_pair, int group_m, int l2_hint, int k_per_stage) {
    if (!(cta_pair == -1 || cta_pair == 1 || cta_pair == 2) || group_m == 0 || group_m < -1 ||
        l2_hint < -1 || l2_hint > 4 || !(k_per_stage == -1 || k_per_stage == 1 || k_per_stage == 2))
        return fail(GBR_ERR_INVALID,
                    "gbr_gemm_tuning: cta_pair in {-1,1,2}, group_m -1 or >= 1, l2_hint -1..4, "
                    "k_per_stage in {-1,1,2}");
    std::lock_guard<std::mutex> lk(g_mu);
    g_gemm_pair = cta_pair;
    g_gemm_group_m = group_m;
    g_gemm_l2_hint = l2_hint;
    g_gemm_k_sub = k_per_stage;
    return GBR_OK;
}

int gbr_gemm_dynamic_schedule(int on) {
    if (on != 0 && on != 1)
        return fail(GBR_ERR_INVALID, "gbr_gemm_dynamic_schedule: on must be 0 or 1");
    std::lock_guard<std::mutex> lk(g_mu);
    g_gemm_dynamic = on;
    return GBR_OK;
}

int gbr_ffma_tuning(int consumer_warps) {
    if (ffma_set_consumer_warps(consumer_warps < 0 ? 8 : consumer_warps) != 0)
        return fail(GBR_ERR_INVALID, "gbr_ffma_tuning: consumer_warps must be -1, 8 or 16");
    return GBR_OK;
}

int gbr_gemm_thin_tail(int on) {
    if (on != 0 && on != 1) return fail(GBR_ERR_INVALID, "gbr_gemm_thin_tail: on must be 0 or 1");
    std::lock_guard<std::mutex> lk(g_mu);
    g_gemm_thin = on;
    return GBR_OK;
}

int gbr_launch_overlap(int on) {
    if (on != 0 && on != 1) return fail(GBR_ERR_INVALID, "gbr_launch_overlap: on must be 0 or 1");
    std::lock_guard<std::mutex> lk(g_mu);
    g_launch_overlap = on;
    return GBR_OK;
}

int gbr_trace_buffer(void* buffer, uint64_t bytes) {
    if (buffer == nullptr) {
        std::lock_guard<std::mutex> lk(g_mu);
        g_trace = nullptr;
        g_trace_cap = 0;
        return GBR_OK;
    }
    const uint64_t region = uint64_t(kTraceMaxCtas) * kTraceRoles * 16u;
    if (bytes < kTraceHeaderBytes + region || (reinterpret_cast<uintptr_t>(buffer) & 15u))
        return fail(GBR_ERR_INVALID,
                    "gbr_trace_buffer: need a 16-byte aligned buffer of at least %llu bytes",
                    (unsigned long long)(kTraceHeaderBytes + region));
    std::lock_guard<std::mutex> lk(g_mu);
    g_trace = static_cast<uint8_t*>(buffer);
    g_trace_cap = uint32_t(std::min<uint64_t>((bytes - kTraceHeaderBytes) / region, 1u << 24));
    return GBR_OK;
}

int gbr_gemm_split_tail(int mode) {
    if (mode < -1 || mode > 1)
        return fail(GBR_ERR_INVALID, "gbr_gemm_split_tail: mode must be -1, 0 or 1");
    std::lock_guard<std::mutex> lk(g_mu);
    g_gemm_split = mode;
    return GBR_OK;
}

int gbr_max_stages(int op, int dtype, int tile_rows, int tile_cols) {
    DevCtx* c;
    int r = get_ctx(&c);
    if (r != GBR_OK) return -r;
    if (op == GBR_OP_GEMM) {
        if (dtype < GBR_F32_FFMA || dtype > GBR_F32_FFMA_CPASYNC)
            return -fail(GBR_ERR_INVALID, "bad dtype %d", dtype);
        return gemm_max_stages(dtype, c->smem_optin);
    }
    if (op == GBR_OP_COPY) {
        if (tile_rows < 1 || tile_rows > 256 || tile_cols < 4 || tile_cols > 256 || tile_cols % 4)
            return -fail(GBR_ERR_INVALID, "bad copy tile %dx%d", tile_rows, tile_cols);
        return copy_max_stages(uint32_t(tile_rows) * uint32_t(tile_cols) * 4u, c->smem_optin);
    }
    return -fail(GBR_ERR_INVALID, "bad op %d", op);
}

int gbr_device_status(gbr_stream_t stream) {
    // Allocates nothing: the regular status block is read only if a regular
    // call has already set up this device (none can have recorded anything
    // otherwise), so callers of gemm_bias_relu_tf32_noalloc may use this too.
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(GBR_ERR_INVALID, "device %d out of range", dev);
    uint32_t* status = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_dev[dev].ready) status = g_dev[dev].status;
    }
    e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t st[kStatusWords] = {};
    if (status != nullptr &&
        (e = cudaMemcpy(st, status, sizeof(st), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "reading the status block");
    if (st[0] == 0) {
        // Calls of gemm_bias_relu_tf32_noalloc record into their own scratch array.
        uint32_t na[4] = {0, 0, 0, 0};
        if (noalloc_take_status(na) == 0) return GBR_OK;
        return fail(GBR_ERR_TIMEOUT,
                    "a pipeline wait of gemm_bias_relu_tf32_noalloc timed out (site 0x%02x, CTA "
                    "%u, item %u); that call's output is undefined",
                    na[1], na[2], na[3]);
    }
    if ((e = cudaMemset(status, 0, sizeof(st))) != cudaSuccess)
        return cuda_fail(e, "clearing the status block");
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    return fail(GBR_ERR_TIMEOUT,
                "a pipeline wait timed out (site 0x%02x, CTA %u, item %u); that call's output "
                "is undefined",
                st[1], st[2], st[3]);
}

int gbr_selftest_gemm_skip_load(const void* A, const void* B, const float* bias, void* C,
                                int64_t M, int64_t N, int64_t K, int dtype, int stages, int cta,
                                int item, uint64_t limit_ns, gbr_stream_t stream) {
    if (dtype == GBR_F32_FFMA_SYNC || dtype == GBR_F32_FFMA_CPASYNC)
        return fail(GBR_ERR_UNSUPPORTED, "self test: runs on the TMA-fed rings only");
    return with_injection(cta, item, limit_ns, [&] {
        return gemm_bias_relu(A, B, bias, C, M, N, K, dtype, stages, stream);
    });
}

int gbr_selftest_noalloc_skip_load(const float* A, const float* B, const float* bias, float* C,
                                   int64_t M, int64_t N, int64_t K, int stages, int cta, int item,
                                   uint64_t limit_ns, gbr_stream_t stream) {
    return with_injection(cta, item, limit_ns, [&] {
        return gemm_bias_relu_tf32_noalloc(A, B, bias, C, M, N, K, stages, stream);
    });
}

int gbr_selftest_copy_skip_load(const void* src, void* dst, int64_t rows, int64_t cols, int stages,
                                int cta, int item, uint64_t limit_ns, gbr_stream_t stream) {
    return with_injection(cta, item, limit_ns, [&] {
        return staged_copy(src, dst, rows, cols, 128, 64, stages, stream);
    });
}

int gbr_selftest_wait_timeout(uint64_t timeout_ns_limit, gbr_stream_t stream) {
    DevCtx* c;
    int r = get_ctx(&c);
    if (r != GBR_OK) return r;
    if (timeout_ns_limit == 0 || timeout_ns_limit > 10000000000ull)
        return fail(GBR_ERR_INVALID, "self-test limit must be in (0, 10 s]");
    KernelCtl ctl = make_ctl(*c);
    ctl.timeout_ns = timeout_ns_limit;
    cudaError_t e = launch_wait_selftest(ctl, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "launching the wait self-test");
    ++g_launches;
    return GBR_OK;
}

int staged_copy(const void* src, void* dst, int64_t rows, int64_t cols, int tile_rows,
                int tile_cols, int stages, gbr_stream_t stream) {
    if (rows < 0 || cols < 0 || rows >= (int64_t(1) << 31) || cols >= (int64_t(1) << 31))
        return fail(GBR_ERR_INVALID, "staged_copy: rows/cols must be in [0, 2^31)");
    if (tile_rows < 1 || tile_rows > 256 || tile_cols < 4 || tile_cols > 256)
        return fail(GBR_ERR_INVALID, "staged_copy: tile must be 1..256 x 4..256");
    if (tile_cols % 4) return fail(GBR_ERR_ALIGN, "staged_copy: tile_cols must be a multiple of 4");
    DevCtx* c;
    int dev = 0;
    int r = get_ctx(&c, &dev);
    if (r != GBR_OK) return r;
    const uint32_t tile_bytes = uint32_t(tile_rows) * uint32_t(tile_cols) * 4u;
    const int smax = copy_max_stages(tile_bytes, c->smem_optin);
    if (stages < 1 || stages > smax)
        return fail(GBR_ERR_SMEM, "staged_copy: stages=%d outside [1, %d] for a %dx%d fp32 tile",
                    stages, smax, tile_rows, tile_cols);
    if (rows == 0 || cols == 0) return GBR_OK;
    if (!src || !dst) return fail(GBR_ERR_INVALID, "staged_copy: NULL buffer");
    if (!aligned16(src) || !aligned16(dst))
        return fail(GBR_ERR_ALIGN, "staged_copy: buffers must be 16-byte aligned");
    if (cols % 4) return fail(GBR_ERR_ALIGN, "staged_copy: cols must be a multiple of 4");
    const size_t bytes = size_t(rows) * size_t(cols) * 4u;
    if (overlaps(src, bytes, dst, bytes)) return fail(GBR_ERR_INVALID, "staged_copy: src and dst overlap");

    CUtensorMap ms, md;
    if ((r = encode_2d(&ms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, src, uint64_t(cols), uint64_t(rows),
                       uint64_t(cols) * 4u, uint32_t(tile_cols), uint32_t(tile_rows),
                       CU_TENSOR_MAP_SWIZZLE_NONE, "copy src")) != GBR_OK)
        return r;
    if ((r = encode_2d(&md, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dst, uint64_t(cols), uint64_t(rows),
                       uint64_t(cols) * 4u, uint32_t(tile_cols), uint32_t(tile_rows),
                       CU_TENSOR_MAP_SWIZZLE_NONE, "copy dst")) != GBR_OK)
        return r;

    CopyArgs a;
    a.rows = int32_t(rows);
    a.cols = int32_t(cols);
    a.tile_rows = tile_rows;
    a.tile_cols = tile_cols;
    a.tiles_c = int32_t(cdiv(cols, tile_cols));
    a.num_tiles = cdiv(rows, tile_rows) * int64_t(a.tiles_c);
    a.stages = stages;
    a.tile_bytes = tile_bytes;
    int lag, cps, hint;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        lag = g_copy_store_lag;
        cps = g_copy_ctas_per_sm;
        hint = g_copy_l2_hint;
    }
    // Auto: the loaded lines are marked evict-first (each is read exactly once);
    // measured on the 256 MiB copy, +4% over no hint.
    a.l2_hint = hint < 0 ? 1u : uint32_t(hint);
    a.inject = t_inject;
    a.store_lag = (lag < 0) ? (stages >= 2 ? 1 : 0) : lag;
    if (a.store_lag == 1 && stages < 2) a.store_lag = 0;
    a.ctl = make_ctl(*c);

    const size_t smem = copy_smem_bytes(stages, tile_bytes);
    int occ = 0;
    if (cudaError_t e2 = copy_prepare(smem))
        return cuda_fail(e2, "cudaFuncSetAttribute(staged copy)");
    r = prepared(dev, {kPrepCopy, 0, 0, 0, int64_t(smem)}, &occ, [&](int* v) {
        const cudaError_t e2 = copy_occupancy(smem, v);
        return e2 == cudaSuccess ? int(GBR_OK) : cuda_fail(e2, "occupancy(staged copy)");
    });
    if (r != GBR_OK) return r;
    cudaError_t e;
    if (occ < 1) return fail(GBR_ERR_SMEM, "staged_copy: kernel does not fit on an SM");
    if (cps > 0 && cps < occ) occ = cps;
    const int64_t grid = std::min<int64_t>(a.num_tiles, int64_t(c->sm_count) * occ);
    e = launch_staged_copy(ms, md, a, int(grid), smem, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "launching staged copy");
    ++g_launches;
    return GBR_OK;
}

int gemm_bias_relu(const void* A, const void* B, const float* bias, void* C, int64_t M, int64_t N,
                   int64_t K, int dtype, int stages, gbr_stream_t stream) {
    if (dtype < GBR_F32_FFMA || dtype > GBR_F32_FFMA_CPASYNC)
        return fail(GBR_ERR_INVALID, "gemm_bias_relu: unknown dtype %d", dtype);
    const int64_t lim = int64_t(1) << 31;
    if (M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim)
        return fail(GBR_ERR_INVALID, "gemm_bias_relu: M, N, K must be in [0, 2^31)");
    DevCtx* c;
    int dev = 0;
    int r = get_ctx(&c, &dev);
    if (r != GBR_OK) return r;
    const int smax = gemm_max_stages(dtype, c->smem_optin);
    if (stages < 1 || stages > smax)
        return fail(GBR_ERR_SMEM, "gemm_bias_relu: stages=%d outside [1, %d] for dtype %d", stages,
                    smax, dtype);
    if (M == 0 || N == 0) return GBR_OK;
    const uint64_t es = dtype == GBR_BF16 ? 2 : 4;
    if (!C || !bias || (K > 0 && (!A || !B)))
        return fail(GBR_ERR_INVALID, "gemm_bias_relu: NULL buffer");
    if (!aligned16(C) || !aligned16(bias) || (K > 0 && (!aligned16(A) || !aligned16(B))))
        return fail(GBR_ERR_ALIGN, "gemm_bias_relu: buffers must be 16-byte aligned");
    if ((uint64_t(N) * es) % 16 || (uint64_t(K) * es) % 16)
        return fail(GBR_ERR_ALIGN,
                    "gemm_bias_relu: row pitches K*%d and N*%d bytes must be multiples of 16",
                    int(es), int(es));
    const size_t c_bytes = size_t(M) * size_t(N) * es;
    if ((K > 0 && (overlaps(C, c_bytes, A, size_t(M) * K * es) ||
                   overlaps(C, c_bytes, B, size_t(K) * N * es))) ||
        overlaps(C, c_bytes, bias, size_t(N) * 4))
        return fail(GBR_ERR_INVALID, "gemm_bias_relu: C overlaps an input");

    GemmShape s;
    memset(&s, 0, sizeof(s));
    s.M = int32_t(M);
    s.N = int32_t(N);
    s.K = int32_t(K);
    s.stages = stages;
    s.bias = bias;
    s.C = C;
    s.ctl = make_ctl(*c);
    s.inject = t_inject;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;

    if (dtype == GBR_F32_FFMA_SYNC) {
        s.m_tiles = int32_t(cdiv(M, kFfmaBM));
        s.n_tiles = int32_t(cdiv(N, kFfmaBN));
        s.num_kb = int32_t(cdiv(K, kFfmaBK));
        s.num_tiles = s.m_tiles * s.n_tiles;
        s.group_m = 8;
        if ((e = launch_gemm_ffma_sync(static_cast<const float*>(A), static_cast<const float*>(B), s,
                                       st)) != cudaSuccess)
            return cuda_fail(e, "launching the homogeneous FFMA GEMM");
        ++g_launches;
        return GBR_OK;
    }

    if (dtype == GBR_F32_FFMA || dtype == GBR_F32_FFMA_CPASYNC) {
        s.A = A;
        s.B = B;
        s.m_tiles = int32_t(cdiv(M, kFfmaBM));
        s.n_tiles = int32_t(cdiv(N, kFfmaBN));
        s.num_kb = int32_t(cdiv(K, kFfmaBK));
        s.num_tiles = s.m_tiles * s.n_tiles;
        s.group_m = 8;
        CUtensorMap ma, mb;
        const void* pa = K > 0 ? A : C;
        const void* pb = K > 0 ? B : C;
        const uint64_t kk = K > 0 ? uint64_t(K) : uint64_t(N);
        if ((r = encode_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, pa, kk, uint64_t(M), kk * 4, 32,
                           128, CU_TENSOR_MAP_SWIZZLE_128B, "A")) != GBR_OK)
            return r;
        if ((r = encode_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, pb, uint64_t(N),
                           K > 0 ? uint64_t(K) : uint64_t(M), uint64_t(N) * 4, 32, 32,
                           CU_TENSOR_MAP_SWIZZLE_128B, "B")) != GBR_OK)
            return r;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            if (!c->ffma_regs_checked) {
                int regs = 0;
                e = ffma_check_registers(&regs);
                c->ffma_regs_checked = true;
                c->ffma_regs_ok = (e == cudaSuccess);
                if (e != cudaSuccess && e != cudaErrorInvalidConfiguration)
                    return cuda_fail(e, "cudaFuncGetAttributes(FFMA GEMM)");
            }
            if (!c->ffma_regs_ok)
                return fail(GBR_ERR_CUDA, "FFMA GEMM kernel was built with too few registers for its role split");
        }
        const size_t smem = ffma_smem_bytes(stages);
        int occ = 0;
        if ((e = ffma_prepare(smem)) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(FFMA)");
        r = prepared(dev, {kPrepFfma, ffma_consumer_warps(), 0, 0, int64_t(smem)}, &occ, [&](int* v) {
            const cudaError_t e2 = ffma_occupancy(smem, v);
            return e2 == cudaSuccess ? int(GBR_OK) : cuda_fail(e2, "occupancy(FFMA)");
        });
        if (r != GBR_OK) return r;
        if (occ < 1) return fail(GBR_ERR_SMEM, "FFMA GEMM does not fit on an SM");
        const int64_t units = int64_t(c->sm_count) * occ;
        // The split tail (TMA producer): the whole tiles of the first rounds in
        // one launch, then the last partial round's k-blocks dealt out evenly
        // to every CTA in a second launch of the split instance.  Not while an
        // event trace is recorded: each launch writes its CTAs' trace from the
        // start, so the second would overwrite the first.
        GemmShape tail = s;
        const size_t split_bytes =
            dtype == GBR_F32_FFMA && s.ctl.trace == nullptr
                ? plan_split(tail, units, ffma_split_scratch(), kSplitMinGainDivOrdered)
                : 0;
        if (split_bytes) {
            void* ws = nullptr;
            if ((r = split_scratch(*c, tail, ffma_split_scratch(), split_bytes, st, &ws, false)) !=
                GBR_OK)
                return r;
            GemmShape whole = s;
            whole.num_tiles = tail.dp_tiles;
            e = launch_gemm_ffma(ma, mb, whole, int(units), smem, st, false, false);
            if (e == cudaSuccess) {
                ++g_launches;
                e = launch_gemm_ffma(ma, mb, tail, int(units), smem, st, false, true);
            }
            cudaFreeAsync(ws, st);
            if (e != cudaSuccess) return cuda_fail(e, "launching FFMA GEMM");
            ++g_launches;
            return GBR_OK;
        }
        const int grid = int(std::min<int64_t>(s.num_tiles, units));
        if ((e = launch_gemm_ffma(ma, mb, s, grid, smem, st, dtype == GBR_F32_FFMA_CPASYNC)) !=
            cudaSuccess)
            return cuda_fail(e, "launching FFMA GEMM");
        ++g_launches;
        return GBR_OK;
    }

    const int kind = dtype == GBR_BF16 ? kUmmaBf16 : kUmmaTf32;
    const CUtensorMapDataType dt =
        dtype == GBR_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const uint32_t bk = uint32_t(128 / es);          // K per stage
    const uint32_t panel_cols = uint32_t(128 / es);  // B panel width; also the C store box width
    int pair = 1;
    if ((r = choose_pair(M, stages, c->smem_optin, &pair)) != GBR_OK) return r;
    if (s.inject.enabled && pair_forced() != 2) {
        // The self test runs one CTA per tile unless gbr_gemm_tuning forces
        // the CTA pair; `cta` then names the pair, both of whose CTAs leave
        // the item unfilled.
        if (stages > umma_max_stages(1, c->smem_optin))
            return fail(GBR_ERR_SMEM, "self test: stages must fit one CTA per tile");
        pair = 1;
    }
    s.k_sub = uint32_t(s.inject.enabled && pair == 1 ? 1
                                                     : choose_k_sub(pair, stages, c->smem_optin));
    s.m_tiles = int32_t(cdiv(M, int64_t(kUmmaBM) * pair));
    s.n_tiles = int32_t(cdiv(N, kUmmaBN));
    s.num_kb = int32_t(cdiv(K, int64_t(bk) * s.k_sub));
    s.num_tiles = s.m_tiles * s.n_tiles;
    s.group_m = group_m_for(pair);
    s.l2_hint = l2_hint_now();
    CUtensorMap ma, mb, mc;
    if ((r = encode_2d(&mc, dt, C, uint64_t(N), uint64_t(M), uint64_t(N) * es, panel_cols, 32,
                       CU_TENSOR_MAP_SWIZZLE_128B, "C")) != GBR_OK)
        return r;
    if ((r = check_umma_regs(*c, kind, false, pair)) != GBR_OK) return r;
    const size_t smem = umma_smem_bytes(stages, pair, int(s.k_sub));
    if ((e = umma_prepare(kind, false, pair, smem)) != cudaSuccess)
        return cuda_fail(e, "cudaFuncSetAttribute(tcgen05 GEMM)");
    const int64_t units = c->sm_count / pair;
    const size_t split_bytes =
        dynamic_wanted(s) ? 0 : plan_split(s, units, umma_split_scratch(pair));
    const int grid = pair * int(split_bytes ? units : std::min<int64_t>(s.num_tiles, units));
    if (K > 0) {
        if ((r = encode_2d(&ma, dt, A, uint64_t(K), uint64_t(M), uint64_t(K) * es, bk, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B, "A")) != GBR_OK)
            return r;
        // B row-major [K, N] as N-major panels of panel_cols x bk (MN-major
        // operand); TF32 panels in the 32-byte-atom swizzle kind::tf32 reads.
        // When N is a whole number of panels, B is seen as a 3-D tensor
        // (column in panel, K, panel), so that one box brings all of a CTA's
        // panels of a K slice, laid out panel after panel; its addresses stay
        // inside B because every panel is whole.
        const CUtensorMapSwizzle swz =
            kind == kUmmaTf32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B;
        s.b_panels_3d = N % int64_t(panel_cols) == 0 ? 1u : 0u;
        if (s.b_panels_3d) {
            const uint64_t dims[3] = {panel_cols, uint64_t(K), uint64_t(N) / panel_cols};
            const uint64_t strides[2] = {uint64_t(N) * es, uint64_t(panel_cols) * es};
            const uint32_t box[3] = {panel_cols, bk, uint32_t(kUmmaBN / pair) / panel_cols};
            r = encode(&mb, dt, 3, B, dims, strides, box, swz, "B panels");
        } else {
            r = encode_2d(&mb, dt, B, uint64_t(N), uint64_t(K), uint64_t(N) * es, panel_cols, bk,
                          swz, "B");
        }
        if (r != GBR_OK) return r;
    } else {
        ma = mc;  // never read: no k-blocks are loaded when K == 0
        mb = mc;
    }
    void* ws = nullptr;
    void* dyn_ws = nullptr;
    if ((r = split_scratch(*c, s, umma_split_scratch(pair), split_bytes, st, &ws)) != GBR_OK ||
        (r = dynamic_scratch(*c, s, st, &dyn_ws)) != GBR_OK) {
        if (ws) cudaFreeAsync(ws, st);
        return r;
    }
    e = launch_gemm_umma(kind, pair, ma, mb, mc, s, grid, smem, st);
    if (ws) cudaFreeAsync(ws, st);
    if (dyn_ws) cudaFreeAsync(dyn_ws, st);
    if (e != cudaSuccess) return cuda_fail(e, "launching tcgen05 GEMM");
    ++g_launches;
    return GBR_OK;
}

int gemm_bias_relu_grouped(const void* X, const void* W, const float* bias, void* C,
                           const int32_t* counts_host, int num_groups, int64_t K, int64_t N,
                           int dtype, int stages, gbr_stream_t stream) {
    if (dtype != GBR_BF16)
        return fail(GBR_ERR_UNSUPPORTED, "gemm_bias_relu_grouped: only GBR_BF16 is built");
    if (num_groups < 1 || num_groups > kMaxGroups)
        return fail(GBR_ERR_INVALID, "gemm_bias_relu_grouped: num_groups must be 1..%d", kMaxGroups);
    if (!counts_host) return fail(GBR_ERR_INVALID, "gemm_bias_relu_grouped: NULL counts");
    const int64_t lim = int64_t(1) << 31;
    if (K < 0 || N < 0 || K >= lim || N >= lim)
        return fail(GBR_ERR_INVALID, "gemm_bias_relu_grouped: K, N must be in [0, 2^31)");
    int64_t T = 0;
    for (int e = 0; e < num_groups; ++e) {
        if (counts_host[e] < 0) return fail(GBR_ERR_INVALID, "gemm_bias_relu_grouped: negative count");
        T += counts_host[e];
    }
    if (T >= lim) return fail(GBR_ERR_INVALID, "gemm_bias_relu_grouped: too many rows");
    DevCtx* c;
    int dev = 0;
    int r = get_ctx(&c, &dev);
    if (r != GBR_OK) return r;
    const int smax = gemm_max_stages(dtype, c->smem_optin);
    if (stages < 1 || stages > smax)
        return fail(GBR_ERR_SMEM, "gemm_bias_relu_grouped: stages=%d outside [1, %d]", stages, smax);
    if (T == 0 || N == 0) return GBR_OK;
    const uint64_t es = 2;
    if (!C || !bias || (K > 0 && (!X || !W)))
        return fail(GBR_ERR_INVALID, "gemm_bias_relu_grouped: NULL buffer");
    if (!aligned16(C) || !aligned16(bias) || (K > 0 && (!aligned16(X) || !aligned16(W))))
        return fail(GBR_ERR_ALIGN, "gemm_bias_relu_grouped: buffers must be 16-byte aligned");
    if ((uint64_t(N) * es) % 16 || (uint64_t(K) * es) % 16)
        return fail(GBR_ERR_ALIGN, "gemm_bias_relu_grouped: K and N must be multiples of 8");
    const size_t c_bytes = size_t(T) * size_t(N) * es;
    if ((K > 0 && (overlaps(C, c_bytes, X, size_t(T) * K * es) ||
                   overlaps(C, c_bytes, W, size_t(num_groups) * K * N * es))) ||
        overlaps(C, c_bytes, bias, size_t(num_groups) * N * 4))
        return fail(GBR_ERR_INVALID, "gemm_bias_relu_grouped: C overlaps an input");

    GemmShape s;
    memset(&s, 0, sizeof(s));
    s.M = int32_t(T);
    s.N = int32_t(N);
    s.K = int32_t(K);
    s.stages = stages;
    s.bias = bias;
    s.C = C;
    s.ctl = make_ctl(*c);
    s.n_tiles = int32_t(cdiv(N, kUmmaBN));
    s.k_sub = uint32_t(k_sub_forced() == 2 ? 2 : 1);
    int pair = 1;
    {
        // Auto: the pair as soon as some expert spans more than one 128-row
        // tile.  Measured on GB300 (K 4096, N 14336), a 128 x 256 one-CTA tile
        // costs about 0.65 of a 256 x 256 pair tile, so the pair is cheaper
        // even where its 256-row tiles pad more rows (skewed experts of 2048
        // down to 32 rows: 1465 against 1107 TFLOP/s); the short tails run as
        // thin tiles.
        int64_t maxn = 0;
        for (int e2 = 0; e2 < num_groups; ++e2) maxn = std::max<int64_t>(maxn, counts_host[e2]);
        int forced;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            forced = g_gemm_pair;
        }
        const int max1 = umma_max_stages(1, c->smem_optin, int(s.k_sub));
        const int max2 = umma_max_stages(2, c->smem_optin, int(s.k_sub));
        if (forced == 1 && stages > max1)
            return fail(GBR_ERR_SMEM, "stages=%d exceeds %d for one CTA per tile", stages, max1);
        if (forced > 0)
            pair = forced;
        else
            pair = (stages > max1 || maxn > 128) ? 2 : 1;
        if (pair == 2 && stages > max2)
            return fail(GBR_ERR_SMEM, "stages=%d exceeds %d for this stage size", stages, max2);
        s.k_sub = uint32_t(choose_k_sub(pair, stages, c->smem_optin));
    }
    s.num_kb = int32_t(cdiv(K, int64_t(64) * s.k_sub));
    s.group_m = group_m_for(pair);
    s.l2_hint = l2_hint_now();
    GroupTable g;
    memset(&g, 0, sizeof(g));
    g.num_groups = num_groups;
    CUtensorMap mc[kMaxGroups];
    int64_t off = 0, tiles = 0;
    int last_valid = -1;
    for (int e = 0; e < num_groups; ++e) {
        const int64_t n_e = counts_host[e];
        g.row_off[e] = int32_t(off);
        g.rows[e] = int32_t(n_e);
        g.m_tiles[e] = int32_t(cdiv(n_e, int64_t(kUmmaBM) * pair));
        g.tile_start[e] = int32_t(tiles);
        tiles += int64_t(g.m_tiles[e]) * s.n_tiles;
        if (n_e > 0) {
            const void* base = static_cast<const uint8_t*>(C) + size_t(off) * size_t(N) * es;
            if ((r = encode_2d(&mc[e], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, uint64_t(N),
                               uint64_t(n_e), uint64_t(N) * es, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B,
                               "C[e]")) != GBR_OK)
                return r;
            last_valid = e;
        }
        off += n_e;
    }
    for (int e = 0; e < num_groups; ++e)
        if (counts_host[e] == 0) mc[e] = mc[last_valid];  // never used: the group has no tiles
    g.tile_start[num_groups] = int32_t(tiles);
    s.num_tiles = int32_t(tiles);
    s.m_tiles = 0;
    // Thin tails: on the CTA pair, an expert's last M-tile with at most 128
    // rows runs transposed (the rows become the MMA's N, rounded up to 16)
    // instead of padding them to 256.
    bool any_thin = false;
    {
        int thin_on;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            thin_on = g_gemm_thin;
        }
        for (int e = 0; e < num_groups; ++e) {
            const int64_t t = int64_t(counts_host[e]) - int64_t(g.m_tiles[e] - 1) * 256;
            if (pair == 2 && thin_on && counts_host[e] > 0 && t <= 128) {
                g.thin[e] = int32_t(t);
                any_thin = true;
            }
        }
    }
    CUtensorMap mx, mw;
    if (K > 0) {
        if ((r = encode_2d(&mx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, uint64_t(K), uint64_t(T),
                           uint64_t(K) * es, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, "X")) != GBR_OK)
            return r;
        const uint64_t dims[3] = {uint64_t(N), uint64_t(K), uint64_t(num_groups)};
        const uint64_t strides[2] = {uint64_t(N) * es, uint64_t(K) * uint64_t(N) * es};
        const uint32_t box[3] = {64, 64, 1};
        if ((r = encode(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B, "W")) != GBR_OK)
            return r;
    } else {
        mx = mc[last_valid];
        mw = mc[last_valid];
    }
    if ((r = check_umma_regs(*c, kUmmaBf16, true, pair)) != GBR_OK) return r;
    const size_t smem = umma_smem_bytes(stages, pair, int(s.k_sub));
    cudaError_t e = umma_prepare(kUmmaBf16, true, pair, smem);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(grouped GEMM)");
    const int64_t units = c->sm_count / pair;
    // Thin tiles are never split (their accumulator is transposed).
    const size_t split_bytes =
        (dynamic_wanted(s) || any_thin) ? 0 : plan_split(s, units, umma_split_scratch(pair));
    const int grid = pair * int(split_bytes ? units : std::min<int64_t>(s.num_tiles, units));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void* ws = nullptr;
    void* dyn_ws = nullptr;
    if ((r = split_scratch(*c, s, umma_split_scratch(pair), split_bytes, st, &ws)) != GBR_OK ||
        (r = dynamic_scratch(*c, s, st, &dyn_ws)) != GBR_OK) {
        if (ws) cudaFreeAsync(ws, st);
        return r;
    }
    e = launch_gemm_umma_grouped(pair, mx, mw, mc, g, s, int64_t(N), grid, smem, st);
    if (ws) cudaFreeAsync(ws, st);
    if (dyn_ws) cudaFreeAsync(dyn_ws, st);
    if (e != cudaSuccess) return cuda_fail(e, "launching grouped GEMM");
    ++g_launches;
    return GBR_OK;
}

// ------------------------------------------------------------ host buffers
int gemm_bias_relu_host(const void* hA, const void* hB, const float* hbias, void* hC, int64_t M,
                        int64_t N, int64_t K, int dtype, int stages, gbr_stream_t stream) {
    if (dtype < GBR_F32_FFMA || dtype > GBR_F32_FFMA_CPASYNC)
        return fail(GBR_ERR_INVALID, "gemm_bias_relu_host: unknown dtype %d", dtype);
    const int64_t lim = int64_t(1) << 31;
    if (M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim)
        return fail(GBR_ERR_INVALID, "gemm_bias_relu_host: M, N, K must be in [0, 2^31)");
    DevCtx* c;
    int r = get_ctx(&c);
    if (r != GBR_OK) return r;
    const int smax = gemm_max_stages(dtype, c->smem_optin);
    if (stages < 1 || stages > smax)
        return fail(GBR_ERR_SMEM, "gemm_bias_relu_host: stages=%d outside [1, %d]", stages, smax);
    if (M == 0 || N == 0) return GBR_OK;
    if (!hC || !hbias || (K > 0 && (!hA || !hB)))
        return fail(GBR_ERR_INVALID, "gemm_bias_relu_host: NULL buffer");
    const size_t es = dtype == GBR_BF16 ? 2 : 4;
    if ((size_t(N) * es) % 16 || (size_t(K) * es) % 16)
        return fail(GBR_ERR_ALIGN, "gemm_bias_relu_host: row pitches must be multiples of 16 bytes");
    auto up = [](size_t x) { return (x + 255u) & ~size_t(255); };
    const size_t a_bytes = size_t(M) * size_t(K) * es, b_bytes = size_t(K) * size_t(N) * es;
    const size_t bias_bytes = size_t(N) * 4, c_bytes = size_t(M) * size_t(N) * es;
    const size_t off_b = up(a_bytes), off_bias = off_b + up(b_bytes), off_c = off_bias + up(bias_bytes);
    const size_t total = off_c + up(c_bytes);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lk(c->host_mu);
    cudaError_t e;
    if (!c->host_ready) {
        for (auto& hs : c->host_streams)
            if ((e = cudaStreamCreateWithFlags(&hs, cudaStreamNonBlocking)) != cudaSuccess)
                return cuda_fail(e, "cudaStreamCreateWithFlags");
        for (auto& ev : c->host_events)
            if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
                return cuda_fail(e, "cudaEventCreateWithFlags");
        c->host_ready = true;
    }
    cudaStream_t s_in = c->host_streams[0], s_cmp = c->host_streams[1], s_out = c->host_streams[2];
    cudaEvent_t* ev = c->host_events;
    void* ws = nullptr;
    if ((e = cudaMallocFromPoolAsync(&ws, total, c->pool, st)) != cudaSuccess)
        return cuda_fail(e, "cudaMallocFromPoolAsync(host GEMM buffers)");
    uint8_t* base = static_cast<uint8_t*>(ws);
    uint8_t *dA = base, *dB = base + off_b, *dC = base + off_c;
    float* dbias = reinterpret_cast<float*>(base + off_bias);

    // M in chunks (multiples of 256 rows): chunk i computes while chunk i + 1
    // is copied in and chunk i - 1 is copied out.  B and bias go first.
    const int64_t want = std::max<int64_t>(1, std::min<int64_t>(kHostChunks, M / 1024));
    const int64_t rows = std::max<int64_t>(256, (cdiv(M, want) + 255) / 256 * 256);
    const int chunks = int(cdiv(M, rows));
    int first_err = GBR_OK;
    std::string first_msg;
    auto note = [&](int code) {
        if (code != GBR_OK && first_err == GBR_OK) {
            first_err = code;
            first_msg = t_last_error;
        }
    };
    auto cu = [&](cudaError_t err, const char* what) {
        if (err != cudaSuccess) note(cuda_fail(err, what));
    };
    cu(cudaEventRecord(ev[0], st), "cudaEventRecord(fork)");
    for (cudaStream_t hs : {s_in, s_cmp, s_out}) cu(cudaStreamWaitEvent(hs, ev[0], 0), "fork");
    cu(cudaMemcpyAsync(dbias, hbias, bias_bytes, cudaMemcpyHostToDevice, s_in), "copy bias in");
    if (K > 0) cu(cudaMemcpyAsync(dB, hB, b_bytes, cudaMemcpyHostToDevice, s_in), "copy B in");
    for (int i = 0; i < chunks; ++i) {
        const int64_t r0 = int64_t(i) * rows, n = std::min<int64_t>(rows, M - r0);
        cudaEvent_t in = ev[1 + 2 * i], done = ev[2 + 2 * i];
        if (K > 0)
            cu(cudaMemcpyAsync(dA + size_t(r0) * size_t(K) * es,
                               static_cast<const uint8_t*>(hA) + size_t(r0) * size_t(K) * es,
                               size_t(n) * size_t(K) * es, cudaMemcpyHostToDevice, s_in),
               "copy A chunk in");
        cu(cudaEventRecord(in, s_in), "cudaEventRecord(in)");
        cu(cudaStreamWaitEvent(s_cmp, in, 0), "wait in");
        if (first_err == GBR_OK)
            note(gemm_bias_relu(dA + size_t(r0) * size_t(K) * es, dB, dbias,
                                dC + size_t(r0) * size_t(N) * es, n, N, K, dtype, stages,
                                reinterpret_cast<gbr_stream_t>(s_cmp)));
        cu(cudaEventRecord(done, s_cmp), "cudaEventRecord(computed)");
        cu(cudaStreamWaitEvent(s_out, done, 0), "wait computed");
        cu(cudaMemcpyAsync(static_cast<uint8_t*>(hC) + size_t(r0) * size_t(N) * es,
                           dC + size_t(r0) * size_t(N) * es, size_t(n) * size_t(N) * es,
                           cudaMemcpyDeviceToHost, s_out),
           "copy C chunk out");
    }
    // Join: the caller's stream continues once the last chunk is back on the
    // host (it waited for every computation, which waited for every copy in).
    cu(cudaEventRecord(ev[kHostEvents - 1], s_out), "cudaEventRecord(join)");
    cu(cudaStreamWaitEvent(st, ev[kHostEvents - 1], 0), "join");
    cu(cudaFreeAsync(ws, st), "cudaFreeAsync(host GEMM buffers)");
    if (first_err != GBR_OK) {
        t_last_error = first_msg;
        return first_err;
    }
    return GBR_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- self test
namespace gbr {
namespace {
__global__ void wait_selftest_kernel(KernelCtl ctl) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_addr(&bar), 1);
        abort_flag = 0;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: the bounded wait must give up.
        mbar_wait(ptx::smem_addr(&bar), 0, ctl, &abort_flag, kSiteSelfTest, 0);
    }
    __syncthreads();
}
}  // namespace

cudaError_t launch_wait_selftest(KernelCtl ctl, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(ctl);
    return cudaGetLastError();
}
}  // namespace gbr
