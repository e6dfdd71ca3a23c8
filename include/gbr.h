/*
 * gbr.h -- C ABI of the warp-specialized TMA/mbarrier pipeline library for
 * NVIDIA GB300 (sm_103a).
 *
 * Two operators, both built as one producer role that streams tiles through
 * an S-slot shared-memory ring guarded by per-slot "full" and "empty"
 * mbarriers (slot = i % S, full wait parity = (i / S) & 1, empty wait parity =
 * ((i / S) & 1) ^ 1), and consumer roles that work on full slots and release
 * them:
 *
 *   gemm_bias_relu          C = ReLU(A * B + bias)
 *   gemm_bias_relu_grouped  the same per expert segment (MoE-style), one launch
 *   gemm_bias_relu_host     gemm_bias_relu on host buffers, copies overlapped
 *   staged_copy             gmem -> smem -> gmem through the ring (TMA both ways)
 *
 * Conventions shared by every entry point
 *   - Tensors are contiguous, row-major, resident in device memory of the
 *     current CUDA device, allocated and owned by the caller.  The library
 *     never frees or retains them after the call's work has finished.
 *   - `stream` is a cudaStream_t (a CUstream_st pointer); NULL is the legacy
 *     default stream.  Every call is asynchronous on that stream.
 *   - Return value: GBR_OK, or an error code for host-side validation or launch
 *     failures, with a message available from gbr_last_error() on the calling
 *     thread.  Nothing is launched when validation fails.
 *   - Device-side failures (a pipeline wait that exceeded its time limit) are
 *     reported by gbr_device_status(), which also clears them.  The status
 *     block keeps the FIRST timeout recorded since the last read.
 *   - Global addresses must be 16-byte aligned and every row pitch must be a
 *     multiple of 16 bytes (the TMA rule): fp32 row lengths a multiple of 4,
 *     bf16 row lengths a multiple of 8.  Otherwise GBR_ERR_ALIGN.
 *   - The library keeps, per device, a 64-byte status block it allocates on
 *     first use, a memory pool for per-call scratch (taken and returned in
 *     stream order: split-tile sums, the dynamic tile counter), the
 *     streams and events of gemm_bias_relu_host, and cached device attributes.
 */
#ifndef GBR_H_
#define GBR_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *gbr_stream_t;

typedef enum {
    GBR_F32_FFMA = 0,     /* fp32 in/out, strict fp32 FMA on CUDA cores        */
    GBR_F32_TF32 = 1,     /* fp32 in/out, TF32 tensor-core multiply, fp32 acc   */
    GBR_BF16 = 2,         /* bf16 A/B/C, fp32 bias, fp32 accumulation in TMEM   */
    GBR_F32_FFMA_SYNC = 3, /* GBR_F32_FFMA computed by the homogeneous loop of
                             "pwwt.cn news/4436243" section 1.1 (all threads
                             load, sync, compute, sync; no roles, no ring):
                             the baseline the pipeline is measured against.
                             stages must be 1.                                 */
    GBR_F32_FFMA_CPASYNC = 4 /* GBR_F32_FFMA with the historical producer: the
                             producer warpgroup fills each ring stage with
                             16-byte cp.async copies and arrives on full[s]
                             with cp.async.mbarrier.arrive, instead of one TMA
                             lane.  Same consumers, ring and results.          */
} gbr_dtype;

typedef enum {
    GBR_OK = 0,
    GBR_ERR_INVALID = 1,     /* bad size, pointer, count or overlapping buffers */
    GBR_ERR_UNSUPPORTED = 2, /* dtype/operator combination not built            */
    GBR_ERR_ALIGN = 3,       /* address or row pitch violates the TMA rule       */
    GBR_ERR_SMEM = 4,        /* stages outside [1, gbr_max_stages(...)]          */
    GBR_ERR_CUDA = 5,        /* CUDA runtime/driver error (message has details)  */
    GBR_ERR_TIMEOUT = 6      /* a device-side pipeline wait gave up              */
} gbr_status;

/*
 * gemm_bias_relu -- C[m,n] = max(0, bias[n] + sum_k A[m,k] * B[k,n]).
 *
 * Defined by the SGEMM test bench of "pwwt.cn news/4436243", section 4.1
 * (inputs A[M,K], B[K,N]; output A*B + bias followed by ReLU), computed by
 * the warp-specialized ring of section 3.4 of the same page and of
 * "gpu_warp_specialization" ("End-to-end flow").
 *
 *   A     [M, K] row-major; fp32 (GBR_F32_*) or bf16 (GBR_BF16).  Read only.
 *         (GBR_F32_FFMA_SYNC reads A and B with plain loads, not TMA.)
 *   B     [K, N] row-major; same type as A.  Read only.
 *   bias  [N] fp32.  Read only.
 *   C     [M, N] row-major; fp32 (GBR_F32_*) or bf16 (GBR_BF16, rounded to
 *         nearest even from the fp32 result).  Written; must not overlap the
 *         inputs.
 *   M, N, K  >= 0 and < 2^31.  M == 0 or N == 0: nothing to do.  K == 0:
 *         C = max(0, bias) in every row.  A and B may be NULL when K == 0.
 *   dtype gbr_dtype.
 *   stages  ring depth S, 1 <= S <= gbr_max_stages(GBR_OP_GEMM, dtype, 0, 0)
 *         (GBR_ERR_SMEM otherwise).  Tiles: FFMA 128x128x32 fp32;
 *         tcgen05 128x256 per CTA, or 256x256 per CTA pair (gbr_gemm_tuning),
 *         with 128 bytes of K per stage (bf16 K=64, tf32 K=32), or 256 bytes
 *         when S <= 3 on the CTA pair (bf16 K=128, tf32 K=64).
 *   stream  see above.
 * Ragged M, N and K need no padding: TMA loads zero-fill outside the tensor
 * and TMA stores drop rows/columns outside it.
 */
int gemm_bias_relu(const void *A, const void *B, const float *bias, void *C, int64_t M,
                   int64_t N, int64_t K, int dtype, int stages, gbr_stream_t stream);

/*
 * gemm_bias_relu_grouped -- per expert e (0 <= e < num_groups):
 *   C[r,n] = max(0, b[e,n] + sum_k X[r,k] * W[e,k,n]) for r in
 *   [off_e, off_e + counts[e]), off_e = counts[0] + ... + counts[e-1].
 *
 * The mixture-of-experts operator that motivates "pwwt.cn news/4436243"
 * (section 1.1), expressed as the same GEMM + bias + ReLU per expert and run
 * as ONE persistent warp-specialized launch over all experts' tiles.
 *
 *   X     [T, K] rows already grouped by expert, T = sum(counts).  Read only.
 *   W     [G, K, N] expert weights.  Read only.
 *   bias  [G, N] fp32.  Read only.
 *   C     [T, N] written row segment by row segment.
 *   counts_host  HOST array of num_groups non-negative row counts (read
 *         during the call only); a zero count gives the expert no tiles.
 *   num_groups  1..32.
 *   dtype GBR_BF16 (GBR_ERR_UNSUPPORTED for the others).
 *   stages  as for gemm_bias_relu.
 * Routing and permutation of tokens are the caller's.
 */
int gemm_bias_relu_grouped(const void *X, const void *W, const float *bias, void *C,
                           const int32_t *counts_host, int num_groups, int64_t K, int64_t N,
                           int dtype, int stages, gbr_stream_t stream);

/*
 * staged_copy -- dst = src, moved tile by tile gmem -> smem -> gmem by TMA.
 *
 * The double-buffered TMA load/store example of "Producer-Consumer Warp
 * Specialization for TMA Operations" generalised to an S-slot ring: one
 * lane loads tile i into slot i % S and one lane stores it back out; the
 * slot is handed back once the store has finished reading shared memory.
 *
 *   src, dst  [rows, cols] of 4-byte elements (fp32 or any 32-bit type; the
 *         copy is bit-exact).  src read only; dst written; they must not overlap.
 *   rows, cols  >= 0 and < 2^31; cols a multiple of 4.  Empty: nothing to do.
 *   tile_rows  1..256; tile_cols 4..256, a multiple of 4 (16-byte rows).
 *   stages  1 <= S <= gbr_max_stages(GBR_OP_COPY, 0, tile_rows, tile_cols),
 *         i.e. S slots of tile_rows * tile_cols * 4 bytes, each rounded up
 *         to a multiple of 128 bytes (TMA's shared-memory alignment), must
 *         fit in one CTA's shared memory (GBR_ERR_SMEM otherwise; at 128x64
 *         fp32 S <= 7).
 */
int staged_copy(const void *src, void *dst, int64_t rows, int64_t cols, int tile_rows,
                int tile_cols, int stages, gbr_stream_t stream);

/*
 * gbr_device_status -- synchronises `stream`, then reports and clears the
 * current device's status block (and the status words of
 * gemm_bias_relu_tf32_noalloc).  It allocates nothing.  Returns GBR_OK,
 * GBR_ERR_TIMEOUT (a pipeline wait in a kernel exceeded its limit; the kernel
 * raised its abort flag, let its own copies in flight finish, released its
 * Tensor Memory and returned, so the context stays usable; the output of
 * that call is undefined), or GBR_ERR_CUDA for a CUDA error seen while
 * synchronising.
 */
int gbr_device_status(gbr_stream_t stream);

/* Message of the last failing call on this thread ("" if none).  The pointer
 * stays valid until the next library call on this thread. */
const char *gbr_last_error(void);

enum { GBR_OP_GEMM = 0, GBR_OP_COPY = 1 };

/* Largest ring depth that fits the current device's per-CTA shared memory:
 * op GBR_OP_GEMM uses `dtype` (tensor-core dtypes: the CTA-pair kernel's
 * limit; one CTA per tile holds 4); GBR_OP_COPY uses tile_rows x tile_cols
 * fp32.  Returns a negative gbr_status on error. */
int gbr_max_stages(int op, int dtype, int tile_rows, int tile_cols);

/* Number of kernels this library has launched in this process. */
long long gbr_launch_count(void);

/* Number of SMs of the current device (negative gbr_status on error). */
int gbr_sm_count(void);

/* Per-wait time limit in nanoseconds for every pipeline wait; 0 restores the
 * default (environment variable GBR_WAIT_TIMEOUT_NS, else 2 s). */
int gbr_set_wait_timeout_ns(uint64_t ns);

/*
 * Staged-copy tuning, process-wide.  store_lag: -1 auto, 0 (release a slot
 * once its own store has read it) or 1 (release the previous slot after the
 * next store is issued; needs stages >= 2).  ctas_per_sm: -1 auto (as many
 * as shared memory allows), else 1..occupancy.  l2_hint: L2 eviction priority
 * of the copied lines: -1 auto (1), 0 none, 1 loads evict_first, 2 stores
 * evict_first, 3 both.
 */
int gbr_copy_tuning(int store_lag, int ctas_per_sm, int l2_hint);

/*
 * Tensor-core GEMM tuning, process-wide (gemm_bias_relu with GBR_BF16 or
 * GBR_F32_TF32, and gemm_bias_relu_grouped).  cta_pair: -1 auto, 1 (one CTA
 * per 128x256 output tile, S <= 4), 2 (a two-CTA cluster per 256x256 tile,
 * cta_group::2 MMA, S <= 6).  Auto picks 2 when there is more than one
 * 128-row tile or S > 4 (grouped: when some expert has more than 128 rows, or
 * S > 4).  group_m: -1 auto, else output-tile rows per raster band.
 * l2_hint: L2 eviction priority of the A/B tile loads: -1 auto (none), 0 none,
 * 1 both evict_last, 2 A evict_first + B evict_last, 3 A evict_last + B
 * evict_first, 4 both evict_normal.  k_per_stage: 1 or 2 slices of 128 bytes
 * of K per ring stage; with 2 a stage is twice as large (so the largest
 * `stages` halves) and each full/empty handshake covers twice the MMAs; -1
 * auto: 2 on the CTA pair whenever `stages` fits (<= 3), else 1.
 */
int gbr_gemm_tuning(int cta_pair, int group_m, int l2_hint, int k_per_stage);

/*
 * Split tail of the tensor-core GEMMs (dense and grouped), for all later calls
 * in the process.  A persistent launch runs T output tiles on U units (CTAs,
 * or CTA pairs); the last T mod U tiles would make a final round that leaves
 * the other units idle.  With the split on, the k-blocks of those tiles are
 * dealt out in equal runs to all U units (at most 4 units share a tile).  Of
 * the units sharing a tile, all but the last to arrive add their fp32 partial
 * sums into a zeroed fp32 copy of the tile (reductions at L2) and count
 * themselves done; the last to arrive waits, with the pipeline time limit,
 * for those counts -- its partners have all started and finish without
 * waiting on anything -- adds the copy to its own accumulator and runs the
 * bias + ReLU epilogue.  Scratch (per call, stream-ordered, zeroed on the
 * stream, from a memory pool the library keeps per device): (T mod U) x tile
 * rows x 256 x 4 bytes plus counters.  Results differ from the unsplit kernel
 * only by the order of fp32 additions; that order follows the arrival of the
 * parts, so a split tile can differ in its last bits from run to run (mode 0
 * makes every launch deterministic).
 *   mode -1: auto (the default): split when the last round shrinks by >= 1/8
 *         of a tile and the predicted saving is >= 1/20 (5%) of the launch's
 *         time; below that the measured gain is within run-to-run noise, so
 *         such launches stay deterministic bit for bit (bf16 8192^3 on a
 *         152-SM GB300 does not split; TF32 4096^3 does).
 *         0: never, 1: whenever some tile can be split.
 * GBR_F32_FFMA follows the same mode with its own combine: the whole tiles run
 * in one launch, then the split tail's runs in a second launch of the same
 * ring; each part of a split tile is stored in its own fp32 slot (sk tiles x
 * 4 x 128 x 128 x 4 bytes), and the last CTA to finish a part adds the parts
 * in part order, so FFMA results are the same bits on every call (they differ
 * from the unsplit kernel's in the order of fp32 additions).  Its auto rule
 * splits from a predicted saving of 1/50 (2%) of the launch (fp32 4096^3 on
 * 152 SMs splits).  GBR_F32_FFMA_CPASYNC and GBR_F32_FFMA_SYNC never split,
 * and GBR_F32_FFMA does not while gbr_trace_buffer is set (its two launches
 * would each write the trace from the start).
 * GBR_ERR_INVALID for other values.  The failure-detection self tests and
 * gemm_bias_relu_tf32_noalloc never split.
 */
int gbr_gemm_split_tail(int mode);

/*
 * Dynamic tile order of the tensor-core GEMMs (dense and grouped), for all
 * later calls in the process.  on = 0 (default): each persistent unit runs
 * tiles unit, unit + units, ... (with the split tail above).  on = 1: the
 * even CTA's producer of each unit takes the next tile from a global atomic
 * counter (a zeroed word from the library's pool) and hands its id to the
 * MMA lane, the epilogue warps and the odd CTA's producer through a 4-slot
 * ring of tile ids in shared memory, guarded by its own full/empty
 * mbarriers; units that finish early take more tiles.  The split tail is off
 * in this mode.  Results equal the static order's bit for bit (every tile
 * adds the same products in the same order).  GBR_ERR_INVALID for other values.
 */
int gbr_gemm_dynamic_schedule(int on);

/*
 * Consumer layout of the strict-fp32 FFMA GEMM (GBR_F32_FFMA, its cp.async
 * variant and the homogeneous baseline's micro-tile), for all later calls in
 * the process.  consumer_warps 8 (-1: the default): 8 consumer warps (2 per
 * warp scheduler) of an 8 x 8 register micro-tile each per 128 x 128 output
 * tile, 384 threads per CTA.  16: 16 consumer warps (4 per scheduler) of
 * 8 x 4, 640 threads per CTA (more warps, but more shared-memory reads per
 * FMA: measured slower).  Results are the same bits either way (each output
 * adds the same products in the same order).  GBR_ERR_INVALID for other
 * values.
 */
int gbr_ffma_tuning(int consumer_warps);

/*
 * Thin tail tiles of gemm_bias_relu_grouped on the CTA pair, for all later
 * calls in the process.  on = 1 (default): an expert's last M-tile with at
 * most 128 rows (t rows) is computed transposed, C^T = W^T X^T, as one
 * M = 256 x N = t rounded up to 16 tcgen05 MMA per K step (the weight panels
 * read as an MN-major A operand, the rows as a K-major B operand), and its
 * epilogue writes the tile column by column; the MMA work of such a tile
 * shrinks from 256 rows to t (rounded up to 16).  The split tail is off in
 * launches with thin tiles.  on = 0: every tile is a 256-row tile.  Results
 * agree to fp32 accumulation order.  GBR_ERR_INVALID for other values.
 */
int gbr_gemm_thin_tail(int on);

/*
 * Programmatic dependent launch of the library's pipeline kernels (the
 * staged copy, the FFMA and tensor-core GEMMs), for
 * all later calls in the process.  on = 1 (default): each is launched so that
 * it may be scheduled before the previous kernel in the stream has finished;
 * its CTAs set up their barriers and Tensor Memory, then wait
 * (griddepcontrol.wait) until that kernel has completed and its memory is
 * visible, before any access to global memory.  Results and stream order are
 * unchanged; back-to-back launches lose the gap between kernels.  on = 0:
 * ordinary launches.  GBR_ERR_INVALID for other values.
 */
int gbr_launch_overlap(int on);

/*
 * gemm_bias_relu_host -- gemm_bias_relu on HOST buffers: copies A, B and bias
 * to the device, computes, and copies C back, overlapping the three.  The
 * device buffers come from the library's stream-ordered pool.  M is cut into
 * up to 8 chunks of whole 256-row tiles: B and bias are copied first, then
 * chunk i of A is copied in while chunk i - 1 is computed and chunk i - 2 is
 * copied out, on three streams of the library joined back into `stream`.
 *   hA [M, K], hB [K, N], hC [M, N] (dtype as for gemm_bias_relu), hbias [N]
 *   fp32: host memory owned by the caller; page-locked memory lets the copies
 *   run asynchronously at full speed.  Stream-ordered: the call returns once
 *   the work is enqueued; hC holds the result, and the inputs may be changed,
 *   only after `stream` has reached that point (e.g. cudaStreamSynchronize).
 *   Row pitches (K and N times the element size) must be multiples of 16
 *   bytes.  Errors as for gemm_bias_relu; after a failed chunk the call still
 *   joins its streams and frees its buffers before returning the error.
 */
int gemm_bias_relu_host(const void *hA, const void *hB, const float *hbias, void *hC, int64_t M,
                        int64_t N, int64_t K, int dtype, int stages, gbr_stream_t stream);

/*
 * gbr_trace_buffer -- event trace of the ring protocol, for all later launches
 * of the staged copy, the FFMA GEMM and the tensor-core GEMMs in the process
 * (buffer NULL: off, the default).  `buffer` is caller-owned device memory,
 * 16-byte aligned, of `bytes` >= 8192 + 32768 bytes.  Layout:
 *   [512 CTAs][4 roles] uint32 event counts (8192 bytes), then per (CTA, role)
 *   a region of cap = (bytes - 8192) / 32768 records of 16 bytes:
 *   { uint64 %globaltimer ns, uint32 item, uint8 role, event, slot, parity }.
 * Roles: 0 producer (empty waits, loads issued), 1 consumer (full waits and
 * slot releases: copy storer, first FFMA consumer warp, MMA lane), 2 first
 * epilogue warp (accumulator full waits, releases), 3 MMA lane on the
 * accumulator ring (empty waits, tile commits).  Events: 0 wait returned
 * (item, slot, parity waited on), 1 issued (recorded before the loads or the
 * commit), 2 released (recorded before the arrive or commit).  A role counts
 * every event and writes the first `cap`; CTAs from 512 on record nothing.
 * Each launch overwrites the counts of the CTAs it runs.  GBR_ERR_INVALID for
 * a misaligned or too small buffer.
 */
int gbr_trace_buffer(void *buffer, uint64_t bytes);

/*
 * Failure-detection self test: launches one CTA that waits, with the given
 * limit, on an mbarrier phase nothing will complete.  The wait gives up, the
 * kernel records a timeout and returns; gbr_device_status() then reports
 * GBR_ERR_TIMEOUT.  No GPU fault or hang is involved.
 */
int gbr_selftest_wait_timeout(uint64_t timeout_ns, gbr_stream_t stream);

/*
 * Failure-detection self tests of the real pipelines.  Each runs the normal
 * call once with one fault planted on the host's instructions: in CTA `cta`,
 * ring item `item` (that CTA's item counter, counted from 0 across its tiles),
 * the producer registers the stage's expected bytes on the full barrier but
 * issues no TMA load, so that stage never fills.  The consumer's bounded wait
 * (limit `limit_ns`, in (0, 10 s]) gives up, records the site, raises the
 * CTA's abort flag; the other roles leave their loops, the producer waits
 * for its own loads in flight, the tensor-core kernel waits for its issued
 * MMAs and frees its Tensor Memory, and the kernel returns.  Other CTAs run
 * normally.  gbr_device_status() then reports GBR_ERR_TIMEOUT with the site
 * (0x21 FFMA consumer, 0x31 MMA issuer or 0x41 epilogue, 0x51 copy storer),
 * the CTA and the item; the output is undefined.  If `cta` or `item` does not
 * exist in that launch nothing is planted and the call completes normally.
 *
 * gbr_selftest_gemm_skip_load: arguments as gemm_bias_relu; dtype GBR_F32_FFMA,
 *   GBR_F32_TF32 or GBR_BF16.  The tensor-core dtypes run one CTA per tile
 *   (`stages` must fit that kernel), unless gbr_gemm_tuning forces the CTA
 *   pair (cta_pair = 2): then `cta` names the pair (unit), both of whose CTAs
 *   leave item `item` unfilled, and the CTA reported is either CTA of it.
 *   After an abort the even CTA of a pair also waits for the loads its peer
 *   issued before either CTA exits.
 * gbr_selftest_copy_skip_load: arguments as staged_copy with 128 x 64 tiles.
 * Returns GBR_OK when launched, GBR_ERR_INVALID for a negative cta or item or
 * a limit out of range, and the errors of the wrapped call.
 */
int gbr_selftest_gemm_skip_load(const void *A, const void *B, const float *bias, void *C,
                                int64_t M, int64_t N, int64_t K, int dtype, int stages, int cta,
                                int item, uint64_t limit_ns, gbr_stream_t stream);
int gbr_selftest_copy_skip_load(const void *src, void *dst, int64_t rows, int64_t cols,
                                int stages, int cta, int item, uint64_t limit_ns,
                                gbr_stream_t stream);

/*
 * gemm_bias_relu_tf32_noalloc -- the GBR_F32_TF32 case of gemm_bias_relu for
 * callers that cannot allocate device memory.  It has no counterpart in the
 * pages; it exists for code that may not call cudaMalloc or cudaMallocAsync:
 * serving loops that must never enter an allocator (allocation can take locks
 * or synchronise the device at unpredictable times), plug-ins whose host
 * framework owns all device allocation, and processes whose device memory is
 * entirely reserved by another allocator, so that an allocation from this
 * library would fail.  It runs the TF32 tensor-core kernel with one CTA per
 * tile and no split (so it needs no per-call scratch) and takes its status
 * words from one file-scope device array of 256 bytes, which the CUDA driver
 * creates on every device that loads this library and keeps until the process
 * exits.  The call allocates nothing, and neither does gbr_device_status().
 *
 *   A [M, K], B [K, N], bias [N], C [M, N]: fp32, as for gemm_bias_relu;
 *   caller-owned device memory.  K and N multiples of 4.  C must not overlap
 *   A, B or bias (GBR_ERR_INVALID).
 *   M, N, K < 2^31 (GBR_ERR_INVALID otherwise, nothing launched).
 *   stages: 1..4 -- this call always runs one CTA per 128x256 tile, whose
 *   ring holds 4 stages on GB300; gbr_max_stages() reports the CTA-pair
 *   kernel's larger limit, which does not apply here (GBR_ERR_SMEM).
 *   stream: as for gemm_bias_relu.
 * The first call on a device looks up the array's device address (once, with
 * that device current) and clears its status words, synchronising the
 * device; make that first call before any stream capture.
 * The array exists once per device, and every call on that device uses it:
 * calls on one device that may overlap on the GPU (different streams, or
 * several host threads) race and give undefined results -- serialise them.
 * Calls on different devices use different arrays.
 * Status: a wait that times out records its site in the array's status
 * words, which keep the FIRST timeout recorded until gbr_device_status(),
 * called with the stream the calls ran on, reads and clears them; timeouts
 * of later calls before that read are not reported separately.
 */
int gemm_bias_relu_tf32_noalloc(const float *A, const float *B, const float *bias, float *C,
                                int64_t M, int64_t N, int64_t K, int stages,
                                gbr_stream_t stream);

/*
 * Failure-detection self test of gemm_bias_relu_tf32_noalloc: the same call
 * with one ring stage left unfilled (CTA `cta`, ring item `item`, limit
 * `limit_ns`), exactly as gbr_selftest_gemm_skip_load does for
 * gemm_bias_relu.  The timeout lands in the no-alloc array's status words,
 * and gbr_device_status() reports it (GBR_ERR_TIMEOUT, site 0x31 MMA issuer
 * or 0x41 epilogue, or the producer's 0x11).  Allocates nothing.
 */
int gbr_selftest_noalloc_skip_load(const float *A, const float *B, const float *bias, float *C,
                                   int64_t M, int64_t N, int64_t K, int stages, int cta, int item,
                                   uint64_t limit_ns, gbr_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GBR_H_ */
