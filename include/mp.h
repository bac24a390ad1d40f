/*
 * mp.h -- dynamic-shape GEMM with epilogue for NVIDIA GB300 (sm_103a).
 *
 *     D = alpha * A * B + beta * C
 *
 * A [M x K] and B [K x N] are bf16, C and D [M x N] are fp32, products are
 * accumulated in fp32.  All matrices are row-major with a leading dimension
 * (elements between the starts of consecutive rows).  The shape (M, N, K) is
 * known only at run time: every call plans its own "polymerization" -- the
 * output is cut into up to four rectangular regions, each covered by one
 * fixed-size micro-kernel with a split-K factor -- and runs the whole plan in
 * one persistent kernel launch.
 *
 * Sources (page titles and sections):
 *   [MP]    "Optimizing Dynamic-Shape Neural Networks on Accelerators via
 *           On-the-Fly Micro-Kernel Polymerization" (MikPoly summary):
 *           section 3 (multi-level accelerator abstraction H, micro-kernel
 *           performance model g_predict, polymerization patterns, cost model
 *           Cost(S,H) = sum_i f_wave * f_pipe, pruned heuristic search),
 *           section 4 (GPU: Patterns I and II; offsets and loop counts passed
 *           as run-time scalars), section 6 (case study (4096,1024,4096)).
 *   [BOLT]  BOLT summary, "Persistent kernel (GEMM/Conv) fusion": the
 *           epilogue form D = alpha*A*W + beta*C.
 *   [DISC]  BladeDISC v0.2.0 release notes, "GEMM merge": shared-operand
 *           merge A x concat(B, C) and same-shape batched GEMM.
 *
 * Conventions for every entry point:
 *   - The caller owns A, B, C, D and the stream; the library owns the handle
 *     and everything it allocates at mp_init (split-K workspace, tile
 *     counters, an operand staging area, the device status word).  mp_gemm and
 *     mp_gemm_batched never allocate.
 *   - Errors are returned as mp_status codes; nothing aborts, throws or falls
 *     back to the CPU.
 *   - A handle serves one host thread and one stream at a time: two calls that
 *     overlap on the device share the split-K workspace and would race.
 */
#ifndef MP_H_
#define MP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mp_handle_s* mp_handle;
/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef void* mp_stream;

typedef enum {
    MP_OK = 0,
    MP_ERR_INVALID_ARG = -1,     /* bad size, pointer, leading dimension or overlap */
    MP_ERR_UNSUPPORTED = -2,     /* valid request this build cannot run (e.g. no sm_103 device) */
    MP_ERR_CUDA = -3,            /* a CUDA runtime/driver call failed */
    MP_ERR_PLAN = -4,            /* the planner produced no valid plan */
    MP_ERR_DEVICE_TIMEOUT = -5,  /* a device-side wait gave up (reported by mp_check) */
    MP_ERR_NO_MEMORY = -6        /* allocation at mp_init failed */
} mp_status;

#define MP_MAX_REGIONS 4
#define MP_MAX_KERNELS 16

/*
 * Hardware description H [MP section 3, "multi-level accelerator
 * abstraction"]: the number of processing engines, each PE's local memory,
 * and the memory shared by all PEs; plus the rates the cost model uses.
 */
typedef struct {
    int32_t num_pe;            /* processing engines (SMs)                      */
    int32_t warps_per_wave;    /* warps resident at once over all PEs; a task
                                  of w warps gets warps_per_wave / w slots     */
    int64_t local_mem_bytes;   /* per-PE local memory (shared memory)           */
    int64_t shared_mem_bytes;  /* memory shared by the PEs (L2)                 */
    double hbm_gbs;            /* global-memory bandwidth, GB/s                 */
    double l2_gbs;             /* shared-memory (L2) to PE bandwidth, GB/s      */
    double mma_tflops;         /* dense bf16 tensor throughput, TFLOP/s         */
} mp_hw;

/*
 * One micro-kernel: a fixed output tile (um x un) with a fixed K step uk
 * [MP section 3, "micro-kernel generation"], and its performance model
 * g_predict(t) = fixed_us + per_step_us * t for a pipeline task of t
 * micro-kernel instances [MP section 3, "micro-kernel performance model"].
 * That section's task runs in three overlapped stages (load, compute, write
 * back); on a PE that runs tasks back to back, a task's write-back overlaps
 * the next task's load and compute, so only the last wave's write-back adds
 * to the time: tail_us, charged once per plan (with the launch and pipeline
 * fill), keeps it out of g_predict.
 * swap = 1 marks the transposed form (D^T = B^T A^T) used for short M.
 * pair = 1 marks a tile computed by a cluster of two CTAs on two SMs with the
 * pair MMA (each CTA holds half of the tile's rows of A and D and half of its
 * columns of B); such a kernel never splits K, and a plan uses either pair
 * kernels only or none.
 */
typedef struct {
    int32_t um, un, uk;
    int32_t warps;             /* warps per task, for wave counting            */
    int32_t swap;
    int32_t pair;
    double fixed_us;           /* per-task time that does not scale with t     */
    double per_step_us;        /* time per micro-kernel instance (one uk step) */
    double tail_us;            /* time added once per plan after the last wave:
                                  its write-back (stage 3), not hidden behind a
                                  next task, plus launch and pipeline fill     */
} mp_kernel_desc;

/* One region R_i of a plan and its cost terms [MP section 3, cost model]. */
typedef struct {
    int32_t kernel;            /* index into the handle's micro-kernel set     */
    int32_t um, un, uk, swap;
    int32_t pair;              /* tile computed by a CTA pair (see mp_kernel_desc) */
    int64_t m0, n0;            /* origin of the region in D                    */
    int64_t m_ext, n_ext;      /* extent of the region                         */
    int32_t splits;            /* split-K factor: K~_i = ceil(K / splits)      */
    int32_t f_num;             /* micro-kernel instances per task              */
    int64_t f_parallel;        /* pipeline tasks = tiles * splits              */
    int64_t f_wave;            /* ceil(f_parallel / slots)                     */
    double f_pipe_us;          /* g_predict(f_num) (+ split-K reduction)       */
} mp_region_info;

typedef struct {
    int32_t pattern;           /* 1: one region; 2: two regions along M or N;
                                  4: body / right / bottom / corner            */
    int32_t num_regions;
    mp_region_info region[MP_MAX_REGIONS];
    double cost_us;            /* Cost(S, H) of the chosen strategy            */
    int64_t total_tasks;
    int32_t evaluated;         /* strategies whose cost was computed           */
    int32_t pruned;            /* strategies skipped by the running best       */
    int64_t workspace_bytes;   /* split-K partials the plan needs              */
} mp_plan_info;

/*
 * Create a handle on CUDA device `device` (must be an sm_103 GB300-class
 * GPU).  Reads the device's SM count and memory sizes into H, allocates the
 * library-owned device memory, and sets the micro-kernels' performance model
 * (g_predict, its tail, the split-K reduction terms):
 *   calib_path NULL: the table measured on GB300 that ships with the library
 *       (<package>/calib/gb300.txt beside <package>/_lib/libmp.so), when it
 *       is readable; otherwise the analytic model;
 *   calib_path "": the analytic model (hand-fitted GB300 constants);
 *   otherwise: the table at calib_path when readable, else the analytic model.
 * A table is plain text, one micro-kernel per line:
 * "um un uk swap fixed_us per_step_us [tail_us]", plus lines
 * "split on_chip sync_us bytes_factor [S]" for the split-K reduction (see
 * mp_set_split_model; without S, on_chip 1 sets every cluster size); '#'
 * starts a comment, and lines that name no kernel of the set are ignored.
 * micro_polymerization_gb300/calibrate.py writes such tables.  The rates in
 * H default to GB300 figures and can be overridden with the environment
 * variables MP_HBM_GBS, MP_L2_GBS and MP_MMA_TFLOPS.  The set holds the
 * CTA-pair micro-kernels only when the device can keep two-CTA clusters of
 * the kernel resident and MP_PAIR is not "0"; they come last, so the other
 * kernels' indices do not depend on them.
 * Errors: MP_ERR_INVALID_ARG (out NULL or bad device), MP_ERR_UNSUPPORTED
 * (not sm_103), MP_ERR_NO_MEMORY, MP_ERR_CUDA.
 */
mp_status mp_init(mp_handle* out, int device, const char* calib_path);

/*
 * Create a planning-only handle from an explicit H and micro-kernel set (no
 * GPU is touched; mp_gemm on it returns MP_ERR_UNSUPPORTED).  Used to check
 * the planner against the pages' worked example.  kernels[0..num_kernels) is
 * copied; num_kernels <= MP_MAX_KERNELS.
 */
mp_status mp_init_host(mp_handle* out, const mp_hw* hw,
                       const mp_kernel_desc* kernels, int32_t num_kernels);

/* Release the handle and all library-owned memory.  NULL is accepted. */
mp_status mp_destroy(mp_handle h);

/*
 * Plan (M, N, K) without running it [MP section 3, "polymerization" and
 * "heuristic search"; section 4, Patterns I and II]: evaluate Cost(S,H) over
 * the strategies the search visits and return the cheapest in *out
 * (optional).  Host only; never touches the device.
 * Errors: MP_ERR_INVALID_ARG (negative size), MP_ERR_PLAN.
 */
mp_status mp_plan(mp_handle h, int64_t M, int64_t N, int64_t K, mp_plan_info* out);

/* Same, for `batch` independent problems of one shape run in one launch. */
mp_status mp_plan_batched(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                          mp_plan_info* out);

/*
 * Plan `count` shapes in one call: mnk holds (M, N, K) triples, host memory,
 * read only; `out` (nullable) receives count plans, as mp_plan would.  Meant
 * for planning a set of shape buckets ahead of time, and for timing the
 * polymerizer itself without a language binding in the loop (MikPoly summary,
 * section 5, cost model overhead: microseconds per shape).  Shapes already in
 * the handle's plan cache are looked up, not searched; a handle made with
 * MP_PLAN_CACHE=0 in the environment keeps no cache, so every call searches.
 * Returns the first error (MP_ERR_INVALID_ARG for a negative or oversized
 * dimension); plans before it are filled in.
 */
mp_status mp_plan_many(mp_handle h, int32_t count, const int64_t* mnk, mp_plan_info* out);

/*
 * Cost of a given strategy under the handle's model [MP section 3, cost
 * model]: the caller fills num_regions and, per region, kernel, m0, n0,
 * m_ext, n_ext and splits; the call fills every other field and cost_us.
 * Used to evaluate the pages' worked example and for exhaustive search.
 * Errors: MP_ERR_INVALID_ARG (unknown kernel), MP_ERR_PLAN (the regions do
 * not tile the output exactly once).
 */
mp_status mp_evaluate_plan(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                           mp_plan_info* inout);

/*
 * The candidate strategies of one shape, for exhaustive search and for the
 * cost-model ablations of [MP section 5, "cost model effectiveness"] (an
 * exhaustive-search variant picks the fastest candidate by running them):
 *   - Pattern I: every micro-kernel with every split-K candidate;
 *   - Pattern II: both cut directions, every micro-kernel for the first
 *     region, cuts on its tile boundaries (every one up to 64 of them, else
 *     64 spread evenly plus the wave-filling ones), every micro-kernel of the
 *     same CTA grouping for the second region, unsplit or split to fill a
 *     wave.
 * Each is filled as by mp_evaluate_plan under the handle's model.  The
 * candidates are sorted by cost_us; the first `capacity` go to `out` (may be
 * NULL with capacity 0) and `*count` receives how many exist.
 * Errors: MP_ERR_INVALID_ARG (bad sizes, count NULL, capacity < 0).
 */
mp_status mp_enumerate_plans(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K, mp_plan_info* out,
                             int32_t capacity, int32_t* count);

/*
 * mp_gemm with an explicit plan instead of the polymerizer's choice: one
 * from mp_plan or mp_enumerate_plans, or regions filled by hand (kernel, m0,
 * n0, m_ext, n_ext, splits; the rest is recomputed as by mp_evaluate_plan).
 * Used for exhaustive search and ablations.  Same arguments, layout rules,
 * ownership and asynchrony as mp_gemm.
 * Errors: as mp_gemm, and MP_ERR_PLAN when the regions do not tile the
 * output exactly once or mix CTA-pair and one-CTA micro-kernels.
 */
mp_status mp_gemm_with_plan(mp_handle h, const mp_plan_info* plan, int64_t M, int64_t N, int64_t K, const void* A,
                            int64_t lda, const void* B, int64_t ldb, const float* C, int64_t ldc, float* D,
                            int64_t ldd, float alpha, float beta, mp_stream stream);

/*
 * Cost model the polymerizer searches with [MP section 5, "cost model
 * effectiveness"]:
 *   MP_PLAN_MIKPOLY (default): Cost(S,H) = sum over regions of f_wave * f_pipe,
 *     floored at the HBM time of the algorithmic bytes;
 *   MP_PLAN_WAVE: the fewest waves (sum of f_wave), which favours large
 *     micro-kernels;
 *   MP_PLAN_PIPE: the fastest pipeline tasks (sum of f_pipe), which favours
 *     small micro-kernels.
 * The plan cache is cleared.  Errors: MP_ERR_INVALID_ARG (unknown mode).
 */
#define MP_PLAN_MIKPOLY 0
#define MP_PLAN_WAVE 1
#define MP_PLAN_PIPE 2
mp_status mp_set_plan_mode(mp_handle h, int32_t mode);

/*
 * D = alpha * A * B + beta * C, asynchronously on `stream`.  Plans the shape
 * (as mp_plan) and issues one persistent kernel launch [MP section 4:
 * offsets and loop counts are run-time scalars of fixed-size micro-kernels;
 * BOLT: the alpha/beta epilogue is fused].
 *   A: device pointer, M x K bf16, row-major, lda >= max(1, K)
 *   B: device pointer, K x N bf16, row-major, ldb >= max(1, N)
 *   C: device pointer, M x N fp32, row-major, ldc >= max(1, N); not read and
 *      may be NULL when beta == 0
 *   D: device pointer, M x N fp32, row-major, ldd >= max(1, N)
 * Any element-aligned pointer and leading dimension is accepted; operands
 * whose rows are not 16-byte aligned are first repacked into the handle's
 * staging area by the library's own kernel.  M == 0 or N == 0 is a no-op;
 * K == 0 gives D = beta * C.  D may equal C only with ldc == ldd; any other
 * overlap of D with A, B or C is MP_ERR_INVALID_ARG.  Repeated calls with the
 * same plan give bitwise-identical D (split-K partials are reduced in a fixed
 * order).  A call may be recorded by CUDA stream capture into a graph: each
 * replay runs the plan and the operand addresses of the capture (no planning
 * on replay), on the data then in those buffers.  The handle's workspace,
 * tile counters and staging area serve replays as they serve calls, so
 * replays and calls of one handle must not overlap on the GPU.
 * Errors: MP_ERR_INVALID_ARG, MP_ERR_UNSUPPORTED (host-only handle or size
 * beyond the staging area), MP_ERR_PLAN, MP_ERR_CUDA (launch failure).
 */
mp_status mp_gemm(mp_handle h, int64_t M, int64_t N, int64_t K,
                  const void* A, int64_t lda,
                  const void* B, int64_t ldb,
                  const float* C, int64_t ldc,
                  float* D, int64_t ldd,
                  float alpha, float beta, mp_stream stream);

/*
 * mp_gemm with an epilogue variant: an activation applied to
 * alpha*A*B + beta*C, and the type of D.  These are the epilogue variants of
 * templated GEMM libraries (BOLT summary, "Persistent kernel (GEMM/Conv)
 * fusion": the alpha/beta epilogue form; activation and output type are the
 * same epilogue's further stages).  The epilogue word is:
 *   bits 0-7: MP_ACT_NONE, MP_ACT_RELU (max(x, 0)) or MP_ACT_GELU
 *             (x * Phi(x) = x/2 * (1 + erf(x / sqrt 2)), computed in fp32);
 *   MP_EPI_OUT_BF16: D is bf16 (row-major, ldd in elements, 2-byte aligned;
 *             each value rounded to nearest even), else fp32.
 * C stays fp32.  C and D must not overlap when D is bf16.  Otherwise the same
 * arguments, rules and asynchrony as mp_gemm; mp_gemm is mp_gemm_ex with 0.
 * Errors: as mp_gemm, and MP_ERR_INVALID_ARG for an unknown epilogue word.
 */
#define MP_ACT_NONE 0
#define MP_ACT_RELU 1
#define MP_ACT_GELU 2
#define MP_EPI_OUT_BF16 0x100
mp_status mp_gemm_ex(mp_handle h, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda, const void* B,
                     int64_t ldb, const float* C, int64_t ldc, void* D, int64_t ldd, float alpha, float beta,
                     int32_t epilogue, mp_stream stream);

/*
 * `batch` same-shape problems in one launch [DISC, "GEMM merge" 2]: problem
 * b uses A + b*strideA, B + b*strideB, C + b*strideC, D + b*strideD (strides
 * in elements, >= 0).  Per-problem rules are those of mp_gemm; the D blocks
 * of different problems must not overlap.  batch == 0 is a no-op.
 */
mp_status mp_gemm_batched(mp_handle h, int64_t batch, int64_t M, int64_t N, int64_t K,
                          const void* A, int64_t lda, int64_t strideA,
                          const void* B, int64_t ldb, int64_t strideB,
                          const float* C, int64_t ldc, int64_t strideC,
                          float* D, int64_t ldd, int64_t strideD,
                          float alpha, float beta, mp_stream stream);

/*
 * D = alpha * A * B + beta * C without a handle and without allocating any
 * device memory.  The pages have no counterpart to this call; it exists for
 * callers that cannot call cudaMalloc: plugin interfaces of inference runtimes
 * that own all device memory, processes that reserve device memory up front,
 * and latency-critical loops where an allocation may synchronize the device.
 *
 * Same operands, layout rules and argument errors as mp_gemm (one problem, on
 * the current device).  A kernel that gives up on a bounded wait records it
 * in a status word of the fixed array; mp_check_noalloc reads it back (there
 * is no handle for mp_check).  Its scratch is a fixed array inside the
 * library, about 48 MiB per GPU, held until the process exits:
 * 16 MiB of split-K partials (the planner never asks for more), 4096 tile
 * counters, a status word, and a 32 MiB staging area for operands whose rows
 * are not 16-byte aligned.  A request that would need more than that -- an
 * unaligned operand above 32 MiB after padding its rows to 8 elements -- is
 * rejected with MP_ERR_UNSUPPORTED before anything runs.
 *
 * The array's device memory is committed when the library's device code
 * loads on a GPU: under CUDA's default lazy module loading that is the first
 * call on the device (with CUDA_MODULE_LOADING=EAGER, when the library
 * loads).  A caller that reserves nearly all device memory for its own pool
 * should make one call before reserving it.  The first call on a device also
 * finds the array's address and clears it with a synchronous cudaMemset;
 * make that first call before any stream capture.
 * Every call shares the array and starts from what the previous call left:
 * the counters a call needs are cleared on `stream` before its kernel.  Calls
 * whose kernels overlap on the GPU (other streams, other host threads) race
 * on the array; issue them on one stream.  No cudaMalloc, cudaFree or other
 * allocating routine is called.
 */
mp_status mp_gemm_noalloc(int64_t M, int64_t N, int64_t K,
                          const void* A, int64_t lda,
                          const void* B, int64_t ldb,
                          const float* C, int64_t ldc,
                          float* D, int64_t ldd,
                          float alpha, float beta, mp_stream stream);

/*
 * mp_check for mp_gemm_noalloc on the current device: synchronize `stream`
 * and read the fixed array's status word.  MP_OK (also when no call has run
 * on this device), MP_ERR_DEVICE_TIMEOUT if one of its kernels gave up on a
 * bounded wait since the last check (the word and the array's tile counters
 * are then cleared), or MP_ERR_CUDA.  Allocates nothing.  No counterpart on
 * the pages, like mp_gemm_noalloc itself.
 */
mp_status mp_check_noalloc(mp_stream stream);

/*
 * Test hook: mp_inject_wait_timeout for the next mp_gemm_noalloc launch on
 * the current device (the same `enable` modes and limit).
 */
mp_status mp_noalloc_inject_wait_timeout(int32_t enable, int64_t limit_ns);

/*
 * Synchronize `stream` and read the device status word: MP_OK, or
 * MP_ERR_DEVICE_TIMEOUT if a kernel gave up on a bounded wait since the last
 * check (the word is then cleared), or MP_ERR_CUDA.
 */
mp_status mp_check(mp_handle h, mp_stream stream);

/*
 * Test and ablation hook: pin every later plan to micro-kernel `kernel`
 * (-1: free choice) and split-K factor `splits` (0: free choice), Pattern I.
 */
mp_status mp_force_plan(mp_handle h, int32_t kernel, int32_t splits);

/*
 * Test hook for failure detection: with enable = 1 the next launch on this
 * handle (of any kernel: GEMM, fused pair, convolution, grouped GEMM)
 * withholds one shared-memory stage of its first work unit, so the
 * consumer's bounded wait runs out after limit_ns nanoseconds (0 keeps the
 * handle's limit, 1 s by default; a positive value also becomes the limit of
 * later launches).  With enable = 2 the GEMM kernel instead makes the
 * split-K sums it stages in its idle operand ring wait for 16 bytes more
 * than it copies (the other kernels treat 2 as 1).  The kernel then stops
 * cleanly and mp_check reports MP_ERR_DEVICE_TIMEOUT.  Nothing faults, traps
 * or hangs.  0 clears a pending injection; other values: MP_ERR_INVALID_ARG.
 */
mp_status mp_inject_wait_timeout(mp_handle h, int32_t enable, int64_t limit_ns);

/* Copy the handle's H and micro-kernel set (either pointer may be NULL). */
mp_status mp_get_hw(mp_handle h, mp_hw* hw, mp_kernel_desc* kernels, int32_t* num_kernels);

/*
 * Replace micro-kernel k's performance model (g_predict and its tail) with
 * measured values; used by calibration.  The plan cache is cleared.
 * Errors: MP_ERR_INVALID_ARG (no such kernel, negative fixed or tail time,
 * per-step time not positive).
 */
mp_status mp_set_kernel_model(mp_handle h, int32_t k, double fixed_us, double per_step_us, double tail_us);

/*
 * Replace the cost model of the split-K reduction (MikPoly summary, section 3:
 * a split tile's tasks each run g_predict(f_num) K steps and then combine
 * their partial sums).  A task of a tile split S > 1 ways costs
 *     g_predict(f_num) + sync_us + bytes_factor * 4 um un / (l2_gbs / num_pe)
 * microseconds (the last term: the tile's fp32 partial at one PE's share of
 * L2 bandwidth).  on_chip = 0 (S = 0) sets the reduction through L2;
 * on_chip = 1 the one through distributed shared memory in clusters of S
 * CTAs, for S in [2, 8], or for every such S when S = 0.  The plan cache is
 * cleared.  Errors: MP_ERR_INVALID_ARG (h NULL, on_chip or S out of range, a
 * negative or NaN term).
 */
mp_status mp_set_split_model(mp_handle h, int32_t on_chip, int32_t S, double sync_us, double bytes_factor);

/*
 * Read one split-K cost entry: (on_chip 0, S 0) or (on_chip 1, S in [2, 8]).
 * Either output pointer may be NULL.  Errors: MP_ERR_INVALID_ARG.
 */
mp_status mp_get_split_model(mp_handle h, int32_t on_chip, int32_t S, double* sync_us, double* bytes_factor);

/*
 * Apply a calibration table (the text format mp_init reads) to a handle:
 * the lines that name a micro-kernel of its set and the "split" lines
 * replace those terms; the rest of the model is kept.  The plan cache is
 * cleared.  Errors: MP_ERR_INVALID_ARG (h or path NULL, file unreadable).
 */
mp_status mp_load_calibration(mp_handle h, const char* path);

/* Static text for a status code. */
const char* mp_status_string(mp_status s);

/*
 * Back-to-back GEMMs in one launch (BOLT summary, "Persistent kernel
 * (GEMM/Conv) fusion"):
 *     D0 = act0(alpha0 * A0 W0 + beta0 * C0)
 *     D1 = alpha1 * D0 W1 + beta1 * C1
 * A0 [M x K0], W0 [K0 x N0] and W1 [N0 x N1] are bf16, row-major; C0
 * [M x N0], C1 and D1 [M x N1] are fp32, row-major; leading dimensions in
 * elements.  D0 is never written to memory: each 128-row block of it stays
 * in the producing CTA's shared memory, rounded to bf16 (the type of the
 * second GEMM's operand), and feeds that CTA's second GEMM (the summary's
 * threadblock residence).  That needs N0 <= 256.  Where two launches are
 * predicted clearly faster, and always for N0 > 256, D0 goes through a bf16
 * buffer instead (mp_set_b2b_mode): the end of the handle's staging area
 * (allocated at mp_init, 1 GiB by default), so mp_gemm_b2b never allocates;
 * that form needs M * round8(N0) * 2 bytes <= half of the area.  act0 is MP_ACT_NONE,
 * MP_ACT_RELU or MP_ACT_GELU (the epilogue variants' activations).  C0 is not
 * read when beta0 == 0, nor C1 when beta1 == 0; C1 may be D1 (same pointer
 * and ld).  Asynchronous on `stream`, like mp_gemm.
 * M == 0 or N1 == 0 is a no-op; K0 == 0 gives D0 = act0(beta0 * C0); N0 == 0
 * gives D1 = beta1 * C1.
 * Errors: MP_ERR_INVALID_ARG (negative size, NULL operand that is read, ld
 * too small, misaligned element, D1 overlapping an input other than an
 * identical C1, unknown act0); MP_ERR_UNSUPPORTED (N0 > 256 with the fused
 * form forced, host-only handle, or an A0, W0 or W1 whose base or row pitch
 * is not 16-byte aligned and that does not fit the staging area, where such
 * operands are copied with padded rows, as in mp_gemm, or a two-launch D0
 * larger than half of the staging area); MP_ERR_CUDA (launch failure).
 */
mp_status mp_gemm_b2b(mp_handle h, int64_t M, int64_t N0, int64_t N1, int64_t K0, const void* A0, int64_t lda0,
                      const void* W0, int64_t ldw0, const float* C0, int64_t ldc0, const void* W1, int64_t ldw1,
                      const float* C1, int64_t ldc1, float* D1, int64_t ldd1, float alpha0, float beta0,
                      float alpha1, float beta1, int32_t act0, mp_stream stream);

/*
 * How mp_gemm_b2b splits a problem (host only; any handle).  A work unit is
 * 128 rows of M and `cpg` consecutive chunks of `bn1` columns of D1; the
 * units of one row block each recompute that block of D0.  `cpg` minimises
 * the cost model: waves of units x (first GEMM + cpg chunks).
 */
typedef struct {
    int32_t n0p;          /* N0 rounded up to 64 */
    int32_t bn1;          /* D1 columns per chunk */
    int32_t chunks;       /* ceil(N1 / bn1) */
    int32_t mblocks;      /* ceil(M / 128) */
    int32_t cpg;          /* chunks per work unit */
    int32_t units;        /* mblocks * ceil(chunks / cpg) */
    int32_t grid;         /* CTAs launched: min(units, #SMs) */
    int32_t num_stages;   /* shared-memory ring depth */
    int32_t stage_bytes;  /* bytes per ring stage */
    int32_t smem_bytes;   /* dynamic shared memory per CTA */
    double cost_us;       /* model estimate of the fused kernel */
    int32_t mode;         /* what mp_gemm_b2b runs: MP_B2B_FUSED or MP_B2B_TWO_LAUNCH */
    double two_launch_cost_us;  /* model estimate of the two-launch form */
} mp_b2b_plan;
mp_status mp_plan_b2b(mp_handle h, int64_t M, int64_t N0, int64_t N1, int64_t K0, mp_b2b_plan* out);

/*
 * Which form mp_gemm_b2b runs.  MP_B2B_FUSED: the fused kernel (D0 stays on
 * chip; N0 <= 256).  MP_B2B_TWO_LAUNCH: mp_gemm_ex writes D0 =
 * act0(alpha0*A0*W0 + beta0*C0) in bf16 (the same rounding as on chip) to
 * the end of the handle's staging area, then mp_gemm runs the second GEMM.
 * MP_B2B_AUTO (the default) keeps the fused kernel unless the two forms'
 * cost models predict the two launches faster, by more than 5% when the
 * handle plans with a measured table (10% with the analytic model), and runs
 * N0 > 256 as two launches (mp_plan_b2b reports the choice).
 * Errors: MP_ERR_INVALID_ARG (unknown mode).
 */
#define MP_B2B_AUTO 0
#define MP_B2B_FUSED 1
#define MP_B2B_TWO_LAUNCH 2
mp_status mp_set_b2b_mode(mp_handle h, int32_t mode);

/*
 * 2-D convolution, stride 1, zero padding, NHWC, as an implicit GEMM (the
 * MikPoly summary, section 5, runs convolutions as GEMMs; here the im2col
 * matrix [N*P*Q, R*S*C] is never built, its tiles are loaded from X):
 *     D[n,p,q,k] = alpha * sum_{r,s,c} X[n, p+r-pad_h, q+s-pad_w, c] * F[r,s,c,k]
 *                + beta * Cin[n,p,q,k]
 * with P = H + 2*pad_h - R + 1, Q = W + 2*pad_w - S + 1.  X [N][H][W][C] and
 * F [R][S][C][K] are bf16, dense; Cin and D [N][P][Q][K] are fp32 with
 * `ldc` / `ldd` elements from one output pixel to the next (>= K).  Cin is
 * not read when beta == 0 and may be D (same pointer and ld).  Asynchronous
 * on `stream`, like mp_gemm.  An empty output (N, K, P or Q <= 0) is a no-op;
 * C == 0 gives D = beta * Cin.
 * Errors: MP_ERR_INVALID_ARG (negative size or padding, R or S < 1, NULL
 * operand that is read, ld < K, misaligned element, D overlapping X, F or a
 * Cin other than D itself); MP_ERR_UNSUPPORTED (host-only handle, or an X or
 * F whose pixel / row pitch is not 16-byte aligned and that does not fit the
 * staging area, where such operands are copied with padded rows);
 * MP_ERR_CUDA (launch failure).
 */
mp_status mp_conv2d(mp_handle h, int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R, int64_t S,
                    int64_t pad_h, int64_t pad_w, const void* X, const void* F, const float* Cin, int64_t ldc,
                    float* D, int64_t ldd, float alpha, float beta, mp_stream stream);

/*
 * How mp_conv2d tiles a problem (host only; any handle).  An output tile is
 * wb x hb x nb pixels (along Q, P and images; at most 128: powers of two with
 * product 128, or sides that divide a small output exactly) by bn output
 * channels, its K loop (R*S*ceil(C/64) steps) cut into `splits`
 * slices; tile shape, bn and splits minimise the cost model (waves of units
 * x the slice's K loop, against the tile's stores, plus the reduction).
 */
typedef struct {
    int32_t wb, hb, nb;       /* output pixels per tile along Q, P and images (product <= 128) */
    int32_t bn;               /* output channels per tile */
    int32_t tiles_q, tiles_p, tiles_n, tiles_k;
    int32_t ksteps;           /* R * S * ceil(C / 64) */
    int32_t tiles;            /* tiles_q * tiles_p * tiles_n * tiles_k */
    int32_t splits;           /* K slices per tile (> 1: partials in the
                                 handle's workspace, summed in split order by
                                 a second kernel) */
    int32_t units;            /* tiles * splits */
    int32_t grid;             /* CTAs launched: min(units, #SMs) */
    int32_t num_stages;
    int32_t stage_bytes;
    int32_t smem_bytes;
    double useful;            /* output pixels / pixels the tiles cover */
    double cost_us;           /* model estimate */
} mp_conv_plan;
mp_status mp_plan_conv(mp_handle h, int64_t N, int64_t H, int64_t W, int64_t C, int64_t K, int64_t R, int64_t S,
                       int64_t pad_h, int64_t pad_w, mp_conv_plan* out);

/*
 * Grouped GEMM: `count` independent problems of any shapes in as few launches
 * as possible (48 problems per launch), D_i = alpha_i * A_i B_i + beta_i * C_i.
 * The BladeDISC v0.2.0 notes merge same-shape GEMMs into a batched GEMM to
 * fill the machine and launch fewer kernels; a group drops the same-shape
 * condition.  Each problem follows mp_gemm's rules (types, layouts, leading
 * dimensions, C not read when beta_i == 0, C_i == D_i allowed); no D_i may
 * overlap another problem's A, B, C or D.  `problems` is a host array, read
 * before the call returns; the work is asynchronous on `stream`.  Problems
 * with M, N == 0 are skipped; K == 0 gives D = beta * C.  count <= 4096.
 * Errors: MP_ERR_INVALID_ARG (a problem breaking mp_gemm's rules, overlapping
 * outputs, count < 0 or > 4096, NULL problems with count > 0);
 * MP_ERR_UNSUPPORTED (host-only handle, or unaligned operands beyond the
 * staging area); MP_ERR_CUDA.
 */
typedef struct {
    int64_t M, N, K;
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    const float* C;
    int64_t ldc;
    float* D;
    int64_t ldd;
    float alpha, beta;
} mp_gemm_problem;
mp_status mp_gemm_grouped(mp_handle h, int32_t count, const mp_gemm_problem* problems, mp_stream stream);

/*
 * How mp_gemm_grouped runs a group (host only; any handle): one tile width
 * bn for all problems, chosen by the cost model (the group's tiles spread
 * over the SMs, against the longest tile).
 */
typedef struct {
    int32_t bn;           /* output columns per tile: 64, 128 or 256 */
    int32_t units;        /* tiles of all non-empty problems */
    int32_t launches;     /* ceil(non-empty problems / 48) */
    int32_t num_stages;
    int32_t stage_bytes;
    int32_t smem_bytes;
    double cost_us;       /* model estimate */
} mp_grouped_plan;
mp_status mp_plan_grouped(mp_handle h, int32_t count, const mp_gemm_problem* problems, mp_grouped_plan* out);

#ifdef __cplusplus
}
#endif

#endif /* MP_H_ */
