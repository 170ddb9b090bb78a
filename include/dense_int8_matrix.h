/*
 * dense_int8_matrix: dense matrix multiply C = A x B on one NVIDIA GB300
 * (sm_103a).  C ABI of libgemm_gb300.so.
 *
 * The operation is the one the TPU's 256x256 INT8 multiply-accumulate array
 * evaluates ("文章导读: Motivation for and Evaluation of the First Tensor
 * Processing Unit", sections "TPU介绍" and "TPU使用的技术"):
 *
 *     C[i][j] = sum_{kk < k} A[i][kk] * B[kk][j]
 *
 * in two forms: int8 x int8 -> int32 (exact) and bf16 x bf16 -> fp32
 * (fp32 accumulation).  The tile configuration of each problem is chosen on
 * the host by the five-step method of patent CN114238853A
 * ("一種矩陣乘分片配置選擇方法及系統", claims 1-7), re-derived for sm_103a.
 *
 * Layout (all operands dense, leading dimensions implied):
 *   A   m x k row-major              A[i][kk] = A[i*k + kk]
 *   Bt  n x k row-major: B stored K-major (transposed), B[kk][j] = Bt[j*k + kk]
 *   C   m x n row-major              C[i][j]  = C[i*n + j]
 *
 * Ownership: the caller owns every buffer.  The library never frees caller
 * memory.  Device scratch (the f16 copies of int8 operands) is taken from a
 * private stream-ordered memory pool inside gemm_*_run and returned to it on
 * the same stream.  A plan is plain data: copy it freely, nothing to free.
 *
 * Asynchrony: gemm_*_run only enqueues work on `stream` (a cudaStream_t;
 * NULL = the legacy default stream) and returns.  Launch errors are returned
 * as GEMM_ERR_CUDA.  Errors found while kernels run (a wait that ran past its
 * time limit) are reported by gemm_device_error().  The library's kernels
 * are launched with programmatic stream serialization, so a call's kernels
 * may start (set up, prefetch into L2) before the work in front of them on
 * the stream has finished; none of them reads or writes A, Bt, C or scratch
 * before that work has completed, so stream order holds as usual.  C must
 * not overlap A or Bt of the same call.
 *
 * Thread safety: every entry point may be called from several host threads.
 */
#ifndef DENSE_INT8_MATRIX_H
#define DENSE_INT8_MATRIX_H

#include <stdint.h>

/* Only the entry points below are exported; the library is built with
 * hidden default visibility. */
#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,        /* null pointer, size out of range, bad plan */
    GEMM_ERR_MISALIGNED = 2,         /* A or Bt not 16-byte aligned, C not 4-byte aligned */
    GEMM_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not sm_103 */
    GEMM_ERR_CUDA = 4,               /* a CUDA runtime call failed */
    GEMM_ERR_OVERFLOW_RISK = 5,      /* int8: k > 131071, so |C| could exceed int32 */
    GEMM_ERR_TIMEOUT = 6             /* a kernel wait ran past its limit (see gemm_device_error) */
} gemm_status;

enum { GEMM_PATH_TENSOR = 0, GEMM_PATH_SKINNY = 1 };
enum { GEMM_DTYPE_I8 = 0, GEMM_DTYPE_BF16 = 1 };

/* Kernel kinds counted by the trace (gemm_trace_*). */
enum {
    GEMM_KERNEL_STAGE = 0,  /* operand staging: int8 -> f16 widening / re-pitching */
    GEMM_KERNEL_TC = 1,     /* tcgen05 tensor-core GEMM */
    GEMM_KERNEL_SKINNY = 2, /* skinny-m GEMM */
    GEMM_KERNEL_REQUANT = 3, /* elementwise requantisation (gemm_i8_run_requant: K-split tiles, skinny path) */
    GEMM_KERNEL_KINDS = 4
};

/* Output types of gemm_i8_run_requant. */
enum { GEMM_OUT_BF16 = 1, GEMM_OUT_I8 = 2 };

#define GEMM_PLAN_VERSION 2
#define GEMM_I8_MAX_K 131071 /* 131071 * 128 * 128 < 2^31 */

/*
 * The selected configuration (patent CN114238853A claim 7: "input the size,
 * select the configuration and its kernel, run").  Filled by gemm_*_plan.
 *
 * Tail split (an addition to the patent's five steps, int8 only): when the
 * tiles do not fill a whole number of waves, the tiles of the last, partial
 * wave are split along K into split_k slices run by otherwise idle CTAs (CTA
 * pairs for the two-SM tile).  The staging kernel zeroes C over those tiles
 * and every slice adds its exact int32 partial sums into C (TMA reduce-add,
 * or atomics when C cannot take TMA); no slice waits on another.  Integer
 * addition is exact and order-free, so the result is bit-identical to the
 * unsplit one.  gemm_*_run recomputes the split for the tile and grid it
 * actually launches.
 */
typedef struct gemm_plan {
    int32_t version;   /* GEMM_PLAN_VERSION */
    int32_t path;      /* GEMM_PATH_* */
    int32_t dtype;     /* GEMM_DTYPE_* */
    int32_t num_sms;   /* SM count the plan was made for */
    int64_t m, k, n;
    int32_t bm, bn, bk;  /* CTA tile; bk = K elements per pipeline stage */
    int32_t stages;      /* depth of the shared-memory operand ring */
    int32_t tiles;       /* output tiles: Thread_Blocks of claim 4 */
    int32_t bpc;         /* CTAs per SM: block_per_cu of claim 6 */
    int32_t grid;        /* CTAs launched (persistent): min(tiles, num_sms * bpc) */
    int32_t waves;       /* ceil(tiles / (num_sms * bpc)): Launch_kernel_times of claim 6 */
    int32_t k_pitch;     /* row pitch (elements) of the staged 16-bit operands */
    int32_t chunk_k;     /* K elements accumulated in fp32 before an exact int32 drain */
    int32_t fallback;    /* 1 if no tile filled the chip (claim 4 S3) */
    int32_t split_k;     /* K slices of each tile in the last, partial wave (1 = none) */
    double ratio;        /* compute-to-memory ratio of the tile (claim 5), flop per byte */
    int64_t workspace_bytes; /* device scratch gemm_*_run takes from its pool (16-bit operand copies) */
    int32_t split_from;  /* tiles [split_from, tiles) are split into split_k K slices */
    int32_t a_on_chip;   /* 1: the two-SM kernel loads int8 A and widens it on chip (no f16 copy of A);
                            int8, bm == 256 and k % 16 == 0 only (see gemm_i8_plan) */
    int64_t reserved[3];
} gemm_plan;

/*
 * Plan an int8 problem (m x k) x (k x n) for the current CUDA device.
 * Routing: m <= 64, or m <= 128 with k % 16 == 0 -> skinny path (streams Bt
 * once, widening it on chip); otherwise the five
 * steps of CN114238853A claim 1 select a (BM, BN) tile.  When the two-SM tile
 * runs a narrow C (n <= 512) with k % 16 == 0, a_on_chip = 1: A is widened
 * from int8 inside the GEMM instead of through a staged f16 copy, which for
 * such shapes would move more bytes than the multiply.  Host-only apart from
 * one cached query of the device's SM count.
 * Errors: GEMM_ERR_INVALID_ARG (out == NULL, m/k/n outside [1, 2^31-1]),
 * GEMM_ERR_OVERFLOW_RISK (k > GEMM_I8_MAX_K), GEMM_ERR_CUDA (no device).
 */
GEMM_API gemm_status gemm_i8_plan(int64_t m, int64_t k, int64_t n, gemm_plan *out);

/* Plan a bf16 problem for the current device (always the tensor-core path). */
GEMM_API gemm_status gemm_bf16_plan(int64_t m, int64_t k, int64_t n, gemm_plan *out);

/*
 * Pure host planner: the same selection for an explicit SM count, with no
 * CUDA call at all.  dtype is GEMM_DTYPE_*.  Same errors as the above.
 */
GEMM_API gemm_status gemm_plan_for_sms(int32_t dtype, int64_t m, int64_t k, int64_t n, int32_t num_sms,
                              gemm_plan *out);

/*
 * C (int32, m x n) = A (int8, m x k) x B, with B given as Bt (int8, n x k).
 * All pointers are device pointers on the current device.  A and Bt must be
 * 16-byte aligned, C 4-byte aligned.  Exact: every element equals the int64
 * sum, which the plan's k limit keeps inside int32.
 * A plan may be edited before the call to force another compiled tile (bm in
 * {64, 128}, bn in {32, 64, 128, 256}) or another grid size (>= 1); every
 * such choice gives the same result.
 * Errors: GEMM_ERR_INVALID_ARG (null pointer, plan not from gemm_i8_plan or
 * of another version, tile not compiled), GEMM_ERR_MISALIGNED,
 * GEMM_ERR_UNSUPPORTED_DEVICE, GEMM_ERR_CUDA.  Nothing is launched when an
 * error is returned.
 */
GEMM_API gemm_status gemm_i8_run(const gemm_plan *plan, const int8_t *A, const int8_t *Bt, int32_t *C,
                        void *stream);

/*
 * C (fp32, m x n) = A (bf16, m x k) x B, B given as Bt (bf16, n x k); bf16
 * values are passed as their 16-bit patterns.  fp32 accumulation:
 * |C - exact| <= 1e-3 * sum_k |a*b| elementwise.  Same rules and errors as
 * gemm_i8_run.
 */
GEMM_API gemm_status gemm_bf16_run(const gemm_plan *plan, const uint16_t *A, const uint16_t *Bt, float *C,
                          void *stream);

/*
 * Requantising int8 GEMM: D = q( (float(C[i][j]) * row_scale[i]) * col_scale[j] )
 * for the exact int32 product C = A x B of gemm_i8_run, the usual consumer of
 * an int8 GEMM (per-row activation scales, per-column weight scales, a
 * narrower output).  The pages do not define requantisation; its arithmetic is
 * the library's and is stated here: every step is one IEEE-754 binary32
 * operation rounded to nearest, ties to even - (1) int32 -> float, (2) times
 * the row scale, (3) times the column scale - then q:
 *   GEMM_OUT_BF16  bfloat16, round to nearest even (overflow gives infinity,
 *                  NaN stays NaN); D holds m x n 16-bit patterns;
 *   GEMM_OUT_I8    int8: nearest integer, ties to even, then clamped to
 *                  [-128, 127]; NaN gives 0; D holds m x n int8.
 * Where one CTA completes a tile of C, the tile is requantised in the GEMM's
 * epilogue and C never reaches memory (the shared-memory staged write-back of
 * "先导杯比赛回顾", section "Epilogue 写回优化", carried one step further).  The
 * tiles of a K split and the skinny path's C are completed in int32 scratch
 * from the library's pool and converted by a second, elementwise kernel.
 * Same plan and operand rules as gemm_i8_run.  row_scale (m floats) and
 * col_scale (n floats) are device pointers, 16-byte aligned; D is a device
 * pointer (2-byte aligned for bfloat16), row pitch n.
 * Errors: GEMM_ERR_INVALID_ARG (null pointer, bad plan or out_type),
 * GEMM_ERR_MISALIGNED, GEMM_ERR_UNSUPPORTED_DEVICE, GEMM_ERR_CUDA.
 */
GEMM_API gemm_status gemm_i8_run_requant(const gemm_plan *plan, const int8_t *A, const int8_t *Bt,
                                         const float *row_scale, const float *col_scale, int32_t out_type, void *D,
                                         void *stream);

/*
 * gemm_i8_run without any device-memory allocation.  The pages have no
 * counterpart to this entry point.
 *
 * For callers that may not allocate device memory, directly or through a
 * library: runtimes that plan all device memory up front and forbid libraries
 * to take more, and latency-critical loops where an allocation could block,
 * synchronise the device or fail mid-run.  The f16 operand copies that
 * gemm_i8_run takes from a memory pool go instead into one fixed scratch
 * array of GEMM_NOALLOC_SCRATCH_BYTES (64 MiB) in the library's device image,
 * which every GPU that loads the library holds until the process exits.  The
 * call makes no cudaMalloc, cudaFree or other allocating call.
 *
 * Same arguments, rules and result as gemm_i8_run.  Extra rules:
 *   - the tensor-core path needs round256(m*k_pitch*2) + round256(n*k_pitch*2)
 *     bytes of scratch; larger problems return GEMM_ERR_INVALID_ARG and
 *     launch nothing; the skinny path needs m*k*2 bytes (at most 32 MiB) for
 *     the f16 copy of A when k % 16 == 0, and none otherwise;
 *   - the first call on each device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it; make that
 *     first call before any stream capture;
 *   - every call shares the one array and it keeps the last call's contents
 *     (each call overwrites what it reads and clears its own time-out word),
 *     so calls whose work overlaps on the GPU race and give wrong results:
 *     order them on one stream or with events;
 *   - a kernel wait that runs past its limit ends the call's kernels early
 *     (C incomplete) and records its code in the device error word that all
 *     entry points share (a static device variable, not an allocation):
 *     gemm_device_error reports it as for gemm_i8_run.
 */
#define GEMM_NOALLOC_SCRATCH_BYTES (64ll << 20)
GEMM_API gemm_status gemm_i8_run_noalloc(const gemm_plan *plan, const int8_t *A, const int8_t *Bt, int32_t *C,
                                void *stream);

/*
 * End-to-end forms: A, Bt and C are HOST pointers (pinned or pageable).  The
 * call takes device buffers from the library's pool, copies A and Bt to the
 * device, runs the plan, copies C back and waits for `stream` to finish, so
 * C is ready when it returns.  Large tensor-path problems (at least 2048
 * rows of C, at least 32 MiB of A, Bt and C together) run as a pipeline on
 * four library streams that
 * follow `stream`: A and Bt are cut into bands of at least 1024 rows (at most
 * 8 each), copied up one band at a time and widened once; each band's arrival
 * completes a rectangle of C, which is multiplied and copied down while later
 * bands go up.  Rectangles run the two-SM 256 x 256 tile, so an edited
 * plan's tile applies only to calls that are not pipelined.  Calls on one
 * device take the pipeline one at a time.
 */
GEMM_API gemm_status gemm_i8_run_host(const gemm_plan *plan, const int8_t *A, const int8_t *Bt, int32_t *C,
                             void *stream);
GEMM_API gemm_status gemm_bf16_run_host(const gemm_plan *plan, const uint16_t *A, const uint16_t *Bt, float *C,
                               void *stream);

/*
 * Waits for `stream`, then reads and clears the current device's error word,
 * which the kernels of every run entry point (gemm_i8_run_noalloc included)
 * write when a wait gives up; the first code since the last read is kept.
 * Returns GEMM_OK, GEMM_ERR_TIMEOUT (a kernel wait ran past its 2 s limit
 * and the kernel returned early; *code gets the stage that gave up) or
 * GEMM_ERR_CUDA.  `code` may be NULL.
 */
GEMM_API gemm_status gemm_device_error(void *stream, int32_t *code);

/*
 * The library's private stream-ordered memory pool on the current device
 * (the scratch of gemm_*_run and the device buffers of gemm_*_run_host):
 * bytes it holds now (*reserved_bytes) and the most bytes in use at once
 * since the pool was created or the mark was last reset (*used_high_bytes).
 * reset_high != 0 restarts that mark from the current use after reading it.
 * For callers that budget device memory; the pool keeps freed memory for the
 * next call and returns it only when the process exits.
 * Errors: GEMM_ERR_INVALID_ARG (NULL output), GEMM_ERR_UNSUPPORTED_DEVICE,
 * GEMM_ERR_CUDA.
 */
GEMM_API gemm_status gemm_pool_usage(int64_t *reserved_bytes, int64_t *used_high_bytes, int32_t reset_high);

/*
 * Tracing.  While enabled, every kernel launch made by gemm_*_run is counted
 * per GEMM_KERNEL_* kind, and every `every`-th gemm_*_run call (the first,
 * the (every+1)-th, ...) records a pair of CUDA events on its stream around
 * each timed unit (at most `capacity` units are recorded): the staging
 * launch and the GEMM launch of the tensor path separately (kinds STAGE and
 * TC); on the skinny tensor-core path the prologue launch (A to f16, C
 * zeroed) and the skinny launch together, as kind SKINNY, because the skinny
 * kernel starts while the prologue runs (programmatic dependent launch).
 * Calls that are not sampled record no events, so sampling keeps the timing
 * from slowing the work it measures.  Back-to-back skinny calls on one
 * stream overlap (each call's kernels start before the previous call's
 * end); an event recorded between two calls, as a sampled call records,
 * makes them run one after the other.  gemm_trace_collect waits for the events and writes,
 * per kind (arrays of GEMM_KERNEL_KINDS entries): the summed device time in
 * ms of the timed units, the number of timed units, and the number of
 * launches counted; it then disables tracing.  every >= 1.
 */
GEMM_API gemm_status gemm_trace_begin(int32_t capacity, int32_t every);
GEMM_API gemm_status gemm_trace_collect(float *ms_per_kind, int32_t *timed_per_kind, int32_t *launches_per_kind);

/* Registers per thread and CTAs per SM of the compiled tensor-core kernel for
 * a tile (-1 / 0 if no such kernel); needs a device. */
GEMM_API gemm_status gemm_tc_kernel_info(int32_t bm, int32_t bn, int32_t dtype, int32_t *regs, int32_t *ctas_per_sm);

/*
 * Failure-detection self-test.  Launches one CTA that waits on a barrier
 * nothing completes, with a limit of `timeout_us` microseconds (1 .. 2e6)
 * instead of the kernels' 2 s.  The wait gives up, records code 5 in the
 * device error word and the kernel returns: a following gemm_device_error()
 * returns GEMM_ERR_TIMEOUT with *code = 5, and the CUDA context stays usable.
 * Nothing faults, traps or hangs.
 */
GEMM_API gemm_status gemm_selftest_wait_timeout(int32_t timeout_us, void *stream);

/* Human-readable name of a status. */
GEMM_API const char *gemm_status_string(gemm_status s);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_INT8_MATRIX_H */
