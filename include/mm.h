/*
 * mm.h -- C ABI of the GB300 (sm_103a) autotuned dense matmul.
 *
 * The library computes C = A.B on one GPU.  Each call builds a tuning key
 * from the problem (shape buckets, alignment factors, element types and
 * layouts), looks it up in a per-device tuning table, and on a miss
 * benchmarks a grouped, prioritised set of hand-written candidate kernels on
 * the device, records the fastest and runs it.  The design follows the burn
 * "autotune" page (rustineverything.app/docs/burn/06-cubecl/autotune) for the
 * key, the plan, the roofline bound and the table, and the PyTorch TunableOp
 * guide (blog.gitcode.com, "PyTorch TunableOp practical guide") for the
 * tuning budget, rotating buffers, result file and validators.
 *
 * Conventions used by every entry point
 * -------------------------------------
 *  Logical shapes: A is M x K, B is K x N, C is M x N (row-major logically),
 *  optionally repeated over a batch.
 *  Layout letters (first = A, second = B):
 *    N  the operand is stored row-major: element (r, c) at r*ld + c.
 *    T  the operand is stored column-major (a transposed view):
 *       element (r, c) at c*ld + r.
 *  C is always stored row-major: element (i, j) at i*ldc + j.
 *  Leading dimensions and batch strides are in ELEMENTS.  Operands are read
 *  in place through their strides; nothing is made contiguous first (burn
 *  "cubecl-backend" page, section "matmul: handing strides to cubek").
 *  Element types: bf16, f16 or f32 for A, B and C.  Accumulation is always
 *  fp32.  f32 inputs may be multiplied as tf32 by tensor-core candidates
 *  (the same page: the kernel may compute f32 as tf32).
 *
 * Ownership: all data pointers and the stream belong to the caller; the
 * library never frees or retains them past the call.  `out` is written only
 * by the chosen kernel's final launch: benchmarking uses private copies
 * (rotating buffers), so an in-place or accumulating output is never
 * corrupted by tuning.  The library owns its scratch (split-K workspaces,
 * rotating sets, flush buffer) and frees it in mm_shutdown().
 *
 * Alignment: lhs, rhs and out must each start on a multiple of their element
 * size (2 bytes for bf16/f16, 4 for f32); a pointer that does not is rejected
 * with MM_ERR_INVALID_ARG before anything is launched.  Other alignments
 * (16-byte bases or leading dimensions) only narrow the candidates.
 *
 * Errors: every entry point returns an mm_status; on failure a thread-local
 * message is available from mm_last_error().  Device pointers are not
 * dereferenced on the host.  Calls are thread-safe; a second caller that
 * misses on a key another thread is tuning waits (bounded) for the result.
 */
#ifndef MM_GB300_H
#define MM_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t mm_status;
#define MM_OK 0
#define MM_ERR_INVALID_ARG 1        /* bad sizes, strides, dtype or layout */
#define MM_ERR_UNSUPPORTED 2        /* this candidate cannot run this problem */
#define MM_ERR_CUDA 3               /* a CUDA runtime/driver call failed */
#define MM_ERR_NO_VALID_CANDIDATE 4 /* every planned candidate failed */
#define MM_ERR_CACHE_VALIDATION 5   /* result file rejected by a validator row */
#define MM_ERR_IO 6                 /* result file unreadable / unwritable */
#define MM_ERR_TIMEOUT 7            /* a kernel's bounded wait gave up */
#define MM_ERR_NOT_FOUND 8          /* key not in the table / unknown name */

typedef enum { MM_BF16 = 0, MM_F16 = 1, MM_F32 = 2 } mm_dtype;

/* Element types of A, B and C (mm_dtype values). */
typedef struct {
  int32_t a, b, c;
} mm_dtypes;

typedef enum { MM_NN = 0, MM_NT = 1, MM_TN = 2, MM_TT = 3 } mm_layout;

/* Batched problems: `batch` matrices; item b of A starts at A + b*stride_a
 * elements (likewise B, C).  A NULL mm_batch* means batch = 1. */
typedef struct {
  int64_t batch;
  int64_t stride_a, stride_b, stride_c;
} mm_batch;

/* Tuning key: a plain 64-byte value; two keys are equal iff memcmp == 0. */
typedef struct {
  uint8_t bytes[64];
} mm_key;

/* Process-wide counters (all devices). */
typedef struct {
  uint64_t calls;          /* mm_autotune_execute / _host calls */
  uint64_t hits;           /* calls whose key was in the in-memory table */
  uint64_t misses;         /* calls that had to tune (or wait for a tuner) */
  uint64_t tunes;          /* completed tuning runs */
  uint64_t launches;       /* kernel launches by the library, all purposes */
  uint64_t bench_launches; /* of which: benchmark launches while tuning */
  double last_tune_ms;     /* host wall time of the last tuning run */
  double total_tune_ms;    /* sum over tuning runs */
} mm_stats;

/* ---------------------------------------------------------------------- */

/*
 * mm_tune_key -- the tuning key of a problem (host only, no GPU needed).
 * Follows the burn "autotune" page, section "tuning key: shape bucketing":
 * m, n, k (and the batch count) anchored to buckets (Balanced: next power of
 * two; MM_AUTOTUNE_LEVEL selects minimal/balanced/extensive/full),
 * per-operand pow2 vectorisation factor of the anchored contiguous dimension
 * (at most 4), per-operand stride alignment factor (largest power of two, at
 * most 2^10, dividing every non-unit stride in bytes, real strides), element
 * types, per-operand layout (Contiguous / MildlyPermuted{transposed,
 * batch_swap}), scale (Small/Medium/Large) and kind (General, MatVec, ...).
 *   out   receives the 64-byte key (required).
 *   text  optional buffer for the canonical text form (space-separated
 *         field=value pairs, NUL-terminated, truncated to text_cap-1).
 * Errors: MM_ERR_INVALID_ARG for negative sizes, ld smaller than the
 * contiguous extent, unknown dtype/layout, batch < 0.
 */
mm_status mm_tune_key(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                      mm_dtypes dt, mm_layout layout, const mm_batch *batch, mm_key *out,
                      char *text, size_t text_cap);

/*
 * mm_autotune_execute -- C = A.B on the current CUDA device, on `stream`
 * (a cudaStream_t; NULL = the legacy default stream).  lhs/rhs/out are
 * device pointers.  On a table hit: one launch of the recorded kernel (the
 * warm path of the autotune page, "first time a key is met": compute the key,
 * look it up, run the fastest).  On a miss with tuning enabled: plan, bound,
 * benchmark on a private stream (ordered after `stream`'s pending work),
 * record, then launch the winner on `stream`.  With tuning disabled a miss
 * runs the always-valid default kernel (TunableOp's Default).  M, N or batch
 * of 0 is a no-op; K = 0 writes zeros.  While `stream` is being captured
 * into a CUDA graph a miss is not tuned: the default kernel is captured; a
 * hit whose recorded winner needs scratch not yet allocated on `stream`
 * (split-K workspaces, repack copies) captures the next candidate of the
 * key's ranking that needs none.
 * Errors: MM_ERR_INVALID_ARG, MM_ERR_CUDA, MM_ERR_NO_VALID_CANDIDATE.
 */
mm_status mm_autotune_execute(const void *lhs, const void *rhs, void *out, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, int64_t ldc, mm_dtypes dt,
                              mm_layout layout, const mm_batch *batch, void *stream);

/*
 * mm_autotune_execute_host -- the same product from HOST buffers: copies
 * lhs and rhs (their strided spans) to library-owned device staging buffers,
 * runs mm_autotune_execute on `stream`, copies the result span back into
 * `out` (host) and synchronises `stream`.  Host buffers may be pageable;
 * pinned buffers make the copies asynchronous-capable and faster.
 * Errors: as mm_autotune_execute, plus MM_ERR_CUDA for allocation failures.
 */
mm_status mm_autotune_execute_host(const void *lhs, const void *rhs, void *out, int64_t M,
                                   int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                   mm_dtypes dt, mm_layout layout, const mm_batch *batch,
                                   void *stream);

/*
 * mm_cache_load / mm_cache_save -- the on-disk tuning table of the current
 * device, a CSV in the format of TunableOp's result file (the guide's section
 * 3.2): "Validator,<NAME>,<value>" rows followed by
 * "MatmulKey,<key text>,<candidate name>,<median ms>,<all candidates>" rows.
 * Validators: MM_VERSION (the library version, the part of mm_version()
 * before '+'), CANDIDATE_CHECKSUM (mm_candidate_checksum() as 16 hex digits:
 * a hash of every candidate name in registry order, so renaming, adding or
 * removing a candidate orphans old entries, as on the autotune page's step
 * 1), DEVICE ("<device name>|sm_<major><minor>": the model, so a table tuned
 * on one unit serves every unit of that model) and CUDA_VERSION (runtime).  Any
 * validator mismatch rejects the WHOLE file (MM_ERR_CACHE_VALIDATION).  A row
 * naming an unknown candidate is skipped; "Default" means the default kernel.
 *   path  NULL -> MM_CACHE_FILE; the device ordinal is inserted before the
 *         extension ("results.csv" -> "results0.csv").
 * Load merges into the in-memory table (existing keys are kept).
 * Errors: MM_ERR_IO, MM_ERR_CACHE_VALIDATION, MM_ERR_INVALID_ARG (no path).
 */
mm_status mm_cache_load(const char *path);
mm_status mm_cache_save(const char *path);

/* Offline tuning (PyTorch TunableOp guide, sections 6-7: record the
 * operations met while tuning is off, tune them later from the file).  With
 * the option "record_untuned" set to a path (env MM_RECORD_UNTUNED), a key
 * missed while tuning is off is appended once per process to that file as
 *   Untuned,<key text>,M,N,K,lda,ldb,ldc,<a type>,<b type>,<c type>,<layout>,
 *   batch,stride_a,stride_b,stride_c
 * mm_tune_file tunes every recorded problem not yet in the current device's
 * table, on library-allocated synthetic operands of the recorded shape and
 * strides (pseudo-random values in [-1, 1); freed before it returns), and
 * sets *tuned to the number tuned;
 * the results can then be written with mm_cache_save.  Runs whether or not
 * the "tuning" option is on.  Errors: MM_ERR_IO if the file cannot be read,
 * MM_ERR_INVALID_ARG for a malformed record, MM_ERR_CUDA, or the tuner's own
 * errors; lines that are not Untuned records are skipped. */
mm_status mm_tune_file(const char *path, int *tuned);
/* Forget every in-memory entry of the current device. */
mm_status mm_cache_clear(void);
/* Number of in-memory entries of the current device (or -1 on error). */
int64_t mm_cache_size(void);

/* Candidate registry: index 0 is the always-valid default (naive) kernel. */
int32_t mm_candidate_count(void);
const char *mm_candidate_name(int32_t index); /* NULL if out of range */
/* Launches of one candidate by this process (benchmark + execute). */
uint64_t mm_candidate_launches(int32_t index);
/* FNV-1a 64 hash of every candidate name (each followed by a newline) in
 * registry order, then of the library version: the CANDIDATE_CHECKSUM
 * validator of the result file.  Host only. */
uint64_t mm_candidate_checksum(void);

/*
 * mm_execute_candidate -- run one candidate directly (no key, no table):
 * the test hook that lets every candidate be compared with the oracle.
 * Errors: MM_ERR_UNSUPPORTED if the candidate cannot run this problem
 * (alignment, dtype, layout or size gate), else as mm_autotune_execute.
 */
mm_status mm_execute_candidate(int32_t index, const void *lhs, const void *rhs, void *out,
                               int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                               int64_t ldc, mm_dtypes dt, mm_layout layout, const mm_batch *batch,
                               void *stream);

/* mm_lookup -- the recorded candidate of a key on the current device, or
 * *index = -1 and MM_ERR_NOT_FOUND. */
mm_status mm_lookup(const mm_key *key, int32_t *index);

/*
 * mm_plan -- the tuning plan of a problem on the current device (test and
 * report hook; follows the autotune page's group rules).  Fills up to `cap`
 * entries of four parallel arrays, in try order: candidate index, group id,
 * tier rank inside the group (0 = the round, 1.. = backups) and whether the
 * candidate supports the problem (unsupported ones are demoted, not
 * dropped).  group_prio/prio, if not NULL, receive the group priority and
 * the in-group priority (before demotion).  Returns the number of entries.
 */
int32_t mm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                mm_dtypes dt, mm_layout layout, const mm_batch *batch, int32_t cap,
                int32_t *cand, int32_t *group, int32_t *tier, int32_t *supported,
                int32_t *group_prio, int32_t *prio);
/* Name of a group id reported by mm_plan ("gemv", "tensor", "naive"). */
const char *mm_group_name(int32_t group);

/*
 * mm_default_candidate -- the candidate a miss that is not tuned runs on the
 * current device (tuning off, or a pending key whose tuner did not finish in
 * time; the TunableOp guide's Default, made a heuristic): a shape-class
 * preference drawn from the GB300 tuning results (M = 1: the streaming
 * GEMVs; M <= 16: the warp-MMA GEMV for A and B row-major, or for B
 * transposed when A's rows are not 16-byte aligned, else the swapped
 * tensor-core split-K; few tiles and deep K:
 * split-K; f32: the 1-SM tile; small outputs: the 128 x 64 tile; otherwise
 * the 2-SM 256 x 256 tile, or the copying form when A's rows are not 16-byte
 * aligned), then the plan's order, first that supports the problem.  Test and
 * report hook; the data pointers are taken as 256-byte aligned.  Returns the
 * candidate index, or -1 for invalid arguments.
 */
int32_t mm_default_candidate(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                             int64_t ldc, mm_dtypes dt, mm_layout layout, const mm_batch *batch);

/*
 * mm_device_peaks -- the roofline peaks the tuner uses on the current device
 * (autotune page, section "roofline and the hundred thousand launches": the
 * probes run once per device): the dense bf16 tensor rate (the peak_tflops
 * option, else GB300's nominal 2.25 PFLOP/s), the memory bandwidth (the
 * peak_gbs option, else a timed device copy of 4 x L2 read and written), and
 * the launch overhead (200 empty launches between two events).  The first
 * call on a device (or the first tune) runs the probes; later calls return
 * the cached values.  Null outputs are skipped.  Errors: MM_ERR_CUDA.
 */
mm_status mm_device_peaks(double *bf16_ops_per_s, double *bytes_per_s, double *launch_ns);

/*
 * mm_roofline_limit_ns -- the tuning time limit of the autotune page,
 * section "roofline and the hundred thousand launches":
 * max(ops/peak_ops, bytes/peak_bytes) / threshold + launch overhead, in ns.
 */
double mm_roofline_limit_ns(double ops, double peak_ops_per_s, double bytes,
                            double peak_bytes_per_s, double threshold, double launch_ns);

/*
 * Options (TunableOp's tuning context, the guide's section 7): names are
 * the MM_* environment variables without the prefix, lower-case:
 *   tuning (1), autotune_cache (1), autotune_level (balanced),
 *   max_tuning_iterations (100), max_tuning_duration_ms (30),
 *   rotating_buffer_mb (-1 = 2 x L2; 0 disables), l2_flush (0),
 *   numerical_check ("" or "atol_rtol"), cache_file (""), decisions
 *   ("" | "stdout" | path), verbose (0), peak_tflops (0 = probe/nominal),
 *   peak_gbs (0 = probe), fault ("" | "<candidate>:<mode>", host-side
 *   fault injection; modes error, nan, slow, wrong, stall: the host sleeps
 *   1.5 s before benchmarking that candidate), record_untuned (""),
 *   pending_wait_ms (120000: how long a miss on a key that another thread is
 *   tuning waits before it runs the default kernel instead), wait_limit_us
 *   (2000000: how long a wait of a 1-SM tensor-core kernel's main loop may
 *   last before the kernel gives up, records MM_ERR_TIMEOUT's cause in its
 *   error word and returns; its drain waits keep 2 s), wait_stall (0; test
 *   hook: 1 makes the MMA warp of those kernels first wait on a barrier that
 *   nothing arrives on, so that the wait limit runs out and the kernel's
 *   abort path runs; it never faults or hangs the device).
 * An environment variable, when set, takes precedence over the API (the
 * environment is read once, at first use).  Errors: MM_ERR_NOT_FOUND for an
 * unknown name, MM_ERR_INVALID_ARG for a bad value.
 */
mm_status mm_set_option(const char *name, const char *value);
/* Current value as text into buf; MM_ERR_NOT_FOUND for an unknown name. */
mm_status mm_get_option(const char *name, char *buf, size_t cap);

mm_status mm_get_stats(mm_stats *out);
void mm_reset_stats(void);

/* Thread-local message of the last failing call on this thread. */
const char *mm_last_error(void);
/* Library version string ("<semver>+<build fingerprint>"). */
const char *mm_version(void);

/*
 * mm_splitk_gemm_noalloc -- C = A.B (batch 1) with the split-K tensor-core
 * kernel, allocating nothing.  No counterpart in the pages this library
 * follows: it serves callers that may not call cudaMalloc/cudaFree -- a
 * server that reserves all device memory for its own pool at start-up, a
 * plugin inside a framework that owns the allocator, a latency-bound loop
 * that cannot take the implicit device synchronisation of an allocation.
 * Arguments are those of mm_autotune_execute without the batch; lhs, rhs and
 * out are device pointers the caller owns; the call is asynchronous on
 * `stream`.  The K-slice partial sums go to a fixed 16 MiB workspace that is
 * part of the library's device image (held on every GPU that loads the
 * library until exit; its last 256 bytes hold an error word): M*N must be
 * at most 2,097,120 (two fp32 slices), else
 * MM_ERR_INVALID_ARG with the limit in the message.  Differences from
 * mm_autotune_execute for the same arguments: K = 0 is rejected
 * (MM_ERR_INVALID_ARG) instead of writing zeros, and K must span at least two
 * 128-byte blocks (K > 64 for bf16/f16, K > 32 for f32), else
 * MM_ERR_UNSUPPORTED; alignment and type rules are those of the tensor-core
 * candidates (16-byte aligned A, B and leading dimensions; f32 only as NT),
 * else MM_ERR_UNSUPPORTED.
 * The first call on a device resolves the workspace's device address
 * (cudaGetSymbolAddress) with that device current; make it before any stream
 * capture.  The address is kept for the life of the process, or until
 * mm_shutdown, which forgets it (call mm_shutdown after a cudaDeviceReset).
 * All calls share the workspace, so calls whose GPU execution overlaps (two
 * streams, two threads) race and must be ordered by the caller.
 * A kernel whose bounded wait gives up records a code in the workspace; the
 * call itself has returned MM_OK by then (it is asynchronous) and its product
 * is wrong.  mm_splitk_gemm_noalloc_status reports it.
 */
mm_status mm_splitk_gemm_noalloc(const void *lhs, const void *rhs, void *out, int64_t M,
                                 int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                 mm_dtypes dt, mm_layout layout, void *stream);

/*
 * mm_splitk_gemm_noalloc_status -- synchronises `stream`, then reads the
 * no-allocation workspace's error word on the current device (a 4-byte copy
 * to the host; nothing is allocated).  MM_OK when no kernel of
 * mm_splitk_gemm_noalloc gave up a bounded wait since the previous query;
 * otherwise clears the word and returns MM_ERR_TIMEOUT (the products of those
 * calls may be wrong).  Errors: MM_ERR_CUDA.
 */
mm_status mm_splitk_gemm_noalloc_status(void *stream);

/* Free every library-owned device buffer and the tables; saves the table of
 * each device to MM_CACHE_FILE first when that option is set and tuning
 * produced new entries.  The library may be used again afterwards. */
void mm_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* MM_GB300_H */
