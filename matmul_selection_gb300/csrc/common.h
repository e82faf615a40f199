// Internal declarations of the GB300 autotuned matmul library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <shared_mutex>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/mm.h"

#include <utility>

namespace mm {

// Programmatic dependent launch.  Every kernel of the library is launched
// with the programmatic-serialization attribute and begins with
// pdl_launch_dependents() (the next kernel on the stream may be scheduled
// into SM slots this grid leaves free) and pdl_wait() (block until the
// previous kernel on the stream has completed and its writes are visible)
// before it touches global memory.  Stream order is thus unchanged for memory;
// what overlaps is the launch of a kernel with the tail of its predecessor.
// Launched without the attribute, pdl_wait() returns at once.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// L2 prefetch of one box of a tensor map (element coordinates x, y, z).  It
// writes no shared memory and returns nothing to the SM, so it may run before
// pdl_wait(): the data it warms is read after the wait, through the coherent
// L2.  The innermost coordinate x must be a multiple of 16 bytes; boxes that
// reach past the tensor are clipped.
__device__ __forceinline__ void prefetch_box_l2(const CUtensorMap *map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}
#endif

// A tensor map over a row-major operand -- `inner` elements a row (stride
// ld_bytes), `outer` rows, `batch` matrices bstride_bytes apart -- used only
// for L2 prefetch boxes of box_inner x box_outer elements (no swizzle: the
// box's row is any multiple of 16 bytes; both extents at most 256).  Needs a
// 16-byte aligned base and strides that are multiples of 16 bytes.
mm_status encode_prefetch_map(CUtensorMap *map, int dtype, const void *base, uint64_t inner,
                              uint64_t outer, uint64_t batch, uint64_t ld_bytes,
                              uint64_t bstride_bytes, uint32_t box_inner, uint32_t box_outer);

// Launch `kern` with the programmatic-serialization attribute and, unless
// `cluster` is 1 x 1 x 1, that cluster shape.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       dim3 cluster, Args &&...args) {
  cudaLaunchAttribute at[2];
  unsigned n = 0;
  at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster.x * cluster.y * cluster.z > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster.x;
    at[n].val.clusterDim.y = cluster.y;
    at[n].val.clusterDim.z = cluster.z;
    ++n;
  }
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  lc.attrs = at;
  lc.numAttrs = n;
  return cudaLaunchKernelEx(&lc, kern, std::forward<Args>(args)...);
}

}  // namespace mm

namespace mm {

constexpr const char *kVersion = "0.2.0";

// ---------------------------------------------------------------- problem
struct Problem {
  const void *A;
  const void *B;
  void *C;
  int64_t M, N, K;
  int64_t lda, ldb, ldc;
  int64_t batch;
  int64_t sA, sB, sC;  // batch strides, elements
  int ta, tb, tc;      // mm_dtype of A, B, C
  bool at, bt;         // A / B stored transposed (layout letter T)
};

inline int dtype_bytes(int t) { return t == MM_F32 ? 4 : 2; }
inline const char *dtype_name(int t) {
  return t == MM_BF16 ? "bf16" : t == MM_F16 ? "f16" : t == MM_F32 ? "f32" : "?";
}

// Elements from the first to one past the last element an operand addresses.
int64_t span_elems(int64_t rows, int64_t cols, int64_t ld, bool trans, int64_t batch,
                   int64_t bstride);
inline int64_t span_a(const Problem &p) { return span_elems(p.M, p.K, p.lda, p.at, p.batch, p.sA); }
inline int64_t span_b(const Problem &p) { return span_elems(p.K, p.N, p.ldb, p.bt, p.batch, p.sB); }
inline int64_t span_c(const Problem &p) { return span_elems(p.M, p.N, p.ldc, false, p.batch, p.sC); }

// Fill a Problem from C-ABI arguments and check it; MM_OK or INVALID_ARG.
mm_status make_problem(Problem *p, const void *lhs, const void *rhs, void *out, int64_t M,
                       int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, mm_dtypes dt,
                       mm_layout layout, const mm_batch *batch);

// ---------------------------------------------------------------- errors
mm_status set_error(mm_status s, const char *fmt, ...);
mm_status cuda_error(cudaError_t e, const char *what);
#define MM_CUDA_TRY(expr)                                     \
  do {                                                        \
    cudaError_t e__ = (expr);                                 \
    if (e__ != cudaSuccess) return ::mm::cuda_error(e__, #expr); \
  } while (0)

// ---------------------------------------------------------------- key
// 64-byte plain key; every byte is defined (zero padding) so memcmp works.
struct KeyPod {
  uint64_t m, n, k, batch;
  uint8_t lhs_pow2, lhs_stride, rhs_pow2, rhs_stride;
  uint8_t elem_lhs, elem_rhs, elem_out;
  uint8_t layout_lhs, layout_rhs;  // Layout enum
  uint8_t scale, kind;
  uint8_t pad[21];
};
static_assert(sizeof(KeyPod) == 64, "key must be 64 bytes");

enum Layout : uint8_t {
  LAYOUT_CONTIGUOUS = 0,
  LAYOUT_MP_T = 1,    // MildlyPermuted{transposed:true,  batch_swap:false}
  LAYOUT_MP_B = 2,    // MildlyPermuted{transposed:false, batch_swap:true}
  LAYOUT_MP_TB = 3,   // MildlyPermuted{transposed:true,  batch_swap:true}
  LAYOUT_HIGHLY = 4,  // HighlyPermuted (not expressible through this ABI)
};
enum Scale : uint8_t { SCALE_SMALL = 0, SCALE_MEDIUM = 1, SCALE_LARGE = 2 };
enum Kind : uint8_t {
  KIND_GENERAL = 0, KIND_MATVEC, KIND_VECMAT, KIND_SCALARVEC, KIND_VECSCALAR,
  KIND_INNER, KIND_OUTER
};
enum Level { LEVEL_MINIMAL = 0, LEVEL_BALANCED = 1, LEVEL_EXTENSIVE = 2, LEVEL_FULL = 3 };

uint64_t anchor(uint64_t x, int level);
KeyPod make_key(const Problem &p, int level);
std::string key_text(const KeyPod &k);
bool parse_key_text(const std::string &s, KeyPod *out);

struct KeyHash {
  size_t operator()(const KeyPod &k) const;
};
struct KeyEq {
  bool operator()(const KeyPod &a, const KeyPod &b) const {
    return std::memcmp(&a, &b, sizeof(KeyPod)) == 0;
  }
};

// ---------------------------------------------------------------- options
struct Options {
  int tuning = 1;
  int autotune_cache = 1;
  int level = LEVEL_BALANCED;
  int max_tuning_iterations = 100;
  double max_tuning_duration_ms = 30.0;
  double rotating_buffer_mb = -1.0;
  int l2_flush = 0;
  std::string numerical_check;  // "" or "atol_rtol"
  std::string cache_file;
  std::string decisions;
  int verbose = 0;
  double peak_tflops = 0.0;
  double peak_gbs = 0.0;
  std::string fault;
  std::string record_untuned;  // path: keys missed with tuning off are appended here
  double pending_wait_ms = 120000.0;  // how long a miss waits for another thread's tuner
  double wait_limit_us = 2000000.0;   // 1-SM tensor-core kernels: main-loop wait limit
  int wait_stall = 0;                 // test hook: 1-SM kernels wait on a barrier nothing arrives on
};
// The current options (env values take precedence over the API), through a
// per-thread copy refreshed when an option changes.
const Options &get_options();
// The same, built afresh under the options lock: for code that may run after
// the calling thread's thread-local objects are gone (exit handlers).
Options snapshot();
mm_status set_option(const std::string &name, const std::string &value);
mm_status get_option(const std::string &name, std::string *value);

// ---------------------------------------------------------------- device
struct DeviceInfo {
  int ordinal = -1;
  int sms = 0;
  int cc_major = 0, cc_minor = 0;
  int64_t l2_bytes = 0;
  int64_t smem_optin = 0;
  int64_t total_mem = 0;
  std::string name, uuid;
};

// Library-owned device buffer that grows on demand.
struct DevBuf {
  void *ptr = nullptr;
  size_t bytes = 0;
  mm_status ensure(size_t need);
  void release();
};

struct TableEntry {
  int winner = 0;               // candidate index
  std::vector<int> ranking;     // valid candidates, fastest first
  double median_ms = 0.0;
  std::string detail;           // "name:median;..." for the result file
  bool from_file = false;
};

struct Peaks {
  bool ready = false;
  double bf16_ops = 0, tf32_ops = 0, bytes_per_s = 0, launch_ns = 0;
  std::string source;
};

struct DeviceState {
  DeviceInfo info;
  int *d_err = nullptr;                  // kernel error word (bounded-wait timeouts)
  cudaStream_t tune_stream = nullptr;
  cudaEvent_t ev_order = nullptr;
  std::mutex scratch_mu;
  // per-(stream, slot) scratch: slot SCRATCH_TICKETS holds zero-initialised
  // counters that kernels leave at zero; SCRATCH_WORKSPACE holds partial sums
  std::map<std::pair<cudaStream_t, int>, DevBuf> scratch;
  DevBuf flush_buf;
  DevBuf stage_a, stage_b, stage_c;        // host-buffer entry point staging
  std::mutex stage_mu;
  // tuning table
  std::shared_mutex table_mu;
  std::unordered_map<KeyPod, std::shared_ptr<const TableEntry>, KeyHash, KeyEq> table;
  std::mutex pending_mu;
  std::condition_variable pending_cv;
  std::unordered_set<KeyPod, KeyHash, KeyEq> pending;
  std::mutex untuned_mu;
  std::unordered_set<KeyPod, KeyHash, KeyEq> untuned;  // keys already recorded this process
  bool file_loaded = false;
  bool dirty = false;
  std::mutex tune_mu;  // one tuning run at a time per device
  Peaks peaks;
};

// The state of the current device (creating it on first use).
mm_status current_device(DeviceState **out);
// Drop every device state (mm_shutdown).
void release_all_devices();
// Forget the no-allocation entry point's per-device workspace addresses.
void noalloc_forget_devices();
void for_each_device(void (*fn)(DeviceState &));

// Scratch of at least `bytes` private to (device, stream, slot).  A new or
// grown buffer is zero-filled (stream-ordered).
enum ScratchSlot { SCRATCH_TICKETS = 0, SCRATCH_WORKSPACE = 1, SCRATCH_REPACK = 2 };
mm_status get_scratch(DeviceState &ds, cudaStream_t s, int slot, size_t bytes, void **out);

// ---------------------------------------------------------------- candidates
enum Group { GROUP_GEMV = 0, GROUP_TENSOR = 1, GROUP_NAIVE = 2, GROUP_COUNT = 3 };
constexpr int PRIORITY_MAX = 3, PRIORITY_HIGH = 2, PRIORITY_MEDIUM = 1, PRIORITY_MIN = 0,
              PRIORITY_NEVER = -1;

struct LaunchCtx {
  cudaStream_t stream;
  DeviceState *dev;
  bool tuning;  // benchmark launch (counted separately)
};

struct Candidate {
  std::string name;
  int group;
  int cfg;  // index into the family's config table
  int (*prio)(const KeyPod &, const Problem &, const DeviceInfo &, int cfg);
  bool (*supports)(const Problem &, const DeviceInfo &, int cfg, std::string *why);
  mm_status (*launch)(const Problem &, LaunchCtx &, int cfg);
};

const std::vector<Candidate> &registry();
uint64_t registry_checksum();
int group_priority(int group, const KeyPod &k, const Problem &p, const DeviceInfo &d);
const char *group_name(int group);
void count_launch(int index, bool tuning);
uint64_t candidate_launches(int index);

// Plan entry: (candidate, group, tier rank, supported, group prio, prio).
struct PlanItem {
  int cand, group, tier, supported, group_prio, prio;
};
std::vector<PlanItem> make_plan(const KeyPod &k, const Problem &p, const DeviceInfo &d);
// The default for a key that is not tuned: the candidates in the order they
// are tried (a shape-class preference, then the plan), and the first of them
// that supports the problem.
std::vector<int> default_order(const KeyPod &k, const Problem &p, const DeviceInfo &d);
int default_candidate(const KeyPod &k, const Problem &p, const DeviceInfo &d);

// Launch one candidate with fault injection and counting applied.
mm_status launch_candidate(int index, const Problem &p, LaunchCtx &ctx);

// ---------------------------------------------------------------- kernels
mm_status launch_naive(const Problem &p, cudaStream_t s);
mm_status launch_l2_flush(void *buf, size_t bytes, cudaStream_t s);
// Pseudo-random values in [-1, 1) of type dtype (offline tuning's operands).
mm_status launch_fill(void *buf, size_t elems, int dtype, unsigned seed, cudaStream_t s);
mm_status launch_empty(cudaStream_t s);
mm_status launch_delay(unsigned long long ns, cudaStream_t s);
mm_status launch_copy_probe(const void *src, void *dst, size_t bytes, cudaStream_t s);
mm_status launch_compare(const void *x, const void *ref, int dtype, int64_t rows, int64_t cols,
                         int64_t ld, int64_t batch, int64_t bstride, double atol, double rtol,
                         int *d_bad, cudaStream_t s);

bool gemv_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why);
mm_status launch_gemv(const Problem &p, LaunchCtx &ctx, int cfg);
int gemv_config_count();
const char *gemv_config_name(int cfg);

bool gemv_fast_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why);
mm_status launch_gemv_fast(const Problem &p, LaunchCtx &ctx, int cfg);
int gemv_fast_config_count();
const char *gemv_fast_config_name(int cfg);
bool gemv_mma_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why);
mm_status launch_gemv_mma(const Problem &p, LaunchCtx &ctx, int cfg);
int gemv_mma_config_count();
const char *gemv_mma_config_name(int cfg);

bool repack_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why);
mm_status launch_repack(const Problem &p, LaunchCtx &ctx, int cfg);
int repack_config_count();
bool repack_config_is_swap(int cfg);  // a small-M (GEMV group) configuration
bool repack_config_is_splitk(int cfg);
const char *repack_config_name(int cfg);

bool tc_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why);
mm_status launch_tc(const Problem &p, LaunchCtx &ctx, int cfg);
// The same configurations on C^T = B^T A^T (operands exchanged, M and N
// swapped, C written transposed): small M becomes the tile's N side.
Problem swap_problem(const Problem &p);
bool tc_swap_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why);
mm_status launch_tc_swapped(const Problem &p, LaunchCtx &ctx, int cfg);
int tc_config_count();
const char *tc_config_name(int cfg);
bool tc_config_is_splitk(int cfg);
int tc_config_index(const char *name);
mm_status launch_tc_splitk_into(const Problem &p, const DeviceInfo &di, int cfg, float *ws,
                                size_t ws_bytes, int *err, cudaStream_t s);

// ---------------------------------------------------------------- tuner
struct ExecResult {
  int candidate = -1;
  bool hit = false;
};
mm_status autotune_execute(const Problem &p, cudaStream_t s, ExecResult *res);
mm_status roofline_peaks(DeviceState &ds, Peaks *out);

// ---------------------------------------------------------------- cache file
mm_status cache_load(DeviceState &ds, const std::string &path);
// Offline tuning (TunableOp's record-untuned / tune-from-file workflow): a key
// missed with tuning off is appended once to a file as "Untuned,<key>,<the
// problem's shape, strides, types and layout>"; tune_file tunes every such
// problem on library-owned synthetic buffers and records the results.
void record_untuned(DeviceState &ds, const KeyPod &key, const Problem &p, const std::string &path);
mm_status tune_file(DeviceState &ds, const std::string &path, int *tuned);
// The miss path: one tuner per key, then the result into the table.
// MM_ERR_PENDING (internal): another thread's tuner of the key did not finish
// within the wait.
constexpr mm_status MM_ERR_PENDING = 100;
// order_after: a stream whose pending work tuning must follow (null: none).
mm_status tune_and_record(DeviceState &ds, const Problem &p, const KeyPod &key, const Options &o,
                          cudaStream_t order_after, TableEntry *out);
// The persistent table, loaded once per device before the first tune.
void sync_table_file(DeviceState &ds, const Options &o);
mm_status cache_save(DeviceState &ds, const std::string &path);
std::string device_file_name(const std::string &path, int ordinal);

// ---------------------------------------------------------------- stats
struct StatsAtomic {
  std::atomic<uint64_t> calls{0}, hits{0}, misses{0}, tunes{0}, launches{0}, bench_launches{0};
  std::atomic<double> last_tune_ms{0.0}, total_tune_ms{0.0};
};
StatsAtomic &stats();

}  // namespace mm
