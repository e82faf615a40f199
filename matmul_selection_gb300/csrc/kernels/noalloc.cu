// Split-K tensor-core GEMM that allocates nothing.
//
// Who needs it: callers that must not call cudaMalloc/cudaFree, for example
// a serving process that reserves all device memory for its own pool at
// start-up and treats any later allocation as an error, a plugin running
// inside a host framework that owns the device allocator, or a latency-bound
// loop that cannot afford the implicit device synchronisation cudaMalloc and
// cudaFree may perform.  The regular entry points allocate their split-K
// workspace on first use; this one uses a fixed workspace compiled into the
// library instead.
//
// The workspace is a file-scope __device__ array of kScratchBytes (16 MiB),
// present on every GPU that loads the library until the process exits.  It
// holds the fp32 partial sums of the K slices and, in its last 256 bytes, the
// kernels' error word.  Host code cannot use the array's name as a device
// address -- on the host it only names a stand-in object -- so the device
// address is obtained with cudaGetSymbolAddress, with the device current, on
// the first call on each device, and kept until mm_shutdown (which forgets it,
// so a call after a device reset resolves it again).  Make the first call on
// a device before any stream capture.
//
// Every call shares the one array and it keeps the last call's contents.  The
// partials need no clearing: each call overwrites every element it later
// reads.  The error word starts at zero (static storage) and is cleared only
// by mm_splitk_gemm_noalloc_status, so that query reports a bounded wait that
// gave up in any call since the previous query.  Calls whose GPU execution
// overlaps -- on two streams, or from two host threads -- race on the array
// and corrupt each other's results; the caller must order them.
#include <mutex>

#include "../common.h"

namespace {
constexpr size_t kScratchBytes = 16u << 20;
constexpr size_t kErrBytes = 256;  // error word area at the end
constexpr size_t kPartialBytes = kScratchBytes - kErrBytes;
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace mm {

namespace {

constexpr int kMaxDevices = 64;

struct StaticSetup {
  bool ready = false;
  void *ptr = nullptr;
  DeviceInfo info;
};
std::mutex g_setup_mu;
StaticSetup g_setup[kMaxDevices];

// Resolve the array's device address and the device's properties, once per
// device until forgotten.  Queries only: nothing here allocates.
mm_status setup_device(int dev, StaticSetup *out) {
  if (dev < 0 || dev >= kMaxDevices) return set_error(MM_ERR_INVALID_ARG, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lk(g_setup_mu);
  StaticSetup &st = g_setup[dev];
  if (!st.ready) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress (static workspace)");
    int v[4] = {0, 0, 0, 0};
    const cudaDeviceAttr attrs[4] = {cudaDevAttrMultiProcessorCount, cudaDevAttrComputeCapabilityMajor,
                                     cudaDevAttrComputeCapabilityMinor,
                                     cudaDevAttrMaxSharedMemoryPerBlockOptin};
    for (int i = 0; i < 4; ++i) {
      e = cudaDeviceGetAttribute(&v[i], attrs[i], dev);
      if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute");
    }
    st.info.ordinal = dev;
    st.info.sms = v[0];
    st.info.cc_major = v[1];
    st.info.cc_minor = v[2];
    st.info.smem_optin = v[3];
    st.ptr = p;
    st.ready = true;
  }
  *out = st;
  return MM_OK;
}

mm_status current_setup(StaticSetup *out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  return setup_device(dev, out);
}

int *error_word(const StaticSetup &su) {
  return reinterpret_cast<int *>(static_cast<char *>(su.ptr) + kPartialBytes);
}

}  // namespace

void noalloc_forget_devices() {
  std::lock_guard<std::mutex> lk(g_setup_mu);
  for (auto &st : g_setup) st = StaticSetup();
}

}  // namespace mm

using namespace mm;

extern "C" mm_status mm_splitk_gemm_noalloc(const void *lhs, const void *rhs, void *out, int64_t M,
                                            int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                            int64_t ldc, mm_dtypes dt, mm_layout layout,
                                            void *stream) {
  Problem p;
  mm_status st = make_problem(&p, lhs, rhs, out, M, N, K, lda, ldb, ldc, dt, layout, nullptr);
  if (st != MM_OK) return st;
  if (M == 0 || N == 0) return MM_OK;
  if (K == 0) return set_error(MM_ERR_INVALID_ARG, "K must be >= 1 (nothing to split)");
  const size_t need2 = 2 * (size_t)M * (size_t)N * sizeof(float);
  if (need2 > kPartialBytes)
    return set_error(MM_ERR_INVALID_ARG,
                     "M x N = %lld x %lld needs %zu bytes for two K slices; the fixed workspace "
                     "holds %zu bytes (M*N <= %zu)",
                     (long long)M, (long long)N, need2, kPartialBytes,
                     kPartialBytes / (2 * sizeof(float)));
  StaticSetup su;
  if ((st = current_setup(&su)) != MM_OK) return st;
  const int cfg = tc_config_index("tc_splitk_128x128_s7");
  if (cfg < 0) return set_error(MM_ERR_UNSUPPORTED, "split-K configuration missing");
  return launch_tc_splitk_into(p, su.info, cfg, static_cast<float *>(su.ptr), kPartialBytes,
                               error_word(su), static_cast<cudaStream_t>(stream));
}

extern "C" mm_status mm_splitk_gemm_noalloc_status(void *stream) {
  StaticSetup su;
  mm_status st = current_setup(&su);
  if (st != MM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
  int code = 0;
  e = cudaMemcpy(&code, error_word(su), sizeof code, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_error(e, "cudaMemcpy (error word)");
  if (code == 0) return MM_OK;
  e = cudaMemset(error_word(su), 0, sizeof(int));
  if (e != cudaSuccess) return cuda_error(e, "cudaMemset (clear the error word)");
  return set_error(MM_ERR_TIMEOUT,
                   "a split-K kernel's bounded wait gave up (code 0x%x); the products of the "
                   "calls since the previous status query may be wrong",
                   code);
}
