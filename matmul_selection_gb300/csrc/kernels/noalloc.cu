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
// holds the fp32 partial sums of the K slices (and, in its last 256 bytes,
// the kernel's error word).  Host code cannot use the array's name as a
// device address -- on the host it only names a stand-in object -- so the
// device address is obtained once per device with cudaGetSymbolAddress and
// cached.  That set-up happens on the first call on each device, with that
// device current; make the first call before any stream capture.
//
// Every call shares the one array and it keeps the last call's contents:
// the error word is cleared at the start of each call (the partials need no
// clearing: each call overwrites every element it later reads).  Calls whose
// GPU execution overlaps -- on two streams, or from two host threads --
// race on the array and corrupt each other's results; the caller must order
// them.
#include <mutex>

#include "../common.h"

namespace {
constexpr size_t kScratchBytes = 16u << 20;
constexpr size_t kErrBytes = 256;  // error word area at the end
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace mm {

namespace {

constexpr int kMaxDevices = 64;

struct StaticSetup {
  std::once_flag once;
  cudaError_t status = cudaSuccess;
  void *ptr = nullptr;
  DeviceInfo info;
};
StaticSetup g_setup[kMaxDevices];

// Resolve the array's device address and the device's properties, once per
// device.  Queries only: nothing here allocates.
mm_status setup_device(int dev, StaticSetup **out) {
  if (dev < 0 || dev >= kMaxDevices) return set_error(MM_ERR_INVALID_ARG, "device ordinal %d", dev);
  StaticSetup &st = g_setup[dev];
  std::call_once(st.once, [&] {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e == cudaSuccess) {
      int sms = 0, maj = 0, min = 0, smem = 0;
      e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev);
      if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
      st.info.ordinal = dev;
      st.info.sms = sms;
      st.info.cc_major = maj;
      st.info.cc_minor = min;
      st.info.smem_optin = smem;
    }
    st.status = e;
    st.ptr = p;
  });
  if (st.status != cudaSuccess) return cuda_error(st.status, "cudaGetSymbolAddress (static workspace)");
  *out = &st;
  return MM_OK;
}

}  // namespace

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
  if (need2 > kScratchBytes - kErrBytes)
    return set_error(MM_ERR_INVALID_ARG,
                     "M x N = %lld x %lld needs %zu bytes for two K slices; the fixed workspace "
                     "holds %zu bytes (M*N <= %zu)",
                     (long long)M, (long long)N, need2, kScratchBytes - kErrBytes,
                     (kScratchBytes - kErrBytes) / (2 * sizeof(float)));
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  StaticSetup *su = nullptr;
  if ((st = setup_device(dev, &su)) != MM_OK) return st;
  const int cfg = tc_config_index("tc_splitk_128x128_s6");
  if (cfg < 0) return set_error(MM_ERR_UNSUPPORTED, "split-K configuration missing");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *base = static_cast<char *>(su->ptr);
  int *err = reinterpret_cast<int *>(base + kScratchBytes - kErrBytes);
  e = cudaMemsetAsync(err, 0, sizeof(int), s);
  if (e != cudaSuccess) return cuda_error(e, "cudaMemsetAsync (error word)");
  return launch_tc_splitk_into(p, su->info, cfg, reinterpret_cast<float *>(base),
                               kScratchBytes - kErrBytes, err, s);
}
