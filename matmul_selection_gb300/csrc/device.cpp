// Per-device state: properties, error word, private tuning stream, scratch.
#include <cudaTypedefs.h>

#include <cstdio>

#include "common.h"

namespace mm {

namespace {
std::mutex g_dev_mu;
std::map<int, std::unique_ptr<DeviceState>> g_devs;

std::string uuid_string(const cudaUUID_t &u) {
  const unsigned char *b = reinterpret_cast<const unsigned char *>(u.bytes);
  char s[64];
  snprintf(s, sizeof s,
           "GPU-%02x%02x%02x%02x-%02x%02x-%02x%02x-%02x%02x-%02x%02x%02x%02x%02x%02x", b[0], b[1],
           b[2], b[3], b[4], b[5], b[6], b[7], b[8], b[9], b[10], b[11], b[12], b[13], b[14], b[15]);
  return s;
}
}  // namespace

mm_status DevBuf::ensure(size_t need) {
  if (ptr && bytes >= need) return MM_OK;
  release();
  size_t sz = (need + (2u << 20) - 1) & ~(size_t)((2u << 20) - 1);
  if (sz == 0) sz = 2u << 20;
  cudaError_t e = cudaMalloc(&ptr, sz);
  if (e != cudaSuccess) {
    ptr = nullptr;
    return cuda_error(e, "cudaMalloc (library scratch)");
  }
  bytes = sz;
  return MM_OK;
}

void DevBuf::release() {
  if (ptr) cudaFree(ptr);
  ptr = nullptr;
  bytes = 0;
}

mm_status current_device(DeviceState **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  auto it = g_devs.find(dev);
  if (it != g_devs.end()) {
    *out = it->second.get();
    return MM_OK;
  }
  auto ds = std::make_unique<DeviceState>();
  cudaDeviceProp prop;
  MM_CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
  ds->info.ordinal = dev;
  ds->info.sms = prop.multiProcessorCount;
  ds->info.cc_major = prop.major;
  ds->info.cc_minor = prop.minor;
  ds->info.l2_bytes = prop.l2CacheSize;
  ds->info.smem_optin = (int64_t)prop.sharedMemPerBlockOptin;
  ds->info.total_mem = (int64_t)prop.totalGlobalMem;
  ds->info.name = prop.name;
  ds->info.uuid = uuid_string(prop.uuid);
  MM_CUDA_TRY(cudaMalloc(&ds->d_err, 64));
  MM_CUDA_TRY(cudaMemset(ds->d_err, 0, 64));
  MM_CUDA_TRY(cudaStreamCreateWithFlags(&ds->tune_stream, cudaStreamNonBlocking));
  MM_CUDA_TRY(cudaEventCreateWithFlags(&ds->ev_order, cudaEventDisableTiming));
  *out = ds.get();
  g_devs[dev] = std::move(ds);
  return MM_OK;
}

void for_each_device(void (*fn)(DeviceState &)) {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  for (auto &kv : g_devs) fn(*kv.second);
}

void release_all_devices() {
  std::lock_guard<std::mutex> lk(g_dev_mu);
  int cur = -1;
  cudaGetDevice(&cur);
  for (auto &kv : g_devs) {
    DeviceState &ds = *kv.second;
    cudaSetDevice(ds.info.ordinal);
    cudaDeviceSynchronize();
    for (auto &s : ds.scratch) s.second.release();
    ds.flush_buf.release();
    ds.stage_a.release();
    ds.stage_b.release();
    ds.stage_c.release();
    if (ds.d_err) cudaFree(ds.d_err);
    if (ds.tune_stream) cudaStreamDestroy(ds.tune_stream);
    if (ds.ev_order) cudaEventDestroy(ds.ev_order);
  }
  g_devs.clear();
  if (cur >= 0) cudaSetDevice(cur);
}

mm_status get_scratch(DeviceState &ds, cudaStream_t s, int slot, size_t bytes, void **out) {
  std::lock_guard<std::mutex> lk(ds.scratch_mu);
  DevBuf &b = ds.scratch[std::make_pair(s, slot)];
  if (!b.ptr || b.bytes < bytes) {
    // Nothing can be allocated while the stream is being captured into a
    // graph (the allocation would end the capture): the candidate declines
    // and the caller moves on to one that needs no new scratch.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) == cudaSuccess && cap != cudaStreamCaptureStatusNone)
      return set_error(MM_ERR_UNSUPPORTED,
                       "scratch of %zu bytes not allocated on this stream before the capture",
                       bytes);
    // The old buffer may still be read by queued work on this stream.
    if (b.ptr) {
      cudaError_t e = cudaStreamSynchronize(s);
      if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize (scratch growth)");
    }
    mm_status st = b.ensure(bytes);
    if (st != MM_OK) return st;
    // counters used by single-pass reductions must start at zero
    cudaError_t e = cudaMemsetAsync(b.ptr, 0, b.bytes, s);
    if (e != cudaSuccess) return cuda_error(e, "cudaMemsetAsync (scratch)");
  }
  *out = b.ptr;
  return MM_OK;
}

mm_status encode_prefetch_map(CUtensorMap *map, int dtype, const void *base, uint64_t inner,
                              uint64_t outer, uint64_t batch, uint64_t ld_bytes,
                              uint64_t bstride_bytes, uint32_t box_inner, uint32_t box_outer) {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  if (!fn) return set_error(MM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  if (batch <= 1) bstride_bytes = ((ld_bytes * outer) + 15) & ~(uint64_t)15;
  const CUtensorMapDataType t = dtype == MM_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                : dtype == MM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cuuint64_t dims[3] = {inner, outer, batch < 1 ? 1 : batch};
  cuuint64_t strides[2] = {ld_bytes, bstride_bytes};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, t, 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(MM_ERR_CUDA, "cuTensorMapEncodeTiled (prefetch map) failed (%d)", (int)r);
  return MM_OK;
}

}  // namespace mm
