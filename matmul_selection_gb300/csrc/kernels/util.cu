// Utility kernels of the tuner: L2 flush, probes and the numerical check.
//
// The probes follow the burn "autotune" page, section "roofline and the
// hundred thousand launches": an almost empty kernel whose repeated launches
// measure the launch overhead, and a memory-copy kernel whose throughput is
// the bandwidth peak of the roofline bound.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../common.h"

namespace mm {

namespace {

__global__ void empty_kernel(int *p) {
  pdl_launch_dependents();
  pdl_wait();
  if (p && blockIdx.x == 0 && threadIdx.x == 0) *p = 0;
}

// Grid-stride 16-byte writes over a buffer larger than L2, evicting it.
__global__ void flush_kernel(uint4 *buf, size_t n16, unsigned seed) {
  pdl_launch_dependents();
  pdl_wait();
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n16; i += stride) buf[i] = make_uint4(seed, (unsigned)i, seed, (unsigned)i);
}

// Grid-stride 16-byte copy: the bandwidth probe.
__global__ void copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, size_t n16) {
  pdl_launch_dependents();
  pdl_wait();
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n16; i += stride) dst[i] = src[i];
}

// Fills n elements of type t with values in [-1, 1): element i gets the top
// bits of a 32-bit integer hash of (seed, i) (the lowbias32 mixer), so that
// offline tuning times its candidates on data that toggles like real operands
// (constant data lets the tensor cores run cooler and faster).
__global__ void fill_kernel(void *buf, size_t n, int t, unsigned seed) {
  pdl_launch_dependents();
  pdl_wait();
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (; i < n; i += stride) {
    uint32_t h = (uint32_t)i * 0x9E3779B9u ^ seed ^ (uint32_t)(i >> 32);
    h ^= h >> 16;
    h *= 0x7feb352du;
    h ^= h >> 15;
    h *= 0x846ca68bu;
    h ^= h >> 16;
    const float v = (float)(h >> 8) * (1.0f / 8388608.0f) - 1.0f;
    if (t == MM_F32)
      static_cast<float *>(buf)[i] = v;
    else if (t == MM_BF16)
      static_cast<__nv_bfloat16 *>(buf)[i] = __float2bfloat16_rn(v);
    else
      static_cast<__half *>(buf)[i] = __float2half_rn(v);
  }
}

// Occupies the stream for about `ns` nanoseconds (one thread, bounded by
// %globaltimer), so that work enqueued behind it meanwhile runs back to back.
__global__ void delay_kernel(unsigned long long ns) {
  pdl_launch_dependents();
  pdl_wait();
  unsigned long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  unsigned long long t = t0;
  while (t - t0 < ns) {
    __nanosleep(1000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  }
}

__device__ __forceinline__ float ld_any(const void *p, int64_t i, int t) {
  if (t == MM_F32) return static_cast<const float *>(p)[i];
  if (t == MM_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
  return __half2float(static_cast<const __half *>(p)[i]);
}

// *bad |= |x - ref| > atol + rtol * |ref| over the logical outputs.
__global__ void compare_kernel(const void *x, const void *ref, int t, int64_t rows, int64_t cols,
                               int64_t ld, int64_t batch, int64_t bstride, float atol, float rtol,
                               int *bad) {
  pdl_launch_dependents();
  pdl_wait();
  int64_t total = rows * cols * batch;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    int64_t b = e / (rows * cols), r = (e / cols) % rows, c = e % cols;
    int64_t off = b * bstride + r * ld + c;
    float a = ld_any(x, off, t), q = ld_any(ref, off, t);
    if (!(fabsf(a - q) <= atol + rtol * fabsf(q))) atomicOr(bad, 1);
  }
}

}  // namespace

mm_status launch_empty(cudaStream_t s) {
  cudaError_t e = launch_pdl(empty_kernel, dim3(1), dim3(32), 0, s, dim3(1), (int *)nullptr);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "empty_kernel launch");
}

mm_status launch_delay(unsigned long long ns, cudaStream_t s) {
  if (ns > 10000000ull) ns = 10000000ull;  // never more than 10 ms
  cudaError_t e = launch_pdl(delay_kernel, dim3(1), dim3(1), 0, s, dim3(1), ns);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "delay_kernel launch");
}

mm_status launch_fill(void *buf, size_t elems, int dtype, unsigned seed, cudaStream_t s) {
  if (!elems) return MM_OK;
  cudaError_t e = launch_pdl(fill_kernel, dim3(2048), dim3(256), 0, s, dim3(1), buf, elems, dtype, seed);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "fill_kernel launch");
}

mm_status launch_l2_flush(void *buf, size_t bytes, cudaStream_t s) {
  static unsigned seed = 1;
  size_t n16 = bytes / 16;
  cudaError_t e = launch_pdl(flush_kernel, dim3(1024), dim3(256), 0, s, dim3(1),
                             static_cast<uint4 *>(buf), n16, seed++);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "flush_kernel launch");
}

mm_status launch_copy_probe(const void *src, void *dst, size_t bytes, cudaStream_t s) {
  cudaError_t e = launch_pdl(copy_kernel, dim3(2048), dim3(256), 0, s, dim3(1),
                             static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), bytes / 16);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "copy_kernel launch");
}

mm_status launch_compare(const void *x, const void *ref, int dtype, int64_t rows, int64_t cols,
                         int64_t ld, int64_t batch, int64_t bstride, double atol, double rtol,
                         int *d_bad, cudaStream_t s) {
  cudaError_t e = launch_pdl(compare_kernel, dim3(1024), dim3(256), 0, s, dim3(1), x, ref, dtype,
                             rows, cols, ld, batch, bstride, (float)atol, (float)rtol, d_bad);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "compare_kernel launch");
}

}  // namespace mm
