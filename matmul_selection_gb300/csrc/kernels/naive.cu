// The always-valid default candidate: one thread per output element.
//
// The burn "autotune" page registers a naive matmul as the first candidate
// because it "should always work": it is the plan's last resort when every
// other candidate is demoted or fails, and TunableOp's Default when tuning is
// off.  It reads both operands through arbitrary strides (any layout, any
// alignment, any batch strides), accumulates in fp32 with FMA in increasing
// k, and rounds to the output type to nearest-even.  K = 0 writes zeros.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../common.h"

namespace mm {

namespace {

__device__ __forceinline__ float ld_elem(const void *p, int64_t i, int t) {
  if (t == MM_F32) return static_cast<const float *>(p)[i];
  if (t == MM_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
  return __half2float(static_cast<const __half *>(p)[i]);
}

__device__ __forceinline__ void st_elem(void *p, int64_t i, int t, float v) {
  if (t == MM_F32)
    static_cast<float *>(p)[i] = v;
  else if (t == MM_BF16)
    static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
  else
    static_cast<__half *>(p)[i] = __float2half_rn(v);
}

template <int TA, int TB>
__global__ void naive_kernel(const void *__restrict__ A, const void *__restrict__ B,
                             void *__restrict__ C, int tc, int64_t M, int64_t N, int64_t K,
                             int64_t a_rs, int64_t a_cs, int64_t a_bs, int64_t b_rs,
                             int64_t b_cs, int64_t b_bs, int64_t ldc, int64_t c_bs,
                             int64_t batch) {
  pdl_launch_dependents();
  pdl_wait();
  int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= N) return;
  for (int64_t b = blockIdx.z; b < batch; b += gridDim.z) {
    for (int64_t i = (int64_t)blockIdx.y * blockDim.y + threadIdx.y; i < M;
         i += (int64_t)gridDim.y * blockDim.y) {
      const int64_t abase = b * a_bs + i * a_rs;
      const int64_t bbase = b * b_bs + j * b_cs;
      float acc = 0.f;
      for (int64_t k = 0; k < K; ++k)
        acc = fmaf(ld_elem(A, abase + k * a_cs, TA), ld_elem(B, bbase + k * b_rs, TB), acc);
      st_elem(C, b * c_bs + i * ldc + j, tc, acc);
    }
  }
}

template <int TA, int TB>
void launch_t(const Problem &p, cudaStream_t s, dim3 grid, dim3 block) {
  int64_t a_rs = p.at ? 1 : p.lda, a_cs = p.at ? p.lda : 1;
  int64_t b_rs = p.bt ? 1 : p.ldb, b_cs = p.bt ? p.ldb : 1;
  launch_pdl(naive_kernel<TA, TB>, grid, block, 0, s, dim3(1), p.A, p.B, p.C, p.tc, p.M, p.N, p.K,
             a_rs, a_cs, p.sA, b_rs, b_cs, p.sB, p.ldc, p.sC, p.batch);
}

}  // namespace

mm_status launch_naive(const Problem &p, cudaStream_t s) {
  if (p.M == 0 || p.N == 0 || p.batch == 0) return MM_OK;
  dim3 block(32, 8);
  int64_t gx = (p.N + 31) / 32;
  if (gx > 2147483647) return set_error(MM_ERR_UNSUPPORTED, "naive: N too large");
  int64_t gy = (p.M + 7) / 8;
  if (gy > 65535) gy = 65535;
  int64_t gz = p.batch > 65535 ? 65535 : p.batch;
  dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)gz);
#define MM_NAIVE_CASE(a, b) \
  if (p.ta == a && p.tb == b) launch_t<a, b>(p, s, grid, block);
  MM_NAIVE_CASE(MM_BF16, MM_BF16)
  else MM_NAIVE_CASE(MM_F16, MM_F16)
  else MM_NAIVE_CASE(MM_F32, MM_F32)
  else MM_NAIVE_CASE(MM_BF16, MM_F16)
  else MM_NAIVE_CASE(MM_BF16, MM_F32)
  else MM_NAIVE_CASE(MM_F16, MM_BF16)
  else MM_NAIVE_CASE(MM_F16, MM_F32)
  else MM_NAIVE_CASE(MM_F32, MM_BF16)
  else MM_NAIVE_CASE(MM_F32, MM_F16)
#undef MM_NAIVE_CASE
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "naive_kernel launch");
  return MM_OK;
}

}  // namespace mm
