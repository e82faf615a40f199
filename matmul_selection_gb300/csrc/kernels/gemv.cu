// Bandwidth-bound GEMV group (M <= 16).
//
// The work is streaming B once from HBM; A (<= 16 rows) is staged in shared
// memory as fp32 from any type, layout and alignment (so a misaligned lda,
// which gates every TMA-fed candidate, does not gate these).  Two variants:
//
//   gemv_n  B stored row-major ([K][N], unit stride along n).  A lane owns
//           16 contiguous bytes of a B row (8 bf16/f16 or 4 f32 columns); the
//           8 warps of a block take interleaved rows of the block's k-slice;
//           each thread keeps MT x VEC fp32 accumulators.
//   gemv_t  B stored transposed ([N][K], unit stride along k).  A warp owns
//           R output columns; lanes stride along k with 16-byte loads and the
//           column's dot products are finished with xor-shuffle reductions.
//
// Both split K over blocks so the grid fills the GPU.  Partial sums of a
// split go to an fp32 workspace; the last block to finish a tile (atomic
// ticket) adds the splits in increasing split order and converts to the
// output type, then re-arms the ticket.  Every sum is in a fixed order, so
// results are bit-identical from run to run.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../common.h"

namespace mm {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

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

// 16 bytes of B elements -> VEC floats.
template <int TB>
__device__ __forceinline__ void unpack(const uint4 &v, float *f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (TB == MM_F32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(w[i]);
  } else if constexpr (TB == MM_BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
      float2 x = __half22float2(h);
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
}

// 16-byte load of VEC elements starting at element e of a row of length len;
// elements past len read as zero (scalar loads at the ragged end).
template <int TB>
__device__ __forceinline__ uint4 load_row16(const char *row, int64_t e, int64_t len) {
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int VEC = 16 / EB;
  if (e + VEC <= len) return __ldcs(reinterpret_cast<const uint4 *>(row + e * EB));
  uint32_t w[4] = {0, 0, 0, 0};
  if constexpr (EB == 4) {
    for (int i = 0; i < 4; ++i)
      if (e + i < len) w[i] = reinterpret_cast<const uint32_t *>(row)[e + i];
  } else {
    for (int i = 0; i < 8; ++i)
      if (e + i < len) {
        uint32_t h = reinterpret_cast<const uint16_t *>(row)[e + i];
        w[i / 2] |= (i & 1) ? (h << 16) : h;
      }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

struct GemvArgs {
  const void *A;
  int ta;
  int64_t a_rs, a_cs, sA;
  const char *B;
  int64_t ldb, sB;  // elements
  void *C;
  int tc;
  int64_t ldc, sC;
  int M, N, K;
  int S, KR;  // splits, k-rows per split
  int n_tiles;
  int batch;
  float *ws;
  unsigned *tickets;
};

// Stage A[b][0..MT)[k0..k0+KR) as fp32 (rows >= M and k >= K are zero).
template <int MT>
__device__ __forceinline__ void stage_a(const GemvArgs &g, float *As, int b, int k0) {
  for (int e = threadIdx.x; e < MT * g.KR; e += kThreads) {
    int m = e / g.KR, kk = e - m * g.KR, k = k0 + kk;
    As[e] = (m < g.M && k < g.K) ? ld_elem(g.A, b * g.sA + m * g.a_rs + (int64_t)k * g.a_cs, g.ta)
                                 : 0.f;
  }
}

// After a block wrote its split's partials for outputs [m][col] (col in
// cols[]), the last block of the tile reduces all splits in order.
// Returns through C directly.  part(m, j) gives the partial of this block.
template <int MT>
__device__ void finish_tile(const GemvArgs &g, int b, int tile, int s, int col0, int ncols,
                            float *blockpart /* smem [MT][ncols] */) {
  const int64_t MN = (int64_t)g.M * g.N;
  if (g.S == 1) {
    for (int e = threadIdx.x; e < MT * ncols; e += kThreads) {
      int m = e / ncols, j = e - m * ncols, n = col0 + j;
      if (m < g.M && n < g.N)
        st_elem(g.C, b * g.sC + (int64_t)m * g.ldc + n, g.tc, blockpart[e]);
    }
    return;
  }
  float *ws_s = g.ws + ((int64_t)s * g.batch + b) * MN;
  for (int e = threadIdx.x; e < MT * ncols; e += kThreads) {
    int m = e / ncols, j = e - m * ncols, n = col0 + j;
    if (m < g.M && n < g.N) __stcg(ws_s + (int64_t)m * g.N + n, blockpart[e]);
  }
  // The barrier orders every thread's partial store before thread 0's
  // release; thread 0's acquire in the last block orders the other blocks'
  // partials before this block's loads (the second barrier extends it).
  __syncthreads();
  __shared__ int last;
  if (threadIdx.x == 0) {
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
                 : "=r"(prev)
                 : "l"(&g.tickets[b * g.n_tiles + tile]), "r"(1u)
                 : "memory");
    last = (prev == (unsigned)g.S - 1);
  }
  __syncthreads();
  if (!last) return;
  for (int e = threadIdx.x; e < MT * ncols; e += kThreads) {
    int m = e / ncols, j = e - m * ncols, n = col0 + j;
    if (m < g.M && n < g.N) {
      const float *p = g.ws + (int64_t)b * MN + (int64_t)m * g.N + n;
      const int64_t sstride = (int64_t)g.batch * MN;
      float sum = 0.f;
      for (int t0 = 0; t0 < g.S; t0 += 8) {  // splits in order, 8 loads in flight
        float x[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = t0 + q < g.S ? __ldcg(p + (int64_t)(t0 + q) * sstride) : 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) sum += x[q];
      }
      st_elem(g.C, b * g.sC + (int64_t)m * g.ldc + n, g.tc, sum);
    }
  }
  if (threadIdx.x == 0) g.tickets[b * g.n_tiles + tile] = 0;  // re-arm for the next launch
}

// ---------------------------------------------------------------- gemv_n
template <int MT, int TB>
__global__ void __launch_bounds__(kThreads) gemv_n_kernel(GemvArgs g) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int VEC = 16 / EB;
  constexpr int TN = 32 * VEC;
  constexpr int U = 4;  // rows in flight per warp per step
  extern __shared__ float smem[];
  float *As = smem;                 // [MT][KR]
  float *red = smem + MT * g.KR;    // [max(kWarps, MT)][TN]; later the block's [MT][TN] sums
  const int tile = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k0 = s * g.KR;
  const int kr = min(g.KR, g.K - k0);
  stage_a<MT>(g, As, b, k0);
  __syncthreads();
  const int col = tile * TN + lane * VEC;
  float acc[MT][VEC];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[m][j] = 0.f;
  const char *Bb = g.B + (int64_t)b * g.sB * EB;
  for (int kk = warp; kk < kr; kk += kWarps * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      int k = kk + kWarps * u;
      v[u] = (k < kr && col < g.N)
                 ? load_row16<TB>(Bb + (int64_t)(k0 + k) * g.ldb * EB, col, g.N)
                 : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      int k = kk + kWarps * u;
      if (k < kr) {
        float bf[VEC];
        unpack<TB>(v[u], bf);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          float a = As[m * g.KR + k];
#pragma unroll
          for (int j = 0; j < VEC; ++j) acc[m][j] = fmaf(a, bf[j], acc[m][j]);
        }
      }
    }
  }
  // fixed-order reduction over the warps, one output row at a time
  float mine[MT];  // this thread's output column (threadIdx.x < TN)
  for (int m = 0; m < MT; ++m) {
#pragma unroll
    for (int j = 0; j < VEC; ++j) red[warp * TN + lane * VEC + j] = acc[m][j];
    __syncthreads();
    float sum = 0.f;
    if (threadIdx.x < TN)
      for (int w = 0; w < kWarps; ++w) sum += red[w * TN + threadIdx.x];
    mine[m] = sum;
    __syncthreads();
  }
  if (threadIdx.x < TN)
    for (int m = 0; m < MT; ++m) red[m * TN + threadIdx.x] = mine[m];
  __syncthreads();
  finish_tile<MT>(g, b, tile, s, tile * TN, TN, red);
}

// ---------------------------------------------------------------- gemv_t
template <int MT, int TB, int R>
__global__ void __launch_bounds__(kThreads) gemv_t_kernel(GemvArgs g) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int VEC = 16 / EB;
  constexpr int NB = kWarps * R;  // output columns per block
  extern __shared__ float smem[];
  float *As = smem;               // [MT][KR]
  float *part = smem + MT * g.KR; // [MT][NB]
  const int tile = blockIdx.x, s = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k0 = s * g.KR;
  const int kr = min(g.KR, g.K - k0);
  stage_a<MT>(g, As, b, k0);
  __syncthreads();
  float acc[R][MT];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
  const char *Bb = g.B + (int64_t)b * g.sB * EB;
  const int n0 = tile * NB + warp * R;
  for (int kv = lane * VEC; kv < kr; kv += 32 * VEC * 2) {
    uint4 v[2][R];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        int k = kv + h * 32 * VEC, n = n0 + r;
        v[h][r] = (k < kr && n < g.N)
                      ? load_row16<TB>(Bb + (int64_t)n * g.ldb * EB + (int64_t)k0 * EB, k, kr)
                      : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int k = kv + h * 32 * VEC;
      if (k >= kr) continue;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float bf[VEC];
        unpack<TB>(v[h][r], bf);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float *a = As + m * g.KR + k;
          float t = acc[r][m];
#pragma unroll
          for (int j = 0; j < VEC; ++j) t = fmaf(a[j], bf[j], t);
          acc[r][m] = t;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float t = acc[r][m];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      acc[r][m] = t;
    }
  if (lane == 0)
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) part[m * NB + warp * R + r] = acc[r][m];
  __syncthreads();
  finish_tile<MT>(g, b, tile, s, tile * NB, NB, part);
}

// ---------------------------------------------------------------- host
constexpr int kGemvR = 2;

struct GemvCfg {
  const char *name;
  bool b_trans;
};
const GemvCfg kCfgs[] = {{"gemv_n", false}, {"gemv_t", true}};

int mt_for(int64_t M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16; }

template <int MT, int TB>
void launch_mt(const GemvArgs &g, bool bt, dim3 grid, size_t smem, cudaStream_t s) {
  if (bt)
    launch_pdl(gemv_t_kernel<MT, TB, kGemvR>, grid, dim3(kThreads), smem, s, dim3(1), g);
  else
    launch_pdl(gemv_n_kernel<MT, TB>, grid, dim3(kThreads), smem, s, dim3(1), g);
}

template <int TB>
void launch_tb(const GemvArgs &g, int mt, bool bt, dim3 grid, size_t smem, cudaStream_t s) {
  switch (mt) {
  case 1: launch_mt<1, TB>(g, bt, grid, smem, s); break;
  case 2: launch_mt<2, TB>(g, bt, grid, smem, s); break;
  case 4: launch_mt<4, TB>(g, bt, grid, smem, s); break;
  case 8: launch_mt<8, TB>(g, bt, grid, smem, s); break;
  default: launch_mt<16, TB>(g, bt, grid, smem, s); break;
  }
}

template <int MT, int TB>
void set_smem_attr(size_t smem) {
  cudaFuncSetAttribute(gemv_n_kernel<MT, TB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaFuncSetAttribute(gemv_t_kernel<MT, TB, kGemvR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)smem);
}

template <int TB>
void set_attr_tb(int mt, size_t smem) {
  switch (mt) {
  case 1: set_smem_attr<1, TB>(smem); break;
  case 2: set_smem_attr<2, TB>(smem); break;
  case 4: set_smem_attr<4, TB>(smem); break;
  case 8: set_smem_attr<8, TB>(smem); break;
  default: set_smem_attr<16, TB>(smem); break;
  }
}

// Split plan: k-rows per split and split count, aiming at ~2 blocks per SM.
void plan_splits(int64_t K, int64_t tiles, int sms, int kr_align, int kr_max, int *KR, int *S) {
  int64_t want_blocks = 2LL * sms;
  int64_t s = (want_blocks + tiles - 1) / tiles;
  if (s < 1) s = 1;
  int64_t kr = (K + s - 1) / s;
  if (kr < 64) kr = 64;
  kr = (kr + kr_align - 1) / kr_align * kr_align;
  if (kr > kr_max) kr = kr_max;
  if (kr > K) kr = (K + kr_align - 1) / kr_align * kr_align;
  *KR = (int)kr;
  *S = (int)((K + kr - 1) / kr);
}

}  // namespace

int gemv_config_count() { return (int)(sizeof kCfgs / sizeof kCfgs[0]); }
const char *gemv_config_name(int cfg) { return kCfgs[cfg].name; }

bool gemv_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why) {
  const GemvCfg &c = kCfgs[cfg];
  auto no = [&](const char *w) {
    if (why) *why = w;
    return false;
  };
  if (p.bt != c.b_trans) return no("B layout does not match this variant");
  if (p.M < 1 || p.M > 16) return no("M must be in [1, 16]");
  if (p.K < 1) return no("K must be >= 1");
  if (p.N > (1LL << 30) || p.K > (1LL << 30)) return no("N or K too large");
  if (p.batch > 65535) return no("batch too large");
  int eb = dtype_bytes(p.tb);
  if (((uintptr_t)p.B) % 16) return no("B not 16-byte aligned");
  if ((p.ldb * eb) % 16) return no("ldb not a multiple of 16 bytes");
  if (p.batch > 1 && (p.sB * eb) % 16) return no("B batch stride not a multiple of 16 bytes");
  (void)d;
  return true;
}

mm_status launch_gemv(const Problem &p, LaunchCtx &ctx, int cfg) {
  const GemvCfg &c = kCfgs[cfg];
  const int eb = dtype_bytes(p.tb), vec = 16 / eb;
  const int mt = mt_for(p.M);
  GemvArgs g;
  g.A = p.A;
  g.ta = p.ta;
  g.a_rs = p.at ? 1 : p.lda;
  g.a_cs = p.at ? p.lda : 1;
  g.sA = p.sA;
  g.B = static_cast<const char *>(p.B);
  g.ldb = p.ldb;
  g.sB = p.sB;
  g.C = p.C;
  g.tc = p.tc;
  g.ldc = p.ldc;
  g.sC = p.sC;
  g.M = (int)p.M;
  g.N = (int)p.N;
  g.K = (int)p.K;
  g.batch = (int)p.batch;
  int sms = ctx.dev->info.sms;
  int tiles;
  size_t smem;
  if (!c.b_trans) {
    const int TN = 32 * vec;
    tiles = (int)((p.N + TN - 1) / TN);
    plan_splits(p.K, (int64_t)tiles * p.batch, sms, 8, 1024, &g.KR, &g.S);
    smem = ((size_t)mt * g.KR + (size_t)(mt > kWarps ? mt : kWarps) * TN) * sizeof(float);
  } else {
    const int NB = kWarps * kGemvR;
    tiles = (int)((p.N + NB - 1) / NB);
    plan_splits(p.K, (int64_t)tiles * p.batch, sms, 32 * vec * 2, 2048, &g.KR, &g.S);
    smem = ((size_t)mt * g.KR + (size_t)mt * NB) * sizeof(float);
  }
  g.n_tiles = tiles;
  g.ws = nullptr;
  g.tickets = nullptr;
  if (g.S > 1) {
    size_t tickets_bytes = (size_t)tiles * p.batch * sizeof(unsigned);
    size_t ws_bytes = (size_t)g.S * p.batch * p.M * p.N * sizeof(float);
    void *t = nullptr, *w = nullptr;
    mm_status st = get_scratch(*ctx.dev, ctx.stream, SCRATCH_TICKETS, tickets_bytes, &t);
    if (st != MM_OK) return st;
    st = get_scratch(*ctx.dev, ctx.stream, SCRATCH_WORKSPACE, ws_bytes, &w);
    if (st != MM_OK) return st;
    g.tickets = static_cast<unsigned *>(t);
    g.ws = static_cast<float *>(w);
  }
  if (smem > 48 * 1024) {
    if (p.tb == MM_BF16) set_attr_tb<MM_BF16>(mt, smem);
    else if (p.tb == MM_F16) set_attr_tb<MM_F16>(mt, smem);
    else set_attr_tb<MM_F32>(mt, smem);
  }
  dim3 grid((unsigned)tiles, (unsigned)g.S, (unsigned)p.batch);
  if (p.tb == MM_BF16) launch_tb<MM_BF16>(g, mt, c.b_trans, grid, smem, ctx.stream);
  else if (p.tb == MM_F16) launch_tb<MM_F16>(g, mt, c.b_trans, grid, smem, ctx.stream);
  else launch_tb<MM_F32>(g, mt, c.b_trans, grid, smem, ctx.stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "gemv kernel launch");
  return MM_OK;
}

}  // namespace mm
