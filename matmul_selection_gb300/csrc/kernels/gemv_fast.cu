// Latency-lean GEMV candidates for small M.
//
// At M <= 8 the product is a single pass over B (33.5 MB for 4096 x 4096
// bf16); on this part a bare 33.5 MB read already costs ~8 us per launch, so
// these kernels are built to add as little as possible to it:
//   * every thread issues its loads of B before anything else (A staging and
//     all synchronisation happen while those loads are in flight);
//   * A is staged with batched loads (all issued, then stored);
//   * no second kernel and no serial tail.
//
//   gemv_n_cluster  B row-major [K][N].  A cluster of 8 CTAs shares one group
//       of CW columns (256 bytes of every row); CTA rank s handles the K rows
//       [s*KS, (s+1)*KS).  In a CTA, 16 lanes cover a row segment with 16-byte
//       loads (2 rows per warp instruction, 32 rows per step).  Partials are
//       summed in a fixed order: the two rows of a warp by shuffle, the 16 warps
//       through shared memory, then the 8 CTAs through distributed shared
//       memory, rank 0..7 in order, each rank finishing CW/8 of the columns.
//   gemv_n_stream  M = 1, B row-major [K][N], no clusters.  About two CTAs an
//       SM: G column groups of 512 bytes x S splits of K, CTA (g, s) streaming
//       the group's row segments over the rows [s*K/S, (s+1)*K/S).  Before the
//       grid waits for its predecessor, each CTA prefetches its row segments
//       into L2 (cp.async.bulk.prefetch.L2): a prefetch returns nothing to the
//       SM, so it cannot observe a stale value (the loads after the wait read
//       the coherent L2), and back-to-back launches keep HBM busy across the
//       kernel boundary.  A clustered grid cannot start early this way (a
//       cluster needs its GPC's slots free at once), and a second kernel adds a
//       grid boundary, so the split sums go to an fp32 workspace and the CTA of
//       the group that arrives last (atomic ticket) adds them in split order,
//       all its loads of them in flight at once.
//   gemv_t_rows  B transposed [N][K].  One warp per output column (row of B)
//       reading the whole row with 16-byte loads; the dot products end in an
//       xor-shuffle reduction.  No cross-warp or cross-CTA combination.  The
//       rows are prefetched into L2 before the wait, as above.  A is staged
//       in shared memory in an order that keeps the lanes' reads of it free
//       of bank conflicts.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>
#include <type_traits>

#include "../common.h"

namespace mm {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCluster = 8;

__device__ __forceinline__ float ld_any(const void *p, int64_t i, int t) {
  if (t == MM_F32) return static_cast<const float *>(p)[i];
  if (t == MM_BF16) return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
  return __half2float(static_cast<const __half *>(p)[i]);
}
__device__ __forceinline__ void st_any(void *p, int64_t i, int t, float v) {
  if (t == MM_F32)
    static_cast<float *>(p)[i] = v;
  else if (t == MM_BF16)
    static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
  else
    static_cast<__half *>(p)[i] = __float2half_rn(v);
}

// 16 bytes of B -> VEC floats.
template <int TB>
__device__ __forceinline__ void unpack16(const uint4 &q, float *f) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
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
      float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
  }
}

// 16-byte load of elements [e, e+VEC) of a row of length len (zeros past it).
template <int TB>
__device__ __forceinline__ uint4 load16(const char *row, int64_t e, int64_t len) {
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int VEC = 16 / EB;
  if (e + VEC <= len) return __ldcs(reinterpret_cast<const uint4 *>(row + e * EB));
  uint32_t w[4] = {0, 0, 0, 0};
  if (e < len) {
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
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

struct FastArgs {
  const void *A;
  int ta;
  int64_t a_rs, a_cs, sA;
  const char *B;
  int64_t ldb, sB;
  void *C;
  int tc;
  int64_t ldc, sC;
  int M, N, K, batch;
  int KS;  // gemv_n_cluster: rows per cluster rank
  // gemv_n_stream
  int G, S;           // column groups, K splits
  float *ws;          // [batch][G][S][CW] split sums
  unsigned *tickets;  // [batch][G] arrival counters, zero between calls
};

// Atomic add with release and acquire semantics at device scope.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Warm L2 with `bytes` (a multiple of 16) at a 16-byte aligned address.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Stage n_elems elements of A (index -> (m, k) by `map`) into smem as fp32,
// loads batched 8 at a time so their latencies overlap.
template <typename Map>
__device__ __forceinline__ void stage_batched(const FastArgs &g, float *dst, int n_elems, Map map) {
  for (int base = threadIdx.x; base < n_elems; base += kThreads * 8) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = base + u * kThreads;
      int64_t off;
      bool ok = e < n_elems && map(e, &off);
      v[u] = ok ? ld_any(g.A, off, g.ta) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = base + u * kThreads;
      if (e < n_elems) dst[e] = v[u];
    }
  }
}

// ---------------------------------------------------------------- gemv_n_cluster
template <int MT, int TB>
__global__ void __launch_bounds__(kThreads, MT == 1 ? 2 : 1) gemv_n_cluster_kernel(const FastArgs g) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int VEC = 16 / EB;
  constexpr int CW = 256 / EB;          // columns per group: 256 bytes of a row
  constexpr int LPR = CW / VEC;         // 16 lanes per row segment
  constexpr int RPW = 32 / LPR;         // 2 rows per warp instruction
  constexpr int STEP = kWarps * RPW;    // 32 rows per step
  constexpr int U = 8;                  // loads in flight per lane
  constexpr int CPR = CW / kCluster;    // columns each rank finishes
  constexpr int APT = MT;               // A elements a thread preloads (slices of <= 512 rows)
  extern __shared__ float fsm[];
  float *As = fsm;                              // [KS][MT]
  float *part = fsm + g.KS * MT;                // [warps][MT][CW], slot 0 ends as the CTA sum
  const int grp = blockIdx.x, b = blockIdx.z;
  uint32_t rank;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
  const int k0 = (int)rank * g.KS;
  const int kr = max(0, min(g.KS, g.K - k0));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sub = lane / LPR, li = lane % LPR;
  const int col = grp * CW + li * VEC;
  const char *Bb = g.B + (int64_t)b * g.sB * EB;
  // this thread's elements of A's slice: issued first, stored after B's loads
  const int na = g.KS * MT;
  float areg[APT];
#pragma unroll
  for (int u = 0; u < APT; ++u) {
    const int e = threadIdx.x + u * kThreads;
    const int kk = e / MT, m = e - kk * MT;
    areg[u] = (e < na && m < g.M && kk < kr)
                  ? ld_any(g.A, (int64_t)b * g.sA + (int64_t)m * g.a_rs + (int64_t)(k0 + kk) * g.a_cs,
                           g.ta)
                  : 0.f;
  }
  float acc[MT][VEC];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[m][j] = 0.f;
  bool staged = false;
  for (int r0 = warp * RPW + sub; r0 < g.KS; r0 += STEP * U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = r0 + u * STEP;
      v[u] = (r < kr) ? load16<TB>(Bb + (int64_t)(k0 + r) * g.ldb * EB, col, g.N)
                      : make_uint4(0, 0, 0, 0);
    }
    if (!staged) {  // B's first loads are in flight; now publish A's slice
#pragma unroll
      for (int u = 0; u < APT; ++u) {
        const int e = threadIdx.x + u * kThreads;
        if (e < na) As[e] = areg[u];
      }
      for (int e = threadIdx.x + APT * kThreads; e < na; e += kThreads) {  // slices > 512 rows
        const int kk = e / MT, m = e - kk * MT;
        As[e] = (m < g.M && kk < kr) ? ld_any(g.A, (int64_t)b * g.sA + (int64_t)m * g.a_rs +
                                                       (int64_t)(k0 + kk) * g.a_cs, g.ta)
                                     : 0.f;
      }
      __syncthreads();
      staged = true;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int r = r0 + u * STEP;
      if (r < kr) {
        float bf[VEC];
        unpack16<TB>(v[u], bf);
        const float *a = As + r * MT;
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
          for (int j = 0; j < VEC; ++j) acc[m][j] = fmaf(a[m], bf[j], acc[m][j]);
      }
    }
  }
  // rows of a warp: fixed-order xor shuffle over the RPW row lanes
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int j = 0; j < VEC; ++j) {
      float x = acc[m][j];
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      acc[m][j] = x;
    }
  if (sub == 0)
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
      for (int j = 0; j < VEC; ++j) part[(warp * MT + m) * CW + li * VEC + j] = acc[m][j];
  __syncthreads();
  // the CTA's sum over warps 0..15 in order, into slot 0
  float cta[2];
  int ncta = 0;
  for (int e = threadIdx.x; e < MT * CW; e += kThreads) {
    float t = 0.f;
    for (int w = 0; w < kWarps; ++w) t += part[w * MT * CW + e];
    cta[ncta++] = t;
  }
  __syncthreads();
  ncta = 0;
  for (int e = threadIdx.x; e < MT * CW; e += kThreads) part[e] = cta[ncta++];
  // all ranks' sums visible cluster-wide
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
  const uint32_t part_addr = (uint32_t)__cvta_generic_to_shared(part);
  for (int e = threadIdx.x; e < MT * CPR; e += kThreads) {
    const int m = e / CPR, c = (int)rank * CPR + (e - m * CPR);
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < kCluster; ++q) {
      uint32_t ra;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                   : "=r"(ra)
                   : "r"(part_addr + (uint32_t)((m * CW + c) * 4)), "r"(q));
      float x;
      asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(x) : "r"(ra) : "memory");
      t += x;
    }
    const int n = grp * CW + c;
    if (m < g.M && n < g.N) st_any(g.C, (int64_t)b * g.sC + (int64_t)m * g.ldc + n, g.tc, t);
  }
  // keep this CTA's shared memory alive until every rank has read it
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// ---------------------------------------------------------------- gemv_n_stream
// A CTA of 512 threads streams the 512-byte row segments of its column group
// over its K rows, a warp per row.  When the rows of a split fit in at most
// four steps of kStreamFixedU rows a warp, the step count is a template
// argument and the loop is unrolled completely, with eight 16-byte loads in
// flight a lane: straight-line code whose loads the compiler can issue ahead
// of the previous step's arithmetic (4096 x 4096 bf16: 6.8 us a call against
// 7.2 us for the rolled loop with four loads in flight, measured back to
// back).  Deeper splits take the rolled loop.  The S partial sums of a group
// are combined by whichever of its CTAs finishes last (an atomic ticket), in
// split order, so the call is a single grid with no second kernel and no
// serial tail of dependent loads.
constexpr int kStreamThreads = 512;
constexpr int kStreamU = 4;       // loads in flight a lane, rolled loop
constexpr int kStreamFixedU = 8;  // loads in flight a lane, unrolled steps
constexpr int kStreamMaxSteps = 4;
constexpr int kStreamSegB = 512;  // bytes of a row segment (one warp, 16 bytes a lane)
constexpr int kStreamCombineMax = 24;  // splits one thread a column adds in the combine

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

// U rows a warp (one 16-byte load a lane each, all in flight): the split's
// rows r0, r0 + RPS, ..., those at or past kr contributing nothing.  Bc points
// at this lane's 16-byte piece of the split's first row (see stream_rows for
// lanes past N), x at the split's first element of A.
template <int TB, typename TAe, int U>
__device__ __forceinline__ void stream_step(const char *Bc, int64_t pitch, const TAe *x, int acs,
                                            int r0, int kr, float *acc) {
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int VEC = 16 / EB;
  constexpr int RPS = kStreamThreads / 32;
  uint4 v[U];
  float a[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int r = r0 + u * RPS;
    v[u] = r < kr ? __ldcs(reinterpret_cast<const uint4 *>(Bc + (int64_t)r * pitch)) : make_uint4(0, 0, 0, 0);
    a[u] = r < kr ? to_f32(x[r * acs]) : 0.f;
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float bf[VEC];
    unpack16<TB>(v[u], bf);
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = fmaf(a[u], bf[j], acc[j]);
  }
}

// The main loop of gemv_n_stream: this lane's 16 bytes of every RPS-th row of
// the CTA's kr rows, starting at row rr.  STEPS > 0: exactly STEPS steps of
// kStreamFixedU rows (the host guarantees kr <= STEPS * RPS * kStreamFixedU),
// unrolled; STEPS = 0: a loop of kStreamU-row steps.  A lane whose first
// column is inside the matrix loads its whole 16-byte piece: rows are 16-byte
// aligned, so the piece cannot cross a page, and the columns past N it picks
// up (row padding, or bytes past the operand's last row) only feed sums that
// are never stored.  A lane past N reads the group's first piece instead (an
// address inside the matrix) into sums that are never stored either.  The
// host keeps (K - 1) * a_cs below 2^31, so A's offsets fit an int.
template <int TB, int TA, int STEPS>
__device__ __forceinline__ void stream_rows(const char *Bk, int64_t ldb, bool lane_in, int col,
                                            int col0, const void *A, int64_t a0, int a_cs,
                                            int rr, int kr, float *acc) {
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int RPS = kStreamThreads / 32;
  using TAe = typename std::conditional<TA == MM_F32, float,
              typename std::conditional<TA == MM_BF16, __nv_bfloat16, __half>::type>::type;
  const int64_t pitch = ldb * EB;
  const char *Bc = Bk + (int64_t)(lane_in ? col : col0) * EB;
  const TAe *x = static_cast<const TAe *>(A) + a0;
  if constexpr (STEPS > 0) {
#pragma unroll
    for (int i = 0; i < STEPS; ++i)
      stream_step<TB, TAe, kStreamFixedU>(Bc, pitch, x, a_cs, rr + i * kStreamFixedU * RPS, kr, acc);
  } else {
    for (int r0 = rr; r0 < kr; r0 += RPS * kStreamU)
      stream_step<TB, TAe, kStreamU>(Bc, pitch, x, a_cs, r0, kr, acc);
  }
}

template <int TB, int TA, int STEPS>
__global__ void __launch_bounds__(kStreamThreads, 2) gemv_n_stream_kernel(const FastArgs g) {
  pdl_launch_dependents();
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int VEC = 16 / EB;
  constexpr int CW = kStreamSegB / EB;              // columns of a group
  constexpr int RPS = kStreamThreads / 32;          // rows per step: one a warp
  constexpr int H = kStreamThreads / CW;            // threads per column in the final sum
  extern __shared__ float part[];                   // [RPS][CW], then [H][CW]
  __shared__ unsigned last;
  const int b = blockIdx.y;
  const int grp = blockIdx.x / g.S, sp = blockIdx.x - grp * g.S;
  const int k0 = (int)((int64_t)sp * g.K / g.S);
  const int kr = (int)((int64_t)(sp + 1) * g.K / g.S) - k0;
  const int col0 = grp * CW;
  const char *Bk = g.B + ((int64_t)b * g.sB + (int64_t)k0 * g.ldb) * EB;  // row k0, column 0
  {  // this CTA's row segments, whole 16-byte pieces, into L2 before the wait
    const int64_t run = ((int64_t)min(CW, g.N - col0) * EB) & ~(int64_t)15;
    if (run > 0)
      for (int r = threadIdx.x; r < kr; r += kStreamThreads)
        prefetch_l2(Bk + ((int64_t)r * g.ldb + col0) * EB, (uint32_t)run);
  }
  pdl_wait();  // A, the workspace, the tickets and C only after the previous kernel
  const int lane = threadIdx.x & 31, rr = threadIdx.x >> 5;
  const int col = col0 + lane * VEC;
  const int64_t a0 = (int64_t)b * g.sA + (int64_t)k0 * g.a_cs;
  float acc[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) acc[j] = 0.f;
  stream_rows<TB, TA, STEPS>(Bk, g.ldb, col < g.N, col, col0, g.A, a0, (int)g.a_cs, rr, kr, acc);
  // the CTA's rows, added in row-phase order
#pragma unroll
  for (int j = 0; j < VEC; ++j) part[rr * CW + lane * VEC + j] = acc[j];
  __syncthreads();
  const int c = threadIdx.x % CW;
  float t = 0.f;
  if (threadIdx.x < CW)
#pragma unroll
    for (int q = 0; q < RPS; ++q) t += part[q * CW + c];
  if (g.S == 1) {
    if (threadIdx.x < CW && col0 + c < g.N) st_any(g.C, (int64_t)b * g.sC + col0 + c, g.tc, t);
    return;
  }
  const int64_t tile = (int64_t)b * g.G + grp;
  float *ws = g.ws + tile * g.S * CW;  // [S][CW] of this group
  if (threadIdx.x < CW) __stcg(ws + (int64_t)sp * CW + c, t);
  // The barrier orders every thread's partial store before thread 0's
  // release; thread 0's acquire (in the last CTA) orders the other CTAs'
  // partials before this CTA's loads, which the second barrier extends to
  // all of its threads.
  __syncthreads();
  if (threadIdx.x == 0) last = atom_add_acq_rel_gpu(g.tickets + tile, 1u) == (unsigned)g.S - 1;
  __syncthreads();
  if (!last) return;
  if (g.S <= kStreamCombineMax) {
    // one thread a column adds the S split sums in split order, all of their
    // loads in flight (no second exchange through shared memory)
    if (threadIdx.x < CW) {
      float x[kStreamCombineMax];
#pragma unroll
      for (int q = 0; q < kStreamCombineMax; ++q)
        x[q] = q < g.S ? __ldcg(ws + (int64_t)q * CW + c) : 0.f;
      float y = x[0];
#pragma unroll
      for (int q = 1; q < kStreamCombineMax; ++q)
        if (q < g.S) y += x[q];
      if (col0 + c < g.N) st_any(g.C, (int64_t)b * g.sC + col0 + c, g.tc, y);
    }
    if (threadIdx.x == 0) g.tickets[tile] = 0;  // ready for the next call on this stream
    return;
  }
  // more splits: H threads a column, thread h adds the splits
  // [h*S/H, (h+1)*S/H) with all of their loads in flight, then the H run sums
  // are added in run order.
  const int h = threadIdx.x / CW;
  const int sb = h * g.S / H, se = (h + 1) * g.S / H;
  float run = 0.f;
  for (int s0 = sb; s0 < se; s0 += 16) {
    float x[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) x[q] = s0 + q < se ? __ldcg(ws + (int64_t)(s0 + q) * CW + c) : 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) run += x[q];
  }
  part[h * CW + c] = run;
  __syncthreads();
  if (threadIdx.x < CW) {
    float y = 0.f;
#pragma unroll
    for (int q = 0; q < H; ++q) y += part[q * CW + c];
    if (col0 + c < g.N) st_any(g.C, (int64_t)b * g.sC + col0 + c, g.tc, y);
  }
  if (threadIdx.x == 0) g.tickets[tile] = 0;  // ready for the next call on this stream
}

// ---------------------------------------------------------------- gemv_t_stream
// M = 1, B transposed (stored [N][K]): output n is the dot product of A with
// the contiguous row n of B, so a CTA can own whole rows and no CTA depends on
// another.  CTA c of about two per SM takes the rows [c*N/C, (c+1)*N/C)
// (prefetched into L2 before the grid dependency wait); thread t holds the
// 16-byte pieces t, t+512, ... of every row (a warp reads 512 contiguous bytes
// of a row) against A's matching elements, one partial dot product per row of
// a block of 16 rows.  Each block is summed across the CTA in a fixed order
// (xor shuffles in a warp, then the 16 warps in order) and written.
// PA (A contiguous, 16-byte aligned, as wide as B's elements, K a whole
// number of pieces): A's piece is one 16-byte load kept packed and unpacked
// at each row, which leaves the registers for eight rows' loads in flight
// (4096 x 4096 bf16, measured back to back: 6.2 us a call against 7.4 us for
// the general form).  Otherwise A's elements are loaded one by one and four
// rows of loads are in flight.
constexpr int kTsThreads = 512;
constexpr int kTsRB = 16;  // rows per block
constexpr int kTsU = 4;    // rows of loads in flight, general form
constexpr int kTsPackedU = 8;  // rows of loads in flight, packed-A form

template <int TB, int TA, bool PA>
__global__ void __launch_bounds__(kTsThreads, 2) gemv_t_stream_kernel(const FastArgs g) {
  pdl_launch_dependents();
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int VEC = 16 / EB;
  constexpr int W = kTsThreads / 32;
  constexpr int U = PA ? kTsPackedU : kTsU;
  using TAe = typename std::conditional<TA == MM_F32, float,
              typename std::conditional<TA == MM_BF16, __nv_bfloat16, __half>::type>::type;
  static_assert(!PA || sizeof(TAe) == EB, "packed A needs A as wide as B");
  __shared__ float red[W][kTsRB];
  const int b = blockIdx.y;
  const int C = gridDim.x, c = blockIdx.x;
  const int r0 = (int)((int64_t)c * g.N / C), r1 = (int)((int64_t)(c + 1) * g.N / C);
  const char *Bb = g.B + (int64_t)b * g.sB * EB;
  const int64_t rowb = g.ldb * EB;
  {  // this CTA's rows, whole 16-byte pieces, into L2 before the wait
    const int64_t run = ((int64_t)g.K * EB) & ~(int64_t)15;
    for (int r = r0 + (int)threadIdx.x; r < r1 && run > 0; r += kTsThreads)
      for (int64_t o = 0; o < run; o += 65536)
        prefetch_l2(Bb + (int64_t)r * rowb + o, (uint32_t)(run - o < 65536 ? run - o : 65536));
  }
  pdl_wait();
  const TAe *Ab = static_cast<const TAe *>(g.A) + (int64_t)b * g.sA;
  const int ppr = (g.K + VEC - 1) / VEC;  // 16-byte pieces of a row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int rb = r0; rb < r1; rb += kTsRB) {
    float acc[kTsRB];
#pragma unroll
    for (int i = 0; i < kTsRB; ++i) acc[i] = 0.f;
    for (int p = threadIdx.x; p < ppr; p += kTsThreads) {
      const int kb = p * VEC;
      const char *bp = Bb + (int64_t)rb * rowb + (int64_t)kb * EB;
      if constexpr (PA) {
        const uint4 araw = *reinterpret_cast<const uint4 *>(Ab + kb);
#pragma unroll
        for (int i0 = 0; i0 < kTsRB; i0 += U) {
          uint4 v[U];
#pragma unroll
          for (int u = 0; u < U; ++u)
            v[u] = rb + i0 + u < r1 ? __ldcs(reinterpret_cast<const uint4 *>(bp + (int64_t)(i0 + u) * rowb))
                                    : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int u = 0; u < U; ++u) {
            float bf[VEC], af[VEC];
            unpack16<TB>(v[u], bf);
            unpack16<TA>(araw, af);
#pragma unroll
            for (int q = 0; q < VEC; ++q) acc[i0 + u] = fmaf(af[q], bf[q], acc[i0 + u]);
          }
        }
      } else {
        const bool tail = kb + VEC > g.K;  // the last piece of a row: elements past K are not B's
        float a[VEC];
#pragma unroll
        for (int q = 0; q < VEC; ++q) a[q] = kb + q < g.K ? to_f32(Ab[(int64_t)(kb + q) * g.a_cs]) : 0.f;
#pragma unroll
        for (int i0 = 0; i0 < kTsRB; i0 += U) {
          uint4 v[U];
#pragma unroll
          for (int u = 0; u < U; ++u)
            v[u] = rb + i0 + u < r1 ? __ldcs(reinterpret_cast<const uint4 *>(bp + (int64_t)(i0 + u) * rowb))
                                    : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int u = 0; u < U; ++u) {
            float bf[VEC];
            unpack16<TB>(v[u], bf);
            if (tail)
#pragma unroll
              for (int q = 0; q < VEC; ++q) bf[q] = kb + q < g.K ? bf[q] : 0.f;
#pragma unroll
            for (int q = 0; q < VEC; ++q) acc[i0 + u] = fmaf(a[q], bf[q], acc[i0 + u]);
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < kTsRB; ++i) {
      float x = acc[i];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      acc[i] = x;
    }
    if (lane == 0)
#pragma unroll
      for (int i = 0; i < kTsRB; ++i) red[warp][i] = acc[i];
    __syncthreads();
    if (threadIdx.x < kTsRB && rb + (int)threadIdx.x < r1) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) t += red[w][threadIdx.x];
      st_any(g.C, (int64_t)b * g.sC + rb + threadIdx.x, g.tc, t);
    }
    __syncthreads();  // red is reused by the next block
  }
}

// ---------------------------------------------------------------- gemv_t_rows
// A warp walks its row of B in chunks of CE = 32 * VEC elements (512 bytes),
// lane l holding elements [l * VEC, (l + 1) * VEC) of a chunk.  A sits in
// shared memory as fp32, one row of KP = (chunks * CE) floats per m, zero past
// K.  With 16-bit B a lane needs 8 floats of A per chunk; stored in k order
// they would be 32 bytes apart from lane to lane, and each 16-byte shared load
// would take two passes.  So each chunk of A is stored as its lanes' first
// four floats (128 of them), then their last four: element l * 8 + h * 4 + q
// of a chunk at position h * 128 + l * 4 + q, and a lane's two loads are
// 16 bytes apart from lane to lane.  With fp32 B (4 floats a lane) k order
// already has that property.
template <int VEC>
__device__ __forceinline__ int trows_k_of_pos(int pos) {
  if constexpr (VEC == 8) {
    const int c = pos >> 8, r = pos & 255;
    const int h = r >> 7, l = (r >> 2) & 31, q = r & 3;
    return (c << 8) + l * 8 + h * 4 + q;
  } else {
    return pos;
  }
}

template <int MT, int TB>
__global__ void __launch_bounds__(kThreads, MT <= 2 ? 2 : 1) gemv_t_rows_kernel(const FastArgs g) {
  pdl_launch_dependents();
  constexpr int EB = TB == MM_F32 ? 4 : 2;
  constexpr int VEC = 16 / EB;
  constexpr int CE = 32 * VEC;
  constexpr int U = 8;
  extern __shared__ float fsm[];  // dynamic shared memory starts 16-byte aligned
  float *As = fsm;  // [MT][KP]
  const int nch = (g.K + CE - 1) / CE;
  const int KP = nch * CE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int n = blockIdx.x * kWarps + warp;
  const char *row = g.B + ((int64_t)b * g.sB + (int64_t)min(n, g.N - 1) * g.ldb) * EB;
  const bool valid = n < g.N;
  if (valid) {  // this warp's row of B, in whole 16-byte pieces of at most 4 KB
    const int64_t bytes = ((int64_t)g.K * EB) & ~(int64_t)15;
    for (int64_t o = (int64_t)lane * 4096; o < bytes; o += 32 * 4096)
      prefetch_l2(row + o, (uint32_t)min((int64_t)4096, bytes - o));
  }
  pdl_wait();
  float acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0.f;
  bool staged = false;
  for (int c0 = 0; c0 < nch; c0 += U) {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int k = (c0 + u) * CE + lane * VEC;
      v[u] = valid && c0 + u < nch ? load16<TB>(row, k, g.K) : make_uint4(0, 0, 0, 0);
    }
    if (!staged) {
      stage_batched(g, As, MT * KP, [&](int e, int64_t *off) {
        const int m = e / KP, k = trows_k_of_pos<VEC>(e - m * KP);
        if (m >= g.M || k >= g.K) return false;
        *off = (int64_t)b * g.sA + (int64_t)m * g.a_rs + (int64_t)k * g.a_cs;
        return true;
      });
      __syncthreads();
      staged = true;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + u;
      if (c < nch) {  // past K both B (load16) and A (staging) are zero
        float bf[VEC];
        unpack16<TB>(v[u], bf);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float *a = As + m * KP + c * CE + lane * 4;
          const float4 a0 = *reinterpret_cast<const float4 *>(a);
          float t = acc[m];
          t = fmaf(a0.x, bf[0], t);
          t = fmaf(a0.y, bf[1], t);
          t = fmaf(a0.z, bf[2], t);
          t = fmaf(a0.w, bf[3], t);
          if constexpr (VEC == 8) {
            const float4 a1 = *reinterpret_cast<const float4 *>(a + 128);
            t = fmaf(a1.x, bf[4], t);
            t = fmaf(a1.y, bf[5], t);
            t = fmaf(a1.z, bf[6], t);
            t = fmaf(a1.w, bf[7], t);
          }
          acc[m] = t;
        }
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float x = acc[m];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if (lane == 0 && valid && m < g.M)
      st_any(g.C, (int64_t)b * g.sC + (int64_t)m * g.ldc + n, g.tc, x);
  }
}

// ---------------------------------------------------------------- host
struct FastCfg {
  const char *name;
  bool b_trans;
  bool stream;  // gemv_n_stream
};
const FastCfg kFastCfgs[] = {
    {"gemv_n_cluster", false, false}, {"gemv_t_rows", true, false}, {"gemv_n_stream", false, true},
    {"gemv_t_stream", true, true}};

constexpr int kStreamMaxM = 1;
constexpr int64_t kStreamMaxSplits = 64;

// gemv_n_stream geometry: column groups of 512 bytes and K splits so that the
// grid holds about two CTAs per SM (a whole number per SM keeps every SM's
// share of the bytes equal).
void stream_plan(int64_t N, int64_t K, int64_t batch, int eb, int sms, int64_t *G, int64_t *S) {
  const int64_t cw = kStreamSegB / eb;
  *G = (N + cw - 1) / cw;
  const int64_t tiles = *G * batch;
  int64_t s = (2 * (int64_t)sms + tiles / 2) / tiles;
  s = std::max<int64_t>(1, std::min<int64_t>(s, std::min<int64_t>(K, kStreamMaxSplits)));
  *S = s;
}

int mt_of(int64_t M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

constexpr int kMaxM = 8;
// shared memory of one CTA: instances that keep two CTAs an SM (MT <= 2)
// stay within half of it; the others (one CTA an SM) may take most of it
size_t max_smem(int mt) { return mt <= 2 ? 96 * 1024 : 200 * 1024; }

size_t smem_n(int mt, int ks, int eb) {
  return ((size_t)ks * mt + (size_t)kWarps * mt * (256 / eb)) * sizeof(float);
}
// gemv_t_rows: A as fp32 rows padded to whole 512-byte chunks of B (at most
// 256 elements a chunk).
size_t smem_t(int mt, int64_t K) { return (size_t)mt * ((K + 255) / 256 * 256) * sizeof(float); }
// gemv_t_stream: CTAs per batch item, about two per SM, at least one row each.
int64_t tstream_ctas(int64_t N, int64_t batch, int sms) {
  const int64_t per = (2 * (int64_t)sms + batch - 1) / batch;
  return std::max<int64_t>(1, std::min<int64_t>(N, per));
}

size_t smem_stream(int eb) { return (size_t)(kStreamThreads / 32) * (kStreamSegB / eb) * sizeof(float); }

int rows_per_rank(int64_t K) {
  int64_t ks = (K + kCluster - 1) / kCluster;
  return (int)((ks + 31) / 32 * 32);
}

template <typename F>
cudaError_t smem_attr(F kern, size_t smem) {
  static std::mutex mu;
  static std::map<const void *, size_t> have;
  std::lock_guard<std::mutex> lk(mu);
  size_t &h = have[reinterpret_cast<const void *>(kern)];
  if (smem <= h || smem <= 48 * 1024) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) h = smem;
  return e;
}

template <int MT, int TB>
mm_status launch_n(const FastArgs &g, int groups, size_t smem, cudaStream_t s) {
  auto kern = gemv_n_cluster_kernel<MT, TB>;
  cudaError_t e = smem_attr(kern, smem);
  if (e != cudaSuccess) return cuda_error(e, "gemv_n_cluster smem attribute");
  e = launch_pdl(kern, dim3((unsigned)groups, kCluster, (unsigned)g.batch), dim3(kThreads), smem,
                 s, dim3(1, kCluster, 1), g);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "gemv_n_cluster launch");
}

template <int MT, int TB>
mm_status launch_t(const FastArgs &g, size_t smem, cudaStream_t s) {
  auto kern = gemv_t_rows_kernel<MT, TB>;
  cudaError_t e = smem_attr(kern, smem);
  if (e != cudaSuccess) return cuda_error(e, "gemv_t_rows smem attribute");
  dim3 grid((unsigned)((g.N + kWarps - 1) / kWarps), (unsigned)g.batch);
  e = launch_pdl(kern, grid, dim3(kThreads), smem, s, dim3(1), g);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "gemv_t_rows launch");
}

// Unrolled steps for a split of at most kr_max rows: 1, 2 or 4 steps of
// kStreamFixedU rows a warp, or 0 (the rolled loop) for deeper splits.
int stream_steps(int64_t kr_max) {
  const int64_t per = (int64_t)(kStreamThreads / 32) * kStreamFixedU;
  const int64_t n = (kr_max + per - 1) / per;
  return n <= 1 ? 1 : n <= 2 ? 2 : n <= kStreamMaxSteps ? kStreamMaxSteps : 0;
}

template <int TB, int TA>
mm_status launch_stream(const FastArgs &g, size_t smem, cudaStream_t s) {
  const dim3 grid((unsigned)(g.G * g.S), (unsigned)g.batch);
  const int64_t kr_max = ((int64_t)g.K + g.S - 1) / g.S;
  cudaError_t e;
  switch (stream_steps(kr_max)) {
  case 1: e = launch_pdl(gemv_n_stream_kernel<TB, TA, 1>, grid, dim3(kStreamThreads), smem, s, dim3(1), g); break;
  case 2: e = launch_pdl(gemv_n_stream_kernel<TB, TA, 2>, grid, dim3(kStreamThreads), smem, s, dim3(1), g); break;
  case 4: e = launch_pdl(gemv_n_stream_kernel<TB, TA, 4>, grid, dim3(kStreamThreads), smem, s, dim3(1), g); break;
  default: e = launch_pdl(gemv_n_stream_kernel<TB, TA, 0>, grid, dim3(kStreamThreads), smem, s, dim3(1), g); break;
  }
  return e == cudaSuccess ? MM_OK : cuda_error(e, "gemv_n_stream launch");
}

template <int TB, int TA>
mm_status launch_tstream(const FastArgs &g, int64_t C, bool packed, cudaStream_t s) {
  const dim3 grid((unsigned)C, (unsigned)g.batch);
  cudaError_t e;
  if constexpr ((TB == MM_F32) == (TA == MM_F32)) {
    e = packed ? launch_pdl(gemv_t_stream_kernel<TB, TA, true>, grid, dim3(kTsThreads), 0, s, dim3(1), g)
               : launch_pdl(gemv_t_stream_kernel<TB, TA, false>, grid, dim3(kTsThreads), 0, s, dim3(1), g);
  } else {
    e = launch_pdl(gemv_t_stream_kernel<TB, TA, false>, grid, dim3(kTsThreads), 0, s, dim3(1), g);
  }
  return e == cudaSuccess ? MM_OK : cuda_error(e, "gemv_t_stream launch");
}

template <int TB>
mm_status launch_tstream_ta(const FastArgs &g, int64_t C, bool packed, cudaStream_t s) {
  if (g.ta == MM_BF16) return launch_tstream<TB, MM_BF16>(g, C, packed, s);
  if (g.ta == MM_F16) return launch_tstream<TB, MM_F16>(g, C, packed, s);
  return launch_tstream<TB, MM_F32>(g, C, packed, s);
}

template <int TB>
mm_status launch_stream_ta(const FastArgs &g, size_t smem, cudaStream_t s) {
  if (g.ta == MM_BF16) return launch_stream<TB, MM_BF16>(g, smem, s);
  if (g.ta == MM_F16) return launch_stream<TB, MM_F16>(g, smem, s);
  return launch_stream<TB, MM_F32>(g, smem, s);
}

template <int TB>
mm_status launch_tb(bool bt, int mt, const FastArgs &g, int groups, size_t smem, cudaStream_t s) {
  switch (mt) {
  case 1: return bt ? launch_t<1, TB>(g, smem, s) : launch_n<1, TB>(g, groups, smem, s);
  case 2: return bt ? launch_t<2, TB>(g, smem, s) : launch_n<2, TB>(g, groups, smem, s);
  case 4: return bt ? launch_t<4, TB>(g, smem, s) : launch_n<4, TB>(g, groups, smem, s);
  default: return bt ? launch_t<8, TB>(g, smem, s) : launch_n<8, TB>(g, groups, smem, s);
  }
}

}  // namespace

int gemv_fast_config_count() { return (int)(sizeof kFastCfgs / sizeof kFastCfgs[0]); }
const char *gemv_fast_config_name(int cfg) { return kFastCfgs[cfg].name; }

bool gemv_fast_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why) {
  auto no = [&](const char *w) {
    if (why) *why = w;
    return false;
  };
  const FastCfg &c = kFastCfgs[cfg];
  if (d.cc_major != 10) return no("needs an sm_10x device");
  if (p.bt != c.b_trans) return no("B layout does not match this variant");
  if (p.M < 1 || p.M > kMaxM) return no("M outside [1, 8]");
  if (p.K < 1 || p.N < 1) return no("empty problem");
  if (p.N >= (1LL << 30) || p.K >= (1LL << 30) || p.batch > 65535) return no("too large");
  const int eb = dtype_bytes(p.tb);
  if ((uintptr_t)p.B % 16) return no("B not 16-byte aligned");
  if ((p.ldb * eb) % 16) return no("ldb not a multiple of 16 bytes");
  if (p.batch > 1 && (p.sB * eb) % 16) return no("B batch stride not a multiple of 16 bytes");
  const int mt = mt_of(p.M);
  size_t smem;
  if (c.stream) {
    if (p.M > kStreamMaxM) return no("M must be 1");
    if (!c.b_trans && (p.K - 1) * (p.at ? p.lda : 1) >= (1LL << 31))
      return no("A's K stride too large for 32-bit offsets");
    if (c.b_trans) {
      smem = 0;
    } else {
      int64_t G, S;
      stream_plan(p.N, p.K, p.batch, eb, d.sms, &G, &S);
      if (G * S >= (1LL << 31)) return no("too many column groups");
      smem = smem_stream(eb);
    }
  } else {
    smem = c.b_trans ? smem_t(mt, p.K) : smem_n(mt, rows_per_rank(p.K), eb);
  }
  if (smem > max_smem(mt) || (int64_t)smem > d.smem_optin)
    return no("A slice too large for shared memory");
  return true;
}

mm_status launch_gemv_fast(const Problem &p, LaunchCtx &ctx, int cfg) {
  std::string why;
  if (!gemv_fast_supports(p, ctx.dev->info, cfg, &why))
    return set_error(MM_ERR_UNSUPPORTED, "%s: %s", kFastCfgs[cfg].name, why.c_str());
  const FastCfg &c = kFastCfgs[cfg];
  const int eb = dtype_bytes(p.tb), mt = mt_of(p.M);
  FastArgs g;
  std::memset(&g, 0, sizeof g);
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
  int groups = 0;
  size_t smem;
  if (c.stream && c.b_trans) {
    const int64_t C = tstream_ctas(p.N, p.batch, ctx.dev->info.sms);
    // A's pieces as single 16-byte loads: A contiguous along K and 16-byte
    // aligned (base and batch stride), as wide as B, K a whole number of pieces
    const int ea = dtype_bytes(p.ta);
    const bool packed = ea == eb && g.a_cs == 1 && (uintptr_t)p.A % 16 == 0 &&
                        (p.batch == 1 || (p.sA * ea) % 16 == 0) && (p.K * eb) % 16 == 0;
    if (p.tb == MM_BF16) return launch_tstream_ta<MM_BF16>(g, C, packed, ctx.stream);
    if (p.tb == MM_F16) return launch_tstream_ta<MM_F16>(g, C, packed, ctx.stream);
    return launch_tstream_ta<MM_F32>(g, C, packed, ctx.stream);
  }
  if (c.stream) {
    int64_t G, S;
    stream_plan(p.N, p.K, p.batch, eb, ctx.dev->info.sms, &G, &S);
    g.G = (int)G;
    g.S = (int)S;
    smem = smem_stream(eb);
    if (S > 1) {
      const size_t ws_bytes = (size_t)p.batch * G * S * (kStreamSegB / eb) * sizeof(float);
      const size_t tickets_bytes = (size_t)p.batch * G * sizeof(unsigned);
      void *w = nullptr, *t = nullptr;
      mm_status st = get_scratch(*ctx.dev, ctx.stream, SCRATCH_WORKSPACE, ws_bytes, &w);
      if (st != MM_OK) return st;
      st = get_scratch(*ctx.dev, ctx.stream, SCRATCH_TICKETS, tickets_bytes, &t);
      if (st != MM_OK) return st;
      g.ws = static_cast<float *>(w);
      g.tickets = static_cast<unsigned *>(t);
    }
    if (p.tb == MM_BF16) return launch_stream_ta<MM_BF16>(g, smem, ctx.stream);
    if (p.tb == MM_F16) return launch_stream_ta<MM_F16>(g, smem, ctx.stream);
    return launch_stream_ta<MM_F32>(g, smem, ctx.stream);
  }
  if (!c.b_trans) {
    g.KS = rows_per_rank(p.K);
    groups = (int)((p.N + 256 / eb - 1) / (256 / eb));
    smem = smem_n(mt, g.KS, eb);
  } else {
    smem = smem_t(mt, p.K);
  }
  if (p.tb == MM_BF16) return launch_tb<MM_BF16>(c.b_trans, mt, g, groups, smem, ctx.stream);
  if (p.tb == MM_F16) return launch_tb<MM_F16>(c.b_trans, mt, g, groups, smem, ctx.stream);
  return launch_tb<MM_F32>(c.b_trans, mt, g, groups, smem, ctx.stream);
}

}  // namespace mm
