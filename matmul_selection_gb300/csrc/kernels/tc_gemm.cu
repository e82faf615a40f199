// Tensor-core GEMM family for sm_103a: tcgen05.mma into TMEM, fed by TMA.
//
// The autotune page's "accelerated" group (cooperative-matrix kernels) and its
// TMA-fed variants are rebuilt here for Blackwell's 5th-generation tensor
// cores.  One kernel template covers every configuration:
//
//   * persistent: one CTA per SM walks the work units (output tile x batch x
//     K split) with a grid stride;
//   * warp-specialised, 7 warps: warps 0 and 6 issue the TMA loads of A and
//     of B, warp 1 allocates TMEM and issues tcgen05.mma (each role runs as a
//     whole warp with warp-uniform loop state; elect.sync picks the issuing
//     lane), warps 2..5 drain accumulators from TMEM (tcgen05.ld) and store
//     them;
//   * an S-stage shared-memory ring guarded by mbarriers (full: TMA bytes
//     landed; empty: the MMAs reading the stage completed, signalled by
//     tcgen05.commit), and two TMEM accumulators so the epilogue of one tile
//     overlaps the main loop of the next;
//   * tiles are 128 x BN x (128 bytes of K) with the 128-byte swizzle; A and B
//     may each be K-major or MN-major (MN-major only for 16-bit types), so
//     transposed views are read in place;
//   * kind::f16 for bf16/f16 inputs, kind::tf32 for f32 inputs (f32 is
//     multiplied as tf32: the burn backend page notes the kernel may run f32
//     as tf32), fp32 accumulation always;
//   * split-K configurations write fp32 partials of each K slice to a
//     workspace, one CTA a (tile, K slice); a second kernel adds the slices
//     in a fixed order (runs of consecutive slices, each in increasing order,
//     then the runs in order; deterministic) and converts.  Split-K regroups
//     additions only (the CMU 15-779 lecture's rfactor / split-K discussion);
//   * every mbarrier wait is bounded (%globaltimer); on expiry the kernel
//     records an error code, tells the other roles to stop, waits for its own
//     MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "../common.h"

namespace mm {

namespace {

constexpr int BM = 128;
// 7 warps: A copies, MMA, 4 epilogue warps, B copies
constexpr int kTcThreads = 224;
// 2-SM kernel with A copied by cp.async (rows TMA cannot address): 7 more
// warps (7..13) copy A, warp 0 relays the copies' completion.  No more copy
// warps than ring stages (see the copies' loop).
constexpr int kCopyWarps = 7;
constexpr int kTcThreadsAsyncA = 224 + 32 * kCopyWarps;
// 1-SM kernel shared memory after the ring: two 4 KB output staging boxes for
// each epilogue warp (32 rows x 128 bytes, 128-byte swizzle; also the fallback
// store path's [32][33] transpose scratch), then the barriers
constexpr uint32_t kEpiStageBytes = 4 * 2 * 4096;
constexpr uint32_t kBarBytes = 256;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s per wait (main loops, default)
constexpr uint64_t kDrainTimeoutNs = 2000000000ull;  // 2 s per drain wait, always

// error codes (first one wins): 0x100 | role
constexpr int kErrProducer = 0x101, kErrMma = 0x102, kErrEpilogue = 0x103, kErrDrain = 0x104,
              kErrReduce = 0x105;

struct TcParams {
  int M, N, K, batch;
  int tiles_m, tiles_n, splits, kb_per_split, num_kb, total_units;
  void *C;
  int64_t ldc, sC;
  int tc;
  int c_vec_ok;
  float *ws;
  int *err;
  uint32_t idesc;
  uint64_t a_desc, b_desc;           // descriptor bits except the start address
  uint32_t a_kstep, b_kstep;         // start-address advance per MMA k-step (16-byte units)
  uint32_t a_box_stride, b_box_stride;  // bytes between the TMA boxes of one stage (MN-major)
  int a_boxes, b_boxes, a_mn, b_mn;
  // MN-major operand whose boxes of one stage come from a single 4-D copy
  // (map over (atom, K, atom index, batch)); 0: one 3-D copy per box
  int a_4d, b_4d;
  // output stored transposed: element (i, j) of the computed product goes to
  // C[j * ldc + i] (the swapped form C^T = B^T A^T of a product with small M)
  int c_trans;
  // test hook: the MMA warp first waits on a barrier nothing arrives on, so
  // that the wait limit runs out and the kernel's abort path runs
  int stall_wait;
  // 2-SM kernel, A copied by cp.async: A itself (K-major), its row and batch
  // strides in bytes, and the piece size (8 or 4 bytes: the largest that
  // divides the base address and both strides)
  const char *a_ptr;
  int64_t a_row_bytes, a_batch_bytes;
  int a_piece;
  // 1-SM kernel: C written by TMA bulk-tensor stores (tmC valid); with
  // splits > 1, tmC maps the fp32 workspace as [splits * batch][M][N]
  int c_tma;
  uint64_t timeout_ns;
  // 2-SM kernel: units [0, full_units) are whole tiles; the remaining tiles
  // of the last partial wave are split along N into two half-width units
  int full_units;
  uint32_t idesc_half;  // instruction descriptor for a half-width unit
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// The producer and MMA roles run as whole warps so that their loop state stays
// warp-uniform; each issuing wrapper below marked "warp-collective" is executed
// by all 32 lanes and elect.sync picks the one lane that performs the operation.

// Warp-collective.
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbarrier wait with acquire semantics at cluster scope (the arrival may be a
// release by the other CTA of the pair).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `parity` to complete.  Executed by a whole warp (every
// lane polls; the result is warp-uniform).  Gives up (false) when the shared
// abort flag is raised or after timeout_ns, raising the flag and recording
// `code` in the error word.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try_wait_scoped(uint32_t bar, uint32_t parity) {
  return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}
// CLUSTER: acquire at cluster scope (for arrivals the other CTA of a pair
// releases).
template <bool CLUSTER = false>
__device__ __noinline__ bool warp_wait_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                            int *err, int code, uint64_t timeout_ns) {
  const uint64_t t0 = global_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (__all_sync(0xffffffffu, mbar_try_wait_scoped<CLUSTER>(bar, parity))) return true;
    int stop = 0;
    if ((threadIdx.x & 31) == 0) {
      if (*abort_flag) {
        stop = 1;
      } else if (global_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicCAS(err, 0, code);
        stop = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
  }
}
template <bool CLUSTER = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int *err, int code, uint64_t timeout_ns) {
  if (__all_sync(0xffffffffu, mbar_try_wait_scoped<CLUSTER>(bar, parity))) return true;
  return warp_wait_slow<CLUSTER>(bar, parity, abort_flag, err, code, timeout_ns);
}

// Bounded wait that ignores the abort flag: used at the end to let copies and
// MMAs already in flight finish before shared memory and TMEM are released.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, int *err, int code,
                                        uint64_t timeout_ns) {
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > timeout_ns) {
      atomicCAS(err, 0, code);
      return;
    }
  }
}

// Lower the barrier's pending transaction count by `bytes` as if they had
// arrived (for copies that were counted but never issued).  Warp-collective.
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.complete_tx.shared::cta.b64 [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
      : "memory");
}

// Warp-collective.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Warp-collective.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// L2 prefetch of one box of a tensor map: no shared memory, no barrier, and
// nothing returned to the SM, so it may run before the grid dependency wait
// (it cannot observe a value the previous kernel has yet to write; the copies
// after the wait read the coherent L2).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap *map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int c0, int c1, int c2,
                                                int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
// Bytes of operand boxes a CTA prefetches into L2 before its grid dependency
// wait (the first k-blocks of its first work unit): a few hundred KB a CTA
// keeps the prefetches of a whole grid well inside L2.
constexpr uint32_t kPrefetchBytes = 256 * 1024;

// Bulk-tensor store of a shared-memory box (one thread), as its own group.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];\n\t"
      "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// This thread's bulk stores, all but the newest N, have read their source.
template <int N>
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// This thread's bulk stores have completed.
__device__ __forceinline__ void tma_store_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Generic-proxy writes to shared memory visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 prefetch of `bytes` (a multiple of 16) at a 16-byte aligned address.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Warp-collective.
template <int ES>
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                     uint32_t idesc, uint32_t accumulate) {
  if constexpr (ES == 2) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Arrive on `bar` once every previously issued tcgen05 op of the issuing
// thread is done.  Warp-collective.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i gets row (lane) i.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- epilogue store
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void store_one(void *C, int tc, int64_t off, float v) {
  if (tc == MM_F32)
    static_cast<float *>(C)[off] = v;
  else if (tc == MM_BF16)
    static_cast<__nv_bfloat16 *>(C)[off] = __float2bfloat16_rn(v);
  else
    static_cast<__half *>(C)[off] = __float2half_rn(v);
}

__device__ __forceinline__ void store_chunk(const TcParams &p, int b, int sp, int row, int col0,
                                            const uint32_t (&r)[32]) {
  if (row >= p.M) return;
  const bool full = col0 + 32 <= p.N;
  if (p.splits > 1) {
    float *dst = p.ws + (((int64_t)sp * p.batch + b) * p.M + row) * (int64_t)p.N + col0;
    if (full && (p.N & 3) == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        reinterpret_cast<float4 *>(dst)[i] =
            make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                        __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    } else {
      for (int i = 0; i < 32; ++i)
        if (col0 + i < p.N) dst[i] = __uint_as_float(r[i]);
    }
    return;
  }
  if (p.c_trans) {
    for (int i = 0; i < 32; ++i)
      if (col0 + i < p.N)
        store_one(p.C, p.tc, (int64_t)b * p.sC + (int64_t)(col0 + i) * p.ldc + row,
                  __uint_as_float(r[i]));
    return;
  }
  const int64_t off = (int64_t)b * p.sC + (int64_t)row * p.ldc + col0;
  if (p.tc == MM_F32) {
    float *dst = static_cast<float *>(p.C) + off;
    if (full && p.c_vec_ok) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        reinterpret_cast<float4 *>(dst)[i] =
            make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                        __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    } else {
      for (int i = 0; i < 32; ++i)
        if (col0 + i < p.N) dst[i] = __uint_as_float(r[i]);
    }
  } else {
    uint16_t *dst = static_cast<uint16_t *>(p.C) + off;
    const bool bf = p.tc == MM_BF16;
    if (full && p.c_vec_ok) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float lo = __uint_as_float(r[8 * i + 2 * j]), hi = __uint_as_float(r[8 * i + 2 * j + 1]);
          w[j] = bf ? pack_bf16(lo, hi) : pack_f16(lo, hi);
        }
        reinterpret_cast<uint4 *>(dst)[i] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
      for (int i = 0; i < 32; ++i)
        if (col0 + i < p.N) {
          float v = __uint_as_float(r[i]);
          if (bf) {
            __nv_bfloat16 h = __float2bfloat16_rn(v);
            dst[i] = *reinterpret_cast<uint16_t *>(&h);
          } else {
            __half h = __float2half_rn(v);
            dst[i] = *reinterpret_cast<uint16_t *>(&h);
          }
        }
    }
  }
}

// A warp's full 32 x 32 chunk (thread i holds row row0 + i), written row by
// row: the values go through a padded [32][33] scratch (conflict-free both
// ways) so that each store instruction writes consecutive columns of one row
// (f32: 128 bytes; 16-bit: two rows of 64 bytes, two columns a lane) instead
// of 16 bytes of 32 different rows.
__device__ __forceinline__ void store_chunk_rows(const TcParams &p, int b, int sp, int row0, int col0,
                                                 const uint32_t (&r)[32], float *scr, int lane) {
#pragma unroll
  for (int j = 0; j < 32; ++j) scr[lane * 33 + j] = __uint_as_float(r[j]);
  __syncwarp();
  if (p.splits > 1) {
    float *dst = p.ws + (((int64_t)sp * p.batch + b) * p.M + row0) * (int64_t)p.N + col0 + lane;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) dst[(int64_t)i * p.N] = scr[i * 33 + lane];
  } else if (p.tc == MM_F32) {
    float *dst = static_cast<float *>(p.C) + (int64_t)b * p.sC + (int64_t)row0 * p.ldc + col0 + lane;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) dst[(int64_t)i * p.ldc] = scr[i * 33 + lane];
  } else if (p.c_vec_ok) {  // two columns a lane: lanes 0-15 row i, lanes 16-31 row i + 1
    const bool bf = p.tc == MM_BF16;
    const int h = lane >> 4, cc = 2 * (lane & 15);
    uint32_t *dst = reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(p.C) + (int64_t)b * p.sC +
                                                 (int64_t)(row0 + h) * p.ldc + col0 + cc);
    const int64_t step = p.ldc;  // two rows of 16-bit elements, in 32-bit words
#pragma unroll 4
    for (int i = 0; i < 32; i += 2) {
      const float lo = scr[(i + h) * 33 + cc], hi = scr[(i + h) * 33 + cc + 1];
      dst[(int64_t)(i / 2) * step] = bf ? pack_bf16(lo, hi) : pack_f16(lo, hi);
    }
  } else {
    const int64_t base = (int64_t)b * p.sC + (int64_t)row0 * p.ldc + col0 + lane;
#pragma unroll 4
    for (int i = 0; i < 32; ++i) store_one(p.C, p.tc, base + (int64_t)i * p.ldc, scr[i * 33 + lane]);
  }
  __syncwarp();  // the scratch is reused by the next chunk
}

// Unit order: K split fastest, then N, then M, then batch.  CTAs that run at
// the same time then hold neighbouring column tiles of the same rows, so the
// output is written in whole rows (a write pattern of 128-byte pieces of
// many different rows reached 2.6 TB/s on GB300, whole rows 6.9 TB/s).
__device__ __forceinline__ void decode_unit(const TcParams &p, int u, int &tm, int &tn, int &b,
                                            int &sp) {
  sp = u % p.splits;
  u /= p.splits;
  tn = u % p.tiles_n;
  u /= p.tiles_n;
  tm = u % p.tiles_m;
  b = u / p.tiles_m;
}

// K blocks of a work unit: split sp takes the contiguous blocks
// [sp * kb_per_split, (sp + 1) * kb_per_split) (all of them without split-K).
__device__ __forceinline__ int unit_kblocks(const TcParams &p, int sp) {
  return min(p.kb_per_split, p.num_kb - sp * p.kb_per_split);
}
__device__ __forceinline__ int unit_kb(const TcParams &p, int sp, int i) {
  return sp * p.kb_per_split + i;
}


// ---------------------------------------------------------------- the kernel
// SK: a split-K configuration.  Each of its CTAs takes exactly one work unit
// (the grid has one CTA a unit), so once the unit's MMAs are done the operand
// ring is idle: the epilogue stages its stores in the ring, and the CTA needs
// no shared memory beyond it (the ring can be a stage deeper) and one TMEM
// accumulator.
template <int BN, int STAGES, int ES, bool SK>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  pdl_launch_dependents();
  constexpr uint32_t A_BYTES = BM * 128;
  constexpr uint32_t B_BYTES = BN * 128;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int BK = 128 / ES;      // K elements per stage (one 128-byte swizzle row)
  constexpr int UMMA_K = 32 / ES;   // K per tcgen05.mma (32 bytes)
  constexpr int KSTEPS = BK / UMMA_K;
  constexpr uint32_t TMEM_COLS = SK ? BN : 2 * BN;
  constexpr int ATOM = 128 / ES;    // elements per 128-byte row (MN-major box width)
  static_assert(!SK || STAGES * STAGE_BYTES >= kEpiStageBytes + 2048,
                "split-K epilogue staging and reduction scratch live in the ring");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *epi_stage = SK ? smem : smem + STAGES * STAGE_BYTES;  // 1024-byte aligned
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES + (SK ? 0 : kEpiStageBytes));
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t stall = drain + 8;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 6);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a split-K CTA takes its one unit (the host launches one CTA a unit); a
  // persistent CTA walks the units with the grid stride
  const int ustep = SK ? p.total_units : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    mbar_init(stall, 1);  // nothing ever arrives on it
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (p.c_tma) prefetch_tmap(&tmC);
  }
  // the first k-blocks of this CTA's first unit into L2, A by warp 0, B by
  // warp 6 (B only when it fills a box: a short B, such as the swapped form
  // of a GEMV with a few rows, is small, shared by every CTA, and its
  // mostly out-of-range boxes measured slower prefetched than not)
  if ((warp == 0 || (warp == 6 && p.N >= BN)) && lane == 0 && (int)blockIdx.x < p.total_units) {
    int tm, tn, b, sp;
    decode_unit(p, blockIdx.x, tm, tn, b, sp);
    const int nk = min(unit_kblocks(p, sp), (int)(kPrefetchBytes / STAGE_BYTES));
    for (int i = 0; i < nk; ++i) {
      const int kb = unit_kb(p, sp, i);
      if (warp == 0) {
        if (!p.a_mn) tma_prefetch_3d(&tmA, kb * BK, tm * BM, b);
        else if (p.a_4d) tma_prefetch_4d(&tmA, 0, kb * BK, tm * (BM / ATOM), b);
        else
          for (int j = 0; j < p.a_boxes; ++j) tma_prefetch_3d(&tmA, tm * BM + j * ATOM, kb * BK, b);
      } else {
        if (!p.b_mn) tma_prefetch_3d(&tmB, kb * BK, tn * BN, b);
        else if (p.b_4d) tma_prefetch_4d(&tmB, 0, kb * BK, tn * (BN / ATOM), b);
        else
          for (int j = 0; j < p.b_boxes; ++j) tma_prefetch_3d(&tmB, tn * BN + j * ATOM, kb * BK, b);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the prologue above touched no global memory

  if (warp == 0 || warp == 6) {
    // ------------------------------------------------------------ TMA producers
    // warp 0 arms the stage and copies A, warp 6 copies B (see the 2-SM
    // kernel for why B bytes landing before the arming are harmless)
    const bool copy_a = warp == 0;
    {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int nfill = 0;  // stage fills this warp issued
      for (int u = blockIdx.x; u < p.total_units && ok; u += ustep) {
        int tm, tn, b, sp;
        decode_unit(p, u, tm, tn, b, sp);
        const int nk = unit_kblocks(p, sp);
        for (int i = 0; i < nk; ++i) {
          const int kb = unit_kb(p, sp, i);
          if (!warp_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.err, kErrProducer,
                         p.timeout_ns)) {
            ok = false;
            break;
          }
          ++nfill;
          const uint32_t fb = full0 + 8 * stage;
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          if (copy_a) {
            mbar_expect_tx(fb, STAGE_BYTES);
            if (!p.a_mn) {
              tma_load_3d(sa, &tmA, fb, kb * BK, tm * BM, b);
            } else if (p.a_4d) {
              tma_load_4d(sa, &tmA, fb, 0, kb * BK, tm * (BM / ATOM), b);
            } else {
              for (int j = 0; j < p.a_boxes; ++j)
                tma_load_3d(sa + j * p.a_box_stride, &tmA, fb, tm * BM + j * ATOM, kb * BK, b);
            }
          } else if (!p.b_mn) {
            tma_load_3d(sb, &tmB, fb, kb * BK, tn * BN, b);
          } else if (p.b_4d) {
            tma_load_4d(sb, &tmB, fb, 0, kb * BK, tn * (BN / ATOM), b);
          } else {
            for (int j = 0; j < p.b_boxes; ++j)
              tma_load_3d(sb + j * p.b_box_stride, &tmB, fb, tn * BN + j * ATOM, kb * BK, b);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // Leave no copy in flight.  Fill f of the ring is phase f / STAGES of
      // stage f % STAGES's full barrier.  Without an abort both warps issue
      // the same fills.  After an abort one warp may have issued up to a
      // ring's worth more (it passed an empty barrier the other gave up on
      // just before it completed): once both have stopped, warp 0 arms the
      // stages that received B without an arming, and takes the B bytes that
      // were counted but never issued off the stages it armed, so that every
      // issued copy, and only those, completes its phase; then it waits for
      // the last phase of every stage filled.
      volatile int *fills = reinterpret_cast<volatile int *>(tmem_slot + 3);
      if (lane == 0) fills[copy_a ? 0 : 1] = nfill;
      asm volatile("bar.sync 2, 64;" ::: "memory");  // warps 0 and 6
      if (copy_a) {
        const int nb = fills[1];
        for (int f = nfill; f < nb; ++f) mbar_expect_tx(full0 + 8 * (f % STAGES), B_BYTES);
        for (int f = nb; f < nfill; ++f) mbar_complete_tx(full0 + 8 * (f % STAGES), B_BYTES);
        const int total = max(nfill, nb);
        for (int f = max(0, total - STAGES); f < total; ++f)
          wait_drain(full0 + 8 * (f % STAGES), (uint32_t)(f / STAGES) & 1u, p.err, kErrProducer,
                     kDrainTimeoutNs);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (whole warp)
    {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      // (test hook: a wait that only its limit ends)
      bool ok = !p.stall_wait || warp_wait(stall, 0, abort_flag, p.err, kErrMma, p.timeout_ns);
      for (int u = blockIdx.x; u < p.total_units && ok; u += ustep) {
        int tm, tn, b, sp;
        decode_unit(p, u, tm, tn, b, sp);

        if (!warp_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, p.err, kErrMma,
                       p.timeout_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int nk = unit_kblocks(p, sp);
        for (int i = 0; i < nk; ++i) {
          if (!warp_wait(full0 + 8 * stage, phase, abort_flag, p.err, kErrMma, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          const uint64_t adesc = p.a_desc | (uint64_t)((sa >> 4) & 0x3FFFu);
          const uint64_t bdesc = p.b_desc | (uint64_t)((sb >> 4) & 0x3FFFu);
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk)
            umma<ES>(d_tmem, adesc + (uint64_t)(kk * p.a_kstep), bdesc + (uint64_t)(kk * p.b_kstep),
                     p.idesc, (i > 0 || kk > 0) ? 1u : 0u);
          umma_commit(empty0 + 8 * stage);  // frees the stage when these MMAs finish
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(tfull0 + 8 * acc);  // accumulator ready for the epilogue
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // every MMA this thread issued is complete before TMEM is released
      umma_commit(drain);
      wait_drain(drain, 0, p.err, kErrDrain, kDrainTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t *my_stage = epi_stage + (warp - 2) * 8192;  // two 4 KB boxes
    float *epi_scr = reinterpret_cast<float *>(my_stage);
    int sbuf = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < p.total_units; u += ustep) {
      int tm, tn, b, sp;
      decode_unit(p, u, tm, tn, b, sp);
      if (!warp_wait(tfull0 + 8 * acc, acc_phase, abort_flag, p.err, kErrEpilogue, p.timeout_ns))
        break;
      tc_fence_after();
      const int row0 = tm * BM + q * 32, row = row0 + lane;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      const bool rows_full = row0 + 32 <= p.M && !p.c_trans;
      if (p.c_tma) {
        // 128-byte rows: 32 f32 or 64 16-bit columns per box; lane = row of the box.
        // Split-K partials are f32 boxes of the workspace map, item sp * batch + b.
        const bool f32 = p.splits > 1 || p.tc == MM_F32, bf = p.tc == MM_BF16;
        const int zc = p.splits > 1 ? sp * p.batch + b : b;
        const int cols = f32 ? 32 : 64;
        // Only boxes that start inside C are staged, and each staged box is
        // stored: the wait below counts on every box written since the other
        // buffer's store having committed its own store (a skipped store would
        // let this box be refilled while its store still reads it).
        const int cend = row0 < p.M ? min(BN, p.N - tn * BN) : 0;
#pragma unroll 1
        for (int c = 0; c < cend; c += cols) {
          uint32_t r0[32], r1[32];
          tmem_ld_32cols(tbase + (uint32_t)c, r0);
          if (!f32) tmem_ld_32cols(tbase + (uint32_t)(c + 32), r1);
          tmem_ld_wait();
          if (lane == 0) tma_store_wait_read<1>();  // this box's previous store has read it
          __syncwarp();
          uint8_t *box = my_stage + sbuf * 4096;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint4 v;
            if (f32) {
              v = make_uint4(r0[4 * j], r0[4 * j + 1], r0[4 * j + 2], r0[4 * j + 3]);
            } else {
              const uint32_t *src = j < 4 ? r0 + 8 * j : r1 + 8 * (j - 4);
              uint32_t w[4];
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const float lo = __uint_as_float(src[2 * t]), hi = __uint_as_float(src[2 * t + 1]);
                w[t] = bf ? pack_bf16(lo, hi) : pack_f16(lo, hi);
              }
              v = make_uint4(w[0], w[1], w[2], w[3]);
            }
            // 128-byte swizzle: 16-byte chunk j of row `lane` at j ^ (lane % 8)
            *reinterpret_cast<uint4 *>(box + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0)  // rows and columns past C are clipped by the copy
            tma_store_3d(&tmC, smem_u32(box), tn * BN + c, row0, zc);
          sbuf ^= 1;
        }
      } else
#pragma unroll 1
      for (int c = 0; c < BN / 32; c += 2) {  // two chunks per TMEM wait
        uint32_t r0[32], r1[32];
        tmem_ld_32cols(tbase + (uint32_t)(c * 32), r0);
        tmem_ld_32cols(tbase + (uint32_t)(c * 32 + 32), r1);
        tmem_ld_wait();
        const int col0 = tn * BN + c * 32;
        if (rows_full && col0 + 64 <= p.N) {
          store_chunk_rows(p, b, sp, row0, col0, r0, epi_scr, lane);
          store_chunk_rows(p, b, sp, row0, col0 + 32, r1, epi_scr, lane);
        } else {
          store_chunk(p, b, sp, row, col0, r0);
          store_chunk(p, b, sp, row, col0 + 32, r1);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if (lane == 0) tma_store_wait_all();  // staging boxes stay valid until the stores finish
    __syncwarp();
  }
  // after an abort, B copies may have been issued into stages never armed:
  // give them time to land before shared memory is released
  if (*abort_flag) {
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 100000ull) __nanosleep(1000);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------- cp.async copies of A
// One piece of `BYTES` (8 or 4) bytes from global to shared memory; the bytes
// past `valid` (0..BYTES) are zero-filled and not read.
template <int BYTES>
__device__ __forceinline__ void cp_async_piece(uint32_t dst, const void *src, uint32_t valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], %2, %3;" ::"r"(dst), "l"(src), "n"(BYTES),
               "r"(valid)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// This thread's cp.async groups, all but the newest N, have landed.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// This thread's generic-proxy writes to shared memory (its landed cp.async
// copies) ordered before later async-proxy reads (the tensor cores of either
// CTA of the pair).
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

// 128 rows x 128 bytes of A (K block kb of rows m0..m0+127, K-major) into a
// stage laid out as the 128-byte-swizzled K-major tile the MMA reads (16-byte
// chunk j of row r at r * 128 + ((j ^ (r % 8)) << 4)), by one warp: lane t
// copies piece t % P of rows t / P, t / P + 32 / P, ... (P pieces a row), so
// each copy instruction reads whole 128-byte row segments.  Rows past M and
// bytes past K are zero-filled.
template <int BYTES, int ES>
__device__ __forceinline__ void copy_a_stage(const TcParams &p, uint32_t sa, int m0, int b, int kb,
                                             int t) {
  constexpr int P = 128 / BYTES;  // pieces a row
  const int pi = t % P;
  const int boff = pi * BYTES;     // byte of the piece in the row's 128
  const int64_t kbyte = (int64_t)kb * 128 + boff;
  const int64_t krow = (int64_t)p.K * ES;
  const uint32_t kvalid = kbyte >= krow ? 0u : (uint32_t)(krow - kbyte < BYTES ? krow - kbyte : BYTES);
  const char *base = p.a_ptr + (int64_t)b * p.a_batch_bytes + kbyte;
  const uint32_t chunk = (uint32_t)(boff >> 4), half = (uint32_t)(boff & 15);
#pragma unroll 4
  for (int r = t / P; r < BM; r += 32 / P) {
    const int m = m0 + r;
    const uint32_t valid = m < p.M ? kvalid : 0u;
    const void *src = valid ? base + (int64_t)m * p.a_row_bytes : p.a_ptr;
    const uint32_t dst = sa + (uint32_t)r * 128u + (((chunk ^ (uint32_t)(r & 7)) << 4) | half);
    cp_async_piece<BYTES>(dst, src, valid);
  }
}

// ---------------------------------------------------------------- 2-SM kernel
// The same pipeline on a CTA pair (cluster of 2) with tcgen05.mma.cta_group::2:
// one MMA instruction computes a 256 x BN tile; each CTA holds 128 rows of A
// and half of the B tile (BN/2 columns) in its own shared memory and receives
// its 128 rows of the accumulator (all BN columns) in its own TMEM.  Only the
// pair's even CTA (the leader) issues MMAs.  Both CTAs' TMA loads complete on
// the leader's "full" barrier (tx = both halves); the leader's commits are
// multicast to the "empty" and "tmem full" barriers of both CTAs; both CTAs'
// epilogue warps arrive on the leader's "tmem empty" barrier.  Each SM thus
// loads half as many B bytes per k-block as the single-SM form.  Every CTA
// loads its own operand tiles: no copy is multicast to another CTA.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t nclusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// Shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Warp-collective.
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t leader_bar, int c0, int c1, int c2) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(leader_bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Warp-collective.
__device__ __forceinline__ void tma_load_4d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t leader_bar, int c0, int c1, int c2,
                                                 int c3) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(leader_bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Warp-collective.
template <int ES>
__device__ __forceinline__ void umma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  if constexpr (ES == 2) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}
// Arrive on the barrier at this offset in every CTA of `mask` once every
// tcgen05 op issued so far by the issuing thread has completed.
// Warp-collective.
__device__ __forceinline__ void umma_commit_multicast(uint32_t bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// Warp-collective.
__device__ __forceinline__ void umma_commit_pair_local(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

constexpr uint32_t kPairSlack = 0;  // shared memory reserved after the ring

// Tile geometry of a 2-SM work unit: row tile, first column, batch, width.
__device__ __forceinline__ void pair_unit(const TcParams &p, int u, int bn, int &tm, int &n0,
                                          int &b, int &nw) {
  int t = u, half = -1;
  if (u >= p.full_units) {
    const int v = u - p.full_units;
    t = p.full_units + (v >> 1);
    half = v & 1;
  }
  // grouped order: groups of up to 8 row tiles, rows fastest inside a group,
  // so a wave's A rows and B columns stay within L2 on large problems
  constexpr int GM = 8;
  const int per_b = p.tiles_m * p.tiles_n;
  b = t / per_b;
  int r = t - b * per_b;
  const int g = r / (GM * p.tiles_n);
  const int rows_g = min(GM, p.tiles_m - g * GM);
  r -= g * GM * p.tiles_n;
  tm = g * GM + r % rows_g;
  const int tn = r / rows_g;
  n0 = tn * bn + (half > 0 ? bn / 2 : 0);
  nw = half < 0 ? bn : bn / 2;
}

// AL: A is copied by cp.async (warps 7..10, 128-byte-swizzled as TMA would
// have laid it out) instead of TMA, for rows that TMA cannot address (a
// leading dimension or base that is not a multiple of 16 bytes).  Each CTA's
// copies complete on a local barrier; warp 0 waits for it, fences the writes
// to the async proxy and arrives on the leader's full barrier (which then
// expects the arming, both CTAs' A arrivals and both CTAs' B bytes).
template <int BN, int STAGES, int ES, bool AL>
__global__ void __launch_bounds__(AL ? kTcThreadsAsyncA : kTcThreads, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBh, const TcParams p) {
  pdl_launch_dependents();
  constexpr int BNH = BN / 2;                 // B columns held by each CTA
  // B's smem slot: a whole number of 64-column boxes (BN = 224: two boxes,
  // the last 16 columns of the second unused by the MMA)
  constexpr int BNH_SLOT = (BNH + 63) / 64 * 64;
  constexpr uint32_t A_BYTES = BM * 128;
  constexpr uint32_t B_BYTES = BNH_SLOT * 128;
  constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  constexpr int BK = 128 / ES;
  constexpr int UMMA_K = 32 / ES;
  constexpr int KSTEPS = BK / UMMA_K;
  // two accumulators of BN columns, allocated as a power of two
  constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  constexpr int ATOM = 128 / ES;
  constexpr int PAIR_M = 2 * BM;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES + kPairSlack);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t tfull0 = empty0 + 8 * STAGES;
  const uint32_t tempty0 = tfull0 + 16;
  const uint32_t drain = tempty0 + 16;
  const uint32_t afull0 = drain + 8;  // AL: this CTA's A copies of a stage landed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 5 + (AL ? STAGES : 0));
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t pos = cluster_ctarank();  // position in the pair
  const bool leader = pos == 0;
  const uint16_t pair_mask = 0x3u;
  const int cid = (int)cluster_id_x(), ncl = (int)nclusters_x();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, AL ? 3 : 1);  // (AL: the arming and both CTAs' A relays)
      mbar_init(empty0 + 8 * s, 1);  // one commit from the leader
      if (AL) mbar_init(afull0 + 8 * s, 32);  // the copying warp's lanes
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 8);  // 4 epilogue warps in each CTA of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmBh);
  }
  if ((warp == 0 || warp == 6) && lane == 0 && cid < p.total_units) {
    // the first k-blocks of this CTA's share of its first unit into L2
    int tm, t0, b, w;
    pair_unit(p, cid, BN, tm, t0, b, w);
    const int nh = w / 2;
    const int m0 = tm * PAIR_M + (int)pos * BM;
    const int n0 = t0 + (int)pos * nh;
    const int kb1 = min(p.num_kb, (int)(kPrefetchBytes / STAGE_BYTES));
    for (int kb = 0; kb < kb1; ++kb) {
      if (warp == 0) {
        if (AL) break;  // (the copying warps prefetch A)
        if (!p.a_mn) tma_prefetch_3d(&tmA, kb * BK, m0, b);
        else if (p.a_4d) tma_prefetch_4d(&tmA, 0, kb * BK, m0 / ATOM, b);
        else
          for (int j = 0; j < p.a_boxes; ++j) tma_prefetch_3d(&tmA, m0 + j * ATOM, kb * BK, b);
      } else {
        if (!p.b_mn) tma_prefetch_3d(&tmB, kb * BK, n0, b);  // box of BN/2 columns: covers this share
        else if (p.b_4d && nh == BNH) tma_prefetch_4d(&tmB, 0, kb * BK, n0 / ATOM, b);
        else
          for (int j = 0; j < (nh + ATOM - 1) / ATOM; ++j)
            tma_prefetch_3d(p.b_4d ? &tmBh : &tmB, n0 + j * ATOM, kb * BK, b);
      }
    }
  }
  if (AL && warp >= 7 && cid < p.total_units) {
    // the copying threads prefetch the first K blocks of their rows of the
    // first unit into L2 (whole 16-byte granules inside each row)
    int tm, t0, b, w;
    pair_unit(p, cid, BN, tm, t0, b, w);
    for (int m = tm * PAIR_M + (int)pos * BM + (int)threadIdx.x - 32 * 7;
         m < min(p.M, tm * PAIR_M + ((int)pos + 1) * BM); m += 32 * kCopyWarps) {
      const uintptr_t row = reinterpret_cast<uintptr_t>(p.a_ptr + (int64_t)b * p.a_batch_bytes +
                                                        (int64_t)m * p.a_row_bytes);
      const int64_t pf = (int64_t)(kPrefetchBytes / STAGE_BYTES) * 128, krow = (int64_t)p.K * ES;
      const int64_t len = krow < pf ? krow : pf;
      const uintptr_t lo = (row + 15) & ~(uintptr_t)15, hi = (row + (uintptr_t)len) & ~(uintptr_t)15;
      if (hi > lo) prefetch_l2_bulk(reinterpret_cast<const void *>(lo), (uint32_t)(hi - lo));
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t leader_full0 = map_to_rank(full0, 0);
  const uint32_t leader_tempty0 = map_to_rank(tempty0, 0);
  pdl_wait();  // the prologue above touched no global memory

  if (warp == 0 || warp == 6) {
    // ------------------------------------------------------------ TMA producers (both CTAs)
    // warp 0 arms the stage and copies A, warp 6 copies B; both wait on the
    // same "empty" barrier.  B bytes may land before the arming: the barrier's
    // transaction count goes transiently negative and its single arrival (the
    // arming) still holds the phase open until A has landed too.
    const bool copy_a = warp == 0;
    {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = cid; u < p.total_units && ok; u += ncl) {
        int tm, t0, b, w;
        pair_unit(p, u, BN, tm, t0, b, w);
        const int nh = w / 2;    // B columns this CTA loads for the unit
        const int m0 = tm * PAIR_M + (int)pos * BM;
        const int n0 = t0 + (int)pos * nh;
        // bytes both CTAs' copies bring (an MN-major B comes in whole boxes)
        const uint32_t nh_bytes = (uint32_t)(p.b_mn ? (nh + ATOM - 1) / ATOM * ATOM : nh) * 128;
        const uint32_t tx = 2 * ((AL ? 0u : A_BYTES) + nh_bytes);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!warp_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.err, kErrProducer,
                         p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t lfb = leader_full0 + 8 * stage;
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          if (copy_a) {
            if (leader) mbar_expect_tx(full0 + 8 * stage, tx);
            if (AL) {
              // relay: this CTA's A copies of the stage have landed
              if (!warp_wait(afull0 + 8 * stage, phase, abort_flag, p.err, kErrProducer,
                             p.timeout_ns)) {
                ok = false;
                break;
              }
              if (lane == 0) {
                if (leader)
                  mbar_arrive(full0 + 8 * stage);
                else
                  mbar_arrive_cluster(lfb);
              }
              __syncwarp();
            } else if (!p.a_mn) {
              tma_load_3d_pair(sa, &tmA, lfb, kb * BK, m0, b);
            } else if (p.a_4d) {
              tma_load_4d_pair(sa, &tmA, lfb, 0, kb * BK, m0 / ATOM, b);
            } else {
              for (int j = 0; j < p.a_boxes; ++j)
                tma_load_3d_pair(sa + j * p.a_box_stride, &tmA, lfb, m0 + j * ATOM, kb * BK, b);
            }
          } else if (!p.b_mn) {
            tma_load_3d_pair(sb, w == BN ? &tmB : &tmBh, lfb, kb * BK, n0, b);
          } else if (p.b_4d && nh == BNH) {
            tma_load_4d_pair(sb, &tmB, lfb, 0, kb * BK, n0 / ATOM, b);
          } else {  // with a 4-D map in tmB, tmBh holds the per-box 3-D map
            for (int j = 0; j < (nh + ATOM - 1) / ATOM; ++j)
              tma_load_3d_pair(sb + j * p.b_box_stride, p.b_4d ? &tmBh : &tmB, lfb, n0 + j * ATOM,
                               kb * BK, b);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // the leader's full barriers see both CTAs' copies land
      if (leader && copy_a)
        for (int s = 0; s < STAGES; ++s) {
          int st = (stage + s) % STAGES;
          uint32_t par = (st < stage) ? phase : phase ^ 1;
          wait_drain(full0 + 8 * st, par, p.err, kErrProducer, kDrainTimeoutNs);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader, whole warp)
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int u = cid; u < p.total_units && ok; u += ncl) {
        int tm_, t0_, b_, w;
        pair_unit(p, u, BN, tm_, t0_, b_, w);
        const uint32_t idesc = w == BN ? p.idesc : p.idesc_half;
        if (!warp_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, p.err, kErrMma,
                       p.timeout_ns))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          // (AL: the other CTA's A relay is a release at cluster scope)
          if (!warp_wait<AL>(full0 + 8 * stage, phase, abort_flag, p.err, kErrMma, p.timeout_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
          const uint64_t adesc = p.a_desc | (uint64_t)((sa >> 4) & 0x3FFFu);
          const uint64_t bdesc = p.b_desc | (uint64_t)((sb >> 4) & 0x3FFFu);
#pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk)
            umma_pair<ES>(d_tmem, adesc + (uint64_t)(kk * p.a_kstep),
                          bdesc + (uint64_t)(kk * p.b_kstep), idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          umma_commit_multicast(empty0 + 8 * stage, pair_mask);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit_multicast(tfull0 + 8 * acc, pair_mask);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      umma_commit_pair_local(drain);
      wait_drain(drain, 0, p.err, kErrDrain, kDrainTimeoutNs);
    }
    __syncwarp();
  } else if (AL && warp >= 7) {
    // ------------------------------------------------------------ A copies (both CTAs)
    // Copying warp c takes the fills c, c + kCopyWarps, ... of the ring, one
    // at a time: it copies the fill, waits for its own copies to land, fences
    // its writes to the async proxy and arrives (32 lanes) on the stage's
    // afull barrier.  The fence of a thread orders all of its earlier copies,
    // so a thread never has a later fill's copies in flight when it fences;
    // the warps together keep up to a ring's worth of fills in flight.
    // A parity wait tells only adjacent phases apart: when a warp waits for
    // the stage of fill f (the consumption of fill f - STAGES), its previous
    // fill f - kCopyWarps needed the consumption of f - kCopyWarps - STAGES,
    // which covers fill f - 2 * STAGES only when kCopyWarps <= STAGES; then
    // the stage's barrier is never two phases behind the one awaited.
    static_assert(kCopyWarps <= STAGES, "copy warps may not run more than a ring ahead");
    const int c = warp - 7, t = lane;
    const int nunits = cid < p.total_units ? (p.total_units - 1 - cid) / ncl + 1 : 0;
    const int64_t nfills = (int64_t)nunits * p.num_kb;
    for (int64_t f = c; f < nfills; f += kCopyWarps) {
      const int stage = (int)(f % STAGES);
      const uint32_t phase = (uint32_t)(f / STAGES) & 1u;
      if (!warp_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, p.err, kErrProducer,
                     p.timeout_ns))
        break;
      int tm, t0, b, w;
      pair_unit(p, cid + (int)(f / p.num_kb) * ncl, BN, tm, t0, b, w);
      const int m0 = tm * PAIR_M + (int)pos * BM, kb = (int)(f % p.num_kb);
      const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
      if (p.a_piece == 8)
        copy_a_stage<8, ES>(p, sa, m0, b, kb, t);
      else
        copy_a_stage<4, ES>(p, sa, m0, b, kb, t);
      cp_async_commit();
      cp_async_wait_group<0>();
      fence_proxy_async_all();
      mbar_arrive(afull0 + 8 * stage);
    }
    cp_async_wait_group<0>();  // no copy in flight when shared memory is released
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = cid; u < p.total_units; u += ncl) {
      int tm, t0, b, w;
      pair_unit(p, u, BN, tm, t0, b, w);
      const int nw = w, n0 = t0;
      if (!warp_wait(tfull0 + 8 * acc, acc_phase, abort_flag, p.err, kErrEpilogue, p.timeout_ns))
        break;
      tc_fence_after();
      const int row = tm * PAIR_M + (int)pos * BM + q * 32 + lane;
      const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
      for (int c = 0; c < nw / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32cols(tbase + (uint32_t)(c * 32), r);
        tmem_ld_wait();
        store_chunk(p, b, 0, row, n0 + c * 32, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(leader_tempty0 + 8 * acc);
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  // After an abort, copies issued into stages that were never armed (B copies
  // ahead of the arming) are not covered by the drain above: give any such
  // copy time to land before shared memory is released.
  if (*abort_flag) {
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 100000ull) __nanosleep(1000);
  }
  // the leader's MMAs (reading both CTAs' smem, writing both TMEMs) are done
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// Sum the split-K partials in a fixed order and convert.  G threads (a power
// of two dividing the block) share a group of V consecutive outputs of the
// flattened [batch][M][N] grid: thread g adds the slices of run g,
// [g * run, (g + 1) * run) with run = ceil(S / G), in increasing order, and
// the G run sums are then added in run order.  G comes from the problem shape
// and the SM count only, so every launch of a problem adds the same numbers in
// the same order; G = 1 is the plain s = 0..S-1 sum.  With V = 4 a slice's
// four outputs come in one 16-byte load (the workspace is 16-byte aligned and
// a slice holds a multiple of four floats).  Loads are issued eight at a time
// so their latencies overlap.  RUNS = false is the G = 1 instance: no shared
// memory and no block barrier, so its blocks fit beside a GEMM CTA that holds
// nearly all of an SM's shared memory, are resident early, and start the
// moment the GEMM's partials are complete.
template <bool RUNS, int V>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const float *__restrict__ ws, int S,
                                                            int G, int batch, int M, int N, void *C,
                                                            int tc, int64_t ldc, int64_t sC,
                                                            int c_trans) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ float runs[];  // [V][256], RUNS only
  if (!RUNS) G = 1;
  const int per = 256 / G;  // output groups a block handles per pass
  const int g = threadIdx.x / per, el = threadIdx.x - g * per;
  const int run = (S + G - 1) / G;
  const int q0 = g * run, q1 = min(S, q0 + run);
  const int64_t total = (int64_t)batch * M * N;  // flattened [batch][M][N]
  const int64_t groups = (total + V - 1) / V;
  const bool narrow = total < (1LL << 32);       // 32-bit index arithmetic suffices
  for (int64_t base = (int64_t)blockIdx.x * per; base < groups; base += (int64_t)gridDim.x * per) {
    const int64_t e0 = (base + el) * V;
    float sum[V];
#pragma unroll
    for (int k = 0; k < V; ++k) sum[k] = 0.f;
    if (e0 < total) {
      const float *pq = ws + (int64_t)q0 * total + e0;
      if (V == 4 && e0 + 4 <= total) {
        for (int q = q0; q < q1; q += 8) {
          float4 v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            v[u] = q + u < q1 ? __ldcs(reinterpret_cast<const float4 *>(pq)) : make_float4(0, 0, 0, 0);
            pq += total;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (q + u < q1) {
              sum[0] += v[u].x;
              sum[1 % V] += v[u].y;
              sum[2 % V] += v[u].z;
              sum[3 % V] += v[u].w;
            }
        }
      } else {
        for (int q = q0; q < q1; q += 8) {
          float v[8][V];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
#pragma unroll
            for (int k = 0; k < V; ++k) v[u][k] = q + u < q1 && e0 + k < total ? __ldcs(pq + k) : 0.f;
            pq += total;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (q + u < q1)
#pragma unroll
              for (int k = 0; k < V; ++k) sum[k] += v[u][k];
        }
      }
    }
    if constexpr (RUNS) {
#pragma unroll
      for (int k = 0; k < V; ++k) runs[k * 256 + threadIdx.x] = sum[k];
      __syncthreads();
      if (g == 0)
        for (int r = 1; r < G; ++r)
#pragma unroll
          for (int k = 0; k < V; ++k) sum[k] += runs[k * 256 + r * per + el];
    }
    if (g == 0 && e0 < total) {
      int64_t rg, j;  // row of [batch][M], column of the group's first output
      if (narrow) {
        const uint32_t r32 = (uint32_t)e0 / (uint32_t)N;
        rg = r32;
        j = (uint32_t)e0 - r32 * (uint32_t)N;
      } else {
        rg = e0 / N;
        j = e0 - rg * N;
      }
#pragma unroll
      for (int k = 0; k < V; ++k) {
        if (e0 + k < total) {
          const int64_t b = batch == 1 ? 0 : rg / M, i = rg - b * M;
          store_one(C, tc, c_trans ? b * sC + j * ldc + i : b * sC + i * ldc + j, sum[k]);
        }
        if (++j == N) {
          j = 0;
          ++rg;
        }
      }
    }
    if constexpr (RUNS) __syncthreads();
  }
}

// ---------------------------------------------------------------- host side
struct TcCfg {
  const char *name;
  int bn;       // tile N (for a pair: the pair's tile N, each CTA loads half of B)
  int stages;
  bool splitk;
  bool pair;    // 2-SM (cta_group::2) kernel, tile M = 256
  bool async_a;  // 2-SM kernel with A copied by cp.async (A rows TMA cannot address)
};

// In the tuner's priority order: where a round ends early (a candidate within
// the roofline limit), the earlier entry wins, so the configurations that are
// fastest on large problems come first.
const TcCfg kCfgs[] = {
    {"tc2_256x256_s7", 256, 7, false, true, false},
    // 224 columns: 19 column tiles for N = 4096, so four row tiles of 256
    // make one full wave of 76 pairs (the 1000-row products)
    {"tc2_256x224_s7", 224, 7, false, true, false},
    {"tc2_256x128_s8", 128, 8, false, true, false},
    // A rows whose leading dimension or base is not a multiple of 16 bytes
    // (lda = 4100 bf16, say), read in place by cp.async: no copy of A
    {"tc2_cpasync_256x256_s7", 256, 7, false, true, true},
    {"tc_128x256_s4", 256, 4, false, false, false},
    {"tc_128x128_s6", 128, 6, false, false, false},
    {"tc_128x64_s8", 64, 8, false, false, false},
    {"tc_splitk_128x128_s7", 128, 7, true, false, false},
    {"tc_splitk_128x64_s8", 64, 8, true, false, false},
};

// 1-SM kernel: the ring, the epilogue staging (split-K configurations stage
// in the ring instead), the barriers and 1 KB of alignment slack.
size_t smem_bytes(int bn, int stages, bool sk) {
  return (size_t)stages * (BM * 128 + bn * 128) + 1024 + (sk ? 0 : kEpiStageBytes) + kBarBytes;
}

size_t smem_bytes_cfg(const TcCfg &c) {
  if (!c.pair) return smem_bytes(c.bn, c.stages, c.splitk);
  return (size_t)c.stages * (BM * 128 + ((c.bn / 2 + 63) / 64 * 64) * 128) + kPairSlack + 1024 + 256;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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
  return fn;
}

CUtensorMapDataType map_dtype(int t) {
  return t == MM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
         : t == MM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
}

// 3-D tiled map over (inner, outer, batch) with the 128-byte swizzle.
mm_status encode_map(CUtensorMap *map, int dtype, const void *base, uint64_t inner, uint64_t outer,
                     uint64_t batch, uint64_t ld_bytes, uint64_t bstride_bytes, uint32_t box_inner,
                     uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return set_error(MM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  cuuint64_t dims[3] = {inner, outer, batch};
  if (batch <= 1) bstride_bytes = ((ld_bytes * outer) + 15) & ~(uint64_t)15;
  cuuint64_t strides[2] = {ld_bytes, bstride_bytes};
  cuuint32_t box[3] = {box_inner, box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, map_dtype(dtype), 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(MM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MM_OK;
}

// 4-D map over an MN-major operand stored as `outer` rows (K) of `inner`
// contiguous elements (M or N): dims (atom, K, inner / atom, batch), so one
// copy brings `nboxes` consecutive atom-wide boxes, laid out in shared memory
// exactly as nboxes separate 3-D boxes.  Needs inner % atom == 0 (an atom never
// crosses the end of a row, so out-of-range atoms still read the fill value).
mm_status encode_map4(CUtensorMap *map, int dtype, const void *base, uint64_t inner,
                      uint64_t outer, uint64_t batch, uint64_t ld_bytes, uint64_t bstride_bytes,
                      uint32_t atom, uint32_t box_k, uint32_t nboxes) {
  auto fn = encode_fn();
  if (!fn) return set_error(MM_ERR_CUDA, "cuTensorMapEncodeTiled unavailable");
  const int es = dtype == MM_F32 ? 4 : 2;
  cuuint64_t dims[4] = {atom, outer, inner / atom, batch};
  if (batch <= 1) bstride_bytes = ((ld_bytes * outer) + 15) & ~(uint64_t)15;
  cuuint64_t strides[3] = {ld_bytes, (uint64_t)atom * es, bstride_bytes};
  cuuint32_t box[4] = {atom, box_k, nboxes, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, map_dtype(dtype), 4, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_error(MM_ERR_CUDA, "cuTensorMapEncodeTiled (4-D) failed (%d)", (int)r);
  return MM_OK;
}

uint64_t smem_desc_bits(uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;  // leading-dimension byte offset
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;  // stride-dimension byte offset
  d |= (uint64_t)1 << 46;                             // descriptor version (tcgen05)
  d |= (uint64_t)2 << 61;                             // 128-byte swizzle
  return d;
}

template <int BN, int STAGES, int ES, bool SK>
mm_status launch_kernel(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc,
                        const TcParams &tp, int grid, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  const size_t smem = smem_bytes(BN, STAGES, SK);
  auto kern = tc_gemm_kernel<BN, STAGES, ES, SK>;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (attr_err != cudaSuccess) return cuda_error(attr_err, "cudaFuncSetAttribute (tc smem)");
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kTcThreads), smem, s, dim3(1), ma, mb, mc, tp);
  if (e != cudaSuccess) return cuda_error(e, "tc_gemm_kernel launch");
  return MM_OK;
}

template <int BN, int STAGES, int ES, bool AL>
struct PairKernel {
  static constexpr int kThreads = AL ? kTcThreadsAsyncA : kTcThreads;
  static cudaLaunchConfig_t config(size_t smem, cudaStream_t s, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t lc = {};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return lc;
  }
  static size_t smem() {
    const TcCfg shape{"", BN, STAGES, false, true, AL};
    return smem_bytes_cfg(shape);
  }
  // Set-up once: shared-memory attribute and how many pairs fit at once.
  static mm_status capacity(int *max_clusters) {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    static int clusters = 0;
    std::call_once(once, [] {
      auto kern = tc2_gemm_kernel<BN, STAGES, ES, AL>;
      err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem());
      if (err == cudaSuccess) {
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t q = config(smem(), nullptr, attr);
        q.gridDim = dim3(2);
        err = cudaOccupancyMaxActiveClusters(&clusters, kern, &q);
      }
    });
    if (err != cudaSuccess) return cuda_error(err, "tc2 kernel set-up");
    if (clusters < 1) return set_error(MM_ERR_UNSUPPORTED, "no cluster of CTA pairs fits on this device");
    *max_clusters = clusters;
    return MM_OK;
  }
  static mm_status launch(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mbh,
                          const TcParams &tp, int clusters, cudaStream_t s) {
    cudaError_t e = launch_pdl(tc2_gemm_kernel<BN, STAGES, ES, AL>, dim3((unsigned)(2 * clusters)),
                               dim3(kThreads), smem(), s, dim3(2), ma, mb, mbh, tp);
    if (e != cudaSuccess) return cuda_error(e, "tc2_gemm_kernel launch");
    return MM_OK;
  }
};

template <int ES>
mm_status pair_capacity(int cfg, int *max_clusters) {
  if (kCfgs[cfg].async_a) return PairKernel<256, 7, ES, true>::capacity(max_clusters);
  if (kCfgs[cfg].bn == 256) return PairKernel<256, 7, ES, false>::capacity(max_clusters);
  if (kCfgs[cfg].bn == 224) return PairKernel<224, 7, ES, false>::capacity(max_clusters);
  return PairKernel<128, 8, ES, false>::capacity(max_clusters);
}

template <int ES>
mm_status dispatch_pair(int cfg, const CUtensorMap &ma, const CUtensorMap &mb,
                        const CUtensorMap &mbh, const TcParams &tp, int clusters,
                        cudaStream_t s) {
  if (kCfgs[cfg].async_a)
    return PairKernel<256, 7, ES, true>::launch(ma, mb, mbh, tp, clusters, s);
  if (kCfgs[cfg].bn == 256) return PairKernel<256, 7, ES, false>::launch(ma, mb, mbh, tp, clusters, s);
  if (kCfgs[cfg].bn == 224) return PairKernel<224, 7, ES, false>::launch(ma, mb, mbh, tp, clusters, s);
  return PairKernel<128, 8, ES, false>::launch(ma, mb, mbh, tp, clusters, s);
}

template <int ES>
mm_status dispatch(int cfg, const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap &mc,
                   const TcParams &tp, int grid, cudaStream_t s) {
  const bool sk = kCfgs[cfg].splitk;
  switch (kCfgs[cfg].bn) {
  case 256: return launch_kernel<256, 4, ES, false>(ma, mb, mc, tp, grid, s);
  case 128:
    return sk ? launch_kernel<128, 7, ES, true>(ma, mb, mc, tp, grid, s)
              : launch_kernel<128, 6, ES, false>(ma, mb, mc, tp, grid, s);
  default:
    return sk ? launch_kernel<64, 8, ES, true>(ma, mb, mc, tp, grid, s)
              : launch_kernel<64, 8, ES, false>(ma, mb, mc, tp, grid, s);
  }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// The largest of 16, 8, 4 (else 2, 1) bytes dividing A's base address and its
// row and batch strides: 16 lets TMA read A, 8 or 4 the cp.async copies.
int a_piece_bytes(const Problem &p) {
  const int es = dtype_bytes(p.ta);
  const uint64_t x = (uint64_t)(uintptr_t)p.A | (uint64_t)(p.lda * es) |
                     (p.batch > 1 ? (uint64_t)(p.sA * es) : 0ull);
  for (int g = 16; g > 1; g /= 2)
    if (x % (uint64_t)g == 0) return g;
  return 1;
}

// The main-loop wait limit of the 1-SM kernels (option wait_limit_us; the
// drain waits keep 2 s, and the 2-SM kernel keeps 2 s throughout).
uint64_t one_sm_wait_limit_ns() {
  const double us = get_options().wait_limit_us;
  return us >= 0 ? (uint64_t)(us * 1000.0) : kWaitTimeoutNs;
}

// Split-K reduction plan: V = 4 outputs a thread when the workspace allows
// 16-byte loads, else 1; G threads a group of V outputs (a power of two
// <= 32), grown while a thread's run is longer than 8 slices and the GPU
// still holds the threads (the run's loads then take one or two trips to L2
// instead of S / 8); about eight blocks of 256 threads an SM.
struct ReducePlan {
  dim3 grid;
  int G, V;
};
ReducePlan reduce_plan(const TcParams &tp, int sms) {
  const int64_t total = (int64_t)tp.batch * tp.M * tp.N;
  const int V = (uintptr_t)tp.ws % 16 == 0 && total % 4 == 0 ? 4 : 1;
  const int64_t groups = ceil_div(total, V);
  int G = 1;
  while (G < 32 && ceil_div(tp.splits, G) > 8 && groups * G * 2 <= (int64_t)sms * 2048) G *= 2;
  const int64_t per = 256 / G;
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(ceil_div(groups, per), (int64_t)sms * 8));
  return {dim3((unsigned)blocks), G, V};
}

// The split-K workspace [splits * batch][M][N] (fp32) as the target of the
// epilogue's bulk-tensor stores, 32 x 32 boxes.  Needs 16-byte aligned rows;
// leaves tp.c_tma at 0 (per-thread stores) otherwise.
mm_status ws_map(CUtensorMap *map, TcParams &tp) {
  const uint64_t row = (uint64_t)tp.N * 4, item = row * (uint64_t)tp.M;
  if ((uintptr_t)tp.ws % 16 || row % 16 || item >= (1ULL << 40)) return MM_OK;
  mm_status st = encode_map(map, MM_F32, tp.ws, tp.N, tp.M, (uint64_t)tp.splits * tp.batch, row,
                            item, 32, 32);
  if (st == MM_OK) tp.c_tma = 1;
  return st;
}

template <bool RUNS, int V>
cudaError_t launch_reduce_t(const ReducePlan &rp, const TcParams &tp, const Problem &p, int c_trans,
                            cudaStream_t s) {
  const size_t smem = RUNS ? (size_t)V * 256 * sizeof(float) : 0;
  return launch_pdl(splitk_reduce_kernel<RUNS, V>, rp.grid, dim3(256), smem, s, dim3(1), tp.ws,
                    tp.splits, rp.G, tp.batch, tp.M, tp.N, p.C, p.tc, p.ldc, p.sC, c_trans);
}

mm_status launch_reduce(const TcParams &tp, int sms, const Problem &p, int c_trans, cudaStream_t s) {
  const ReducePlan rp = reduce_plan(tp, sms);
  cudaError_t e;
  if (rp.G > 1)
    e = rp.V == 4 ? launch_reduce_t<true, 4>(rp, tp, p, c_trans, s)
                  : launch_reduce_t<true, 1>(rp, tp, p, c_trans, s);
  else
    e = rp.V == 4 ? launch_reduce_t<false, 4>(rp, tp, p, c_trans, s)
                  : launch_reduce_t<false, 1>(rp, tp, p, c_trans, s);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "splitk_reduce_kernel launch");
}

// Split count for a split-K configuration: enough units to fill the SMs.
void choose_splits(int64_t tiles, int64_t num_kb, int sms, int *splits, int *kb_per) {
  int64_t s = sms / (tiles > 0 ? tiles : 1);
  if (s < 2) s = 2;
  if (s > num_kb) s = num_kb;
  int64_t per = ceil_div(num_kb, s);
  *kb_per = (int)per;
  *splits = (int)ceil_div(num_kb, per);
}

// Split-K (every CTA one unit): fp32 partials to tp.ws by bulk-tensor stores
// where TMA can describe the workspace, then the reduction kernel, which
// spreads the sums over every SM.  (Adding the partials inside the GEMM's
// grid instead -- by the CTA that finishes a tile's last slice, or by all of
// a tile's CTAs after waiting for one another -- measured slower on every
// split-K shape: the CTAs it keeps resident hold back the next call's CTAs.)
template <int ES>
mm_status run_splitk(const Problem &p, TcParams &tp, int cfg, const CUtensorMap &ma,
                     const CUtensorMap &mb, int sms, int c_trans, cudaStream_t s) {
  CUtensorMap mw = ma;
  mm_status st = ws_map(&mw, tp);
  if (st != MM_OK) return st;
  st = dispatch<ES>(cfg, ma, mb, mw, tp, tp.total_units, s);
  if (st != MM_OK) return st;
  return launch_reduce(tp, sms, p, c_trans, s);
}

}  // namespace

// Split-K launch into a workspace the caller provides (no allocation here).
// Picks the largest split count <= the usual choice whose fp32 partials fit
// in ws_bytes; needs at least two K slices.
mm_status launch_tc_splitk_into(const Problem &p, const DeviceInfo &di, int cfg, float *ws,
                                size_t ws_bytes, int *err, cudaStream_t s) {
  std::string why;
  if (!kCfgs[cfg].splitk) return set_error(MM_ERR_INVALID_ARG, "not a split-K configuration");
  if (!tc_supports(p, di, cfg, &why))
    return set_error(MM_ERR_UNSUPPORTED, "%s: %s", kCfgs[cfg].name, why.c_str());
  const TcCfg &c = kCfgs[cfg];
  const int es = dtype_bytes(p.ta);
  const int bk = 128 / es, atom = 128 / es, umma_k = 32 / es;
  const int bn = c.bn;
  TcParams tp;
  std::memset(&tp, 0, sizeof tp);
  tp.M = (int)p.M;
  tp.N = (int)p.N;
  tp.K = (int)p.K;
  tp.batch = (int)p.batch;
  tp.tiles_m = (int)ceil_div(p.M, BM);
  tp.tiles_n = (int)ceil_div(p.N, bn);
  tp.num_kb = (int)ceil_div(p.K, bk);
  const int64_t tiles = (int64_t)tp.tiles_m * tp.tiles_n * tp.batch;
  choose_splits(tiles, tp.num_kb, di.sms, &tp.splits, &tp.kb_per_split);
  const size_t slice_bytes = (size_t)tp.batch * (size_t)p.M * (size_t)p.N * sizeof(float);
  const int64_t fit = slice_bytes ? (int64_t)(ws_bytes / slice_bytes) : 0;
  if (fit < 2)
    return set_error(MM_ERR_INVALID_ARG,
                     "problem too large for the fixed workspace: two K slices need %zu bytes, "
                     "the workspace holds %zu",
                     2 * slice_bytes, ws_bytes);
  if (tp.splits > fit) {
    int64_t per = ceil_div(tp.num_kb, fit);
    tp.kb_per_split = (int)per;
    tp.splits = (int)ceil_div(tp.num_kb, per);
  }
  if (tp.splits < 2) return set_error(MM_ERR_INVALID_ARG, "split-K needs at least two K slices");
  const int64_t units = tiles * tp.splits;
  if (units >= (1LL << 31)) return set_error(MM_ERR_UNSUPPORTED, "too many work units");
  tp.total_units = (int)units;
  CUtensorMap ma, mb;
  mm_status st;
  if (!p.at)
    st = encode_map(&ma, p.ta, p.A, p.K, p.M, p.batch, p.lda * es, p.sA * es, bk, BM);
  else
    st = encode_map(&ma, p.ta, p.A, p.M, p.K, p.batch, p.lda * es, p.sA * es, atom, bk);
  if (st != MM_OK) return st;
  if (p.bt)
    st = encode_map(&mb, p.tb, p.B, p.K, p.N, p.batch, p.ldb * es, p.sB * es, bk, bn);
  else
    st = encode_map(&mb, p.tb, p.B, p.N, p.K, p.batch, p.ldb * es, p.sB * es, atom, bk);
  if (st != MM_OK) return st;
  tp.C = p.C;
  tp.ldc = p.ldc;
  tp.sC = p.sC;
  tp.tc = p.tc;
  const int ec = dtype_bytes(p.tc);
  tp.c_vec_ok = ((uintptr_t)p.C % 16 == 0) && ((p.ldc * ec) % 16 == 0) &&
                (p.batch <= 1 || (p.sC * ec) % 16 == 0);
  tp.err = err;
  tp.timeout_ns = one_sm_wait_limit_ns();
  tp.stall_wait = get_options().wait_stall;
  tp.a_mn = p.at ? 1 : 0;
  tp.b_mn = p.bt ? 0 : 1;
  const uint32_t fmt = p.ta == MM_F16 ? 0u : p.ta == MM_BF16 ? 1u : 2u;
  tp.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)tp.a_mn << 15) |
             ((uint32_t)tp.b_mn << 16) | ((uint32_t)(bn >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
  const uint32_t mn_atom_bytes = (uint32_t)bk * 128u;
  tp.a_desc = tp.a_mn ? smem_desc_bits(mn_atom_bytes, 1024) : smem_desc_bits(16, 1024);
  tp.b_desc = tp.b_mn ? smem_desc_bits(mn_atom_bytes, 1024) : smem_desc_bits(16, 1024);
  tp.a_kstep = tp.a_mn ? (uint32_t)(umma_k * 128) >> 4 : 32u >> 4;
  tp.b_kstep = tp.b_mn ? (uint32_t)(umma_k * 128) >> 4 : 32u >> 4;
  tp.a_boxes = tp.a_mn ? BM / atom : 1;
  tp.b_boxes = tp.b_mn ? bn / atom : 1;
  tp.a_box_stride = mn_atom_bytes;
  tp.b_box_stride = mn_atom_bytes;
  tp.ws = ws;
  return es == 2 ? run_splitk<2>(p, tp, cfg, ma, mb, di.sms, 0, s)
                 : run_splitk<4>(p, tp, cfg, ma, mb, di.sms, 0, s);
}

int tc_config_index(const char *name) {
  for (int i = 0; i < tc_config_count(); ++i)
    if (std::strcmp(kCfgs[i].name, name) == 0) return i;
  return -1;
}

int tc_config_count() { return (int)(sizeof kCfgs / sizeof kCfgs[0]); }
const char *tc_config_name(int cfg) { return kCfgs[cfg].name; }
bool tc_config_is_splitk(int cfg) { return kCfgs[cfg].splitk; }

bool tc_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why) {
  auto no = [&](const char *w) {
    if (why) *why = w;
    return false;
  };
  const TcCfg &c = kCfgs[cfg];
  if (d.cc_major != 10 || d.cc_minor != 3) return no("needs an sm_103 device");
  if (p.ta != p.tb) return no("A and B must have the same type");
  if (p.M < 1 || p.N < 1 || p.K < 1) return no("empty problem");
  if (p.M >= (1LL << 31) || p.N >= (1LL << 31) || p.K >= (1LL << 31) || p.batch >= (1LL << 31))
    return no("dimension too large");
  const int es = dtype_bytes(p.ta);
  if (es == 4 && (p.at || !p.bt)) return no("f32 (tf32) needs K-major A and B (layout NT)");
  if (p.batch > 1 && (p.sA <= 0 || p.sB <= 0)) return no("zero batch stride");
  if (c.async_a) {
    if (p.at) return no("A must be stored row-major (K-major) for the cp.async copies");
    if (a_piece_bytes(p) == 16) return no("A is TMA-aligned: the plain configuration applies");
    if (a_piece_bytes(p) < 4) return no("A rows not 4-byte aligned");
    if ((p.K * es) % a_piece_bytes(p)) return no("K * element size not a multiple of the copy piece");
  } else {
    if ((uintptr_t)p.A % 16) return no("A not 16-byte aligned");
    if ((p.lda * es) % 16) return no("lda not a multiple of 16 bytes (TMA stride rule)");
    if (p.batch > 1 && (p.sA * es) % 16) return no("A batch stride not a multiple of 16 bytes");
  }
  if ((uintptr_t)p.B % 16) return no("B not 16-byte aligned");
  if ((p.ldb * es) % 16) return no("ldb not a multiple of 16 bytes (TMA stride rule)");
  if (p.batch > 1 && (p.sB * es) % 16) return no("B batch stride not a multiple of 16 bytes");
  if (p.lda * es >= (1LL << 40) || p.ldb * es >= (1LL << 40) || p.sA * es >= (1LL << 40) ||
      p.sB * es >= (1LL << 40))
    return no("stride too large for TMA");
  if ((int64_t)smem_bytes_cfg(c) > d.smem_optin) return no("not enough shared memory");
  if (c.splitk) {
    const int64_t num_kb = ceil_div(p.K, 128 / es);
    if (num_kb < 2) return no("split-K needs at least two K blocks");
  }
  return true;
}

namespace {
mm_status launch_tc_impl(const Problem &p, LaunchCtx &ctx, int cfg, bool c_trans);
}

mm_status launch_tc(const Problem &p, LaunchCtx &ctx, int cfg) {
  return launch_tc_impl(p, ctx, cfg, false);
}

// C^T = B^T A^T: the problem with the operands exchanged and M, N swapped;
// C keeps its place and is written transposed.
Problem swap_problem(const Problem &p) {
  Problem q = p;
  q.A = p.B;
  q.ta = p.tb;
  q.at = !p.bt;
  q.lda = p.ldb;
  q.sA = p.sB;
  q.B = p.A;
  q.tb = p.ta;
  q.bt = !p.at;
  q.ldb = p.lda;
  q.sB = p.sA;
  q.M = p.N;
  q.N = p.M;
  return q;
}

bool tc_swap_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why) {
  return tc_supports(swap_problem(p), d, cfg, why);
}

mm_status launch_tc_swapped(const Problem &p, LaunchCtx &ctx, int cfg) {
  return launch_tc_impl(swap_problem(p), ctx, cfg, true);
}

namespace {
mm_status launch_tc_impl(const Problem &p, LaunchCtx &ctx, int cfg, bool c_trans) {
  std::string why;
  if (!tc_supports(p, ctx.dev->info, cfg, &why))
    return set_error(MM_ERR_UNSUPPORTED, "%s: %s", kCfgs[cfg].name, why.c_str());
  const TcCfg &c = kCfgs[cfg];
  const int es = dtype_bytes(p.ta);
  const int bk = 128 / es, atom = 128 / es, umma_k = 32 / es;
  const int bn = c.bn;
  const int bn_cta = c.pair ? bn / 2 : bn;  // B columns one CTA loads
  const int tile_m = c.pair ? 2 * BM : BM;
  CUtensorMap ma, mb;
  mm_status st;
  // B: logical K x N.  K-major when stored transposed (T), MN-major when N.
  if (p.bt)
    st = encode_map(&mb, p.tb, p.B, p.K, p.N, p.batch, p.ldb * es, p.sB * es, bk, bn_cta);
  else
    st = encode_map(&mb, p.tb, p.B, p.N, p.K, p.batch, p.ldb * es, p.sB * es, atom, bk);
  if (st != MM_OK) return st;
  // A: logical M x K.  K-major when stored row-major (N), MN-major when T;
  // copied by cp.async instead where TMA cannot address its rows (the map
  // argument then only repeats B's)
  if (c.async_a)
    ma = mb;
  else if (!p.at)
    st = encode_map(&ma, p.ta, p.A, p.K, p.M, p.batch, p.lda * es, p.sA * es, bk, BM);
  else
    st = encode_map(&ma, p.ta, p.A, p.M, p.K, p.batch, p.lda * es, p.sA * es, atom, bk);
  if (st != MM_OK) return st;
  // MN-major operands: one 4-D copy per stage instead of one copy per
  // 128-byte-wide box, where the MN extent is a whole number of boxes
  const int a_nbox = BM / atom, b_nbox = bn_cta / atom;
  const bool a_4d = p.at && a_nbox > 1 && p.M % atom == 0;
  const bool b_4d = !p.bt && b_nbox > 1 && p.N % atom == 0;
  const CUtensorMap mb3 = mb;  // per-box map (half-width units of the pair kernel)
  if (a_4d) {
    st = encode_map4(&ma, p.ta, p.A, p.M, p.K, p.batch, p.lda * es, p.sA * es, atom, bk, a_nbox);
    if (st != MM_OK) return st;
  }
  if (b_4d) {
    st = encode_map4(&mb, p.tb, p.B, p.N, p.K, p.batch, p.ldb * es, p.sB * es, atom, bk, b_nbox);
    if (st != MM_OK) return st;
  }

  TcParams tp;
  std::memset(&tp, 0, sizeof tp);
  tp.a_4d = a_4d ? 1 : 0;
  tp.b_4d = b_4d ? 1 : 0;
  tp.c_trans = c_trans ? 1 : 0;
  tp.M = (int)p.M;
  tp.N = (int)p.N;
  tp.K = (int)p.K;
  tp.batch = (int)p.batch;
  tp.tiles_m = (int)ceil_div(p.M, tile_m);
  tp.tiles_n = (int)ceil_div(p.N, bn);
  tp.num_kb = (int)ceil_div(p.K, bk);
  const int64_t tiles = (int64_t)tp.tiles_m * tp.tiles_n * tp.batch;
  if (c.splitk) {
    choose_splits(tiles, tp.num_kb, ctx.dev->info.sms, &tp.splits, &tp.kb_per_split);
  } else {
    tp.splits = 1;
    tp.kb_per_split = tp.num_kb;
  }
  int64_t units = tiles * tp.splits;
  int pair_clusters = 0;
  tp.full_units = (int)std::min<int64_t>(units, (1LL << 31) - 1);
  if (c.pair) {
    st = es == 2 ? pair_capacity<2>(cfg, &pair_clusters) : pair_capacity<4>(cfg, &pair_clusters);
    if (st != MM_OK) return st;
    // split the last partial wave's tiles in half along N when that keeps it
    // within one round (only where a half tile still fills whole TMA boxes)
    const int64_t rem = tiles % pair_clusters;
    if (bn == 256 && tiles > pair_clusters && rem > 0 && 2 * rem <= pair_clusters) {
      tp.full_units = (int)(tiles - rem);
      units = tiles + rem;
    }
  }
  if (units >= (1LL << 31)) return set_error(MM_ERR_UNSUPPORTED, "too many work units");
  tp.total_units = (int)units;
  tp.C = p.C;
  tp.ldc = p.ldc;
  tp.sC = p.sC;
  tp.tc = p.tc;
  const int ec = dtype_bytes(p.tc);
  tp.c_vec_ok = ((uintptr_t)p.C % 16 == 0) && ((p.ldc * ec) % 16 == 0) &&
                (p.batch <= 1 || (p.sC * ec) % 16 == 0);
  tp.err = ctx.dev->d_err;
  tp.timeout_ns = c.pair ? kWaitTimeoutNs : one_sm_wait_limit_ns();
  tp.stall_wait = c.pair ? 0 : get_options().wait_stall;
  if (c.async_a) {
    tp.a_ptr = static_cast<const char *>(p.A);
    tp.a_row_bytes = p.lda * es;
    tp.a_batch_bytes = p.batch > 1 ? p.sA * es : 0;
    tp.a_piece = a_piece_bytes(p);
  }
  tp.a_mn = p.at ? 1 : 0;
  tp.b_mn = p.bt ? 0 : 1;
  const uint32_t fmt = p.ta == MM_F16 ? 0u : p.ta == MM_BF16 ? 1u : 2u;
  const uint32_t idesc_base = (1u << 4)                  // D: f32
                              | (fmt << 7) | (fmt << 10)  // A, B types
                              | ((uint32_t)tp.a_mn << 15) // A major (1 = MN)
                              | ((uint32_t)tp.b_mn << 16) // B major (1 = MN)
                              | ((uint32_t)(tile_m >> 4) << 24);  // M / 16 (256 for a pair)
  tp.idesc = idesc_base | ((uint32_t)(bn >> 3) << 17);             // N / 8
  tp.idesc_half = idesc_base | ((uint32_t)(bn >> 4) << 17);        // N / 16: half width
  // K-major: 8-row groups 1024 B apart, K advances 32 B inside the swizzle row.
  // MN-major: boxes of 128 bytes x bk rows; atoms along MN are bk*128 B apart,
  // 8-row K groups 1024 B apart, K advances umma_k rows (umma_k * 128 B).
  const uint32_t mn_atom_bytes = (uint32_t)bk * 128u;
  tp.a_desc = tp.a_mn ? smem_desc_bits(mn_atom_bytes, 1024) : smem_desc_bits(16, 1024);
  tp.b_desc = tp.b_mn ? smem_desc_bits(mn_atom_bytes, 1024) : smem_desc_bits(16, 1024);
  tp.a_kstep = tp.a_mn ? (uint32_t)(umma_k * 128) >> 4 : 32u >> 4;
  tp.b_kstep = tp.b_mn ? (uint32_t)(umma_k * 128) >> 4 : 32u >> 4;
  tp.a_boxes = tp.a_mn ? BM / atom : 1;
  tp.b_boxes = tp.b_mn ? (bn_cta + atom - 1) / atom : 1;
  tp.a_box_stride = mn_atom_bytes;
  tp.b_box_stride = mn_atom_bytes;
  if (c.pair) {
    // B map for half-width units (K-major B loads bn/4 rows per CTA)
    CUtensorMap mbh = b_4d ? mb3 : mb;
    if (p.bt && tp.full_units < tp.total_units) {
      st = encode_map(&mbh, p.tb, p.B, p.K, p.N, p.batch, p.ldb * es, p.sB * es, bk, bn_cta / 2);
      if (st != MM_OK) return st;
    }
    const int clusters = (int)std::min<int64_t>(units, pair_clusters);
    return es == 2 ? dispatch_pair<2>(cfg, ma, mb, mbh, tp, clusters, ctx.stream)
                   : dispatch_pair<4>(cfg, ma, mb, mbh, tp, clusters, ctx.stream);
  }
  const int sms = ctx.dev->info.sms;
  if (c.splitk) {
    void *w = nullptr;
    size_t ws_bytes = (size_t)tp.splits * tp.batch * (size_t)p.M * p.N * sizeof(float);
    st = get_scratch(*ctx.dev, ctx.stream, SCRATCH_WORKSPACE, ws_bytes, &w);
    if (st != MM_OK) return st;
    tp.ws = static_cast<float *>(w);
    return es == 2 ? run_splitk<2>(p, tp, cfg, ma, mb, sms, tp.c_trans, ctx.stream)
                   : run_splitk<4>(p, tp, cfg, ma, mb, sms, tp.c_trans, ctx.stream);
  }
  const int grid = (int)std::min<int64_t>(units, sms);
  // C by bulk-tensor stores where TMA can describe it, else the per-thread path
  CUtensorMap mc = ma;
  if (!c_trans && (uintptr_t)p.C % 16 == 0 && (p.ldc * ec) % 16 == 0 &&
             (p.batch <= 1 || (p.sC * ec) % 16 == 0) && p.ldc * ec < (1LL << 40) &&
             p.sC * ec < (1LL << 40)) {
    st = encode_map(&mc, p.tc, p.C, p.N, p.M, p.batch, p.ldc * ec, p.sC * ec, 128 / ec, 32);
    if (st != MM_OK) return st;
    tp.c_tma = 1;
  }
  return es == 2 ? dispatch<2>(cfg, ma, mb, mc, tp, grid, ctx.stream)
                 : dispatch<4>(cfg, ma, mb, mc, tp, grid, ctx.stream);
}

}  // namespace

}  // namespace mm
