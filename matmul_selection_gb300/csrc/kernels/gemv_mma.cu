// Small-M GEMV on the warp-level tensor-core instruction (mma.sync):
//
//   gemv_n_mma  2 <= M <= 16, B row-major [K][N], A row-major [M][K], A and B
//       both bf16 or both f16.  The product is a single pass over B, so what
//       matters is the stream, not the multiply rate: a CTA of 8 warps owns a
//       column group of 64 columns (128 bytes of every row) and a K slice of
//       whole 16-row chunks; warp w takes the chunks w, w + 8, ... of the
//       slice.  Each chunk (16 rows of B's group, and the 16 x 16 tile of A
//       at the same k, rows past M zero) is copied by cp.async into one of
//       the warp's four shared-memory stages, 128-byte rows with the 16-byte
//       pieces XOR-swizzled by the row, so that ldmatrix reads them without
//       bank conflicts: ldmatrix.trans gives B's "col" fragments, ldmatrix
//       gives A's, and eight m16n8k16 MMAs (fp32 accumulators) cover the
//       chunk's 16 x 64 outputs.  The copies land through the generic proxy
//       and the MMA reads registers, so no proxy fence is needed.  The warps'
//       sums are added in warp order, the CTA's 16 x 64 split sum goes to a
//       workspace, and the CTA that takes a group's last ticket adds the S
//       split sums in split order (as gemv_n_stream): one grid a call.
//       Before its grid dependency wait each CTA prefetches its rows of B
//       into L2, a few tensor-map boxes a CTA.
//
//   gemv_t_mma  the same with B transposed (stored [N][K], each output
//       column a contiguous row of B): a chunk of B is then one 32-row half
//       of the group x 32 k (64 bytes a row, so a copy instruction touches 8
//       rows), stored in shared memory as 64-byte rows with the 16-byte
//       pieces XOR-swizzled by row pair, and read by plain ldmatrix, whose
//       8 x 8 matrices of (n, k) are exactly the MMA's "col" fragments of B;
//       two k steps of 16 a chunk, A's tile 16 x 32 k.  The warps' chunk
//       stride (8) keeps each warp on one half, so a warp accumulates 32
//       columns and the CTA adds the four warps of each half.  B's L2 boxes
//       are 256 k x 8 rows.
//
// A need not be 16-byte aligned: its chunks are copied in 8-byte pieces when
// its base or leading dimension is only 8-byte aligned (lda = 4100 bf16, for
// instance), so a misaligned A needs no copy of its own.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "../common.h"

namespace mm {

namespace {

constexpr int kMmaWarps = 8;
constexpr int kMmaThreads = kMmaWarps * 32;
constexpr int kMmaCW = 64;                       // columns of a group
constexpr int kMmaRowB = kMmaCW * 2;             // bytes of a group's row (16-bit B)
constexpr int kMmaStages = 4;                    // chunks in flight a warp
constexpr int kMmaStageB = 16 * kMmaRowB + 512;  // B's 16 rows, then A's 16 x 32 bytes
constexpr int kMmaMaxSplits = 16;
constexpr size_t kMmaSmem = (size_t)kMmaWarps * kMmaStages * kMmaStageB;
// B transposed: a chunk is 32 rows of n x 32 k (64 bytes a row), then A's 16 x 64 bytes
constexpr int kTRows = 32;
constexpr int kTRowB = 64;
constexpr int kTStageB = kTRows * kTRowB + 16 * kTRowB;
constexpr size_t kMmaSmemT = (size_t)kMmaWarps * kMmaStages * kTStageB;

struct MmaArgs {
  const char *A;
  int64_t lda, sA;  // elements
  const char *B;
  int64_t ldb, sB;
  void *C;
  int tc;
  int64_t ldc, sC;
  int M, N, K, batch;
  int G, S;           // column groups, K splits (in whole 16-row chunks)
  int cq, crem;       // chunks / S and chunks % S: split sp has chunks [sp*cq + min(sp, crem), + cq + (sp < crem))
  float *ws;          // [batch][G][S][16][64] split sums
  unsigned *tickets;  // [batch][G] arrival counters, zero between calls
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// 16 bytes (16-byte aligned source), the bytes past `valid` zero-filled.
__device__ __forceinline__ void cp16(uint32_t dst, const void *src, uint32_t valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid)
               : "memory");
}
// 8 bytes (8-byte aligned source), the bytes past `valid` zero-filled.
__device__ __forceinline__ void cp8(uint32_t dst, const void *src, uint32_t valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;" ::"r"(dst), "l"(src), "r"(valid)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldm_x4(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                       uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
__device__ __forceinline__ void ldm_x4_trans(uint32_t a, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                             uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(a));
}
// D (16 x 8, fp32) += A (16 x 16) . B (16 x 8), 16-bit inputs of type TT.
template <int TT>
__device__ __forceinline__ void mma_16816(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
  if constexpr (TT == MM_BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}
constexpr int kPfRows = 32;  // rows of B an L2 prefetch box covers (a group wide, 4 KB)
constexpr int kPfTK = 256;   // B transposed: a box is 256 k x 8 rows of n (4 KB)
constexpr int kPfTN = 8;
__device__ __forceinline__ void store_out(void *C, int tc, int64_t i, float v) {
  if (tc == MM_F32)
    static_cast<float *>(C)[i] = v;
  else if (tc == MM_BF16)
    static_cast<__nv_bfloat16 *>(C)[i] = __float2bfloat16_rn(v);
  else
    static_cast<__half *>(C)[i] = __float2half_rn(v);
}
__device__ __forceinline__ int clampi(int v, int lo, int hi) { return v < lo ? lo : v > hi ? hi : v; }

// TT: the element type of A and B.  XP: the piece size A is copied in (16 or
// 8 bytes).  STEPS > 0: no warp has more than STEPS chunks, and the chunk
// loop is unrolled STEPS times (a trip count the compiler can see lets it
// schedule the copies and MMAs of consecutive chunks together: 9.96 against
// 10.40 us a call at M = 16, 4096 x 4096, measured back to back); STEPS = 0:
// a loop.  EVEN: every warp has exactly STEPS chunks, all inside K and every
// group inside N (the host checks), so no copy needs a bound.  BT: B is
// stored transposed ([N][K]); its chunks are described at gemv_t_mma above.
template <int TT, int XP, int STEPS, bool EVEN, bool BT>
__global__ void __launch_bounds__(kMmaThreads, 2)
    gemv_mma_kernel(const MmaArgs g, const __grid_constant__ CUtensorMap tmB) {
  pdl_launch_dependents();
  constexpr int NB = (BT ? kTRows : kMmaCW) / 8;  // 8-column blocks a warp accumulates
  constexpr int STB = BT ? kTStageB : kMmaStageB;  // bytes of a stage
  constexpr int AOFF = BT ? kTRows * kTRowB : 16 * kMmaRowB;  // A's tile in a stage
  extern __shared__ __align__(128) uint8_t dsm[];
  __shared__ unsigned last;
  const int b = blockIdx.y;
  const int grp = blockIdx.x / g.S, sp = blockIdx.x - grp * g.S;
  // the first crem splits take one 16-row unit more (no division before the prefetch)
  const int c0 = sp * g.cq + min(sp, g.crem), c1 = c0 + g.cq + (sp < g.crem ? 1 : 0);
  const int col0 = grp * kMmaCW;
  const char *Bb = g.B + (int64_t)b * g.sB * 2;
  const char *Ab = g.A + (int64_t)b * g.sA * 2;
  {  // this CTA's rows of B into L2 before the wait, in boxes of 64 columns x
     // 32 rows (4 KB).  Measured at 4096 x 4096, M = 8 / 16 / 16 with lda =
     // 4100, us a call back to back: one request a row of 128 bytes 9.66 /
     // 9.81 / 9.99; boxes of 256 rows 9.38 / 9.70 / 9.79, 128 rows 9.36 /
     // 9.66 / 9.79, 64 rows 9.31 / 9.65 / 9.68, 32 rows 9.29 / 9.62 / 9.64,
     // 16 rows 9.29 / 9.65 / 9.66
    const int r0 = c0 * 16;
    if constexpr (BT) {  // rows col0 .. col0 + 63 of B's [N][K], k from r0
      const int nbox = ((c1 - c0) * 16 + kPfTK - 1) / kPfTK * (kMmaCW / kPfTN);
      for (int t = (int)threadIdx.x; t < nbox; t += kMmaThreads)
        prefetch_box_l2(&tmB, r0 + (t / (kMmaCW / kPfTN)) * kPfTK, col0 + (t % (kMmaCW / kPfTN)) * kPfTN, b);
    } else {
      const int nbox = ((c1 - c0) * 16 + kPfRows - 1) / kPfRows;
      for (int t = (int)threadIdx.x; t < nbox; t += kMmaThreads)
        prefetch_box_l2(&tmB, col0, r0 + t * kPfRows, b);
    }
  }
  pdl_wait();  // A, the workspace, the tickets and C only after the previous kernel
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the split's chunks: B row-major, one a 16-row unit; B transposed, two a
  // pair of 16-k units (one for each 32-row half of the group; past an odd
  // count's last unit zero-filled).  Warp w takes chunks w, w + 8, ...: with
  // B transposed always the same half, w % 2.
  const int nun = BT ? 2 * ((c1 - c0 + 1) >> 1) : c1 - c0;
  const int mine = EVEN ? STEPS : nun > warp ? (nun - warp + kMmaWarps - 1) / kMmaWarps : 0;
  const int half = warp & 1;
  const int kend = min(g.K, c1 * 16);  // no k past the split is read
  uint8_t *wbase = dsm + (size_t)warp * kMmaStages * STB;
  // a group wholly inside N over whole 16-row units copies B unchecked
  const bool b_whole = EVEN || (col0 + kMmaCW <= g.N && g.K % 16 == 0);
  // copies of the warp's i-th chunk into stage i % kMmaStages (an empty group
  // past the last chunk keeps the wait counts uniform)
  auto issue = [&](int i) {
    if (i < mine) {
      const int c = warp + i * kMmaWarps;  // within the split
      const uint32_t dst = smem_addr(wbase + (size_t)(i % kMmaStages) * STB);
      if constexpr (BT) {
        const int k0 = (c0 + 2 * (c >> 1)) * 16;
        const bool whole = b_whole && (EVEN || k0 + 32 <= kend);
        // B: the half's 32 rows of n x 4 pieces of 8 k (64 bytes, k0 .. k0 +
        // 31); lane: piece lane % 4 of rows lane / 4 + 8 j
        const int p = lane & 3, k = k0 + p * 8;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int row = (lane >> 2) + 8 * j, n = col0 + half * kTRows + row;
          const uint32_t d = dst + row * kTRowB + ((p ^ ((row >> 1) & 3)) << 4);
          if (whole) {
            cp16(d, Bb + ((int64_t)n * g.ldb + k) * 2, 16u);
          } else {
            const int valid = n < g.N ? clampi(kend - k, 0, 8) * 2 : 0;
            cp16(d, valid ? Bb + ((int64_t)n * g.ldb + k) * 2 : g.B, (uint32_t)valid);
          }
        }
        // A: rows below M of the 16 x 64-byte tile at the same k
        if constexpr (XP == 16) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int e = lane + 32 * j, m = e >> 2, q = e & 3, ka = k0 + q * 8;
            if (m < g.M) {
              const int valid = whole ? 16 : clampi(kend - ka, 0, 8) * 2;
              cp16(dst + AOFF + m * kTRowB + ((q ^ ((m >> 1) & 3)) << 4),
                   valid ? Ab + ((int64_t)m * g.lda + ka) * 2 : g.A, (uint32_t)valid);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int e = lane + 32 * j, m = e >> 3, q = e & 7, ka = k0 + q * 4;
            if (m < g.M) {
              const int valid = whole ? 8 : clampi(kend - ka, 0, 4) * 2;
              cp8(dst + AOFF + m * kTRowB + (((q >> 1) ^ ((m >> 1) & 3)) << 4) + (q & 1) * 8,
                  valid ? Ab + ((int64_t)m * g.lda + ka) * 2 : g.A, (uint32_t)valid);
            }
          }
        }
      } else {
        const int cu = c0 + c;  // the 16-row unit
        if (b_whole) {
          // B: 16 rows x 8 pieces; lane: pieces lane % 8 of rows lane / 8 + 4 j
          const char *src = Bb + ((int64_t)(cu * 16 + lane / 8) * g.ldb + col0 + (lane % 8) * 8) * 2;
          const int64_t step4 = 4 * g.ldb * 2;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int row = lane / 8 + 4 * j, piece = lane % 8;
            cp16(dst + row * kMmaRowB + ((piece ^ (row & 7)) << 4), src + j * step4, 16u);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int row = lane / 8 + 4 * j, piece = lane % 8;
            const int r = cu * 16 + row, n = col0 + piece * 8;
            const int valid = r < g.K ? clampi(g.N - n, 0, 8) * 2 : 0;
            const char *src = valid ? Bb + ((int64_t)r * g.ldb + n) * 2 : g.B;
            cp16(dst + row * kMmaRowB + ((piece ^ (row & 7)) << 4), src, (uint32_t)valid);
          }
        }
        // A: rows below M of the 16 x 32-byte tile (k = 16 cu .. + 15), k
        // past K zero
        const int k0 = cu * 16;
        if constexpr (XP == 16) {
          const int m = lane >> 1, h = lane & 1;
          if (m < g.M) {
            const int valid = EVEN ? 16 : clampi(g.K - (k0 + 8 * h), 0, 8) * 2;
            const char *src = valid ? Ab + ((int64_t)m * g.lda + k0 + 8 * h) * 2 : g.A;
            cp16(dst + AOFF + m * 32 + ((h ^ ((m >> 2) & 1)) << 4), src, (uint32_t)valid);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int e = lane + 32 * j, m = e >> 2, q = e & 3, h = q >> 1;
            if (m < g.M) {
              const int valid = EVEN ? 8 : clampi(g.K - (k0 + 4 * q), 0, 4) * 2;
              const char *src = valid ? Ab + ((int64_t)m * g.lda + k0 + 4 * q) * 2 : g.A;
              cp8(dst + AOFF + m * 32 + ((h ^ ((m >> 2) & 1)) << 4) + (q & 1) * 8, src,
                  (uint32_t)valid);
            }
          }
        }
      }
    }
    cp_commit();
  };
  // A's rows from M on (the MMA's rows past the problem) zero in every stage,
  // cleared once here and never copied: whole rows, whatever the swizzle
  if (g.M < 16) {
    constexpr int APIECES = BT ? 16 * kTRowB / 16 : 16 * 32 / 16;  // 16-byte pieces of A's tile
#pragma unroll
    for (int st = 0; st < kMmaStages; ++st)
#pragma unroll
      for (int e = lane; e < APIECES; e += 32) {
        const int m = e / (APIECES / 16);
        if (m >= g.M)
          *reinterpret_cast<uint4 *>(wbase + (size_t)st * STB + AOFF + e * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    __syncwarp();  // ordered before any lane's fragment loads
  }
#pragma unroll
  for (int i = 0; i < kMmaStages - 1; ++i) issue(i);
  float acc[NB][4];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[nb][q] = 0.f;
  // one chunk: its fragments and MMAs
  auto compute = [&](int i) {
    const uint32_t base = smem_addr(wbase + (size_t)(i % kMmaStages) * STB);
    const int mat = lane >> 3, r = lane & 7;
    if constexpr (BT) {
      // two k steps of 16; A's matrices (m 0-7, k lo), (m 8-15, k lo), (m 0-7,
      // k hi), (m 8-15, k hi); B's (block, k lo), (block, k hi), (block + 1,
      // k lo), (block + 1, k hi), rows of n read without a transpose
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        uint32_t a[4];
        {
          const int m = (mat & 1) * 8 + r, q = 2 * s + (mat >> 1);
          ldm_x4(base + AOFF + m * kTRowB + ((q ^ ((m >> 1) & 3)) << 4), a[0], a[1], a[2], a[3]);
        }
#pragma unroll
        for (int nb = 0; nb < NB; nb += 2) {
          const int nrow = (nb + (mat >> 1)) * 8 + r, q = 2 * s + (mat & 1);
          uint32_t b0, b1, b2, b3;
          ldm_x4(base + nrow * kTRowB + ((q ^ ((nrow >> 1) & 3)) << 4), b0, b1, b2, b3);
          mma_16816<TT>(acc[nb], a, b0, b1);
          mma_16816<TT>(acc[nb + 1], a, b2, b3);
        }
      }
    } else {
      // A's fragments: matrices (m 0-7, k 0-7), (m 8-15, k 0-7), (m 0-7, k 8-15), (m 8-15, k 8-15)
      uint32_t a[4];
      {
        const int m = (mat & 1) * 8 + r, h = mat >> 1;
        ldm_x4(base + AOFF + m * 32 + ((h ^ ((m >> 2) & 1)) << 4), a[0], a[1], a[2], a[3]);
      }
      // B's fragments, two column blocks an ldmatrix: matrices (k 0-7, block),
      // (k 8-15, block), (k 0-7, block + 1), (k 8-15, block + 1)
#pragma unroll
      for (int nb = 0; nb < NB; nb += 2) {
        const int krow = (mat & 1) * 8 + r, piece = nb + (mat >> 1);
        uint32_t b0, b1, b2, b3;
        ldm_x4_trans(base + krow * kMmaRowB + ((piece ^ (krow & 7)) << 4), b0, b1, b2, b3);
        mma_16816<TT>(acc[nb], a, b0, b1);
        mma_16816<TT>(acc[nb + 1], a, b2, b3);
      }
    }
  };
  if constexpr (STEPS > 0) {
#pragma unroll
    for (int i = 0; i < STEPS; ++i) {
      issue(i + kMmaStages - 1);
      cp_wait<kMmaStages - 1>();  // this lane's copies of chunk i have landed
      __syncwarp();               // ... and every lane's
      if (i < mine) compute(i);
      __syncwarp();  // every lane done with the stage before it is refilled
    }
  } else {
    for (int i = 0; i < mine; ++i) {
      issue(i + kMmaStages - 1);
      cp_wait<kMmaStages - 1>();
      __syncwarp();
      compute(i);
      __syncwarp();
    }
  }
  cp_wait<0>();
  __syncwarp();
  // the warp's sums into its own stages (no copy is in flight there): all 64
  // columns, or with B transposed its half's 32
  constexpr int PLD = kMmaCW + 1;
  static_assert(kMmaStages * STB >= 16 * PLD * 4, "a warp's sums fit its stages");
  {
    float *pw = reinterpret_cast<float *>(wbase);
    const int gr = lane >> 2, t = lane & 3, cb = BT ? half * kTRows : 0;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      pw[gr * PLD + cb + nb * 8 + 2 * t] = acc[nb][0];
      pw[gr * PLD + cb + nb * 8 + 2 * t + 1] = acc[nb][1];
      pw[(gr + 8) * PLD + cb + nb * 8 + 2 * t] = acc[nb][2];
      pw[(gr + 8) * PLD + cb + nb * 8 + 2 * t + 1] = acc[nb][3];
    }
  }
  __syncthreads();
  // the CTA's sums, warps added in order (with B transposed the four warps
  // of the column's half): 16 x 64 outputs, 4 a thread
  constexpr int OPT = 16 * kMmaCW / kMmaThreads;
  float tv[OPT];
#pragma unroll
  for (int j = 0; j < OPT; ++j) {
    const int o = threadIdx.x + j * kMmaThreads, m = o / kMmaCW, n = o % kMmaCW;
    float s = 0.f;
    if constexpr (BT) {
#pragma unroll
      for (int w = n / kTRows; w < kMmaWarps; w += 2)
        s += reinterpret_cast<const float *>(dsm + (size_t)w * kMmaStages * STB)[m * PLD + n];
    } else {
#pragma unroll
      for (int w = 0; w < kMmaWarps; ++w)
        s += reinterpret_cast<const float *>(dsm + (size_t)w * kMmaStages * STB)[m * PLD + n];
    }
    tv[j] = s;
  }
  auto store = [&](int o, float v) {
    const int m = o / kMmaCW, n = col0 + o % kMmaCW;
    if (m < g.M && (EVEN || n < g.N)) store_out(g.C, g.tc, (int64_t)b * g.sC + (int64_t)m * g.ldc + n, v);
  };
  if (g.S == 1) {
#pragma unroll
    for (int j = 0; j < OPT; ++j) store(threadIdx.x + j * kMmaThreads, tv[j]);
    return;
  }
  const int64_t tile = (int64_t)b * g.G + grp;
  float *ws = g.ws + tile * g.S * (16 * kMmaCW);  // [S][16 * 64] of this group
#pragma unroll
  for (int j = 0; j < OPT; ++j) __stcg(ws + (int64_t)sp * 16 * kMmaCW + threadIdx.x + j * kMmaThreads, tv[j]);
  // The barrier orders every thread's split-sum stores before thread 0's
  // release; thread 0's acquire (in the last CTA) orders the other CTAs'
  // sums before this CTA's loads, which the second barrier extends to all of
  // its threads.
  __syncthreads();
  if (threadIdx.x == 0) last = atom_add_acq_rel(g.tickets + tile) == (unsigned)g.S - 1;
  __syncthreads();
  if (!last) return;
#pragma unroll
  for (int j = 0; j < OPT; ++j) {
    const int o = threadIdx.x + j * kMmaThreads;
    float x[kMmaMaxSplits];
#pragma unroll
    for (int q = 0; q < kMmaMaxSplits; ++q)
      x[q] = q < g.S ? __ldcg(ws + (int64_t)q * 16 * kMmaCW + o) : 0.f;
    float y = x[0];
#pragma unroll
    for (int q = 1; q < kMmaMaxSplits; ++q)
      if (q < g.S) y += x[q];
    store(o, y);
  }
  if (threadIdx.x == 0) g.tickets[tile] = 0;  // ready for the next call on this stream
}

// Column groups and K splits: about two CTAs an SM and no more (a second
// partial round of CTAs measured slower than fewer splits), each split at
// least one chunk a warp.
void mma_plan(int64_t N, int64_t K, int64_t batch, int sms, int *G, int *S) {
  const int64_t g = (N + kMmaCW - 1) / kMmaCW, nch = (K + 15) / 16;
  int64_t s = (2 * (int64_t)sms) / std::max<int64_t>(1, g * batch);
  s = std::min<int64_t>(s, std::min<int64_t>(kMmaMaxSplits, nch / kMmaWarps));
  *G = (int)g;
  *S = (int)std::max<int64_t>(1, s);
}

// Unrolled steps for the most chunks a warp gets: 2, 4, 8 or 16, else 0 (a
// loop).  A split of u 16-row units has u chunks, or with B transposed 2 *
// ceil(u / 2).
int mma_steps(const MmaArgs &g, bool bt) {
  const int nch = (g.K + 15) / 16, per_split = (nch + g.S - 1) / g.S;
  const int chunks = bt ? 2 * ((per_split + 1) / 2) : per_split;
  const int per_warp = (chunks + kMmaWarps - 1) / kMmaWarps;
  return per_warp <= 2 ? 2 : per_warp <= 4 ? 4 : per_warp <= 8 ? 8 : per_warp <= 16 ? 16 : 0;
}

template <bool BT, int TT, int XP, int STEPS, bool EVEN = false>
mm_status launch_mma(const MmaArgs &g, const CUtensorMap &tm, cudaStream_t s) {
  auto kern = gemv_mma_kernel<TT, XP, STEPS, EVEN, BT>;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  constexpr size_t smem = BT ? kMmaSmemT : kMmaSmem;
  std::call_once(once, [&] {
    attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  });
  if (attr != cudaSuccess) return cuda_error(attr, "gemv_mma shared memory attribute");
  cudaError_t e = launch_pdl(kern, dim3((unsigned)(g.G * g.S), (unsigned)g.batch),
                             dim3(kMmaThreads), smem, s, dim3(1), g, tm);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "gemv_mma launch");
}

template <bool BT, int TT, int XP>
mm_status launch_steps(const MmaArgs &g, const CUtensorMap &tm, cudaStream_t s) {
  // every split kMmaWarps * steps whole chunks, every group whole
  const bool even = g.N % kMmaCW == 0 && g.K % 16 == 0 && g.crem == 0 && g.cq % kMmaWarps == 0;
  if (even) switch (g.cq / kMmaWarps) {
    case 2: return launch_mma<BT, TT, XP, 2, true>(g, tm, s);
    case 4: return launch_mma<BT, TT, XP, 4, true>(g, tm, s);
    case 8: return launch_mma<BT, TT, XP, 8, true>(g, tm, s);
    case 16: return launch_mma<BT, TT, XP, 16, true>(g, tm, s);
    default: break;
    }
  switch (mma_steps(g, BT)) {
  case 2: return launch_mma<BT, TT, XP, 2>(g, tm, s);
  case 4: return launch_mma<BT, TT, XP, 4>(g, tm, s);
  case 8: return launch_mma<BT, TT, XP, 8>(g, tm, s);
  case 16: return launch_mma<BT, TT, XP, 16>(g, tm, s);
  default: return launch_mma<BT, TT, XP, 0>(g, tm, s);
  }
}

template <bool BT>
mm_status launch_types(const MmaArgs &g, const CUtensorMap &tm, int ta, bool x16, cudaStream_t s) {
  if (ta == MM_BF16)
    return x16 ? launch_steps<BT, MM_BF16, 16>(g, tm, s) : launch_steps<BT, MM_BF16, 8>(g, tm, s);
  return x16 ? launch_steps<BT, MM_F16, 16>(g, tm, s) : launch_steps<BT, MM_F16, 8>(g, tm, s);
}

const char *const kMmaNames[2] = {"gemv_n_mma", "gemv_t_mma"};  // B row-major, B transposed

}  // namespace

int gemv_mma_config_count() { return 2; }
const char *gemv_mma_config_name(int cfg) { return kMmaNames[cfg]; }

bool gemv_mma_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why) {
  auto no = [&](const char *w) {
    if (why) *why = w;
    return false;
  };
  if (d.cc_major != 10) return no("needs an sm_10x device");
  if (p.at) return no("A must be row-major");
  if (p.bt != (cfg == 1)) return no(cfg == 1 ? "B must be transposed" : "B must be row-major");
  if (p.ta != p.tb || (p.ta != MM_BF16 && p.ta != MM_F16)) return no("A and B: both bf16 or both f16");
  if (p.M < 2 || p.M > 16) return no("M outside [2, 16]");
  if (p.N < 1 || p.K < 1) return no("empty problem");
  if (p.N >= (1LL << 30) || p.K >= (1LL << 30) || p.batch > 65535) return no("too large");
  if ((uintptr_t)p.B % 16 || (p.ldb * 2) % 16 || (p.batch > 1 && (p.sB * 2) % 16))
    return no("B's rows not 16-byte aligned");
  if ((uintptr_t)p.A % 8 || (p.lda * 2) % 8 || (p.batch > 1 && (p.sA * 2) % 8))
    return no("A rows not 8-byte aligned");
  if ((int64_t)d.smem_optin < (int64_t)(cfg == 1 ? kMmaSmemT : kMmaSmem))
    return no("not enough shared memory");
  return true;
}

mm_status launch_gemv_mma(const Problem &p, LaunchCtx &ctx, int cfg) {
  std::string why;
  if (!gemv_mma_supports(p, ctx.dev->info, cfg, &why))
    return set_error(MM_ERR_UNSUPPORTED, "%s: %s", kMmaNames[cfg], why.c_str());
  MmaArgs g;
  std::memset(&g, 0, sizeof g);
  g.A = static_cast<const char *>(p.A);
  g.lda = p.lda;
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
  mma_plan(p.N, p.K, p.batch, ctx.dev->info.sms, &g.G, &g.S);
  const int nch = (g.K + 15) / 16;
  g.cq = nch / g.S;
  g.crem = nch % g.S;
  if (g.S > 1) {
    const size_t ws_bytes = (size_t)p.batch * g.G * g.S * 16 * kMmaCW * sizeof(float);
    const size_t tickets_bytes = (size_t)p.batch * g.G * sizeof(unsigned);
    void *w = nullptr, *t = nullptr;
    mm_status st = get_scratch(*ctx.dev, ctx.stream, SCRATCH_WORKSPACE, ws_bytes, &w);
    if (st != MM_OK) return st;
    st = get_scratch(*ctx.dev, ctx.stream, SCRATCH_TICKETS, tickets_bytes, &t);
    if (st != MM_OK) return st;
    g.ws = static_cast<float *>(w);
    g.tickets = static_cast<unsigned *>(t);
  }
  const bool x16 = (uintptr_t)p.A % 16 == 0 && (p.lda * 2) % 16 == 0 &&
                   (p.batch == 1 || (p.sA * 2) % 16 == 0);
  // B, for the L2 prefetch boxes: [K][N] in boxes a group wide, or [N][K]
  // in boxes of 256 k x 8 rows
  alignas(64) CUtensorMap tm;
  const bool bt = cfg == 1;
  mm_status st = bt ? encode_prefetch_map(&tm, p.tb, p.B, (uint64_t)p.K, (uint64_t)p.N,
                                          (uint64_t)p.batch, (uint64_t)p.ldb * 2,
                                          (uint64_t)p.sB * 2, kPfTK, kPfTN)
                    : encode_prefetch_map(&tm, p.tb, p.B, (uint64_t)p.N, (uint64_t)p.K,
                                          (uint64_t)p.batch, (uint64_t)p.ldb * 2,
                                          (uint64_t)p.sB * 2, kMmaCW, kPfRows);
  if (st != MM_OK) return st;
  return bt ? launch_types<true>(g, tm, p.ta, x16, ctx.stream)
            : launch_types<false>(g, tm, p.ta, x16, ctx.stream);
}

}  // namespace mm
