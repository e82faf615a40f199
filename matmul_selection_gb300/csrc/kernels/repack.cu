// Tensor-core candidates for operands that TMA cannot read in place.
//
// The key's stride factor records when a leading dimension (or base) is not
// 16-byte aligned (e.g. a bf16 lda of 4100: 8200-byte rows, stride factor
// 3); TMA-fed kernels cannot describe such an operand (burn "autotune" page:
// the stride alignment decides whether TMA-style kernels can run).  These
// candidates copy each misaligned operand once per call into library scratch
// with its leading dimension rounded up to 16 bytes, then run a tensor-core
// configuration on the copy.  The copy moves each misaligned operand once
// more through HBM; for the large shapes that need it this is a few percent
// of the product's time, against the naive kernel otherwise left.  The swap
// variant (GEMV group) serves small M: it copies the few rows of A and runs
// the split-K configuration on C^T = B^T A^T.
#include <algorithm>
#include <type_traits>

#include "../common.h"

namespace mm {

namespace {

// Copy `rows` rows of `row_bytes` from a strided source to a strided
// destination, G bytes a piece (G divides every address and size).  Grid y
// walks the rows of all batch items (one division a row), grid x a row's
// pieces; each thread issues its U loads before its U stores.
constexpr int kRepackU = 4;
template <int G>
__global__ void __launch_bounds__(256) repack_kernel(const char *__restrict__ src,
                                                     char *__restrict__ dst, int64_t rows,
                                                     int64_t row_bytes, int64_t src_ld,
                                                     int64_t dst_ld, int64_t batch, int64_t src_bs,
                                                     int64_t dst_bs) {
  pdl_launch_dependents();
  pdl_wait();
  using T = typename std::conditional<
      G == 16, uint4,
      typename std::conditional<G == 8, uint2,
                                typename std::conditional<G == 4, uint32_t, uint16_t>::type>::type>::type;
  const int64_t units = row_bytes / G;
  const int64_t nrows = batch * rows;
  for (int64_t rr = blockIdx.y; rr < nrows; rr += gridDim.y) {
    const int64_t b = rr / rows, r = rr - b * rows;
    const char *s = src + b * src_bs + r * src_ld;
    char *d = dst + b * dst_bs + r * dst_ld;
    for (int64_t u0 = (int64_t)blockIdx.x * (256 * kRepackU) + threadIdx.x; u0 < units;
         u0 += (int64_t)gridDim.x * (256 * kRepackU)) {
      T v[kRepackU];
#pragma unroll
      for (int k = 0; k < kRepackU; ++k) {
        const int64_t u = u0 + k * 256;
        if (u < units) v[k] = *reinterpret_cast<const T *>(s + u * G);
      }
#pragma unroll
      for (int k = 0; k < kRepackU; ++k) {
        const int64_t u = u0 + k * 256;
        if (u < units) *reinterpret_cast<T *>(d + u * G) = v[k];
      }
    }
  }
}

struct RepackCfg {
  const char *name;
  const char *inner;  // tensor-core configuration run on the copies
  bool swap;          // run it on C^T = B^T A^T (small M: a copy of A is cheap)
};
const RepackCfg kRepackCfgs[] = {
    {"tc2_repack_256x256", "tc2_256x256_s7", false},
    {"tc2_repack_256x224", "tc2_256x224_s7", false},
    {"tc_repack_128x128", "tc_128x128_s6", false},
    {"tc_repack_128x64", "tc_128x64_s8", false},
    {"tc_repack_splitk_128x128", "tc_splitk_128x128_s7", false},
    {"tc_repack_splitk_128x64", "tc_splitk_128x64_s8", false},
    {"gemv_swap_tc_repack_splitk_128x64", "tc_splitk_128x64_s8", true},
};

struct Plan {
  bool a, b;               // which operands are copied
  int64_t lda2, ldb2;      // leading dimensions of the copies (elements)
  int64_t sA2, sB2;        // batch strides of the copies (elements)
  size_t bytes_a, bytes_b; // scratch bytes for each copy
  Problem q;               // the problem on the copies (pointers filled at launch)
};

bool aligned16(const void *p, int64_t ld, int64_t bs, int64_t batch, int es) {
  return (uintptr_t)p % 16 == 0 && (ld * es) % 16 == 0 && (batch <= 1 || (bs * es) % 16 == 0);
}

// Rows / row length of an operand as stored.
void storage_shape(int64_t rows_logical, int64_t cols_logical, bool trans, int64_t *rows,
                   int64_t *row_elems) {
  *rows = trans ? cols_logical : rows_logical;
  *row_elems = trans ? rows_logical : cols_logical;
}

Plan make_plan_for(const Problem &p) {
  Plan pl;
  const int es = dtype_bytes(p.ta);
  const int64_t round = 16 / es;
  pl.a = !aligned16(p.A, p.lda, p.sA, p.batch, es);
  pl.b = !aligned16(p.B, p.ldb, p.sB, p.batch, es);
  int64_t ra, ea, rb, eb;
  storage_shape(p.M, p.K, p.at, &ra, &ea);
  storage_shape(p.K, p.N, p.bt, &rb, &eb);
  pl.lda2 = (ea + round - 1) / round * round;
  pl.ldb2 = (eb + round - 1) / round * round;
  pl.sA2 = ra * pl.lda2;
  pl.sB2 = rb * pl.ldb2;
  pl.bytes_a = pl.a ? (size_t)(p.batch * pl.sA2 * es + 256) : 0;
  pl.bytes_b = pl.b ? (size_t)(p.batch * pl.sB2 * es + 256) : 0;
  pl.q = p;
  if (pl.a) {
    pl.q.lda = pl.lda2;
    pl.q.sA = pl.sA2;
  }
  if (pl.b) {
    pl.q.ldb = pl.ldb2;
    pl.q.sB = pl.sB2;
  }
  return pl;
}

int inner_index(int cfg) { return tc_config_index(kRepackCfgs[cfg].inner); }

mm_status repack(const void *src, void *dst, int64_t rows, int64_t row_bytes, int64_t src_ld,
                 int64_t dst_ld, int64_t batch, int64_t src_bs, int64_t dst_bs, int sms,
                 cudaStream_t s) {
  auto ok = [&](int g) {
    return (uintptr_t)src % g == 0 && (uintptr_t)dst % g == 0 && row_bytes % g == 0 &&
           src_ld % g == 0 && dst_ld % g == 0 && (batch <= 1 || (src_bs % g == 0 && dst_bs % g == 0));
  };
  int g = ok(16) ? 16 : ok(8) ? 8 : ok(4) ? 4 : 2;
  // x: enough blocks to cover a row, y: the rows (capped; the kernel strides),
  // about 16 blocks an SM in all
  const int64_t nrows = std::max<int64_t>(1, batch * rows);
  const int64_t per_block = 256LL * kRepackU;
  const int64_t cap = (int64_t)sms * 16;
  int64_t gx = std::max<int64_t>(1, (row_bytes / g + per_block - 1) / per_block);
  gx = std::min<int64_t>(gx, cap);
  const int64_t gy = std::min<int64_t>({nrows, 65535, std::max<int64_t>(1, cap / gx)});
  const char *sp = static_cast<const char *>(src);
  char *dp = static_cast<char *>(dst);
  auto kern = g == 16 ? repack_kernel<16> : g == 8 ? repack_kernel<8> : g == 4 ? repack_kernel<4>
                                                                           : repack_kernel<2>;
  cudaError_t e = launch_pdl(kern, dim3((unsigned)gx, (unsigned)gy), dim3(256), 0, s, dim3(1), sp,
                             dp, rows, row_bytes, src_ld, dst_ld, batch, src_bs, dst_bs);
  return e == cudaSuccess ? MM_OK : cuda_error(e, "repack_kernel launch");
}

}  // namespace

int repack_config_count() { return (int)(sizeof kRepackCfgs / sizeof kRepackCfgs[0]); }
bool repack_config_is_swap(int cfg) { return kRepackCfgs[cfg].swap; }
bool repack_config_is_splitk(int cfg) { return tc_config_is_splitk(inner_index(cfg)); }
const char *repack_config_name(int cfg) { return kRepackCfgs[cfg].name; }

bool repack_supports(const Problem &p, const DeviceInfo &d, int cfg, std::string *why) {
  auto no = [&](const char *w) {
    if (why) *why = w;
    return false;
  };
  if (p.ta != p.tb) return no("A and B must have the same type");
  if (p.M < 1 || p.N < 1 || p.K < 1) return no("empty problem");
  const int es = dtype_bytes(p.ta);
  if (((uintptr_t)p.A | (uintptr_t)p.B) % es) return no("operands not element-aligned");
  Plan pl = make_plan_for(p);
  if (!pl.a && !pl.b) return no("both operands TMA-aligned: the plain configuration applies");
  const int inner = inner_index(cfg);
  if (inner < 0) return no("inner configuration missing");
  // the inner configuration must accept the aligned copies
  Problem q = pl.q;
  static char aligned_dummy[256] __attribute__((aligned(256)));
  if (pl.a) q.A = aligned_dummy;
  if (pl.b) q.B = aligned_dummy;
  return kRepackCfgs[cfg].swap ? tc_swap_supports(q, d, inner, why) : tc_supports(q, d, inner, why);
}

mm_status launch_repack(const Problem &p, LaunchCtx &ctx, int cfg) {
  std::string why;
  if (!repack_supports(p, ctx.dev->info, cfg, &why))
    return set_error(MM_ERR_UNSUPPORTED, "%s: %s", kRepackCfgs[cfg].name, why.c_str());
  Plan pl = make_plan_for(p);
  const int es = dtype_bytes(p.ta);
  void *scr = nullptr;
  mm_status st = get_scratch(*ctx.dev, ctx.stream, SCRATCH_REPACK, pl.bytes_a + pl.bytes_b + 512, &scr);
  if (st != MM_OK) return st;
  char *base = reinterpret_cast<char *>(((uintptr_t)scr + 255) & ~(uintptr_t)255);
  Problem q = pl.q;
  const int sms = ctx.dev->info.sms;
  if (pl.a) {
    int64_t rows, row_elems;
    storage_shape(p.M, p.K, p.at, &rows, &row_elems);
    st = repack(p.A, base, rows, row_elems * es, p.lda * es, pl.lda2 * es, p.batch, p.sA * es,
                pl.sA2 * es, sms, ctx.stream);
    if (st != MM_OK) return st;
    q.A = base;
    base += (pl.bytes_a + 255) & ~(size_t)255;
  }
  if (pl.b) {
    int64_t rows, row_elems;
    storage_shape(p.K, p.N, p.bt, &rows, &row_elems);
    st = repack(p.B, base, rows, row_elems * es, p.ldb * es, pl.ldb2 * es, p.batch, p.sB * es,
                pl.sB2 * es, sms, ctx.stream);
    if (st != MM_OK) return st;
    q.B = base;
  }
  return kRepackCfgs[cfg].swap ? launch_tc_swapped(q, ctx, inner_index(cfg))
                               : launch_tc(q, ctx, inner_index(cfg));
}

}  // namespace mm
