// Tuning key and problem validation.
//
// The key follows the burn "autotune" page, section "tuning key: shape
// bucketing" (cubek's MatmulAutotuneKey = definition + analysis):
//   * m, n, k anchored (Balanced: round up to a power of two; Minimal base
//     2.5, Extensive base 1.5, Full: no bucketing);
//   * pow2 factor: trailing zero bits of the anchored size of the operand's
//     contiguous dimension, at most 4;
//   * stride factor: largest power of two (exponent, at most 10) dividing every
//     non-unit stride in bytes -- real strides, because alignment decides
//     whether TMA-fed kernels can run;
//   * element types; per-operand layout (Contiguous / MildlyPermuted);
//   * analysis: scale from the anchored sizes (< 512 Small, < 2048 Medium,
//     else Large) and the matmul kind.
// The anchored batch count is also part of the key.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <sstream>

#include "common.h"

namespace mm {

static thread_local std::string g_last_error;

mm_status set_error(mm_status s, const char *fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

mm_status cuda_error(cudaError_t e, const char *what) {
  return set_error(MM_ERR_CUDA, "%s failed: %s (%d)", what, cudaGetErrorString(e), (int)e);
}

const char *last_error_cstr() { return g_last_error.c_str(); }

int64_t span_elems(int64_t rows, int64_t cols, int64_t ld, bool trans, int64_t batch,
                   int64_t bstride) {
  if (rows <= 0 || cols <= 0 || batch <= 0) return 0;
  int64_t outer = trans ? cols : rows, inner = trans ? rows : cols;
  int64_t one = (outer - 1) * ld + inner;
  return batch > 1 ? (batch - 1) * bstride + one : one;
}

mm_status make_problem(Problem *p, const void *lhs, const void *rhs, void *out, int64_t M,
                       int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, mm_dtypes dt,
                       mm_layout layout, const mm_batch *batch) {
  if (!p) return set_error(MM_ERR_INVALID_ARG, "null problem");
  if (M < 0 || N < 0 || K < 0) return set_error(MM_ERR_INVALID_ARG, "negative size");
  for (int t : {dt.a, dt.b, dt.c})
    if (t != MM_BF16 && t != MM_F16 && t != MM_F32)
      return set_error(MM_ERR_INVALID_ARG, "unknown dtype %d", t);
  if ((int)layout < 0 || (int)layout > 3)
    return set_error(MM_ERR_INVALID_ARG, "unknown layout %d", (int)layout);
  p->A = lhs;
  p->B = rhs;
  p->C = out;
  p->M = M;
  p->N = N;
  p->K = K;
  p->lda = lda;
  p->ldb = ldb;
  p->ldc = ldc;
  p->ta = dt.a;
  p->tb = dt.b;
  p->tc = dt.c;
  p->at = (layout == MM_TN || layout == MM_TT);
  p->bt = (layout == MM_NT || layout == MM_TT);
  p->batch = batch ? batch->batch : 1;
  p->sA = batch ? batch->stride_a : 0;
  p->sB = batch ? batch->stride_b : 0;
  p->sC = batch ? batch->stride_c : 0;
  if (p->batch < 0) return set_error(MM_ERR_INVALID_ARG, "negative batch");
  if (p->sA < 0 || p->sB < 0 || p->sC < 0)
    return set_error(MM_ERR_INVALID_ARG, "negative batch stride");
  // leading dimensions must cover the contiguous extent
  int64_t a_inner = p->at ? M : K, b_inner = p->bt ? K : N;
  if (lda < (a_inner > 1 ? a_inner : 1) || ldb < (b_inner > 1 ? b_inner : 1) ||
      ldc < (N > 1 ? N : 1))
    return set_error(MM_ERR_INVALID_ARG,
                     "leading dimension too small (lda=%lld ldb=%lld ldc=%lld for M=%lld N=%lld "
                     "K=%lld layout=%d)",
                     (long long)lda, (long long)ldb, (long long)ldc, (long long)M, (long long)N,
                     (long long)K, (int)layout);
  if (p->batch > 1) {
    // output items must not overlap each other (inputs may, e.g. broadcast B)
    int64_t one_c = span_elems(M, N, ldc, false, 1, 0);
    if (p->sC < one_c && M > 0 && N > 0)
      return set_error(MM_ERR_INVALID_ARG, "stride_c %lld smaller than one output (%lld)",
                       (long long)p->sC, (long long)one_c);
  }
  bool empty = (M == 0 || N == 0 || p->batch == 0);
  if (!empty && !out) return set_error(MM_ERR_INVALID_ARG, "null output");
  if (!empty && K > 0 && (!lhs || !rhs)) return set_error(MM_ERR_INVALID_ARG, "null input");
  // every kernel reads and writes whole elements: an operand must start on a
  // multiple of its element size
  if ((uintptr_t)lhs % dtype_bytes(p->ta) || (uintptr_t)rhs % dtype_bytes(p->tb) ||
      (uintptr_t)out % dtype_bytes(p->tc))
    return set_error(MM_ERR_INVALID_ARG, "operand pointer not aligned to its element size");
  return MM_OK;
}

uint64_t anchor(uint64_t x, int level) {
  if (level == LEVEL_FULL || x <= 1) return x;
  double base = level == LEVEL_MINIMAL ? 2.5 : level == LEVEL_EXTENSIVE ? 1.5 : 2.0;
  double p = 1.0;
  while (p < (double)x) p *= base;
  return (uint64_t)std::ceil(p);
}

static int trailing_zeros(uint64_t v, int cap) {
  if (v == 0) return cap;
  int n = 0;
  while ((v & 1) == 0 && n < cap) {
    v >>= 1;
    ++n;
  }
  return n;
}

static uint8_t layout_of(bool trans, bool batch_swap) {
  if (!trans && !batch_swap) return LAYOUT_CONTIGUOUS;
  if (trans && !batch_swap) return LAYOUT_MP_T;
  if (!trans) return LAYOUT_MP_B;
  return LAYOUT_MP_TB;
}

KeyPod make_key(const Problem &p, int level) {
  KeyPod k;
  std::memset(&k, 0, sizeof k);
  k.m = anchor((uint64_t)p.M, level);
  k.n = anchor((uint64_t)p.N, level);
  k.k = anchor((uint64_t)p.K, level);
  k.batch = anchor((uint64_t)p.batch, level);
  // contiguous dimension of each operand
  k.lhs_pow2 = (uint8_t)trailing_zeros(p.at ? k.m : k.k, 4);
  k.rhs_pow2 = (uint8_t)trailing_zeros(p.bt ? k.k : k.n, 4);
  int ea = dtype_bytes(p.ta), eb = dtype_bytes(p.tb);
  int fa = trailing_zeros((uint64_t)(p.lda * ea), 10);
  int fb = trailing_zeros((uint64_t)(p.ldb * eb), 10);
  if (p.batch > 1) {
    int ga = trailing_zeros((uint64_t)(p.sA * ea), 10);
    int gb = trailing_zeros((uint64_t)(p.sB * eb), 10);
    fa = ga < fa ? ga : fa;
    fb = gb < fb ? gb : fb;
  }
  k.lhs_stride = (uint8_t)fa;
  k.rhs_stride = (uint8_t)fb;
  k.elem_lhs = (uint8_t)p.ta;
  k.elem_rhs = (uint8_t)p.tb;
  k.elem_out = (uint8_t)p.tc;
  bool a_swap = p.batch > 1 && p.sA < span_elems(p.M, p.K, p.lda, p.at, 1, 0);
  bool b_swap = p.batch > 1 && p.sB < span_elems(p.K, p.N, p.ldb, p.bt, 1, 0);
  k.layout_lhs = layout_of(p.at, a_swap);
  k.layout_rhs = layout_of(p.bt, b_swap);
  if (k.m < 512 && k.n < 512 && k.k < 512)
    k.scale = SCALE_SMALL;
  else if (k.m < 2048 && k.n < 2048 && k.k < 2048)
    k.scale = SCALE_MEDIUM;
  else
    k.scale = SCALE_LARGE;
  if (k.m == 1 && k.n == 1)
    k.kind = KIND_INNER;
  else if (k.k == 1 && k.m == 1)
    k.kind = KIND_SCALARVEC;
  else if (k.k == 1 && k.n == 1)
    k.kind = KIND_VECSCALAR;
  else if (k.k == 1)
    k.kind = KIND_OUTER;
  else if (k.m == 1)
    k.kind = KIND_VECMAT;
  else if (k.n == 1)
    k.kind = KIND_MATVEC;
  else
    k.kind = KIND_GENERAL;
  return k;
}

static const char *kLayoutNames[] = {
    "Contiguous", "MildlyPermuted{transposed:true,batch_swap:false}",
    "MildlyPermuted{transposed:false,batch_swap:true}",
    "MildlyPermuted{transposed:true,batch_swap:true}", "HighlyPermuted"};
static const char *kScaleNames[] = {"Small", "Medium", "Large"};
static const char *kDtypeNames[] = {"bf16", "f16", "f32"};
static const char *kKindNames[] = {"General",   "MatVec",       "VecMat",      "ScalarVec",
                                   "VecScalar", "InnerProduct", "OuterProduct"};

std::string key_text(const KeyPod &k) {
  char buf[512];
  snprintf(buf, sizeof buf,
           "m=%llu n=%llu k=%llu batch=%llu lhs_pow2=%u lhs_stride=%u rhs_pow2=%u rhs_stride=%u "
           "elem_lhs=%s elem_rhs=%s elem_out=%s layout_lhs=%s layout_rhs=%s scale=%s kind=%s",
           (unsigned long long)k.m, (unsigned long long)k.n, (unsigned long long)k.k,
           (unsigned long long)k.batch, k.lhs_pow2, k.lhs_stride, k.rhs_pow2, k.rhs_stride,
           dtype_name(k.elem_lhs), dtype_name(k.elem_rhs), dtype_name(k.elem_out),
           kLayoutNames[k.layout_lhs < 5 ? k.layout_lhs : 4],
           kLayoutNames[k.layout_rhs < 5 ? k.layout_rhs : 4], kScaleNames[k.scale < 3 ? k.scale : 2],
           kKindNames[k.kind < 7 ? k.kind : 0]);
  return buf;
}

static int index_of(const char *const *names, int n, const std::string &v) {
  for (int i = 0; i < n; ++i)
    if (v == names[i]) return i;
  return -1;
}

bool parse_key_text(const std::string &s, KeyPod *out) {
  KeyPod k;
  std::memset(&k, 0, sizeof k);
  std::istringstream is(s);
  std::string tok;
  int seen = 0;
  while (is >> tok) {
    size_t eq = tok.find('=');
    if (eq == std::string::npos) return false;
    std::string f = tok.substr(0, eq), v = tok.substr(eq + 1);
    auto num = [&](uint64_t *dst) {
      char *end = nullptr;
      unsigned long long x = strtoull(v.c_str(), &end, 10);
      if (!end || *end) return false;
      *dst = x;
      return true;
    };
    auto small = [&](uint8_t *dst) {
      uint64_t x;
      if (!num(&x) || x > 255) return false;
      *dst = (uint8_t)x;
      return true;
    };
    auto dty = [&](uint8_t *dst) {
      int i = index_of(kDtypeNames, 3, v);
      if (i < 0) return false;
      *dst = (uint8_t)i;
      return true;
    };
    bool ok;
    if (f == "m") ok = num(&k.m);
    else if (f == "n") ok = num(&k.n);
    else if (f == "k") ok = num(&k.k);
    else if (f == "batch") ok = num(&k.batch);
    else if (f == "lhs_pow2") ok = small(&k.lhs_pow2);
    else if (f == "lhs_stride") ok = small(&k.lhs_stride);
    else if (f == "rhs_pow2") ok = small(&k.rhs_pow2);
    else if (f == "rhs_stride") ok = small(&k.rhs_stride);
    else if (f == "elem_lhs") ok = dty(&k.elem_lhs);
    else if (f == "elem_rhs") ok = dty(&k.elem_rhs);
    else if (f == "elem_out") ok = dty(&k.elem_out);
    else if (f == "layout_lhs" || f == "layout_rhs") {
      int i = index_of(kLayoutNames, 5, v);
      ok = i >= 0;
      if (ok) (f == "layout_lhs" ? k.layout_lhs : k.layout_rhs) = (uint8_t)i;
    } else if (f == "scale") {
      int i = index_of(kScaleNames, 3, v);
      ok = i >= 0;
      if (ok) k.scale = (uint8_t)i;
    } else if (f == "kind") {
      int i = index_of(kKindNames, 7, v);
      ok = i >= 0;
      if (ok) k.kind = (uint8_t)i;
    } else
      ok = false;
    if (!ok) return false;
    ++seen;
  }
  if (seen != 15) return false;
  *out = k;
  return true;
}

size_t KeyHash::operator()(const KeyPod &k) const {
  // FNV-1a over the 64 bytes
  const uint8_t *b = reinterpret_cast<const uint8_t *>(&k);
  uint64_t h = 1469598103934665603ull;
  for (size_t i = 0; i < sizeof k; ++i) {
    h ^= b[i];
    h *= 1099511628211ull;
  }
  return (size_t)h;
}

}  // namespace mm
