// extern "C" entry points declared in include/mm.h.
#include <cstdio>

#include "common.h"

namespace mm {
const char *last_error_cstr();
}

using namespace mm;

extern "C" {

const char *mm_last_error(void) { return last_error_cstr(); }

const char *mm_version(void) {
#ifndef MM_BUILD_ID
#define MM_BUILD_ID "dev"
#endif
  static const std::string v = std::string(kVersion) + "+" + MM_BUILD_ID;
  return v.c_str();
}

mm_status mm_tune_key(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                      mm_dtypes dt, mm_layout layout, const mm_batch *batch, mm_key *out,
                      char *text, size_t text_cap) {
  if (!out) return set_error(MM_ERR_INVALID_ARG, "null key output");
  Problem p;
  // no data pointers are needed for a key: validate with a dummy output
  static char dummy[16] __attribute__((aligned(16)));
  mm_status st = make_problem(&p, dummy, dummy, dummy, M, N, K, lda, ldb, ldc, dt, layout, batch);
  if (st != MM_OK) return st;
  KeyPod k = make_key(p, get_options().level);
  std::memcpy(out->bytes, &k, sizeof k);
  if (text && text_cap) {
    std::string t = key_text(k);
    size_t n = t.size() < text_cap - 1 ? t.size() : text_cap - 1;
    std::memcpy(text, t.data(), n);
    text[n] = 0;
  }
  return MM_OK;
}

mm_status mm_autotune_execute(const void *lhs, const void *rhs, void *out, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, int64_t ldc, mm_dtypes dt,
                              mm_layout layout, const mm_batch *batch, void *stream) {
  Problem p;
  mm_status st = make_problem(&p, lhs, rhs, out, M, N, K, lda, ldb, ldc, dt, layout, batch);
  if (st != MM_OK) return st;
  return autotune_execute(p, (cudaStream_t)stream, nullptr);
}

mm_status mm_autotune_execute_host(const void *lhs, const void *rhs, void *out, int64_t M,
                                   int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                   mm_dtypes dt, mm_layout layout, const mm_batch *batch,
                                   void *stream) {
  Problem p;
  mm_status st = make_problem(&p, lhs, rhs, out, M, N, K, lda, ldb, ldc, dt, layout, batch);
  if (st != MM_OK) return st;
  if (M == 0 || N == 0 || p.batch == 0) return MM_OK;
  DeviceState *ds = nullptr;
  st = current_device(&ds);
  if (st != MM_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  size_t ba = (size_t)span_a(p) * dtype_bytes(p.ta), bb = (size_t)span_b(p) * dtype_bytes(p.tb);
  size_t bc = (size_t)span_c(p) * dtype_bytes(p.tc);
  std::lock_guard<std::mutex> lk(ds->stage_mu);
  if ((st = ds->stage_a.ensure(ba)) != MM_OK) return st;
  if ((st = ds->stage_b.ensure(bb)) != MM_OK) return st;
  if ((st = ds->stage_c.ensure(bc)) != MM_OK) return st;
  if (ba) MM_CUDA_TRY(cudaMemcpyAsync(ds->stage_a.ptr, lhs, ba, cudaMemcpyHostToDevice, s));
  if (bb) MM_CUDA_TRY(cudaMemcpyAsync(ds->stage_b.ptr, rhs, bb, cudaMemcpyHostToDevice, s));
  Problem q = p;
  q.A = ds->stage_a.ptr;
  q.B = ds->stage_b.ptr;
  q.C = ds->stage_c.ptr;
  st = autotune_execute(q, s, nullptr);
  if (st != MM_OK) return st;
  // copy back only the logical rows, so the caller's padding is untouched
  size_t es = dtype_bytes(p.tc);
  size_t width = (size_t)N * es, pitch = (size_t)ldc * es;
  if (p.batch == 1 || p.sC == M * ldc) {
    MM_CUDA_TRY(cudaMemcpy2DAsync(out, pitch, ds->stage_c.ptr, pitch, width,
                                  (size_t)(M * p.batch), cudaMemcpyDeviceToHost, s));
  } else {
    for (int64_t b = 0; b < p.batch; ++b)
      MM_CUDA_TRY(cudaMemcpy2DAsync((char *)out + b * p.sC * es, pitch,
                                    (char *)ds->stage_c.ptr + b * p.sC * es, pitch, width,
                                    (size_t)M, cudaMemcpyDeviceToHost, s));
  }
  MM_CUDA_TRY(cudaStreamSynchronize(s));
  return MM_OK;
}

mm_status mm_cache_load(const char *path) {
  DeviceState *ds = nullptr;
  mm_status st = current_device(&ds);
  if (st != MM_OK) return st;
  std::string f;
  if (path) {
    f = path;
  } else {
    Options o = get_options();
    if (o.cache_file.empty()) return set_error(MM_ERR_INVALID_ARG, "no path and no cache_file");
    f = device_file_name(o.cache_file, ds->info.ordinal);
  }
  std::lock_guard<std::mutex> tl(ds->tune_mu);
  ds->file_loaded = true;
  return cache_load(*ds, f);
}

mm_status mm_cache_save(const char *path) {
  DeviceState *ds = nullptr;
  mm_status st = current_device(&ds);
  if (st != MM_OK) return st;
  std::string f;
  if (path) {
    f = path;
  } else {
    Options o = get_options();
    if (o.cache_file.empty()) return set_error(MM_ERR_INVALID_ARG, "no path and no cache_file");
    f = device_file_name(o.cache_file, ds->info.ordinal);
  }
  return cache_save(*ds, f);
}

mm_status mm_tune_file(const char *path, int *tuned) {
  if (!path || !tuned) return set_error(MM_ERR_INVALID_ARG, "null path or count");
  *tuned = 0;
  DeviceState *ds = nullptr;
  mm_status st = current_device(&ds);
  if (st != MM_OK) return st;
  return tune_file(*ds, path, tuned);
}

mm_status mm_cache_clear(void) {
  DeviceState *ds = nullptr;
  mm_status st = current_device(&ds);
  if (st != MM_OK) return st;
  std::unique_lock<std::shared_mutex> lk(ds->table_mu);
  ds->table.clear();
  ds->dirty = false;
  return MM_OK;
}

int64_t mm_cache_size(void) {
  DeviceState *ds = nullptr;
  if (current_device(&ds) != MM_OK) return -1;
  std::shared_lock<std::shared_mutex> lk(ds->table_mu);
  return (int64_t)ds->table.size();
}

int32_t mm_candidate_count(void) { return (int32_t)registry().size(); }

const char *mm_candidate_name(int32_t index) {
  const auto &r = registry();
  if (index < 0 || index >= (int32_t)r.size()) return nullptr;
  return r[index].name.c_str();
}

uint64_t mm_candidate_launches(int32_t index) { return candidate_launches(index); }

uint64_t mm_candidate_checksum(void) { return registry_checksum(); }

mm_status mm_execute_candidate(int32_t index, const void *lhs, const void *rhs, void *out,
                               int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                               int64_t ldc, mm_dtypes dt, mm_layout layout, const mm_batch *batch,
                               void *stream) {
  Problem p;
  mm_status st = make_problem(&p, lhs, rhs, out, M, N, K, lda, ldb, ldc, dt, layout, batch);
  if (st != MM_OK) return st;
  if (index < 0 || index >= (int32_t)registry().size())
    return set_error(MM_ERR_INVALID_ARG, "candidate index %d out of range", index);
  if (M == 0 || N == 0 || p.batch == 0) return MM_OK;
  DeviceState *ds = nullptr;
  st = current_device(&ds);
  if (st != MM_OK) return st;
  LaunchCtx ctx{(cudaStream_t)stream, ds, false};
  if (K == 0 && index != 0) {
    std::string why;
    if (!registry()[index].supports(p, ds->info, registry()[index].cfg, &why))
      return set_error(MM_ERR_UNSUPPORTED, "%s: %s", registry()[index].name.c_str(), why.c_str());
  }
  return launch_candidate(index, p, ctx);
}

mm_status mm_lookup(const mm_key *key, int32_t *index) {
  if (!key || !index) return set_error(MM_ERR_INVALID_ARG, "null argument");
  *index = -1;
  DeviceState *ds = nullptr;
  mm_status st = current_device(&ds);
  if (st != MM_OK) return st;
  KeyPod k;
  std::memcpy(&k, key->bytes, sizeof k);
  std::shared_lock<std::shared_mutex> lk(ds->table_mu);
  auto it = ds->table.find(k);
  if (it == ds->table.end()) return set_error(MM_ERR_NOT_FOUND, "key not in the table");
  *index = it->second->winner;
  return MM_OK;
}

int32_t mm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                mm_dtypes dt, mm_layout layout, const mm_batch *batch, int32_t cap, int32_t *cand,
                int32_t *group, int32_t *tier, int32_t *supported, int32_t *group_prio,
                int32_t *prio) {
  Problem p;
  static char dummy[256] __attribute__((aligned(256)));
  if (make_problem(&p, dummy, dummy, dummy, M, N, K, lda, ldb, ldc, dt, layout, batch) != MM_OK)
    return -1;
  DeviceState *ds = nullptr;
  if (current_device(&ds) != MM_OK) return -1;
  auto plan = make_plan(make_key(p, get_options().level), p, ds->info);
  int32_t n = 0;
  for (const auto &it : plan) {
    if (n >= cap) break;
    if (cand) cand[n] = it.cand;
    if (group) group[n] = it.group;
    if (tier) tier[n] = it.tier;
    if (supported) supported[n] = it.supported;
    if (group_prio) group_prio[n] = it.group_prio;
    if (prio) prio[n] = it.prio;
    ++n;
  }
  return n;
}

const char *mm_group_name(int32_t g) { return group_name(g); }

int32_t mm_default_candidate(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                             int64_t ldc, mm_dtypes dt, mm_layout layout, const mm_batch *batch) {
  Problem p;
  static char dummy[256] __attribute__((aligned(256)));
  if (make_problem(&p, dummy, dummy, dummy, M, N, K, lda, ldb, ldc, dt, layout, batch) != MM_OK)
    return -1;
  DeviceState *ds = nullptr;
  if (current_device(&ds) != MM_OK) return -1;
  return default_candidate(make_key(p, get_options().level), p, ds->info);
}

mm_status mm_set_option(const char *name, const char *value) {
  if (!name || !value) return set_error(MM_ERR_INVALID_ARG, "null option name/value");
  return set_option(name, value);
}

mm_status mm_get_option(const char *name, char *buf, size_t cap) {
  if (!name || !buf || !cap) return set_error(MM_ERR_INVALID_ARG, "null argument");
  std::string v;
  mm_status st = get_option(name, &v);
  if (st != MM_OK) return st;
  size_t n = v.size() < cap - 1 ? v.size() : cap - 1;
  std::memcpy(buf, v.data(), n);
  buf[n] = 0;
  return MM_OK;
}

mm_status mm_get_stats(mm_stats *out) {
  if (!out) return set_error(MM_ERR_INVALID_ARG, "null stats");
  StatsAtomic &s = stats();
  out->calls = s.calls.load();
  out->hits = s.hits.load();
  out->misses = s.misses.load();
  out->tunes = s.tunes.load();
  out->launches = s.launches.load();
  out->bench_launches = s.bench_launches.load();
  out->last_tune_ms = s.last_tune_ms.load();
  out->total_tune_ms = s.total_tune_ms.load();
  return MM_OK;
}

void mm_reset_stats(void) {
  StatsAtomic &s = stats();
  s.calls = 0;
  s.hits = 0;
  s.misses = 0;
  s.tunes = 0;
  s.launches = 0;
  s.bench_launches = 0;
  s.last_tune_ms = 0.0;
  s.total_tune_ms = 0.0;
}

void mm_shutdown(void) {
  Options o = get_options();
  if (!o.cache_file.empty() && o.autotune_cache)
    for_each_device([](DeviceState &ds) {
      Options oo = get_options();
      if (ds.dirty) cache_save(ds, device_file_name(oo.cache_file, ds.info.ordinal));
    });
  release_all_devices();
  noalloc_forget_devices();
}

}  // extern "C"
