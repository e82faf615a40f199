// The tuner: table lookup on the warm path, benchmarking on a miss.
//
// Warm path (burn "autotune" page, section "first time a key is met"):
// compute the key, look it up in the in-memory table, launch the recorded
// candidate.  Miss: sync the persistent table, mark the key pending, plan
// the rounds, bound the problem with the roofline, benchmark, record, run.
//
// Benchmark of one candidate merges the page's adaptive rule with
// TunableOp's budget (PyTorch TunableOp guide, section 4):
//   * one untimed warm-up launch (module load, first-touch);
//   * a 3-iteration screening pass: a candidate whose median is more than
//     1.5x the best median so far is dropped;
//   * then iterations until min(max_tuning_iterations, max_tuning_duration)
//     is reached (at least one);
//   * a candidate with 2 samples inside the roofline time limit short-circuits
//     the round: no further candidate of that round is measured;
//   * the fastest MEDIAN wins; ties go to the lower candidate index;
//   * unless the round ended inside the limit, the finalists (medians within
//     10 % of the winner's, at most three) are re-timed in interleaved chunks
//     of 30 calls and the lowest re-timed median is recorded (the winner's curse: the
//     fastest of several noisy medians is biased low).
// Iterations run in chunks (3 for the screening pass, then up to 10), each
// enqueued behind a short delay kernel so that they run back to back on the
// device.  A sample is the mean of a chunk, timed by one pair of events
// around it (as TunableOp times a loop of calls): events between the calls
// would stop a launch from overlapping its predecessor's tail, which is how
// the library's kernels run in a stream.  With the L2 flush on, the flush
// kernels sit between the calls, so each call is then timed on its own.
// Every timed iteration runs on its own rotating copy of the inputs and its
// own private output (TunableOp's rotating buffer; the page's out.copy()), so
// the user's output is never written by tuning and repeated runs do not
// measure a warm L2.  An optional L2 flush runs between iterations, outside
// the timed events.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <fstream>
#include <thread>

#include "common.h"

namespace mm {

namespace {

struct CandResult {
  int index = -1;
  std::string state = "skipped";  // ok, unsupported, error, slow, timeout, numeric, skipped
  std::vector<float> times;       // samples (ms per call)
  int iters = 0;                  // timed calls
  double final_median = NAN;      // finalists: median of the re-timed chunks
  double median = NAN, mean = NAN;
  bool short_circuit = false;
  std::string err;
};

double median_of(std::vector<float> v) {
  if (v.empty()) return NAN;
  std::sort(v.begin(), v.end());
  size_t n = v.size();
  return n % 2 ? v[n / 2] : 0.5 * ((double)v[n / 2 - 1] + (double)v[n / 2]);
}

struct FaultSpec {
  std::string name, mode;
};
FaultSpec parse_fault(const std::string &s) {
  FaultSpec f;
  size_t c = s.rfind(':');
  if (c != std::string::npos) {
    f.name = s.substr(0, c);
    f.mode = s.substr(c + 1);
  }
  return f;
}

// Private copies of the inputs and private outputs used while benchmarking.
struct Rotation {
  std::vector<void *> allocs;
  std::vector<Problem> sets;
  ~Rotation() {
    for (void *p : allocs) cudaFree(p);
  }
};

size_t align_off(const void *p) { return (size_t)((uintptr_t)p & 255u); }

mm_status alloc_like(Rotation &r, const void *src, size_t bytes, void **out) {
  void *base = nullptr;
  cudaError_t e = cudaMalloc(&base, bytes + 256);
  if (e != cudaSuccess) return cuda_error(e, "cudaMalloc (rotating buffer)");
  r.allocs.push_back(base);
  // keep the caller's alignment modulo 256 so that alignment gates agree
  *out = (char *)base + align_off(src);
  return MM_OK;
}

mm_status make_rotation(DeviceState &ds, const Problem &p, const Options &o, Rotation &r) {
  size_t ba = (size_t)span_a(p) * dtype_bytes(p.ta);
  size_t bb = (size_t)span_b(p) * dtype_bytes(p.tb);
  size_t bc = (size_t)span_c(p) * dtype_bytes(p.tc);
  bool rotate = o.rotating_buffer_mb != 0.0;
  size_t set_bytes = (rotate ? ba + bb : 0) + bc + 768;
  double want = o.rotating_buffer_mb < 0 ? 2.0 * (double)ds.info.l2_bytes
                                         : o.rotating_buffer_mb * 1048576.0;
  size_t free_b = 0, total_b = 0;
  cudaMemGetInfo(&free_b, &total_b);
  double cap = std::min((double)free_b * 0.5, 16.0 * (1ull << 30));
  int R = 1;
  if (rotate && set_bytes > 0) {
    R = (int)std::ceil(want / (double)set_bytes);
    R = std::max(1, std::min(R, 64));
    while (R > 1 && (double)R * (double)set_bytes > cap) --R;
  }
  for (int i = 0; i < R; ++i) {
    Problem q = p;
    if (rotate) {
      void *a = nullptr, *b = nullptr;
      mm_status st = alloc_like(r, p.A, ba, &a);
      if (st != MM_OK) return st;
      st = alloc_like(r, p.B, bb, &b);
      if (st != MM_OK) return st;
      MM_CUDA_TRY(cudaMemcpyAsync(a, p.A, ba, cudaMemcpyDeviceToDevice, ds.tune_stream));
      MM_CUDA_TRY(cudaMemcpyAsync(b, p.B, bb, cudaMemcpyDeviceToDevice, ds.tune_stream));
      q.A = a;
      q.B = b;
    }
    void *c = nullptr;
    mm_status st = alloc_like(r, p.C, bc, &c);
    if (st != MM_OK) return st;
    q.C = c;
    r.sets.push_back(q);
  }
  return MM_OK;
}

const char *state_json(const CandResult &r) { return r.state.c_str(); }

}  // namespace

// ---------------------------------------------------------------- peaks
mm_status roofline_peaks(DeviceState &ds, Peaks *out) {
  if (ds.peaks.ready) {
    *out = ds.peaks;
    return MM_OK;
  }
  Options o = get_options();
  Peaks pk;
  cudaStream_t s = ds.tune_stream;
  // compute: the option, else the nominal dense tensor rates of the part
  // (bf16 2.25 PFLOP/s, tf32 1.1 PFLOP/s per GB300); tf32 scaled alike.
  double bf16 = o.peak_tflops > 0 ? o.peak_tflops * 1e12 : 2.25e15;
  pk.bf16_ops = bf16;
  pk.tf32_ops = bf16 * (1.1 / 2.25);
  std::string src = o.peak_tflops > 0 ? "compute=option" : "compute=nominal";
  cudaEvent_t e0, e1;
  MM_CUDA_TRY(cudaEventCreate(&e0));
  MM_CUDA_TRY(cudaEventCreate(&e1));
  // launch overhead: 200 empty launches between two events
  for (int i = 0; i < 20; ++i) launch_empty(s);
  MM_CUDA_TRY(cudaEventRecord(e0, s));
  for (int i = 0; i < 200; ++i) launch_empty(s);
  MM_CUDA_TRY(cudaEventRecord(e1, s));
  MM_CUDA_TRY(cudaEventSynchronize(e1));
  float ms = 0;
  cudaEventElapsedTime(&ms, e0, e1);
  pk.launch_ns = ms * 1e6 / 200.0;
  if (o.peak_gbs > 0) {
    pk.bytes_per_s = o.peak_gbs * 1e9;
    src += ",memory=option";
  } else {
    // bandwidth: best of 5 copies of a buffer of 4 x L2 (read + write bytes)
    size_t bytes = (size_t)std::max<int64_t>(ds.info.l2_bytes * 4, 64 << 20);
    void *a = nullptr, *b = nullptr;
    MM_CUDA_TRY(cudaMalloc(&a, bytes));
    MM_CUDA_TRY(cudaMalloc(&b, bytes));
    cudaMemsetAsync(a, 0, bytes, s);
    float best = 1e30f;
    for (int i = 0; i < 6; ++i) {
      cudaEventRecord(e0, s);
      launch_copy_probe(a, b, bytes, s);
      cudaEventRecord(e1, s);
      cudaEventSynchronize(e1);
      float t = 0;
      cudaEventElapsedTime(&t, e0, e1);
      if (i > 0) best = std::min(best, t);
    }
    cudaFree(a);
    cudaFree(b);
    pk.bytes_per_s = 2.0 * (double)bytes / (best * 1e-3);
    src += ",memory=probe";
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  pk.ready = true;
  pk.source = src;
  ds.peaks = pk;
  *out = pk;
  return MM_OK;
}

// ---------------------------------------------------------------- benchmark
namespace {

struct BenchEnv {
  DeviceState *ds;
  Rotation *rot;
  Options opts;
  FaultSpec fault;
  double limit_ms;
  std::vector<cudaEvent_t> ev;  // 2 per iteration of a chunk
  void *ref = nullptr;          // numerical-check reference output (set 0 layout)
  int *d_bad = nullptr;
  double atol = 0, rtol = 0;
};

// One chunk of `chunk` back-to-back calls of a candidate, timed by one event
// pair; *ms = mean per call.  False when a launch fails or no timing results.
bool time_chunk(int idx, BenchEnv &env, int base, int chunk, float *ms) {
  DeviceState &ds = *env.ds;
  LaunchCtx ctx{ds.tune_stream, &ds, true};
  const int R = (int)env.rot->sets.size();
  launch_delay(40000ull * (unsigned long long)chunk, ds.tune_stream);
  cudaEventRecord(env.ev[0], ds.tune_stream);
  for (int i = 0; i < chunk; ++i)
    if (launch_candidate(idx, env.rot->sets[(base + i) % R], ctx) != MM_OK) return false;
  cudaEventRecord(env.ev[1], ds.tune_stream);
  if (cudaStreamSynchronize(ds.tune_stream) != cudaSuccess) return false;
  float t = NAN;
  if (cudaEventElapsedTime(&t, env.ev[0], env.ev[1]) != cudaSuccess || !(t > 0)) return false;
  t /= (float)chunk;
  if (env.fault.name == registry()[idx].name) {
    if (env.fault.mode == "nan") return false;
    if (env.fault.mode == "slow") t *= 1000.f;
  }
  *ms = t;
  return true;
}

CandResult bench_candidate(int idx, BenchEnv &env, double best_ms) {
  CandResult r;
  r.index = idx;
  const auto &reg = registry();
  DeviceState &ds = *env.ds;
  std::string why;
  if (!reg[idx].supports(env.rot->sets[0], ds.info, reg[idx].cfg, &why)) {
    r.state = "unsupported";
    r.err = why;
    return r;
  }
  LaunchCtx ctx{ds.tune_stream, &ds, true};
  const int R = (int)env.rot->sets.size();
  cudaMemsetAsync(ds.d_err, 0, 64, ds.tune_stream);
  // warm-up
  mm_status st = launch_candidate(idx, env.rot->sets[0], ctx);
  cudaError_t ce = cudaStreamSynchronize(ds.tune_stream);
  if (st != MM_OK || ce != cudaSuccess) {
    r.state = "error";
    r.err = st != MM_OK ? std::string(mm_last_error()) : cudaGetErrorString(ce);
    return r;
  }
  bool faulty = env.fault.name == reg[idx].name;
  if (faulty && env.fault.mode == "stall")  // a slow host-side benchmark (tests the pending wait)
    std::this_thread::sleep_for(std::chrono::milliseconds(1500));
  int n = 0;
  double total = 0;
  int in_limit = 0;
  bool first = true;
  const int max_it = std::max(1, env.opts.max_tuning_iterations);
  while (true) {
    int chunk = first ? std::min(3, max_it) : std::min(10, max_it - n);
    if (chunk <= 0) break;
    // hold the stream while the chunk is enqueued, so its iterations run back
    // to back and the events time the device, not the host's launch latency
    launch_delay(40000ull * (unsigned long long)chunk, ds.tune_stream);
    const bool per_call = env.opts.l2_flush && ds.flush_buf.ptr;
    if (!per_call) cudaEventRecord(env.ev[0], ds.tune_stream);
    for (int i = 0; i < chunk; ++i) {
      const Problem &q = env.rot->sets[(n + i) % R];
      if (per_call) {
        launch_l2_flush(ds.flush_buf.ptr, ds.flush_buf.bytes, ds.tune_stream);
        cudaEventRecord(env.ev[2 * i], ds.tune_stream);
      }
      st = launch_candidate(idx, q, ctx);
      if (per_call) cudaEventRecord(env.ev[2 * i + 1], ds.tune_stream);
      if (st != MM_OK) break;
    }
    if (!per_call) cudaEventRecord(env.ev[1], ds.tune_stream);
    ce = cudaStreamSynchronize(ds.tune_stream);
    if (st != MM_OK || ce != cudaSuccess) {
      r.state = "error";
      r.err = st != MM_OK ? std::string(mm_last_error()) : cudaGetErrorString(ce);
      return r;
    }
    const int samples = per_call ? chunk : 1;
    for (int i = 0; i < samples; ++i) {
      float ms = NAN;
      if (cudaEventElapsedTime(&ms, env.ev[2 * i], env.ev[2 * i + 1]) != cudaSuccess) ms = NAN;
      if (!per_call) ms /= (float)chunk;
      if (faulty && env.fault.mode == "nan") ms = NAN;
      if (faulty && env.fault.mode == "slow") ms *= 1000.f;
      if (!(ms > 0) || !std::isfinite(ms)) {
        r.state = "error";
        r.err = "the profiled window resolved no device timing";
        return r;
      }
      r.times.push_back(ms);
      total += per_call ? ms : ms * chunk;
      if (ms <= env.limit_ms) ++in_limit;
    }
    r.iters += chunk;
    n += chunk;
    if (first) {
      first = false;
      double med = median_of(r.times);
      if (std::isfinite(best_ms) && med > 1.5 * best_ms) {
        r.state = "slow";
        break;
      }
    }
    if (in_limit >= 2) {
      r.short_circuit = true;
      break;
    }
    if (n >= max_it || total >= env.opts.max_tuning_duration_ms) break;
  }
  int err_word = 0;
  cudaMemcpy(&err_word, ds.d_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (err_word != 0) {
    r.state = "timeout";
    char b[96];
    snprintf(b, sizeof b, "kernel wait gave up (code 0x%x)", err_word);
    r.err = b;
    cudaMemset(ds.d_err, 0, 64);
    return r;
  }
  if (r.state != "slow") r.state = "ok";
  r.median = median_of(r.times);
  double s = 0;
  for (float t : r.times) s += t;
  r.mean = s / (double)r.times.size();
  // optional numerical check against the default kernel's output
  if (env.ref && r.state == "ok") {
    const Problem &q = env.rot->sets[0];
    bool wrong = faulty && env.fault.mode == "wrong";
    launch_candidate(idx, q, ctx);
    cudaMemsetAsync(env.d_bad, 0, sizeof(int), ds.tune_stream);
    launch_compare(q.C, env.ref, q.tc, q.M, q.N, q.ldc, q.batch, q.sC, env.atol, env.rtol,
                   env.d_bad, ds.tune_stream);
    int bad = 0;
    cudaMemcpyAsync(&bad, env.d_bad, sizeof(int), cudaMemcpyDeviceToHost, ds.tune_stream);
    cudaStreamSynchronize(ds.tune_stream);
    if (bad || wrong) {
      r.state = "numeric";
      r.err = "failed the numerical check against the default kernel";
    }
  }
  return r;
}

std::string fin_json(const CandResult &r) {
  if (!std::isfinite(r.final_median)) return "";
  char b[64];
  snprintf(b, sizeof b, ", \"final_ms\": %.6g", r.final_median);
  return b;
}

void log_decision(const Options &o, const KeyPod &key, const std::vector<CandResult> &res,
                  int winner, double limit_ms, const Peaks &pk, double ops, double bytes,
                  int rotating_sets, bool l2_flush) {
  if (o.decisions.empty()) return;
  std::string s = "{\"key\": \"" + key_text(key) + "\", \"fastest_index\": " +
                  std::to_string(winner) + ", \"fastest\": \"" +
                  (winner >= 0 ? registry()[winner].name : std::string("")) + "\"";
  char b[512];
  snprintf(b, sizeof b, ", \"rotating_sets\": %d, \"l2_flush\": %s", rotating_sets,
           l2_flush ? "true" : "false");
  s += b;
  snprintf(b, sizeof b,
           ", \"bounds\": {\"compute\": {\"amount\": %.0f, \"peak_per_s\": %.6g}, \"memory\": "
           "{\"amount\": %.0f, \"peak_per_s\": %.6g}, \"threshold\": 0.8, \"launch_overhead_ns\": "
           "%.1f, \"source\": \"%s\"}, \"limit_ns\": %.0f, \"candidates\": [",
           ops, ops > 0 && key.elem_lhs == MM_F32 ? pk.tf32_ops : pk.bf16_ops, bytes,
           pk.bytes_per_s, pk.launch_ns, pk.source.c_str(), limit_ms * 1e6);
  s += b;
  bool firstc = true;
  for (const auto &r : res) {
    if (r.index < 0) continue;
    snprintf(b, sizeof b,
             "%s{\"index\": %d, \"name\": \"%s\", \"state\": \"%s\", \"median_ms\": %.6g, "
             "\"mean_ms\": %.6g, \"n\": %d, \"samples\": %zu%s%s}",
             firstc ? "" : ", ", r.index, registry()[r.index].name.c_str(), state_json(r),
             std::isfinite(r.median) ? r.median : -1.0, std::isfinite(r.mean) ? r.mean : -1.0,
             r.iters, r.times.size(), r.short_circuit ? ", \"short_circuit\": true" : "",
             fin_json(r).c_str());
    s += b;
    firstc = false;
  }
  s += "]}\n";
  if (o.decisions == "stdout") {
    fputs(s.c_str(), stdout);
    fflush(stdout);
  } else {
    FILE *f = fopen(o.decisions.c_str(), "a");
    if (f) {
      fputs(s.c_str(), f);
      fclose(f);
    }
  }
}

mm_status tune(DeviceState &ds, const Problem &p, const KeyPod &key, const Options &o,
               TableEntry *entry) {
  auto t0 = std::chrono::steady_clock::now();
  std::vector<PlanItem> plan = make_plan(key, p, ds.info);
  if (plan.empty()) return set_error(MM_ERR_NO_VALID_CANDIDATE, "empty tuning plan");
  Peaks pk;
  mm_status st = roofline_peaks(ds, &pk);
  if (st != MM_OK) return st;
  double ops = (double)p.M * (double)p.N * (double)std::max<int64_t>(0, 2 * p.K - 1) * (double)p.batch;
  double bytes = ((double)p.M * p.K * dtype_bytes(p.ta) + (double)p.K * p.N * dtype_bytes(p.tb) +
                  (double)p.M * p.N * dtype_bytes(p.tc)) * (double)p.batch;
  double peak_ops = (p.ta == MM_F32 || p.tb == MM_F32) ? pk.tf32_ops : pk.bf16_ops;
  double limit_ms = mm_roofline_limit_ns(ops, peak_ops, bytes, pk.bytes_per_s, 0.8, pk.launch_ns) * 1e-6;

  std::vector<CandResult> res(registry().size());
  int winner = -1;
  int rotating_sets = 0;
  bool flushed = false;
  if (plan.size() == 1) {
    // a single candidate is recorded without measuring it (the page's step 2)
    winner = plan[0].cand;
    res[winner].index = winner;
    res[winner].state = "ok";
  } else {
    Rotation rot;
    // order the private stream after the caller's pending work
    st = make_rotation(ds, p, o, rot);
    if (st != MM_OK) return st;
    BenchEnv env;
    env.ds = &ds;
    env.rot = &rot;
    env.opts = o;
    env.fault = parse_fault(o.fault);
    env.limit_ms = limit_ms;
    env.ev.resize(20);
    rotating_sets = (int)rot.sets.size();
    for (auto &e : env.ev) MM_CUDA_TRY(cudaEventCreate(&e));
    if (o.l2_flush) {
      st = ds.flush_buf.ensure((size_t)std::max<int64_t>(2 * ds.info.l2_bytes, 64 << 20));
      if (st != MM_OK) return st;
      flushed = true;
    }
    std::vector<void *> extra;
    if (!o.numerical_check.empty()) {
      size_t u = o.numerical_check.find('_');
      env.atol = atof(o.numerical_check.substr(0, u).c_str());
      env.rtol = atof(o.numerical_check.substr(u + 1).c_str());
      size_t bc = (size_t)span_c(p) * dtype_bytes(p.tc) + 256;
      void *ref = nullptr;
      MM_CUDA_TRY(cudaMalloc(&ref, bc));
      MM_CUDA_TRY(cudaMalloc(&env.d_bad, 16));
      extra.push_back(ref);
      extra.push_back(env.d_bad);
      Problem q = rot.sets[0];
      char *refp = (char *)ref + align_off(q.C);
      q.C = refp;
      env.ref = refp;
      LaunchCtx ctx{ds.tune_stream, &ds, true};
      st = launch_candidate(0, q, ctx);  // the Default: reference result
      if (st != MM_OK) return st;
    }
    double best = INFINITY;
    size_t pi = 0;
    bool done = false;
    while (pi < plan.size() && !done) {
      int g = plan[pi].group;
      size_t gend = pi;
      while (gend < plan.size() && plan[gend].group == g) ++gend;
      // tiers of this group, in order
      size_t ti = pi;
      while (ti < gend) {
        int tier = plan[ti].tier;
        size_t tend = ti;
        while (tend < gend && plan[tend].tier == tier) ++tend;
        int round_best = -1;
        for (size_t j = ti; j < tend; ++j) {
          int c = plan[j].cand;
          res[c] = bench_candidate(c, env, best);
          if (res[c].state == "ok") {
            if (res[c].median < best) best = res[c].median;
            if (round_best < 0 || res[c].median < res[round_best].median ||
                (res[c].median == res[round_best].median && c < round_best))
              round_best = c;
          }
          if (res[c].short_circuit && res[c].state == "ok") break;
        }
        if (round_best >= 0) {
          winner = round_best;
          done = true;
          break;
        }
        ti = tend;  // whole round failed: its backups
      }
      pi = gend;  // group failed: next group
    }
    // Finalists (medians within 10 % of the winner's, at most three) are
    // re-timed in interleaved chunks before the choice is recorded, so that
    // one lucky or unlucky set of samples does not decide alone.  Not after a
    // round ended inside the roofline limit, nor with the L2 flush on.
    if (winner >= 0 && !res[winner].short_circuit && !(o.l2_flush && ds.flush_buf.ptr)) {
      std::vector<int> fin;
      for (const auto &r : res)
        if (r.index >= 0 && r.state == "ok" && r.median <= 1.10 * res[winner].median)
          fin.push_back(r.index);
      std::stable_sort(fin.begin(), fin.end(),
                       [&](int a, int b) { return res[a].median < res[b].median; });
      if (fin.size() > 3) fin.resize(3);
      if (fin.size() >= 2) {
        std::vector<std::vector<float>> t(fin.size());
        // chunks of 30 calls: closer to a long back-to-back run, where a call
        // overlaps its predecessor's tail (the first call of a chunk cannot)
        for (int round = 0; round < 3; ++round)
          for (size_t f = 0; f < fin.size(); ++f) {
            float ms;
            if (time_chunk(fin[f], env, round * 30, 30, &ms)) t[f].push_back(ms);
          }
        int pick = -1;
        for (size_t f = 0; f < fin.size(); ++f) {
          if (t[f].empty()) continue;
          res[fin[f]].final_median = median_of(t[f]);
          if (pick < 0 || res[fin[f]].final_median < res[pick].final_median ||
              (res[fin[f]].final_median == res[pick].final_median && fin[f] < pick))
            pick = fin[f];
        }
        if (pick >= 0) winner = pick;
      }
    }
    for (auto &e : env.ev) cudaEventDestroy(e);
    cudaStreamSynchronize(ds.tune_stream);
    for (void *x : extra) cudaFree(x);
  }
  log_decision(o, key, res, winner, limit_ms, pk, ops, bytes, rotating_sets, flushed);
  if (winner < 0) {
    std::string why;
    for (const auto &r : res)
      if (r.index >= 0 && !r.err.empty()) why += registry()[r.index].name + ": " + r.err + "; ";
    return set_error(MM_ERR_NO_VALID_CANDIDATE, "no candidate gave a valid result (%s)",
                     why.c_str());
  }
  // ranking: valid results, fastest median first; the default last if absent
  std::vector<int> ok;
  for (const auto &r : res)
    if (r.index >= 0 && (r.state == "ok" || r.state == "slow")) ok.push_back(r.index);
  std::stable_sort(ok.begin(), ok.end(), [&](int a, int b) {
    double ma = std::isfinite(res[a].median) ? res[a].median : INFINITY;
    double mb = std::isfinite(res[b].median) ? res[b].median : INFINITY;
    return ma < mb || (ma == mb && a < b);
  });
  ok.erase(std::remove(ok.begin(), ok.end(), winner), ok.end());
  ok.insert(ok.begin(), winner);
  if (std::find(ok.begin(), ok.end(), 0) == ok.end()) ok.push_back(0);
  entry->winner = winner;
  entry->ranking = ok;
  entry->median_ms = std::isfinite(res[winner].median) ? res[winner].median : 0.0;
  std::string detail;
  for (int c : ok) {
    char b[128];
    snprintf(b, sizeof b, "%s%s:%.6g", detail.empty() ? "" : ";", registry()[c].name.c_str(),
             std::isfinite(res[c].median) ? res[c].median : -1.0);
    detail += b;
  }
  entry->detail = detail;
  double ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t0).count();
  stats().last_tune_ms.store(ms);
  double tot = stats().total_tune_ms.load();
  while (!stats().total_tune_ms.compare_exchange_weak(tot, tot + ms)) {
  }
  stats().tunes.fetch_add(1);
  return MM_OK;
}

// Launch the first candidate of an entry's ranking that supports p.
mm_status run_entry(DeviceState &ds, const TableEntry &e, const Problem &p, cudaStream_t s,
                    ExecResult *res) {
  LaunchCtx ctx{s, &ds, false};
  const auto &reg = registry();
  for (int c : e.ranking) {
    std::string why;
    if (c < 0 || c >= (int)reg.size()) continue;
    if (!reg[c].supports(p, ds.info, reg[c].cfg, &why)) continue;
    const mm_status st = launch_candidate(c, p, ctx);
    // a candidate that declines at launch (scratch it cannot allocate while
    // the stream is captured) leaves the call to the next one in the ranking
    if (st == MM_ERR_UNSUPPORTED) continue;
    if (res) res->candidate = c;
    return st;
  }
  if (res) res->candidate = 0;
  return launch_candidate(0, p, ctx);
}

// The default for a miss that is not tuned (tuning off, a pending key whose
// tuner did not finish in time): the shape-class heuristic's choice, then the
// key's plan, first that supports the problem; the next one if a launch fails.
mm_status launch_default(DeviceState &ds, const KeyPod &key, const Problem &p, LaunchCtx &ctx,
                         ExecResult *res) {
  const auto &reg = registry();
  for (int c : default_order(key, p, ds.info)) {
    std::string why;
    if (!reg[c].supports(p, ds.info, reg[c].cfg, &why)) continue;
    if (launch_candidate(c, p, ctx) == MM_OK) {
      if (res) res->candidate = c;
      return MM_OK;
    }
  }
  if (res) res->candidate = 0;
  return launch_candidate(0, p, ctx);
}

// Runs from exit(): the main thread's thread-local objects (get_options's
// per-thread copy among them) are already destroyed, so the options are read
// through a fresh snapshot.
void save_at_exit_fn() {
  const Options o = snapshot();
  if (o.cache_file.empty() || !o.autotune_cache) return;
  for_each_device([](DeviceState &ds) {
    const Options oo = snapshot();
    if (ds.dirty) cache_save(ds, device_file_name(oo.cache_file, ds.info.ordinal));
  });
}

}  // namespace

void sync_table_file(DeviceState &ds, const Options &o) {
  if (!o.autotune_cache || o.cache_file.empty() || ds.file_loaded) return;
  std::unique_lock<std::mutex> tl(ds.tune_mu);
  if (ds.file_loaded) return;
  ds.file_loaded = true;
  cache_load(ds, device_file_name(o.cache_file, ds.info.ordinal));  // absent file: fine
  static std::once_flag reg_exit;
  std::call_once(reg_exit, [] { atexit(save_at_exit_fn); });
}

mm_status tune_and_record(DeviceState &ds, const Problem &p, const KeyPod &key, const Options &o,
                          cudaStream_t order_after, TableEntry *out) {
  {  // pending protocol: one tuner per key; others wait (bounded)
    std::unique_lock<std::mutex> pl(ds.pending_mu);
    {  // tuned meanwhile by another caller
      std::shared_lock<std::shared_mutex> lk(ds.table_mu);
      auto it = ds.table.find(key);
      if (it != ds.table.end()) {
        *out = *it->second;
        return MM_OK;
      }
    }
    if (ds.pending.count(key)) {
      ds.pending_cv.wait_for(pl, std::chrono::duration<double, std::milli>(o.pending_wait_ms),
                             [&] { return !ds.pending.count(key); });
      pl.unlock();
      std::shared_lock<std::shared_mutex> lk(ds.table_mu);
      auto it = ds.table.find(key);
      if (it != ds.table.end()) {
        *out = *it->second;
        return MM_OK;
      }
      return MM_ERR_PENDING;
    }
    ds.pending.insert(key);
  }
  mm_status st;
  {
    std::lock_guard<std::mutex> tl(ds.tune_mu);
    if (order_after) {  // the private stream starts after the caller's pending work
      cudaEventRecord(ds.ev_order, order_after);
      cudaStreamWaitEvent(ds.tune_stream, ds.ev_order, 0);
    }
    st = tune(ds, p, key, o, out);
  }
  {
    std::lock_guard<std::mutex> pl(ds.pending_mu);
    if (st == MM_OK) {
      std::unique_lock<std::shared_mutex> lk(ds.table_mu);
      ds.table[key] = std::make_shared<const TableEntry>(*out);
      ds.dirty = true;
    }
    ds.pending.erase(key);
  }
  ds.pending_cv.notify_all();
  return st;
}

mm_status autotune_execute(const Problem &p, cudaStream_t s, ExecResult *res) {
  stats().calls.fetch_add(1, std::memory_order_relaxed);
  if (p.M == 0 || p.N == 0 || p.batch == 0) return MM_OK;
  DeviceState *dsp = nullptr;
  mm_status st = current_device(&dsp);
  if (st != MM_OK) return st;
  DeviceState &ds = *dsp;
  LaunchCtx ctx{s, &ds, false};
  if (p.K == 0) {  // an empty sum: zeros, no tuning
    if (res) res->candidate = 0;
    return launch_candidate(0, p, ctx);
  }
  const Options &o = get_options();
  KeyPod key = make_key(p, o.level);
  {
    std::shared_lock<std::shared_mutex> lk(ds.table_mu);
    auto it = ds.table.find(key);
    if (it != ds.table.end()) {
      std::shared_ptr<const TableEntry> e = it->second;
      lk.unlock();
      stats().hits.fetch_add(1, std::memory_order_relaxed);
      if (res) res->hit = true;
      return run_entry(ds, *e, p, s, res);
    }
  }
  stats().misses.fetch_add(1, std::memory_order_relaxed);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cap);
  if (cap != cudaStreamCaptureStatusNone) {
    // capture: the naive kernel (needs no scratch, which could not be
    // allocated while the stream is captured)
    if (res) res->candidate = 0;
    return launch_candidate(0, p, ctx);
  }
  if (!o.tuning) {
    if (!o.record_untuned.empty()) record_untuned(ds, key, p, o.record_untuned);
    return launch_default(ds, key, p, ctx, res);
  }
  // sync the persistent table once per device
  if (o.autotune_cache && !o.cache_file.empty() && !ds.file_loaded) {
    sync_table_file(ds, o);
    std::shared_lock<std::shared_mutex> lk(ds.table_mu);
    auto it = ds.table.find(key);
    if (it != ds.table.end()) {
      std::shared_ptr<const TableEntry> e = it->second;
      lk.unlock();
      if (res) res->hit = true;
      return run_entry(ds, *e, p, s, res);
    }
  }
  TableEntry entry;
  st = tune_and_record(ds, p, key, o, s ? s : cudaStreamLegacy, &entry);
  if (st == MM_ERR_PENDING) {  // another thread's tuner did not finish in time
    std::shared_lock<std::shared_mutex> lk(ds.table_mu);
    auto it = ds.table.find(key);
    if (it != ds.table.end()) {
      std::shared_ptr<const TableEntry> e = it->second;
      lk.unlock();
      return run_entry(ds, *e, p, s, res);
    }
    lk.unlock();
    return launch_default(ds, key, p, ctx, res);
  }
  if (st != MM_OK) return st;
  return run_entry(ds, entry, p, s, res);
}

}  // namespace mm

extern "C" mm_status mm_device_peaks(double *bf16_ops_per_s, double *bytes_per_s,
                                     double *launch_ns) {
  mm::DeviceState *ds = nullptr;
  mm_status st = mm::current_device(&ds);
  if (st != MM_OK) return st;
  mm::Peaks pk;
  {
    std::lock_guard<std::mutex> lk(ds->tune_mu);  // the tuner computes them under this lock too
    st = mm::roofline_peaks(*ds, &pk);
  }
  if (st != MM_OK) return st;
  if (bf16_ops_per_s) *bf16_ops_per_s = pk.bf16_ops;
  if (bytes_per_s) *bytes_per_s = pk.bytes_per_s;
  if (launch_ns) *launch_ns = pk.launch_ns;
  return MM_OK;
}

extern "C" double mm_roofline_limit_ns(double ops, double peak_ops_per_s, double bytes,
                                       double peak_bytes_per_s, double threshold,
                                       double launch_ns) {
  double c = peak_ops_per_s > 0 ? ops / peak_ops_per_s : 0.0;
  double m = peak_bytes_per_s > 0 ? bytes / peak_bytes_per_s : 0.0;
  double t = (c > m ? c : m) / (threshold > 0 ? threshold : 1.0);
  return t * 1e9 + launch_ns;
}
