// Tuning options.  Modelled on TunableOp's tuning context (PyTorch TunableOp
// guide, section 7): every option has an MM_* environment variable and an API
// setter; the environment is read once, at first use, and takes precedence
// over values set through the API.
#include <cstdlib>
#include <mutex>

#include "common.h"

namespace mm {

namespace {

struct OptDef {
  const char *name;  // API name; env name = "MM_" + upper(name)
};
const OptDef kDefs[] = {{"tuning"},          {"autotune_cache"},
                        {"autotune_level"},  {"max_tuning_iterations"},
                        {"max_tuning_duration_ms"}, {"rotating_buffer_mb"},
                        {"l2_flush"},        {"numerical_check"},
                        {"cache_file"},      {"decisions"},
                        {"verbose"},         {"peak_tflops"},
                        {"peak_gbs"},        {"fault"},
                        {"record_untuned"},  {"pending_wait_ms"},
                        {"wait_limit_us"},   {"wait_stall"}};

std::mutex g_mu;
Options g_api;
std::map<std::string, std::string> g_env;
std::once_flag g_env_once;

std::string env_name(const char *n) {
  std::string s = "MM_";
  for (const char *c = n; *c; ++c) s += (char)toupper((unsigned char)*c);
  return s;
}

void read_env() {
  for (const auto &d : kDefs) {
    const char *v = getenv(env_name(d.name).c_str());
    if (v) g_env[d.name] = v;
  }
}

bool known(const std::string &n) {
  for (const auto &d : kDefs)
    if (n == d.name) return true;
  return false;
}

bool parse_int(const std::string &v, int *out) {
  char *end = nullptr;
  long x = strtol(v.c_str(), &end, 10);
  if (v.empty() || !end || *end) return false;
  *out = (int)x;
  return true;
}
bool parse_double(const std::string &v, double *out) {
  char *end = nullptr;
  double x = strtod(v.c_str(), &end);
  if (v.empty() || !end || *end) return false;
  *out = x;
  return true;
}

// Apply one (name, value) to an Options; false if the value is malformed.
bool apply(Options &o, const std::string &n, const std::string &v) {
  if (n == "tuning") return parse_int(v, &o.tuning);
  if (n == "autotune_cache") return parse_int(v, &o.autotune_cache);
  if (n == "autotune_level") {
    if (v == "minimal") o.level = LEVEL_MINIMAL;
    else if (v == "balanced") o.level = LEVEL_BALANCED;
    else if (v == "extensive") o.level = LEVEL_EXTENSIVE;
    else if (v == "full") o.level = LEVEL_FULL;
    else return false;
    return true;
  }
  if (n == "max_tuning_iterations") return parse_int(v, &o.max_tuning_iterations);
  if (n == "max_tuning_duration_ms") return parse_double(v, &o.max_tuning_duration_ms);
  if (n == "rotating_buffer_mb") return parse_double(v, &o.rotating_buffer_mb);
  if (n == "l2_flush") return parse_int(v, &o.l2_flush);
  if (n == "numerical_check") {
    if (!v.empty()) {
      size_t u = v.find('_');
      double a, r;
      if (u == std::string::npos || !parse_double(v.substr(0, u), &a) ||
          !parse_double(v.substr(u + 1), &r))
        return false;
    }
    o.numerical_check = v;
    return true;
  }
  if (n == "cache_file") { o.cache_file = v; return true; }
  if (n == "decisions") { o.decisions = v; return true; }
  if (n == "verbose") return parse_int(v, &o.verbose);
  if (n == "peak_tflops") return parse_double(v, &o.peak_tflops);
  if (n == "peak_gbs") return parse_double(v, &o.peak_gbs);
  if (n == "fault") { o.fault = v; return true; }
  if (n == "record_untuned") { o.record_untuned = v; return true; }
  if (n == "pending_wait_ms") return parse_double(v, &o.pending_wait_ms) && o.pending_wait_ms >= 0;
  if (n == "wait_limit_us") return parse_double(v, &o.wait_limit_us) && o.wait_limit_us >= 0;
  if (n == "wait_stall") return parse_int(v, &o.wait_stall);
  return false;
}

std::string show(const Options &o, const std::string &n) {
  char b[64];
  if (n == "tuning") return std::to_string(o.tuning);
  if (n == "autotune_cache") return std::to_string(o.autotune_cache);
  if (n == "autotune_level") {
    const char *L[] = {"minimal", "balanced", "extensive", "full"};
    return L[o.level];
  }
  if (n == "max_tuning_iterations") return std::to_string(o.max_tuning_iterations);
  if (n == "max_tuning_duration_ms") { snprintf(b, sizeof b, "%g", o.max_tuning_duration_ms); return b; }
  if (n == "rotating_buffer_mb") { snprintf(b, sizeof b, "%g", o.rotating_buffer_mb); return b; }
  if (n == "l2_flush") return std::to_string(o.l2_flush);
  if (n == "numerical_check") return o.numerical_check;
  if (n == "cache_file") return o.cache_file;
  if (n == "decisions") return o.decisions;
  if (n == "verbose") return std::to_string(o.verbose);
  if (n == "peak_tflops") { snprintf(b, sizeof b, "%g", o.peak_tflops); return b; }
  if (n == "peak_gbs") { snprintf(b, sizeof b, "%g", o.peak_gbs); return b; }
  if (n == "fault") return o.fault;
  if (n == "record_untuned") return o.record_untuned;
  if (n == "pending_wait_ms") { snprintf(b, sizeof b, "%g", o.pending_wait_ms); return b; }
  if (n == "wait_limit_us") { snprintf(b, sizeof b, "%g", o.wait_limit_us); return b; }
  if (n == "wait_stall") return std::to_string(o.wait_stall);
  return "";
}

}  // namespace

std::atomic<uint64_t> g_version{1};

Options snapshot() {
  std::call_once(g_env_once, read_env);
  std::lock_guard<std::mutex> lk(g_mu);
  Options o = g_api;
  for (const auto &kv : g_env) apply(o, kv.first, kv.second);  // env wins
  return o;
}

// Each thread keeps a copy that is refreshed when an option changes, so the
// warm path reads options without a lock or a string copy.
const Options &get_options() {
  thread_local uint64_t seen = 0;
  thread_local Options cached;
  uint64_t v = g_version.load(std::memory_order_acquire);
  if (v != seen) {
    cached = snapshot();
    seen = v;
  }
  return cached;
}

mm_status set_option(const std::string &name, const std::string &value) {
  std::call_once(g_env_once, read_env);
  if (!known(name)) return set_error(MM_ERR_NOT_FOUND, "unknown option '%s'", name.c_str());
  std::lock_guard<std::mutex> lk(g_mu);
  Options o = g_api;
  if (!apply(o, name, value))
    return set_error(MM_ERR_INVALID_ARG, "bad value '%s' for option '%s'", value.c_str(),
                     name.c_str());
  g_api = o;
  g_version.fetch_add(1, std::memory_order_release);
  return MM_OK;
}

mm_status get_option(const std::string &name, std::string *value) {
  if (!known(name)) return set_error(MM_ERR_NOT_FOUND, "unknown option '%s'", name.c_str());
  *value = show(get_options(), name);
  return MM_OK;
}

}  // namespace mm
