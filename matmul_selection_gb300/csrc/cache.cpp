// On-disk tuning table.
//
// Format follows TunableOp's result file (PyTorch TunableOp guide, section
// 3.2): "Validator,<NAME>,<value>" rows, then one row per result with the
// operator, its parameters, the solution name and the time.  Here:
//   MatmulKey,<canonical key text>,<candidate name>,<median ms>,<ranking>
// where <ranking> lists "name:median_ms" of every valid candidate, fastest
// first, separated by ';' -- kept so an entry can be inspected after the fact
// (burn "autotune" page, section "cache: in-memory table and default.db").
// Validators (mismatch of any one rejects the WHOLE file, as TunableOp's
// ValidateAll does): MM_VERSION (the library version), CANDIDATE_CHECKSUM
// (the candidate set), DEVICE (the device model and architecture, not one
// unit: a table tuned on one GB300 serves every GB300, as TunableOp's result
// file names the GPU architecture) and CUDA_VERSION (the runtime).
// A row naming an unknown candidate is skipped; "Default" names the default
// (naive) kernel, as TunableOp's hand-edit rule allows.
#include <algorithm>
#include <cstdio>
#include <fstream>
#include <sstream>

#include "common.h"

namespace mm {

namespace {

std::vector<std::pair<std::string, std::string>> validators(const DeviceState &ds) {
  char cks[32];
  snprintf(cks, sizeof cks, "%016llx", (unsigned long long)registry_checksum());
  int rt = 0;
  cudaRuntimeGetVersion(&rt);
  char dev[256];
  snprintf(dev, sizeof dev, "%s|sm_%d%d", ds.info.name.c_str(), ds.info.cc_major, ds.info.cc_minor);
  return {{"MM_VERSION", kVersion},
          {"CANDIDATE_CHECKSUM", cks},
          {"DEVICE", dev},
          {"CUDA_VERSION", std::to_string(rt)}};
}

// CSV fields: a field holding ',' or '"' is written in double quotes with
// embedded quotes doubled (the key text contains commas).
std::string csv_field(const std::string &f) {
  if (f.find_first_of(",\"") == std::string::npos) return f;
  std::string q = "\"";
  for (char c : f) {
    if (c == '"') q += '"';
    q += c;
  }
  return q + "\"";
}

std::vector<std::string> csv_split(const std::string &s) {
  std::vector<std::string> out;
  std::string cur;
  bool quoted = false;
  for (size_t i = 0; i < s.size(); ++i) {
    char c = s[i];
    if (quoted) {
      if (c == '"') {
        if (i + 1 < s.size() && s[i + 1] == '"') {
          cur += '"';
          ++i;
        } else {
          quoted = false;
        }
      } else {
        cur += c;
      }
    } else if (c == '"') {
      quoted = true;
    } else if (c == ',') {
      out.push_back(cur);
      cur.clear();
    } else {
      cur += c;
    }
  }
  out.push_back(cur);
  return out;
}

std::vector<std::string> split(const std::string &s, char d, size_t max_fields) {
  std::vector<std::string> out;
  size_t start = 0;
  while (out.size() + 1 < max_fields) {
    size_t c = s.find(d, start);
    if (c == std::string::npos) break;
    out.push_back(s.substr(start, c - start));
    start = c + 1;
  }
  out.push_back(s.substr(start));
  return out;
}

int candidate_index(const std::string &name) {
  if (name == "Default") return 0;
  const auto &reg = registry();
  for (int i = 0; i < (int)reg.size(); ++i)
    if (reg[i].name == name) return i;
  return -1;
}

}  // namespace

std::string device_file_name(const std::string &path, int ordinal) {
  size_t slash = path.find_last_of('/');
  size_t dot = path.find_last_of('.');
  std::string ord = std::to_string(ordinal);
  if (dot == std::string::npos || (slash != std::string::npos && dot < slash))
    return path + ord;
  return path.substr(0, dot) + ord + path.substr(dot);
}

mm_status cache_load(DeviceState &ds, const std::string &path) {
  std::ifstream f(path);
  if (!f) return set_error(MM_ERR_IO, "cannot open '%s'", path.c_str());
  std::map<std::string, std::string> seen;
  std::vector<std::vector<std::string>> rows;
  std::string line;
  while (std::getline(f, line)) {
    if (!line.empty() && line.back() == '\r') line.pop_back();
    if (line.empty()) continue;
    if (line.rfind("Validator,", 0) == 0) {
      auto v = split(line, ',', 3);
      if (v.size() == 3) seen[v[1]] = v[2];
      continue;
    }
    rows.push_back(csv_split(line));
  }
  for (const auto &kv : validators(ds)) {
    auto it = seen.find(kv.first);
    if (it == seen.end())
      return set_error(MM_ERR_CACHE_VALIDATION, "'%s': validator %s missing", path.c_str(),
                       kv.first.c_str());
    if (it->second != kv.second)
      return set_error(MM_ERR_CACHE_VALIDATION, "'%s': validator %s is '%s', expected '%s'",
                       path.c_str(), kv.first.c_str(), it->second.c_str(), kv.second.c_str());
  }
  std::unique_lock<std::shared_mutex> lk(ds.table_mu);
  for (const auto &r : rows) {
    if (r.size() < 3 || r[0] != "MatmulKey") continue;
    KeyPod k;
    if (!parse_key_text(r[1], &k)) continue;
    int w = candidate_index(r[2]);
    if (w < 0) continue;  // unknown solution name: skip this row
    if (ds.table.count(k)) continue;
    TableEntry e;
    e.winner = w;
    e.ranking.push_back(w);
    e.median_ms = r.size() > 3 ? atof(r[3].c_str()) : 0.0;
    if (r.size() > 4) {
      e.detail = r[4];
      for (const auto &tok : split(r[4], ';', 1 << 20)) {
        size_t c = tok.rfind(':');
        int i = candidate_index(tok.substr(0, c));
        if (i >= 0 && std::find(e.ranking.begin(), e.ranking.end(), i) == e.ranking.end())
          e.ranking.push_back(i);
      }
    }
    if (std::find(e.ranking.begin(), e.ranking.end(), 0) == e.ranking.end()) e.ranking.push_back(0);
    e.from_file = true;
    ds.table[k] = std::make_shared<const TableEntry>(e);
  }
  return MM_OK;
}

mm_status cache_save(DeviceState &ds, const std::string &path) {
  std::vector<std::string> lines;
  {
    std::shared_lock<std::shared_mutex> lk(ds.table_mu);
    for (const auto &kv : ds.table) {
      const TableEntry &e = *kv.second;
      char ms[64];
      snprintf(ms, sizeof ms, "%.6g", e.median_ms);
      lines.push_back("MatmulKey," + csv_field(key_text(kv.first)) + "," +
                      csv_field(registry()[e.winner].name) + "," + ms + "," + csv_field(e.detail));
    }
  }
  std::sort(lines.begin(), lines.end());
  std::string tmp = path + ".tmp";
  {
    std::ofstream f(tmp, std::ios::trunc);
    if (!f) return set_error(MM_ERR_IO, "cannot write '%s'", tmp.c_str());
    for (const auto &kv : validators(ds)) f << "Validator," << kv.first << "," << kv.second << "\n";
    for (const auto &l : lines) f << l << "\n";
    if (!f) return set_error(MM_ERR_IO, "write to '%s' failed", tmp.c_str());
  }
  if (std::rename(tmp.c_str(), path.c_str()) != 0)
    return set_error(MM_ERR_IO, "cannot rename '%s' to '%s'", tmp.c_str(), path.c_str());
  ds.dirty = false;
  return MM_OK;
}

namespace {
std::mutex g_untuned_file_mu;

const char *layout_letters(const Problem &p) {
  static const char *L[] = {"NN", "NT", "TN", "TT"};
  return L[(p.at ? 2 : 0) + (p.bt ? 1 : 0)];
}

bool parse_dtype(const std::string &s, int *t) {
  if (s == "bf16") *t = MM_BF16;
  else if (s == "f16") *t = MM_F16;
  else if (s == "f32") *t = MM_F32;
  else return false;
  return true;
}
}  // namespace

void record_untuned(DeviceState &ds, const KeyPod &key, const Problem &p, const std::string &path) {
  {
    std::lock_guard<std::mutex> lk(ds.untuned_mu);
    if (!ds.untuned.insert(key).second) return;  // once per key and process
  }
  char b[512];
  snprintf(b, sizeof b, ",%lld,%lld,%lld,%lld,%lld,%lld,%s,%s,%s,%s,%lld,%lld,%lld,%lld\n",
           (long long)p.M, (long long)p.N, (long long)p.K, (long long)p.lda, (long long)p.ldb,
           (long long)p.ldc, dtype_name(p.ta), dtype_name(p.tb), dtype_name(p.tc), layout_letters(p),
           (long long)p.batch, (long long)p.sA, (long long)p.sB, (long long)p.sC);
  const std::string line = "Untuned," + csv_field(key_text(key)) + b;
  std::lock_guard<std::mutex> lk(g_untuned_file_mu);
  FILE *f = fopen(path.c_str(), "a");
  if (!f) return;  // recording is best effort; the call itself already ran
  fputs(line.c_str(), f);
  fclose(f);
}

mm_status tune_file(DeviceState &ds, const std::string &path, int *tuned) {
  *tuned = 0;
  std::ifstream in(path);
  if (!in) return set_error(MM_ERR_IO, "cannot read %s", path.c_str());
  const Options o = get_options();
  sync_table_file(ds, o);
  std::string line;
  int lineno = 0;
  while (std::getline(in, line)) {
    ++lineno;
    if (line.empty()) continue;
    std::vector<std::string> f = csv_split(line);
    if (f.size() != 16 || f[0] != "Untuned") continue;  // not a record of this format
    Problem p{};
    long long v[6], bs[4];
    for (int i = 0; i < 6; ++i) v[i] = atoll(f[2 + i].c_str());
    for (int i = 0; i < 4; ++i) bs[i] = atoll(f[12 + i].c_str());
    if (!parse_dtype(f[8], &p.ta) || !parse_dtype(f[9], &p.tb) || !parse_dtype(f[10], &p.tc) ||
        f[11].size() != 2)
      return set_error(MM_ERR_INVALID_ARG, "%s:%d: malformed record", path.c_str(), lineno);
    p.M = v[0], p.N = v[1], p.K = v[2], p.lda = v[3], p.ldb = v[4], p.ldc = v[5];
    p.at = f[11][0] == 'T';
    p.bt = f[11][1] == 'T';
    p.batch = bs[0], p.sA = bs[1], p.sB = bs[2], p.sC = bs[3];
    if (p.M < 1 || p.N < 1 || p.K < 1 || p.batch < 1)
      return set_error(MM_ERR_INVALID_ARG, "%s:%d: empty problem", path.c_str(), lineno);
    const KeyPod key = make_key(p, o.level);
    {
      std::shared_lock<std::shared_mutex> lk(ds.table_mu);
      if (ds.table.count(key)) continue;  // already tuned
    }
    // synthetic operands of the recorded shape
    DevBuf a, bb, c;
    struct Release {
      DevBuf &x, &y, &z;
      ~Release() {
        x.release();
        y.release();
        z.release();
      }
    } release{a, bb, c};
    const size_t na = (size_t)span_a(p) * dtype_bytes(p.ta) + 256;
    const size_t nb = (size_t)span_b(p) * dtype_bytes(p.tb) + 256;
    const size_t nc = (size_t)span_c(p) * dtype_bytes(p.tc) + 256;
    mm_status st;
    if ((st = a.ensure(na)) != MM_OK || (st = bb.ensure(nb)) != MM_OK || (st = c.ensure(nc)) != MM_OK)
      return st;
    // pseudo-random operands: every candidate computes the same product, but
    // constant data would let compute-bound candidates run at a lower power
    if ((st = launch_fill(a.ptr, na / dtype_bytes(p.ta), p.ta, 1u, ds.tune_stream)) != MM_OK ||
        (st = launch_fill(bb.ptr, nb / dtype_bytes(p.tb), p.tb, 2u, ds.tune_stream)) != MM_OK)
      return st;
    p.A = a.ptr;
    p.B = bb.ptr;
    p.C = c.ptr;
    TableEntry e;
    st = tune_and_record(ds, p, key, o, nullptr, &e);
    if (st != MM_OK && st != MM_ERR_PENDING) return st;
    MM_CUDA_TRY(cudaStreamSynchronize(ds.tune_stream));
    if (st == MM_OK) ++*tuned;
  }
  return MM_OK;
}

}  // namespace mm
