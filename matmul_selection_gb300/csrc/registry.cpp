// Candidate registry, group priorities and the tuning plan.
//
// Plan rules (burn "autotune" page, section "one op, thirty-odd candidates"):
// each candidate belongs to a group; group priority and in-group priority
// are functions of the key (MAX 3, HIGH 2, MEDIUM 1, MIN 0, NEVER -1; a
// negative value skips it for that key).  Groups are tried from the highest
// priority down and once a candidate of a group gives a valid result no later
// group is tried.  Inside a group only the top tier forms the round; lower
// tiers are backups.  Candidates that cannot run the problem are demoted to
// MIN instead of being dropped, so the plan is never empty; the first entry
// (naive) always works.
//
// The page's table of group rules did not survive; the rules here are ours:
//   gemv   : MAX when the anchored m <= 16, else NEVER;
//   tensor : HIGH; inside it plain tile configs are HIGH, split-K configs are
//            HIGH when the output has too few tiles to fill the GPU and k is
//            deep (anchored 128 x 128 tiles * 2 <= SMs and k >= 1024), else
//            MIN (backup);
//   naive  : MIN.
#include <algorithm>

#include "common.h"

namespace mm {

namespace {

int prio_naive(const KeyPod &, const Problem &, const DeviceInfo &, int) { return PRIORITY_MIN; }
int prio_gemv(const KeyPod &, const Problem &, const DeviceInfo &, int) { return PRIORITY_HIGH; }
// Split-K: worth measuring when 128 x 128 tiles fill at most half the SMs and
// K is deep enough to split.
int prio_splitk(const KeyPod &k, const DeviceInfo &d) {
  uint64_t tiles = ((k.m + 127) / 128) * ((k.n + 127) / 128) * (k.batch ? k.batch : 1);
  if (tiles * 2 <= (uint64_t)d.sms && k.k >= 1024) return PRIORITY_HIGH;
  return PRIORITY_MIN;
}

int prio_tc(const KeyPod &k, const Problem &, const DeviceInfo &d, int cfg) {
  return tc_config_is_splitk(cfg) ? prio_splitk(k, d) : PRIORITY_HIGH;
}

int prio_repack(const KeyPod &k, const Problem &, const DeviceInfo &d, int cfg) {
  return repack_config_is_splitk(cfg) ? prio_splitk(k, d) : PRIORITY_HIGH;
}

bool naive_supports(const Problem &, const DeviceInfo &, int, std::string *) { return true; }
mm_status naive_launch(const Problem &p, LaunchCtx &ctx, int) { return launch_naive(p, ctx.stream); }

std::vector<Candidate> build_registry() {
  std::vector<Candidate> r;
  r.push_back({"naive", GROUP_NAIVE, 0, prio_naive, naive_supports, naive_launch});
  for (int i = 0; i < gemv_config_count(); ++i)
    r.push_back({gemv_config_name(i), GROUP_GEMV, i, prio_gemv, gemv_supports, launch_gemv});
  for (int i = 0; i < gemv_fast_config_count(); ++i)
    r.push_back({gemv_fast_config_name(i), GROUP_GEMV, i, prio_gemv, gemv_fast_supports,
                 launch_gemv_fast});
  for (int i = 0; i < gemv_mma_config_count(); ++i)
    r.push_back({gemv_mma_config_name(i), GROUP_GEMV, i, prio_gemv, gemv_mma_supports,
                 launch_gemv_mma});
  for (int i = 0; i < tc_config_count(); ++i)
    r.push_back({tc_config_name(i), GROUP_TENSOR, i, prio_tc, tc_supports, launch_tc});
  for (int i = 0; i < repack_config_count(); ++i) {
    const bool small_m = repack_config_is_swap(i);
    r.push_back({repack_config_name(i), small_m ? GROUP_GEMV : GROUP_TENSOR, i,
                 small_m ? prio_gemv : prio_repack, repack_supports, launch_repack});
  }
  // small-M products on the tensor cores: C^T = B^T A^T puts M on the tile's
  // N side (zero-padded to 64) and the long N on its 128-row side; split-K
  // spreads the single row of tiles over the SMs
  const struct {
    const char *name, *cfg;
  } swaps[] = {{"gemv_swap_tc_splitk_128x64_s8", "tc_splitk_128x64_s8"},
               {"gemv_swap_tc_128x64_s8", "tc_128x64_s8"}};
  for (const auto &sw : swaps)
    r.push_back({sw.name, GROUP_GEMV, tc_config_index(sw.cfg), prio_gemv, tc_swap_supports,
                 launch_tc_swapped});
  return r;
}

std::vector<std::atomic<uint64_t>> &launch_counters() {
  static std::vector<std::atomic<uint64_t>> c(registry().size());
  return c;
}

}  // namespace

const std::vector<Candidate> &registry() {
  static const std::vector<Candidate> r = build_registry();
  return r;
}

uint64_t registry_checksum() {
  // FNV-1a 64 over "name\n" of every candidate in registry order, then the
  // library version: adding, removing, renaming or reordering a candidate
  // changes it (the autotune page's compute_checksum over candidate names).
  uint64_t h = 1469598103934665603ull;
  auto mix = [&](const std::string &s) {
    for (unsigned char c : s) {
      h ^= c;
      h *= 1099511628211ull;
    }
  };
  for (const auto &c : registry()) mix(c.name + "\n");
  mix(kVersion);
  return h;
}

const char *group_name(int g) {
  switch (g) {
  case GROUP_GEMV: return "gemv";
  case GROUP_TENSOR: return "tensor";
  case GROUP_NAIVE: return "naive";
  default: return nullptr;
  }
}

int group_priority(int g, const KeyPod &k, const Problem &, const DeviceInfo &) {
  switch (g) {
  case GROUP_GEMV: return k.m <= 16 ? PRIORITY_MAX : PRIORITY_NEVER;
  case GROUP_TENSOR: return PRIORITY_HIGH;
  default: return PRIORITY_MIN;
  }
}

void count_launch(int index, bool tuning) {
  auto &c = launch_counters();
  if (index >= 0 && index < (int)c.size()) c[index].fetch_add(1, std::memory_order_relaxed);
  stats().launches.fetch_add(1, std::memory_order_relaxed);
  if (tuning) stats().bench_launches.fetch_add(1, std::memory_order_relaxed);
}

uint64_t candidate_launches(int index) {
  auto &c = launch_counters();
  if (index < 0 || index >= (int)c.size()) return 0;
  return c[index].load();
}

std::vector<PlanItem> make_plan(const KeyPod &k, const Problem &p, const DeviceInfo &d) {
  const auto &reg = registry();
  // group order: first appearance in the registry
  std::vector<int> order;
  for (const auto &c : reg)
    if (std::find(order.begin(), order.end(), c.group) == order.end()) order.push_back(c.group);
  struct G {
    int group, gprio;
    std::vector<PlanItem> items;
  };
  std::vector<G> groups;
  for (int g : order) {
    G gr{g, group_priority(g, k, p, d), {}};
    if (gr.gprio < 0) continue;
    for (int i = 0; i < (int)reg.size(); ++i) {
      if (reg[i].group != g) continue;
      int pr = reg[i].prio(k, p, d, reg[i].cfg);
      std::string why;
      bool sup = reg[i].supports(p, d, reg[i].cfg, &why);
      int eff = pr;
      if (eff >= 0 && !sup) eff = PRIORITY_MIN;  // demote, never drop
      if (eff < 0) continue;
      gr.items.push_back({i, g, eff, sup ? 1 : 0, gr.gprio, pr});
    }
    if (!gr.items.empty()) groups.push_back(std::move(gr));
  }
  std::stable_sort(groups.begin(), groups.end(),
                   [](const G &a, const G &b) { return a.gprio > b.gprio; });
  std::vector<PlanItem> plan;
  for (auto &gr : groups) {
    std::vector<int> tiers;
    for (auto &it : gr.items) tiers.push_back(it.tier);  // effective priority for now
    std::sort(tiers.begin(), tiers.end(), std::greater<int>());
    tiers.erase(std::unique(tiers.begin(), tiers.end()), tiers.end());
    for (size_t t = 0; t < tiers.size(); ++t)
      for (auto &it : gr.items)
        if (it.tier == tiers[t]) {
          PlanItem x = it;
          x.tier = (int)t;
          plan.push_back(x);
        }
  }
  return plan;
}

// The default for a key that is not tuned (tuning off, or a pending key whose
// tuner did not finish in time): a preference list by shape class, each entry
// the candidate that won that class on a GB300 (the committed tuning table),
// then the plan's order; the first that supports the problem is taken.
//   m = 1                  : gemv_n_stream / gemv_t_stream (B row-major / transposed)
//   m <= 16, A and B       : gemv_n_mma (it also reads an A whose rows are only
//     row-major              8-byte aligned in place)
//   m <= 16, B transposed, : gemv_t_mma (A read in place), then the swapped
//     A not 16-byte aligned  split-K on a copy of A
//   m <= 16 otherwise      : the swapped tensor-core split-K
//   few tiles, deep k      : split-K (the split-K group rule)
//   f32 inputs             : tc_128x256_s4, tc_128x128_s6
//   small outputs          : tc_128x64_s8 (m*n <= 512 x 512: latency)
//   otherwise              : tc2_256x256_s7, or its copying form
std::vector<int> default_order(const KeyPod &k, const Problem &p, const DeviceInfo &d) {
  std::vector<const char *> pref;
  const bool aligned_a = k.lhs_stride >= 4;
  if (k.m <= 1) {
    pref = {p.bt ? "gemv_t_stream" : "gemv_n_stream"};
  } else if (k.m <= 16) {
    const char *swap = aligned_a ? "gemv_swap_tc_splitk_128x64_s8" : "gemv_swap_tc_repack_splitk_128x64";
    if (!p.bt)
      pref = {"gemv_n_mma", swap};  // the first supports only row-major A and B
    else if (!aligned_a)
      pref = {"gemv_t_mma", swap};
    else
      pref = {swap, "gemv_t_mma"};
  } else if (prio_splitk(k, d) == PRIORITY_HIGH) {
    pref = {aligned_a ? "tc_splitk_128x128_s7" : "tc_repack_splitk_128x128"};
  } else if (p.ta == MM_F32) {
    pref = {"tc_128x256_s4", "tc_128x128_s6"};
  } else if (k.m * k.n <= 512 * 512 && k.batch <= 1) {
    pref = {"tc_128x64_s8"};
  } else if (k.batch > 1) {
    pref = {"tc_128x256_s4"};
  } else {
    pref = {aligned_a ? "tc2_256x256_s7" : "tc2_repack_256x256"};
  }
  std::vector<int> order;
  const auto &reg = registry();
  for (const char *name : pref)
    for (int i = 0; i < (int)reg.size(); ++i)
      if (reg[i].name == name) order.push_back(i);
  for (const PlanItem &it : make_plan(k, p, d))
    if (std::find(order.begin(), order.end(), it.cand) == order.end()) order.push_back(it.cand);
  return order;
}

int default_candidate(const KeyPod &k, const Problem &p, const DeviceInfo &d) {
  const auto &reg = registry();
  for (int c : default_order(k, p, d)) {
    std::string why;
    if (reg[c].supports(p, d, reg[c].cfg, &why)) return c;
  }
  return 0;
}

// Host-side fault injection: "<candidate name>:error" makes that candidate's
// launch fail without launching anything.
static bool fault_error(const std::string &spec, const std::string &name) {
  if (spec.empty()) return false;
  size_t c = spec.rfind(':');
  if (c == std::string::npos) return false;
  return spec.substr(0, c) == name && spec.substr(c + 1) == "error";
}

mm_status launch_candidate(int index, const Problem &p, LaunchCtx &ctx) {
  const auto &reg = registry();
  if (index < 0 || index >= (int)reg.size())
    return set_error(MM_ERR_INVALID_ARG, "candidate index %d out of range", index);
  const Candidate &c = reg[index];
  std::string why;
  if (!c.supports(p, ctx.dev->info, c.cfg, &why))
    return set_error(MM_ERR_UNSUPPORTED, "%s: %s", c.name.c_str(), why.c_str());
  const Options &o = get_options();
  if (!o.fault.empty() && fault_error(o.fault, c.name))
    return set_error(MM_ERR_CUDA, "%s: injected launch error", c.name.c_str());
  mm_status st = c.launch(p, ctx, c.cfg);
  if (st == MM_OK) count_launch(index, ctx.tuning);
  return st;
}

StatsAtomic &stats() {
  static StatsAtomic s;
  return s;
}

}  // namespace mm
