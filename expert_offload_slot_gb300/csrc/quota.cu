// Offline cache shaping of MoE-CORE (host code only; declared in include/moeslot.h):
//   moe_plan_quotas  per-layer slot quotas for a fixed budget from a replay of a
//                    profiling trace's hit-rate curves;
//   moe_profile_lut  the initial table from a domain profile: each layer's quota of
//                    experts of highest mean router probability.
//
// Source: MoE-CORE "Mechanism".  A fixed decode-cache budget is not split evenly:
// slots move in steps of delta-K from layers whose hit rate stays above the
// median and barely drops when shrunk to layers at least tau_low below the median
// whose hit rate rises the most when grown, and only when the receiver gains more
// than the donor loses.  The cache starts from the experts of highest mean router
// score on a profiling set.
//
// Hit-rate curve h_l(K): one layer's cache of K slots, filled from the profile,
// replayed over the trace with the pool's own history score (MoE-CORE score,
// Minus Recent Score or LRU, fp32 in the order the pool computes it) and victim
// rule (lowest free slot, else the lowest-score slot this step does not need, ties
// to the lower slot; a miss with no victim is not cached).  h = hits / needed
// experts, both integer counts; everything after that is float64.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>
#include <vector>

#include "moeslot_internal.cuh"

namespace {

using moeslot::set_last_error;

struct Trace {
  const int32_t* ids;    // [steps][L][T][k]
  const float* probs;    // [steps][L][T][E]
  int steps, L, T, k, E;
  const int32_t* ids_at(int s, int l) const { return ids + (((size_t)s * L + l) * T) * k; }
  const float* probs_at(int s, int l) const { return probs + (((size_t)s * L + l) * T) * E; }
};

// Experts of layer l by descending mean probability (float64 sum over (step, token) in
// order, divided by their count), ties to the lower id.
std::vector<int> profile_order(const Trace& tr, int l) {
  std::vector<double> total(tr.E, 0.0);
  for (int s = 0; s < tr.steps; ++s)
    for (int t = 0; t < tr.T; ++t) {
      const float* p = tr.probs_at(s, l) + (size_t)t * tr.E;
      for (int e = 0; e < tr.E; ++e) total[e] = total[e] + (double)p[e];
    }
  const double n = (double)tr.steps * tr.T;
  std::vector<double> mean(tr.E);
  for (int e = 0; e < tr.E; ++e) mean[e] = total[e] / n;
  std::vector<int> order(tr.E);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return mean[a] > mean[b]; });
  return order;
}

// One layer's cache of K slots over the trace; returns (hits, needed experts).
struct LayerReplay {
  const moe_config& cfg;
  int E, K, W;
  std::vector<int> lut, owner, last_sel;
  std::vector<float> score, ema, hist_s;
  std::vector<uint8_t> hist_sel;
  int t = 0;

  LayerReplay(const moe_config& c, int K_) : cfg(c), E(c.num_experts), K(K_), W(c.window) {
    lut.assign(E, -1);
    owner.assign(K, -1);
    last_sel.assign(E, -1);
    score.assign(E, 0.f);
    ema.assign(E, 0.f);
    hist_s.assign((size_t)W * E, 0.f);
    hist_sel.assign((size_t)W * E, 0);
  }

  void scores(const int32_t* ids, const float* probs, int T, int k) {
    std::vector<float> s(E, 0.f);
    for (int tt = 0; tt < T; ++tt)
      for (int e = 0; e < E; ++e) s[e] = s[e] + probs[(size_t)tt * E + e];
    for (int e = 0; e < E; ++e) s[e] = s[e] / (float)T;
    std::vector<uint8_t> sel(E, 0);
    for (int i = 0; i < T * k; ++i) sel[ids[i]] = 1;
    const int ring = t % W;
    const float lam = cfg.ema_decay, oml = 1.0f - cfg.ema_decay;
    for (int e = 0; e < E; ++e) {
      hist_s[(size_t)ring * E + e] = s[e];
      hist_sel[(size_t)ring * E + e] = sel[e];
      ema[e] = lam * ema[e] + oml * (sel[e] ? 1.f : 0.f);
      if (sel[e]) last_sel[e] = t;
    }
    if (cfg.evict_policy == MOE_EVICT_MRS) {
      for (int e = 0; e < E; ++e) {
        float acc = 0.f;
        for (int j = W - 1; j >= 0; --j) acc = acc + hist_s[(size_t)(((t - j) % W + W) % W) * E + e];
        score[e] = acc - s[e];
      }
    } else if (cfg.evict_policy == MOE_EVICT_CORE) {
      std::vector<float> c(E), a(E);
      float cmax = -INFINITY, mmax = -INFINITY, smax = -INFINITY, amax = -INFINITY;
      for (int e = 0; e < E; ++e) {
        int cnt = 0;
        for (int j = 0; j < W; ++j) cnt += hist_sel[(size_t)j * E + e];
        c[e] = (float)cnt;
        a[e] = (float)((long long)t - last_sel[e]);
        cmax = std::max(cmax, c[e]);
        mmax = std::max(mmax, ema[e]);
        smax = std::max(smax, s[e]);
        amax = std::max(amax, a[e]);
      }
      const float w0 = cfg.core_w[0], w1 = cfg.core_w[1], w2 = cfg.core_w[2], w3 = cfg.core_w[3];
      for (int e = 0; e < E; ++e) {
        const float ch = cmax > 0.f ? c[e] / cmax : 0.f;
        const float mh = mmax > 0.f ? ema[e] / mmax : 0.f;
        const float gh = smax > 0.f ? s[e] / smax : 0.f;
        const float rh = amax > 0.f ? 1.0f - a[e] / amax : 1.0f;
        const float p0 = w0 * ch, p1 = w1 * mh, p2 = w2 * gh, p3 = w3 * rh;
        score[e] = ((p0 + p1) + p2) + p3;
      }
    } else {
      for (int e = 0; e < E; ++e) score[e] = (float)last_sel[e];
    }
    ++t;
  }

  // returns (hits, needed) of this step
  std::pair<long long, long long> plan(const int32_t* ids, int n) {
    std::vector<int> U(ids, ids + n);
    std::sort(U.begin(), U.end());
    U.erase(std::unique(U.begin(), U.end()), U.end());
    std::vector<uint8_t> prot(K, 0);
    long long hits = 0;
    for (int e : U)
      if (lut[e] >= 0) {
        prot[lut[e]] = 1;
        ++hits;
      }
    for (int e : U) {
      if (lut[e] >= 0) continue;
      int victim = -1;
      for (int s2 = 0; s2 < K && victim < 0; ++s2)
        if (owner[s2] < 0) victim = s2;
      if (victim < 0) {
        float best = 0.f;
        for (int s2 = 0; s2 < K; ++s2) {
          if (prot[s2]) continue;
          const float sc = score[owner[s2]];
          if (victim < 0 || sc < best) {
            victim = s2;
            best = sc;
          }
        }
      }
      if (victim < 0) continue;   // every slot holds an expert this step needs
      if (owner[victim] >= 0) lut[owner[victim]] = -1;
      owner[victim] = e;
      lut[e] = victim;
      prot[victim] = 1;
    }
    return {hits, (long long)U.size()};
  }
};

double hit_rate(const moe_config& cfg, const Trace& tr, int l, int K, const std::vector<int>& order) {
  long long hits = 0, needed = 0;
  if (K <= 0) return 0.0;
  LayerReplay r(cfg, K);
  for (int i = 0; i < K && i < tr.E; ++i) {
    r.lut[order[i]] = i;
    r.owner[i] = order[i];
  }
  for (int s = 0; s < tr.steps; ++s) {
    r.scores(tr.ids_at(s, l), tr.probs_at(s, l), tr.T, tr.k);
    const auto hn = r.plan(tr.ids_at(s, l), tr.T * tr.k);
    hits += hn.first;
    needed += hn.second;
  }
  return needed ? (double)hits / (double)needed : 0.0;
}

moe_status check_trace(const moe_config* cfg, const int32_t* ids, const float* probs, int32_t steps, int32_t T) {
  size_t w13 = 0;
  moe_status st = moe_expert_layout(cfg, &w13, nullptr, nullptr, nullptr, nullptr);
  if (st != MOE_OK) return st;
  if (!probs || steps < 1 || T < 1) return set_last_error(MOE_ERR_INVALID, "trace: NULL probs or empty trace");
  if (ids) {
    const size_t n = (size_t)steps * cfg->num_layers * T * cfg->top_k;
    for (size_t i = 0; i < n; ++i)
      if (ids[i] < 0 || ids[i] >= cfg->num_experts) return set_last_error(MOE_ERR_INVALID, "trace: expert id out of range");
  }
  return MOE_OK;
}

}  // namespace

MOE_API moe_status moe_plan_quotas(const moe_config* cfg, const int32_t* ids, const float* probs, int32_t steps,
                                   int32_t T, int32_t budget, int32_t delta_k, double tau_low, int32_t* quota,
                                   double* hit) {
  moe_status st = check_trace(cfg, ids, probs, steps, T);
  if (st != MOE_OK) return st;
  if (!ids || !quota) return set_last_error(MOE_ERR_INVALID, "moe_plan_quotas: NULL ids or quota");
  if (budget < 0 || delta_k < 1 || !(tau_low >= 0.0))
    return set_last_error(MOE_ERR_INVALID, "moe_plan_quotas: budget >= 0, delta_k >= 1, tau_low >= 0");
  const int L = cfg->num_layers, E = cfg->num_experts;
  const Trace tr{ids, probs, steps, L, T, cfg->top_k, E};
  std::vector<std::vector<int>> order(L);
  for (int l = 0; l < L; ++l) order[l] = profile_order(tr, l);
  std::vector<std::vector<double>> memo(L, std::vector<double>(E + 1, NAN));
  auto h = [&](int l, int k) -> double {
    if (std::isnan(memo[l][k])) memo[l][k] = hit_rate(*cfg, tr, l, k, order[l]);
    return memo[l][k];
  };
  std::vector<int> K(L);
  for (int l = 0; l < L; ++l) K[l] = std::min(E, budget / L + (l < budget % L ? 1 : 0));
  for (int round = 0; round < L * E + 1; ++round) {
    std::vector<double> cur(L), srt;
    for (int l = 0; l < L; ++l) cur[l] = h(l, K[l]);
    srt = cur;
    std::sort(srt.begin(), srt.end());
    const double med = (L % 2) ? srt[L / 2] : (srt[L / 2 - 1] + srt[L / 2]) / 2.0;
    int donor = -1, recv = -1;
    double drop = 0.0, gain = 0.0;
    for (int l = 0; l < L; ++l) {
      if (K[l] - delta_k >= 1 && h(l, K[l] - delta_k) >= med) {
        const double d = cur[l] - h(l, K[l] - delta_k);
        if (donor < 0 || d < drop) {
          donor = l;
          drop = d;
        }
      }
    }
    for (int l = 0; l < L; ++l) {
      if (l != donor && cur[l] <= med - tau_low && K[l] + delta_k <= E) {
        const double g = h(l, K[l] + delta_k) - cur[l];
        if (recv < 0 || g > gain) {
          recv = l;
          gain = g;
        }
      }
    }
    if (donor < 0 || recv < 0 || !(gain > drop)) break;
    K[donor] -= delta_k;
    K[recv] += delta_k;
  }
  for (int l = 0; l < L; ++l) {
    quota[l] = K[l];
    if (hit) hit[l] = h(l, K[l]);
  }
  return MOE_OK;
}

MOE_API moe_status moe_profile_lut(const moe_config* cfg, const float* probs, int32_t steps, int32_t T,
                                   const int32_t* quota, int32_t* lut) {
  moe_status st = check_trace(cfg, nullptr, probs, steps, T);
  if (st != MOE_OK) return st;
  if (!quota || !lut) return set_last_error(MOE_ERR_INVALID, "moe_profile_lut: NULL quota or lut");
  const int L = cfg->num_layers, E = cfg->num_experts;
  long long total = 0;
  for (int l = 0; l < L; ++l) {
    if (quota[l] < 0 || quota[l] > E) return set_last_error(MOE_ERR_INVALID, "moe_profile_lut: quota out of 0..E");
    total += quota[l];
  }
  if (total > cfg->num_slots) return set_last_error(MOE_ERR_INVALID, "moe_profile_lut: quotas exceed num_slots");
  const Trace tr{nullptr, probs, steps, L, T, cfg->top_k, E};
  int next = 0;
  for (int l = 0; l < L; ++l) {
    for (int e = 0; e < E; ++e) lut[(size_t)l * E + e] = -1;
    const std::vector<int> order = profile_order(tr, l);
    for (int i = 0; i < quota[l]; ++i) lut[(size_t)l * E + order[i]] = next++;
  }
  return MOE_OK;
}
