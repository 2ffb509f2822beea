// Steps a1 (router projection) and a2 (gate + top-k).
//
// a1: z[t, e] = sum_h x[t, h] * W_r[e, h] + b[e]   (RapidMoE §2.1: the gate is a
//     linear projection of the token).  fp32 accumulation of bf16/fp32 inputs.
// a2: one warp per token.  Top-k by descending logit with ties to the lower
//     expert id (RapidMoE §2.1); the k weights are renormalised (CAP §II-A,
//     Eq. 1): softmax-renorm exp(z_j - z_max) / sum_topk exp(z_i - z_max), or
//     sigmoid-renorm sigma(z_j) / sum_topk sigma(z_i).  It also writes the
//     per-expert probability (full softmax or sigmoid) used by the routing
//     history, and the gap between the k-th and (k+1)-th logit.
#include "gate_body.cuh"

namespace moeslot {

constexpr int kRouteWarps = 8;   // experts per CTA (one per warp)
constexpr int kRouteTok = 8;     // tokens per CTA row

template <typename AT>
__global__ void __launch_bounds__(kRouteWarps * 32)
route_logits_kernel(const AT* __restrict__ x, const AT* __restrict__ wr, const float* __restrict__ b,
                    float* __restrict__ z, int T, int E, int H) {
  constexpr int C = Vec16<AT>::C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouteWarps + warp;
  const int t0 = blockIdx.y * kRouteTok;
  if (e >= E) return;
  const int nt = min(kRouteTok, T - t0);
  float acc[kRouteTok];
#pragma unroll
  for (int r = 0; r < kRouteTok; ++r) acc[r] = 0.f;
  const AT* wrow = wr + (size_t)e * H;
  for (int h = lane * C; h < H; h += 32 * C) {
    float wv[C];
    Vec16<AT>::load(wrow + h, wv);
#pragma unroll
    for (int r = 0; r < kRouteTok; ++r) {
      if (r < nt) {
        float xv[C];
        Vec16<AT>::load(x + (size_t)(t0 + r) * H + h, xv);
#pragma unroll
        for (int c = 0; c < C; ++c) acc[r] = fmaf(wv[c], xv[c], acc[r]);
      }
    }
  }
  const float bias = b[e];
#pragma unroll
  for (int r = 0; r < kRouteTok; ++r) {
    if (r < nt) {
      float v = warp_sum(acc[r]);
      if (lane == 0) z[(size_t)(t0 + r) * E + e] = v + bias;
    }
  }
}

int launch_route_logits(const PoolDev& p, int layer, const void* x, int T, const void* router_w,
                        const float* router_b, float* logits, cudaStream_t s) {
  dim3 grid((p.E + kRouteWarps - 1) / kRouteWarps, (T + kRouteTok - 1) / kRouteTok);
  const size_t wofs = (size_t)layer * p.E * p.H;
  const float* b = router_b + (size_t)layer * p.E;
  if (p.adt == MOE_BF16) {
    route_logits_kernel<uint16_t><<<grid, kRouteWarps * 32, 0, s>>>(
        (const uint16_t*)x, (const uint16_t*)router_w + wofs, b, logits, T, p.E, p.H);
  } else {
    route_logits_kernel<float><<<grid, kRouteWarps * 32, 0, s>>>(
        (const float*)x, (const float*)router_w + wofs, b, logits, T, p.E, p.H);
  }
  return 1;
}

// ------------------------------------------------------------------ gate + top-k
constexpr int kGateWarps = 8;

// z: the logits [T][E]; or, with nsp > 0, nsp partial sums [nsp][T][E] of the
// projection (tensor-core router), added in split order, plus the bias.
__global__ void __launch_bounds__(kGateWarps * 32)
gate_topk_kernel(const float* __restrict__ z, int nsp, const float* __restrict__ bias, int T, int E, int k,
                 int gating, int32_t* __restrict__ ids, float* __restrict__ w, float* __restrict__ probs,
                 float* __restrict__ gap, unsigned long long* stats, const int32_t* __restrict__ aes_row,
                 float aes_alpha) {
  __shared__ float zsel[kGateWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kGateWarps + warp;
  if (t >= T) return;
  float v[kMaxPerLane];
  bool taken[kMaxPerLane];
  float zmax = -INFINITY;
#pragma unroll
  for (int j = 0; j < kMaxPerLane; ++j) {
    const int e = lane + 32 * j;
    taken[j] = e >= E;
    if (e >= E) {
      v[j] = -INFINITY;
    } else if (nsp > 0) {
      float acc = 0.f;
      for (int sp = 0; sp < nsp; ++sp) acc += z[((size_t)sp * T + t) * E + e];
      v[j] = acc + bias[e];
    } else {
      v[j] = z[(size_t)t * E + e];
    }
    zmax = fmaxf(zmax, v[j]);
  }
  zmax = warp_max(zmax);

  // per-expert probability for the routing history
  if (gating == MOE_GATE_SOFTMAX_RENORM) {
    float part = 0.f, ex[kMaxPerLane];
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
      ex[j] = taken[j] ? 0.f : expf(v[j] - zmax);
      part += ex[j];
    }
    const float den = warp_sum(part);
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j)
      if (!taken[j]) probs[(size_t)t * E + lane + 32 * j] = ex[j] / den;
  } else {
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j)
      if (!taken[j]) probs[(size_t)t * E + lane + 32 * j] = 1.f / (1.f + expf(-v[j]));
  }

  // top-k: k rounds of a warp arg-max (ties to the lower expert id), plus one
  // more round for the best unselected logit when k < E
  float next_best = INFINITY;
  const int rounds = k < E ? k + 1 : k;
  for (int r = 0; r < rounds; ++r) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
      const int e = lane + 32 * j;
      if (!taken[j] && (v[j] > bv || (v[j] == bv && e < be))) { bv = v[j]; be = e; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
    }
    if (r < k) {
#pragma unroll
      for (int j = 0; j < kMaxPerLane; ++j)
        if (lane + 32 * j == be) taken[j] = true;
      if (lane == 0) {
        ids[(size_t)t * k + r] = be;
        zsel[warp][r] = bv;
      }
    } else {
      next_best = bv;
    }
  }
  __syncwarp();
  if (aes_row && k < E) aes_warp(v, taken, zsel[warp], next_best, t, E, k, aes_alpha, aes_row, ids, stats);
  const float zk = zsel[warp][k - 1];
  const float g = k < E ? zk - next_best : INFINITY;
  if (lane == 0) {
    gap[t] = g;
    if (g < 1e-4f) atomicAdd(&stats[ST_NEAR_TIES], 1ull);
  }
  // renormalised weights of the k selected experts
  float num = 0.f;
  if (lane < k) {
    const float zj = zsel[warp][lane];
    num = gating == MOE_GATE_SOFTMAX_RENORM ? expf(zj - zmax) : 1.f / (1.f + expf(-zj));
  }
  const float den = warp_sum(num);
  if (lane < k) w[(size_t)t * k + lane] = num / den;
}

// ------------------------------------------------------------------ fused decode routing
// For a handful of tokens (T <= kFusedRouteT): one CTA per expert computes that
// expert's logits for every token — each thread issues all of its W_r and x
// loads at once, then a block reduction — and the last CTA to finish (ticket
// counter, self-resetting) runs the gate/top-k warps over all tokens.  One
// launch and two dependent memory round trips instead of two launches.
constexpr int kFusedRouteT = 32;
constexpr int kFusedRouteThreads = 256;

template <typename AT>
__global__ void __launch_bounds__(kFusedRouteThreads)
route_gate_fused_kernel(const AT* __restrict__ x, const AT* __restrict__ wr, const float* __restrict__ b,
                        float* __restrict__ z, int T, int E, int H, int k, int gating, int32_t* ids, float* w,
                        float* probs, float* gap, unsigned long long* stats, int32_t* ticket,
                        const int32_t* aes_row, float aes_alpha) {
  constexpr int C = Vec16<AT>::C;
  constexpr int kMaxChunks = 4;        // H <= kMaxChunks * C * kFusedRouteThreads
  __shared__ float red[kFusedRouteThreads / 32][kFusedRouteT];
  __shared__ float zsel[kFusedRouteThreads / 32][32];
  __shared__ int last;
  const int e = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float wv[kMaxChunks][C];
  bool has[kMaxChunks];
#pragma unroll
  for (int q = 0; q < kMaxChunks; ++q) {
    const int h = (q * kFusedRouteThreads + threadIdx.x) * C;
    has[q] = h < H;
    if (has[q]) Vec16<AT>::load(wr + (size_t)e * H + h, wv[q]);
  }
  float acc[kFusedRouteT];
#pragma unroll
  for (int t = 0; t < kFusedRouteT; ++t) {
    acc[t] = 0.f;
    if (t < T) {
#pragma unroll
      for (int q = 0; q < kMaxChunks; ++q) {
        if (has[q]) {
          float xv[C];
          Vec16<AT>::load(x + (size_t)t * H + (q * kFusedRouteThreads + threadIdx.x) * C, xv);
#pragma unroll
          for (int c = 0; c < C; ++c) acc[t] = fmaf(wv[q][c], xv[c], acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kFusedRouteT; ++t) {
    if (t < T) {
      const float v = warp_sum(acc[t]);
      if (lane == 0) red[warp][t] = v;
    }
  }
  __syncthreads();
  if (threadIdx.x < T) {
    float v = 0.f;
    for (int w2 = 0; w2 < kFusedRouteThreads / 32; ++w2) v += red[w2][threadIdx.x];
    z[(size_t)threadIdx.x * E + e] = v + b[e];
  }
  // last CTA to finish runs the gate for every token
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(ticket, 1);
    last = old == (int)gridDim.x - 1;
    if (last) *ticket = 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  for (int t = warp; t < T; t += kFusedRouteThreads / 32)
    gate_one_token(z, t, E, k, gating, ids, w, probs, gap, stats, zsel[warp], aes_row, aes_alpha);
}

int launch_route_gate_fused(const PoolDev& p, int layer, const void* x, int T, const void* router_w,
                            const float* router_b, const Scratch& sc, cudaStream_t s) {
  const size_t wofs = (size_t)layer * p.E * p.H;
  const float* b = router_b + (size_t)layer * p.E;
  const int32_t* aes_row = p.aes_on ? p.lut + (size_t)layer * p.E : nullptr;   // the table at the step's start
  if (p.adt == MOE_BF16) {
    route_gate_fused_kernel<uint16_t><<<p.E, kFusedRouteThreads, 0, s>>>(
        (const uint16_t*)x, (const uint16_t*)router_w + wofs, b, sc.logits, T, p.E, p.H, p.k, p.gating, sc.ids,
        sc.w, sc.probs, sc.gap, p.stats, sc.ticket, aes_row, p.aes_alpha);
  } else {
    route_gate_fused_kernel<float><<<p.E, kFusedRouteThreads, 0, s>>>(
        (const float*)x, (const float*)router_w + wofs, b, sc.logits, T, p.E, p.H, p.k, p.gating, sc.ids, sc.w,
        sc.probs, sc.gap, p.stats, sc.ticket, aes_row, p.aes_alpha);
  }
  return 1;
}

bool route_fused_ok(const PoolDev& p, int T) {
  const int C = p.adt == MOE_BF16 ? 8 : 4;
  return T <= kFusedRouteT && p.H <= 4 * C * kFusedRouteThreads;
}

int launch_gate_topk(const PoolDev& p, const float* logits, int nsp, const float* bias, int T, int32_t* ids,
                     float* w, float* probs, float* gap, cudaStream_t s, const int32_t* aes_row) {
  const int grid = (T + kGateWarps - 1) / kGateWarps;
  gate_topk_kernel<<<grid, kGateWarps * 32, 0, s>>>(logits, nsp, bias, T, p.E, p.k, p.gating, ids, w, probs, gap,
                                                     p.stats, aes_row, p.aes_alpha);
  return 1;
}

}  // namespace moeslot
