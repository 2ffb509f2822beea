// Device code of step a2 for one token (gate + top-k by one warp), and the
// 16-byte activation loads, shared by the routing kernels and the decode-layer
// kernel.  See k_route.cu for the sources.
#pragma once
#include "moeslot_internal.cuh"

namespace moeslot {

constexpr int kMaxPerLane = 8;   // E <= 256: logits per lane of a gate warp

template <typename AT> struct Vec16;
template <> struct Vec16<float> {
  static constexpr int C = 4;
  __device__ __forceinline__ static void load(const float* p, float* v) {
    float4 q = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
  }
};
template <> struct Vec16<uint16_t> {   // bf16 bit patterns
  static constexpr int C = 8;
  __device__ __forceinline__ static void load(const uint16_t* p, float* v) {
    uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
    v[0] = bf16lo(q.x); v[1] = bf16hi(q.x); v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
    v[4] = bf16lo(q.z); v[5] = bf16hi(q.z); v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
  }
};

// Approximate expert substitution (MoE-CORE "Mechanism"), opt-in: after a warp's top-k of
// token t (ids[t][0..k) in rank order, this lane's logits v and selection flags taken,
// the selected logits zsel in rank order, the best unselected logit `boundary`), each
// selected expert that is not resident (res_row: the layer's table row at the step's
// start) and whose logit is within alpha of the boundary takes, in rank order, the
// token's best resident unselected expert (ties to the lower id), one each; it keeps the
// missed expert's position and so its weight.  k < E only.
__device__ __forceinline__ void aes_warp(const float* v, bool* taken, const float* zsel, float boundary, int t,
                                         int E, int k, float alpha, const int32_t* __restrict__ res_row,
                                         int32_t* ids, unsigned long long* stats) {
  const int lane = threadIdx.x & 31;
  bool res[kMaxPerLane];
#pragma unroll
  for (int j = 0; j < kMaxPerLane; ++j) {
    const int e = lane + 32 * j;
    res[j] = e < E && res_row[e] >= 0;
  }
  __syncwarp();   // ids[t][..] as lane 0 wrote them
  int n = 0;
  for (int r = 0; r < k; ++r) {
    const int e = ids[(size_t)t * k + r];
    if (res_row[e] >= 0 || !(zsel[r] - boundary <= alpha)) continue;
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
      const int ee = lane + 32 * j;
      if (!taken[j] && res[j] && (v[j] > bv || (v[j] == bv && ee < be))) { bv = v[j]; be = ee; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
    }
    if (be == 0x7fffffff) break;        // no resident unselected expert left
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j)
      if (lane + 32 * j == be) taken[j] = true;
    if (lane == 0) ids[(size_t)t * k + r] = be;
    ++n;
  }
  if (lane == 0 && n) atomicAdd(&stats[ST_AES], (unsigned long long)n);
  __syncwarp();
}

// One warp: gate and top-k of token t from its logits z[t][0..E).  zsel_w: k floats
// of shared memory private to the warp.
__device__ __forceinline__ void gate_one_token(const float* __restrict__ z, int t, int E, int k, int gating,
                                               int32_t* ids, float* w, float* probs, float* gap,
                                               unsigned long long* stats, float* zsel_w,
                                               const int32_t* aes_row = nullptr, float aes_alpha = 0.f) {
  const int lane = threadIdx.x & 31;
  float v[kMaxPerLane];
  bool taken[kMaxPerLane];
  float zmax = -INFINITY;
#pragma unroll
  for (int j = 0; j < kMaxPerLane; ++j) {
    const int e = lane + 32 * j;
    taken[j] = e >= E;
    v[j] = e < E ? __ldcg(z + (size_t)t * E + e) : -INFINITY;
    zmax = fmaxf(zmax, v[j]);
  }
  zmax = warp_max(zmax);
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
        zsel_w[r] = bv;
      }
    } else {
      next_best = bv;
    }
  }
  __syncwarp();
  if (aes_row && k < E) aes_warp(v, taken, zsel_w, next_best, t, E, k, aes_alpha, aes_row, ids, stats);
  const float zk = zsel_w[k - 1];
  const float g = k < E ? zk - next_best : INFINITY;
  if (lane == 0) {
    gap[t] = g;
    if (g < 1e-4f) atomicAdd(&stats[ST_NEAR_TIES], 1ull);
  }
  float num = 0.f;
  if (lane < k) {
    const float zj = zsel_w[lane];
    num = gating == MOE_GATE_SOFTMAX_RENORM ? expf(zj - zmax) : 1.f / (1.f + expf(-zj));
  }
  const float den = warp_sum(num);
  if (lane < k) w[(size_t)t * k + lane] = num / den;
  __syncwarp();
}

// Unsigned key of a logit whose integer order is the float order: NaN ranks as -inf
// and -0 as +0 (equal logits tie, the lower id first); 0 is below every key and marks
// a taken or absent expert.
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (isnan(v)) v = -INFINITY;
  if (v == 0.f) v = 0.f;
  const uint32_t b = __float_as_uint(v);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// One warp: gate and top-k of token t from its logits zs[t][0..E) in shared memory, as
// gate_one_token (same selection, weights and probabilities), each arg-max round taken
// by two warp reductions (the largest key, then the lowest expert id holding it).
// PER: logits per lane (E <= 32 * PER).  ids_s / w_s: the token's k ids and weights in
// rank order (shared memory); flag_s (shared memory, optional): set to 1 for every
// selected expert.  When ids is not null the warp also writes the global routing outputs
// (ids, w, probs, gap) and the near-tie count.
template <int PER>
__device__ __forceinline__ void gate_warp_keys(const float* zs, int t, int E, int k, int gating, int32_t* ids_s,
                                               float* w_s, int32_t* ids, float* w, float* probs, float* gap,
                                               unsigned long long* stats, int* flag_s) {
  const int lane = threadIdx.x & 31;
  float v[PER];
  uint32_t key[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const int e = lane + 32 * j;
    v[j] = e < E ? zs[(size_t)t * E + e] : -INFINITY;
    key[j] = e < E ? logit_key(v[j]) : 0u;
  }
  float zmax = -INFINITY, zmine = 0.f, next_best = INFINITY;
  const int rounds = k < E ? k + 1 : k;
  for (int r = 0; r < rounds; ++r) {
    uint32_t bk = 0u, be = 0xffffffffu;
#pragma unroll
    for (int j = 0; j < PER; ++j)
      if (key[j] > bk) { bk = key[j]; be = (uint32_t)(lane + 32 * j); }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t emin = __reduce_min_sync(0xffffffffu, bk == kmax ? be : 0xffffffffu);
    const float val = key_logit(kmax);
    if (r == 0) zmax = val;
    if (r < k) {
#pragma unroll
      for (int j = 0; j < PER; ++j)
        if ((uint32_t)(lane + 32 * j) == emin) key[j] = 0u;
      if (lane == r) zmine = val;
      if (lane == 0) {
        ids_s[t * k + r] = (int32_t)emin;
        if (flag_s) flag_s[emin] = 1;
        if (ids) ids[(size_t)t * k + r] = (int32_t)emin;
      }
    } else {
      next_best = val;
    }
  }
  float num = 0.f;
  if (lane < k) num = gating == MOE_GATE_SOFTMAX_RENORM ? expf(zmine - zmax) : 1.f / (1.f + expf(-zmine));
  const float den = warp_sum(num);
  if (lane < k) {
    w_s[t * k + lane] = num / den;
    if (ids) w[(size_t)t * k + lane] = num / den;
  }
  if (ids) {
    const float zk = __shfl_sync(0xffffffffu, zmine, k - 1);
    const float g = k < E ? zk - next_best : INFINITY;
    if (lane == 0) {
      gap[t] = g;
      if (g < 1e-4f) atomicAdd(&stats[ST_NEAR_TIES], 1ull);
    }
    if (gating == MOE_GATE_SOFTMAX_RENORM) {
      float part = 0.f, ex[PER];
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        ex[j] = lane + 32 * j < E ? expf(v[j] - zmax) : 0.f;
        part += ex[j];
      }
      const float pden = warp_sum(part);
#pragma unroll
      for (int j = 0; j < PER; ++j)
        if (lane + 32 * j < E) probs[(size_t)t * E + lane + 32 * j] = ex[j] / pden;
    } else {
#pragma unroll
      for (int j = 0; j < PER; ++j)
        if (lane + 32 * j < E) probs[(size_t)t * E + lane + 32 * j] = 1.f / (1.f + expf(-v[j]));
    }
  }
  __syncwarp();
}

// Every token of a step gated by the CTA's NW warps, one token per warp at a time.
template <int PER>
__device__ __forceinline__ void gate_tokens_warps(const float* zs, int T, int E, int k, int gating, int32_t* ids_s,
                                                  float* w_s, int32_t* ids, float* w, float* probs, float* gap,
                                                  unsigned long long* stats, int NW, int* flag_s) {
  for (int t = threadIdx.x >> 5; t < T; t += NW)
    gate_warp_keys<PER>(zs, t, E, k, gating, ids_s, w_s, ids, w, probs, gap, stats, flag_s);
}

// Gate and top-k of token t by a whole CTA of NT >= E threads, thread e holding
// expert e (the decode layer kernel: a token's last routing CTA has all its
// threads free, and one warp's serial arg-max rounds are the long pole).  Same
// results as gate_one_token: softmax (or sigmoid) probabilities of every expert,
// the k largest logits in descending order with ties to the lower expert id
// (expert e is the r-th largest for r = #{e' : z[e'] > z[e] or (z[e'] == z[e]
// and e' < e)}; NaN ranks as -inf), the gap to the best unselected logit, and
// the renormalised weights of the selected.
struct GateCtaScratch {
  float zs[kMaxPerLane * 32 + 4];   // logits as ranked
  float zsel[36];                   // selected logits by rank, then the best unselected
  float red[32];                    // per-warp partials
  float bcast;
  int byrank[kMaxPerLane * 32];     // expert of each rank (substitution only)
  uint8_t resr[kMaxPerLane * 32];   // whether the expert of each rank is resident
};

template <int NT>
__device__ __forceinline__ void gate_token_cta(const float* __restrict__ z, int t, int E, int k, int gating,
                                               int32_t* ids, float* w, float* probs, float* gap,
                                               unsigned long long* stats, GateCtaScratch& gs,
                                               const int32_t* aes_row = nullptr, float aes_alpha = 0.f) {
  static_assert(NT >= kMaxPerLane * 32, "one thread per expert");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NW = NT / 32;
  const int E4 = (E + 3) & ~3;
  const float v = tid < E ? __ldcg(z + (size_t)t * E + tid) : -INFINITY;
  if (tid < E4) gs.zs[tid] = tid < E && !isnan(v) ? v : -INFINITY;   // padding never outranks: index >= E
  // max of the logits (NaN ignored)
  float m = warp_max(v);
  if (lane == 0) gs.red[warp] = m;
  __syncthreads();
  if (tid == 0) {
    float mm = gs.red[0];
    for (int i = 1; i < NW; ++i) mm = fmaxf(mm, gs.red[i]);
    gs.bcast = mm;
  }
  __syncthreads();
  const float zmax = gs.bcast;
  // per-expert probability for the routing history
  float ex = 0.f;
  if (gating == MOE_GATE_SOFTMAX_RENORM) {
    ex = tid < E ? expf(v - zmax) : 0.f;
    const float part = warp_sum(ex);
    __syncthreads();   // every thread has read bcast
    if (lane == 0) gs.red[warp] = part;
    __syncthreads();
    if (tid == 0) {
      float den = 0.f;
      for (int i = 0; i < NW; ++i) den += gs.red[i];
      gs.bcast = den;
    }
    __syncthreads();
    if (tid < E) probs[(size_t)t * E + tid] = ex / gs.bcast;
  } else if (tid < E) {
    probs[(size_t)t * E + tid] = 1.f / (1.f + expf(-v));
  }
  // rank of expert tid
  if (tid < E) {
    const float u = gs.zs[tid];
    int rank = 0;
    for (int e0 = 0; e0 < E4; e0 += 4) {
      const float4 q = *reinterpret_cast<const float4*>(gs.zs + e0);
      rank += (q.x > u || (q.x == u && e0 < tid)) ? 1 : 0;
      rank += (q.y > u || (q.y == u && e0 + 1 < tid)) ? 1 : 0;
      rank += (q.z > u || (q.z == u && e0 + 2 < tid)) ? 1 : 0;
      rank += (q.w > u || (q.w == u && e0 + 3 < tid)) ? 1 : 0;
    }
    if (rank <= k) gs.zsel[rank] = u;
    if (rank < k) ids[(size_t)t * k + rank] = tid;
    if (aes_row) {
      gs.byrank[rank] = tid;
      gs.resr[rank] = aes_row[tid] >= 0 ? 1 : 0;
    }
  }
  __syncthreads();
  if (aes_row && k < E && tid == 0) {
    // approximate expert substitution, as aes_warp: low-score misses in rank order take the
    // resident unselected experts in rank order
    const float bnd = gs.zsel[k];
    int j = k, n = 0;
    for (int r = 0; r < k; ++r) {
      if (gs.resr[r] || !(gs.zsel[r] - bnd <= aes_alpha)) continue;
      while (j < E && !gs.resr[j]) ++j;
      if (j >= E) break;
      ids[(size_t)t * k + r] = gs.byrank[j];
      ++j;
      ++n;
    }
    if (n) atomicAdd(&stats[ST_AES], (unsigned long long)n);
  }
  if (warp == 0) {
    const float zk = gs.zsel[k - 1];
    const float g = k < E ? zk - gs.zsel[k] : INFINITY;
    if (lane == 0) {
      gap[t] = g;
      if (g < 1e-4f) atomicAdd(&stats[ST_NEAR_TIES], 1ull);
    }
    float num = 0.f;
    if (lane < k) {
      const float zj = gs.zsel[lane];
      num = gating == MOE_GATE_SOFTMAX_RENORM ? expf(zj - zmax) : 1.f / (1.f + expf(-zj));
    }
    const float den = warp_sum(num);
    if (lane < k) w[(size_t)t * k + lane] = num / den;
  }
}

}  // namespace moeslot
