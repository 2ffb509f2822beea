// Steps a3 (routing history and eviction score), a4 (expert_id -> slot_id
// rewrite and miss detection), a5 (victim choice and table update) and a7
// (stable permutation of token rows by expert, and the work list the expert
// kernels consume).  One CTA per layer call: the victim sequence of a layer is
// a chain of dependent decisions, and the whole working set (E <= 256 experts,
// one layer's slots) fits a CTA.
//
// Sources: SeqMoE "Mechanism" (slot pool shared by all layers at one fixed
// base; a table rewrites expert_id to slot_id; the device owns the cache
// metadata and starts the miss copy; a per-slot tag grows with every new
// occupant); MoE-CORE "Mechanism" (per-layer decode cache; score from the
// selection count over a window, an EMA of selections, the current router
// score and the age since the last selection, each normalised across the
// layer, nonnegative weights, evict the lowest); HybriMoE "Mechanism" (Minus
// Recent Score); RapidMoE §4.3 (token-averaged router score for multi-token
// steps).
//
// Score arithmetic uses explicitly rounded fp32 operations in a fixed order
// (no contraction), because the scores decide integer victim choices.
#include "moeslot_internal.cuh"

namespace moeslot {

constexpr int kPlanThreads = 1024;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kMaxE = 256;

struct PlanArgs {
  PoolDev p;
  Scratch sc;
  int layer, T, flags, region, npad;
  const int32_t* ids;
  const float* w;
  const float* probs;
};

// Orderable key: (score ascending, slot ascending).  -0 is folded into +0.
__device__ __forceinline__ unsigned long long score_key(float sc, int slot) {
  if (sc == 0.f) sc = 0.f;
  uint32_t u = __float_as_uint(sc);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (uint32_t)slot;
}

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w < v ? w : v;
  }
  return v;
}

// Block-wide minimum; every thread must call it.  `red` holds kPlanWarps entries.
__device__ unsigned long long block_min_u64(unsigned long long v, unsigned long long* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = warp_min_u64(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    unsigned long long r = lane < kPlanWarps ? red[lane] : ~0ull;
    r = warp_min_u64(r);
    if (lane == 0) red[0] = r;
  }
  __syncthreads();
  const unsigned long long out = red[0];
  __syncthreads();
  return out;
}

__device__ float block_max_f(float v, float* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = warp_max(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    float r = lane < kPlanWarps ? red[lane] : -INFINITY;
    r = warp_max(r);
    if (lane == 0) red[0] = r;
  }
  __syncthreads();
  const float out = red[0];
  __syncthreads();
  return out;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  __shared__ int cnt[kMaxE];
  __shared__ int offs[kMaxE + 1];
  __shared__ int base[kMaxE];
  __shared__ int wcnt[kPlanWarps][kMaxE];
  __shared__ int miss_list[kMaxE];
  __shared__ int bypass_rid[kMaxE];   // one-step record of a miss that got no slot, or -1
  __shared__ int pos_of[kMaxE];       // work-list position of each expert, or -1
  __shared__ unsigned long long red64[kPlanWarps];
  __shared__ float redf[kPlanWarps];
  __shared__ int sh_misc[8];   // 0: n_miss, 1: epoch, 2: hits, 3: n_copy, 4: bypass, 5: evictions, 6: n_work

  const PoolDev& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E, k = p.k, T = a.T, l = a.layer, W = p.W;
  const int Tk = T * k;

  for (int e = tid; e < E; e += kPlanThreads) {
    cnt[e] = 0;
    bypass_rid[e] = -1;
    pos_of[e] = -1;
  }
  if (tid < 8) sh_misc[tid] = 0;
  __syncthreads();
  for (int i = tid; i < Tk; i += kPlanThreads) {
    const int e = a.ids[i];
    if ((unsigned)e >= (unsigned)E) set_status(p.status, MOE_ERR_BOUNDS);
    else atomicAdd(&cnt[e], 1);
  }
  __syncthreads();

  // ------------------------------------------------------------ a3 history
  if (a.flags & PLAN_HISTORY) {
    const int t = p.step[l];
    const int ring = t % W;
    float s = 0.f, m = 0.f;
    int count = 0, age = 0;
    const bool mine = tid < E;
    if (mine) {
      const int e = tid;
      for (int tt = 0; tt < T; ++tt) s = __fadd_rn(s, a.probs[(size_t)tt * E + e]);
      s = __fdiv_rn(s, (float)T);
      const int sel = cnt[e] > 0 ? 1 : 0;
      const size_t he = ((size_t)l * W + ring) * E + e;
      p.hist_s[he] = s;
      p.hist_sel[he] = (uint8_t)sel;
      const size_t le = (size_t)l * E + e;
      m = __fadd_rn(__fmul_rn(p.lam, p.ema[le]), __fmul_rn(p.one_minus_lam, sel ? 1.f : 0.f));
      p.ema[le] = m;
      if (sel) p.last_sel[le] = t;
      age = t - p.last_sel[le];
      for (int j = 0; j < W; ++j) count += p.hist_sel[((size_t)l * W + j) * E + e];
    }
    float sc = 0.f;
    if (p.policy == MOE_EVICT_CORE) {
      // all threads take part in the reductions
      const float cmax = block_max_f(mine ? (float)count : -INFINITY, redf);
      const float mmax = block_max_f(mine ? m : -INFINITY, redf);
      const float smax = block_max_f(mine ? s : -INFINITY, redf);
      const float amax = block_max_f(mine ? (float)age : -INFINITY, redf);
      if (mine) {
        const float c_hat = cmax > 0.f ? __fdiv_rn((float)count, cmax) : 0.f;
        const float m_hat = mmax > 0.f ? __fdiv_rn(m, mmax) : 0.f;
        const float g_hat = smax > 0.f ? __fdiv_rn(s, smax) : 0.f;
        const float r_hat = amax > 0.f ? __fsub_rn(1.f, __fdiv_rn((float)age, amax)) : 1.f;
        sc = __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(p.cw0, c_hat), __fmul_rn(p.cw1, m_hat)),
                                 __fmul_rn(p.cw2, g_hat)),
                       __fmul_rn(p.cw3, r_hat));
      }
    } else if (p.policy == MOE_EVICT_MRS) {
      if (mine) {
        float acc = 0.f;
        for (int j = W - 1; j >= 0; --j) {         // oldest step of the window first
          const int idx = ((t - j) % W + W) % W;
          acc = __fadd_rn(acc, p.hist_s[((size_t)l * W + idx) * E + tid]);
        }
        sc = __fsub_rn(acc, s);
      }
    } else {
      if (mine) sc = (float)p.last_sel[(size_t)l * E + tid];
    }
    if (mine) p.score[(size_t)l * E + tid] = sc;
    __syncthreads();
    if (tid == 0) {
      p.step[l] = t + 1;
      atomicAdd(&p.stats[ST_STEPS], 1ull);
    }
  }

  // ------------------------------------------------------- a4/a5 table, misses
  if (a.flags & PLAN_CACHE) {
    if (tid == 0) sh_misc[1] = *p.epoch + 1;
    __syncthreads();
    const int ep = sh_misc[1];
    // protect resident needed experts; list misses in ascending expert id
    int is_miss = 0;
    if (tid < E && cnt[tid] > 0) {
      const int sl = p.lut[(size_t)l * E + tid];
      if (sl >= 0 && sl < p.S) {
        p.prot_epoch[sl] = ep;
        atomicAdd(&sh_misc[2], 1);
      } else {
        if (sl >= p.S) set_status(p.status, MOE_ERR_BOUNDS);
        is_miss = 1;
      }
    }
    // compaction by warp ballots (all lanes of warps 0..7 take part)
    unsigned miss_bal = 0;
    if (warp < (kMaxE / 32)) {
      miss_bal = __ballot_sync(0xffffffffu, is_miss);
      if (lane == 0) wcnt[0][warp] = __popc(miss_bal);
    }
    __syncthreads();
    if (warp < (kMaxE / 32) && is_miss) {
      int before = 0;
      for (int w2 = 0; w2 < warp; ++w2) before += wcnt[0][w2];
      miss_list[before + __popc(miss_bal & ((1u << lane) - 1u))] = tid;
    }
    if (tid == 0) {
      int n = 0;
      for (int w2 = 0; w2 < kMaxE / 32; ++w2) n += wcnt[0][w2];
      sh_misc[0] = n;
    }
    __syncthreads();
    const int n_miss = sh_misc[0];
    const size_t rec = p.lay.rec;
    for (int mi = 0; mi < n_miss; ++mi) {
      const int e = miss_list[mi];
      // lowest free slot
      unsigned long long key = ~0ull;
      for (int s2 = tid; s2 < p.S; s2 += kPlanThreads)
        if (p.owner[s2] < 0) { key = (unsigned long long)s2; break; }
      key = block_min_u64(key, red64);
      int victim = key == ~0ull ? -1 : (int)key;
      if (victim < 0) {
        // lowest score among this layer's slots that this step does not need
        key = ~0ull;
        for (int s2 = tid; s2 < p.S; s2 += kPlanThreads) {
          const int o = p.owner[s2];
          if (o >= 0 && o < p.L * E && o / E == l && p.prot_epoch[s2] != ep) {
            const unsigned long long kk = score_key(p.score[o], s2);
            key = kk < key ? kk : key;
          }
        }
        key = block_min_u64(key, red64);
        if (key == ~0ull) {
          // lowest score among other layers' slots
          for (int s2 = tid; s2 < p.S; s2 += kPlanThreads) {
            const int o = p.owner[s2];
            if (o >= 0 && o < p.L * E && o / E != l) {
              const unsigned long long kk = score_key(p.score[o], s2);
              key = kk < key ? kk : key;
            }
          }
          key = block_min_u64(key, red64);
        }
        victim = key == ~0ull ? -1 : (int)(key & 0xffffffffu);
      }
      if (tid == 0) {
        if (victim < 0) {
          // no slot can be freed: copy into a one-step record for this call only
          const int b = sh_misc[4];
          sh_misc[4] = b + 1;
          int rid = 0;
          if (b < p.n_bypass) rid = p.S + b;
          else set_status(p.status, MOE_ERR_CAPACITY);
          bypass_rid[e] = rid;
          const int nc = sh_misc[3];
          a.sc.copies[nc].src = p.host_dev + ((size_t)l * E + e) * rec;
          a.sc.copies[nc].dst = p.records + (size_t)rid * rec;
          sh_misc[3] = nc + 1;
        } else {
          const int old = p.owner[victim];
          if (old >= 0) {
            if (old < p.L * E) p.lut[old] = -1;
            else set_status(p.status, MOE_ERR_BOUNDS);
            sh_misc[5] += 1;
          }
          p.owner[victim] = l * E + e;
          p.lut[(size_t)l * E + e] = victim;
          p.tag[victim] += 1u;
          p.prot_epoch[victim] = ep;
          const int nc = sh_misc[3];
          a.sc.copies[nc].src = p.host_dev + ((size_t)l * E + e) * rec;
          a.sc.copies[nc].dst = p.slots + (size_t)victim * rec;
          sh_misc[3] = nc + 1;
        }
      }
      __syncthreads();
    }
    if (tid == 0) {
      *a.sc.n_copy = sh_misc[3];
      *p.epoch = ep;
      atomicAdd(&p.stats[ST_HITS], (unsigned long long)sh_misc[2]);
      atomicAdd(&p.stats[ST_MISSES], (unsigned long long)n_miss);
      atomicAdd(&p.stats[ST_BYPASS], (unsigned long long)sh_misc[4]);
      atomicAdd(&p.stats[ST_EVICT], (unsigned long long)sh_misc[5]);
      atomicAdd(&p.stats[ST_BYTES], (unsigned long long)sh_misc[3] * rec);   // slot fills + one-step records
    }
    __syncthreads();
  } else if (tid == 0) {
    *a.sc.n_copy = 0;
  }

  // ------------------------------------------------------ a7 permutation
  if (a.flags & PLAN_PERMUTE) {
    // exclusive scan of the per-expert counts (warp 0, 32 experts per pass)
    if (warp == 0) {
      int run = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int c = e < E ? cnt[e] : 0;
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        if (e < E) offs[e] = run + inc - c;
        run += __shfl_sync(0xffffffffu, inc, 31);
      }
      if (lane == 0) offs[E] = run;
    }
    __syncthreads();
    for (int e = tid; e < E; e += kPlanThreads) base[e] = offs[e];
    for (int e = tid; e <= E; e += kPlanThreads) a.sc.offs[e] = offs[e];
    __syncthreads();
    // stable scatter, 1024 entries per pass
    for (int c0 = 0; c0 < Tk; c0 += kPlanThreads) {
      const int i = c0 + tid;
      int e = -1;
      if (i < Tk) {
        e = a.ids[i];
        if ((unsigned)e >= (unsigned)E) e = -1;
      }
      for (int j = tid; j < kPlanWarps * E; j += kPlanThreads) wcnt[j / E][j % E] = 0;
      __syncthreads();
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (e >= 0 && rank == 0) wcnt[warp][e] = __popc(peers);
      __syncthreads();
      for (int ee = tid; ee < E; ee += kPlanThreads) {
        int run = 0;
        for (int w2 = 0; w2 < kPlanWarps; ++w2) {
          const int c = wcnt[w2][ee];
          wcnt[w2][ee] = run;
          run += c;
        }
        cnt[ee] = run;    // this pass's total for the expert (counts are no longer needed)
      }
      __syncthreads();
      if (e >= 0) {
        const int r = base[e] + wcnt[warp][e] + rank;
        a.sc.perm_tok[r] = i / k;
        a.sc.perm_w[r] = a.w[i];
        a.sc.perm_ent[r] = i;
      }
      __syncthreads();
      for (int ee = tid; ee < E; ee += kPlanThreads) base[ee] += cnt[ee];
      __syncthreads();
    }
    // slot read by every (t, j) entry
    for (int i = tid; i < Tk; i += kPlanThreads) {
      const int e = a.ids[i];
      int sl = -1;
      if ((unsigned)e < (unsigned)E) {
        if (a.flags & PLAN_STAGED) sl = -2;      // read from a staging region
        else sl = p.lut[(size_t)l * E + e];
      }
      a.sc.slots_out[i] = sl;
    }
    // work list: experts with rows, ascending id, then the shared expert
    int has = 0;
    if (tid < E) has = (offs[tid + 1] - offs[tid]) > 0;
    unsigned has_bal = 0;
    if (warp < kMaxE / 32) {
      has_bal = __ballot_sync(0xffffffffu, has);
      if (lane == 0) red64[warp] = __popc(has_bal);
    }
    __syncthreads();
    if (warp < kMaxE / 32 && has) {
      int before = 0;
      for (int w2 = 0; w2 < warp; ++w2) before += (int)red64[w2];
      const int pos = before + __popc(has_bal & ((1u << lane) - 1u));
      const int e = tid;
      int rid;
      if (a.flags & PLAN_STAGED) {
        rid = p.rid_staging0 + a.region * E + e;
      } else {
        const int sl = p.lut[(size_t)l * E + e];
        rid = (sl >= 0 && sl < p.S) ? sl : (bypass_rid[e] >= 0 ? bypass_rid[e] : 0);
      }
      WorkEntry we;
      we.rec = p.records + (size_t)rid * p.lay.rec;
      we.row0 = offs[e];
      we.n = offs[e + 1] - offs[e];
      we.expert = e;
      we.rid = rid;
      a.sc.work[pos] = we;
      pos_of[e] = pos;
    }
    if (tid == 0) {
      int n = 0;
      for (int w2 = 0; w2 < kMaxE / 32; ++w2) n += (int)red64[w2];
      if (p.shared) {
        WorkEntry we;
        we.rid = p.rid_shared0 + l;
        we.rec = p.records + (size_t)we.rid * p.lay.rec;
        we.row0 = Tk;
        we.n = T;
        we.expert = -1;
        a.sc.work[n] = we;
        n += 1;
      }
      *a.sc.n_work = n;
      sh_misc[6] = n;
    }
    if (p.shared) {
      for (int t = tid; t < T; t += kPlanThreads) {
        a.sc.perm_tok[Tk + t] = t;
        a.sc.perm_w[Tk + t] = 1.f;
      }
    }
    // dense routing weights for the tensor-core path: wmat[pos][t] = w of token t for that entry
    if (a.npad > 0) {
      __syncthreads();
      const int nw = sh_misc[6];
      const int np = a.npad;
      for (int j = tid; j < nw * np; j += kPlanThreads) a.sc.wmat[j] = 0.f;
      __syncthreads();
      for (int i = tid; i < Tk; i += kPlanThreads) {
        const int e = a.ids[i];
        if ((unsigned)e < (unsigned)E && pos_of[e] >= 0) a.sc.wmat[(size_t)pos_of[e] * np + i / k] = a.w[i];
      }
      if (p.shared)
        for (int t = tid; t < T; t += kPlanThreads) a.sc.wmat[(size_t)(nw - 1) * np + t] = 1.f;
    }
  }
}

int launch_plan(const PoolDev& p, const Scratch& sc, int layer, int T, const int32_t* ids, const float* w,
                const float* probs, int flags, int region, int npad, cudaStream_t s) {
  PlanArgs a;
  a.p = p;
  a.sc = sc;
  a.layer = layer;
  a.T = T;
  a.flags = flags;
  a.region = region;
  a.npad = npad;
  a.ids = ids;
  a.w = w;
  a.probs = probs;
  plan_kernel<<<1, kPlanThreads, 0, s>>>(a);
  return 1;
}

}  // namespace moeslot
