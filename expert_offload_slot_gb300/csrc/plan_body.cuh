// Device code of steps a3/a4/a5/a7 (routing history, table, victims,
// permutation), shared by the plan kernel and the decode-layer kernel.  See
// k_plan.cu for the sources and the latency plan.
#pragma once
#include "moeslot_internal.cuh"

namespace moeslot {

constexpr int kMaxE = 256;
constexpr int kTokBlock = 32;
constexpr int kOwnerSmemMax = 24576;   // slots whose owner is staged in shared memory
constexpr int kIdsSmemMax = 4096;      // routing entries (T*k) staged in shared memory
constexpr int kStageUnroll = 8;        // loads in flight per thread while staging

struct PlanArgs {
  PoolDev p;
  Scratch sc;
  int layer, T, flags, region, npad;
  const int32_t* ids;
  const float* w;
  const float* probs;
  int owner_cap;        // slots staged in shared memory (S, or 0 for the global-memory path)
  int tok_rows;         // rows of the token staging area
  bool zero_sync = true;                 // zero the expert kernel's counters (false: the caller does)
  const uint32_t* snap_wait = nullptr;   // if set: before writing the table, wait for *snap_wait >= snap_target
  uint32_t snap_target = 0;              // (other CTAs' reads of this layer's table row)
  uint32_t* slots_flag = nullptr;        // if set: released once the table holds this step's slots
  int gather_bn = 128;                   // gather path: token rows per tile (64, 128 or 256)
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

// Block-wide minimum over NT threads; every thread must call it.  `red` holds NT / 32 entries.
template <int NT>
__device__ unsigned long long block_min_u64(unsigned long long v, unsigned long long* red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  v = warp_min_u64(v);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (warp == 0) {
    unsigned long long r = lane < NT / 32 ? red[lane] : ~0ull;
    r = warp_min_u64(r);
    if (lane == 0) red[0] = r;
  }
  __syncthreads();
  const unsigned long long out = red[0];
  __syncthreads();
  return out;
}

struct SmemLayout {
  size_t hs, hsel, tok, owner, prot, ids, w, pfs, total;
};

__host__ __device__ inline size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

__host__ __device__ inline SmemLayout plan_smem_layout(int E, int W, int tok_rows, int owner_cap, int nwarps) {
  SmemLayout L;
  size_t off = 0;
  L.hs = off;
  off = align16(off + (size_t)W * E * 4);
  L.hsel = off;
  off = align16(off + (size_t)W * E);
  L.tok = off;   // token staging, later reused by the permutation's per-warp counts
  const size_t tok_bytes = (size_t)tok_rows * E * 4, wc_bytes = (size_t)nwarps * E * 4;
  off = align16(off + (tok_bytes > wc_bytes ? tok_bytes : wc_bytes));
  L.owner = off;
  off = align16(off + (size_t)owner_cap * 4);
  L.prot = off;
  off = align16(off + (size_t)((owner_cap + 31) / 32) * 4);
  L.ids = off;
  off = align16(off + (size_t)kIdsSmemMax * 4);
  L.w = off;
  off = align16(off + (size_t)kIdsSmemMax * 4);
  L.pfs = off;   // the layer's pending-prefetch slot of each expert
  off = align16(off + (size_t)E * 4);
  L.total = off;
  return L;
}

// Copy n elements global -> shared with kStageUnroll loads in flight per thread (NT threads).
template <int NT, typename T>
__device__ __forceinline__ void stage_copy(T* dst, const T* __restrict__ src, int n) {
  for (int j0 = threadIdx.x; j0 < n; j0 += NT * kStageUnroll) {
    T v[kStageUnroll];
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) {
      const int j = j0 + u * NT;
      if (j < n) v[u] = src[j];
    }
#pragma unroll
    for (int u = 0; u < kStageUnroll; ++u) {
      const int j = j0 + u * NT;
      if (j < n) dst[j] = v[u];
    }
  }
}

// Asynchronous global -> shared copy of n bytes (cp.async, no registers): 16-byte
// pieces while both addresses are 16-byte aligned, the rest with plain loads.  The
// copies land by the next cp_async_wait_all() of each issuing thread.
template <int NT>
__device__ __forceinline__ void stage_async(void* dst, const void* src, size_t n) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  const char* sp = static_cast<const char*>(src);
  size_t n16 = ((d | reinterpret_cast<uintptr_t>(sp)) & 15u) == 0 ? n / 16 : 0;
  for (size_t i = threadIdx.x; i < n16; i += NT)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + (uint32_t)(16 * i)), "l"(sp + 16 * i) : "memory");
  for (size_t i = 16 * n16 + threadIdx.x; i < n; i += NT) static_cast<char*>(dst)[i] = sp[i];
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The parts of the plan's input that do not depend on the step's routing (the
// layer's history rings and the owner of every slot): started early, in flight
// until plan_body waits for them.
template <int NT>
__device__ void plan_prestage(const PlanArgs& a, uint8_t* dsm) {
  const PoolDev& p = a.p;
  const int E = p.E, l = a.layer, W = p.W;
  const SmemLayout SL = plan_smem_layout(E, W, a.tok_rows, a.owner_cap, NT / 32);
  if (a.flags & PLAN_HISTORY) {
    stage_async<NT>(dsm + SL.hs, p.hist_s + (size_t)l * W * E, (size_t)W * E * 4);
    stage_async<NT>(dsm + SL.hsel, p.hist_sel + (size_t)l * W * E, (size_t)W * E);
  }
  if ((a.flags & PLAN_CACHE) && a.owner_cap >= p.S) stage_async<NT>(dsm + SL.owner, p.owner, (size_t)p.S * 4);
}

// The plan of one layer call, run by all NT threads of one CTA.  dsm: dynamic shared
// memory laid out by plan_smem_layout(E, W, a.tok_rows, a.owner_cap, NT / 32);
// prestaged: plan_prestage<NT> already ran on this CTA.
template <int NT>
__device__ void plan_body(const PlanArgs& a, uint8_t* dsm, bool prestaged = false) {
  constexpr int kPlanThreads = NT;
  constexpr int kPlanWarps = NT / 32;
  __shared__ int cnt[kMaxE];
  __shared__ int offs[kMaxE + 1];
  __shared__ int base[kMaxE];
  __shared__ int lut_s[kMaxE];
  __shared__ float score_s[kMaxE];
  __shared__ int miss_list[kMaxE];
  __shared__ int victim_s[kMaxE];
  __shared__ int old_s[kMaxE];
  __shared__ int bypass_rid[kMaxE];   // one-step record of a miss that got no slot, or -1
  __shared__ int pos_of[kMaxE];       // work-list position of each expert, or -1
  __shared__ int missed[kMaxE];       // 1 if the expert was not resident at the start of this step
  __shared__ int wtmp[3][kMaxE / 32];
  __shared__ unsigned long long red64[kPlanWarps];
  __shared__ float red4[kPlanWarps][4];
  __shared__ int sh_misc[12];   // 0 n_miss, 2 hits, 4 bypass, 5 evictions, 6 n_work

  const PoolDev& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = p.E, k = p.k, T = a.T, l = a.layer, W = p.W;
  const int Tk = T * k;
  const SmemLayout SL = plan_smem_layout(E, W, a.tok_rows, a.owner_cap, kPlanWarps);
  float* hs = reinterpret_cast<float*>(dsm + SL.hs);
  uint8_t* hsel = dsm + SL.hsel;
  float* tok = reinterpret_cast<float*>(dsm + SL.tok);
  int* wcnt = reinterpret_cast<int*>(dsm + SL.tok);          // [kPlanWarps][E], after the history phase
  int* owner_s = reinterpret_cast<int*>(dsm + SL.owner);
  uint32_t* prot = reinterpret_cast<uint32_t*>(dsm + SL.prot);
  const bool owner_in_smem = a.owner_cap >= p.S;
  // routing entries: shared memory when they fit, else global memory
  const bool ids_in_smem = Tk <= kIdsSmemMax;
  int32_t* ids_s = reinterpret_cast<int32_t*>(dsm + SL.ids);
  float* w_s = reinterpret_cast<float*>(dsm + SL.w);
  const int32_t* ids = ids_in_smem ? ids_s : a.ids;
  const float* wrt = ids_in_smem ? w_s : a.w;

  // ------------------------------------------------------------ stage (one round trip)
  for (int e = tid; e < E; e += kPlanThreads) {
    cnt[e] = 0;
    bypass_rid[e] = -1;
    pos_of[e] = -1;
    missed[e] = 0;
  }
  if (tid < 12) sh_misc[tid] = 0;
  // arrival counters and readiness flags of the expert kernel that follows
  if (a.zero_sync)
    for (int i = tid; i < a.sc.n_ffn_sync; i += kPlanThreads) a.sc.ffn_sync[i] = 0;
  const bool hist = (a.flags & PLAN_HISTORY) != 0;
  const bool cache = (a.flags & PLAN_CACHE) != 0;
  int t_step = 0;
  float ema0 = 0.f;
  int last0 = -1;
  if (!prestaged) plan_prestage<NT>(a, dsm);
  if (ids_in_smem) {
    stage_async<NT>(ids_s, a.ids, (size_t)Tk * 4);
    if (a.w && (a.flags & PLAN_PERMUTE)) stage_async<NT>(w_s, a.w, (size_t)Tk * 4);
  }
  if (hist) {
    t_step = p.step[l];
    // short steps stage the probabilities; longer ones are summed from global memory below
    if (T <= kTokBlock) stage_async<NT>(tok, a.probs, (size_t)T * E * 4);
    if (tid < E) {
      ema0 = p.ema[(size_t)l * E + tid];
      last0 = p.last_sel[(size_t)l * E + tid];
    }
  }
  int* pfs = reinterpret_cast<int*>(dsm + SL.pfs);
  const bool pf = cache && p.pf_used;
  if (cache) {
    if (tid < E) lut_s[tid] = p.lut[(size_t)l * E + tid];
    if (pf && tid < E) pfs[tid] = p.pf_slot[(size_t)l * E + tid];
    if (owner_in_smem)
      for (int j = tid; j < (p.S + 31) / 32; j += kPlanThreads) prot[j] = 0u;
  }
  cp_async_wait_all();
  __syncthreads();
  for (int i = tid; i < Tk; i += kPlanThreads) {
    const int e = ids[i];
    if ((unsigned)e >= (unsigned)E) set_status(p.status, MOE_ERR_BOUNDS);
    else atomicAdd(&cnt[e], 1);
  }
  __syncthreads();

  // ------------------------------------------------------------ a3 history
  float s = 0.f;                      // this thread's expert's router score of the step (tid < E)
  if (hist) {
    const int t = t_step;
    const int ring = t % W;
    const bool mine = tid < E;
    float m = 0.f;
    int count = 0, age = 0;
    if (mine) {
      const int e = tid;
      // token-averaged probability: one sum per expert in ascending token order
      if (T <= kTokBlock) {
        for (int tt = 0; tt < T; ++tt) s = __fadd_rn(s, tok[tt * E + e]);
      } else {
        // coalesced across the threads (consecutive experts); 16 loads in flight, then the adds in order
        const float* pe = a.probs + e;
        int tt = 0;
        for (; tt + 16 <= T; tt += 16) {
          float v[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = pe[(size_t)(tt + q) * E];
#pragma unroll
          for (int q = 0; q < 16; ++q) s = __fadd_rn(s, v[q]);
        }
        for (; tt < T; ++tt) s = __fadd_rn(s, pe[(size_t)tt * E]);
      }
      s = __fdiv_rn(s, (float)T);
      const int sel = cnt[e] > 0 ? 1 : 0;
      hs[ring * E + e] = s;
      hsel[ring * E + e] = (uint8_t)sel;
      const size_t he = ((size_t)l * W + ring) * E + e;
      p.hist_s[he] = s;
      p.hist_sel[he] = (uint8_t)sel;
      m = __fadd_rn(__fmul_rn(p.lam, ema0), __fmul_rn(p.one_minus_lam, sel ? 1.f : 0.f));
      p.ema[(size_t)l * E + e] = m;
      int last = last0;
      if (sel) {
        last = t;
        p.last_sel[(size_t)l * E + e] = t;
      }
      age = t - last;
      for (int j = 0; j < W; ++j) count += hsel[j * E + e];
    }
    float sc = 0.f;
    if (p.policy == MOE_EVICT_CORE) {
      // the four layer maxima in one block reduction
      float v4[4] = {mine ? (float)count : -INFINITY, mine ? m : -INFINITY, mine ? s : -INFINITY,
                     mine ? (float)age : -INFINITY};
#pragma unroll
      for (int q = 0; q < 4; ++q) v4[q] = warp_max(v4[q]);
      if (lane == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) red4[warp][q] = v4[q];
      }
      __syncthreads();
      if (warp == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float r = lane < kPlanWarps ? red4[lane][q] : -INFINITY;
          r = warp_max(r);
          if (lane == 0) red4[0][q] = r;
        }
      }
      __syncthreads();
      const float cmax = red4[0][0], mmax = red4[0][1], smax = red4[0][2], amax = red4[0][3];
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
          acc = __fadd_rn(acc, hs[idx * E + tid]);
        }
        sc = __fsub_rn(acc, s);
      }
    } else {
      if (mine) sc = (float)(t - age);             // last selection step, -1 if never
    }
    if (mine) {
      p.score[(size_t)l * E + tid] = sc;
      score_s[tid] = sc;
    }
    if (tid == 0) {
      p.step[l] = t + 1;
      atomicAdd(&p.stats[ST_STEPS], 1ull);
    }
    __syncthreads();
  } else if (cache) {
    if (tid < E) score_s[tid] = p.score[(size_t)l * E + tid];
    __syncthreads();
  }

  // ------------------------------------------------------- a4/a5 table, misses
  if (cache) {
    const int S = p.S;
    const size_t rec = p.lay.rec;
    int ep = 0;
    if (!owner_in_smem) ep = *p.epoch + 1;
    // protect resident needed experts; list misses in ascending expert id
    int is_miss = 0;
    if (tid < E && cnt[tid] > 0) {
      const int sl = lut_s[tid];
      if (sl >= 0 && sl < S) {
        if (owner_in_smem) atomicOr(&prot[sl >> 5], 1u << (sl & 31));
        else p.prot_epoch[sl] = ep;
        atomicAdd(&sh_misc[2], 1);
      } else {
        if (sl >= S) set_status(p.status, MOE_ERR_BOUNDS);
        is_miss = 1;
        missed[tid] = 1;
      }
    }
    unsigned miss_bal = 0;
    if (warp < (kMaxE / 32)) {
      miss_bal = __ballot_sync(0xffffffffu, is_miss);
      if (lane == 0) wtmp[0][warp] = __popc(miss_bal);
    }
    __syncthreads();
    if (warp < (kMaxE / 32) && is_miss) {
      int before = 0;
      for (int w2 = 0; w2 < warp; ++w2) before += wtmp[0][w2];
      miss_list[before + __popc(miss_bal & ((1u << lane) - 1u))] = tid;
    }
    if (tid == 0) {
      int n = 0;
      for (int w2 = 0; w2 < kMaxE / 32; ++w2) n += wtmp[0][w2];
      sh_misc[0] = n;
    }
    __syncthreads();
    const int n_miss = sh_misc[0];
    // victims, one miss at a time (ascending expert id): lowest free slot, else the
    // lowest-score slot of this layer that this step does not need, else of another layer
    // a slot whose prefetch copy may still be in flight (its tag not yet written back) is
    // never a victim: the late copy would overwrite the new occupant
    auto busy = [&](int s2) -> bool {
      return pf && *reinterpret_cast<const volatile uint32_t*>(p.landed + s2) != p.pf_tag[s2];
    };
    for (int mi = 0; mi < n_miss; ++mi) {
      // a miss whose expert is pending (its prefetch not committed): the pending slot takes it
      const int pend = pf ? pfs[miss_list[mi]] : -1;
      unsigned long long key = ~0ull;
      for (int s2 = tid; pend < 0 && s2 < S; s2 += kPlanThreads) {
        const int o = owner_in_smem ? owner_s[s2] : p.owner[s2];
        if (o == -1) { key = (unsigned long long)s2; break; }
      }
      if (pend < 0) key = block_min_u64<NT>(key, red64);
      int victim = pend >= 0 ? pend : key == ~0ull ? -1 : (int)key;
      if (victim < 0) {
        key = ~0ull;
        for (int s2 = tid; s2 < S; s2 += kPlanThreads) {
          const int o = owner_in_smem ? owner_s[s2] : p.owner[s2];
          const bool pr = owner_in_smem ? ((prot[s2 >> 5] >> (s2 & 31)) & 1u) != 0u : p.prot_epoch[s2] == ep;
          if (o >= 0 && o < p.L * E && o / E == l && !pr && !busy(s2)) {
            const unsigned long long kk = score_key(score_s[o - l * E], s2);
            key = kk < key ? kk : key;
          }
        }
        key = block_min_u64<NT>(key, red64);
        if (key == ~0ull) {
          for (int s2 = tid; s2 < S; s2 += kPlanThreads) {
            const int o = owner_in_smem ? owner_s[s2] : p.owner[s2];
            if (o >= 0 && o < p.L * E && o / E != l && !busy(s2)) {
              const unsigned long long kk = score_key(p.score[o], s2);
              key = kk < key ? kk : key;
            }
          }
          key = block_min_u64<NT>(key, red64);
        }
        victim = key == ~0ull ? -1 : (int)(key & 0xffffffffu);
      }
      if (tid == 0) {
        const int e = miss_list[mi];
        victim_s[mi] = victim;
        if (victim < 0) {
          old_s[mi] = -1;
          const int b = sh_misc[4]++;
          int rid = 0;
          if (b < p.n_bypass) rid = S + b;
          else set_status(p.status, MOE_ERR_CAPACITY);
          bypass_rid[e] = rid;
        } else {
          const int old = pend >= 0 ? -3 : owner_in_smem ? owner_s[victim] : p.owner[victim];
          old_s[mi] = old;             // -3: the expert's own pending slot
          if (old >= 0) sh_misc[5] += 1;
          if (old >= 0 && old / E == l) lut_s[old - l * E] = -1;   // the row stays current in shared memory
          if (owner_in_smem) {
            owner_s[victim] = l * E + e;
            prot[victim >> 5] |= 1u << (victim & 31);
          } else {
            p.owner[victim] = l * E + e;
            p.prot_epoch[victim] = ep;
          }
          lut_s[e] = victim;
        }
      }
      __syncthreads();
    }
    if (a.snap_wait) {
      // the table row may change only once every reader has its copy (bounded wait: the
      // pool's wait limit of global time, 1 s by default)
      if (tid == 0) {
        uint64_t t0, now;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
        uint32_t v = 0;
        do {
          asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a.snap_wait) : "memory");
          asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
        } while (v < a.snap_target && now - t0 < p.wait_ns);
        if (v < a.snap_target) set_status(p.status, MOE_ERR_TIMEOUT);
      }
      __syncthreads();
    }
    // apply the decisions in parallel: table, owners, tags, copy list (one copy per miss)
    if (tid < n_miss) {
      const int e = miss_list[tid], v = victim_s[tid], old = old_s[tid];
      CopyJob job;
      job.src = p.host_dev + ((size_t)l * E + e) * rec;
      if (v >= 0) {
        if (old >= 0 && old < p.L * E) p.lut[old] = -1;
        if (old == -3) {               // a pending prefetch of e, demanded before its commit
          p.pf_expert[v] = -1;
          p.pf_slot[(size_t)l * E + e] = -1;
          atomicAdd(&p.stats[ST_PF_DEMANDED], 1ull);
        }
        p.lut[(size_t)l * E + e] = v;
        p.owner[v] = l * E + e;
        atomicAdd(&p.tag[v], 1u);
        job.dst = p.records + (size_t)v * rec;
      } else {
        job.dst = p.records + (size_t)bypass_rid[e] * rec;
      }
      a.sc.copies[tid] = job;
    }
    if (tid == 0) {
      *a.sc.n_copy = n_miss;
      if (!owner_in_smem) *p.epoch = ep;
      atomicAdd(&p.stats[ST_HITS], (unsigned long long)sh_misc[2]);
      atomicAdd(&p.stats[ST_MISSES], (unsigned long long)n_miss);
      atomicAdd(&p.stats[ST_BYPASS], (unsigned long long)sh_misc[4]);
      atomicAdd(&p.stats[ST_EVICT], (unsigned long long)sh_misc[5]);
      atomicAdd(&p.stats[ST_BYTES], (unsigned long long)n_miss * rec);   // slot fills + one-step records
    }
  } else if (tid == 0) {
    *a.sc.n_copy = 0;
  }
  if (a.slots_flag) {
    // the table is final for this step: copies may move to the chosen slots
    __threadfence();
    __syncthreads();
    if (tid == 0)
      asm volatile("fence.acq_rel.gpu;\n red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.slots_flag) : "memory");
  }

  // ------------------------------------------------ asynchronous prefetch (SeqMoE)
  // Issue: up to pf_per_step minus this step's misses (the copy volume already committed to
  // the layer, HybriMoE's priority) of the layer's experts the step does not need, neither
  // resident nor pending, highest router score first; each takes the lowest free slot, else
  // the lowest-score slot of this layer the step does not need.  The slot turns pending
  // (owner -2 - its expert) with a fresh tag, and the request goes to the host thread through the
  // mapped control region.  Commit: every pending slot whose written-back tag equals its
  // own becomes resident; a stale or superseded write-back never matches.
  if (cache && p.pf_used) {
    __syncthreads();
    const int S = p.S;
    const int n_miss = sh_misc[0];
    int* pfs = reinterpret_cast<int*>(dsm + SL.pfs);
    auto busy = [&](int s2) -> bool {
      return *reinterpret_cast<const volatile uint32_t*>(p.landed + s2) != p.pf_tag[s2];
    };
    if (tid == 0) {
      int b = p.pf_per_step - n_miss;
      b = min(b, kPfRing - (int)(*p.pf_head - p.pf_ctl->tail));
      b = min(b, kPfMaxPending - *p.pf_n);
      sh_misc[7] = b > 0 ? b : 0;
      sh_misc[8] = 0;
    }
    __syncthreads();
    const int budget = sh_misc[7];
    const int ep = owner_in_smem ? 0 : *p.epoch;
    // candidates are fixed when the phase starts (an expert this phase evicts is not one)
    const bool cand = tid < E && cnt[tid] == 0 && lut_s[tid] < 0 && pfs[tid] < 0;
    for (int b = 0; b < budget; ++b) {
      unsigned long long ck = ~0ull;
      if (cand && pfs[tid] < 0) ck = score_key(-s, tid);
      ck = block_min_u64<NT>(ck, red64);
      if (ck == ~0ull) break;
      const int e = (int)(ck & 0xffffffffu);
      unsigned long long key = ~0ull;
      for (int s2 = tid; s2 < S; s2 += kPlanThreads) {
        const int o = owner_in_smem ? owner_s[s2] : p.owner[s2];
        if (o == -1) { key = (unsigned long long)s2; break; }
      }
      key = block_min_u64<NT>(key, red64);
      int v = key == ~0ull ? -1 : (int)key;
      if (v < 0) {
        key = ~0ull;
        for (int s2 = tid; s2 < S; s2 += kPlanThreads) {
          const int o = owner_in_smem ? owner_s[s2] : p.owner[s2];
          const bool pr = owner_in_smem ? ((prot[s2 >> 5] >> (s2 & 31)) & 1u) != 0u : p.prot_epoch[s2] == ep;
          if (o >= 0 && o < p.L * E && o / E == l && !pr && !busy(s2)) {
            const unsigned long long kk = score_key(score_s[o - l * E], s2);
            key = kk < key ? kk : key;
          }
        }
        key = block_min_u64<NT>(key, red64);
        v = key == ~0ull ? -1 : (int)(key & 0xffffffffu);
      }
      if (v < 0) break;
      if (tid == 0) {
        const int old = owner_in_smem ? owner_s[v] : p.owner[v];
        if (old >= 0 && old < p.L * E) {
          p.lut[old] = -1;
          if (old / E == l) lut_s[old - l * E] = -1;
          atomicAdd(&p.stats[ST_EVICT], 1ull);
        }
        if (owner_in_smem) owner_s[v] = -2 - (l * E + e);    // pending: -2 - the expert it will hold
        p.owner[v] = -2 - (l * E + e);
        p.pf_expert[v] = l * E + e;
        p.pf_slot[(size_t)l * E + e] = v;
        pfs[e] = v;
        const uint32_t tg = atomicAdd(&p.tag[v], 1u) + 1u;
        p.pf_tag[v] = tg;
        const int k2 = sh_misc[8];
        volatile PfReq* r = &p.pf_ctl->req[(*p.pf_head + (uint32_t)k2) % kPfRing];   // mapped host memory
        r->slot = v;
        r->flat = l * E + e;
        r->tag = tg;
        p.pf_list[*p.pf_n + k2] = v;
        sh_misc[8] = k2 + 1;
      }
      __syncthreads();
    }
    if (tid == 0) {
      const int issued = sh_misc[8];
      if (issued > 0) {
        *p.pf_n += issued;
        const uint32_t h = *p.pf_head + (uint32_t)issued;
        *p.pf_head = h;
        __threadfence_system();        // the requests before the head that publishes them
        p.pf_ctl->head = h;
        atomicAdd(&p.stats[ST_PF_ISSUED], (unsigned long long)issued);
      }
      // commits, in request order
      const int n = *p.pf_n;
      int w = 0, committed = 0;
      for (int i = 0; i < n; ++i) {
        const int q = p.pf_list[i];
        const int x = p.pf_expert[q];
        if (x < 0) continue;                                        // demanded before its commit
        if (*reinterpret_cast<const volatile uint32_t*>(p.landed + q) == p.pf_tag[q]) {
          p.owner[q] = x;
          p.lut[x] = q;
          p.pf_slot[x] = -1;
          p.pf_expert[q] = -1;
          if (x / E == l) lut_s[x - l * E] = q;
          if (owner_in_smem) owner_s[q] = x;
          ++committed;
          continue;
        }
        p.pf_list[w++] = q;
      }
      *p.pf_n = w;
      if (committed) atomicAdd(&p.stats[ST_PF_COMMITTED], (unsigned long long)committed);
      // the GPU's position and the miss flag, for the host thread
      p.pf_ctl->layer = l;
      p.pf_ctl->step = t_step;
      if (n_miss > 0) p.pf_ctl->demand = p.pf_ctl->demand + 1u;
    }
    __syncthreads();
  }

  // ------------------------------------------------------ a7 permutation
  if (a.flags & PLAN_PERMUTE) {
    if (!cache && tid < E) lut_s[tid] = p.lut[(size_t)l * E + tid];
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
    if (Tk <= kPlanThreads) {
      // one entry per thread: its rank among the earlier entries of the same expert
      const int i = tid;
      int e = -1;
      if (i < Tk) {
        e = ids[i];
        if ((unsigned)e >= (unsigned)E) e = -1;
      }
      if (e >= 0) {
        int rank = 0;
        for (int j = 0; j < i; ++j) rank += ids[j] == e;
        const int r = offs[e] + rank;
        a.sc.perm_tok[r] = i / k;
        a.sc.perm_w[r] = wrt[i];
        a.sc.perm_ent[r] = i;
        if (a.flags & PLAN_GATHER) a.sc.inv[i] = r;
      }
    }
    // stable scatter, kPlanThreads entries per pass
    for (int c0 = 0; Tk > kPlanThreads && c0 < Tk; c0 += kPlanThreads) {
      const int i = c0 + tid;
      int e = -1;
      if (i < Tk) {
        e = ids[i];
        if ((unsigned)e >= (unsigned)E) e = -1;
      }
      for (int j = tid; j < kPlanWarps * E; j += kPlanThreads) wcnt[j] = 0;
      __syncthreads();
      const unsigned peers = __match_any_sync(0xffffffffu, e);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (e >= 0 && rank == 0) wcnt[warp * E + e] = __popc(peers);
      __syncthreads();
      for (int ee = tid; ee < E; ee += kPlanThreads) {
        int run = 0;
        for (int w2 = 0; w2 < kPlanWarps; ++w2) {
          const int c = wcnt[w2 * E + ee];
          wcnt[w2 * E + ee] = run;
          run += c;
        }
        cnt[ee] = run;    // this pass's total for the expert (the full counts are in offs)
      }
      __syncthreads();
      if (e >= 0) {
        const int r = base[e] + wcnt[warp * E + e] + rank;
        a.sc.perm_tok[r] = i / k;
        a.sc.perm_w[r] = wrt[i];
        a.sc.perm_ent[r] = i;
        if (a.flags & PLAN_GATHER) a.sc.inv[i] = r;
      }
      __syncthreads();
      for (int ee = tid; ee < E; ee += kPlanThreads) base[ee] += cnt[ee];
      __syncthreads();
    }
    // slot read by every (t, j) entry
    for (int i = tid; i < Tk; i += kPlanThreads) {
      const int e = ids[i];
      int sl = -1;
      if ((unsigned)e < (unsigned)E) sl = (a.flags & PLAN_STAGED) ? -2 : lut_s[e];
      a.sc.slots_out[i] = sl;
    }
    // work list: experts with rows, ascending id, then the shared expert
    int has = 0;
    if (tid < E) has = (offs[tid + 1] - offs[tid]) > 0;
    unsigned has_bal = 0, hit_bal = 0, mis_bal = 0;
    if (warp < kMaxE / 32) {
      has_bal = __ballot_sync(0xffffffffu, has);
      hit_bal = __ballot_sync(0xffffffffu, has && !(tid < E && missed[tid]));
      mis_bal = __ballot_sync(0xffffffffu, has && (tid < E && missed[tid]));
      if (lane == 0) {
        red64[warp] = __popc(has_bal);
        wtmp[1][warp] = __popc(hit_bal);
        wtmp[2][warp] = __popc(mis_bal);
      }
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
        const int sl = lut_s[e];
        rid = (sl >= 0 && sl < p.S) ? sl : (bypass_rid[e] >= 0 ? bypass_rid[e] : 0);
      }
      WorkEntry we;
      we.rec = p.records + (size_t)rid * p.lay.rec;
      we.row0 = offs[e];
      we.n = offs[e + 1] - offs[e];
      we.expert = e;
      we.rid = rid;
      // UMIA (residual-split records): critical when the step's token-averaged probability s
      // reaches (theta * beta[l]) * gamma of the call's phase
      we.crit = 1;
      if (p.wdt == MOE_RESPLIT_Q4R4) {
        const float g = (a.flags & PLAN_STAGED) ? p.umia_gamma_prefill : p.umia_gamma_decode;
        const float thr = __fmul_rn(__fmul_rn(p.umia_theta, p.umia_beta[l]), g);
        we.crit = s >= thr ? 1 : 0;
        if (we.crit) atomicAdd(&p.stats[ST_CRIT], 1ull);
      }
      a.sc.work[pos] = we;
      pos_of[e] = pos;
      // entries that need no copy this step, and entries that do (both in expert order)
      const unsigned lower = (1u << lane) - 1u;
      if (missed[e]) {
        int b = 0;
        for (int w2 = 0; w2 < warp; ++w2) b += wtmp[2][w2];
        a.sc.elist[(E + 1) + b + __popc(mis_bal & lower)] = pos;
      } else {
        int b = 0;
        for (int w2 = 0; w2 < warp; ++w2) b += wtmp[1][w2];
        a.sc.elist[b + __popc(hit_bal & lower)] = pos;
      }
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
        we.crit = 1;                          // the shared expert runs at high precision
        if (p.wdt == MOE_RESPLIT_Q4R4) atomicAdd(&p.stats[ST_CRIT], 1ull);
        a.sc.work[n] = we;
        n += 1;
      }
      int nh = 0, nm = 0;
      for (int w2 = 0; w2 < kMaxE / 32; ++w2) {
        nh += wtmp[1][w2];
        nm += wtmp[2][w2];
      }
      if (p.shared) a.sc.elist[nh++] = n - 1;    // the shared expert is always resident
      a.sc.ecount[0] = nh;
      a.sc.ecount[1] = nm;
      *a.sc.n_work = n;
      sh_misc[6] = n;
    }
    if (p.shared) {
      for (int t = tid; t < T; t += kPlanThreads) {
        a.sc.perm_tok[Tk + t] = t;
        a.sc.perm_w[Tk + t] = 1.f;
      }
    }
    __syncthreads();
    // gather path: first token tile of every entry (entries in ascending expert id, shared last)
    if ((a.flags & PLAN_GATHER) && warp == 0) {
      const int bn = a.gather_bn;
      int run = 0;
      for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        const int c = e < E ? offs[e + 1] - offs[e] : 0;
        const int v = (c + bn - 1) / bn;
        int inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        if (e < E && c > 0) a.sc.ntile0[pos_of[e]] = run + inc - v;
        run += __shfl_sync(0xffffffffu, inc, 31);
      }
      if (lane == 0) {
        const int nw = sh_misc[6];
        if (p.shared) {
          a.sc.ntile0[nw - 1] = run;
          run += (T + bn - 1) / bn;
        }
        a.sc.ntile0[nw] = run;
        *a.sc.n_rows = Tk + (p.shared ? T : 0);
      }
    }
    // dense routing weights for the tensor-core path: wmat[pos][t] = w of token t for that entry
    if (a.npad > 0) {
      const int nw = sh_misc[6];
      const int np = a.npad;
      for (int j = tid; j < nw * np; j += kPlanThreads) a.sc.wmat[j] = 0.f;
      __syncthreads();
      for (int i = tid; i < Tk; i += kPlanThreads) {
        const int e = ids[i];
        if ((unsigned)e < (unsigned)E && pos_of[e] >= 0) a.sc.wmat[(size_t)pos_of[e] * np + i / k] = wrt[i];
      }
      if (p.shared)
        for (int t = tid; t < T; t += kPlanThreads) a.sc.wmat[(size_t)(nw - 1) * np + t] = 1.f;
    }
  }
}


// Dynamic shared memory of plan_body<NT> for calls of up to Tmax tokens;
// *owner_cap_out = slots whose owner is staged (S, or 0 when they do not fit).
template <int NT>
inline size_t plan_smem_bytes_nt(const PoolDev& p, int Tmax, int* owner_cap_out, int* tok_rows_out,
                                 size_t budget = 200 * 1024) {
  // T <= 32 stages the probabilities themselves (up to 32 rows); larger T reads them
  // from global memory
  (void)Tmax;
  const int tok_rows = kTokBlock;
  int cap = p.S <= kOwnerSmemMax ? p.S : 0;
  SmemLayout L = plan_smem_layout(p.E, p.W, tok_rows, cap, NT / 32);
  if (L.total > budget) {          // very large pools: owners stay in global memory
    cap = 0;
    L = plan_smem_layout(p.E, p.W, tok_rows, 0, NT / 32);
  }
  if (owner_cap_out) *owner_cap_out = cap;
  if (tok_rows_out) *tok_rows_out = tok_rows;
  return L.total;
}

}  // namespace moeslot
