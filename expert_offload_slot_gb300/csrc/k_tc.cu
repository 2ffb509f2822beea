// Step a8 (SwiGLU experts) and a9 (combine) on the 5th-generation tensor cores
// (tcgen05, accumulators in TMEM, operands staged in shared memory by TMA).
//
// Expert (RapidMoE §4.5, Eq. 7): y = W_down (SiLU(W_gate x) ⊙ W_up x).
// Combine (CAP §II-A, Eq. 1): out[t] = sum_j w[t,j] y_j(t) (+ shared expert).
//
// Orientation ("swap AB"): the MMA's M dimension is 128 weight rows and N the
// tokens, so a decode step with a handful of tokens still fills M.  Every
// token of the step is a column of B (N = T rounded up to 16); columns of
// tokens an expert does not serve are masked in the epilogue, which costs
// tensor-core work only — the bound is the weight stream from HBM.
//
//   gate_up: per (work entry u, 128-row tile of I):
//              D_g = W_gate[tile] · xᵀ,  D_u = W_up[tile] · xᵀ     (K = H)
//            epilogue: hbuf[u][t][i] = w(u,t) · SiLU(D_g) · D_u   (bf16; 0 if t
//            is not routed to u) — the routing weight is folded in here.
//   down:    per 128-row tile of H:  D = sum over entries u, K = I of
//              W_down_u[tile] · hbuf[u]ᵀ
//            i.e. the combine is accumulated in TMEM in a fixed order (entries
//            ascending, shared expert last); epilogue: out[t][h] = D (bf16).
//
// When there are fewer output tiles than SMs, each tile's reduction (K for
// gate_up, the entry list for down) is split over several CTAs; each writes
// an fp32 partial tile and the last CTA to arrive sums the partials in split
// order (deterministic) and runs the epilogue.
//
// CTA roles (192 threads): warp 0 lane 0 issues TMA loads into a ring of
// shared-memory stages; warp 1 allocates TMEM and its lane 0 issues the MMAs;
// warps 2..5 (one warpgroup, TMEM lanes 0..127) run the epilogue.  Every
// mbarrier wait is bounded (about one second of global time); a wait that
// gives up records MOE_ERR_TIMEOUT in the status word, and the kernel drains
// its own copies and MMAs (again with bounded waits) before freeing TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "moeslot_internal.cuh"

namespace moeslot {

struct TcMaps {
  CUtensorMap w13;   // [R records][2I rows][H]  bf16, box 64 x 128 x 1
  CUtensorMap w2;    // [R records][H rows][I]   bf16, box 64 x 128 x 1
};

namespace tc {

constexpr int BM = 128;          // weight rows per tile (MMA M)
constexpr int BK = 64;           // K elements per stage (one 128-byte swizzle row)
constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kModeGateUp = 0, kModeDown = 1;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait: false after ~1 s of global time.
__device__ __noinline__ bool mbar_wait(uint64_t* b, uint32_t parity) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try(b, parity)) return true;
    if ((it & 255u) == 0 && global_ns() - t0 > 1000000000ull) return false;
  }
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// tcgen05 ------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] · B[smem desc]ᵀ, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane (load and wait in one block).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B and a 64-element bf16 box width).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor: kind::f16, A = B = bf16, D = fp32, both K-major, M = 128.
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}

struct Args {
  const WorkEntry* work;
  const int32_t* n_work;
  int T, N, H, I, num_sms, stages;
  const float* wmat;   // [E+1][N]
  uint16_t* hbuf;      // [E+1][N][I]
  uint16_t* out;       // [T][H]
  float* partial;
  int32_t* counters;
  int32_t* status;
};

struct Plan {             // the unit decomposition, identical in every role
  int tiles, splits, units, kblocks, mt_per_entry, n_work;
};

template <int MODE>
__device__ __forceinline__ Plan make_plan(const Args& a) {
  Plan p;
  p.n_work = *a.n_work;
  if (MODE == kModeGateUp) {
    p.mt_per_entry = (a.I + BM - 1) / BM;
    p.tiles = p.n_work * p.mt_per_entry;
    p.kblocks = (a.H + BK - 1) / BK;
    int sp = p.tiles > 0 ? (a.num_sms + p.tiles - 1) / p.tiles : 1;
    sp = min(sp, min(p.kblocks, 8));
    p.splits = max(sp, 1);
  } else {
    p.mt_per_entry = (a.H + BM - 1) / BM;
    p.tiles = p.n_work > 0 ? p.mt_per_entry : 0;
    p.kblocks = (a.I + BK - 1) / BK;
    int sp = p.tiles > 0 ? (a.num_sms + p.tiles - 1) / p.tiles : 1;
    sp = min(sp, min(p.n_work, 16));
    p.splits = max(sp, 1);
  }
  p.units = p.tiles * p.splits;
  return p;
}

// Iterations of one unit: (entry, k-block) pairs in order.
struct UnitRange {
  int tile, split, mt, u0, u1, kb0, kb1;
};

template <int MODE>
__device__ __forceinline__ UnitRange unit_range(const Plan& p, int unit) {
  UnitRange r;
  r.tile = unit / p.splits;
  r.split = unit % p.splits;
  if (MODE == kModeGateUp) {
    r.u0 = r.tile / p.mt_per_entry;
    r.u1 = r.u0 + 1;
    r.mt = r.tile % p.mt_per_entry;
    r.kb0 = r.split * p.kblocks / p.splits;
    r.kb1 = (r.split + 1) * p.kblocks / p.splits;
  } else {
    r.mt = r.tile;
    r.u0 = r.split * p.n_work / p.splits;
    r.u1 = (r.split + 1) * p.n_work / p.splits;
    r.kb0 = 0;
    r.kb1 = p.kblocks;
  }
  return r;
}

__device__ __forceinline__ float silu(float v) { return v / (1.f + expf(-v)); }

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
tc_expert_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b, Args a) {
  constexpr int NACC = MODE == kModeGateUp ? 2 : 1;
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t tfull_bar, tempty_bar, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh, last_sh;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const int S = a.stages;
  const uint32_t a_bytes = BM * BK * 2;                       // 16 KB per A tile
  const uint32_t b_bytes = (uint32_t)N * BK * 2;              // N rows of 128 B
  const uint32_t stage_bytes = ((NACC * a_bytes + b_bytes) + 1023) & ~1023u;
  uint32_t ncols = 32;
  while (ncols < (uint32_t)(NACC * N)) ncols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tfull_bar, 1);
    mbar_init(&tempty_bar, 4);
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, ncols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_sh;

  const Plan pl = make_plan<MODE>(a);
  const uint32_t idesc = idesc_bf16(N);

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < pl.units && ok; unit += gridDim.x) {
        const UnitRange r = unit_range<MODE>(pl, unit);
        for (int u = r.u0; u < r.u1 && ok; ++u) {
          const int rid = a.work[u].rid;
          for (int kb = r.kb0; kb < r.kb1; ++kb, ++it) {
            const int s = it % S;
            if (it >= (uint32_t)S && !mbar_wait(&empty_bar[s], ((it / S) - 1) & 1)) { ok = false; break; }
            if (abort_sh) { ok = false; break; }
            uint8_t* st = smem + (size_t)s * stage_bytes;
            mbar_expect_tx(&full_bar[s], NACC * a_bytes + b_bytes);
            const int k0 = kb * BK;
            if (MODE == kModeGateUp) {
              tma_load_3d(st, &map_a, &full_bar[s], k0, r.mt * BM, rid);
              tma_load_3d(st + a_bytes, &map_a, &full_bar[s], k0, a.I + r.mt * BM, rid);
              tma_load_3d(st + 2 * a_bytes, &map_b, &full_bar[s], k0, 0, 0);
            } else {
              tma_load_3d(st, &map_a, &full_bar[s], k0, r.mt * BM, rid);
              tma_load_3d(st + a_bytes, &map_b, &full_bar[s], k0, 0, u);
            }
          }
        }
      }
      if (!ok) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
      }
      // drain: the last fill of every stage must have landed before the CTA exits
      const uint32_t issued = it;
      for (int s = 0; s < S; ++s) {
        if ((uint32_t)s < issued) {
          const uint32_t last = issued - 1 - ((issued - 1 - s) % S);
          mbar_wait(&full_bar[s], (last / S) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < pl.units && ok; unit += gridDim.x, ++local) {
        const UnitRange r = unit_range<MODE>(pl, unit);
        if (local > 0 && !mbar_wait(&tempty_bar, (local - 1) & 1)) { ok = false; break; }
        fence_after();
        uint32_t acc = 0;
        for (int u = r.u0; u < r.u1 && ok; ++u) {
          for (int kb = r.kb0; kb < r.kb1; ++kb, ++it) {
            const int s = it % S;
            if (!mbar_wait(&full_bar[s], (it / S) & 1) || abort_sh) { ok = false; break; }
            fence_after();
            const uint32_t base = smem_u32(smem + (size_t)s * stage_bytes);
            const uint64_t da = desc_sw128(base);
            const uint64_t db = desc_sw128(base + NACC * a_bytes);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // advance 16 bf16 = 32 bytes along K inside the swizzle atom
              mma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, acc);
              if (MODE == kModeGateUp) mma_bf16(tmem + N, da + (a_bytes >> 4) + 2 * kk, db + 2 * kk, idesc, acc);
              acc = 1;
            }
            mma_commit(&empty_bar[s]);
          }
        }
        if (ok) mma_commit(&tfull_bar);
      }
      if (!ok) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
      }
      // drain: all issued MMAs complete before TMEM is freed
      mma_commit(&drain_bar);
      mbar_wait(&drain_bar, 0);
    }
  } else {
    // ------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;          // tile row == TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16);
    // Every epilogue warp runs the same number of iterations and reaches every
    // named barrier even after a timeout, so no warp can be left waiting.
    int local = 0;
    for (int unit = blockIdx.x; unit < pl.units; unit += gridDim.x, ++local) {
      const UnitRange r = unit_range<MODE>(pl, unit);
      bool live = !abort_sh;
      if (live && !mbar_wait(&tfull_bar, local & 1)) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
        live = false;
      }
      if (live) fence_after();
      const int m = r.mt * BM + row;                           // output row (i for gate_up, h for down)
      const int mlimit = MODE == kModeGateUp ? a.I : a.H;
      if (pl.splits == 1) {
        if (!live) continue;
        for (int c0 = 0; c0 < N; c0 += 16) {
          float d0[16], d1[16];
          tmem_ld16(trow + c0, d0);
          if (MODE == kModeGateUp) tmem_ld16(trow + N + c0, d1);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c0 + j;
            if (m < mlimit) {
              if (MODE == kModeGateUp) {
                const float wgt = t < a.T ? a.wmat[(size_t)r.u0 * N + t] : 0.f;
                const float hv = wgt != 0.f ? wgt * silu(d0[j]) * d1[j] : 0.f;
                a.hbuf[((size_t)r.u0 * N + t) * a.I + m] = f32_to_bf16_rn(hv);
              } else if (t < a.T) {
                a.out[(size_t)t * a.H + m] = f32_to_bf16_rn(d0[j]);
              }
            }
          }
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty_bar);
      } else {
        if (live) {
          // this split's partial tile, [acc][column][row] fp32
          float* mine = a.partial + ((size_t)r.tile * pl.splits + r.split) * NACC * N * BM;
          for (int c0 = 0; c0 < N; c0 += 16) {
            float d0[16], d1[16];
            tmem_ld16(trow + c0, d0);
            if (MODE == kModeGateUp) tmem_ld16(trow + N + c0, d1);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              mine[(size_t)(c0 + j) * BM + row] = d0[j];
              if (MODE == kModeGateUp) mine[(size_t)N * BM + (size_t)(c0 + j) * BM + row] = d1[j];
            }
          }
          fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty_bar);
          __threadfence();
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == 2 && lane == 0) {
          last_sh = 0;
          if (!abort_sh) {
            const int old = atomicAdd(&a.counters[r.tile], 1);
            if (old == pl.splits - 1) {
              last_sh = 1;
              a.counters[r.tile] = 0;
            }
          }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (last_sh && live) {
          __threadfence();
          const float* base = a.partial + (size_t)r.tile * pl.splits * NACC * N * BM;
          for (int t = 0; t < N; ++t) {
            float s0 = 0.f, s1 = 0.f;
            for (int sp = 0; sp < pl.splits; ++sp) {       // fixed order: deterministic
              const float* pt = base + (size_t)sp * NACC * N * BM;
              s0 += __ldcg(pt + (size_t)t * BM + row);
              if (MODE == kModeGateUp) s1 += __ldcg(pt + (size_t)N * BM + (size_t)t * BM + row);
            }
            if (m < mlimit) {
              if (MODE == kModeGateUp) {
                const float wgt = t < a.T ? a.wmat[(size_t)r.u0 * N + t] : 0.f;
                const float hv = wgt != 0.f ? wgt * silu(s0) * s1 : 0.f;
                a.hbuf[((size_t)r.u0 * N + t) * a.I + m] = f32_to_bf16_rn(hv);
              } else if (t < a.T) {
                a.out[(size_t)t * a.H + m] = f32_to_bf16_rn(s0);
              }
            }
          }
        }
        asm volatile("bar.sync 1, 128;" ::: "memory");
      }
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) tmem_dealloc(tmem, ncols);
}

// ----------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// bf16 tensor [d2][d1][d0] (d0 contiguous), byte strides s1 (d1), s2 (d2); box BK x rows x 1, 128B swizzle.
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
                 uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {(cuuint32_t)BK, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
void configure_once() {
  static bool done = false;
  if (!done) {
    cudaFuncSetAttribute(tc_expert_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget + 1024);
    done = true;
  }
}

int stages_for(int nacc, int N) {
  const int stage = ((nacc * BM * BK * 2 + N * BK * 2) + 1023) & ~1023;
  int s = kSmemBudget / stage;
  if (s > kMaxStages) s = kMaxStages;
  return s;
}

}  // namespace tc

TcMaps* tc_maps_create(const PoolDev& p, const Scratch& sc) {
  (void)sc;
  TcMaps* m = new TcMaps();
  const uint64_t H = p.H, I = p.I, R = p.n_records, rec = p.lay.rec;
  bool ok = tc::make_map_3d(&m->w13, p.records + p.lay.off13, H, 2 * I, R, H * 2, rec, tc::BM) &&
            tc::make_map_3d(&m->w2, p.records + p.lay.off2, I, H, R, I * 2, rec, tc::BM);
  if (!ok) {
    delete m;
    return nullptr;
  }
  return m;
}

void tc_maps_destroy(TcMaps* m) { delete m; }

int tc_npad(int T) { return (T + 15) / 16 * 16; }

static tc::Args tc_args(const PoolDev& p, const Scratch& sc, int T) {
  tc::Args a;
  a.work = sc.work;
  a.n_work = sc.n_work;
  a.T = T;
  a.N = tc_npad(T);
  a.H = p.H;
  a.I = p.I;
  a.num_sms = sm_count();
  a.wmat = sc.wmat;
  a.hbuf = sc.hbuf;
  a.out = nullptr;
  a.partial = sc.partial;
  a.counters = sc.counters;
  a.status = p.status;
  return a;
}

int launch_tc_gate_up(const PoolDev& p, const Scratch& sc, const TcMaps* m, int T, const void* x, cudaStream_t s) {
  tc::Args a = tc_args(p, sc, T);
  a.stages = tc::stages_for(2, a.N);
  CUtensorMap xm;   // x [T][H] as a 3-D map with one "record"
  if (!tc::make_map_3d(&xm, x, (uint64_t)p.H, (uint64_t)T, 1, (uint64_t)p.H * 2, (uint64_t)p.H * 2 * T, a.N)) {
    return -1;
  }
  tc::configure_once<tc::kModeGateUp>();
  const size_t smem = (size_t)a.stages * (((2 * tc::BM * tc::BK * 2 + a.N * tc::BK * 2) + 1023) & ~1023) + 1024;
  tc::tc_expert_kernel<tc::kModeGateUp><<<sm_count(), tc::kThreads, smem, s>>>(m->w13, xm, a);
  return 1;
}

int launch_tc_down(const PoolDev& p, const Scratch& sc, const TcMaps* m, int T, void* out, cudaStream_t s) {
  tc::Args a = tc_args(p, sc, T);
  a.out = static_cast<uint16_t*>(out);
  a.stages = tc::stages_for(1, a.N);
  CUtensorMap hm;   // hbuf [E+1][N][I]
  const uint64_t I = p.I, N = a.N;
  if (!tc::make_map_3d(&hm, sc.hbuf, I, N, (uint64_t)p.E + 1, I * 2, N * I * 2, a.N)) return -1;
  tc::configure_once<tc::kModeDown>();
  const size_t smem = (size_t)a.stages * (((tc::BM * tc::BK * 2 + a.N * tc::BK * 2) + 1023) & ~1023) + 1024;
  tc::tc_expert_kernel<tc::kModeDown><<<sm_count(), tc::kThreads, smem, s>>>(m->w2, hm, a);
  return 1;
}

}  // namespace moeslot
