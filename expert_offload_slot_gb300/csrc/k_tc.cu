// Step a8 (SwiGLU experts) and a9 (combine) on the 5th-generation tensor cores
// (tcgen05, accumulators in TMEM, operands staged in shared memory by the
// Tensor Memory Accelerator).
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
// Weights: a bf16 expert record is stored as 128-row x 64-column tiles
// already in the 128-byte-swizzled order the MMA descriptor reads (w13 as
// [I/128][H/64][gate, up], w2 as [H/128][I/64]), so every pipeline stage is
// ONE contiguous bulk copy (32 KB gate+up, or 16 KB down) that streams from
// HBM at full burst length.  Activations (x, h) come through TMA tensor maps.
//
// Large token counts (T > 256) use the gather modes: tokens are grouped by
// expert (x rows gathered once), each (entry, token tile of 64, 128 or 256 rows,
// 128-row tile) is a unit, gate/up writes w * SiLU(g) * u per expert row, down writes one bf16
// row per (token, expert) and a combine kernel sums each token's k rows in
// ascending expert order (plus the shared expert).
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
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <cstring>

#include "gate_body.cuh"
#include "moeslot_internal.cuh"
#include "plan_body.cuh"

namespace moeslot {

struct TcMaps {
  // bf16 weights need no tensor map (tiled records, bulk copies); fp8 weights are
  // read as 128-row x 64-byte tiles of the record array: w13 [n_records][2I][H]
  // and w2 [n_records][H][I] (row-major codes)
  bool fp8 = false;
  CUtensorMap w13{}, w2{};
  // bf16 pools, streaming decode path: 16-row segments of the tiled records, as
  // [n_records][mt][tile (kb, gate/up)][row][128 B] and [n_records][mt][kb][row][128 B]
  bool stream = false;
  CUtensorMap sw13{}, sw2{};
};

namespace tc {

constexpr int BM = 128;          // weight rows per tile (MMA M)
constexpr int BK = 64;           // K elements per stage (one 128-byte swizzle row)
constexpr int kThreads = 192;
constexpr int kMaxStages = 8;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kModeGateUp = 0, kModeDown = 1, kModeGateUpGather = 2, kModeDownGather = 3;
constexpr uint32_t kTileBytes = BM * BK * 2;   // one 128 x 64 bf16 tile

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

// Tiled tensor loads of 4 and 5 dimensions (coordinates innermost first); the
// 5-dimensional one carries the weights' evict-first L2 policy.
__device__ __forceinline__ uint64_t l2_evict_first_policy();
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], "
      "[%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d_ef(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                               int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, "
      "%4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "l"(l2_evict_first_policy())
      : "memory");
}

// Contiguous global -> shared copy by the bulk-copy engine, completing on `bar`.
// Expert weights are read once per layer step, so they are marked evict-first
// in L2: the stream then does not push out the small state every layer
// re-reads (tables, history, activations, the code of the other kernels).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(l2_evict_first_policy())
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
  const int32_t* sel;        // gate_up dense: the entries to process (indices into work), or null for all
  const int32_t* sel_count;
  const int32_t* ntile0;     // gather modes: first token tile of each entry ([E+2], prefix)
  const uint8_t* records;    // record array base
  size_t rec, off13, off2;   // record bytes, w13 / w2 tile offsets
  int T, N, H, I, num_sms, stages;
  int max_split_units;       // capacity of `partial` in (tile, split) units of this call's size
  const float* wmat;         // dense: [E+1][N] routing weight per (entry, token)
  const float* perm_w;       // gather: routing weight of each expert-sorted row
  uint16_t* hbuf;            // dense: [E+1][N][I]; gather: h rows [rows][I]
  uint16_t* out;             // dense down: [T][H]; gather down: Y rows [rows][H]
  float* partial;
  int32_t* counters;
  int32_t* status;
  uint64_t wait_ns;          // limit of every wait on another CTA (global-timer ns)
};

__host__ __device__ constexpr bool is_gate_up(int mode) { return mode == kModeGateUp || mode == kModeGateUpGather; }
__host__ __device__ constexpr bool is_gather(int mode) { return mode >= kModeGateUpGather; }

struct Plan {             // the unit decomposition, identical in every role
  int tiles, splits, units, kblocks, mt_per_entry, n_work, n_sel, n_ntiles;
};

// Split count that keeps the most SMs busy: units = tiles * s spread over
// the grid, utilisation (units / grid) / ceil(units / grid); ties to fewer splits.
__device__ __forceinline__ int best_splits(int tiles, int smax, int grid, int cap) {
  if (tiles <= 0) return 1;
  int best = 1;
  float best_eff = 0.f;
  for (int sp = 1; sp <= smax; ++sp) {
    const int units = tiles * sp;
    if (sp > 1 && units > cap) break;          // the partial buffer holds at most `cap` units
    const int rounds = (units + grid - 1) / grid;
    const float eff = (float)units / (float)(rounds * grid);
    if (eff > best_eff + 1e-6f) { best_eff = eff; best = sp; }
  }
  return best;
}

template <int MODE>
__device__ __forceinline__ Plan make_plan(const Args& a, int grid) {
  Plan p;
  p.n_work = *a.n_work;
  p.n_ntiles = 0;
  if (MODE == kModeGateUp) {
    p.n_sel = a.sel ? *a.sel_count : p.n_work;
    p.mt_per_entry = (a.I + BM - 1) / BM;
    p.tiles = p.n_sel * p.mt_per_entry;
    p.kblocks = (a.H + BK - 1) / BK;
    p.splits = best_splits(p.tiles, min(p.kblocks, 8), grid, a.max_split_units);
  } else if (MODE == kModeDown) {
    p.n_sel = p.n_work;
    p.mt_per_entry = (a.H + BM - 1) / BM;
    p.tiles = p.n_work > 0 ? p.mt_per_entry : 0;
    p.kblocks = (a.I + BK - 1) / BK;
    p.splits = best_splits(p.tiles, min(max(p.n_work, 1), 16), grid, a.max_split_units);
  } else {
    p.n_sel = p.n_work;
    p.n_ntiles = a.ntile0[p.n_work];
    p.mt_per_entry = MODE == kModeGateUpGather ? (a.I + BM - 1) / BM : (a.H + BM - 1) / BM;
    p.kblocks = MODE == kModeGateUpGather ? (a.H + BK - 1) / BK : (a.I + BK - 1) / BK;
    p.tiles = p.n_ntiles * p.mt_per_entry;
    p.splits = 1;
  }
  p.units = p.tiles * p.splits;
  return p;
}

// One unit: rows mt of entry range [u0, u1), K blocks [kb0, kb1), token tile nt (gather).
struct UnitRange {
  int tile, split, mt, u0, u1, kb0, kb1, nt;
};

template <int MODE>
__device__ __forceinline__ UnitRange unit_range(const Plan& p, const Args& a, int unit) {
  UnitRange r;
  r.tile = unit / p.splits;
  r.split = unit % p.splits;
  r.nt = 0;
  if (MODE == kModeGateUp) {
    const int si = r.tile / p.mt_per_entry;
    r.u0 = a.sel ? a.sel[si] : si;
    r.u1 = r.u0 + 1;
    r.mt = r.tile % p.mt_per_entry;
    r.kb0 = r.split * p.kblocks / p.splits;
    r.kb1 = (r.split + 1) * p.kblocks / p.splits;
  } else if (MODE == kModeDown) {
    r.mt = r.tile;
    r.u0 = r.split * p.n_work / p.splits;
    r.u1 = (r.split + 1) * p.n_work / p.splits;
    r.kb0 = 0;
    r.kb1 = p.kblocks;
  } else {
    // unit = ntile0[u] * MT + mt * nts(u) + nt: entries' units are consecutive
    const int MT = p.mt_per_entry;
    int lo = 0, hi = p.n_work - 1;
    while (lo < hi) {                      // last u with ntile0[u] * MT <= unit
      const int mid = (lo + hi + 1) >> 1;
      if (a.ntile0[mid] * MT <= unit) lo = mid;
      else hi = mid - 1;
    }
    const int nts = a.ntile0[lo + 1] - a.ntile0[lo];
    const int local = unit - a.ntile0[lo] * MT;
    r.u0 = lo;
    r.u1 = lo + 1;
    r.mt = local / nts;
    r.nt = local % nts;
    r.kb0 = 0;
    r.kb1 = p.kblocks;
  }
  return r;
}

__device__ __forceinline__ float silu(float v) { return v / (1.f + expf(-v)); }

// Four fp8 e4m3 codes (little-endian in w) as floats; the decode is exact.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* v) {
  const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
  const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}

// Two floats rounded to bf16 (nearest, ties to even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Epilogue store of one 16-column chunk.  Gate/up: d0 = W_gate x, d1 = W_up x;
// down: d0 = D.  Column j is token c0+j (dense) or row row_base+c0+j (gather).
template <int MODE>
__device__ __forceinline__ void store_chunk(const Args& a, const UnitRange& r, int m, int c0, const float* d0,
                                            const float* d1, int row_base, int row_end) {
  const int N = a.N;
  if (MODE == kModeGateUp) {
    if (m >= a.I) return;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int t = c0 + j;
      const float wgt = t < a.T ? a.wmat[(size_t)r.u0 * N + t] : 0.f;
      const float hv = wgt != 0.f ? wgt * silu(d0[j]) * d1[j] : 0.f;
      a.hbuf[((size_t)r.u0 * N + t) * a.I + m] = f32_to_bf16_rn(hv);
    }
  } else if (MODE == kModeDown) {
    if (m >= a.H) return;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (c0 + j < a.T) a.out[(size_t)(c0 + j) * a.H + m] = f32_to_bf16_rn(d0[j]);
  } else if (MODE == kModeGateUpGather) {
    if (m >= a.I) return;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int row = row_base + c0 + j;
      if (row < row_end) a.hbuf[(size_t)row * a.I + m] = f32_to_bf16_rn(a.perm_w[row] * silu(d0[j]) * d1[j]);
    }
  } else {
    if (m >= a.H) return;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int row = row_base + c0 + j;
      if (row < row_end) a.out[(size_t)row * a.H + m] = f32_to_bf16_rn(d0[j]);
    }
  }
}

// Weight formats: bf16 records pre-tiled in the MMA's swizzled order (bulk
// copies), or fp8 e4m3 row-major records with one fp32 scale per 128 x 128
// block (TMA tiles of codes, expanded to bf16 in place by converter warps, the
// block scale applied in the expansion).
constexpr int kWfBf16 = 0, kWfFp8 = 1;
constexpr int kConvWarps = 4;         // fused decode kernels
constexpr int kGatherConvWarps = 8;   // prefill gather kernel

// NCT converter threads (ct = 0..NCT-1): expand the fp8 code tiles q < nt of one
// stage in place.  Each tile slot is 16 KB; its codes (128 rows x 64 bytes = 512
// chunks of 16 bytes) sit in the upper 8 KB.  Every thread reads its 512 / NCT
// chunks of each tile, then (after the named barrier, all reads done) writes them
// back as bf16 (code * scale, one rounding) in the 128-byte-swizzled order.  Every
// converter thread calls this for every stage, work or not, so the named barrier
// is always complete.
template <int NCT, int BAR = 3>
__device__ __forceinline__ void fp8_expand_stage(uint8_t* st, int nt, float s0, float s1, int ct, bool work) {
  constexpr int MPER = 512 / NCT;
  uint4 raw[2][MPER];
  if (work) {
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (q < nt) {
#pragma unroll
        for (int m = 0; m < MPER; ++m)
          raw[q][m] = *reinterpret_cast<const uint4*>(st + q * kTileBytes + kTileBytes / 2 + (ct + NCT * m) * 16);
      }
  }
  asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NCT) : "memory");
  if (!work) return;
#pragma unroll
  for (int q = 0; q < 2; ++q)
    if (q < nt) {
      const float sv = q ? s1 : s0;
#pragma unroll
      for (int m = 0; m < MPER; ++m) {
        const int c16 = ct + NCT * m, row = c16 >> 2, cq = c16 & 3;   // 16 codes: columns cq*16..+16
        const uint32_t w4[4] = {raw[q][m].x, raw[q][m].y, raw[q][m].z, raw[q][m].w};
        uint32_t o[8];
#pragma unroll
        for (int wq = 0; wq < 4; ++wq) {
          float v[4];
          e4m3x4_to_f32(w4[wq], v);
          o[2 * wq] = pack_bf16x2(v[0] * sv, v[1] * sv);
          o[2 * wq + 1] = pack_bf16x2(v[2] * sv, v[3] * sv);
        }
        uint8_t* rowp = st + q * kTileBytes + row * 128;
        const int c0 = 2 * cq;
        *reinterpret_cast<uint4*>(rowp + ((c0 ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(rowp + (((c0 + 1) ^ (row & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // generic writes -> MMA reads
}

// fp8 record geometry for the converters: scale tables at os13 ([2I/128][H/128]
// fp32) and os2 ([H/128][I/128]).
struct Fp8Args {
  size_t os13, os2;
  int sc_h, sc_i;               // H / 128, I / 128
};

template <int WF> struct GatherShape {
  static constexpr int threads = kThreads + (WF == kWfFp8 ? 32 * kGatherConvWarps : 0);
};

// Gather modes (T > 256 tokens): unit = (entry u, token tile nt of N = 64, 128 or 256
// rows, 128-row tile mt), full K (the plan's ntile0 counts tiles of the same N).  Gate/up: A = gate and up tiles of the entry, B = its gathered x
// rows; epilogue h = w * SiLU(g) * u per row.  Down: A = W_down tile, B = its h
// rows; epilogue one bf16 row of y per (token, expert).
template <int MODE, int WF>
__global__ void __launch_bounds__(GatherShape<WF>::threads, 1)
tc_gather_kernel(const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_w, Args a,
                 Fp8Args w8) {
  constexpr int NACC = is_gate_up(MODE) ? 2 : 1;
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t conv_bar[WF == kWfFp8 ? kMaxStages : 1];
  __shared__ __align__(8) uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
  __shared__ float scale_sh[WF == kWfFp8 ? 2 : 1][WF == kWfFp8 ? 128 : 1];
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const int S = a.stages;
  const uint32_t a_bytes = NACC * kTileBytes;                 // 16 KB (down) or 32 KB (gate + up)
  const uint32_t b_bytes = (uint32_t)N * BK * 2;              // N rows of 128 B
  const uint32_t stage_bytes = (a_bytes + b_bytes + 1023) & ~1023u;
  const int nbuf = 2 * NACC * N <= 512 ? 2 : 1;
  const uint32_t acc_cols = (uint32_t)(NACC * N);
  uint32_t ncols = 32;
  while (ncols < (uint32_t)nbuf * acc_cols) ncols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      if (WF == kWfFp8) mbar_init(&conv_bar[s], 32 * kGatherConvWarps / 2);   // one group per stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 4);
    }
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, ncols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_sh;

  const Plan pl = make_plan<MODE>(a, gridDim.x);
  const uint32_t idesc = idesc_bf16(N);
  const int kb_per_row = is_gate_up(MODE) ? (a.H + BK - 1) / BK : (a.I + BK - 1) / BK;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < pl.units && ok; unit += gridDim.x) {
        const UnitRange r = unit_range<MODE>(pl, a, unit);
        const WorkEntry we = a.work[r.u0];
        const uint8_t* wbase = a.records + (size_t)we.rid * a.rec + (is_gate_up(MODE) ? a.off13 : a.off2) +
                               (size_t)r.mt * kb_per_row * a_bytes;
        const int brow = we.row0 + r.nt * N;
        for (int kb = r.kb0; kb < r.kb1; ++kb, ++it) {
          const int s = it % S;
          if (it >= (uint32_t)S && !mbar_wait(&empty_bar[s], ((it / S) - 1) & 1)) { ok = false; break; }
          if (abort_sh) { ok = false; break; }
          uint8_t* st = smem + (size_t)s * stage_bytes;
          if (WF == kWfFp8) {
            const uint32_t raw = kTileBytes / 2;
            mbar_expect_tx(&full_bar[s], NACC * raw + b_bytes);
            if (is_gate_up(MODE)) {
              tma_load_3d(st + raw, &map_w, &full_bar[s], kb * BK, r.mt * BM, we.rid);
              tma_load_3d(st + kTileBytes + raw, &map_w, &full_bar[s], kb * BK, a.I + r.mt * BM, we.rid);
            } else {
              tma_load_3d(st + raw, &map_w, &full_bar[s], kb * BK, r.mt * BM, we.rid);
            }
          } else {
            mbar_expect_tx(&full_bar[s], a_bytes + b_bytes);
            bulk_load(st, wbase + (size_t)kb * a_bytes, a_bytes, &full_bar[s]);
          }
          tma_load_3d(st + a_bytes, &map_b, &full_bar[s], kb * BK, brow, 0);
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
        const UnitRange r = unit_range<MODE>(pl, a, unit);
        const int buf = local % nbuf, use = local / nbuf;
        if (use > 0 && !mbar_wait(&tempty_bar[buf], (use - 1) & 1)) { ok = false; break; }
        fence_after();
        const uint32_t dacc = tmem + (uint32_t)buf * acc_cols;
        uint32_t acc = 0;
        for (int kb = r.kb0; kb < r.kb1; ++kb, ++it) {
          const int s = it % S;
          if (!mbar_wait(WF == kWfFp8 ? &conv_bar[s] : &full_bar[s], (it / S) & 1) || abort_sh) { ok = false; break; }
          fence_after();
          const uint32_t base = smem_u32(smem + (size_t)s * stage_bytes);
          const uint64_t da = desc_sw128(base);
          const uint64_t db = desc_sw128(base + a_bytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // advance 16 bf16 = 32 bytes along K inside the swizzle atom
            mma_bf16(dacc, da + 2 * kk, db + 2 * kk, idesc, acc);
            if (NACC == 2) mma_bf16(dacc + N, da + (kTileBytes >> 4) + 2 * kk, db + 2 * kk, idesc, acc);
            acc = 1;
          }
          mma_commit(&empty_bar[s]);
        }
        if (ok) mma_commit(&tfull_bar[buf]);
      }
      if (!ok) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
      }
      // drain: all issued MMAs complete before TMEM is freed
      mma_commit(&drain_bar);
      mbar_wait(&drain_bar, 0);
    }
  } else if (warp < kThreads / 32) {
    // ------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;          // tile row == TMEM lane
    const uint32_t trow0 = tmem + ((uint32_t)(q * 32) << 16);
    int local = 0;
    for (int unit = blockIdx.x; unit < pl.units; unit += gridDim.x, ++local) {
      const UnitRange r = unit_range<MODE>(pl, a, unit);
      const int buf = local % nbuf;
      const uint32_t trow = trow0 + (uint32_t)buf * acc_cols;
      if (abort_sh) continue;
      if (!mbar_wait(&tfull_bar[buf], (local / nbuf) & 1)) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
        continue;
      }
      fence_after();
      const int m = r.mt * BM + row;                           // output row (i for gate/up, h for down)
      const WorkEntry we = a.work[r.u0];
      const int row_base = we.row0 + r.nt * N, row_end = we.row0 + we.n;
      for (int c0 = 0; c0 < N; c0 += 16) {
        float d0[16], d1[16];
        tmem_ld16(trow + c0, d0);
        if (NACC == 2) tmem_ld16(trow + N + c0, d1);
        store_chunk<MODE>(a, r, m, c0, d0, d1, row_base, row_end);
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[buf]);
    }
  } else if (WF == kWfFp8) {
    // ------------------------------------------------------------- converter warps (fp8)
    const int ct = threadIdx.x - kThreads;        // 0 .. 32 * kGatherConvWarps - 1
    const int grp = ct >= 16 * kGatherConvWarps ? 1 : 0, gct = ct - grp * 16 * kGatherConvWarps;
    uint32_t it = 0;
    int local = 0;
    bool stop = false;
    for (int unit = blockIdx.x; unit < pl.units; unit += gridDim.x, ++local) {
      const UnitRange r = unit_range<MODE>(pl, a, unit);
      const WorkEntry we = a.work[r.u0];
      const float* scl =
          reinterpret_cast<const float*>(a.records + (size_t)we.rid * a.rec + (is_gate_up(MODE) ? w8.os13 : w8.os2));
      const int b0 = r.kb0 / 2, nblk = (r.kb1 - 1) / 2 - b0 + 1;
      const int sbuf = local & 1;
      if (ct < nblk) {
        scale_sh[sbuf][ct] = scl[(size_t)(is_gate_up(MODE) ? r.mt * w8.sc_h : r.mt * w8.sc_i) + b0 + ct];
      } else if (is_gate_up(MODE) && ct >= 64 && ct - 64 < nblk) {
        scale_sh[sbuf][ct] = scl[(size_t)(a.I / BM + r.mt) * w8.sc_h + b0 + (ct - 64)];
      }
      asm volatile("bar.sync 3, %0;" ::"n"(32 * kGatherConvWarps) : "memory");
      for (int kb = r.kb0; kb < r.kb1; ++kb, ++it) {
        // two groups of converter warps take alternate stages, so that two expansions are in
        // flight (each group's own named barrier orders its in-place reads before its writes)
        if ((int)(it & 1u) != grp) continue;
        const int s = it % S;
        if (!stop && (!mbar_wait(&full_bar[s], (it / S) & 1) || abort_sh)) {
          stop = true;
          set_status(a.status, MOE_ERR_TIMEOUT);
          abort_sh = 1;
        }
        const float s0 = scale_sh[sbuf][kb / 2 - b0];
        const float s1 = is_gate_up(MODE) ? scale_sh[sbuf][64 + kb / 2 - b0] : 0.f;
        if (grp == 0)
          fp8_expand_stage<16 * kGatherConvWarps, 4>(smem + (size_t)s * stage_bytes, NACC, s0, s1, gct, !stop);
        else
          fp8_expand_stage<16 * kGatherConvWarps, 5>(smem + (size_t)s * stage_bytes, NACC, s0, s1, gct, !stop);
        if (!stop) mbar_arrive(&conv_bar[s]);
      }
      asm volatile("bar.sync 3, %0;" ::"n"(32 * kGatherConvWarps) : "memory");   // before the scale buffer is reused
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) tmem_dealloc(tmem, ncols);
}

// ----------------------------------------------------------------- fused decode FFN
// One persistent kernel per layer for the dense token path (cooperative launch:
// every CTA is resident, so CTAs may wait on each other with bounded spins).
// Work units in one global order, which CTA c walks as c, c+G, c+2G, ...:
//   1. gate/up tiles of the entries already resident,
//   2. down tiles of those entries,
//   3. gate/up tiles of the entries copied this step (in copy-job order),
//   4. down tiles of those entries;
// meanwhile this step's misses are pulled from the mapped host pool (NVLink-C2C
// reads) into their records, one job after another: by kCopyCtas copy-only CTAs
// with all their threads in the decode layer kernel, else by two copy warps in
// every CTA.  A unit waits only for what it reads: the part of a copied record
// it reads (jdone[job] for the gate/up tiles, jdone_w2[job] for the rest: every
// copying CTA has released its slice), or the complete h of its entry
// (hready[u] == the entry's gate/up tiles).  So the resident experts' whole FFN
// overlaps the link-bound copies.
// A down unit covers one entry and writes an fp32 partial tile; once every
// CTA's partials are written, all CTAs sum them element-parallel in entry order
// (ascending expert id, shared expert last).  The order is fixed, and the split
// counts depend on the entry count alone, so the output does not depend on
// which experts happened to be resident.
// Partial tiles are row-major ([128 rows][columns]) so that each epilogue
// thread (one row) moves its columns with 16-byte accesses.
constexpr int kCopyWarps = 2;
constexpr int kCopyCtas = 32;   // CTAs that copy first in a decode layer call with misses (local lists)
constexpr int kUnitQ = 32;      // a CTA's queue of units handed out (it is at most stages + TMEM buffers ahead)
constexpr int kCopyUnroll = 8;   // 16-byte host reads in flight per copy lane
constexpr int kFusedBufs = 8;
template <int WF> struct FusedShape {
  static constexpr int conv_warps = WF == kWfFp8 ? kConvWarps : 0;
  static constexpr int conv_warp0 = kThreads / 32;               // after the epilogue warps
  static constexpr int copy_warp0 = conv_warp0 + conv_warps;
  static constexpr int threads = (copy_warp0 + kCopyWarps) * 32;
};

// A step's entry lists derived by every CTA itself from the gated routing and
// a snapshot of the layer's table row taken before the plan may change it
// (decode layer kernel): same positions and order as the plan's work list.
constexpr int kLocalMaxTk = 256;   // routing entries (T * k) the local lists take
struct LocalPlan {
  int n, nh, nm, tk, k;
  int elist[2][kMaxE + 1];         // resident entries, entries copied this step (work positions)
  int expert[kMaxE + 1];           // expert of each work position (-1: the shared expert)
  int rid[kMaxE + 1];              // record of each resident entry
  int32_t ids[kLocalMaxTk];        // the step's routing
  float w[kLocalMaxTk];
  int16_t epos[kMaxE];             // work position of each expert with tokens
};

struct FusedArgs {
  const LocalPlan* lp;          // null: the plan's work lists in global memory
  int cta0_plans;               // CTA 0 runs the plan first (copying CTAs are counted after it)
  // with lp: a miss j (j-th copied entry) is copied from the host pool into landing
  // record rid_land0 + j at once, read from there, and written to its slot once the
  // plan has chosen it (slots_ready: the table holds this step's slots)
  const uint32_t* slots_ready;
  const uint8_t* host_layer;    // host pool records of this layer (device view)
  const int32_t* lut_row;       // this layer's table row
  int rid_land0, S;
  const CopyJob* jobs;
  const int32_t* n_jobs;
  uint32_t tile16;              // bytes of a record the miss copy moves, in 16 B units
  uint32_t part16;              // its first part, all that gate/up units read (bf16: the W_gate/W_up
                                // tiles; fp8: the whole record), in 16 B units
  // fp8 records: scale tables at os13 ([2I/128][H/128] fp32) and os2 ([H/128][I/128])
  size_t os13, os2;
  int sc_h, sc_i;               // scale row lengths: H / 128 and I / 128
  const int32_t* elist;         // [2][E1]: resident entries, copied entries (work positions, ascending)
  const int32_t* ecount;        // [2]
  int E1;                       // E + 1
  float* gu_partial;            // gate/up split partials
  int gu_cap;                   // (tile, split) partials gu_partial holds at this call's token count
  float* dn_partial;            // per-entry down partials
  int dn_cap;                   // (tile, split) partials dn_partial holds at this call's token count
  int32_t* gu_cnt;              // [E1 * MT_I] split arrivals per gate/up tile    } zeroed by the plan
  uint32_t* dn_done;            // CTAs whose down units are all written           } kernel before
  uint32_t* hready;             // [E1] finished gate/up tiles per entry           } every launch
  uint32_t* jdone;              // [E1] CTAs done with each copy job's first part  }
  uint32_t* jdone_w2;           // [E1] ... and with the whole record              }
  uint32_t* next_unit;          // the next resident entries' unit to hand out     }
  uint32_t* next_miss;          // the next copied entries' unit to hand out       }
};

struct FSched {
  int n, nh, nm, mt_i, kb_h, mt_h, kb_i, sg, sd, cols;
  int p0, p1, p2, p3, total;
};

__device__ __forceinline__ FSched fused_sched(const Args& a, const FusedArgs& f, int G) {
  FSched s;
  if (f.lp) {
    s.n = f.lp->n;
    s.nh = f.lp->nh;
    s.nm = f.lp->nm;
  } else {
    s.n = *a.n_work;
    s.nh = f.ecount[0];
    s.nm = f.ecount[1];
  }
  G -= f.cta0_plans;
  s.mt_i = (a.I + BM - 1) / BM;
  s.kb_h = (a.H + BK - 1) / BK;
  s.mt_h = (a.H + BM - 1) / BM;
  s.kb_i = (a.I + BK - 1) / BK;
  s.cols = (a.T + 3) & ~3;            // partial columns kept: the tokens, rounded up to 4
  // Splits: the fewest that give every CTA about two gate/up units and one down
  // unit (all units of a step share one round-robin schedule, so per-phase wave
  // quantisation matters little, while every unit costs a partial round trip).
  const int gu_tiles = s.n * s.mt_i;
  const int gcap = f.gu_cap;
  s.sg = max(1, min(min(s.kb_h, 8), (2 * G + gu_tiles - 1) / max(gu_tiles, 1)));
  while (s.sg > 1 && gu_tiles * s.sg > gcap) --s.sg;
  const int dn_tiles = s.n * s.mt_h;
  const int dcap = f.dn_cap;
  s.sd = max(1, min(min(s.kb_i, 4), (G + dn_tiles - 1) / max(dn_tiles, 1)));
  while (s.sd > 1 && dn_tiles * s.sd > dcap) --s.sd;
  s.p0 = s.nh * s.mt_i * s.sg;
  s.p1 = s.nh * s.mt_h * s.sd;
  s.p2 = s.nm * s.mt_i * s.sg;
  s.p3 = s.nm * s.mt_h * s.sd;
  s.total = s.p0 + s.p1 + s.p2 + s.p3;
  return s;
}

struct FUnit {
  int gu, miss, li, u, mt, sp, kb0, kb1;
};

__device__ __forceinline__ FUnit fused_unit(const FSched& s, const FusedArgs& f, int g) {
  FUnit r;
  int loc = g, rem;
  if (loc < s.p0 + s.p1) {
    // resident entries: all gate/up units, then all down units, each entry-major (an
    // entry's h completes early, and its down units come soon after)
    r.miss = 0;
    r.gu = loc < s.p0;
    if (!r.gu) loc -= s.p0;
    const int per = r.gu ? s.mt_i * s.sg : s.mt_h * s.sd;
    r.li = loc / per;
    rem = loc - r.li * per;
  } else {
    // copied entries, job by job: its gate/up units, then its down units (the order in
    // which the two parts of its record land)
    loc -= s.p0 + s.p1;
    const int gu_per = s.mt_i * s.sg, job_per = gu_per + s.mt_h * s.sd;
    r.miss = 1;
    r.li = loc / job_per;
    rem = loc - r.li * job_per;
    r.gu = rem < gu_per;
    if (!r.gu) rem -= gu_per;
  }
  const int spn = r.gu ? s.sg : s.sd, kbn = r.gu ? s.kb_h : s.kb_i;
  r.mt = rem / spn;
  r.sp = rem - r.mt * spn;
  r.kb0 = r.sp * kbn / spn;
  r.kb1 = (r.sp + 1) * kbn / spn;
  r.u = f.lp ? f.lp->elist[r.miss][r.li] : f.elist[r.miss * f.E1 + r.li];
  return r;
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Release this thread's prior writes (and, after a CTA barrier, the CTA's) and add 1.
__device__ __forceinline__ void release_add(uint32_t* p) {
  asm volatile("fence.acq_rel.gpu;\n red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p) : "memory");
}

// Wait until *p >= target, for at most limit_ns of global time (1 s unless the
// pool's wait limit was changed); gives up at once if another CTA has already
// recorded an error, so one failure cannot chain into many timeouts.
__device__ __noinline__ bool wait_count(const uint32_t* p, uint32_t target, const int32_t* status, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire(p) >= target) return true;
    if ((it & 15u) == 15u) {
      if (*reinterpret_cast<const volatile int32_t*>(status) != 0) return false;
      if (global_ns() - t0 > limit_ns) return false;
    }
    __nanosleep(64);
  }
}

// Record copies, job by job and part by part (first the gate/up part, which releases
// jdone[j], then the rest, which releases jdone_w2[j]; both count the copying CTAs):
// nthr threads of each of ncta CTAs copy; thread tid of copying CTA cidx takes the
// 16-byte chunks wb + lane + u * stride (u < kCopyUnroll) of the lattice rows
// wb = w0 + i * kCopyUnroll * stride, w0 = its warp's first chunk, that fall in the
// part.  The loops run on wb, so all lanes of a warp take the same trip count (the
// warp-wide shuffles below need that).
__device__ __noinline__ void copy_records(const Args& a, const FusedArgs& f, uint32_t nthr, uint32_t tid,
                                        uint32_t cidx, uint32_t ncta) {
  const int lane = threadIdx.x & 31;
  const uint32_t stride = ncta * nthr;
  const uint32_t step = stride * kCopyUnroll;
  const uint32_t w0 = cidx * nthr + (tid & ~31u);
  auto first_row = [&](uint32_t lo) { return lo <= w0 ? w0 : w0 + (lo - w0) / step * step; };
  // slot record the plan gave expert e (null: none, the miss stays in its landing record)
  auto slot_record = [&](int e) -> uint4* {
    int slot = -1;
    if (lane == 0) slot = __ldcg(f.lut_row + e);
    slot = __shfl_sync(0xffffffffu, slot, 0);
    return slot >= 0 && slot < f.S ? reinterpret_cast<uint4*>(const_cast<uint8_t*>(a.records) + (size_t)slot * a.rec)
                                   : nullptr;
  };
  // chunks [lo, hi) of rows wb < wend: src -> dst
  auto copy_range = [&](const uint4* src, uint4* dst, uint32_t lo, uint32_t hi, uint32_t wend) {
    for (uint32_t wb = first_row(lo); wb < min(hi, wend); wb += step) {
      const uint32_t base = wb + lane;
      uint4 v[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const uint32_t idx = base + (uint32_t)u * stride;
        if (idx >= lo && idx < hi) v[u] = __ldcs(src + idx);
      }
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) {
        const uint32_t idx = base + (uint32_t)u * stride;
        if (idx >= lo && idx < hi) __stcs(dst + idx, v[u]);
      }
    }
  };
  const uint32_t n = f.lp ? (uint32_t)f.lp->nm : (uint32_t)__ldcg(f.n_jobs);
  // local lists: each miss lands in its landing record at once; from the moment the
  // table is seen final (slots_ready), its chunks go to the chosen slot as well.
  // (j_dual, p_dual, c_dual): the first job, part and row written to both; what came
  // before is copied over at the end.
  bool planned = !f.lp;
  uint32_t j_dual = n, p_dual = 0, c_dual = 0;
  for (uint32_t j = 0; j < n; ++j) {
    const uint4* src;
    uint4* dst;
    uint4* dst2 = nullptr;
    int e = -1;
    if (f.lp) {
      e = f.lp->expert[f.lp->elist[1][j]];
      src = reinterpret_cast<const uint4*>(f.host_layer + (size_t)e * a.rec);
      dst = reinterpret_cast<uint4*>(const_cast<uint8_t*>(a.records) + (size_t)(f.rid_land0 + (int)j) * a.rec);
      if (planned) dst2 = slot_record(e);
    } else {
      src = reinterpret_cast<const uint4*>(f.jobs[j].src);
      dst = reinterpret_cast<uint4*>(f.jobs[j].dst);
    }
    for (uint32_t part = 0; part < 2; ++part) {
      const uint32_t lo = part ? f.part16 : 0u, hi = part ? f.tile16 : f.part16;
      for (uint32_t wb = first_row(lo); wb < hi; wb += step) {
        if (!planned) {
          uint32_t pv = 0;
          if (lane == 0) pv = ld_acquire(f.slots_ready);
          planned = __shfl_sync(0xffffffffu, pv, 0) != 0u;
          if (planned) {
            dst2 = slot_record(e);
            j_dual = j;
            p_dual = part;
            c_dual = wb;
          }
        }
        const uint32_t base = wb + lane;
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
          const uint32_t idx = base + (uint32_t)u * stride;
          if (idx >= lo && idx < hi) v[u] = __ldcs(src + idx);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
          const uint32_t idx = base + (uint32_t)u * stride;
          if (idx >= lo && idx < hi) {
            __stcs(dst + idx, v[u]);
            if (dst2) __stcs(dst2 + idx, v[u]);
          }
        }
      }
      __threadfence();
      asm volatile("bar.sync 2, %0;" ::"r"(nthr) : "memory");
      if (tid == 0) release_add(part ? &f.jdone_w2[j] : &f.jdone[j]);
    }
  }
  if (f.lp && n > 0) {
    // the chunks that landed before the table was seen final, into their slots: this
    // thread re-reads only what it wrote
    if (!planned) {
      bool ok = true;
      if (lane == 0) ok = wait_count(f.slots_ready, 1u, a.status, a.wait_ns);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) set_status(a.status, MOE_ERR_TIMEOUT);
      planned = ok;
    }
    for (uint32_t j = 0; planned && j < n && j <= j_dual; ++j) {
      uint4* dst = slot_record(f.lp->expert[f.lp->elist[1][j]]);
      if (!dst) continue;
      const uint4* src = reinterpret_cast<const uint4*>(a.records + (size_t)(f.rid_land0 + (int)j) * a.rec);
      for (uint32_t part = 0; part < 2; ++part) {
        const bool before = j < j_dual || part < p_dual;
        if (!before && part > p_dual) break;
        copy_range(src, dst, part ? f.part16 : 0u, part ? f.tile16 : f.part16, before ? f.tile16 : c_dual);
      }
    }
  }
}

// 32 KB of weight tiles plus two activation tiles of N x 64 bf16 (1 KB aligned)
__host__ __device__ constexpr uint32_t fused_stage_bytes(int N) {
  return (2 * kTileBytes + 2u * (uint32_t)N * BK * 2 + 1023u) & ~1023u;
}

__device__ __forceinline__ void st_f4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

// The fused FFN of one layer call, run by every CTA of a cooperative grid of
// kFusedThreads-thread CTAs; smem_raw: the CTA's dynamic shared memory.  pre()
// runs on every thread between the CTA's setup (barriers, TMEM) and the first
// read of the step's work lists, and returns false if they will not come.
template <int WF, typename Pre>
__device__ __forceinline__ void fused_ffn(const CUtensorMap* map_x_p, const CUtensorMap* map_h_p,
                                          const CUtensorMap* map_w13_p, const CUtensorMap* map_w2_p, const Args& a,
                                          const FusedArgs& f, uint8_t* smem_raw, Pre pre) {
  using Shape = FusedShape<WF>;
  const CUtensorMap& map_x = *map_x_p;
  const CUtensorMap& map_h = *map_h_p;
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t tfull_bar[kFusedBufs], tempty_bar[kFusedBufs], drain_bar;
  __shared__ __align__(8) uint64_t conv_bar[WF == kWfFp8 ? kMaxStages : 1];   // stage expanded to bf16
  __shared__ float scale_sh[WF == kWfFp8 ? 2 : 1][WF == kWfFp8 ? 128 : 1];    // the unit's block scales
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh, last_sh;
  __shared__ FSched sched_sh;
  __shared__ float wloc_sh[32];                                              // routing weights of one entry (local lists)
  __shared__ int unit_q[kUnitQ];                                             // this CTA's units, in the order taken
  __shared__ volatile int unit_n;                                            // entries of unit_q published
  __shared__ volatile int epi_unit_sh[2], conv_unit_sh[2];                   // a unit handed to the epilogue / converter warps
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = a.N;
  const int S = a.stages;
  const int G = gridDim.x;
  // A stage holds 32 KB of weights and up to two activation tiles:
  //   gate/up: [gate tile | up tile | x tile], one K block;
  //   down:    [W tile kb | W tile kb+1 | h tile kb | h tile kb+1], two K blocks.
  const uint32_t b_bytes = (uint32_t)N * BK * 2;
  const uint32_t stage_bytes = fused_stage_bytes(N);
  // as many TMEM accumulator buffers as fit (up to 8): the MMA warp runs ahead of the epilogue
  const int nbuf = min(kFusedBufs, 512 / (2 * N));
  const uint32_t acc_cols = (uint32_t)(2 * N);
  uint32_t ncols = 32;
  while (ncols < (uint32_t)nbuf * acc_cols) ncols <<= 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      if (WF == kWfFp8) mbar_init(&conv_bar[s], 32 * kConvWarps);
    }
    for (int b = 0; b < kFusedBufs; ++b) {
      mbar_init(&tfull_bar[b], 1);
      mbar_init(&tempty_bar[b], 4);
    }
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, ncols);
  fence_before();
  __syncthreads();
  fence_after();
  const bool go = pre();
  // Local lists and a step with misses: CTAs cta0_plans .. + kCopyCtas - 1 first copy the
  // misses with all their threads, so that the other CTAs' stores and fences never queue
  // behind host reads, and take expert units only afterwards.  Otherwise the copy warps of
  // every CTA copy.
  const int ncopy = go && f.lp && f.lp->nm > 0 ? min(kCopyCtas, G - f.cta0_plans - 1) : 0;
  const bool copy_cta = ncopy > 0 && (int)blockIdx.x >= f.cta0_plans && (int)blockIdx.x < f.cta0_plans + ncopy;
  const uint32_t njd = ncopy > 0 ? (uint32_t)ncopy : (uint32_t)(G - f.cta0_plans);   // CTAs releasing each job
  if (threadIdx.x == 0) {
    unit_n = 0;
    if (go) {
      sched_sh = fused_sched(a, f, G);   // the unit decomposition, identical in every role and CTA
    } else {
      sched_sh = FSched{};
      abort_sh = 1;
    }
  }
  __syncthreads();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t idesc = idesc_bf16(N);

  // Units are handed out at run time: the producer takes the next unit of the step's
  // schedule from a grid-wide counter whenever it moves on, so CTAs that finish early
  // (or join late: the planner, the copy CTAs) take more; the CTA's other roles read
  // the units it took, in order, from unit_q (-1 ends the list).  The producer is at
  // most stages + TMEM buffers units ahead of the epilogue, well inside kUnitQ.
  auto publish_unit = [&](int k, int g) {
    unit_q[k % kUnitQ] = g;
    __threadfence_block();
    unit_n = k + 1;
  };
  auto unit_at = [&](int k) -> int {   // bounded wait (~1 s); -1 also after a timeout
    if (unit_n <= k) {
      const uint64_t t0 = global_ns();
      while (unit_n <= k) {
        if (abort_sh || global_ns() - t0 > a.wait_ns) {
          set_status(a.status, MOE_ERR_TIMEOUT);
          abort_sh = 1;
          return -1;
        }
        __nanosleep(32);
      }
    }
    __threadfence_block();
    return unit_q[k % kUnitQ];
  };

  if (copy_cta) copy_records(a, f, blockDim.x, threadIdx.x, (uint32_t)((int)blockIdx.x - f.cta0_plans), (uint32_t)ncopy);
  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      const FSched sc = sched_sh;
      uint32_t it = 0;
      bool ok = true;
      int pend_s[kMaxStages], pend_kb[kMaxStages], pend_nk[kMaxStages];
      int npub = 0;   // units published; the list ends with -1 right after them, never over one
      // Two queues: the resident entries' units (next_unit, one taken ahead) and the copied
      // entries' units, job by job (next_miss).  A copied entry's unit whose part of the
      // record has landed goes first, so the copies' tail is spread over every CTA that is
      // between units then; once the resident units are gone, the copied ones in any case.
      constexpr uint32_t kNone = 0xffffffffu;
      const uint32_t nhit = (uint32_t)(sc.p0 + sc.p1), nmu = (uint32_t)sc.total - nhit;
      const int gu_per = sc.mt_i * sc.sg, job_per = gu_per + sc.mt_h * sc.sd;
      // A CTA that starts on expert work at once (not the planner, not a copy CTA) takes
      // its first resident unit by its own index, without a round trip to the grid's
      // counter; the counter hands out the units after those.
      const int first = (int)blockIdx.x - f.cta0_plans - ncopy;
      const uint32_t nfirst = (uint32_t)(G - f.cta0_plans - ncopy);
      uint32_t hn = !go ? kNone : first >= 0 ? (uint32_t)first : nfirst + atomicAdd(f.next_unit, 1u);
      // The counter's answer for the next unit is read only when the next unit starts (after
      // this one's loads went out), so its round trip never holds up a unit's first load.
      uint32_t hraw = 0;
      bool hpend = false;
      for (;;) {
        if (hpend) {
          hn = nfirst + hraw;
          hpend = false;
        }
        if (!ok || abort_sh || !go) break;
        uint32_t g = kNone;
        if (nmu > 0) {
          const uint32_t m = *reinterpret_cast<volatile uint32_t*>(f.next_miss);
          bool take = m < nmu && hn >= nhit;
          if (m < nmu && !take) {
            const int j = (int)m / job_per;
            const uint32_t* part = (int)m - j * job_per < gu_per ? &f.jdone[j] : &f.jdone_w2[j];
            take = *reinterpret_cast<const volatile uint32_t*>(part) >= njd;
          }
          if (take) {
            const uint32_t got = atomicAdd(f.next_miss, 1u);
            if (got < nmu) g = nhit + got;
          }
        }
        bool ask = false;
        if (g == kNone && hn < nhit) {
          g = hn;
          ask = true;
        }
        if (g == kNone) break;
        publish_unit(npub, (int)g);
        ++npub;
        if (ask) {
          // the next one, while this one's loads go out; asked only after the publish, whose
          // fence would otherwise wait for the counter's round trip
          hraw = atomicAdd(f.next_unit, 1u);
          hpend = true;
        }
        const FUnit r = fused_unit(sc, f, (int)g);
        int rid = 0;
        if (!r.miss) rid = f.lp ? f.lp->rid[r.u] : a.work[r.u].rid;
        if (r.miss) {
          // a copied record: every copying CTA's slice of the part this unit reads must
          // have landed (down units too: their weight tiles go out before h is complete)
          if (!wait_count(r.gu ? &f.jdone[r.li] : &f.jdone_w2[r.li], njd, a.status, a.wait_ns)) { ok = false; break; }
          asm volatile("fence.proxy.async.global;" ::: "memory");   // generic writes -> bulk-copy reads
          // the landing record, or the plan's choice (slot or one-step record)
          rid = f.lp ? f.rid_land0 + r.li : __ldcg(&a.work[r.u].rid);
        }
        // down: h of this entry complete?  If not yet, weight tiles are issued
        // ahead and their h tiles once it is (at the latest when the ring is full)
        bool h_ok = r.gu || ld_acquire(&f.hready[r.u]) >= (uint32_t)sc.mt_i;
        if (!r.gu && h_ok) asm volatile("fence.proxy.async.global;" ::: "memory");
        int npend = 0;
        auto resolve = [&]() -> bool {
          if (!wait_count(&f.hready[r.u], (uint32_t)sc.mt_i, a.status, a.wait_ns)) return false;
          asm volatile("fence.proxy.async.global;" ::: "memory");   // h written by other CTAs -> TMA reads
          for (int q = 0; q < npend; ++q)
            for (int j = 0; j < pend_nk[q]; ++j)
              tma_load_3d(smem + (size_t)pend_s[q] * stage_bytes + 2 * kTileBytes + j * b_bytes, &map_h,
                          &full_bar[pend_s[q]], (pend_kb[q] + j) * BK, 0, r.u);
          npend = 0;
          h_ok = true;
          return true;
        };
        const uint8_t* wbase = a.records + (size_t)rid * a.rec + (r.gu ? a.off13 : a.off2) +
                               (size_t)r.mt * (r.gu ? sc.kb_h * 2 * kTileBytes : sc.kb_i * kTileBytes);
        const int kstep = r.gu ? 1 : 2;
        for (int kb = r.kb0; kb < r.kb1; kb += kstep, ++it) {
          const int s = it % S;
          const int nk = min(kstep, r.kb1 - kb);
          if (!h_ok && npend == S && !resolve()) { ok = false; break; }
          if (it >= (uint32_t)S && !mbar_wait(&empty_bar[s], ((it / S) - 1) & 1)) { ok = false; break; }
          if (abort_sh) { ok = false; break; }
          uint8_t* st = smem + (size_t)s * stage_bytes;
          if (WF == kWfFp8) {
            // fp8 code tiles (128 rows x 64 bytes) into the upper half of each bf16 tile slot
            const uint32_t raw = kTileBytes / 2;
            mbar_expect_tx(&full_bar[s], (r.gu ? 2u : (uint32_t)nk) * raw + (uint32_t)nk * b_bytes);
            if (r.gu) {
              tma_load_3d(st + raw, &map_w13_p[0], &full_bar[s], kb * BK, r.mt * BM, rid);
              tma_load_3d(st + kTileBytes + raw, &map_w13_p[0], &full_bar[s], kb * BK, a.I + r.mt * BM, rid);
            } else {
              for (int j = 0; j < nk; ++j)
                tma_load_3d(st + j * kTileBytes + raw, &map_w2_p[0], &full_bar[s], (kb + j) * BK, r.mt * BM, rid);
            }
          } else {
            const uint32_t wb = r.gu ? 2 * kTileBytes : (uint32_t)nk * kTileBytes;
            mbar_expect_tx(&full_bar[s], wb + (uint32_t)nk * b_bytes);
            bulk_load(st, wbase + (size_t)kb * (r.gu ? 2 * kTileBytes : kTileBytes), wb, &full_bar[s]);
          }
          if (r.gu) {
            tma_load_3d(st + 2 * kTileBytes, &map_x, &full_bar[s], kb * BK, 0, 0);
          } else if (h_ok) {
            for (int j = 0; j < nk; ++j)
              tma_load_3d(st + 2 * kTileBytes + j * b_bytes, &map_h, &full_bar[s], (kb + j) * BK, 0, r.u);
          } else {
            pend_s[npend] = s;
            pend_kb[npend] = kb;
            pend_nk[npend] = nk;
            ++npend;
          }
        }
        if (ok && npend > 0 && !resolve()) ok = false;
      }
      publish_unit(npub, -1);
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
      const FSched sc = sched_sh;
      uint32_t it = 0;
      int local = 0;
      bool ok = true;
      for (;; ++local) {
        const int g = unit_at(local);
        if (g < 0 || !ok) break;
        const FUnit r = fused_unit(sc, f, g);
        const int buf = local % nbuf, use = local / nbuf;
        if (use > 0 && !mbar_wait(&tempty_bar[buf], (use - 1) & 1)) { ok = false; break; }
        fence_after();
        const uint32_t dacc = tmem + (uint32_t)buf * acc_cols;
        uint32_t acc = 0;
        const int kstep = r.gu ? 1 : 2;
        for (int kb = r.kb0; kb < r.kb1; kb += kstep, ++it) {
          const int s = it % S;
          if (!mbar_wait(WF == kWfFp8 ? &conv_bar[s] : &full_bar[s], (it / S) & 1) || abort_sh) { ok = false; break; }
          fence_after();
          const uint32_t base = smem_u32(smem + (size_t)s * stage_bytes);
          if (r.gu) {
            const uint64_t da = desc_sw128(base);
            const uint64_t db = desc_sw128(base + 2 * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // advance 16 bf16 = 32 bytes along K inside the swizzle atom
              mma_bf16(dacc, da + 2 * kk, db + 2 * kk, idesc, acc);
              mma_bf16(dacc + N, da + (kTileBytes >> 4) + 2 * kk, db + 2 * kk, idesc, acc);
              acc = 1;
            }
          } else {
            const int nk = min(2, r.kb1 - kb);
            for (int j = 0; j < nk; ++j) {
              const uint64_t da = desc_sw128(base + j * kTileBytes);
              const uint64_t db = desc_sw128(base + 2 * kTileBytes + j * b_bytes);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                mma_bf16(dacc, da + 2 * kk, db + 2 * kk, idesc, acc);
                acc = 1;
              }
            }
          }
          mma_commit(&empty_bar[s]);
        }
        if (ok) mma_commit(&tfull_bar[buf]);
      }
      if (!ok) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
      }
      mma_commit(&drain_bar);
      mbar_wait(&drain_bar, 0);
    }
  } else if (warp < kThreads / 32) {
    // ------------------------------------------------------------- epilogue (warps 2..5)
    // Every epilogue warp runs the same units and reaches every named barrier,
    // even after a timeout, so no warp is left waiting.
    const FSched sc = sched_sh;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t trow0 = tmem + ((uint32_t)(q * 32) << 16);
    const int cols = sc.cols;
    int local = 0;
    for (;; ++local) {
      // one thread waits for the unit; the barrier hands it to all four warps, so they
      // always run the same units (two slots: a slot is rewritten only after the next barrier)
      if (threadIdx.x == 64) epi_unit_sh[local & 1] = unit_at(local);
      asm volatile("bar.sync 1, 128;" ::: "memory");
      const int g = epi_unit_sh[local & 1];
      if (g < 0) break;
      const FUnit r = fused_unit(sc, f, g);
      const int buf = local % nbuf;
      const uint32_t trow = trow0 + (uint32_t)buf * acc_cols;
      bool live = !abort_sh;
      if (live && !mbar_wait(&tfull_bar[buf], (local / nbuf) & 1)) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
        live = false;
      }
      if (live) fence_after();
      if (r.gu) {
        // ------------------------------ gate/up: h[u][t][m] = w(u,t) SiLU(g) u
        const int m = r.mt * BM + row;
        const float* wrow = a.wmat + (size_t)r.u * N;
        if (f.lp) {
          // routing weight of each token for this entry, from the step's routing (N <= 32 here)
          const int et = threadIdx.x - 64;
          if (et < N) {
            const int e = f.lp->expert[r.u];
            float wv = 0.f;
            if (et < a.T) {
              if (e < 0) {
                wv = 1.f;
              } else {
                for (int j = 0; j < f.lp->k; ++j)
                  if (f.lp->ids[et * f.lp->k + j] == e) wv += f.lp->w[et * f.lp->k + j];
              }
            }
            wloc_sh[et] = wv;
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
          wrow = wloc_sh;
        }
        uint16_t* hrow = a.hbuf + (size_t)r.u * N * a.I + m;
        auto store_h = [&](int c0, const float* g16, const float* u16) {
          if (m >= a.I) return;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int t = c0 + j;
            const float wgt = t < a.T ? wrow[t] : 0.f;
            const float hv = wgt != 0.f ? wgt * silu(g16[j]) * u16[j] : 0.f;
            hrow[(size_t)t * a.I] = f32_to_bf16_rn(hv);
          }
        };
        bool done_h = false;   // this CTA wrote the finished h tile
        if (sc.sg == 1) {
          if (live) {
            for (int c0 = 0; c0 < N; c0 += 16) {
              float d0[16], d1[16];
              tmem_ld16(trow + c0, d0);
              tmem_ld16(trow + N + c0, d1);
              store_h(c0, d0, d1);
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty_bar[buf]);
            done_h = true;
          }
        } else {
          // split partial [2][row][cols]: gate then up, this thread's row contiguous
          const size_t tile = (size_t)r.u * sc.mt_i + r.mt;
          const size_t pstride = (size_t)2 * BM * cols;
          if (live) {
            float* mine = f.gu_partial + (tile * sc.sg + r.sp) * pstride + (size_t)row * cols;
            for (int c0 = 0; c0 < N; c0 += 16) {
              float d0[16], d1[16];
              tmem_ld16(trow + c0, d0);
              tmem_ld16(trow + N + c0, d1);
#pragma unroll
              for (int j = 0; j < 16; j += 4) {
                if (c0 + j < cols) {
                  st_f4(mine + c0 + j, d0[j], d0[j + 1], d0[j + 2], d0[j + 3]);
                  st_f4(mine + (size_t)BM * cols + c0 + j, d1[j], d1[j + 1], d1[j + 2], d1[j + 3]);
                }
              }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty_bar[buf]);
          }
          // One acquire-release add per CTA: it releases this CTA's partials (every thread's
          // stores are ordered before it by the barrier), and the last split to arrive
          // acquires the others' (its threads' loads are ordered after it by the next barrier).
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (warp == 2 && lane == 0) {
            last_sh = 0;
            if (!abort_sh) {
              const uint32_t old = atom_add_acq_rel(reinterpret_cast<uint32_t*>(&f.gu_cnt[tile]), 1u);
              if (old == (uint32_t)sc.sg - 1) {
                last_sh = 1;
                f.gu_cnt[tile] = 0;
              }
            }
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (last_sh && live) {
            const float* base = f.gu_partial + tile * sc.sg * pstride + (size_t)row * cols;
            for (int c0 = 0; c0 < N; c0 += 16) {
              float s0[16], s1[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) { s0[j] = 0.f; s1[j] = 0.f; }
              // 4 columns at a time: every split's gate and up values in flight, added in split order
#pragma unroll
              for (int h4 = 0; h4 < 16; h4 += 4) {
                if (c0 + h4 >= cols) continue;
                float4 v0[8], v1[8];
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                  if (b < sc.sg) {
                    const float* pt = base + (size_t)b * pstride + c0 + h4;
                    v0[b] = __ldcg(reinterpret_cast<const float4*>(pt));
                    v1[b] = __ldcg(reinterpret_cast<const float4*>(pt + (size_t)BM * cols));
                  }
                }
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                  if (b < sc.sg) {
                    float* a0 = s0 + h4;
                    float* a1 = s1 + h4;
                    a0[0] += v0[b].x; a0[1] += v0[b].y; a0[2] += v0[b].z; a0[3] += v0[b].w;
                    a1[0] += v1[b].x; a1[1] += v1[b].y; a1[2] += v1[b].z; a1[3] += v1[b].w;
                  }
                }
              }
              store_h(c0, s0, s1);
            }
            done_h = true;
          }
        }
        // publish: this entry has one more finished gate/up tile (the barrier orders
        // every thread's h stores before the one release, which is cumulative)
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (warp == 2 && lane == 0 && done_h && !abort_sh) release_add(&f.hready[r.u]);
      } else {
        // ------------------------------ down: this entry's partial [row][cols]
        if (live) {
          float* mine = f.dn_partial + (((size_t)r.u * sc.mt_h + r.mt) * sc.sd + r.sp) * ((size_t)BM * cols) +
                        (size_t)row * cols;
          for (int c0 = 0; c0 < cols; c0 += 16) {
            float d0[16];
            tmem_ld16(trow + c0, d0);
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              if (c0 + j < cols) st_f4(mine + c0 + j, d0[j], d0[j + 1], d0[j + 2], d0[j + 3]);
          }
          fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty_bar[buf]);
        }
      }
    }
    __threadfence();   // this thread's partials, before the CTA reports them written
  } else if (WF == kWfFp8 && warp < Shape::copy_warp0) {
    // ------------------------------------------------------------- converter warps (fp8)
    // Per stage: every thread reads its 4 x 16 code bytes of each tile, then (all
    // reads done) writes them back as bf16 (code * block scale, one rounding) in
    // the 128-byte-swizzled order, over the same slot.  The unit's block scales
    // are staged in shared memory at unit start (a copied record's only after
    // its first stage has landed, which orders them after the copy).
    // Every converter thread passes every named barrier of every stage, also after
    // a timeout (then it only skips the work), so none is left waiting.
    const FSched sc = sched_sh;
    const int ct = threadIdx.x - Shape::conv_warp0 * 32;        // 0..127
    uint32_t it = 0;
    int local = 0;
    bool stop = false;
    for (;; ++local) {
      if (ct == 0) conv_unit_sh[local & 1] = unit_at(local);   // handed to all four converter warps
      asm volatile("bar.sync 3, %0;" ::"n"(32 * kConvWarps) : "memory");
      const int g = conv_unit_sh[local & 1];
      if (g < 0) break;
      const FUnit r = fused_unit(sc, f, g);
      const float* scl = nullptr;
      const int b0 = r.kb0 / 2, nblk = (r.kb1 - 1) / 2 - b0 + 1;   // 128-wide scale blocks the unit spans (<= 64)
      const int sbuf = local & 1;
      // gate (or down) scales at [0, 64), up scales at [64, 128)
      auto stage_scales = [&]() {
        if (stop) return;
        // a copied entry's record is read once its first stage has landed (L2, not L1:
        // other CTAs wrote it)
        const int rid = r.miss ? (f.lp ? f.rid_land0 + r.li : __ldcg(&a.work[r.u].rid))
                               : (f.lp ? f.lp->rid[r.u] : a.work[r.u].rid);
        scl = reinterpret_cast<const float*>(a.records + (size_t)rid * a.rec + (r.gu ? f.os13 : f.os2));
        if (ct < nblk) {
          scale_sh[sbuf][ct] = __ldcg(scl + (size_t)(r.gu ? r.mt * f.sc_h : r.mt * f.sc_i) + b0 + ct);
        } else if (r.gu && ct >= 64 && ct - 64 < nblk) {
          scale_sh[sbuf][ct] = __ldcg(scl + (size_t)(a.I / BM + r.mt) * f.sc_h + b0 + (ct - 64));
        }
      };
      if (!r.miss) stage_scales();
      const int kstep = r.gu ? 1 : 2;
      bool first = true;
      for (int kb = r.kb0; kb < r.kb1; kb += kstep, ++it) {
        const int s = it % S;
        if (!stop && (!mbar_wait(&full_bar[s], (it / S) & 1) || abort_sh)) {
          stop = true;
          set_status(a.status, MOE_ERR_TIMEOUT);
          abort_sh = 1;
        }
        if (first) {
          if (r.miss) stage_scales();
          asm volatile("bar.sync 3, %0;" ::"n"(32 * kConvWarps) : "memory");
          first = false;
        }
        const int nt = r.gu ? 2 : min(2, r.kb1 - kb);
        const float s0 = scale_sh[sbuf][kb / 2 - b0];
        const float s1 = r.gu ? scale_sh[sbuf][64 + kb / 2 - b0] : (nt > 1 ? scale_sh[sbuf][(kb + 1) / 2 - b0] : 0.f);
        fp8_expand_stage<32 * kConvWarps>(smem + (size_t)s * stage_bytes, nt, s0, s1, ct, !stop);
        if (!stop) mbar_arrive(&conv_bar[s]);
      }
      asm volatile("bar.sync 3, %0;" ::"n"(32 * kConvWarps) : "memory");   // before the scale buffer is reused
    }
  } else if (!f.lp && go) {
    // ------------------------------------------------------------- copy warps
    copy_records(a, f, 32u * kCopyWarps, (uint32_t)(warp - Shape::copy_warp0) * 32u + lane, blockIdx.x, (uint32_t)G);
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) tmem_dealloc(tmem, ncols);

  // ---- combine: once every CTA's down partials are written, all threads of all
  // CTAs sum them element-parallel, each element over (entry, split) in order
  if (threadIdx.x == 0) {
    last_sh = 0;
    if (!abort_sh) {
      release_add(f.dn_done);
      last_sh = wait_count(f.dn_done, (uint32_t)G, a.status, a.wait_ns) ? 1 : 0;
      if (!last_sh) set_status(a.status, MOE_ERR_TIMEOUT);
    }
  }
  __syncthreads();
  if (last_sh) {
    __threadfence();
    const FSched sc = sched_sh;
    const uint32_t cols = (uint32_t)sc.cols;
    const uint32_t tile_el = (uint32_t)BM * cols;
    const uint32_t total_el = (uint32_t)sc.mt_h * tile_el;
    const size_t ustride = (size_t)sc.mt_h * sc.sd * tile_el;
    const int parts = sc.n * sc.sd;
    for (uint32_t e0 = blockIdx.x * blockDim.x + threadIdx.x; e0 < total_el; e0 += (uint32_t)G * blockDim.x) {
      const uint32_t mt = e0 / tile_el;
      const uint32_t rem = e0 - mt * tile_el;
      const uint32_t rw = rem / cols, t = rem - rw * cols;
      const uint32_t m = mt * BM + rw;
      if (t >= (uint32_t)a.T || m >= (uint32_t)a.H) continue;
      const float* base = f.dn_partial + (size_t)mt * sc.sd * tile_el + rem;
      // part q = (entry u, split sp), q = u * sd + sp, at base + u * ustride + sp * tile_el.
      // Each batch's addresses come straight from q (past the end: the last part again, never
      // added), so its 16 loads are independent and all in flight at once.
      float acc = 0.f;
      const int sd = sc.sd;
      if (f.lp) {
        // local lists: only the token's own entries (every other entry's partial for it is
        // +-0, its h column being zero), in the token's gate rank order, then the shared
        // expert: a fixed order for a given routing
        const LocalPlan& lp = *f.lp;
        const int kq = lp.k, kp = kq + (lp.n > 0 && lp.expert[lp.n - 1] < 0 ? 1 : 0);
        const int tparts = kp * sd;
        for (int p0 = 0; p0 < tparts; p0 += 16) {
          float v[16];
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const int q = min(p0 + b, tparts - 1);
            const int j = sd == 1 ? q : q / sd;
            const int e = j < kq ? lp.ids[t * kq + j] : -1;
            const int u = (unsigned)e < (unsigned)kMaxE ? lp.epos[e] : lp.n - 1;
            v[b] = __ldcg(base + (size_t)u * ustride + (size_t)(q - j * sd) * tile_el);
          }
#pragma unroll
          for (int b = 0; b < 16; ++b)
            if (p0 + b < tparts) acc += v[b];
        }
      } else {
        for (int p0 = 0; p0 < parts; p0 += 16) {
          float v[16];
#pragma unroll
          for (int b = 0; b < 16; ++b) {
            const int q = min(p0 + b, parts - 1);
            const int u = sd == 1 ? q : q / sd;
            v[b] = __ldcg(base + (size_t)u * ustride + (size_t)(q - u * sd) * tile_el);
          }
#pragma unroll
          for (int b = 0; b < 16; ++b)
            if (p0 + b < parts) acc += v[b];
        }
      }
      a.out[(size_t)t * a.H + m] = f32_to_bf16_rn(acc);
    }
  }
}

// ----------------------------------------------------------------- streaming decode FFN (one token)
// With one token, a layer call is one matrix-vector product per expert: each
// weight streams from HBM once and feeds one multiply-add, which the CUDA cores
// keep up with, so the tensor cores buy nothing.  What costs time on the
// tensor-core path at this size is its structure: gate/up tiles
// split along K (partials, arrivals and a reduction per tile before the down
// projection may start) and a grid-wide combine of per-entry down partials.
// This path has neither:
//   phase 1: unit = (work entry u, 16 rows of a 128-row tile of I), all of K.  The
//            unit's gate and up rows stream through a shared-memory ring (the 2 KB
//            16-row segments of the swizzled 128 x 64 tiles); each
//            compute warp owns two rows of gate and of up and finishes
//            h = w(u,t) SiLU(W_gate x_t) (W_up x_t) itself, in fp32, into global
//            scratch (rows past I as 0).
//   arrival: every CTA's phase-1 units are done (one grid-wide counter).
//   phase 2: unit = 16 rows of H, every entry in work order (ascending expert id,
//            shared expert last): each stage carries W_down row segments of one
//            entry and the matching slice of its h; each compute warp owns two
//            output rows and sums over entries and K in registers, and writes
//            out directly: no partials, no combine.  A CTA issues the weight
//            segments of its first phase-2 stages before the arrival (they need
//            no h) and their h slices after it.
// A stage is one tiled tensor load (phase 2: two, W_down and h): the 16-row segments of
// 8 tiles, 32 KB, arrive in one request instead of sixteen 2 KB copies.
// Misses are copied as on the tensor-core path (copy CTAs, landing records);
// a copied entry's phase-1 units wait for its gate/up part and its phase-2
// stages for the rest.  Every sum runs in one fixed order (each lane's partial in
// stage and element order, then a butterfly over the lanes), and no unit's rows
// depend on which experts are resident, so neither does the output.
// Tokens the path takes.  The code is written for up to four, but measured on the
// Qwen3-shaped layer it beats the tensor-core path only at one token (all experts
// resident: 35.7-39.8 vs 43 us per call); at four it is slower (83 vs ~60 us): its
// 16-row units read each tile as 2 KB pieces, whose loads wait far longer than
// the tensor-core path's contiguous 32 KB stages.
constexpr int kStreamMaxT = 1;
constexpr int kStreamRows = 16;                  // rows per unit
constexpr int kStreamKb = 8;                     // 64-column K blocks per stage
constexpr int kStreamWarps = 8;                  // compute warps; warp kStreamWarps issues the copies
constexpr int kStreamThreads = (kStreamWarps + 1) * 32;
constexpr uint32_t kStreamSeg = kStreamRows * 128;            // one row segment of a tile: 2 KB
constexpr uint32_t kStreamStage = 2 * kStreamKb * kStreamSeg; // 32 KB: gate and up segments of 8 K blocks
constexpr uint32_t kStreamHOff = kStreamKb * kStreamSeg;      // phase 2: h slices after the W_down segments
constexpr int kStreamQ = 64;
constexpr int kStreamEnd1 = -2, kStreamEnd = -1, kStreamP2 = 1 << 30;

// 8 bf16 weights (one 16-byte chunk) as floats
__device__ __forceinline__ void unpack8_bf16(const uint4& w, float* f) {
  f[0] = bf16lo(w.x); f[1] = bf16hi(w.x); f[2] = bf16lo(w.y); f[3] = bf16hi(w.y);
  f[4] = bf16lo(w.z); f[5] = bf16hi(w.z); f[6] = bf16lo(w.w); f[7] = bf16hi(w.w);
}

// dot product of 8 weights with 8 activations, in element order
__device__ __forceinline__ float dot8(const float* w, const float* v, float acc) {
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = fmaf(w[i], v[i], acc);
  return acc;
}

// 16 bytes from shared memory at a shared-window address (explicitly shared: the
// ring's pointers come from aligned integer arithmetic, so the compiler cannot tell
// they address shared memory and would emit generic loads)
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float butterfly_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// smem_raw: the CTA's dynamic shared memory; pre(): as for fused_ffn.  bf16 tiled
// records, local lists (f.lp), T <= kStreamMaxT.
// map_w13 / map_w2: the row-segment maps of the records (TcMaps::sw13 / sw2); map_h: h as
// [work position][T][Ip / 64][64] fp32, boxes of 8 K blocks of every token.
template <typename Pre>
__device__ __forceinline__ void stream_ffn(const CUtensorMap* map_w13, const CUtensorMap* map_w2,
                                           const CUtensorMap* map_h, const Args& a, const FusedArgs& f,
                                           const uint16_t* __restrict__ x, uint8_t* smem_raw, Pre pre) {
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ int unit_q[kStreamQ];
  __shared__ volatile int unit_n;
  __shared__ volatile int abort_sh;
  __shared__ int jpos_sh[kMaxE + 1];     // copied index of each work position, or -1
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  const int T = a.T, H = a.H, I = a.I;
  const int S = a.stages;
  const int kb_h = (H + 63) / 64, kb_i = (I + 63) / 64, mt_i = (I + 127) / 128, mt_h = (H + 127) / 128;
  const int Hp = kb_h * 64, Ip = kb_i * 64;
  const int rg_tile = 128 / kStreamRows;
  float* xs = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = reinterpret_cast<uint8_t*>(xs) + (((size_t)T * Hp * 4 + 1023) & ~(size_t)1023);
  float* hf = reinterpret_cast<float*>(a.hbuf);   // [work position][T][Ip] fp32

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kStreamWarps);
    }
    unit_n = 0;
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool go = pre();
  if (!go && threadIdx.x == 0) abort_sh = 1;
  const LocalPlan* lp = f.lp;
  const int n = go ? lp->n : 0, nh = go ? lp->nh : 0, nm = go ? lp->nm : 0;
  const int ncopy = go && nm > 0 ? min(kCopyCtas, G - f.cta0_plans - 1) : 0;
  const bool copy_cta = ncopy > 0 && (int)blockIdx.x >= f.cta0_plans && (int)blockIdx.x < f.cta0_plans + ncopy;
  const uint32_t njd = (uint32_t)max(ncopy, 1);
  if (go) {
    for (int i = threadIdx.x; i <= kMaxE; i += blockDim.x) jpos_sh[i] = -1;
    __syncthreads();
    for (int j = threadIdx.x; j < nm; j += blockDim.x) jpos_sh[lp->elist[1][j]] = j;
    __syncthreads();
  }
  if (copy_cta) copy_records(a, f, blockDim.x, threadIdx.x, (uint32_t)((int)blockIdx.x - f.cta0_plans), (uint32_t)ncopy);
  const int per1 = mt_i * rg_tile;                  // phase-1 units per entry
  const uint32_t n1 = (uint32_t)(n * per1);         // resident entries' units first, then copied
  const uint32_t n2 = (uint32_t)(mt_h * rg_tile);   // phase-2 units
  uint32_t* p1_done = f.dn_done;
  auto publish = [&](int k, int g) {
    unit_q[k % kStreamQ] = g;
    __threadfence_block();
    unit_n = k + 1;
  };
  auto unit_at = [&](int k) -> int {   // bounded wait; kStreamEnd after a timeout
    if (unit_n <= k) {
      const uint64_t t0 = global_ns();
      while (unit_n <= k) {
        if (abort_sh || global_ns() - t0 > a.wait_ns) {
          set_status(a.status, MOE_ERR_TIMEOUT);
          abort_sh = 1;
          return kStreamEnd;
        }
        __nanosleep(32);
      }
    }
    __threadfence_block();
    return unit_q[k % kStreamQ];
  };
  // record of work position u: resident slot record, or the landing record of its copy job
  auto record_of = [&](int u) -> int { return jpos_sh[u] >= 0 ? f.rid_land0 + jpos_sh[u] : lp->rid[u]; };

  if (warp == kStreamWarps) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0;
      int npub = 0;
      bool ok = go;
      auto slot = [&](int& s) -> bool {   // the next ring stage, once its previous fill is consumed
        s = (int)(it % (uint32_t)S);
        if (it >= (uint32_t)S && !mbar_wait(&empty_bar[s], ((it / S) - 1) & 1)) return false;
        return !abort_sh;
      };
      // phase 1: a CTA that starts on expert work at once takes its first unit by index
      const int first = (int)blockIdx.x - f.cta0_plans - ncopy;
      const uint32_t nfirst = (uint32_t)(G - f.cta0_plans - ncopy);
      uint32_t g = first >= 0 ? (uint32_t)first : nfirst + atomicAdd(f.next_unit, 1u);
      while (ok && g < n1) {
        const int li = (int)g / per1, rem = (int)g - li * per1;
        const int mt = rem / rg_tile, rg = rem - mt * rg_tile;
        const bool miss = li >= nh;
        const int u = miss ? lp->elist[1][li - nh] : lp->elist[0][li];
        if (miss) {
          // the copied record's gate/up part, written by the copy CTAs
          if (!wait_count(&f.jdone[li - nh], njd, a.status, a.wait_ns)) { ok = false; break; }
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        publish(npub++, (int)g);
        // the next one, while this one's loads go out (its value is read after them; asked
        // after the publish, whose fence would otherwise wait for the counter's round trip)
        const uint32_t graw = atomicAdd(f.next_unit, 1u);
        const int rid = record_of(u);
        for (int kb0 = 0; kb0 < kb_h; kb0 += kStreamKb, ++it) {
          int s;
          if (!slot(s)) { ok = false; break; }
          // tiles 2 kb0 .. 2 kb0 + 15 (gate, up of 8 K blocks; past the last: zeros), rows rg * 16 ..
          mbar_expect_tx(&full_bar[s], kStreamStage);
          tma_load_5d_ef(ring + (size_t)s * kStreamStage, map_w13, &full_bar[s], 0, rg * kStreamRows, 2 * kb0, mt, rid);
        }
        g = nfirst + graw;
      }
      publish(npub++, kStreamEnd1);
      // phase 2: units handed out by a second counter.  Until every CTA's h is written,
      // stages go out with their W_down segments only; their h slices follow the arrival.
      bool h_ok = false;
      int pend_s[kMaxStages], pend_u[kMaxStages], pend_kb[kMaxStages], npend = 0;
      auto issue_h = [&](int s, int u, int kb0) {   // K blocks kb0 .. kb0 + 7 of every token's h
        tma_load_4d(ring + (size_t)s * kStreamStage + kStreamHOff, map_h, &full_bar[s], 0, kb0, 0, u);
      };
      auto arrival = [&]() -> bool {
        if (!wait_count(p1_done, (uint32_t)(G - f.cta0_plans) * kStreamWarps, a.status, a.wait_ns)) return false;
        asm volatile("fence.proxy.async.global;" ::: "memory");   // h written by every CTA -> bulk reads
        h_ok = true;
        for (int q = 0; q < npend; ++q) issue_h(pend_s[q], pend_u[q], pend_kb[q]);
        npend = 0;
        return true;
      };
      while (ok) {
        // one unit at a time: a CTA reaching phase 2 early must not hold a second unit that
        // a CTA arriving later would start sooner
        const uint32_t g2 = atomicAdd(f.next_miss, 1u);
        if (g2 >= n2) break;
        publish(npub++, kStreamP2 | (int)g2);
        const int mt = (int)g2 / rg_tile, rg = (int)g2 - mt * rg_tile;
        for (int u = 0; ok && u < n; ++u) {
          if (jpos_sh[u] >= 0) {
            // a copied record's W_down part (it lands after every gate/up part, so the
            // arrival comes first: the stages already issued get their h meanwhile)
            if (!h_ok && npend > 0 && !arrival()) { ok = false; break; }
            if (!wait_count(&f.jdone_w2[jpos_sh[u]], njd, a.status, a.wait_ns)) { ok = false; break; }
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
          const int rid = record_of(u);
          for (int kb0 = 0; kb0 < kb_i; kb0 += kStreamKb, ++it) {
            // every ring stage waiting for its h slice: the arrival first (the oldest stage
            // cannot be consumed before it)
            if (!h_ok && npend == S && !arrival()) { ok = false; break; }
            int s;
            if (!slot(s)) { ok = false; break; }
            // W_down tiles kb0 .. kb0 + 7 (past the last: zeros), rows rg * 16 .., and the h slice
            mbar_expect_tx(&full_bar[s], kStreamHOff + (uint32_t)T * kStreamKb * 256);
            tma_load_5d_ef(ring + (size_t)s * kStreamStage, map_w2, &full_bar[s], 0, rg * kStreamRows, kb0, mt, rid);
            if (h_ok) {
              issue_h(s, u, kb0);
            } else {
              pend_s[npend] = s;
              pend_u[npend] = u;
              pend_kb[npend] = kb0;
              ++npend;
            }
          }
        }
      }
      if (ok && npend > 0 && !arrival()) ok = false;
      publish(npub++, kStreamEnd);
      if (!ok) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
        // stages still waiting for their h slice get one anyway (in-bounds reads of the
        // scratch), so that their weight copies can be waited for below
        for (int q = 0; q < npend; ++q) issue_h(pend_s[q], pend_u[q], pend_kb[q]);
        npend = 0;
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
  } else {
    // ------------------------------------------------------------- compute warps
    constexpr int NC = kStreamWarps * 32;
    // x staged once as fp32 [T][Hp], zero past H
    for (int i = threadIdx.x; i < T * (Hp / 8); i += NC) {
      const int t = i / (Hp / 8), c = i - t * (Hp / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (go && c * 8 < H) v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H + c * 8));
      float f[8];
      unpack8_bf16(v, f);
      reinterpret_cast<float4*>(xs)[2 * i] = make_float4(f[0], f[1], f[2], f[3]);
      reinterpret_cast<float4*>(xs)[2 * i + 1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(NC) : "memory");
    uint32_t it = 0;
    const uint32_t xs_a = smem_u32(xs), ring_a = smem_u32(ring);
    auto stage_wait = [&](int s) {
      if (!abort_sh && !mbar_try(&full_bar[s], (it / S) & 1) && !mbar_wait(&full_bar[s], (it / S) & 1)) {
        set_status(a.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
      }
    };
    for (int k = 0;; ++k) {
      const int g = unit_at(k);
      if (g == kStreamEnd) break;
      if (g == kStreamEnd1) {
        // this warp's h stores are done: one release per warp (the warp barrier orders
        // the lanes' stores before lane 0's cumulative release)
        __syncwarp();
        if (lane == 0 && !abort_sh) release_add(p1_done);
        continue;
      }
      if (!(g & kStreamP2)) {
        // ---- phase 1: rows warp and warp + 8 of 16 rows of tile mt of entry u's gate and up
        const int li = g / per1, rem = g - li * per1;
        const int mt = rem / rg_tile, rg = rem - mt * rg_tile;
        const int u = li >= nh ? lp->elist[1][li - nh] : lp->elist[0][li];
        // lane t: the routing weight of token t for this entry (1 for the shared expert), read
        // from the step's routing once per unit, while the unit's first stage is in flight
        float wt_lane = 0.f;
        if (lane < T) {
          const int e = lp->expert[u], kk = lp->k;
          if (e < 0) {
            wt_lane = 1.f;
          } else {
            for (int j = 0; j < kk; ++j)
              if (lp->ids[lane * kk + j] == e) wt_lane += lp->w[lane * kk + j];
          }
        }
        float acc[4][kStreamMaxT];
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
          for (int t = 0; t < kStreamMaxT; ++t) acc[p][t] = 0.f;
        for (int kb0 = 0; kb0 < kb_h; kb0 += kStreamKb, ++it) {
          const int s = (int)(it % (uint32_t)S);
          stage_wait(s);
          const int nk = min(kStreamKb, kb_h - kb0);
          if (!abort_sh) {
            // this lane's chunks c = lane and lane + 32 of the stage (chunk c % 8 of K block
            // c / 8): a chunk's shared-memory loads first, then its multiply-adds
            const uint32_t st = ring_a + (uint32_t)s * kStreamStage;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int c = lane + 32 * cc, kbi = c >> 3, q = c & 7;
              if (kbi < nk) {
                uint4 xq[kStreamMaxT][2], wq[4];
#pragma unroll
                for (int t = 0; t < kStreamMaxT; ++t) {
                  if (t < T) {
                    const uint32_t xa = xs_a + (uint32_t)(t * Hp + (kb0 + kbi) * 64 + q * 8) * 4u;
                    xq[t][0] = lds128(xa);
                    xq[t][1] = lds128(xa + 16);
                  }
                }
#pragma unroll
                for (int pr = 0; pr < 4; ++pr) {   // gate row warp, gate row warp + 8, up row warp, up row warp + 8
                  const int m = pr >> 1, lr = warp + 8 * (pr & 1);
                  wq[pr] = lds128(st + (uint32_t)(kbi * 2 + m) * kStreamSeg + lr * 128 + ((q ^ (lr & 7)) << 4));
                }
#pragma unroll
                for (int pr = 0; pr < 4; ++pr) {
                  float wv[8];
                  unpack8_bf16(wq[pr], wv);   // once per chunk, for every token
#pragma unroll
                  for (int t = 0; t < kStreamMaxT; ++t) {
                    if (t < T) {
                      const float xv[8] = {__uint_as_float(xq[t][0].x), __uint_as_float(xq[t][0].y),
                                           __uint_as_float(xq[t][0].z), __uint_as_float(xq[t][0].w),
                                           __uint_as_float(xq[t][1].x), __uint_as_float(xq[t][1].y),
                                           __uint_as_float(xq[t][1].z), __uint_as_float(xq[t][1].w)};
                      acc[pr][t] = dot8(wv, xv, acc[pr][t]);
                    }
                  }
                }
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
          const int i = mt * 128 + rg * kStreamRows + warp + 8 * ri;
#pragma unroll
          for (int t = 0; t < kStreamMaxT; ++t) {
            if (t < T) {
              const float gs = butterfly_sum(acc[ri][t]);
              const float us = butterfly_sum(acc[2 + ri][t]);
              const float wt = __shfl_sync(0xffffffffu, wt_lane, t);
              if (lane == 0 && i < Ip) hf[((size_t)u * T + t) * Ip + i] = i < I && wt != 0.f ? wt * silu(gs) * us : 0.f;
            }
          }
        }
      } else {
        // ---- phase 2: rows 2 warp and 2 warp + 1 of 16 rows of tile mt of H, every entry
        const int g2 = g & ~kStreamP2;
        const int mt = g2 / rg_tile, rg = g2 - mt * rg_tile;
        float acc[2][kStreamMaxT];
#pragma unroll
        for (int ri = 0; ri < 2; ++ri)
#pragma unroll
          for (int t = 0; t < kStreamMaxT; ++t) acc[ri][t] = 0.f;
        for (int u = 0; u < n; ++u) {
          for (int kb0 = 0; kb0 < kb_i; kb0 += kStreamKb, ++it) {
            const int s = (int)(it % (uint32_t)S);
            stage_wait(s);
            const int nk = min(kStreamKb, kb_i - kb0);
            if (!abort_sh) {
              // this lane's chunks c = lane and lane + 32: a chunk's h slices and W_down rows
              // first, then its multiply-adds
              const uint32_t st = ring_a + (uint32_t)s * kStreamStage;
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const int c = lane + 32 * cc, kbi = c >> 3, q = c & 7;
                if (kbi < nk) {
                  uint4 hq[kStreamMaxT][2], wq[2];
#pragma unroll
                  for (int t = 0; t < kStreamMaxT; ++t) {
                    if (t < T) {
                      const uint32_t hp = st + kStreamHOff + (uint32_t)t * kStreamKb * 256 + (uint32_t)(kbi * 64 + q * 8) * 4u;
                      hq[t][0] = lds128(hp);
                      hq[t][1] = lds128(hp + 16);
                    }
                  }
#pragma unroll
                  for (int ri = 0; ri < 2; ++ri) {
                    const int lr = 2 * warp + ri;
                    wq[ri] = lds128(st + (uint32_t)kbi * kStreamSeg + lr * 128 + ((q ^ (lr & 7)) << 4));
                  }
#pragma unroll
                  for (int ri = 0; ri < 2; ++ri) {
                    float wv[8];
                    unpack8_bf16(wq[ri], wv);   // once per chunk, for every token
#pragma unroll
                    for (int t = 0; t < kStreamMaxT; ++t) {
                      if (t < T) {
                        const float hv[8] = {__uint_as_float(hq[t][0].x), __uint_as_float(hq[t][0].y),
                                             __uint_as_float(hq[t][0].z), __uint_as_float(hq[t][0].w),
                                             __uint_as_float(hq[t][1].x), __uint_as_float(hq[t][1].y),
                                             __uint_as_float(hq[t][1].z), __uint_as_float(hq[t][1].w)};
                        acc[ri][t] = dot8(wv, hv, acc[ri][t]);
                      }
                    }
                  }
                }
              }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[s]);
          }
        }
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
          const int m = mt * 128 + rg * kStreamRows + 2 * warp + ri;
#pragma unroll
          for (int t = 0; t < kStreamMaxT; ++t) {
            if (t < T) {
              const float v = butterfly_sum(acc[ri][t]);
              if (lane == 0 && m < H && !abort_sh) a.out[(size_t)t * H + m] = f32_to_bf16_rn(v);
            }
          }
        }
      }
    }
  }
}

template <int WF>
__global__ void __launch_bounds__(FusedShape<WF>::threads, 1)
tc_fused_decode_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_h,
                       const __grid_constant__ CUtensorMap map_w13, const __grid_constant__ CUtensorMap map_w2, Args a,
                       FusedArgs f) {
  extern __shared__ uint8_t smem_raw[];
  fused_ffn<WF>(&map_x, &map_h, &map_w13, &map_w2, a, f, smem_raw, [] { return true; });
}


// ----------------------------------------------------------------- decode layer kernel
// A decode call with few tokens (T <= 32) and bf16 or fp8 weights is one
// cooperative launch: steps a1/a2 (router and gate), a3-a5/a7 (history, table,
// victims, permutation) and the fused FFN (a6, a8, a9), without the launch gaps
// and global round trips of three kernels.
//   route: CTA 1 + t * nblk + b, t < T, b < nblk, computes the logits of token
//          t for experts [b * eb, (b + 1) * eb); the last CTA of token t
//          (ticket) runs its gate and top-k in one warp;
//   plan:  CTA 0 starts copying the plan's routing-independent inputs (history
//          rings, slot owners) into shared memory at once, and once every token
//          is gated runs the plan, from shared memory that the FFN's stage ring
//          reuses later;
//   FFN:   local lists (T k <= kLocalMaxTk): every CTA snapshots the
//          layer's table row at kernel start and, once every token is gated,
//          derives the step's entry lists from the routing and the snapshot.
//          Resident entries start at once (the plan never evicts an expert the
//          step uses); each copied entry is pulled from the host pool into a
//          landing record at once and computed from there, and written to its
//          slot once the plan has chosen it.  Otherwise every CTA waits for the
//          plan's work lists.
// Fast gate (streaming variant, local lists, no substitution): no ticket and no gating CTA; each
// routing CTA adds one to route_done once its logits are written, and every CTA,
// once all are, stages the step's logits [T][E] in shared memory and gates every
// token itself, one warp per token (CTA 0 also writes the routing outputs the plan
// and the routing dump read).
// Counters: route_done counts T gates (fast gate: T * nblk routing CTAs) plus CTA
// 0's zeroing of the expert counters; tickets reset on their last arrival; plan_done,
// snap_done, slots_ready (and, after a timeout, the others) are reset by the
// last CTA to leave, so each launch starts from zero.
struct DecodeArgs {
  int local;                // every CTA derives the step's entry lists itself (T * k <= kLocalMaxTk)
  int fast;                 // (streaming variant, local lists, no substitution) every CTA gates every token itself
  int zoff;                 // fast: byte offset in dynamic shared memory of the staged logits [T][E]
  const uint16_t* x;        // [T][H] bf16
  const uint16_t* wr;       // this layer's router [E][H] bf16
  const float* rb;          // [E]
  float* z;                 // [T][E] logits scratch
  int eb, nblk;             // experts per routing CTA, routing CTAs per token
  PlanArgs plan;
  uint32_t* dsync;          // counters, one per 128-byte line (kSyncLine ints): route_done, plan_done, exit
                            // count, CTAs holding their copy of the layer's table row, table final, then
                            // the ticket of token t at line kDsTicket + t
};
// Every counter that many CTAs poll or add to has a line of its own, so that the
// polls of one do not queue in front of the atomics of another.
constexpr int kSyncLine = 32;
constexpr int kDsRoute = 0, kDsPlan = 1, kDsExit = 2, kDsSnap = 3, kDsSlots = 4, kDsTicket = 8;

constexpr int kDecodeMaxT = 32;
constexpr int kRouterMaxSplits = 32;   // K splits of the tensor-core router
constexpr int kRouteChunks = 16;   // router-row loads in flight per lane (H <= 4096 in one round)

// STREAM: the CUDA-core streaming FFN (bf16 tiled records, T <= kStreamMaxT, local lists)
// instead of the tensor-core one.
template <int WF, bool STREAM> struct DecodeShape {
  static constexpr int threads = STREAM ? kStreamThreads : FusedShape<WF>::threads;
};

template <int WF, bool STREAM>
__global__ void __launch_bounds__(DecodeShape<WF, STREAM>::threads, 1)
tc_decode_layer_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_h,
                       const __grid_constant__ CUtensorMap map_w13, const __grid_constant__ CUtensorMap map_w2,
                       Args a, FusedArgs f, DecodeArgs d) {
  constexpr int NT = DecodeShape<WF, STREAM>::threads;
  // programmatic dependent launch: this grid may start while the previous kernel of the
  // stream drains.  Everything below reads data earlier kernels wrote, so the wait comes
  // first; the trigger after it lets the next layer call's grid be launched early (it waits
  // the same way), which also keeps every kernel before the previous one complete here.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint8_t smem_raw[];
  __shared__ volatile int flag_sh;
  __shared__ LocalPlan lp_sh;
  __shared__ int lut_snap[kMaxE];
  __shared__ int cnt_sh[kMaxE];
  uint8_t* dsm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = a.T, H = a.H, E = d.plan.p.E;
  const int G = gridDim.x;
  uint32_t* route_done = d.dsync + kDsRoute * kSyncLine;
  uint32_t* plan_done = d.dsync + kDsPlan * kSyncLine;
  uint32_t* exit_cnt = d.dsync + kDsExit * kSyncLine;
  uint32_t* snap_done = d.dsync + kDsSnap * kSyncLine;
  uint32_t* slots_ready = d.dsync + kDsSlots * kSyncLine;
  auto ticket = [&](int t) -> uint32_t* { return d.dsync + (kDsTicket + t) * kSyncLine; };
  const PoolDev& p = d.plan.p;
  const int l = d.plan.layer;
  // the fast gate exists in the streaming variant only (compiled out of the other, where it
  // measured slower: several tokens per warp)
  const bool fast = STREAM && d.fast;

  // this CTA's copy of the layer's table row, taken before the plan may change it: loaded
  // now; a routing CTA stores and releases it after its logits, off the routing's path
  constexpr int kSnapPer = (kMaxE + NT - 1) / NT;
  int snap_v[kSnapPer];
  const bool routing = blockIdx.x >= 1 && (int)blockIdx.x <= T * d.nblk;
  auto take_snapshot = [&]() {
#pragma unroll
    for (int i = 0; i < kSnapPer; ++i) {
      const int e = threadIdx.x + i * NT;
      if (e < E) lut_snap[e] = snap_v[i];
    }
    __syncthreads();
    if (threadIdx.x == 0) release_add(snap_done);
  };
  if (d.local) {
    for (int e = threadIdx.x; e < kMaxE; e += NT) cnt_sh[e] = 0;   // ordered before its use by later barriers
#pragma unroll
    for (int i = 0; i < kSnapPer; ++i) {
      const int e = threadIdx.x + i * NT;
      snap_v[i] = e < E ? p.lut[(size_t)l * E + e] : -1;
    }
    if (!routing) take_snapshot();
  }
  if (blockIdx.x == 0) {
    plan_prestage<NT>(d.plan, dsm);
    // the expert kernel's counters start from zero: one more arrival on route_done
    // (which every CTA waits for) publishes that
    for (int i = threadIdx.x; i < d.plan.sc.n_ffn_sync; i += NT) d.plan.sc.ffn_sync[i] = 0;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) release_add(route_done);
  }
  // ---- route: logits of token t for one block of experts, then (last CTA) its gate
  if (routing) {
    const int rb = blockIdx.x - 1;
    const int t = rb / d.nblk, b = rb - t * d.nblk;
    const uint16_t* xrow = d.x + (size_t)t * H;   // read by every warp: L1 after the first
    const int e0 = b * d.eb, e1 = min(E, e0 + d.eb);
    for (int e = e0 + warp; e < e1; e += NT / 32) {
      const uint16_t* wrow = d.wr + (size_t)e * H;
      float acc = 0.f;
      // the row's 16-byte chunks of this lane and the matching x chunks, kRouteChunks of
      // each in flight at once
      for (int h0 = lane * 8; h0 < H; h0 += 32 * 8 * kRouteChunks) {
        uint4 wq[kRouteChunks], xq[kRouteChunks];
#pragma unroll
        for (int c = 0; c < kRouteChunks; ++c) {
          const int h = h0 + c * 32 * 8;
          if (h < H) {
            wq[c] = __ldg(reinterpret_cast<const uint4*>(wrow + h));
            xq[c] = __ldg(reinterpret_cast<const uint4*>(xrow + h));
          }
        }
#pragma unroll
        for (int c = 0; c < kRouteChunks; ++c) {
          const int h = h0 + c * 32 * 8;
          if (h < H) {
            const uint4 q = xq[c];
            acc = fmaf(bf16lo(wq[c].x), bf16lo(q.x), acc);
            acc = fmaf(bf16hi(wq[c].x), bf16hi(q.x), acc);
            acc = fmaf(bf16lo(wq[c].y), bf16lo(q.y), acc);
            acc = fmaf(bf16hi(wq[c].y), bf16hi(q.y), acc);
            acc = fmaf(bf16lo(wq[c].z), bf16lo(q.z), acc);
            acc = fmaf(bf16hi(wq[c].z), bf16hi(q.z), acc);
            acc = fmaf(bf16lo(wq[c].w), bf16lo(q.w), acc);
            acc = fmaf(bf16hi(wq[c].w), bf16hi(q.w), acc);
          }
        }
      }
      acc = warp_sum(acc);
      if (lane == 0) d.z[(size_t)t * E + e] = acc + d.rb[e];
    }
    __syncthreads();
    if (fast) {
      // this CTA's logits (ordered before the release by the barrier)
      if (threadIdx.x == 0) release_add(route_done);
    } else if (threadIdx.x == 0) {
      // one acquire-release add: it releases this CTA's logits (ordered before it by the
      // barrier), and the token's last CTA acquires every other CTA's
      const uint32_t old = atom_add_acq_rel(ticket(t), 1u);
      flag_sh = old == (uint32_t)d.nblk - 1;
      if (flag_sh) *ticket(t) = 0u;
    }
    __syncthreads();
    if (!fast && flag_sh) {
      // the token's gate by the whole CTA (measured faster here than one warp's arg-max
      // rounds); scratch: this CTA's dynamic shared memory (substitution reads the layer's
      // table row: the plan changes it only after every gate)
      gate_token_cta<NT>(d.z, t, E, d.plan.p.k, d.plan.p.gating, d.plan.sc.ids, d.plan.sc.w, d.plan.sc.probs,
                         d.plan.sc.gap, d.plan.p.stats, *reinterpret_cast<GateCtaScratch*>(dsm),
                         p.aes_on ? p.lut + (size_t)l * E : nullptr, p.aes_alpha);
      __syncthreads();
      if (threadIdx.x == 0) release_add(route_done);
    }
    __syncthreads();
    if (d.local) take_snapshot();
  }

  // ---- plan (CTA 0, once every token is gated) while the other CTAs set up;
  // then every CTA runs the FFN once the plan is published
  FusedArgs fl = f;
  if (d.local) {
    fl.lp = &lp_sh;
    fl.cta0_plans = 1;
    fl.slots_ready = slots_ready;
    fl.host_layer = p.host_dev + (size_t)l * E * p.lay.rec;
    fl.lut_row = p.lut + (size_t)l * E;
    fl.rid_land0 = p.rid_land0;
    fl.S = p.S;
  }
  auto pre = [&]() -> bool {
    // every token gated, or (fast gate) every logit written, and the counters zeroed
    if (threadIdx.x == 0) {
      const uint32_t target = (uint32_t)(fast ? T * d.nblk : T) + 1u;
      flag_sh = wait_count(route_done, target, a.status, a.wait_ns) ? 1 : 0;
      if (!flag_sh) set_status(a.status, MOE_ERR_TIMEOUT);
    }
    __syncthreads();
    if (!flag_sh) {
      if (blockIdx.x == 0) cp_async_wait_all();   // the prestaged copies land before this CTA moves on
      return false;
    }
    // (thread 0's acquire of route_done and the barrier order every thread's reads of the routing)
    if (d.local) {
      // the step's entry lists, as the plan orders them: experts with tokens ascending,
      // then the shared expert; resident / copied by the table row at the step's start
      const int tk = T * p.k;
      // cnt_sh (zeroed at kernel start): 1 for every expert with tokens
      if (fast) {
        // the step's logits into shared memory, then one warp per token
        float* zs = reinterpret_cast<float*>(dsm + d.zoff);
        const int n = T * E;
        if ((E & 3) == 0) {
          for (int i = threadIdx.x; i < n / 4; i += NT)
            reinterpret_cast<float4*>(zs)[i] = __ldcg(reinterpret_cast<const float4*>(d.z) + i);
        } else {
          for (int i = threadIdx.x; i < n; i += NT) zs[i] = __ldcg(d.z + i);
        }
        __syncthreads();
        // CTA 0 also writes the routing outputs
        int32_t* gids = blockIdx.x == 0 ? d.plan.sc.ids : nullptr;
        if (E <= 128)
          gate_tokens_warps<4>(zs, T, E, p.k, p.gating, lp_sh.ids, lp_sh.w, gids, d.plan.sc.w, d.plan.sc.probs,
                               d.plan.sc.gap, p.stats, NT / 32, cnt_sh);
        else
          gate_tokens_warps<kMaxPerLane>(zs, T, E, p.k, p.gating, lp_sh.ids, lp_sh.w, gids, d.plan.sc.w,
                                         d.plan.sc.probs, d.plan.sc.gap, p.stats, NT / 32, cnt_sh);
        if (gids) __threadfence();   // the routing outputs, before the plan reads them
      } else {
        for (int i = threadIdx.x; i < tk; i += NT) {
          const int e = __ldcg(d.plan.sc.ids + i);
          lp_sh.ids[i] = e;
          lp_sh.w[i] = __ldcg(d.plan.sc.w + i);
          if ((unsigned)e < (unsigned)E) cnt_sh[e] = 1;
        }
      }
      __syncthreads();
      if (warp == 0) {
        // the step's entry lists, as the plan orders them: experts with tokens ascending,
        // then the shared expert; resident / copied by the table row at the step's start
        int pos_run = 0, nh_run = 0, nm_run = 0;
        const unsigned lower = (1u << lane) - 1u;
        for (int e0 = 0; e0 < E; e0 += 32) {
          const int e = e0 + lane;
          const bool has = e < E && cnt_sh[e] > 0;
          const int sl = has ? lut_snap[e] : -1;
          const bool hit = has && sl >= 0 && sl < p.S;
          const unsigned mhas = __ballot_sync(0xffffffffu, has), mhit = __ballot_sync(0xffffffffu, hit),
                         mmis = __ballot_sync(0xffffffffu, has && !hit);
          if (has) {
            const int pos = pos_run + __popc(mhas & lower);
            lp_sh.epos[e] = (int16_t)pos;
            lp_sh.expert[pos] = e;
            lp_sh.rid[pos] = hit ? sl : -1;
            if (hit) lp_sh.elist[0][nh_run + __popc(mhit & lower)] = pos;
            else lp_sh.elist[1][nm_run + __popc(mmis & lower)] = pos;
          }
          pos_run += __popc(mhas);
          nh_run += __popc(mhit);
          nm_run += __popc(mmis);
        }
        if (lane == 0) {
          if (p.shared) {
            lp_sh.expert[pos_run] = -1;
            lp_sh.rid[pos_run] = p.rid_shared0 + l;
            lp_sh.elist[0][nh_run++] = pos_run;
            ++pos_run;
          }
          lp_sh.n = pos_run;
          lp_sh.nh = nh_run;
          lp_sh.nm = nm_run;
          lp_sh.tk = tk;
          lp_sh.k = p.k;
        }
      }
      __syncthreads();
    }
    if (blockIdx.x == 0) {
      // the plan: history, victims, table, copy jobs, permutation (for the routing dump)
      plan_body<NT>(d.plan, dsm, true);
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) release_add(plan_done);
    }
    if (!d.local) {
      // the plan's work lists
      if (threadIdx.x == 0) {
        flag_sh = wait_count(plan_done, 1u, a.status, a.wait_ns) ? 1 : 0;
        if (!flag_sh) set_status(a.status, MOE_ERR_TIMEOUT);
      }
      __syncthreads();
      if (!flag_sh) return false;
      __threadfence();
    }
    __syncthreads();
    return true;
  };
  if constexpr (STREAM) {
    // The planner takes no streaming units: at one token the plan lasts about as long as
    // the FFN, and the FFN's phase barrier would wait for it (the other CTAs count G - 1
    // arrivals).  The streaming variant always runs on local lists.
    if (blockIdx.x == 0)
      pre();
    else
      stream_ffn(&map_w13, &map_w2, &map_h, a, fl, d.x, smem_raw, pre);
  } else {
    fused_ffn<WF>(&map_x, &map_h, &map_w13, &map_w2, a, fl, smem_raw, pre);
  }
  // ---- leave: the last CTA resets the counters for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t old = atomicAdd(exit_cnt, 1u);
    if (old == (uint32_t)G - 1) {
      *route_done = 0u;
      *plan_done = 0u;
      *snap_done = 0u;
      *slots_ready = 0u;
      for (int t = 0; t < kDecodeMaxT; ++t) *ticket(t) = 0u;
      *exit_cnt = 0u;
    }
  }
}

// ----------------------------------------------------------------- router GEMM (T > 32)
// z = X W_r^T for many tokens on the tensor cores (RapidMoE §2.1: the gate is a
// linear projection): unit = (128-token tile mt, K split sp), M = the tokens,
// N = the experts (padded to 16), fp32 accumulators in TMEM.  Each unit writes
// its partial [T][E] slice; the gate kernel adds the splits in order and the
// bias, so the logits are deterministic.
struct RouterArgs {
  int T, E, N, kb_h, nsp;
  float* part;          // [nsp][T][E]
  int32_t* status;
};

__global__ void __launch_bounds__(kThreads, 1)
tc_router_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, RouterArgs r) {
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t tfull_bar, drain_bar;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_sh;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = r.N;
  const uint32_t a_bytes = kTileBytes, b_bytes = (uint32_t)N * BK * 2;
  const uint32_t stage_bytes = (a_bytes + b_bytes + 1023) & ~1023u;
  const int S = min(kMaxStages, (int)(kSmemBudget / stage_bytes));
  uint32_t ncols = 32;
  while (ncols < (uint32_t)N) ncols <<= 1;
  const int mt = blockIdx.x / r.nsp, sp = blockIdx.x - mt * r.nsp;
  const int kb0 = sp * r.kb_h / r.nsp, kb1 = (sp + 1) * r.kb_h / r.nsp;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&tfull_bar, 1);
    mbar_init(&drain_bar, 1);
    abort_sh = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(&tmem_base_sh, ncols);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = tmem_base_sh;
  if (warp == 0) {
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = it % S;
        if (it >= (uint32_t)S && !mbar_wait(&empty_bar[s], ((it / S) - 1) & 1)) { ok = false; break; }
        uint8_t* st = smem + (size_t)s * stage_bytes;
        mbar_expect_tx(&full_bar[s], a_bytes + b_bytes);
        tma_load_3d(st, &map_x, &full_bar[s], kb * BK, mt * BM, 0);
        tma_load_3d(st + a_bytes, &map_w, &full_bar[s], kb * BK, 0, 0);
      }
      if (!ok) {
        set_status(r.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
      }
      const uint32_t issued = it;
      for (int s = 0; s < S; ++s) {
        if ((uint32_t)s < issued) {
          const uint32_t last = issued - 1 - ((issued - 1 - s) % S);
          mbar_wait(&full_bar[s], (last / S) & 1);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(N);
      uint32_t it = 0, acc = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb, ++it) {
        const int s = it % S;
        if (!mbar_wait(&full_bar[s], (it / S) & 1) || abort_sh) { ok = false; break; }
        fence_after();
        const uint32_t base = smem_u32(smem + (size_t)s * stage_bytes);
        const uint64_t da = desc_sw128(base), db = desc_sw128(base + a_bytes);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          mma_bf16(tmem, da + 2 * kk, db + 2 * kk, idesc, acc);
          acc = 1;
        }
        mma_commit(&empty_bar[s]);
      }
      if (!ok) {
        set_status(r.status, MOE_ERR_TIMEOUT);
        abort_sh = 1;
      }
      mma_commit(&tfull_bar);
      mbar_wait(&tfull_bar, 0);
    }
  } else {
    // epilogue: TMEM lane = token row of the tile
    const int q = warp & 3, row = q * 32 + lane;
    const int t = mt * BM + row;
    if (mbar_wait(&tfull_bar, 0) && !abort_sh) {
      fence_after();
      for (int c0 = 0; c0 < N; c0 += 16) {
        float d[16];
        tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + c0, d);
        if (t < r.T) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < r.E) r.part[((size_t)sp * r.T + t) * r.E + c0 + j] = d[j];
        }
      }
    } else {
      set_status(r.status, MOE_ERR_TIMEOUT);
    }
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1) tmem_dealloc(tmem, ncols);
}

// ----------------------------------------------------------------- gather / combine (T > 256)
// x rows in expert-sorted order: xp[r] = x[perm_tok[r]] (shared-expert rows included).
__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm_tok,
                                   const int32_t* __restrict__ n_rows, uint16_t* __restrict__ xp, int H) {
  const int rows = *n_rows;
  const int vec = H / 8;   // uint4 per row
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)perm_tok[r] * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)r * H);
    for (int c = threadIdx.x; c < vec; c += blockDim.x) dst[c] = src[c];
  }
}

// out[t] = sum over the token's k rows in ascending expert id of Y[row] (+ its shared-expert row).
__global__ void combine_rows_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ inv, int T, int k,
                                    int shared, uint16_t* __restrict__ out, int H) {
  const int t = blockIdx.x;
  if (t >= T) return;
  int rows[32];
  for (int j = 0; j < k; ++j) rows[j] = inv[t * k + j];
  for (int j = 1; j < k; ++j) {            // rows are grouped by ascending expert id
    const int v = rows[j];
    int q = j - 1;
    while (q >= 0 && rows[q] > v) { rows[q + 1] = rows[q]; --q; }
    rows[q + 1] = v;
  }
  for (int h2 = threadIdx.x; h2 < H / 2; h2 += blockDim.x) {
    float s0 = 0.f, s1 = 0.f;
    for (int j = 0; j < k; ++j) {
      const uint32_t v = reinterpret_cast<const uint32_t*>(y + (size_t)rows[j] * H)[h2];
      s0 += bf16lo(v);
      s1 += bf16hi(v);
    }
    if (shared) {
      const uint32_t v = reinterpret_cast<const uint32_t*>(y + (size_t)(T * k + t) * H)[h2];
      s0 += bf16lo(v);
      s1 += bf16hi(v);
    }
    reinterpret_cast<uint32_t*>(out + (size_t)t * H)[h2] =
        (uint32_t)f32_to_bf16_rn(s0) | ((uint32_t)f32_to_bf16_rn(s1) << 16);
  }
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


int stages_for(int nacc, int N) {
  const int stage = ((nacc * BM * BK * 2 + N * BK * 2) + 1023) & ~1023;
  int s = kSmemBudget / stage;
  if (s > kMaxStages) s = kMaxStages;
  return s;
}

template <int MODE, int WF>
int launch_mode(Args a, const CUtensorMap& mb, const CUtensorMap& mw, const Fp8Args& w8, cudaStream_t s) {
  constexpr int NACC = is_gate_up(MODE) ? 2 : 1;
  a.stages = stages_for(NACC, a.N);
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!configured[dev & 63]) {
    cudaFuncSetAttribute(tc_gather_kernel<MODE, WF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         kSmemBudget + 1024);
    configured[dev & 63] = true;
  }
  const size_t smem = (size_t)a.stages * (((NACC * BM * BK * 2 + a.N * BK * 2) + 1023) & ~1023) + 1024;
  tc_gather_kernel<MODE, WF><<<sm_count(), GatherShape<WF>::threads, smem, s>>>(mb, mw, a, w8);
  return 1;
}

}  // namespace tc

// uint8 tensor [d2][d1][d0] (d0 contiguous), byte strides s1, s2; box 64 x 128 x 1, no swizzle.
static bool make_map_u8_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                           uint64_t s2) {
  auto fn = tc::encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {s1, s2};
  cuuint32_t box[3] = {(cuuint32_t)tc::BK, (cuuint32_t)tc::BM, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tiled map without swizzle (the bf16 records are stored swizzled already), zero fill
// past the edges.  strides: the rank - 1 outer strides in bytes.
static bool make_map_nd(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                        const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = tc::encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(m, dt, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

TcMaps* tc_maps_create(const PoolDev& p, const Scratch& sc) {
  (void)sc;
  if (!tc::encode_fn()) return nullptr;
  TcMaps* m = new TcMaps();
  if (p.wdt == MOE_BF16) {
    // 16-row segments of 8 consecutive tiles: w13 tiles (kb, gate/up) of one 128-row block mt of
    // I, w2 tiles kb of one 128-row block of H, in any record
    const uint64_t kb_h = (p.H + 63) / 64, kb_i = (p.I + 63) / 64, mt_i = (p.I + 127) / 128, mt_h = (p.H + 127) / 128;
    const cuuint64_t d13[5] = {128, 128, 2 * kb_h, mt_i, (cuuint64_t)p.n_records};
    const cuuint64_t s13[4] = {128, tc::kTileBytes, 2 * kb_h * tc::kTileBytes, p.lay.rec};
    const cuuint32_t b13[5] = {128, tc::kStreamRows, 2 * tc::kStreamKb, 1, 1};
    const cuuint64_t d2[5] = {128, 128, kb_i, mt_h, (cuuint64_t)p.n_records};
    const cuuint64_t s2[4] = {128, tc::kTileBytes, kb_i * tc::kTileBytes, p.lay.rec};
    const cuuint32_t b2[5] = {128, tc::kStreamRows, tc::kStreamKb, 1, 1};
    m->stream = make_map_nd(&m->sw13, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, p.records + p.lay.off13, d13, s13, b13) &&
                make_map_nd(&m->sw2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, p.records + p.lay.off2, d2, s2, b2);
  }
  if (p.wdt == MOE_FP8_E4M3_B128) {
    m->fp8 = true;
    const uint64_t H = p.H, I = p.I, n = p.n_records, rec = p.lay.rec;
    if (!make_map_u8_3d(&m->w13, p.records + p.lay.off13, H, 2 * I, n, H, rec) ||
        !make_map_u8_3d(&m->w2, p.records + p.lay.off2, I, H, n, I, rec)) {
      delete m;
      return nullptr;
    }
  }
  return m;
}

// fp8 weights on the tensor cores: shapes whose tiles and scale rows the kernels cover
bool tc_fp8_ok(const PoolDev& p) {
  return p.H % 128 == 0 && p.I % 128 == 0 && p.H / 128 <= 64 && p.I / 128 <= 64 && p.lay.off2 % 16 == 0 &&
         p.lay.rec % 16 == 0;
}

// Landing records for the copied entries of one decode layer call with local lists:
// at most min(T k, E) entries, T <= kDecodeMaxT and T k <= kLocalMaxTk.
int decode_landing_records(const PoolDev& p, int max_tokens) {
  const bool tc = p.adt == MOE_BF16 && (p.wdt == MOE_BF16 || (p.wdt == MOE_FP8_E4M3_B128 && tc_fp8_ok(p)));
  if (!tc || p.E > kMaxE || p.k > tc::kLocalMaxTk) return 0;
  const int t = std::min(std::min(max_tokens, tc::kDecodeMaxT), tc::kLocalMaxTk / p.k);
  return std::min(p.E, t * p.k);
}

void tc_maps_destroy(TcMaps* m) { delete m; }

int tc_npad(int T) { return (T + 15) / 16 * 16; }

// Gate/up split partials: up to 8 splits of every (entry, 128-row tile), capped at 64 MB.
size_t tc_partial_floats(const PoolDev& p, int npad_max) {
  const size_t need = (size_t)(p.E + 1) * ((p.I + 127) / 128) * 8 * 2 * npad_max * tc::BM;
  return std::min(need, (size_t)16 << 20);
}

// Per-entry down partials: one split always fits; up to 4 within 64 MB.
size_t tc_dn_partial_floats(const PoolDev& p, int npad_max) {
  const size_t one = (size_t)(p.E + 1) * ((p.H + 127) / 128) * npad_max * tc::BM;
  return std::max(one, std::min(4 * one, (size_t)16 << 20));
}

// tile data of a record (the w13 tiles, then the w2 tiles), in 16-byte units
static uint32_t tile16(const PoolDev& p) {
  const size_t kb_i = (p.I + 63) / 64, mt_h = (p.H + 127) / 128;
  return (uint32_t)((p.lay.off2 + mt_h * kb_i * tc::kTileBytes) / 16);
}

// [gu_cnt: (E+1) * MT_I, padded to a 128-byte line][dn_done: a line of its own][hready: E+1]
// [jdone: E+1][jdone_w2: E+1, padded][next_unit: a line][next_miss: a line]
static int dn_done_index(const PoolDev& p) {
  const int mt_i = (p.I + 127) / 128;
  return ((p.E + 1) * mt_i + tc::kSyncLine - 1) / tc::kSyncLine * tc::kSyncLine;
}
static int next_unit_index(const PoolDev& p) {
  return (dn_done_index(p) + tc::kSyncLine + 3 * (p.E + 1) + tc::kSyncLine - 1) / tc::kSyncLine * tc::kSyncLine;
}
int tc_ffn_sync_ints(const PoolDev& p) { return next_unit_index(p) + 2 * tc::kSyncLine; }

// decode layer kernel counters: a line for each of kDsTicket named ones and for every token's ticket
int tc_dsync_ints() { return (tc::kDsTicket + tc::kDecodeMaxT) * tc::kSyncLine; }

static tc::Args tc_args(const PoolDev& p, const Scratch& sc, int T, int N) {
  tc::Args a;
  a.work = sc.work;
  a.n_work = sc.n_work;
  a.sel = nullptr;
  a.sel_count = nullptr;
  a.ntile0 = sc.ntile0;
  a.records = p.records;
  a.rec = p.lay.rec;
  a.off13 = p.lay.off13;
  a.off2 = p.lay.off2;
  a.T = T;
  a.N = N;
  a.H = p.H;
  a.I = p.I;
  a.num_sms = sm_count();
  a.stages = 1;
  a.wmat = sc.wmat;
  a.perm_w = sc.perm_w;
  a.hbuf = sc.hbuf;
  a.out = nullptr;
  a.partial = sc.partial;
  a.counters = sc.ffn_sync;
  a.status = p.status;
  a.wait_ns = p.wait_ns;
  a.max_split_units = 0;
  return a;
}

int gather_tile_rows(const PoolDev& p, int T) {
  const long long rows = (long long)T * p.k;   // routed rows of the call
  if (rows >= 192LL * p.E) return 256;
  // fp8 records are expanded to bf16 once per unit: smaller tiles would expand each weight
  // tile more often (measured slower), so they keep 128 rows
  return rows >= 96LL * p.E || p.wdt == MOE_FP8_E4M3_B128 ? 128 : 64;
}

// Gather path: xp = x rows by expert; h = gate/up per row; y = down per row; out = combine.
int launch_tc_gather(const PoolDev& p, const Scratch& sc, const TcMaps* m, int T, const void* x, void* out,
                     cudaStream_t s) {
  const int rows_max = T * p.k + (p.shared ? T : 0);
  tc::gather_rows_kernel<<<2 * sm_count(), 256, 0, s>>>(static_cast<const uint16_t*>(x), sc.perm_tok, sc.n_rows,
                                                         sc.xp, p.H);
  const int bn = gather_tile_rows(p, T);
  tc::Args a = tc_args(p, sc, T, bn);
  a.max_split_units = 0;
  a.hbuf = static_cast<uint16_t*>(sc.h);
  CUtensorMap xm;
  if (!tc::make_map_3d(&xm, sc.xp, (uint64_t)p.H, (uint64_t)rows_max, 1, (uint64_t)p.H * 2,
                       (uint64_t)p.H * 2 * rows_max, bn))
    return -1;
  tc::Fp8Args w8;
  w8.os13 = p.lay.offs13;
  w8.os2 = p.lay.offs2;
  w8.sc_h = p.H / 128;
  w8.sc_i = p.I / 128;
  const bool fp8 = m->fp8;
  int n = 1 + (fp8 ? tc::launch_mode<tc::kModeGateUpGather, tc::kWfFp8>(a, xm, m->w13, w8, s)
                   : tc::launch_mode<tc::kModeGateUpGather, tc::kWfBf16>(a, xm, xm, w8, s));
  tc::Args b = a;
  b.out = sc.y;
  CUtensorMap hm;
  if (!tc::make_map_3d(&hm, sc.h, (uint64_t)p.I, (uint64_t)rows_max, 1, (uint64_t)p.I * 2,
                       (uint64_t)p.I * 2 * rows_max, bn))
    return -1;
  n += fp8 ? tc::launch_mode<tc::kModeDownGather, tc::kWfFp8>(b, hm, m->w2, w8, s)
           : tc::launch_mode<tc::kModeDownGather, tc::kWfBf16>(b, hm, hm, w8, s);
  tc::combine_rows_kernel<<<T, 256, 0, s>>>(sc.y, sc.inv, T, p.k, p.shared, static_cast<uint16_t*>(out), p.H);
  return n + 1;
}


// Arguments of the fused FFN for a call of T tokens (dense token columns).
static bool fused_setup(const PoolDev& p, const Scratch& sc, int T, const void* x, void* out, tc::Args* ap,
                        tc::FusedArgs* fp, CUtensorMap* xm, CUtensorMap* hm) {
  const int N = tc_npad(T);
  tc::Args a = tc_args(p, sc, T, N);
  a.out = static_cast<uint16_t*>(out);
  a.stages = std::min<int>(tc::kMaxStages, (int)(tc::kSmemBudget / tc::fused_stage_bytes(N)));
  if (!tc::make_map_3d(xm, x, (uint64_t)p.H, (uint64_t)T, 1, (uint64_t)p.H * 2, (uint64_t)p.H * 2 * T, N))
    return false;
  const uint64_t I = p.I;
  if (!tc::make_map_3d(hm, sc.hbuf, I, (uint64_t)N, (uint64_t)p.E + 1, I * 2, (uint64_t)N * I * 2, N)) return false;
  tc::FusedArgs f;
  f.lp = nullptr;
  f.cta0_plans = 0;
  f.slots_ready = nullptr;
  f.host_layer = nullptr;
  f.lut_row = nullptr;
  f.rid_land0 = 0;
  f.S = p.S;
  f.jobs = sc.copies;
  f.n_jobs = sc.n_copy;
  // a bf16 record's tile data; an fp8 record whole (codes, then its scale tables)
  f.tile16 = p.wdt == MOE_FP8_E4M3_B128 ? (uint32_t)(p.lay.rec / 16) : tile16(p);
  f.part16 = p.wdt == MOE_FP8_E4M3_B128 ? f.tile16 : (uint32_t)(p.lay.off2 / 16);
  f.os13 = p.lay.offs13;
  f.os2 = p.lay.offs2;
  f.sc_h = p.H / 128;
  f.sc_i = p.I / 128;
  f.elist = sc.elist;
  f.ecount = sc.ecount;
  f.E1 = p.E + 1;
  // the partial buffers' capacities in (tile, split) partials of this call's columns (the
  // token count rounded up to 4), worked out here so that no kernel divides 64-bit sizes
  const size_t cols = (size_t)((T + 3) & ~3);
  f.gu_partial = sc.partial;
  f.gu_cap = (int)std::min<size_t>(sc.partial_floats / (2 * cols * tc::BM), (size_t)INT32_MAX);
  f.dn_partial = sc.dn_partial;
  f.dn_cap = (int)std::min<size_t>(sc.dn_partial_floats / (cols * tc::BM), (size_t)INT32_MAX);
  f.gu_cnt = sc.ffn_sync;
  f.dn_done = reinterpret_cast<uint32_t*>(sc.ffn_sync + dn_done_index(p));
  f.hready = f.dn_done + tc::kSyncLine;
  f.jdone = f.hready + (p.E + 1);
  f.jdone_w2 = f.jdone + (p.E + 1);
  f.next_unit = reinterpret_cast<uint32_t*>(sc.ffn_sync + next_unit_index(p));
  f.next_miss = f.next_unit + tc::kSyncLine;
  *ap = a;
  *fp = f;
  return true;
}

static size_t fused_smem(int N, int stages) { return (size_t)stages * tc::fused_stage_bytes(N) + 1024; }

// pdl: programmatic dependent launch — the grid may be launched while the previous kernel
// of the stream drains; the kernel waits for it (griddepcontrol.wait) before reading
// anything.  If the driver refuses the combination with a cooperative launch, the launch
// is repeated without it and later launches do not ask again.
static int launch_cooperative(const void* fn, int threads, size_t smem, cudaStream_t s, void** args,
                              bool pdl = false) {
  static bool pdl_refused = false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl && !pdl_refused ? 2 : 1;
  if (cudaLaunchKernelExC(&cfg, fn, args) == cudaSuccess) return 1;
  if (cfg.numAttrs == 2) {
    cudaGetLastError();
    pdl_refused = true;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelExC(&cfg, fn, args) == cudaSuccess) return 1;
  }
  return -2;
}

static void set_smem_attr_once(const void* fn, bool* configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (!configured[dev & 63]) {
    cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBudget + 1024);
    configured[dev & 63] = true;
  }
}

// Fused dense decode FFN (miss copies + gate/up + down + combine), one cooperative launch.
template <int WF>
static int launch_fused_decode_wf(const PoolDev& p, const Scratch& sc, const TcMaps* m, int T, const void* x,
                                  void* out, cudaStream_t s) {
  tc::Args a;
  tc::FusedArgs f;
  CUtensorMap xm, hm;
  if (!fused_setup(p, sc, T, x, out, &a, &f, &xm, &hm)) return -1;
  CUtensorMap w13 = WF == tc::kWfFp8 ? m->w13 : xm, w2 = WF == tc::kWfFp8 ? m->w2 : xm;
  static bool configured[64] = {};
  const void* fn = reinterpret_cast<const void*>(tc::tc_fused_decode_kernel<WF>);
  set_smem_attr_once(fn, configured);
  void* args[] = {&xm, &hm, &w13, &w2, &a, &f};
  return launch_cooperative(fn, tc::FusedShape<WF>::threads, fused_smem(a.N, a.stages), s, args);
}

int launch_tc_fused_decode(const PoolDev& p, const Scratch& sc, const TcMaps* m, int T, const void* x, void* out,
                           cudaStream_t s) {
  return m->fp8 ? launch_fused_decode_wf<tc::kWfFp8>(p, sc, m, T, x, out, s)
                : launch_fused_decode_wf<tc::kWfBf16>(p, sc, m, T, x, out, s);
}

// Shared memory of the decode layer kernel's plan (NT threads), 0 if it does not fit.
template <int NT>
static size_t decode_plan_smem(const PoolDev& p, int T, int* cap, int* rows) {
  const size_t b = plan_smem_bytes_nt<NT>(p, T, cap, rows, tc::kSmemBudget - 1024);
  return b + 16 <= (size_t)tc::kSmemBudget ? b + 16 : 0;
}

bool tc_decode_layer_ok(const PoolDev& p, const Scratch& sc, int T) {
  int cap = 0, rows = 0;
  const size_t psm = p.wdt == MOE_FP8_E4M3_B128
                         ? decode_plan_smem<tc::FusedShape<tc::kWfFp8>::threads>(p, T, &cap, &rows)
                         : decode_plan_smem<tc::FusedShape<tc::kWfBf16>::threads>(p, T, &cap, &rows);
  return sc.dsync != nullptr && p.adt == MOE_BF16 && T >= 1 && T <= tc::kDecodeMaxT && tc_npad(T) <= sc.npad_max &&
         p.H % 8 == 0 && (size_t)p.H * 2 + 16 <= (size_t)tc::kSmemBudget && psm > 0;
}

// Router, gate, plan and fused FFN of one decode call, one cooperative launch.
template <int WF, bool STREAM>
static int launch_decode_layer_impl(const PoolDev& p, const Scratch& sc, const TcMaps* m, int layer, int T,
                                    const void* x, const void* router_w, const float* router_b, void* out,
                                    cudaStream_t s);

template <int WF>
static int launch_decode_layer_wf(const PoolDev& p, const Scratch& sc, const TcMaps* m, int layer, int T,
                                  const void* x, const void* router_w, const float* router_b, void* out,
                                  cudaStream_t s) {
  // bf16 pools and one to four tokens: the CUDA-core streaming FFN
  if constexpr (WF == tc::kWfBf16) {
    if (m->stream && T <= tc::kStreamMaxT && T * p.k <= tc::kLocalMaxTk && p.E <= kMaxE &&
        std::min(T * p.k, p.E) <= p.n_land &&
        (size_t)(p.E + 1) * T * ((p.I + 63) / 64 * 64) * 4 <= (size_t)(p.E + 1) * sc.npad_max * p.I * 2 &&
        (size_t)T * ((p.H + 63) / 64 * 64) * 4 + 1024 + 2 * tc::kStreamStage <= (size_t)tc::kSmemBudget)
      return launch_decode_layer_impl<WF, true>(p, sc, m, layer, T, x, router_w, router_b, out, s);
  }
  return launch_decode_layer_impl<WF, false>(p, sc, m, layer, T, x, router_w, router_b, out, s);
}

template <int WF, bool STREAM>
static int launch_decode_layer_impl(const PoolDev& p, const Scratch& sc, const TcMaps* m, int layer, int T,
                                    const void* x, const void* router_w, const float* router_b, void* out,
                                    cudaStream_t s) {
  constexpr int NT = tc::DecodeShape<WF, STREAM>::threads;
  tc::Args a;
  tc::FusedArgs f;
  CUtensorMap xm, hm;
  if (!fused_setup(p, sc, T, x, out, &a, &f, &xm, &hm)) return -1;
  CUtensorMap w13 = WF == tc::kWfFp8 ? m->w13 : xm, w2 = WF == tc::kWfFp8 ? m->w2 : xm;
  tc::DecodeArgs d;
  d.x = static_cast<const uint16_t*>(x);
  d.wr = static_cast<const uint16_t*>(router_w) + (size_t)layer * p.E * p.H;
  d.rb = router_b + (size_t)layer * p.E;
  d.z = sc.logits;
  const int G = sm_count();
  int nblk = std::max(1, std::min((G - 1) / T, (p.E + 7) / 8));   // CTA 0 plans, the others route
  d.eb = (p.E + nblk - 1) / nblk;
  d.nblk = (p.E + d.eb - 1) / d.eb;
  PlanArgs& pa = d.plan;
  pa.p = p;
  pa.sc = sc;
  pa.layer = layer;
  pa.T = T;
  pa.flags = PLAN_HISTORY | PLAN_CACHE | PLAN_PERMUTE;
  pa.region = 0;
  pa.npad = a.N;
  pa.ids = sc.ids;
  pa.w = sc.w;
  pa.probs = sc.probs;
  // local lists: the copied entries (at most min(T k, E)) land in the landing records
  d.local = T * p.k <= tc::kLocalMaxTk && p.E <= kMaxE && std::min(T * p.k, p.E) <= p.n_land ? 1 : 0;
  pa.zero_sync = false;                      // CTA 0 zeroes the counters at kernel start
  pa.snap_wait = d.local ? sc.dsync + tc::kDsSnap * tc::kSyncLine : nullptr;
  pa.slots_flag = d.local ? sc.dsync + tc::kDsSlots * tc::kSyncLine : nullptr;
  pa.snap_target = (uint32_t)G;
  const size_t psm = decode_plan_smem<NT>(p, T, &pa.owner_cap, &pa.tok_rows);
  if (psm == 0) return -1;
  d.dsync = sc.dsync;
  size_t ffn_smem = fused_smem(a.N, a.stages);
  if (STREAM) {
    // h as [work position][T][Ip / 64][64] fp32 in the h scratch; boxes of 8 K blocks x T tokens
    const uint64_t kb_i = (p.I + 63) / 64, Ip = kb_i * 64;
    const cuuint64_t dh[4] = {64, kb_i, (cuuint64_t)T, (cuuint64_t)p.E + 1};
    const cuuint64_t sh[3] = {256, Ip * 4, (cuuint64_t)T * Ip * 4};
    const cuuint32_t bh[4] = {64, tc::kStreamKb, (cuuint32_t)T, 1};
    if (!make_map_nd(&hm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, sc.hbuf, dh, sh, bh)) return -1;
    w13 = m->sw13;
    w2 = m->sw2;
    // [x: T x H fp32, whole K blocks, 1 KB aligned][ring of 32 KB stages]
    const size_t xb = ((size_t)T * ((p.H + 63) / 64 * 64) * 4 + 1023) & ~(size_t)1023;
    a.stages = std::min<int>(tc::kMaxStages, (int)((tc::kSmemBudget - xb) / tc::kStreamStage));
    ffn_smem = 1024 + xb + (size_t)a.stages * tc::kStreamStage;
  }
  size_t smem = std::max(std::max(ffn_smem, psm + 1024), (size_t)p.H * 2 + 16 + 1024);
  // fast gate: the staged logits after the plan's shared memory (CTA 0 prestages the plan's
  // inputs while it gates)
  const size_t zoff = (psm + 15) & ~(size_t)15, zend = zoff + (size_t)T * p.E * 4 + 16;
  // (the streaming variant, one token: a gate per token on its own routing CTA measured
  // faster once a warp has to gate several tokens)
  d.fast = STREAM && d.local && !p.aes_on && T <= NT / 32 && zend <= (size_t)tc::kSmemBudget + 1024 ? 1 : 0;
  d.zoff = (int)zoff;
  if (d.fast) smem = std::max(smem, zend);
  static bool configured[64] = {};
  const void* fn = reinterpret_cast<const void*>(tc::tc_decode_layer_kernel<WF, STREAM>);
  set_smem_attr_once(fn, configured);
  void* args[] = {&xm, &hm, &w13, &w2, &a, &f, &d};
  return launch_cooperative(fn, NT, smem, s, args, /*pdl=*/true);
}

int launch_tc_decode_layer(const PoolDev& p, const Scratch& sc, const TcMaps* m, int layer, int T, const void* x,
                           const void* router_w, const float* router_b, void* out, cudaStream_t s) {
  return m->fp8 ? launch_decode_layer_wf<tc::kWfFp8>(p, sc, m, layer, T, x, router_w, router_b, out, s)
                : launch_decode_layer_wf<tc::kWfBf16>(p, sc, m, layer, T, x, router_w, router_b, out, s);
}


// Router on the tensor cores for T > 32 tokens: partial logits per K split.
bool tc_router_ok(const PoolDev& p, const Scratch& sc, int T) {
  return sc.rpart != nullptr && p.adt == MOE_BF16 && T > 32 && T <= sc.tmax && p.E <= 256 && p.H % 64 == 0;
}

int launch_tc_router(const PoolDev& p, const Scratch& sc, int layer, const void* x, int T, const void* router_w,
                     int* nsp_out, cudaStream_t s) {
  const int mtiles = (T + tc::BM - 1) / tc::BM;
  const int kb_h = p.H / tc::BK;
  const int G = sm_count();
  int nsp = std::max(1, std::min(std::min(kb_h, tc::kRouterMaxSplits), G / mtiles));
  tc::RouterArgs r;
  r.T = T;
  r.E = p.E;
  r.N = (p.E + 15) / 16 * 16;
  r.kb_h = kb_h;
  r.nsp = nsp;
  r.part = sc.rpart;
  r.status = p.status;
  CUtensorMap xm, wm;
  if (!tc::make_map_3d(&xm, x, (uint64_t)p.H, (uint64_t)T, 1, (uint64_t)p.H * 2, (uint64_t)p.H * 2 * T, tc::BM))
    return -1;
  const uint16_t* wr = static_cast<const uint16_t*>(router_w) + (size_t)layer * p.E * p.H;
  if (!tc::make_map_3d(&wm, wr, (uint64_t)p.H, (uint64_t)p.E, 1, (uint64_t)p.H * 2, (uint64_t)p.H * 2 * p.E, r.N))
    return -1;
  static bool configured[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!configured[dev & 63]) {
    cudaFuncSetAttribute(tc::tc_router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBudget + 1024);
    configured[dev & 63] = true;
  }
  const uint32_t stage = (tc::kTileBytes + (uint32_t)r.N * tc::BK * 2 + 1023) & ~1023u;
  const int S = std::min(tc::kMaxStages, (int)(tc::kSmemBudget / stage));
  tc::tc_router_kernel<<<mtiles * nsp, tc::kThreads, (size_t)S * stage + 1024, s>>>(xm, wm, r);
  *nsp_out = nsp;
  return 1;
}

}  // namespace moeslot
