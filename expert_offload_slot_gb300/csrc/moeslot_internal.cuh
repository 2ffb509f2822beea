// Internal declarations of libmoeslot: the pool object, the per-call work
// list shared between kernels, and small device helpers.  Nothing here is
// part of the C ABI (include/moeslot.h is).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moeslot.h"

namespace moeslot {

// One expert that this call must evaluate: its record (slot, staging region,
// host pool for a bypassed miss, or the shared expert), and its rows
// [row0, row0 + n) of the expert-sorted token order.
struct WorkEntry {
  const uint8_t* rec;
  int32_t row0;
  int32_t n;
  int32_t expert;   // routed expert id, or -1 for the shared expert
  int32_t rid;      // record index in the pool's record array
  int32_t crit;     // residual-split records: 1 = high precision (UMIA critical set)
};

// One device-started miss copy: record bytes from the mapped host pool to a slot.
struct CopyJob {
  const uint8_t* src;
  uint8_t* dst;
};

enum StatIdx {
  ST_STEPS = 0, ST_HITS, ST_MISSES, ST_BYPASS, ST_EVICT, ST_BYTES, ST_NEAR_TIES, ST_STAGED,
  ST_PF_ISSUED, ST_PF_COMMITTED, ST_PF_DEMANDED, ST_AES, ST_CRIT, ST_COUNT
};

// Asynchronous prefetch (SeqMoE "Mechanism"): the control region in pinned, mapped host
// memory.  The device writes requests and its position; the pool's host thread takes the
// requests in order, copies each record into its slot on a stream of its own, and then
// writes the request's tag into the pool's landed[slot] (device memory), in stream order.
constexpr int kPfRing = 256;              // requests the ring holds
constexpr int kPfMaxPending = 256;        // slots pending at once
constexpr int kPfMaxPerStep = 8;
struct PfReq {
  int32_t slot;
  int32_t flat;        // l * E + e
  uint32_t tag;
  int32_t pad;
};
struct PfCtl {
  volatile uint32_t head;     // requests written by the device
  volatile uint32_t tail;     // requests taken by the host thread
  volatile int32_t layer;     // GPU position: the last layer call that planned ...
  volatile int32_t step;      // ... and that layer's step
  volatile uint32_t demand;   // miss flag: bumped by every layer call with demand misses
  volatile uint32_t pad[3];
  PfReq req[kPfRing];
};

// Plan-kernel switches.
enum PlanFlags {
  PLAN_HISTORY = 1,    // a3: update routing history and eviction scores
  PLAN_CACHE = 2,      // a4/a5: table rewrite, misses, victims, copy list
  PLAN_PERMUTE = 4,    // a7 + work list
  PLAN_STAGED = 8,     // work list points into a staging region (identity table)
  PLAN_GATHER = 16     // also write inv, ntile0, n_rows for the gather path
};

struct Layout {
  size_t rec, off13, off2, offs13, offs2;
  size_t offr13, offh2, offsr13, offsh2;   // residual-split records: W^R, W^H_down and their scales
};

struct PoolDev {           // device-side pointers handed to kernels by value
  int32_t L, E, k, H, I, S, W;
  int32_t wdt, adt, gating, shared, policy;
  float lam, one_minus_lam, cw0, cw1, cw2, cw3;
  Layout lay;
  const uint8_t* host_dev;     // device-visible base of the mapped host pool
  // One record array: [S slots | n_bypass one-step records | n_land landing records |
  // 2E staging | L shared].
  uint8_t* records;
  int32_t n_bypass, rid_land0, n_land, rid_staging0, rid_shared0, n_records;
  uint8_t* slots;              // == records: the fixed base of the slot pool
  uint8_t* staging;            // records + rid_staging0 * rec, or null
  const uint8_t* shared_w;     // records + rid_shared0 * rec, or null
  int32_t* lut;                // [L*E]
  int32_t* owner;              // [S]
  uint32_t* tag;               // [S]
  int32_t* prot_epoch;         // [S]
  int32_t* epoch;              // [1]
  float* hist_s;               // [L][W][E]
  uint8_t* hist_sel;           // [L][W][E]
  float* ema;                  // [L][E]
  int32_t* last_sel;           // [L][E]
  float* score;                // [L][E]
  int32_t* step;               // [L]
  int32_t* status;             // sticky
  unsigned long long* stats;   // [ST_COUNT]
  uint64_t wait_ns;            // limit of a kernel's wait on another CTA (global-timer ns)
  // asynchronous prefetch: pf_used once it was ever enabled (pending slots are handled from
  // then on); pf_per_step > 0 while the plans issue requests
  int32_t pf_used, pf_per_step;
  int32_t* pf_expert;          // [S] l*E+e whose prefetch the slot holds (owner -2), or -1
  int32_t* pf_slot;            // [L*E] slot of the expert's pending prefetch, or -1
  uint32_t* pf_tag;            // [S] tag the slot's last prefetch was issued with
  const uint32_t* landed;      // [S] tag the host wrote back once that copy had landed
  int32_t* pf_list;            // [kPfMaxPending] pending slots, in request order
  int32_t* pf_n;               // [1]
  uint32_t* pf_head;           // [1] the device's count of requests written
  PfCtl* pf_ctl;               // control region, device view of the mapped host memory
  // approximate expert substitution (opt-in): the gates rewrite low-score misses
  int32_t aes_on;
  float aes_alpha;
  // UMIA (residual-split records): an expert of the step is critical when its token-averaged
  // router probability reaches (theta * beta[l]) * gamma (gamma of the decode or the prefill phase)
  float umia_theta, umia_gamma_decode, umia_gamma_prefill;
  const float* umia_beta;      // [L]
};

struct Scratch {
  int32_t tmax;       // max_tokens of the pool
  float* logits;      // [Tmax, E]
  float* probs;       // [Tmax, E]
  int32_t* ids;       // [Tmax, k]
  float* w;           // [Tmax, k]
  float* gap;         // [Tmax]
  int32_t* slots_out; // [Tmax, k]
  int32_t* perm_tok;  // [Tmax*k + Tmax]   token of each expert-sorted row
  float* perm_w;      // [Tmax*k + Tmax]   routing weight of each row
  int32_t* perm_ent;  // [Tmax*k]          flat entry t*k+j of each row
  int32_t* offs;      // [E+1]
  WorkEntry* work;    // [E+1]
  int32_t* n_work;    // [1]
  CopyJob* copies;    // [E+1]
  int32_t* n_copy;    // [1]
  int32_t* ticket;    // [1] last-CTA ticket of the fused routing kernel (self-resetting)
  void* h;            // [(Tmax*k + Tmax), I] act dtype
  // tensor-core decode path (dense token columns)
  int32_t npad_max;   // largest padded token count of that path (<= 256)
  float* wmat;        // [E+1][npad] routing weight of each token for each work entry (0 if not routed)
  uint16_t* hbuf;     // [E+1][npad][I] bf16: w * SiLU(g) * u
  float* partial;     // gate/up split partials
  size_t partial_floats;
  float* dn_partial;  // per-entry down partials of the fused decode kernel
  size_t dn_partial_floats;
  int32_t* ffn_sync;  // arrival counters and readiness flags of the fused decode kernel,
  int32_t n_ffn_sync; // zeroed by the plan kernel before every expert launch
  uint32_t* dsync;    // [tc_dsync_ints()] counters of the decode layer kernel (reset by its last CTA)
  float* rpart;       // [32][Tmax][E] K-split partial logits of the tensor-core router (Tmax > 32)
  int32_t* elist;     // [2][E+1]: work entries already resident / copied this step
  int32_t* ecount;    // [2]
  // tensor-core gather path (T > npad_max)
  int32_t* inv;       // [Tmax*k]   expert-sorted row of each flat entry t*k+j
  int32_t* ntile0;    // [E+2]      first token tile of each work entry (prefix; tiles of gather_tile_rows)
  int32_t* n_rows;    // [1]        expert-sorted rows of this call (T*k [+ T shared])
  uint16_t* xp;       // [(Tmax*k + Tmax), H] x rows in expert-sorted order
  uint16_t* y;        // [(Tmax*k + Tmax), H] per-row expert outputs
};

// ----------------------------------------------------------------- device helpers
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40);  // quiet NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// ----------------------------------------------------------------- launchers
// Each returns the number of kernels it launched (0 or more); errors from the
// launch itself surface through cudaGetLastError in the caller.
int launch_route_logits(const PoolDev& p, int layer, const void* x, int T, const void* router_w,
                        const float* router_b, float* logits, cudaStream_t s);
// logits [T][E], or (nsp > 0) nsp partial projections [nsp][T][E] summed in order plus bias
int launch_gate_topk(const PoolDev& p, const float* logits, int nsp, const float* bias, int T, int32_t* ids,
                     float* w, float* probs, float* gap, cudaStream_t s, const int32_t* aes_row = nullptr);
// one launch for router + gate when T and H are small enough (decode)
bool route_fused_ok(const PoolDev& p, int T);
int launch_route_gate_fused(const PoolDev& p, int layer, const void* x, int T, const void* router_w,
                            const float* router_b, const Scratch& sc, cudaStream_t s);
int launch_plan(const PoolDev& p, const Scratch& sc, int layer, int T, const int32_t* ids, const float* w,
                const float* probs, int flags, int region, int npad, cudaStream_t s);
// ctas: grid size (0: two CTAs per SM)
int launch_miss_copy(const PoolDev& p, const Scratch& sc, cudaStream_t s, int ctas = 0);
// part: -1 every entry; 0 / 1 (residual-split pools) the resident / the copied entries of the plan's lists
int launch_ffn_gate_up(const PoolDev& p, const Scratch& sc, int T, const void* x, cudaStream_t s, int part = -1);
int launch_ffn_down(const PoolDev& p, const Scratch& sc, int T, void* out, cudaStream_t s);

// tensor-core (tcgen05) expert path: bf16 weights, T <= 256 tokens
struct TcMaps;                      // host-side tensor maps of a pool (k_tc.cu)
TcMaps* tc_maps_create(const PoolDev& p, const Scratch& sc);
bool tc_fp8_ok(const PoolDev& p);   // fp8 pool shapes the tensor-core kernels take
int decode_landing_records(const PoolDev& p, int max_tokens);   // landing records the decode layer kernel needs
void tc_maps_destroy(TcMaps* m);
int tc_npad(int T);                 // padded token count (multiple of 16)
// scratch sizes for a pool whose dense path takes up to npad_max token columns
size_t tc_partial_floats(const PoolDev& p, int npad_max);      // Scratch::partial
size_t tc_dn_partial_floats(const PoolDev& p, int npad_max);   // Scratch::dn_partial
int tc_ffn_sync_ints(const PoolDev& p);                         // Scratch::ffn_sync
int tc_dsync_ints();                                          // Scratch::dsync
// Token rows per tile of the gather path for a call of T tokens, from its routed rows per
// expert on average: 256 from 192 (one weight tile then serves twice the tokens), 128 from
// 96 (and always for fp8 records), else 64 (fewer padding rows loaded and multiplied for
// experts with few tokens).
int gather_tile_rows(const PoolDev& p, int T);
int launch_tc_gather(const PoolDev& p, const Scratch& sc, const TcMaps* m, int T, const void* x, void* out,
                     cudaStream_t s);
int launch_tc_fused_decode(const PoolDev& p, const Scratch& sc, const TcMaps* m, int T, const void* x, void* out,
                           cudaStream_t s);
// router + gate + plan + fused FFN of a decode call in one cooperative launch (bf16, T <= 32)
bool tc_decode_layer_ok(const PoolDev& p, const Scratch& sc, int T);
// router projection on the tensor cores (bf16, T > 32): partial logits, *nsp_out splits
bool tc_router_ok(const PoolDev& p, const Scratch& sc, int T);
int launch_tc_router(const PoolDev& p, const Scratch& sc, int layer, const void* x, int T, const void* router_w,
                     int* nsp_out, cudaStream_t s);
int launch_tc_decode_layer(const PoolDev& p, const Scratch& sc, const TcMaps* m, int layer, int T, const void* x,
                           const void* router_w, const float* router_b, void* out, cudaStream_t s);
int launch_load_slot(const PoolDev& p, const Scratch& sc, int layer, int expert, int slot, cudaStream_t s);
int launch_rebuild_owner(const PoolDev& p, cudaStream_t s);

int sm_count();
moe_status set_last_error(moe_status st, const char* msg);   // text for moe_last_error()

}  // namespace moeslot
