// C ABI of libmoeslot (declared in include/moeslot.h): argument checks, the
// pool's device memory, and the per-layer launch sequence.
//
// Decode / slot-pool forward of one layer, all on the caller's stream:
//   route_logits -> gate_topk -> plan (history, table, victims, permutation)
//   -> miss_copy (device-started, from the mapped host pool) -> gate_up -> down
// Nothing in that sequence synchronises with the host or allocates, so it can
// be captured in a CUDA graph (SeqMoE "Mechanism": the graph never waits for
// the host to notice a miss).
//
// Staged prefill (MoE-CORE "Mechanism"): two staging regions, each one whole
// MoE layer; layer l reads region l mod 2; while it computes, the other region
// receives layer l+1 on the pool's copy stream (once layer l-1 has released it).
#include <atomic>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <string>
#include <thread>
#include <vector>

#include "moeslot_internal.cuh"

using namespace moeslot;

namespace moeslot {
int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}
}  // namespace moeslot

static thread_local std::string g_err;

static moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

namespace moeslot {
moe_status set_last_error(moe_status st, const char* msg) {
  g_err = msg;
  return st;
}
}  // namespace moeslot

#define CUDA_TRY(call)                                                                    \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess) return fail(MOE_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
  } while (0)

struct moe_pool {
  moe_config cfg;
  int device = 0;
  PoolDev d;
  Scratch sc;
  const uint8_t* host_pool = nullptr;
  size_t host_bytes = 0;
  const void* router_w = nullptr;
  const float* router_b = nullptr;
  int last_T = 0;
  bool last_gap_valid = false;
  cudaStream_t copy_stream = nullptr;
  cudaEvent_t ready[2] = {nullptr, nullptr};
  cudaEvent_t released[2] = {nullptr, nullptr};
  int staged_layer[2] = {-1, -1};
  int ready_pending = -1;             // region whose copy is the last on copy_stream, ready not yet recorded
  uint64_t staged_count = 0;
  uint64_t launches = 0;
  std::vector<void*> allocs;
  bool prof_on = false;
  std::vector<cudaEvent_t> prof_ev;   // [L][MOE_NUM_STAGES + 1]
  std::vector<uint8_t> prof_fused;    // [L]: the layer's last call ran as one decode layer kernel
  TcMaps* tc_maps = nullptr;          // tensor maps of the record array (bf16 weights)
  cudaStream_t side = nullptr;        // miss copies run here, beside gate/up over resident experts
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // asynchronous prefetch: the mapped control region, the host thread and its stream
  PfCtl* pf_ctl = nullptr;            // host view
  uint32_t* pf_tagbuf = nullptr;      // pinned: the tags the thread writes back, [kPfRing]
  cudaStream_t pf_stream = nullptr;
  std::thread pf_thread;
  std::atomic<bool> pf_stop{false};
  std::atomic<uint32_t> pf_taken{0};  // requests the thread has enqueued
  std::atomic<uint32_t> pf_corrupt{0};
  std::atomic<uint64_t> pf_bytes{0};
};

constexpr uint64_t kDefaultWaitNs = 1000000000ull;   // 1 s

static size_t elt_bytes(int dt) { return dt == MOE_F32 ? 4 : dt == MOE_BF16 ? 2 : 1; }   // RESPLIT: bytes of codes

static moe_status check_config(const moe_config* c) {
  if (!c) return fail(MOE_ERR_INVALID, "config is NULL");
  if (c->num_layers < 1) return fail(MOE_ERR_INVALID, "num_layers must be >= 1");
  if (c->num_experts < 1 || c->num_experts > 256) return fail(MOE_ERR_INVALID, "num_experts must be in 1..256");
  if (c->top_k < 1 || c->top_k > c->num_experts || c->top_k > 32)
    return fail(MOE_ERR_INVALID, "top_k must be in 1..min(num_experts, 32)");
  if (c->num_slots < 1) return fail(MOE_ERR_INVALID, "num_slots must be >= 1");
  if (c->window < 1 || c->window > 64) return fail(MOE_ERR_INVALID, "window must be in 1..64");
  if (c->max_tokens < 1) return fail(MOE_ERR_INVALID, "max_tokens must be >= 1");
  if (c->gating != MOE_GATE_SOFTMAX_RENORM && c->gating != MOE_GATE_SIGMOID_RENORM)
    return fail(MOE_ERR_INVALID, "unknown gating");
  if (c->evict_policy < MOE_EVICT_CORE || c->evict_policy > MOE_EVICT_LRU)
    return fail(MOE_ERR_INVALID, "unknown evict_policy");
  if (c->staging_regions != 0 && c->staging_regions != 2)
    return fail(MOE_ERR_INVALID, "staging_regions must be 0 or 2");
  if (c->has_shared_expert != 0 && c->has_shared_expert != 1)
    return fail(MOE_ERR_INVALID, "has_shared_expert must be 0 or 1");
  if (!(c->ema_decay >= 0.f && c->ema_decay <= 1.f)) return fail(MOE_ERR_INVALID, "ema_decay must be in [0, 1]");
  for (int i = 0; i < 4; ++i)
    if (!(c->core_w[i] >= 0.f)) return fail(MOE_ERR_INVALID, "core_w must be nonnegative");
  const bool ok_pair = (c->weight_dtype == MOE_F32 && c->act_dtype == MOE_F32) ||
                       (c->weight_dtype == MOE_BF16 && c->act_dtype == MOE_BF16) ||
                       (c->weight_dtype == MOE_FP8_E4M3_B128 && c->act_dtype == MOE_BF16) ||
                       (c->weight_dtype == MOE_RESPLIT_Q4R4 && c->act_dtype == MOE_BF16);
  if (!ok_pair)
    return fail(MOE_ERR_INVALID, "supported (weight, act) dtypes: (f32,f32), (bf16,bf16), (fp8,bf16), (resplit,bf16)");
  const int cw = (int)(16 / elt_bytes(c->weight_dtype));
  const int ca = (int)(16 / elt_bytes(c->act_dtype));
  const int q = cw > ca ? cw : ca;
  if (c->hidden < q || c->hidden % q || c->inter < q || c->inter % q)
    return fail(MOE_ERR_INVALID, "hidden and inter must be positive multiples of %d for these dtypes", q);
  if ((c->weight_dtype == MOE_FP8_E4M3_B128 || c->weight_dtype == MOE_RESPLIT_Q4R4) && (c->hidden % 128 || c->inter % 128))
    return fail(MOE_ERR_INVALID, "fp8 and residual-split weights need hidden and inter multiples of 128");
  return MOE_OK;
}

static Layout layout_of(const moe_config* c) {
  Layout L{};
  const size_t eb = elt_bytes(c->weight_dtype);
  const size_t H = c->hidden, I = c->inter;
  if (c->weight_dtype == MOE_RESPLIT_Q4R4) {
    // [q13 | r13 | l2 | h2 | sq13 | sr13 | sl2 | sh2]
    const size_t IH = I * H, s13 = 2 * I * (H / 128) * 4, s2 = H * (I / 128) * 4;
    L.off13 = 0;
    L.offr13 = IH;
    L.off2 = 2 * IH;
    L.offh2 = 2 * IH + IH / 2;
    L.offs13 = 3 * IH + IH / 2;
    L.offsr13 = L.offs13 + s13;
    L.offs2 = L.offsr13 + s13;
    L.offsh2 = L.offs2 + s2;
    L.rec = (L.offsh2 + s2 + 4095) / 4096 * 4096;
    return L;
  }
  if (c->weight_dtype == MOE_BF16) {
    // 128 x 64 tiles in 128-byte-swizzled order: w13 [I/128][H/64][gate, up], w2 [H/128][I/64]
    const size_t mt_i = (I + 127) / 128, kb_h = (H + 63) / 64, mt_h = (H + 127) / 128, kb_i = (I + 63) / 64;
    const size_t w13 = 2 * mt_i * kb_h * 16384, w2 = mt_h * kb_i * 16384;
    L.off13 = 0;
    L.off2 = w13;
    L.offs13 = L.offs2 = w13 + w2;
    L.rec = (w13 + w2 + 4095) / 4096 * 4096;
    return L;
  }
  const size_t w13 = 2 * I * H * eb, w2 = H * I * eb;
  size_t s13 = 0, s2 = 0;
  if (c->weight_dtype == MOE_FP8_E4M3_B128) {
    s13 = (2 * I / 128) * (H / 128) * 4;
    s2 = (H / 128) * (I / 128) * 4;
  }
  L.off13 = 0;
  L.off2 = w13;
  L.offs13 = w13 + w2;
  L.offs2 = w13 + w2 + s13;
  const size_t raw = w13 + w2 + s13 + s2;
  L.rec = (raw + 4095) / 4096 * 4096;
  return L;
}

// The API functions below were declared extern "C" by moeslot.h, so their
// definitions keep C linkage.

MOE_API const char* moe_last_error(void) { return g_err.c_str(); }

MOE_API moe_status moe_expert_layout(const moe_config* cfg, size_t* w13_off, size_t* w2_off, size_t* s13_off,
                                     size_t* s2_off, size_t* record_bytes) {
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const Layout L = layout_of(cfg);
  if (w13_off) *w13_off = L.off13;
  if (w2_off) *w2_off = L.off2;
  if (s13_off) *s13_off = L.offs13;
  if (s2_off) *s2_off = L.offs2;
  if (record_bytes) *record_bytes = L.rec;
  return MOE_OK;
}

MOE_API moe_status moe_host_alloc(size_t bytes, void** out) {
  if (!out || bytes == 0) return fail(MOE_ERR_INVALID, "moe_host_alloc: bad arguments");
  *out = nullptr;
  cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocMapped | cudaHostAllocPortable);
  if (e != cudaSuccess) {
    *out = nullptr;
    return fail(MOE_ERR_OOM, "cudaHostAlloc(%zu): %s", bytes, cudaGetErrorString(e));
  }
  return MOE_OK;
}

MOE_API moe_status moe_host_free(void* p) {
  if (!p) return MOE_OK;
  CUDA_TRY(cudaFreeHost(p));
  return MOE_OK;
}

static moe_status pool_alloc(moe_pool* P, void** out, size_t bytes) {
  *out = nullptr;
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(out, bytes);
  if (e != cudaSuccess) {
    *out = nullptr;
    cudaGetLastError();
    return fail(MOE_ERR_OOM, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
  }
  P->allocs.push_back(*out);
  return MOE_OK;
}

template <typename T>
static moe_status palloc(moe_pool* P, T** out, size_t count, int fill_byte) {
  void* v = nullptr;
  moe_status st = pool_alloc(P, &v, count * sizeof(T));
  if (st != MOE_OK) return st;
  *out = static_cast<T*>(v);
  if (cudaMemset(v, fill_byte, count * sizeof(T)) != cudaSuccess)
    return fail(MOE_ERR_CUDA, "cudaMemset failed");
  return MOE_OK;
}

static void prefetch_stop(moe_pool* P) {
  if (P->pf_thread.joinable()) {
    P->pf_stop.store(true);
    P->pf_thread.join();
  }
}

static void pool_free_all(moe_pool* P) {
  prefetch_stop(P);
  if (P->pf_stream) cudaStreamSynchronize(P->pf_stream);
  if (P->pf_stream) cudaStreamDestroy(P->pf_stream);
  if (P->pf_ctl) cudaFreeHost(P->pf_ctl);
  if (P->pf_tagbuf) cudaFreeHost(P->pf_tagbuf);
  if (P->tc_maps) tc_maps_destroy(P->tc_maps);
  P->tc_maps = nullptr;
  for (void* p : P->allocs) cudaFree(p);
  P->allocs.clear();
  for (cudaEvent_t e : P->prof_ev) cudaEventDestroy(e);
  P->prof_ev.clear();
  for (int r = 0; r < 2; ++r) {
    if (P->ready[r]) cudaEventDestroy(P->ready[r]);
    if (P->released[r]) cudaEventDestroy(P->released[r]);
  }
  if (P->copy_stream) cudaStreamDestroy(P->copy_stream);
  if (P->side) cudaStreamDestroy(P->side);
  if (P->ev_fork) cudaEventDestroy(P->ev_fork);
  if (P->ev_join) cudaEventDestroy(P->ev_join);
}

MOE_API moe_status moe_pool_create(const moe_config* cfg, const void* host_pool, size_t host_pool_bytes,
                                   const void* router_w, const float* router_b, const void* shared_w, int device,
                                   moe_pool** out) {
  if (!out) return fail(MOE_ERR_INVALID, "out is NULL");
  *out = nullptr;
  moe_status st = check_config(cfg);
  if (st != MOE_OK) return st;
  const Layout lay = layout_of(cfg);
  const size_t L = cfg->num_layers, E = cfg->num_experts;
  if (!host_pool) return fail(MOE_ERR_INVALID, "host_pool is NULL");
  if ((E + 1) * (lay.rec / 16) >= (1ull << 32))
    return fail(MOE_ERR_INVALID, "expert record too large for the copy kernel's 32-bit index space");
  if (host_pool_bytes < L * E * lay.rec)
    return fail(MOE_ERR_INVALID, "host_pool_bytes %zu < L*E*record_bytes %zu", host_pool_bytes, L * E * lay.rec);
  if (!router_w || !router_b) return fail(MOE_ERR_INVALID, "router weights are NULL");
  if ((reinterpret_cast<uintptr_t>(router_w) & 15) || (reinterpret_cast<uintptr_t>(router_b) & 3))
    return fail(MOE_ERR_INVALID, "router_w must be 16-byte aligned and router_b 4-byte aligned");
  if (cfg->has_shared_expert && !shared_w) return fail(MOE_ERR_INVALID, "shared_w is NULL but has_shared_expert");
  int ndev = 0;
  CUDA_TRY(cudaGetDeviceCount(&ndev));
  if (device < 0 || device >= ndev) return fail(MOE_ERR_INVALID, "device %d out of range", device);
  CUDA_TRY(cudaSetDevice(device));

  // The pool must be page-locked host memory: the staging copies are
  // asynchronous DMA and the miss kernel reads it through its mapped address.
  // (On a Grace host pageable memory is device-reachable too, so the memory
  // type is checked explicitly.)
  cudaPointerAttributes attr;
  void* hdev = nullptr;
  if (cudaPointerGetAttributes(&attr, host_pool) != cudaSuccess || attr.type != cudaMemoryTypeHost ||
      cudaHostGetDevicePointer(&hdev, const_cast<void*>(host_pool), 0) != cudaSuccess || !hdev) {
    cudaGetLastError();
    return fail(MOE_ERR_INVALID, "host_pool is not pinned, mapped host memory");
  }

  moe_pool* P = new moe_pool();
  P->cfg = *cfg;
  P->device = device;
  P->host_pool = static_cast<const uint8_t*>(host_pool);
  P->host_bytes = host_pool_bytes;
  P->router_w = router_w;
  P->router_b = router_b;
  PoolDev& d = P->d;
  d.L = cfg->num_layers; d.E = cfg->num_experts; d.k = cfg->top_k; d.H = cfg->hidden; d.I = cfg->inter;
  d.S = cfg->num_slots; d.W = cfg->window;
  d.wdt = cfg->weight_dtype; d.adt = cfg->act_dtype; d.gating = cfg->gating;
  d.shared = cfg->has_shared_expert; d.policy = cfg->evict_policy;
  d.lam = cfg->ema_decay;
  d.one_minus_lam = 1.0f - cfg->ema_decay;
  d.cw0 = cfg->core_w[0]; d.cw1 = cfg->core_w[1]; d.cw2 = cfg->core_w[2]; d.cw3 = cfg->core_w[3];
  d.lay = lay;
  d.host_dev = static_cast<const uint8_t*>(hdev);
  d.wait_ns = kDefaultWaitNs;

  const size_t S = d.S, W = d.W, Tm = cfg->max_tokens, k = d.k;
  const size_t rows = Tm * k + Tm;
  const size_t asz = elt_bytes(cfg->act_dtype);
#define PA(ptr, n, fill)                         \
  do {                                           \
    st = palloc(P, &(ptr), (n), (fill));         \
    if (st != MOE_OK) goto fail_out;             \
  } while (0)
  {
    // one record array: [S slots | one-step records for misses that get no slot |
    // landing records of the decode layer kernel | 2E staging | L shared]
    const long long need = std::min<long long>((long long)E, (long long)Tm * (long long)k) - (long long)S;
    d.n_bypass = need > 0 ? (int)need : 0;
    d.rid_land0 = (int)S + d.n_bypass;
    d.n_land = decode_landing_records(d, cfg->max_tokens);
    d.rid_staging0 = d.rid_land0 + d.n_land;
    const int n_stage = cfg->staging_regions == 2 ? 2 * (int)E : 0;
    d.rid_shared0 = d.rid_staging0 + n_stage;
    d.n_records = d.rid_shared0 + (cfg->has_shared_expert ? (int)L : 0);
    PA(d.records, (size_t)d.n_records * lay.rec, 0);
    d.slots = d.records;
    d.staging = n_stage ? d.records + (size_t)d.rid_staging0 * lay.rec : nullptr;
    d.shared_w = cfg->has_shared_expert ? d.records + (size_t)d.rid_shared0 * lay.rec : nullptr;
    if (cfg->has_shared_expert &&
        cudaMemcpy(const_cast<uint8_t*>(d.shared_w), shared_w, L * lay.rec, cudaMemcpyDefault) != cudaSuccess) {
      st = fail(MOE_ERR_CUDA, "copying the shared experts failed");
      goto fail_out;
    }
  }
  PA(d.lut, L * E, 0xff);
  PA(d.owner, S, 0xff);
  PA(d.tag, S, 0);
  PA(d.prot_epoch, S, 0);
  PA(d.epoch, 1, 0);
  PA(d.hist_s, L * W * E, 0);
  PA(d.hist_sel, L * W * E, 0);
  PA(d.ema, L * E, 0);
  PA(d.last_sel, L * E, 0xff);
  PA(d.score, L * E, 0);
  PA(d.step, L, 0);
  PA(d.status, 1, 0);
  PA(d.stats, ST_COUNT, 0);
  {
    int32_t* pe = nullptr;
    uint32_t* ld = nullptr;
    PA(pe, S, 0xff);
    d.pf_expert = pe;
    PA(d.pf_slot, L * E, 0xff);
    PA(d.pf_tag, S, 0);
    PA(ld, S, 0);
    d.landed = ld;
    PA(d.pf_list, kPfMaxPending, 0);
    PA(d.pf_n, 1, 0);
    PA(d.pf_head, 1, 0);
    float* ub = nullptr;
    PA(ub, L, 0);
    std::vector<float> ones(L, 1.f);
    if (cudaMemcpy(ub, ones.data(), sizeof(float) * L, cudaMemcpyHostToDevice) != cudaSuccess) {
      st = fail(MOE_ERR_CUDA, "initialising the UMIA coefficients failed");
      goto fail_out;
    }
    d.umia_beta = ub;
    d.umia_theta = 0.f;
    d.umia_gamma_decode = d.umia_gamma_prefill = 1.f;
  }
  P->sc.tmax = (int32_t)Tm;
  PA(P->sc.logits, Tm * E, 0);
  PA(P->sc.probs, Tm * E, 0);
  PA(P->sc.ids, Tm * k, 0);
  PA(P->sc.w, Tm * k, 0);
  PA(P->sc.gap, Tm, 0);
  PA(P->sc.slots_out, Tm * k, 0);
  PA(P->sc.perm_tok, rows, 0);
  PA(P->sc.perm_w, rows, 0);
  PA(P->sc.perm_ent, Tm * k, 0);
  PA(P->sc.offs, E + 1, 0);
  PA(P->sc.work, E + 1, 0);
  PA(P->sc.n_work, 1, 0);
  PA(P->sc.copies, E + 1, 0);
  PA(P->sc.n_copy, 1, 0);
  PA(P->sc.ticket, 1, 0);
  PA(P->sc.elist, 2 * (E + 1), 0);     // written by the plan kernel for every pool
  PA(P->sc.ecount, 2, 0);
  {
    uint8_t* hb = nullptr;
    PA(hb, rows * (size_t)d.I * asz, 0);
    P->sc.h = hb;
  }
  if (cfg->weight_dtype == MOE_BF16 ||
      (cfg->weight_dtype == MOE_FP8_E4M3_B128 && cfg->act_dtype == MOE_BF16 && tc_fp8_ok(d))) {
    // tensor-core expert path (T <= 256): dense routing weights, h buffer, split partials
    const int np = std::min(tc_npad((int)Tm), 256);
    P->sc.npad_max = np;
    PA(P->sc.wmat, (E + 1) * (size_t)np, 0);
    PA(P->sc.hbuf, (E + 1) * (size_t)np * d.I, 0);
    P->sc.partial_floats = tc_partial_floats(d, np);
    PA(P->sc.partial, P->sc.partial_floats, 0);
    P->sc.dn_partial_floats = tc_dn_partial_floats(d, np);
    PA(P->sc.dn_partial, P->sc.dn_partial_floats, 0);
    P->sc.n_ffn_sync = tc_ffn_sync_ints(d);
    PA(P->sc.ffn_sync, P->sc.n_ffn_sync, 0);
    PA(P->sc.dsync, tc_dsync_ints(), 0);
    if (Tm > 32 && cfg->act_dtype == MOE_BF16) PA(P->sc.rpart, (size_t)32 * Tm * E, 0);
    if ((size_t)tc_npad((int)Tm) > (size_t)np) {
      // gather path for calls with more tokens than the dense path takes
      PA(P->sc.inv, Tm * k, 0);
      PA(P->sc.ntile0, E + 2, 0);
      PA(P->sc.n_rows, 1, 0);
      PA(P->sc.xp, rows * (size_t)d.H, 0);
      PA(P->sc.y, rows * (size_t)d.H, 0);
    }
    P->tc_maps = tc_maps_create(d, P->sc);
    if (!P->tc_maps) {
      st = fail(MOE_ERR_CUDA, "creating the tensor maps of the record array failed");
      goto fail_out;
    }
  } else {
    P->sc.npad_max = 0;
  }
#undef PA
  if (cudaStreamCreateWithFlags(&P->side, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&P->ev_fork, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&P->ev_join, cudaEventDisableTiming) != cudaSuccess) {
    st = fail(MOE_ERR_CUDA, "creating the side stream failed");
    goto fail_out;
  }
  if (cudaStreamCreateWithFlags(&P->copy_stream, cudaStreamNonBlocking) != cudaSuccess) {
    st = fail(MOE_ERR_CUDA, "cudaStreamCreate failed");
    goto fail_out;
  }
  for (int r = 0; r < 2; ++r) {
    if (cudaEventCreateWithFlags(&P->ready[r], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&P->released[r], cudaEventDisableTiming) != cudaSuccess) {
      st = fail(MOE_ERR_CUDA, "cudaEventCreate failed");
      goto fail_out;
    }
    cudaEventRecord(P->ready[r], P->copy_stream);
    cudaEventRecord(P->released[r], P->copy_stream);
  }
  if (cudaDeviceSynchronize() != cudaSuccess) {
    st = fail(MOE_ERR_CUDA, "pool initialisation failed: %s", cudaGetErrorString(cudaGetLastError()));
    goto fail_out;
  }
  *out = P;
  return MOE_OK;
fail_out:
  pool_free_all(P);
  delete P;
  return st;
}

MOE_API moe_status moe_pool_destroy(moe_pool* P) {
  if (!P) return MOE_OK;
  cudaSetDevice(P->device);
  cudaDeviceSynchronize();
  pool_free_all(P);
  delete P;
  return MOE_OK;
}

MOE_API moe_status moe_set_lut(moe_pool* P, const int32_t* lut_host, void* stream) {
  if (!P || !lut_host) return fail(MOE_ERR_INVALID, "moe_set_lut: NULL argument");
  const int L = P->d.L, E = P->d.E, S = P->d.S;
  std::vector<int32_t> owner(S, -1);
  for (int i = 0; i < L * E; ++i) {
    const int s = lut_host[i];
    if (s < -1 || s >= S) return fail(MOE_ERR_INVALID, "lut[%d] = %d is not a slot id or -1", i, s);
    if (s >= 0) {
      if (owner[s] >= 0) return fail(MOE_ERR_INVALID, "slot %d assigned twice", s);
      owner[s] = i;
    }
  }
  CUDA_TRY(cudaSetDevice(P->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CUDA_TRY(cudaStreamSynchronize(s));
  if (P->d.pf_used) {
    // every prefetch copy lands before the slots are refilled; no slot stays pending
    moe_status st = moe_prefetch_drain(P);
    if (st != MOE_OK) return st;
    CUDA_TRY(cudaMemset(P->d.pf_expert, 0xff, sizeof(int32_t) * S));
    CUDA_TRY(cudaMemset(P->d.pf_slot, 0xff, sizeof(int32_t) * L * E));
    CUDA_TRY(cudaMemset(P->d.pf_n, 0, sizeof(int32_t)));
    CUDA_TRY(cudaMemcpy(const_cast<uint32_t*>(P->d.landed), P->d.pf_tag, sizeof(uint32_t) * S,
                        cudaMemcpyDeviceToDevice));
  }
  CUDA_TRY(cudaMemcpy(P->d.lut, lut_host, sizeof(int32_t) * L * E, cudaMemcpyHostToDevice));
  CUDA_TRY(cudaMemcpy(P->d.owner, owner.data(), sizeof(int32_t) * S, cudaMemcpyHostToDevice));
  P->launches += launch_rebuild_owner(P->d, s);
  const size_t rec = P->d.lay.rec;
  for (int sl = 0; sl < S; ++sl) {
    if (owner[sl] < 0) continue;
    CUDA_TRY(cudaMemcpyAsync(P->d.records + (size_t)sl * rec, P->host_pool + (size_t)owner[sl] * rec, rec,
                             cudaMemcpyHostToDevice, s));
  }
  CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

MOE_API moe_status moe_load_slot(moe_pool* P, int32_t layer, int32_t expert, int32_t slot, void* stream) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  if (layer < 0 || layer >= P->d.L || expert < 0 || expert >= P->d.E || slot < 0 || slot >= P->d.S)
    return fail(MOE_ERR_INVALID, "moe_load_slot: layer/expert/slot out of range");
  if (P->d.pf_used) return fail(MOE_ERR_INVALID, "moe_load_slot: not available on a pool that has used prefetch");
  CUDA_TRY(cudaSetDevice(P->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  P->launches += launch_load_slot(P->d, P->sc, layer, expert, slot, s);
  P->launches += launch_miss_copy(P->d, P->sc, s);
  CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

// Staging (MoE-CORE's two prefill regions): a layer's records are copied into a
// region on the pool's copy stream once the layer that used the region last has
// released it.  The copy's `ready` event is recorded only when its layer is about
// to run (mark_ready), not right after the copy is issued: where the copy stream
// and the caller's stream share one hardware work queue, a record issued right
// after a long copy holds back everything the caller enqueues behind it (the next
// layer's kernels) until that copy ends, which serialises copies and compute.  The
// record still comes right after its copy in the copy stream's order, because a
// pending record is made before any later copy is issued.
static void mark_ready(moe_pool* P, int r) {
  if (P->ready_pending == r) {
    cudaEventRecord(P->ready[r], P->copy_stream);
    P->ready_pending = -1;
  }
}

static void stage_layer(moe_pool* P, int layer, int r) {
  const size_t bytes = (size_t)P->d.E * P->d.lay.rec;
  if (P->ready_pending >= 0) mark_ready(P, P->ready_pending);
  cudaStreamWaitEvent(P->copy_stream, P->released[r], 0);
  cudaMemcpyAsync(P->d.staging + (size_t)r * bytes, P->host_pool + (size_t)layer * bytes, bytes,
                  cudaMemcpyHostToDevice, P->copy_stream);
  P->ready_pending = r;
  P->staged_layer[r] = layer;
  P->staged_count += 1;
}

// CTAs of a residual-split call's miss copy: enough host reads in flight for the link (32 x 512
// threads x 8 x 16 B = 2 MB), leaving the other SMs to the gate/up kernel running beside it
constexpr int kSideCopyCtas = 32;

static moe_status run_layer(moe_pool* P, int layer, const void* x, int T, void* out, bool staged,
                            const int32_t* ids_in, const float* w_in, const float* probs_in, cudaStream_t s) {
  PoolDev& d = P->d;
  Scratch& sc = P->sc;
  const int32_t* ids = ids_in ? ids_in : sc.ids;
  const float* w = w_in ? w_in : sc.w;
  const float* probs = probs_in ? probs_in : sc.probs;
  int region = 0;
  if (staged) {
    // this layer's region (copied during the previous layer's call, else now), then the next
    // layer's copy into the other region, issued before this layer's kernels so that it runs
    // beside them
    region = layer % 2;
    if (P->staged_layer[region] != layer) stage_layer(P, layer, region);
    mark_ready(P, region);
    if (layer + 1 < d.L && P->staged_layer[1 - region] != layer + 1) stage_layer(P, layer + 1, 1 - region);
    CUDA_TRY(cudaStreamWaitEvent(s, P->ready[region], 0));
  }
  const int NB = MOE_NUM_STAGES + 1;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (P->prof_on) cudaStreamIsCapturing(s, &cap);
  auto mark = [&](int i) {
    if (!P->prof_on) return;
    // inside a stream capture an event needs the external flag to become an event-record node
    if (cap == cudaStreamCaptureStatusActive)
      cudaEventRecordWithFlags(P->prof_ev[(size_t)layer * NB + i], s, cudaEventRecordExternal);
    else
      cudaEventRecord(P->prof_ev[(size_t)layer * NB + i], s);
  };
  mark(0);
  const bool tc = P->tc_maps != nullptr;                 // bf16 or fp8 weights: tensor-core path
  const bool use_tc = tc && tc_npad(T) <= sc.npad_max;   // dense token columns
  const bool gather = tc && !use_tc;                     // expert-grouped token tiles
  if (use_tc && !ids_in && !staged && tc_decode_layer_ok(d, sc, T)) {
    // router, gate, plan, miss copies, gate/up, down and combine in one cooperative kernel;
    // its profile is one interval (mark 0 to mark 4)
    if (P->prof_on) P->prof_fused[layer] = 1;
    const int n = launch_tc_decode_layer(d, sc, P->tc_maps, layer, T, x, P->router_w, P->router_b, out, s);
    if (n == -1) return fail(MOE_ERR_INVALID, "x must be 16-byte aligned for the tensor-core path");
    if (n < 0) return fail(MOE_ERR_CUDA, "cooperative launch failed: %s", cudaGetErrorString(cudaGetLastError()));
    P->launches += n;
    mark(4);
    CUDA_TRY(cudaGetLastError());
    P->last_T = T;
    P->last_gap_valid = true;
    return MOE_OK;
  }
  if (P->prof_on) P->prof_fused[layer] = 0;
  if (!ids_in) {
    if (route_fused_ok(d, T)) {
      P->launches += launch_route_gate_fused(d, layer, x, T, P->router_w, P->router_b, sc, s);
    } else if (tc_router_ok(d, sc, T)) {
      int nsp = 0;
      const int n = launch_tc_router(d, sc, layer, x, T, P->router_w, &nsp, s);
      if (n < 0) return fail(MOE_ERR_INVALID, "x must be 16-byte aligned for the tensor-core router");
      P->launches += n;
      P->launches += launch_gate_topk(d, sc.rpart, nsp, P->router_b + (size_t)layer * d.E, T, sc.ids, sc.w,
                                      sc.probs, sc.gap, s, d.aes_on ? d.lut + (size_t)layer * d.E : nullptr);
    } else {
      P->launches += launch_route_logits(d, layer, x, T, P->router_w, P->router_b, sc.logits, s);
      P->launches += launch_gate_topk(d, sc.logits, 0, nullptr, T, sc.ids, sc.w, sc.probs, sc.gap, s,
                                      d.aes_on ? d.lut + (size_t)layer * d.E : nullptr);
    }
  }
  mark(1);
  const int flags = staged ? (PLAN_HISTORY | PLAN_PERMUTE | PLAN_STAGED) : (PLAN_HISTORY | PLAN_CACHE | PLAN_PERMUTE);
  P->launches += launch_plan(d, sc, layer, T, ids, w, probs, gather ? (flags | PLAN_GATHER) : flags, region,
                             use_tc ? tc_npad(T) : 0, s);
  mark(2);
  if (use_tc) {
    // miss copies, gate/up and down + combine in one cooperative kernel
    mark(3);
    const int n = launch_tc_fused_decode(d, sc, P->tc_maps, T, x, out, s);
    if (n == -1) return fail(MOE_ERR_INVALID, "x must be 16-byte aligned for the tensor-core path");
    if (n < 0) return fail(MOE_ERR_CUDA, "cooperative launch failed: %s", cudaGetErrorString(cudaGetLastError()));
    P->launches += n;
  } else if (gather) {
    if (!staged) P->launches += launch_miss_copy(d, sc, s);
    mark(3);
    const int n = launch_tc_gather(d, sc, P->tc_maps, T, x, out, s);
    if (n < 0) return fail(MOE_ERR_INVALID, "x must be 16-byte aligned for the tensor-core path");
    P->launches += n;
  } else if (!staged && d.wdt == MOE_RESPLIT_Q4R4) {
    // The miss copies on the side stream, beside gate/up over the resident entries (the plan
    // never evicts an expert the step uses, so the copies write no slot those read); gate/up
    // over the copied entries once they have landed, then down + combine over all entries.
    CUDA_TRY(cudaEventRecord(P->ev_fork, s));
    CUDA_TRY(cudaStreamWaitEvent(P->side, P->ev_fork, 0));
    P->launches += launch_miss_copy(d, sc, P->side, kSideCopyCtas);
    CUDA_TRY(cudaEventRecord(P->ev_join, P->side));
    mark(3);
    P->launches += launch_ffn_gate_up(d, sc, T, x, s, 0);
    CUDA_TRY(cudaStreamWaitEvent(s, P->ev_join, 0));
    P->launches += launch_ffn_gate_up(d, sc, T, x, s, 1);
    P->launches += launch_ffn_down(d, sc, T, out, s);
  } else {
    if (!staged) P->launches += launch_miss_copy(d, sc, s);
    mark(3);
    P->launches += launch_ffn_gate_up(d, sc, T, x, s);
    P->launches += launch_ffn_down(d, sc, T, out, s);
  }
  mark(4);
  if (staged) {
    CUDA_TRY(cudaEventRecord(P->released[region], s));
  }
  CUDA_TRY(cudaGetLastError());
  if (ids_in) {
    // keep the supplied routing for moe_get_routing
    CUDA_TRY(cudaMemcpyAsync(sc.ids, ids_in, sizeof(int32_t) * T * d.k, cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(sc.w, w_in, sizeof(float) * T * d.k, cudaMemcpyDeviceToDevice, s));
    CUDA_TRY(cudaMemcpyAsync(sc.probs, probs_in, sizeof(float) * T * d.E, cudaMemcpyDeviceToDevice, s));
  }
  P->last_T = T;
  P->last_gap_valid = ids_in == nullptr;
  return MOE_OK;
}

static int layer_quota_host(moe_pool* P, int layer) {
  // K_l: slots layer l holds now (host copy of the owner table; AUTO mode only)
  std::vector<int32_t> owner(P->d.S);
  cudaMemcpy(owner.data(), P->d.owner, sizeof(int32_t) * P->d.S, cudaMemcpyDeviceToHost);
  int n = 0;
  for (int o : owner)
    if (o >= 0 && o / P->d.E == layer) ++n;
  return n;
}

MOE_API moe_status moe_forward(moe_pool* P, int32_t layer, const void* x, int32_t T, void* out, int32_t mode,
                               void* stream) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  if (layer < 0 || layer >= P->d.L) return fail(MOE_ERR_INVALID, "layer %d out of range", layer);
  if (T < 0) return fail(MOE_ERR_INVALID, "T must be >= 0");
  if (T > P->cfg.max_tokens) return fail(MOE_ERR_CAPACITY, "T=%d exceeds max_tokens=%d", T, P->cfg.max_tokens);
  if (mode != MOE_MODE_AUTO && mode != MOE_MODE_DECODE && mode != MOE_MODE_PREFILL_STAGED)
    return fail(MOE_ERR_INVALID, "unknown mode %d", mode);
  if (T == 0) return MOE_OK;
  if (!x || !out) return fail(MOE_ERR_INVALID, "x/out is NULL");
  if (x == out) return fail(MOE_ERR_INVALID, "out must not alias x");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(MOE_ERR_INVALID, "x and out must be 16-byte aligned");
  if (mode == MOE_MODE_PREFILL_STAGED && P->cfg.staging_regions != 2)
    return fail(MOE_ERR_INVALID, "staged prefill needs staging_regions == 2");
  CUDA_TRY(cudaSetDevice(P->device));
  bool staged = mode == MOE_MODE_PREFILL_STAGED;
  if (mode == MOE_MODE_AUTO && P->cfg.staging_regions == 2) {
    const int Kl = layer_quota_host(P, layer);
    staged = T >= Kl / P->d.k;
  }
  return run_layer(P, layer, x, T, out, staged, nullptr, nullptr, nullptr, static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_forward_routed(moe_pool* P, int32_t layer, const void* x, int32_t T, const int32_t* ids,
                                      const float* w, const float* probs, void* out, void* stream) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  if (layer < 0 || layer >= P->d.L) return fail(MOE_ERR_INVALID, "layer %d out of range", layer);
  if (T < 0) return fail(MOE_ERR_INVALID, "T must be >= 0");
  if (T > P->cfg.max_tokens) return fail(MOE_ERR_CAPACITY, "T=%d exceeds max_tokens=%d", T, P->cfg.max_tokens);
  if (T == 0) return MOE_OK;
  if (!x || !out || !ids || !w || !probs) return fail(MOE_ERR_INVALID, "NULL argument");
  if (x == out) return fail(MOE_ERR_INVALID, "out must not alias x");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15)
    return fail(MOE_ERR_INVALID, "x and out must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(ids) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(probs)) & 3)
    return fail(MOE_ERR_INVALID, "ids, w and probs must be 4-byte aligned");
  CUDA_TRY(cudaSetDevice(P->device));
  return run_layer(P, layer, x, T, out, false, ids, w, probs, static_cast<cudaStream_t>(stream));
}

MOE_API moe_status moe_update_scores(moe_pool* P, int32_t layer, const int32_t* ids, const float* probs, int32_t T,
                                     void* stream) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  if (layer < 0 || layer >= P->d.L) return fail(MOE_ERR_INVALID, "layer %d out of range", layer);
  if (T < 1) return fail(MOE_ERR_INVALID, "T must be >= 1");
  if (T > P->cfg.max_tokens) return fail(MOE_ERR_CAPACITY, "T=%d exceeds max_tokens=%d", T, P->cfg.max_tokens);
  if (!ids || !probs) return fail(MOE_ERR_INVALID, "NULL argument");
  CUDA_TRY(cudaSetDevice(P->device));
  P->launches += launch_plan(P->d, P->sc, layer, T, ids, nullptr, probs, PLAN_HISTORY, 0, 0,
                             static_cast<cudaStream_t>(stream));
  CUDA_TRY(cudaGetLastError());
  return MOE_OK;
}

// ---------------------------------------------------------------- asynchronous prefetch
// The pool's only host thread (SeqMoE "Mechanism"): it polls the mapped control region,
// takes the device's requests in order and, on a stream of its own that no compute waits
// for, copies each record from the host pool into its slot and then writes the request's
// tag into landed[slot]; the device commits the slot only when that tag matches its own.
// It also reads the GPU's position and miss flag: when the layer call now running has
// demand misses (their copies use the same link), it holds the next prefetch back until
// the position moves on, for at most one record's copy time.
static void prefetch_main(moe_pool* P) {
  cudaSetDevice(P->device);
  PfCtl* c = P->pf_ctl;
  const size_t rec = P->d.lay.rec;
  const auto defer = std::chrono::nanoseconds((long long)(rec / 200.0));   // ~200 GB/s host link
  uint32_t tail = P->pf_taken.load(), inflight = 0, seen_demand = c->demand;
  while (!P->pf_stop.load()) {
    const uint32_t head = c->head;
    if (head == tail) {
      std::this_thread::sleep_for(std::chrono::microseconds(2));
      continue;
    }
    std::atomic_thread_fence(std::memory_order_acquire);   // the requests were written before the head
    const uint32_t dm = c->demand;
    if (dm != seen_demand) {
      seen_demand = dm;
      const int32_t l0 = c->layer, s0 = c->step;
      const auto t0 = std::chrono::steady_clock::now();
      while (c->layer == l0 && c->step == s0 && std::chrono::steady_clock::now() - t0 < defer &&
             !P->pf_stop.load())
        std::this_thread::sleep_for(std::chrono::microseconds(2));
    }
    const volatile PfReq& q = c->req[tail % kPfRing];
    const int32_t slot = q.slot, flat = q.flat;
    uint32_t tag = q.tag;
    uint32_t bad = P->pf_corrupt.load();
    while (bad > 0 && !P->pf_corrupt.compare_exchange_weak(bad, bad - 1)) {
    }
    if (bad > 0) tag += 0x5A5A0000u;   // a wrong tag (test injection): the device must not commit it
    if (inflight >= kPfRing / 2) {     // the tag buffer entry about to be reused has been read
      cudaStreamSynchronize(P->pf_stream);
      inflight = 0;
    }
    uint32_t* tb = P->pf_tagbuf + (tail % kPfRing);
    *tb = tag;
    if (slot >= 0 && slot < P->d.S && flat >= 0 && flat < P->d.L * P->d.E) {
      cudaMemcpyAsync(P->d.records + (size_t)slot * rec, P->host_pool + (size_t)flat * rec, rec,
                      cudaMemcpyHostToDevice, P->pf_stream);
      cudaMemcpyAsync(const_cast<uint32_t*>(P->d.landed) + slot, tb, sizeof(uint32_t), cudaMemcpyHostToDevice,
                      P->pf_stream);
      P->pf_bytes.fetch_add(rec);
      ++inflight;
    }
    ++tail;
    c->tail = tail;
    P->pf_taken.store(tail);
  }
}

MOE_API moe_status moe_prefetch_enable(moe_pool* P, int32_t per_step) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  if (per_step < 0 || per_step > kPfMaxPerStep) return fail(MOE_ERR_INVALID, "per_step must be 0..%d", kPfMaxPerStep);
  CUDA_TRY(cudaSetDevice(P->device));
  if (per_step > 0 && !P->pf_ctl) {
    void* c = nullptr;
    void* dc = nullptr;
    CUDA_TRY(cudaHostAlloc(&c, sizeof(PfCtl), cudaHostAllocMapped | cudaHostAllocPortable));
    std::memset(c, 0, sizeof(PfCtl));
    P->pf_ctl = static_cast<PfCtl*>(c);
    CUDA_TRY(cudaHostGetDevicePointer(&dc, c, 0));
    void* tb = nullptr;
    CUDA_TRY(cudaHostAlloc(&tb, sizeof(uint32_t) * kPfRing, cudaHostAllocPortable));
    P->pf_tagbuf = static_cast<uint32_t*>(tb);
    CUDA_TRY(cudaStreamCreateWithFlags(&P->pf_stream, cudaStreamNonBlocking));
    P->d.pf_ctl = static_cast<PfCtl*>(dc);
    P->d.pf_used = 1;
  }
  if (per_step > 0 && !P->pf_thread.joinable()) {
    P->pf_stop.store(false);
    P->pf_thread = std::thread(prefetch_main, P);
  }
  P->d.pf_per_step = per_step;
  return MOE_OK;
}

MOE_API moe_status moe_prefetch_drain(moe_pool* P) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  if (!P->pf_ctl) return MOE_OK;
  CUDA_TRY(cudaSetDevice(P->device));
  CUDA_TRY(cudaDeviceSynchronize());               // every plan that may write a request has run
  const uint32_t head = P->pf_ctl->head;
  const auto t0 = std::chrono::steady_clock::now();
  while (P->pf_taken.load() - head > 0x7fffffffu) {  // taken < head (wrapping)
    if (!P->pf_thread.joinable() || std::chrono::steady_clock::now() - t0 > std::chrono::seconds(10))
      return fail(MOE_ERR_TIMEOUT, "moe_prefetch_drain: the prefetch thread did not take the requests");
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
  CUDA_TRY(cudaStreamSynchronize(P->pf_stream));
  return MOE_OK;
}

MOE_API moe_status moe_prefetch_inject_wrong_tags(moe_pool* P, uint32_t n) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  P->pf_corrupt.fetch_add(n);
  return MOE_OK;
}

MOE_API moe_status moe_set_umia(moe_pool* P, float theta, const float* beta, float gamma_decode,
                                float gamma_prefill) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  if (!(theta >= 0.f && gamma_decode >= 0.f && gamma_prefill >= 0.f && theta < INFINITY))
    return fail(MOE_ERR_INVALID, "theta and the gammas must be finite and >= 0");
  CUDA_TRY(cudaSetDevice(P->device));
  std::vector<float> b((size_t)P->d.L, 1.f);
  if (beta)
    for (int l = 0; l < P->d.L; ++l) {
      if (!(beta[l] >= 0.f && beta[l] < INFINITY)) return fail(MOE_ERR_INVALID, "beta must be finite and >= 0");
      b[l] = beta[l];
    }
  CUDA_TRY(cudaMemcpy(const_cast<float*>(P->d.umia_beta), b.data(), sizeof(float) * b.size(), cudaMemcpyHostToDevice));
  P->d.umia_theta = theta;
  P->d.umia_gamma_decode = gamma_decode;
  P->d.umia_gamma_prefill = gamma_prefill;
  return MOE_OK;
}

MOE_API moe_status moe_set_aes(moe_pool* P, int32_t on, float alpha) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  if (on && !(alpha >= 0.f && alpha < INFINITY)) return fail(MOE_ERR_INVALID, "alpha must be finite and >= 0");
  P->d.aes_on = on ? 1 : 0;
  P->d.aes_alpha = on ? alpha : 0.f;
  return MOE_OK;
}

MOE_API moe_status moe_set_wait_limit(moe_pool* P, uint64_t ns) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  if (ns == 0) ns = kDefaultWaitNs;
  if (ns < 1000ull || ns > 10000000000ull) return fail(MOE_ERR_INVALID, "wait limit must be 1 us .. 10 s (0: default)");
  P->d.wait_ns = ns;
  return MOE_OK;
}

MOE_API moe_status moe_get_status(moe_pool* P) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  CUDA_TRY(cudaSetDevice(P->device));
  CUDA_TRY(cudaDeviceSynchronize());
  int32_t st = 0;
  CUDA_TRY(cudaMemcpy(&st, P->d.status, sizeof st, cudaMemcpyDeviceToHost));
  return static_cast<moe_status>(st);
}

MOE_API moe_status moe_clear_status(moe_pool* P) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  CUDA_TRY(cudaSetDevice(P->device));
  CUDA_TRY(cudaDeviceSynchronize());
  CUDA_TRY(cudaMemset(P->d.status, 0, sizeof(int32_t)));
  // counters a timed-out launch may have left behind
  if (P->sc.dsync) CUDA_TRY(cudaMemset(P->sc.dsync, 0, tc_dsync_ints() * sizeof(uint32_t)));
  if (P->sc.ticket) CUDA_TRY(cudaMemset(P->sc.ticket, 0, sizeof(int32_t)));
  return MOE_OK;
}

MOE_API moe_status moe_get_routing(moe_pool* P, int32_t* ids, float* w, float* probs, float* gap, int32_t* slots,
                                   int32_t* perm, int32_t* offs, int32_t cap_T, int32_t* T_out) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  const int T = P->last_T, k = P->d.k, E = P->d.E;
  if (T_out) *T_out = T;
  if (cap_T < T) return fail(MOE_ERR_CAPACITY, "cap_T=%d < last T=%d", cap_T, T);
  CUDA_TRY(cudaSetDevice(P->device));
  CUDA_TRY(cudaDeviceSynchronize());
  if (T == 0) return MOE_OK;
  if (ids) CUDA_TRY(cudaMemcpy(ids, P->sc.ids, sizeof(int32_t) * T * k, cudaMemcpyDeviceToHost));
  if (w) CUDA_TRY(cudaMemcpy(w, P->sc.w, sizeof(float) * T * k, cudaMemcpyDeviceToHost));
  if (probs) CUDA_TRY(cudaMemcpy(probs, P->sc.probs, sizeof(float) * T * E, cudaMemcpyDeviceToHost));
  if (gap) {
    if (P->last_gap_valid) CUDA_TRY(cudaMemcpy(gap, P->sc.gap, sizeof(float) * T, cudaMemcpyDeviceToHost));
    else
      for (int t = 0; t < T; ++t) gap[t] = INFINITY;
  }
  if (slots) CUDA_TRY(cudaMemcpy(slots, P->sc.slots_out, sizeof(int32_t) * T * k, cudaMemcpyDeviceToHost));
  if (perm) CUDA_TRY(cudaMemcpy(perm, P->sc.perm_ent, sizeof(int32_t) * T * k, cudaMemcpyDeviceToHost));
  if (offs) CUDA_TRY(cudaMemcpy(offs, P->sc.offs, sizeof(int32_t) * (E + 1), cudaMemcpyDeviceToHost));
  return MOE_OK;
}

MOE_API moe_status moe_get_state(moe_pool* P, int32_t* lut, int32_t* owner, uint32_t* tag, float* score) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  CUDA_TRY(cudaSetDevice(P->device));
  CUDA_TRY(cudaDeviceSynchronize());
  const size_t LE = (size_t)P->d.L * P->d.E, S = P->d.S;
  if (lut) CUDA_TRY(cudaMemcpy(lut, P->d.lut, sizeof(int32_t) * LE, cudaMemcpyDeviceToHost));
  if (owner) CUDA_TRY(cudaMemcpy(owner, P->d.owner, sizeof(int32_t) * S, cudaMemcpyDeviceToHost));
  if (tag) CUDA_TRY(cudaMemcpy(tag, P->d.tag, sizeof(uint32_t) * S, cudaMemcpyDeviceToHost));
  if (score) CUDA_TRY(cudaMemcpy(score, P->d.score, sizeof(float) * LE, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

MOE_API moe_status moe_read_slot(moe_pool* P, int32_t slot, void* out, size_t out_bytes) {
  if (!P || !out) return fail(MOE_ERR_INVALID, "NULL argument");
  if (slot < 0 || slot >= P->d.S) return fail(MOE_ERR_INVALID, "moe_read_slot: slot %d out of [0, %d)", slot, P->d.S);
  if (out_bytes < P->d.lay.rec) return fail(MOE_ERR_INVALID, "moe_read_slot: buffer of %zu bytes < record %zu", out_bytes,
                                            P->d.lay.rec);
  CUDA_TRY(cudaSetDevice(P->device));
  CUDA_TRY(cudaDeviceSynchronize());
  CUDA_TRY(cudaMemcpy(out, P->d.records + (size_t)slot * P->d.lay.rec, P->d.lay.rec, cudaMemcpyDeviceToHost));
  return MOE_OK;
}

MOE_API moe_status moe_get_stats(moe_pool* P, moe_stats* out) {
  if (!P || !out) return fail(MOE_ERR_INVALID, "NULL argument");
  CUDA_TRY(cudaSetDevice(P->device));
  CUDA_TRY(cudaDeviceSynchronize());
  unsigned long long v[ST_COUNT];
  CUDA_TRY(cudaMemcpy(v, P->d.stats, sizeof v, cudaMemcpyDeviceToHost));
  out->steps = v[ST_STEPS];
  out->hits = v[ST_HITS];
  out->misses = v[ST_MISSES];
  out->bypass = v[ST_BYPASS];
  out->evictions = v[ST_EVICT];
  out->bytes_copied = v[ST_BYTES];
  out->near_ties = v[ST_NEAR_TIES];
  out->staged_layers = P->staged_count;
  out->prefetch_issued = v[ST_PF_ISSUED];
  out->prefetch_committed = v[ST_PF_COMMITTED];
  out->prefetch_demanded = v[ST_PF_DEMANDED];
  out->prefetch_bytes = P->pf_bytes.load();
  out->aes_substitutions = v[ST_AES];
  out->critical_entries = v[ST_CRIT];
  return MOE_OK;
}

MOE_API uint64_t moe_launch_count(const moe_pool* P) { return P ? P->launches : 0; }

MOE_API moe_status moe_profile_enable(moe_pool* P, int32_t on) {
  if (!P) return fail(MOE_ERR_INVALID, "pool is NULL");
  CUDA_TRY(cudaSetDevice(P->device));
  if (on && P->prof_ev.empty()) {
    const size_t n = (size_t)P->d.L * (MOE_NUM_STAGES + 1);
    P->prof_ev.resize(n, nullptr);
    P->prof_fused.assign((size_t)P->d.L, 0);
    for (size_t i = 0; i < n; ++i) CUDA_TRY(cudaEventCreate(&P->prof_ev[i]));
  }
  P->prof_on = on != 0;
  return MOE_OK;
}

MOE_API moe_status moe_profile_read(moe_pool* P, int32_t layer, float* stage_ms) {
  if (!P || !stage_ms) return fail(MOE_ERR_INVALID, "NULL argument");
  if (layer < 0 || layer >= P->d.L) return fail(MOE_ERR_INVALID, "layer out of range");
  if (P->prof_ev.empty()) return fail(MOE_ERR_INVALID, "profiling was never enabled");
  CUDA_TRY(cudaSetDevice(P->device));
  const size_t b = (size_t)layer * (MOE_NUM_STAGES + 1);
  if (P->prof_fused[layer]) {
    // one kernel: every stage is attributed to the expert stage
    for (int i = 0; i < MOE_NUM_STAGES; ++i) stage_ms[i] = 0.f;
    CUDA_TRY(cudaEventSynchronize(P->prof_ev[b + MOE_NUM_STAGES]));
    CUDA_TRY(cudaEventElapsedTime(&stage_ms[MOE_STAGE_FFN], P->prof_ev[b], P->prof_ev[b + MOE_NUM_STAGES]));
    return MOE_OK;
  }
  for (int i = 0; i < MOE_NUM_STAGES; ++i) {
    CUDA_TRY(cudaEventSynchronize(P->prof_ev[b + i + 1]));
    CUDA_TRY(cudaEventElapsedTime(&stage_ms[i], P->prof_ev[b + i], P->prof_ev[b + i + 1]));
  }
  return MOE_OK;
}
