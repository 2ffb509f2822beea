/*
 * moeslot.h — C ABI of a routed Mixture-of-Experts layer whose experts are read
 * from one shared, fixed-address slot pool on a single GB300 GPU (sm_103a).
 *
 * What the layer computes (one call of moe_forward, one MoE layer, T tokens):
 *   a1 router        z = x · W_rᵀ + b                      RapidMoE §2.1
 *   a2 gate + top-k  softmax- or sigmoid-renormalised over the k largest
 *                    logits                                  RapidMoE §2.1; CAP §II-A Eq. 1
 *   a3 history       per-expert routing history and eviction score
 *                    (MoE-CORE windowed/EMA score, HybriMoE Minus Recent
 *                    Score, or LRU)                          MoE-CORE "Mechanism"; HybriMoE "Mechanism"
 *   a4 table         expert_id -> slot_id lookup; resident/missing detection
 *                                                            SeqMoE "Mechanism"
 *   a5 victims       a missing expert takes a free slot or the lowest-score
 *                    slot that this step does not need       MoE-CORE / HybriMoE "Mechanism"
 *   a6 miss copy     started by the device: a kernel reads the expert from
 *                    the pinned, mapped host pool into its slot  SeqMoE "Mechanism"
 *   a7 permute       token rows grouped by expert (stable)
 *   a8 experts       SwiGLU: W_down (SiLU(W_gate x) ⊙ W_up x)   RapidMoE §4.5 Eq. 7
 *   a9 combine       out[t] = Σ_j w[t,j] · y_j (+ shared expert, weight 1)
 *                                                            CAP §II-A Eq. 1; RapidMoE Table 2
 *   a10 staging      large prefills read whole layers from two swapped
 *                    layer-sized staging regions             MoE-CORE "Mechanism"
 *
 * Conventions
 *   - Every call is stream-ordered and asynchronous unless it says otherwise.
 *   - Argument errors are returned synchronously (MOE_ERR_INVALID) and nothing
 *     is launched.
 *   - Errors the device finds (an out-of-range id or slot) are written once
 *     into a sticky device status word; moe_get_status() reads it.  Kernels
 *     never trap.
 *   - No C++ exception crosses this boundary.
 *   - The pool owns every device buffer it allocates (slots, staging regions,
 *     table, history, per-call scratch).  The caller owns the host pool, the
 *     router and shared-expert weights, x and out.
 *   - A decode call (MOE_MODE_DECODE) performs no host synchronisation and
 *     allocates nothing, so a sequence of such calls can be captured into a
 *     CUDA graph.  MOE_MODE_AUTO on a pool with staging regions does
 *     synchronise (see moe_forward).
 *   - Every device-side wait (a copy landing, another CTA's arrival) is
 *     bounded; one that runs out records MOE_ERR_TIMEOUT, and the kernel
 *     drains its own copies and returns.
 *   - One pool must not be used from two streams at once: calls on one pool
 *     share its scratch and its table.
 *
 * Expert record (the unit of the host pool, of a slot and of a staging region;
 * SeqMoE "Mechanism": one fixed-base pool of [num_slots, record] entries).
 * moe_expert_layout() returns the offsets; moe_pack_expert_record() writes a
 * record from plain row-major W_gate, W_up, W_down.  The layout depends on
 * weight_dtype:
 *   MOE_F32, MOE_FP8_E4M3_B128 (row-major):
 *     w13  [2I, H]: rows 0..I-1 are W_gate, rows I..2I-1 are W_up
 *     w2   [H, I]:  W_down
 *     s13  [2I/128, H/128] fp32 block scales   (MOE_FP8_E4M3_B128 only)
 *     s2   [H/128, I/128]  fp32 block scales   (MOE_FP8_E4M3_B128 only)
 *     Element (i, j) of a block-scaled fp8 matrix is e4m3(q[i,j]) * scale[i/128][j/128].
 *   MOE_BF16 (tiled; NOT row-major): each matrix is cut into tiles of 128 rows
 *     x 64 columns (16384 bytes; rows and columns past the matrix are zero),
 *     and inside a tile element (r, c) is at byte
 *         r*128 + ((c/8) XOR (r mod 8))*16 + (c mod 8)*2
 *     (the tensor cores' 128-byte-swizzled operand order, so a pipeline stage
 *     is one contiguous copy).  Tile order:
 *     w13 at w13_off: tile (m, b, g) of W_gate (g = 0) or W_up (g = 1), rows
 *         128m.., columns 64b.., at ((m*ceil(H/64) + b)*2 + g) * 16384
 *     w2 at w2_off:   tile (m, b) of W_down at (m*ceil(I/64) + b) * 16384
 *     So element (i, j) of W_up is at byte
 *         w13_off + (((i/128)*ceil(H/64) + j/64)*2 + 1)*16384 + tile byte of (i mod 128, j mod 64).
 *     A row-major bf16 record gives wrong outputs without any error: pack
 *     bf16 records with moe_pack_expert_record.
 *   MOE_RESPLIT_Q4R4 (RapidMoE §4.4 Alg. 3, with a codec defined here): gate/up
 *     stored as W^Q plus a residual W^R, down stored twice (W^L, W^H), as
 *     symmetric integer codes per 128-column group, scale = group amax /
 *     (2^(b-1) - 1), code = round-half-even(w / scale) (fp32), row-major, in this
 *     order (IH = I * H bytes):
 *       q13  [2I][H/2]  4-bit codes of W^Q (gate rows, then up rows)   at 0
 *       r13  [2I][H/2]  4-bit codes of W^R = Quantize(W - W^Q, 4)      at IH
 *       l2   [H][I/2]   4-bit codes of W^L_down                        at 2 IH
 *       h2   [H][I]     8-bit codes of W^H_down                        at 2.5 IH
 *       sq13, sr13 [2I][H/128], then sl2, sh2 [H][I/128]: fp32 scales, from 3.5 IH
 *     A byte holds columns 2j (low nibble) and 2j+1 (high nibble), two's
 *     complement.  moe_expert_layout returns (q13, l2, sq13, sl2, record).
 *     Critical experts (moe_set_umia) run W^Q + W^R and W^H_down, the others
 *     W^Q and W^L_down.  H and I multiples of 128; activations bf16.
 *   Every record is padded to a multiple of 4096 bytes.
 */
#ifndef MOESLOT_H
#define MOESLOT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef struct moe_pool moe_pool;   /* opaque */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,    /* bad argument or configuration                      */
  MOE_ERR_OOM = 2,        /* a device allocation failed                         */
  MOE_ERR_CUDA = 3,       /* a CUDA runtime call failed                         */
  MOE_ERR_CAPACITY = 4,   /* T exceeds the pool's max_tokens, or a one-step
                             record / static scratch is too small              */
  MOE_ERR_TIMEOUT = 5,    /* a bounded device-side wait gave up                 */
  MOE_ERR_TAG = 6,        /* reserved (a prefetch whose tag does not match is
                             simply not committed)                             */
  MOE_ERR_BOUNDS = 7      /* the device met an expert id or slot out of range   */
} moe_status;

enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_FP8_E4M3_B128 = 2,            /* dtypes   */
       MOE_RESPLIT_Q4R4 = 3 };                                       /* residual-split weights */
enum { MOE_GATE_SOFTMAX_RENORM = 0, MOE_GATE_SIGMOID_RENORM = 1 };  /* gating   */
enum { MOE_EVICT_CORE = 0, MOE_EVICT_MRS = 1, MOE_EVICT_LRU = 2 };  /* policy   */
enum { MOE_MODE_AUTO = 0, MOE_MODE_DECODE = 1, MOE_MODE_PREFILL_STAGED = 2 };

typedef struct {
  int32_t num_layers;        /* L                                                  */
  int32_t num_experts;       /* E routed experts per layer, 1..256                 */
  int32_t top_k;             /* k, 1..min(E, 32)                                   */
  int32_t hidden;            /* H: multiple of 4 (f32), 8 (bf16), 16 and 128 (fp8) */
  int32_t inter;             /* I: same rule as H                                  */
  int32_t num_slots;         /* S slots in the shared pool, >= 1                   */
  int32_t weight_dtype;      /* MOE_F32, MOE_BF16 or MOE_FP8_E4M3_B128             */
  int32_t act_dtype;         /* MOE_F32 or MOE_BF16 (x, out, router weights)       */
  int32_t gating;            /* MOE_GATE_*                                         */
  int32_t has_shared_expert; /* 0 or 1: one always-resident shared expert / layer  */
  int32_t evict_policy;      /* MOE_EVICT_*                                        */
  int32_t window;            /* W steps of routing history, 1..64 (16 typical)     */
  float ema_decay;           /* lambda of the selection EMA (0.9 typical)          */
  float core_w[4];           /* MoE-CORE weights: count, EMA, score, recency       */
  int32_t staging_regions;   /* 0, or 2 for double-buffered full-layer prefill     */
  int32_t max_tokens;        /* largest T any call on this pool will pass          */
} moe_config;

typedef struct {   /* cumulative counters of a pool */
  uint64_t steps;            /* history updates performed                          */
  uint64_t hits;             /* needed experts found resident                      */
  uint64_t misses;           /* needed experts not resident                        */
  uint64_t bypass;           /* misses that got no slot (every slot held an expert
                                this step needs): copied into a one-step record   */
  uint64_t evictions;        /* occupants replaced                                 */
  uint64_t bytes_copied;     /* host -> device bytes moved by miss copies          */
  uint64_t near_ties;        /* tokens whose k-th/(k+1)-th logit gap is < 1e-4     */
  uint64_t staged_layers;    /* layers copied into a staging region               */
  uint64_t prefetch_issued;  /* prefetch requests the device wrote (moe_prefetch_enable) */
  uint64_t prefetch_committed; /* prefetched slots committed on a matching tag      */
  uint64_t prefetch_demanded;  /* pending prefetches a step needed before their commit */
  uint64_t prefetch_bytes;   /* record bytes the host thread copied for prefetches */
  uint64_t aes_substitutions; /* (token, expert) misses replaced by a resident expert */
  uint64_t critical_entries; /* residual-split experts run at high precision (UMIA) */
} moe_stats;

/* Byte layout of one expert record for `cfg` (see the header comment).  Any
 * output pointer may be NULL.  Returns MOE_ERR_INVALID for a bad config.
 * Host only: no CUDA call. */
MOE_API moe_status moe_expert_layout(const moe_config* cfg, size_t* w13_off, size_t* w2_off,
                                     size_t* s13_off, size_t* s2_off, size_t* record_bytes);

/* Write one expert's record (the layout of the header comment) from plain
 * row-major matrices.  Host memory in and out; no CUDA call, no allocation,
 * safe from any thread.
 *   w_gate [I, H], w_up [I, H], w_down [H, I]: row-major, elements in the
 *       storage of cfg->weight_dtype (MOE_F32: float; MOE_BF16: bf16 bit
 *       patterns, uint16; MOE_FP8_E4M3_B128: e4m3 codes, uint8;
 *       MOE_RESPLIT_Q4R4: float, which this call quantizes as the header states)
 *   s_gate [I/128, H/128], s_up [I/128, H/128], s_down [H/128, I/128]: fp32
 *       block scales, MOE_FP8_E4M3_B128 only (NULL otherwise)
 *   record: record_bytes >= moe_expert_layout's record_bytes; the padding is
 *       zeroed.  Host-pool record (l, e) goes to host_pool + (l*E + e)*record_bytes.
 * MOE_ERR_INVALID for a bad config, a NULL matrix or a short buffer. */
MOE_API moe_status moe_pack_expert_record(const moe_config* cfg, const void* w_gate, const void* w_up,
                                          const void* w_down, const float* s_gate, const float* s_up,
                                          const float* s_down, void* record, size_t record_bytes);

/* Pinned, mapped host memory for a host pool (cudaHostAlloc with the mapped
 * and portable flags).  Blocking.  Free it with moe_host_free. */
MOE_API moe_status moe_host_alloc(size_t bytes, void** out);
MOE_API moe_status moe_host_free(void* p);

/* Create a pool on `device`.  Blocking; allocates all device memory the pool
 * will ever use (slots: num_slots records at one fixed base address —
 * SeqMoE "Mechanism": a pool of cache slots shared by every MoE layer at a
 * fixed base, experts kept in pinned, mapped host memory; MoE-CORE
 * "Mechanism": two layer-sized regions for full-layer prefill).
 *   host_pool       caller-owned pinned host memory (moe_host_alloc, or
 *                   cudaHostAlloc/cudaHostRegister with the mapped flag) holding
 *                   L*E expert records, record (l, e) at (l*E + e)*record_bytes;
 *                   it must stay valid and unchanged while the pool lives
 *   host_pool_bytes at least L*E*record_bytes
 *   router_w        device, [L][E][H] in act_dtype; caller-owned, outlives pool
 *   router_b        device, fp32 [L][E]; caller-owned, outlives pool
 *   shared_w        device, L expert records (one shared expert per layer) when
 *                   cfg->has_shared_expert, else NULL; caller-owned
 * The table starts empty (every expert missing, every slot free). */
MOE_API moe_status moe_pool_create(const moe_config* cfg, const void* host_pool, size_t host_pool_bytes,
                                   const void* router_w, const float* router_b, const void* shared_w,
                                   int device, moe_pool** out);
MOE_API moe_status moe_pool_destroy(moe_pool* pool);   /* blocking; NULL is a no-op */

/* Replace the whole expert_id -> slot_id table (SeqMoE "Mechanism").
 *   lut_host  host, int32 [L*E]: slot id, or -1 for "not resident"; each slot
 *             may appear at most once.
 * Every assigned slot is filled from the host pool on `stream` and its tag is
 * incremented.  Routing history is kept.  Blocking on the host only for the
 * small table upload: the slot copies (one record per assigned slot) are still
 * running when the call returns, so work on another stream that reads the pool
 * (moe_forward included) must first wait for `stream`. */
MOE_API moe_status moe_set_lut(moe_pool* pool, const int32_t* lut_host, void* stream);

/* Host-initiated placement of expert (layer, expert) into `slot`: the slot's
 * occupant is evicted, a previous slot of this expert becomes free, the record
 * is copied by the device-side copy kernel and the slot's tag incremented
 * (SeqMoE "Mechanism": a slot's tag grows with every new occupant, so a copy
 * into it can be told apart from the next).  Stream-ordered on `stream`. */
MOE_API moe_status moe_load_slot(moe_pool* pool, int32_t layer, int32_t expert, int32_t slot, void* stream);

/* One MoE layer forward (steps a1..a9, or a10 for a staged prefill).
 *   x     device [T, H] act_dtype;   out  device [T, H] act_dtype (may not alias x)
 *   T     0..max_tokens; T == 0 returns MOE_OK and does nothing
 *   mode  MOE_MODE_DECODE: slot pool path, misses copied by the device;
 *         MOE_MODE_PREFILL_STAGED: the whole layer is read from a staging
 *         region (needs staging_regions == 2); the history is still updated;
 *         MOE_MODE_AUTO: staged when staging_regions == 2 and
 *         T >= floor(K_l / k), K_l being the slots layer l holds now
 *         (MoE-CORE "Mechanism"), else the slot pool path.  To count K_l
 *         the call reads the pool's slot owners back to the host, so AUTO on
 *         a pool with staging regions SYNCHRONISES the host with the device
 *         and cannot be captured in a CUDA graph; pass MOE_MODE_DECODE or
 *         MOE_MODE_PREFILL_STAGED to choose without a synchronisation.
 * A staged call stages layer l (if not already there), then queues layer l+1
 * into the other region (after layer l-1 has released it) ahead of layer l's
 * kernels, so that the copy runs beside them; it synchronises the host with
 * nothing but makes `stream` wait for the pool's internal copy stream. */
MOE_API moe_status moe_forward(moe_pool* pool, int32_t layer, const void* x, int32_t T, void* out,
                               int32_t mode, void* stream);

/* Same as a slot-pool moe_forward, with the routing supplied by the caller
 * (steps a3..a9 only):
 *   ids   device int32 [T, k], distinct experts per token
 *   w     device fp32 [T, k] routing weights used in the combine
 *   probs device fp32 [T, E] per-expert probabilities used for the history */
MOE_API moe_status moe_forward_routed(moe_pool* pool, int32_t layer, const void* x, int32_t T,
                                      const int32_t* ids, const float* w, const float* probs,
                                      void* out, void* stream);

/* Step a3 alone: one history/score update of `layer` from device ids [T, k]
 * and device fp32 probs [T, E] (MoE-CORE "Mechanism": selection count over a
 * window, EMA of selections, current router score, age since the last
 * selection; HybriMoE "Mechanism": Minus Recent Score; RapidMoE §4.3: the
 * router score of a T-token step is the token-averaged probability, summed in
 * ascending token order).  Stream-ordered; the table is not touched. */
MOE_API moe_status moe_update_scores(moe_pool* pool, int32_t layer, const int32_t* ids, const float* probs,
                                     int32_t T, void* stream);

/* Asynchronous prefetch (SeqMoE "Mechanism"; HybriMoE "Mechanism" for the order).
 * per_step > 0 starts the pool's one host thread and makes every layer call's plan
 * issue up to per_step minus that step's misses prefetches for its layer: the
 * experts the step does not need, neither resident nor pending, highest router
 * score first, each into the lowest free slot or the lowest-score slot of the
 * layer the step does not need.  Such a slot turns pending (not resident, never a
 * victim) and its tag grows by one.  The device writes the request (slot, expert,
 * tag) and its position and a miss flag into a mapped control region; the thread
 * copies the record into the slot on a stream of its own and then writes the tag
 * into device memory, in stream order.  A later plan commits the slot only if that
 * tag equals the slot's tag, so a stale or wrong write-back is never committed; a
 * step that needs a pending expert copies it into that slot itself.  No kernel ever
 * waits for the thread.  per_step 0 stops issuing (slots already pending are still
 * committed or demanded); 0..8.  Set it before capturing calls into a CUDA graph:
 * a captured call keeps the setting it was captured with.  Once prefetch was used,
 * moe_load_slot is refused; moe_set_lut drains it first. */
MOE_API moe_status moe_prefetch_enable(moe_pool* pool, int32_t per_step);
/* Blocking: every request issued so far has been copied and its tag written back. */
MOE_API moe_status moe_prefetch_drain(moe_pool* pool);
/* Fault injection on the host side: the next n tags the thread writes back are wrong
 * (their slots are never committed). */
MOE_API moe_status moe_prefetch_inject_wrong_tags(moe_pool* pool, uint32_t n);

/* Approximate expert substitution (MoE-CORE "Mechanism"), off by default.  It
 * CHANGES RESULTS: with on = 1, a token's selected expert that is not resident at
 * the start of the step and whose router logit is within alpha of the best
 * logit the token did not select (the rank-(k+1) boundary) is replaced, in rank
 * order, by the token's best resident unselected expert (ties to the lower id),
 * which keeps the missed expert's routing weight.  A miss above the band still
 * takes the exact copy.  The rest of the step (history, table, misses, experts,
 * combine) sees the rewritten routing; moe_get_routing returns it.  Applies to
 * the calls issued after it (a captured call keeps its setting). */
MOE_API moe_status moe_set_aes(moe_pool* pool, int32_t on, float alpha);

/* UMIA (RapidMoE §4.3, Eq. 3-4) for MOE_RESPLIT_Q4R4 pools: an expert a step uses
 * runs at high precision when its token-averaged router probability reaches
 * Theta(l, t) = (theta * beta[l]) * gamma_t (fp32), gamma_t = gamma_decode for
 * slot-pool calls and gamma_prefill for staged prefill calls; the shared expert
 * always does.  beta: host float [L] (NULL: all 1).  Defaults: theta 0 (every
 * expert critical), beta 1, gammas 1.  Blocking only for the beta upload; applies
 * to the calls issued after it. */
MOE_API moe_status moe_set_umia(moe_pool* pool, float theta, const float* beta, float gamma_decode,
                                float gamma_prefill);

/* Limit of every wait a kernel of this pool makes on another CTA of its grid
 * (a miss record landing, the routing or the plan being published, a tile's
 * partial sums, the final arrival before the combine): `ns` nanoseconds of
 * global time, 1 s by default (ns == 0 restores it); 1 us .. 10 s.  A wait
 * that runs out records MOE_ERR_TIMEOUT; the kernel then skips its remaining
 * work, waits for its own copies and tensor-core operations (those waits keep
 * their 1 s limit), frees its tensor memory and returns.  The output of that
 * call is undefined and its table changes may not have reached the slots:
 * after moe_clear_status, moe_set_lut restores a consistent pool.  Host-side
 * setting; applies to the calls issued after it.  Short limits are for tests
 * of this path. */
MOE_API moe_status moe_set_wait_limit(moe_pool* pool, uint64_t ns);

/* Blocking: synchronises the device, returns the sticky device status (MOE_OK
 * if no device-side error was recorded).  moe_clear_status resets it. */
MOE_API moe_status moe_get_status(moe_pool* pool);
MOE_API moe_status moe_clear_status(moe_pool* pool);

/* Blocking: host copies of the last forward's routing (any pointer may be NULL),
 * for parity checks: the top-k ids and renormalised weights (RapidMoE §2.1;
 * CAP §II-A Eq. 1), the full probabilities, the expert_id -> slot_id rewrite
 * (SeqMoE "Mechanism") and the expert-sorted permutation of token rows.
 *   ids [T,k] int32, w [T,k] fp32, probs [T,E] fp32, gap [T] fp32 (the k-th
 *   minus the (k+1)-th fp32 logit; +inf when k == E or the routing was
 *   supplied), slots [T,k] int32 (slot read; -1 = a one-step copy, -2 = a
 *   staging region),
 *   perm [T*k] int32 (flat entry t*k+j at each expert-sorted row),
 *   offs [E+1] int32 (row offset of each expert).  *T_out receives T. */
MOE_API moe_status moe_get_routing(moe_pool* pool, int32_t* ids, float* w, float* probs, float* gap,
                                   int32_t* slots, int32_t* perm, int32_t* offs, int32_t cap_T,
                                   int32_t* T_out);

/* Blocking: host copies of the cache state (any pointer may be NULL).
 *   lut [L*E] int32, owner [S] int32 (l*E+e, -1 free, -2 - (l*E+e) holding a
 *   pending prefetch of (l, e)), tag [S] uint32,
 *   score [L*E] fp32 (eviction score as of each layer's last update). */
MOE_API moe_status moe_get_state(moe_pool* pool, int32_t* lut, int32_t* owner, uint32_t* tag, float* score);

/* Blocking: host copy of the record held by `slot` (0 <= slot < num_slots),
 * record_bytes of moe_expert_layout into `out` (host, at least that many bytes,
 * out_bytes says how many).  For checks: a slot owned by (l, e) holds the bytes
 * of host record l*E+e.  MOE_ERR_INVALID on a bad slot or a short buffer. */
MOE_API moe_status moe_read_slot(moe_pool* pool, int32_t slot, void* out, size_t out_bytes);

/* Blocking: cumulative counters. */
MOE_API moe_status moe_get_stats(moe_pool* pool, moe_stats* out);

/* Per-stage timing with CUDA events (off by default).  While enabled, every
 * forward records pool-owned events on its stream between its stages (inside
 * a captured graph they become event nodes); moe_profile_read returns, for the
 * latest forward of `layer`, the elapsed milliseconds of each stage.  When the
 * forward ran as one decode layer kernel (bf16 weights, T <= 32: router, gate,
 * plan and experts in one launch) the whole call is reported under
 * MOE_STAGE_FFN and the other stages are 0.  Enabling creates
 * L*(MOE_NUM_STAGES+1) events and is blocking. */
enum { MOE_STAGE_ROUTE = 0,     /* router GEMV + gate/top-k                        */
       MOE_STAGE_PLAN = 1,      /* history, table, victims, permutation            */
       MOE_STAGE_COPY = 2,      /* miss copies run as their own kernel (0 when the
                                   expert kernel does them itself)                 */
       MOE_STAGE_FFN = 3,       /* expert gate/up, down and weighted combine       */
       MOE_NUM_STAGES = 4 };
MOE_API moe_status moe_profile_enable(moe_pool* pool, int32_t on);
MOE_API moe_status moe_profile_read(moe_pool* pool, int32_t layer, float* stage_ms /* [MOE_NUM_STAGES] */);

/* Offline cache shaping (MoE-CORE "Mechanism"): host code only, no CUDA call.
 * A profiling trace of the routing drives both calls:
 *   ids    host int32 [steps][L][T][k]   the experts each token selected
 *   probs  host fp32  [steps][L][T][E]   the router probabilities (as moe_get_routing
 *                                        returns them)
 * moe_plan_quotas splits a budget of `budget` slots over the L layers.  Layer l's
 * hit-rate curve h_l(K) is a replay of its trace through a K-slot cache filled
 * from the profile (below) with this config's eviction policy, window, EMA rate
 * and weights; h = hits / needed experts.  It starts from the uniform split
 * (floor(budget/L), one more for the first budget mod L layers, at most E) and
 * then moves delta_k slots at a time from the donor (hit rate still >= the median
 * after shrinking, at least one slot left; the smallest drop) to the receiver (hit
 * rate <= median - tau_low, at most E slots; the largest gain), ties to the lower
 * layer, as long as the gain exceeds the drop.  quota [L] receives the slot
 * counts, hit [L] (or NULL) h_l at them.
 * moe_profile_lut writes the initial table lut [L*E] for moe_set_lut: layer l's
 * quota[l] experts of highest mean probability over the trace (ties to the lower
 * id), slots numbered layer by layer in that order; the quotas must sum to at
 * most cfg->num_slots.
 * MOE_ERR_INVALID for a bad config or trace (an id outside 0..E-1). */
MOE_API moe_status moe_plan_quotas(const moe_config* cfg, const int32_t* ids, const float* probs, int32_t steps,
                                   int32_t T, int32_t budget, int32_t delta_k, double tau_low, int32_t* quota,
                                   double* hit);
MOE_API moe_status moe_profile_lut(const moe_config* cfg, const float* probs, int32_t steps, int32_t T,
                                   const int32_t* quota, int32_t* lut);

/* Router projection + gate/top-k (steps a1, a2) with no device allocation.
 * The pages have no counterpart: this exists for callers that cannot call
 * cudaMalloc where they route tokens — code running while a CUDA graph is
 * captured in global capture mode, or hosts whose framework owns the device
 * memory budget and forbids third-party allocations — and so cannot create a
 * moe_pool.  The fp32 logits scratch is a file-scope device array of
 * MOE_NOALLOC_MAX_LOGITS floats held by every device that loads the library
 * until exit; T * num_experts above it returns MOE_ERR_CAPACITY.  All calls on
 * a device share that array: calls whose kernels overlap on the GPU race.
 * Runs on the current device and on `stream`; the first call on a device looks
 * up the array's device address (cudaGetSymbolAddress), so make it before any
 * stream capture.  Calls no allocating routine.
 *   x         device [T, hidden] act_dtype (MOE_F32 or MOE_BF16)
 *   router_w  device [num_experts, hidden] act_dtype (one layer's W_r)
 *   router_b  device fp32 [num_experts]
 *   ids [T, top_k] int32, w [T, top_k] fp32, probs [T, num_experts] fp32,
 *   gap [T] fp32: device outputs, as moe_get_routing describes them.
 * x and router_w must be 16-byte aligned (they are read 16 bytes at a time),
 * the other pointers 4-byte aligned.  Argument errors, misalignment included,
 * return MOE_ERR_INVALID before anything is launched; T == 0 returns MOE_OK. */
#define MOE_NOALLOC_MAX_LOGITS 65536
MOE_API moe_status moe_route_topk_noalloc(int32_t num_experts, int32_t top_k, int32_t hidden, int32_t act_dtype,
                                          int32_t gating, const void* x, int32_t T, const void* router_w,
                                          const float* router_b, int32_t* ids, float* w, float* probs, float* gap,
                                          void* stream);

/* Number of kernel launches the library issued since the pool was created. */
MOE_API uint64_t moe_launch_count(const moe_pool* pool);

/* Text of the last error returned on this thread ("" if none). */
MOE_API const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOESLOT_H */
