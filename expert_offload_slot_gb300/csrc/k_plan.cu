// Steps a3 (routing history and eviction score), a4 (expert_id -> slot_id
// rewrite and miss detection), a5 (victim choice and table update) and a7
// (stable permutation of token rows by expert, and the work lists the expert
// kernels consume).  One CTA per layer call: the victims of a layer are a
// chain of dependent decisions and the whole working set fits a CTA.
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
// Latency plan: everything the decisions read (the layer's ring history, the
// step's probabilities, the table row, the owner of every slot) is staged into
// shared memory in one round trip; victims come from block arg-mins over
// shared memory; the table, owners, tags and copy list are then written in
// parallel without reading global memory again.
//
// Score arithmetic uses explicitly rounded fp32 operations in a fixed order
// (no contraction), because the scores decide integer victim choices.  The
// token average sums each expert's probabilities in ascending token order.
#include "plan_body.cuh"

namespace moeslot {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  extern __shared__ __align__(16) uint8_t dsm[];
  plan_body<kPlanThreads>(a, dsm);
}

size_t plan_smem_bytes(const PoolDev& p, int Tmax, int* owner_cap_out, int* tok_rows_out) {
  return plan_smem_bytes_nt<kPlanThreads>(p, Tmax, owner_cap_out, tok_rows_out);
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
  a.gather_bn = gather_tile_rows(p, T);
  const size_t smem = plan_smem_bytes(p, sc.tmax, &a.owner_cap, &a.tok_rows);
  static size_t configured = 0;
  if (smem > configured) {
    cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    configured = smem;
  }
  plan_kernel<<<1, kPlanThreads, smem, s>>>(a);
  return 1;
}

}  // namespace moeslot
