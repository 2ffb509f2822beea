// moe_route_topk_noalloc: router projection + gate/top-k for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they need routing:
// code that runs while a CUDA graph is being captured in global capture mode
// (an allocation there invalidates the capture), and hosts whose framework
// owns the whole device memory budget through its own allocator and forbids
// third-party allocations.  Such callers cannot create a moe_pool (which
// allocates its scratch), so this entry point keeps the only scratch it needs
// — the fp32 logits [T, E] — in a file-scope __device__ array instead.
//
// The array is MOE_NOALLOC_MAX_LOGITS floats (256 KiB).  It lives in every
// device that loads this library until the process exits, and all calls on a
// device share it: two calls whose kernels overlap on the GPU race on it.
// It is fully overwritten by every call, so nothing needs clearing.
//
// In host code the array's name is only a host-side stand-in, not a device
// address: the device address is looked up once per device with
// cudaGetSymbolAddress (on the first call made with that device current) and
// cached.  That first call therefore makes a runtime call that is not a
// stream operation; make it before any stream capture.
//
// The kernels are the library's own router and gate kernels, launched with
// the scratch address in place of a pool's buffer.
#include <mutex>

#include "moeslot_internal.cuh"

namespace moeslot {

static __device__ __align__(256) float g_noalloc_logits[MOE_NOALLOC_MAX_LOGITS];
static __device__ __align__(256) unsigned long long g_noalloc_stats[ST_COUNT];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_logits_addr[kMaxDevices] = {};
unsigned long long* g_stats_addr[kMaxDevices] = {};
}  // namespace

}  // namespace moeslot

using namespace moeslot;

MOE_API moe_status moe_route_topk_noalloc(int32_t num_experts, int32_t top_k, int32_t hidden, int32_t act_dtype,
                                          int32_t gating, const void* x, int32_t T, const void* router_w,
                                          const float* router_b, int32_t* ids, float* w, float* probs, float* gap,
                                          void* stream) {
  if (num_experts < 1 || num_experts > 256) return set_last_error(MOE_ERR_INVALID, "num_experts must be in 1..256");
  if (top_k < 1 || top_k > num_experts || top_k > 32)
    return set_last_error(MOE_ERR_INVALID, "top_k must be in 1..min(num_experts, 32)");
  if (act_dtype != MOE_F32 && act_dtype != MOE_BF16)
    return set_last_error(MOE_ERR_INVALID, "act_dtype must be MOE_F32 or MOE_BF16");
  if (gating != MOE_GATE_SOFTMAX_RENORM && gating != MOE_GATE_SIGMOID_RENORM)
    return set_last_error(MOE_ERR_INVALID, "unknown gating");
  const int per16 = act_dtype == MOE_F32 ? 4 : 8;
  if (hidden < per16 || hidden % per16)
    return set_last_error(MOE_ERR_INVALID, "hidden must be a positive multiple of 16 bytes of act_dtype");
  if (T < 0) return set_last_error(MOE_ERR_INVALID, "T must be >= 0");
  if ((long long)T * num_experts > MOE_NOALLOC_MAX_LOGITS)
    return set_last_error(MOE_ERR_CAPACITY,
                          "T * num_experts exceeds MOE_NOALLOC_MAX_LOGITS (65536), the static scratch size");
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !router_b || !ids || !w || !probs || !gap)
    return set_last_error(MOE_ERR_INVALID, "NULL argument");
  // the router kernel reads x and router_w 16 bytes at a time; the rest are 4-byte elements
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(router_w)) & 15)
    return set_last_error(MOE_ERR_INVALID, "x and router_w must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(router_b) | reinterpret_cast<uintptr_t>(ids) | reinterpret_cast<uintptr_t>(w) |
       reinterpret_cast<uintptr_t>(probs) | reinterpret_cast<uintptr_t>(gap)) & 3)
    return set_last_error(MOE_ERR_INVALID, "router_b, ids, w, probs and gap must be 4-byte aligned");

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return set_last_error(MOE_ERR_CUDA, "no usable current device");
  float* logits = nullptr;
  unsigned long long* stats = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_logits_addr[dev]) {
      void* a = nullptr;
      void* b = nullptr;
      if (cudaGetSymbolAddress(&a, g_noalloc_logits) != cudaSuccess || !a)
        return set_last_error(MOE_ERR_CUDA, "cudaGetSymbolAddress of the logits scratch failed");
      if (cudaGetSymbolAddress(&b, g_noalloc_stats) != cudaSuccess || !b)
        return set_last_error(MOE_ERR_CUDA, "cudaGetSymbolAddress of the counter failed");
      g_logits_addr[dev] = static_cast<float*>(a);
      g_stats_addr[dev] = static_cast<unsigned long long*>(b);
    }
    logits = g_logits_addr[dev];
    stats = g_stats_addr[dev];
  }
  PoolDev p = {};
  p.E = num_experts;
  p.k = top_k;
  p.H = hidden;
  p.adt = act_dtype;
  p.gating = gating;
  p.stats = stats;   // near-tie counter of this entry point; never read back
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  launch_route_logits(p, 0, x, T, router_w, router_b, logits, s);
  launch_gate_topk(p, logits, 0, nullptr, T, ids, w, probs, gap, s);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : set_last_error(MOE_ERR_CUDA, cudaGetErrorString(e));
}
