// Step a6: the device-started miss copy (SeqMoE "Mechanism": the device owns
// the cache metadata and starts the miss copy itself, from a kernel on the
// main stream, out of a pinned, mapped host pool, so a captured graph never
// waits for the host).  On GB300 the mapped host pool is read over
// NVLink-C2C with 16-byte loads; the slot is written with 16-byte stores.
//
// The copy list is produced on the device by the plan kernel, so the grid is
// fixed at launch: each CTA takes an equal share of every record.
#include "moeslot_internal.cuh"

namespace moeslot {

constexpr int kCopyThreads = 512;
constexpr int kCopyUnroll = 8;

// Every (job, 16-byte chunk) pair is one index of a flat space; each thread
// keeps kCopyUnroll independent loads from the host in flight before storing.
// The job of an index is idx / rec16, taken as the high word of idx * magic
// with magic = ceil(2^64 / rec16): exact for every idx < 2^32.
__global__ void __launch_bounds__(kCopyThreads)
miss_copy_kernel(const CopyJob* __restrict__ jobs, const int32_t* __restrict__ n_jobs, uint32_t rec16,
                 unsigned long long magic) {
  const uint32_t n = (uint32_t)*n_jobs;
  if (n == 0) return;
  const uint32_t total = n * rec16;
  const uint32_t stride = gridDim.x * kCopyThreads;
  for (uint32_t base = blockIdx.x * kCopyThreads + threadIdx.x; base < total; base += stride * kCopyUnroll) {
    uint4 v[kCopyUnroll];
    uint4* dst[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const uint32_t idx = base + u * stride;
      dst[u] = nullptr;
      if (idx < total) {
        const uint32_t j = (uint32_t)__umul64hi((unsigned long long)idx, magic);
        const uint32_t c = idx - j * rec16;
        v[u] = __ldcs(reinterpret_cast<const uint4*>(jobs[j].src) + c);
        dst[u] = reinterpret_cast<uint4*>(jobs[j].dst) + c;
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u)
      if (dst[u]) __stcs(dst[u], v[u]);
  }
}

int launch_miss_copy(const PoolDev& p, const Scratch& sc, cudaStream_t s, int ctas) {
  const uint32_t rec16 = (uint32_t)(p.lay.rec / 16);
  const unsigned long long magic = ~0ull / rec16 + 1ull;
  miss_copy_kernel<<<ctas > 0 ? ctas : 2 * sm_count(), kCopyThreads, 0, s>>>(sc.copies, sc.n_copy, rec16, magic);
  return 1;
}

// Host-initiated placement (moe_load_slot): one thread updates the table —
// the slot's occupant leaves, a previous slot of the expert becomes free, the
// slot's tag grows — and writes a one-element copy list for miss_copy_kernel.
__global__ void load_slot_kernel(PoolDev p, Scratch sc, int layer, int expert, int slot) {
  const int le = layer * p.E + expert;
  const int prev = p.lut[le];
  if (prev == slot) {
    *sc.n_copy = 0;
    return;
  }
  if (prev >= 0 && prev < p.S) p.owner[prev] = -1;
  const int occ = p.owner[slot];
  if (occ >= 0 && occ < p.L * p.E) p.lut[occ] = -1;
  p.owner[slot] = le;
  p.lut[le] = slot;
  p.tag[slot] += 1u;
  sc.copies[0].src = p.host_dev + (size_t)le * p.lay.rec;
  sc.copies[0].dst = p.records + (size_t)slot * p.lay.rec;
  *sc.n_copy = 1;
}

int launch_load_slot(const PoolDev& p, const Scratch& sc, int layer, int expert, int slot, cudaStream_t s) {
  load_slot_kernel<<<1, 1, 0, s>>>(p, sc, layer, expert, slot);
  return 1;
}

// After a whole-table upload: every occupied slot got a new occupant.
__global__ void rebuild_owner_kernel(PoolDev p) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s < p.S && p.owner[s] >= 0) p.tag[s] += 1u;
}

int launch_rebuild_owner(const PoolDev& p, cudaStream_t s) {
  rebuild_owner_kernel<<<(p.S + 255) / 256, 256, 0, s>>>(p);
  return 1;
}

}  // namespace moeslot
