// Steps a8 (SwiGLU experts) and a9 (weighted combine) for the memory-bound
// token counts of decode.
//
// Expert (RapidMoE §4.5, Eq. 7): y = W_down (SiLU(W_gate x) ⊙ W_up x), SiLU on
// the gate projection only.  Combine (CAP §II-A, Eq. 1; RapidMoE Table 2):
// out[t] = sum_j w[t, j] * y_j(t) (+ the shared expert with weight 1).
//
// With a handful of tokens per expert the layer streams U expert records from
// HBM once and does a few FMAs per weight: the bound is HBM bandwidth.  Two
// kernels:
//   gate_up : every warp owns a contiguous, balanced range of (expert, row i)
//             pairs over all active experts; it streams gate row i and up row
//             I+i once with 16-byte loads and serves every token of that expert
//             from L1, writing h = SiLU(g) * u for each token row.
//   down    : every CTA owns a block of output features; for each active expert
//             in ascending id (shared expert last) it streams those W_down rows
//             once and accumulates w * (W_down h) per token in shared memory.
//             The combine is therefore fused, deterministic and atomic-free.
// Weights may be fp32, bf16, or fp8 e4m3 with 128x128 fp32 block scales (the
// scale multiplies each 16-element partial dot product, which stays inside
// one 128-wide block), or residual-split codes (RapidMoE §4.4 Alg. 3): 4-bit
// W^Q and W^R for gate/up, 4-bit W^L or 8-bit W^H for down, fp32 scales per
// 128-column group.  A critical expert (UMIA, RapidMoE §4.3) reads W^Q and
// W^R (each weight q * sq + r * sr, fp32) and W^H_down; the others read W^Q
// and W^L_down only.
#include <cuda_fp8.h>

#include "moeslot_internal.cuh"

namespace moeslot {

struct FfnArgs {
  const WorkEntry* work;
  const int32_t* n_work;
  const void* x;
  const int32_t* perm_tok;
  const float* perm_w;
  void* h;
  void* out;
  int H, I, T;
  size_t off13, off2, offs13, offs2;
  size_t offr13, offh2, offsr13, offsh2;   // residual-split records
  const int32_t* sel;        // residual-split gate/up: the work positions to process (null: all)
  const int32_t* sel_count;
};

template <typename WT> struct WTraits;
template <> struct WTraits<float> {
  static constexpr int CW = 4;
  static constexpr bool kScaled = false;
  __device__ __forceinline__ static void cvt(const uint4& q, float* v) {
    v[0] = __uint_as_float(q.x); v[1] = __uint_as_float(q.y);
    v[2] = __uint_as_float(q.z); v[3] = __uint_as_float(q.w);
  }
};
template <> struct WTraits<uint16_t> {
  static constexpr int CW = 8;
  static constexpr bool kScaled = false;
  __device__ __forceinline__ static void cvt(const uint4& q, float* v) {
    v[0] = bf16lo(q.x); v[1] = bf16hi(q.x); v[2] = bf16lo(q.y); v[3] = bf16hi(q.y);
    v[4] = bf16lo(q.z); v[5] = bf16hi(q.z); v[6] = bf16lo(q.w); v[7] = bf16hi(q.w);
  }
};
template <> struct WTraits<uint8_t> {   // fp8 e4m3 codes
  static constexpr int CW = 16;
  static constexpr bool kScaled = true;
  __device__ __forceinline__ static void pair(uint32_t w, float* v) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
    const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
  }
  __device__ __forceinline__ static void cvt(const uint4& q, float* v) {
    pair(q.x, v); pair(q.y, v + 4); pair(q.z, v + 8); pair(q.w, v + 12);
  }
};

// N activation elements starting at p (16-byte aligned) as fp32.
template <typename AT, int N> struct Act;
template <int N> struct Act<float, N> {
  __device__ __forceinline__ static void load(const float* p, float* v) {
#pragma unroll
    for (int q = 0; q < N / 4; ++q) {
      const float4 f = *reinterpret_cast<const float4*>(p + 4 * q);
      v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
    }
  }
  __device__ __forceinline__ static void store1(float* p, float v) { *p = v; }
};
template <int N> struct Act<uint16_t, N> {
  __device__ __forceinline__ static void load(const uint16_t* p, float* v) {
#pragma unroll
    for (int q = 0; q < N / 8; ++q) {
      const uint4 u = *reinterpret_cast<const uint4*>(p + 8 * q);
      v[8 * q + 0] = bf16lo(u.x); v[8 * q + 1] = bf16hi(u.x);
      v[8 * q + 2] = bf16lo(u.y); v[8 * q + 3] = bf16hi(u.y);
      v[8 * q + 4] = bf16lo(u.z); v[8 * q + 5] = bf16hi(u.z);
      v[8 * q + 6] = bf16lo(u.w); v[8 * q + 7] = bf16hi(u.w);
    }
    if constexpr (N % 8 == 4) {   // a last 8-byte group
      const uint2 u = *reinterpret_cast<const uint2*>(p + N - 4);
      v[N - 4] = bf16lo(u.x); v[N - 3] = bf16hi(u.x);
      v[N - 2] = bf16lo(u.y); v[N - 1] = bf16hi(u.y);
    }
  }
  __device__ __forceinline__ static void store1(uint16_t* p, float v) { *p = f32_to_bf16_rn(v); }
};

__device__ __forceinline__ float silu(float a) { return a / (1.f + expf(-a)); }

constexpr int kFfnWarps = 8;
constexpr int kTokChunk = 8;    // tokens served per pass over a weight row

template <typename WT, typename AT>
__global__ void __launch_bounds__(kFfnWarps * 32)
ffn_gate_up_kernel(FfnArgs a) {
  constexpr int CW = WTraits<WT>::CW;
  constexpr int UNR = CW == 16 ? 2 : 4;
  constexpr int NT = kTokChunk;
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kFfnWarps + (threadIdx.x >> 5);
  const int nw = gridDim.x * kFfnWarps;
  const int n_work = *a.n_work;
  const int H = a.H, I = a.I;
  const long long total = (long long)n_work * I;
  const long long p0 = total * gw / nw, p1 = total * (gw + 1) / nw;
  const AT* __restrict__ x = static_cast<const AT*>(a.x);
  AT* __restrict__ hout = static_cast<AT*>(a.h);

  for (long long pp = p0; pp < p1; ++pp) {
    const int u = (int)(pp / I), i = (int)(pp % I);
    const WorkEntry ent = a.work[u];
    const WT* __restrict__ gate = reinterpret_cast<const WT*>(ent.rec + a.off13) + (size_t)i * H;
    const WT* __restrict__ up = gate + (size_t)I * H;
    const float* sg = nullptr;
    const float* su = nullptr;
    if constexpr (WTraits<WT>::kScaled) {
      const float* s13 = reinterpret_cast<const float*>(ent.rec + a.offs13);
      sg = s13 + (size_t)(i / 128) * (H / 128);
      su = s13 + (size_t)((I + i) / 128) * (H / 128);
    }
    for (int tc = 0; tc < ent.n; tc += NT) {
      const int nr = min(NT, ent.n - tc);
      int tok[NT];
#pragma unroll
      for (int r = 0; r < NT; ++r) tok[r] = r < nr ? a.perm_tok[ent.row0 + tc + r] : 0;
      float ag[NT], au[NT];
#pragma unroll
      for (int r = 0; r < NT; ++r) { ag[r] = 0.f; au[r] = 0.f; }
      for (int h0 = lane * CW; h0 < H; h0 += 32 * CW * UNR) {
        uint4 rg[UNR], ru[UNR];
#pragma unroll
        for (int q = 0; q < UNR; ++q) {
          const int h = h0 + q * 32 * CW;
          if (h < H) {
            rg[q] = __ldcs(reinterpret_cast<const uint4*>(gate + h));
            ru[q] = __ldcs(reinterpret_cast<const uint4*>(up + h));
          }
        }
#pragma unroll
        for (int q = 0; q < UNR; ++q) {
          const int h = h0 + q * 32 * CW;
          if (h < H) {
            float wg[CW], wu[CW];
            WTraits<WT>::cvt(rg[q], wg);
            WTraits<WT>::cvt(ru[q], wu);
            float gs = 1.f, us = 1.f;
            if constexpr (WTraits<WT>::kScaled) { gs = sg[h / 128]; us = su[h / 128]; }
#pragma unroll
            for (int r = 0; r < NT; ++r) {
              if (r < nr) {
                float xv[CW];
                Act<AT, CW>::load(x + (size_t)tok[r] * H + h, xv);
                float dg = 0.f, du = 0.f;
#pragma unroll
                for (int c = 0; c < CW; ++c) { dg = fmaf(wg[c], xv[c], dg); du = fmaf(wu[c], xv[c], du); }
                if constexpr (WTraits<WT>::kScaled) { ag[r] = fmaf(gs, dg, ag[r]); au[r] = fmaf(us, du, au[r]); }
                else { ag[r] += dg; au[r] += du; }
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < NT; ++r) {
        if (r < nr) {
          const float g = warp_sum(ag[r]);
          const float uu = warp_sum(au[r]);
          if (lane == 0) Act<AT, 8>::store1(hout + (size_t)(ent.row0 + tc + r) * I + i, silu(g) * uu);
        }
      }
    }
  }
}

// ---------------------------------------------------------------- residual-split records
// 8 two's-complement nibbles of a little-endian word: element k is bits 4k .. 4k+3.
__device__ __forceinline__ void nib8(uint32_t w, float* v) {
#pragma unroll
  for (int k = 0; k < 8; ++k) v[k] = (float)((int)(w << (28 - 4 * k)) >> 28);
}
__device__ __forceinline__ void int8x4(uint32_t w, float* v) {
#pragma unroll
  for (int k = 0; k < 4; ++k) v[k] = (float)((int)(w << (24 - 8 * k)) >> 24);
}
// 32 weights of one 16-byte chunk of nibbles: q * sq (+ r * sr for a critical entry), fp32
__device__ __forceinline__ void decode32(const uint4& q, float sq, const uint4& r, float sr, bool crit, float* w) {
  const uint32_t wq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    nib8(wq[j], w + 8 * j);
#pragma unroll
    for (int k = 0; k < 8; ++k) w[8 * j + k] *= sq;
  }
  if (crit) {
    const uint32_t wr[4] = {r.x, r.y, r.z, r.w};
    float c[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      nib8(wr[j], c);
#pragma unroll
      for (int k = 0; k < 8; ++k) w[8 * j + k] = fmaf(c[k], sr, w[8 * j + k]);
    }
  }
}

// gate/up: the work is (entry, chunk of NT tokens, row i) units, entries in order, each entry's
// units chunk-major; every warp owns a contiguous, equal range of units, so an entry with many
// tokens (the shared expert) spreads over many warps.  Each lane takes 32 columns (16 bytes of
// codes) at a time and decodes them once for the unit's tokens.
template <typename AT>
__global__ void __launch_bounds__(kFfnWarps * 32, 2)
ffn_resplit_gate_up_kernel(FfnArgs a) {
  constexpr int NT = 4;   // tokens per unit: four keep the kernel at two CTAs per SM
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kFfnWarps + (threadIdx.x >> 5);
  const int nw = gridDim.x * kFfnWarps;
  const int n_work = a.sel ? *a.sel_count : *a.n_work;   // the selected entries, or all
  auto entry = [&](int j) -> const WorkEntry& { return a.work[a.sel ? a.sel[j] : j]; };
  const int H = a.H, I = a.I;
  long long total = 0;
  for (int u = 0; u < n_work; ++u) total += (long long)((entry(u).n + NT - 1) / NT) * I;
  const long long p0 = total * gw / nw, p1 = total * (gw + 1) / nw;
  const AT* __restrict__ x = static_cast<const AT*>(a.x);
  AT* __restrict__ hout = static_cast<AT*>(a.h);
  const int G = H / 128;
  int u = 0;
  long long base = 0;                            // first unit of entry u
  for (long long pp = p0; pp < p1; ++pp) {
    while (u < n_work && pp >= base + (long long)((entry(u).n + NT - 1) / NT) * I) {
      base += (long long)((entry(u).n + NT - 1) / NT) * I;
      ++u;
    }
    if (u >= n_work) break;
    const WorkEntry ent = entry(u);
    const long long local = pp - base;
    const int tc = (int)(local / I) * NT, i = (int)(local % I);
    const bool crit = ent.crit != 0;
    const uint8_t* qg = ent.rec + a.off13 + (size_t)i * (H / 2);
    const uint8_t* qu = ent.rec + a.off13 + (size_t)(I + i) * (H / 2);
    const uint8_t* rg = ent.rec + a.offr13 + (size_t)i * (H / 2);
    const uint8_t* ru = ent.rec + a.offr13 + (size_t)(I + i) * (H / 2);
    const float* sqg = reinterpret_cast<const float*>(ent.rec + a.offs13) + (size_t)i * G;
    const float* squ = reinterpret_cast<const float*>(ent.rec + a.offs13) + (size_t)(I + i) * G;
    const float* srg = reinterpret_cast<const float*>(ent.rec + a.offsr13) + (size_t)i * G;
    const float* sru = reinterpret_cast<const float*>(ent.rec + a.offsr13) + (size_t)(I + i) * G;
    const int nr = min(NT, ent.n - tc);
    int tok[NT];
#pragma unroll
    for (int r = 0; r < NT; ++r) tok[r] = r < nr ? a.perm_tok[ent.row0 + tc + r] : 0;
    float ag[NT], au[NT];
#pragma unroll
    for (int r = 0; r < NT; ++r) { ag[r] = 0.f; au[r] = 0.f; }
    for (int h = lane * 32; h < H; h += 32 * 32) {
      const uint4 cqg = __ldcs(reinterpret_cast<const uint4*>(qg + h / 2));
      const uint4 cqu = __ldcs(reinterpret_cast<const uint4*>(qu + h / 2));
      uint4 crg = make_uint4(0u, 0u, 0u, 0u), cru = crg;
      if (crit) {
        crg = __ldcs(reinterpret_cast<const uint4*>(rg + h / 2));
        cru = __ldcs(reinterpret_cast<const uint4*>(ru + h / 2));
      }
      float wg[32], wu[32];
      decode32(cqg, sqg[h / 128], crg, crit ? srg[h / 128] : 0.f, crit, wg);
      decode32(cqu, squ[h / 128], cru, crit ? sru[h / 128] : 0.f, crit, wu);
#pragma unroll
      for (int r = 0; r < NT; ++r) {
        if (r < nr) {
          float xv[32];
          Act<AT, 32>::load(x + (size_t)tok[r] * H + h, xv);
          float dg = 0.f, du = 0.f;
#pragma unroll
          for (int c = 0; c < 32; ++c) { dg = fmaf(wg[c], xv[c], dg); du = fmaf(wu[c], xv[c], du); }
          ag[r] += dg;
          au[r] += du;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < NT; ++r) {
      if (r < nr) {
        const float g = warp_sum(ag[r]);
        const float uu = warp_sum(au[r]);
        if (lane == 0) Act<AT, 8>::store1(hout + (size_t)(ent.row0 + tc + r) * I + i, silu(g) * uu);
      }
    }
  }
}

constexpr int kDownRowsPerWarp = 2;
constexpr int kDownRows = kFfnWarps * kDownRowsPerWarp;   // output features per CTA

template <typename WT, typename AT>
__global__ void __launch_bounds__(kFfnWarps * 32)
ffn_down_combine_kernel(FfnArgs a) {
  constexpr int CW = WTraits<WT>::CW;
  constexpr int NT = kTokChunk;
  constexpr int RPW = kDownRowsPerWarp;
  extern __shared__ float acc_s[];   // [kDownRows][T]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, I = a.I, T = a.T;
  const int h0 = blockIdx.x * kDownRows;
  for (int j = threadIdx.x; j < kDownRows * T; j += blockDim.x) acc_s[j] = 0.f;
  __syncthreads();
  const int n_work = *a.n_work;
  const AT* __restrict__ hin = static_cast<const AT*>(a.h);
  int hr[RPW];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) hr[rr] = min(h0 + warp * RPW + rr, H - 1);
  for (int u = 0; u < n_work; ++u) {
    const WorkEntry ent = a.work[u];
    const WT* __restrict__ w2 = reinterpret_cast<const WT*>(ent.rec + a.off2);
    const float* s2 = nullptr;
    if constexpr (WTraits<WT>::kScaled) s2 = reinterpret_cast<const float*>(ent.rec + a.offs2);
    for (int tc = 0; tc < ent.n; tc += NT) {
      const int nr = min(NT, ent.n - tc);
      float acc[RPW][NT];
#pragma unroll
      for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
        for (int r = 0; r < NT; ++r) acc[rr][r] = 0.f;
      for (int i0 = lane * CW; i0 < I; i0 += 32 * CW) {
        float wv[RPW][CW];
        float sc[RPW];
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
          const uint4 q = __ldcs(reinterpret_cast<const uint4*>(w2 + (size_t)hr[rr] * I + i0));
          WTraits<WT>::cvt(q, wv[rr]);
          sc[rr] = 1.f;
          if constexpr (WTraits<WT>::kScaled) sc[rr] = s2[(size_t)(hr[rr] / 128) * (I / 128) + i0 / 128];
        }
#pragma unroll
        for (int r = 0; r < NT; ++r) {
          if (r < nr) {
            float hv[CW];
            Act<AT, CW>::load(hin + (size_t)(ent.row0 + tc + r) * I + i0, hv);
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) {
              float d = 0.f;
#pragma unroll
              for (int c = 0; c < CW; ++c) d = fmaf(wv[rr][c], hv[c], d);
              if constexpr (WTraits<WT>::kScaled) acc[rr][r] = fmaf(sc[rr], d, acc[rr][r]);
              else acc[rr][r] += d;
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < NT; ++r) {
        if (r < nr) {
          const int row = ent.row0 + tc + r;
          const int t = a.perm_tok[row];
          const float wgt = a.perm_w[row];
#pragma unroll
          for (int rr = 0; rr < RPW; ++rr) {
            const float v = warp_sum(acc[rr][r]);
            if (lane == 0 && h0 + warp * RPW + rr < H) {
              float* dst = &acc_s[(warp * RPW + rr) * T + t];
              *dst = *dst + wgt * v;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  AT* __restrict__ out = static_cast<AT*>(a.out);
  for (int j = threadIdx.x; j < kDownRows * T; j += blockDim.x) {
    const int t = j / kDownRows, rr = j % kDownRows;
    if (h0 + rr < H) Act<AT, 8>::store1(out + (size_t)t * H + h0 + rr, acc_s[rr * T + t]);
  }
}

// down + combine for residual-split records: as ffn_down_combine_kernel, reading W^H_down (8-bit,
// 16 columns per lane chunk) for a critical entry and W^L_down (4-bit, 32 columns) otherwise
template <typename AT>
__global__ void __launch_bounds__(kFfnWarps * 32, 3)
ffn_resplit_down_kernel(FfnArgs a) {
  constexpr int NT = kTokChunk;
  constexpr int RPW = kDownRowsPerWarp;
  extern __shared__ float acc_s[];   // [kDownRows][T]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H, I = a.I, T = a.T;
  const int h0 = blockIdx.x * kDownRows;
  for (int j = threadIdx.x; j < kDownRows * T; j += blockDim.x) acc_s[j] = 0.f;
  __syncthreads();
  const int n_work = *a.n_work;
  const AT* __restrict__ hin = static_cast<const AT*>(a.h);
  const int G = I / 128;
  int hr[RPW];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) hr[rr] = min(h0 + warp * RPW + rr, H - 1);
  for (int u = 0; u < n_work; ++u) {
    const WorkEntry ent = a.work[u];
    const bool crit = ent.crit != 0;
    const uint8_t* w2 = ent.rec + (crit ? a.offh2 : a.off2);
    const float* s2 = reinterpret_cast<const float*>(ent.rec + (crit ? a.offsh2 : a.offs2));
    const int cw = crit ? 16 : 32;                 // columns per 16-byte chunk
    const size_t row_bytes = crit ? (size_t)I : (size_t)I / 2;
    for (int tc = 0; tc < ent.n; tc += NT) {
      const int nr = min(NT, ent.n - tc);
      float acc[RPW][NT];
#pragma unroll
      for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
        for (int r = 0; r < NT; ++r) acc[rr][r] = 0.f;
      for (int i0 = lane * cw; i0 < I; i0 += 32 * cw) {
        uint32_t w[RPW][4];
        float sc[RPW];
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr) {
          const uint4 q = __ldcs(reinterpret_cast<const uint4*>(w2 + (size_t)hr[rr] * row_bytes + (crit ? (size_t)i0 : (size_t)i0 / 2)));
          w[rr][0] = q.x;
          w[rr][1] = q.y;
          w[rr][2] = q.z;
          w[rr][3] = q.w;
          sc[rr] = s2[(size_t)hr[rr] * G + i0 / 128];
        }
        // one word of codes at a time (few registers, so more warps per SM): each (row, token)
        // product still runs over the chunk's columns in ascending order
        float d[RPW][NT];
#pragma unroll
        for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
          for (int r = 0; r < NT; ++r) d[rr][r] = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float wv[RPW][8];
#pragma unroll
          for (int rr = 0; rr < RPW; ++rr) {
            if (crit) int8x4(w[rr][j], wv[rr]);
            else nib8(w[rr][j], wv[rr]);
          }
#pragma unroll
          for (int r = 0; r < NT; ++r) {
            if (r < nr) {
              float hv[8];
              const AT* hp = hin + (size_t)(ent.row0 + tc + r) * I + i0;
              if (crit) {
                Act<AT, 4>::load(hp + 4 * j, hv);
#pragma unroll
                for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
                  for (int c = 0; c < 4; ++c) d[rr][r] = fmaf(wv[rr][c], hv[c], d[rr][r]);
              } else {
                Act<AT, 8>::load(hp + 8 * j, hv);
#pragma unroll
                for (int rr = 0; rr < RPW; ++rr)
#pragma unroll
                  for (int c = 0; c < 8; ++c) d[rr][r] = fmaf(wv[rr][c], hv[c], d[rr][r]);
              }
            }
          }
        }
#pragma unroll
        for (int r = 0; r < NT; ++r)
          if (r < nr)
#pragma unroll
            for (int rr = 0; rr < RPW; ++rr) acc[rr][r] = fmaf(sc[rr], d[rr][r], acc[rr][r]);
      }
#pragma unroll
      for (int r = 0; r < NT; ++r) {
        if (r < nr) {
          const int row = ent.row0 + tc + r;
          const int t = a.perm_tok[row];
          const float wgt = a.perm_w[row];
#pragma unroll
          for (int rr = 0; rr < RPW; ++rr) {
            const float v = warp_sum(acc[rr][r]);
            if (lane == 0 && h0 + warp * RPW + rr < H) {
              float* dst = &acc_s[(warp * RPW + rr) * T + t];
              *dst = *dst + wgt * v;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  AT* __restrict__ out = static_cast<AT*>(a.out);
  for (int j = threadIdx.x; j < kDownRows * T; j += blockDim.x) {
    const int t = j / kDownRows, rr = j % kDownRows;
    if (h0 + rr < H) Act<AT, 8>::store1(out + (size_t)t * H + h0 + rr, acc_s[rr * T + t]);
  }
}

static FfnArgs ffn_args(const PoolDev& p, const Scratch& sc, int T, const void* x, void* out) {
  FfnArgs a;
  a.work = sc.work;
  a.n_work = sc.n_work;
  a.x = x;
  a.perm_tok = sc.perm_tok;
  a.perm_w = sc.perm_w;
  a.h = sc.h;
  a.out = out;
  a.H = p.H;
  a.I = p.I;
  a.T = T;
  a.off13 = p.lay.off13;
  a.off2 = p.lay.off2;
  a.offs13 = p.lay.offs13;
  a.offs2 = p.lay.offs2;
  a.offr13 = p.lay.offr13;
  a.offh2 = p.lay.offh2;
  a.offsr13 = p.lay.offsr13;
  a.offsh2 = p.lay.offsh2;
  a.sel = nullptr;
  a.sel_count = nullptr;
  return a;
}

int launch_ffn_gate_up(const PoolDev& p, const Scratch& sc, int T, const void* x, cudaStream_t s, int part) {
  FfnArgs a = ffn_args(p, sc, T, x, nullptr);
  if (part >= 0 && p.wdt == MOE_RESPLIT_Q4R4) {
    a.sel = sc.elist + (size_t)part * (p.E + 1);
    a.sel_count = sc.ecount + part;
  }
  const int grid = 2 * sm_count();
  if (p.wdt == MOE_F32) ffn_gate_up_kernel<float, float><<<grid, kFfnWarps * 32, 0, s>>>(a);
  else if (p.wdt == MOE_BF16) ffn_gate_up_kernel<uint16_t, uint16_t><<<grid, kFfnWarps * 32, 0, s>>>(a);
  else if (p.wdt == MOE_RESPLIT_Q4R4) ffn_resplit_gate_up_kernel<uint16_t><<<grid, kFfnWarps * 32, 0, s>>>(a);
  else ffn_gate_up_kernel<uint8_t, uint16_t><<<grid, kFfnWarps * 32, 0, s>>>(a);
  return 1;
}

template <typename WT, typename AT>
static void launch_down_t(const FfnArgs& a, int T, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    cudaFuncSetAttribute(ffn_down_combine_kernel<WT, AT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         200 * 1024);
    configured = true;
  }
  const size_t smem = (size_t)kDownRows * T * sizeof(float);
  ffn_down_combine_kernel<WT, AT><<<(a.H + kDownRows - 1) / kDownRows, kFfnWarps * 32, smem, s>>>(a);
}

int launch_ffn_down(const PoolDev& p, const Scratch& sc, int T, void* out, cudaStream_t s) {
  const FfnArgs a = ffn_args(p, sc, T, nullptr, out);
  if (p.wdt == MOE_F32) {
    launch_down_t<float, float>(a, T, s);
  } else if (p.wdt == MOE_BF16) {
    launch_down_t<uint16_t, uint16_t>(a, T, s);
  } else if (p.wdt == MOE_RESPLIT_Q4R4) {
    static bool configured = false;
    if (!configured) {
      cudaFuncSetAttribute(ffn_resplit_down_kernel<uint16_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           200 * 1024);
      configured = true;
    }
    const size_t smem = (size_t)kDownRows * T * sizeof(float);
    ffn_resplit_down_kernel<uint16_t><<<(a.H + kDownRows - 1) / kDownRows, kFfnWarps * 32, smem, s>>>(a);
  } else {
    launch_down_t<uint8_t, uint16_t>(a, T, s);
  }
  return 1;
}

}  // namespace moeslot
