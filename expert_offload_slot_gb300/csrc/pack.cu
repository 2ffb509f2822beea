// moe_pack_expert_record: host-side packing of one expert from plain row-major
// matrices into the record format the pool's kernels read (declared in
// include/moeslot.h).  Host code only: no CUDA call, no allocation.
//
// bf16 records are cut into 128-row x 64-column tiles stored in the order the
// tensor cores' 128-byte-swizzled shared-memory operand layout reads them, so
// that one pipeline stage of the expert kernels is one contiguous bulk copy:
//   element (r, c) of a tile sits at byte r*128 + ((c/8) XOR (r mod 8))*16 + (c mod 8)*2;
//   w13 holds tiles [ceil(I/128)][ceil(H/64)][gate, up], w2 tiles [ceil(H/128)][ceil(I/64)];
//   rows and columns beyond the matrix are zero.
// fp32 and fp8 records are row-major (fp8 followed by its 128x128 block scales).
// Residual-split records (RapidMoE §4.4 Alg. 3, with the codec defined in the
// header) are encoded here from fp32 matrices: symmetric integer codes per
// 128-column group, scale = group amax / (2^(bits-1) - 1), code =
// round-half-even(w / scale), all in fp32 (this file is compiled without
// floating-point contraction, so each operation rounds once).
#include <cmath>
#include <cstring>
#include <vector>

#include "moeslot_internal.cuh"

namespace {

constexpr size_t kTileBytes = 128 * 64 * 2;

// byte offset of element (r, c) inside one swizzled 128 x 64 bf16 tile
inline size_t tile_byte(size_t r, size_t c) { return r * 128 + (((c >> 3) ^ (r & 7)) << 4) + (c & 7) * 2; }

// scatter a row-major bf16 matrix [R, C] into tiles; tile (mt, kb) starts at base + tile_off(mt, kb)
template <typename F>
void scatter_tiles(uint8_t* base, const uint16_t* m, size_t R, size_t C, F tile_off) {
  for (size_t i = 0; i < R; ++i)
    for (size_t j = 0; j < C; ++j) {
      uint8_t* t = base + tile_off(i / 128, j / 64);
      std::memcpy(t + tile_byte(i % 128, j % 64), m + i * C + j, 2);
    }
}

// codes [R][C] and scales [R][C/128] of a row-major fp32 matrix
void quant_groups(const float* w, size_t R, size_t C, int bits, std::vector<int8_t>& q, std::vector<float>& sc) {
  const float qmax = (float)((1 << (bits - 1)) - 1);
  q.assign(R * C, 0);
  sc.assign(R * (C / 128), 1.f);
  for (size_t r = 0; r < R; ++r)
    for (size_t g = 0; g < C / 128; ++g) {
      const float* src = w + r * C + g * 128;
      float amax = 0.f;
      for (int j = 0; j < 128; ++j) amax = std::fmax(amax, std::fabs(src[j]));
      const float scale = amax > 0.f ? amax / qmax : 1.f;
      sc[r * (C / 128) + g] = scale;
      for (int j = 0; j < 128; ++j) {
        float v = std::nearbyint(src[j] / scale);
        v = std::fmin(std::fmax(v, -qmax), qmax);
        q[r * C + g * 128 + j] = (int8_t)v;
      }
    }
}

void put_nibbles(uint8_t* dst, const std::vector<int8_t>& q) {
  for (size_t j = 0; j < q.size() / 2; ++j)
    dst[j] = (uint8_t)((q[2 * j] & 0x0F) | ((q[2 * j + 1] & 0x0F) << 4));
}

void pack_resplit(uint8_t* out, const float* w_gate, const float* w_up, const float* w_down, size_t H, size_t I) {
  const size_t IH = I * H;
  std::vector<float> w13(2 * IH);
  std::memcpy(w13.data(), w_gate, IH * sizeof(float));
  std::memcpy(w13.data() + IH, w_up, IH * sizeof(float));
  std::vector<int8_t> q13, r13, l2, h2;
  std::vector<float> sq13, sr13, sl2, sh2;
  quant_groups(w13.data(), 2 * I, H, 4, q13, sq13);
  std::vector<float> res(2 * IH);
  for (size_t i = 0; i < 2 * I; ++i)
    for (size_t h = 0; h < H; ++h) {
      const float deq = (float)q13[i * H + h] * sq13[i * (H / 128) + h / 128];
      res[i * H + h] = w13[i * H + h] - deq;
    }
  quant_groups(res.data(), 2 * I, H, 4, r13, sr13);
  quant_groups(w_down, H, I, 4, l2, sl2);
  quant_groups(w_down, H, I, 8, h2, sh2);
  const size_t s13 = 2 * I * (H / 128) * 4, s2 = H * (I / 128) * 4;
  uint8_t* p = out;
  put_nibbles(p, q13);
  put_nibbles(p + IH, r13);
  put_nibbles(p + 2 * IH, l2);
  std::memcpy(p + 2 * IH + IH / 2, h2.data(), IH);
  uint8_t* sp = p + 3 * IH + IH / 2;
  std::memcpy(sp, sq13.data(), s13);
  std::memcpy(sp + s13, sr13.data(), s13);
  std::memcpy(sp + 2 * s13, sl2.data(), s2);
  std::memcpy(sp + 2 * s13 + s2, sh2.data(), s2);
}

}  // namespace

MOE_API moe_status moe_pack_expert_record(const moe_config* cfg, const void* w_gate, const void* w_up,
                                          const void* w_down, const float* s_gate, const float* s_up,
                                          const float* s_down, void* record, size_t record_bytes) {
  size_t off13 = 0, off2 = 0, offs13 = 0, offs2 = 0, rec = 0;
  moe_status st = moe_expert_layout(cfg, &off13, &off2, &offs13, &offs2, &rec);
  if (st != MOE_OK) return st;
  if (!w_gate || !w_up || !w_down || !record)
    return moeslot::set_last_error(MOE_ERR_INVALID, "moe_pack_expert_record: NULL matrix or record");
  if (record_bytes < rec)
    return moeslot::set_last_error(MOE_ERR_INVALID, "moe_pack_expert_record: record buffer shorter than record_bytes");
  const int wdt = cfg->weight_dtype;
  if (wdt == MOE_FP8_E4M3_B128 && (!s_gate || !s_up || !s_down))
    return moeslot::set_last_error(MOE_ERR_INVALID, "moe_pack_expert_record: fp8 records need the block scales");
  const size_t H = cfg->hidden, I = cfg->inter;
  uint8_t* out = static_cast<uint8_t*>(record);
  std::memset(out, 0, rec);
  if (wdt == MOE_RESPLIT_Q4R4) {
    pack_resplit(out, static_cast<const float*>(w_gate), static_cast<const float*>(w_up),
                 static_cast<const float*>(w_down), H, I);
    return MOE_OK;
  }
  if (wdt == MOE_BF16) {
    const size_t kb_h = (H + 63) / 64, kb_i = (I + 63) / 64;
    const uint16_t* g = static_cast<const uint16_t*>(w_gate);
    const uint16_t* u = static_cast<const uint16_t*>(w_up);
    const uint16_t* d = static_cast<const uint16_t*>(w_down);
    scatter_tiles(out + off13, g, I, H, [&](size_t mt, size_t kb) { return ((mt * kb_h + kb) * 2 + 0) * kTileBytes; });
    scatter_tiles(out + off13, u, I, H, [&](size_t mt, size_t kb) { return ((mt * kb_h + kb) * 2 + 1) * kTileBytes; });
    scatter_tiles(out + off2, d, H, I, [&](size_t mt, size_t kb) { return (mt * kb_i + kb) * kTileBytes; });
    return MOE_OK;
  }
  const size_t eb = wdt == MOE_F32 ? 4 : 1;
  std::memcpy(out + off13, w_gate, I * H * eb);
  std::memcpy(out + off13 + I * H * eb, w_up, I * H * eb);
  std::memcpy(out + off2, w_down, H * I * eb);
  if (wdt == MOE_FP8_E4M3_B128) {
    const size_t n_half = (I / 128) * (H / 128);
    std::memcpy(out + offs13, s_gate, n_half * 4);
    std::memcpy(out + offs13 + n_half * 4, s_up, n_half * 4);
    std::memcpy(out + offs2, s_down, (H / 128) * (I / 128) * 4);
  }
  return MOE_OK;
}
