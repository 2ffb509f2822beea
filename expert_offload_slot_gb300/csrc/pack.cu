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
#include <cstring>

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
