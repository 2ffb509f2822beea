"""Seeded generators for every input of the routed-MoE slot-pool layer.

Recipe (the same for every consumer):
  * expert matrices W_gate, W_up, W_down ~ N(0, 0.02), stored as fp32, bf16
    (round-to-nearest-even) or fp8 e4m3 with one fp32 scale per 128x128 block
    (scale = block amax / 448, codes by torch's e4m3 conversion);
  * router weight W_r ~ N(0, 0.02) in the activation dtype; router bias
    b_e = -s * ln(rank_e) for a seeded permutation rank of 1..E (Zipf(s));
  * decode hidden states: an independent AR(1) stream per (layer, token lane),
    x_0 ~ N(0,1), x_t = rho * x_{t-1} + sqrt(1 - rho^2) * eps;
  * prefill hidden states: i.i.d. N(0,1);
  * initial slot fill: per layer a seeded random choice of its quota of experts.

Small cases are drawn with numpy (Philox) on the host; full-size weights are
drawn with torch's device generator (Philox) chunk by chunk, because tens of
GB cannot be drawn on the host in reasonable time.  Per-tensor seeds are a
hash of (workload, layer, tensor name, base seed).

Nothing here computes any part of the MoE layer; storage encodings (bf16
rounding, fp8 block quantisation) only produce the stored weights.
"""
import hashlib
import math

import numpy as np

from .configs import F32, BF16, FP8_E4M3_B128, RESPLIT_Q4R4, Workload, resplit_offsets

FP8_MAX = 448.0


def seed_for(wl_name: str, layer: int, tensor: str, base_seed: int = 0) -> int:
    h = hashlib.sha256(f"{wl_name}/{layer}/{tensor}/{base_seed}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def np_rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(seed))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Storage helper for generators only (widening is exact)."""
    return (b.astype(np.uint32) << 16).view(np.float32)


def quantize_fp8_blocks(w: np.ndarray):
    """fp32 [R, C] (R, C multiples of 128) -> (uint8 e4m3 codes [R,C], fp32 scales [R/128, C/128])."""
    import torch
    R, C = w.shape
    assert R % 128 == 0 and C % 128 == 0
    t = torch.from_numpy(np.ascontiguousarray(w, dtype=np.float32))
    blk = t.view(R // 128, 128, C // 128, 128)
    amax = blk.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    q = (blk / scale[:, None, :, None]).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    codes = q.view(torch.uint8).reshape(R, C).numpy().copy()
    return codes, scale.numpy().astype(np.float32)


# ----------------------------------------------------------------------------
# host (numpy) generators: small cases and everything the CPU tests touch
# ----------------------------------------------------------------------------

def expert_fp32(wl: Workload, layer: int, expert: int, base_seed: int = 0):
    """The three expert matrices as drawn (fp32, before storage rounding)."""
    g = np_rng(seed_for(wl.name, layer, f"expert{expert}", base_seed))
    w_gate = (g.standard_normal((wl.I, wl.H), dtype=np.float32) * np.float32(0.02))
    w_up = (g.standard_normal((wl.I, wl.H), dtype=np.float32) * np.float32(0.02))
    w_down = (g.standard_normal((wl.H, wl.I), dtype=np.float32) * np.float32(0.02))
    return w_gate, w_up, w_down


def quantize_groups(w: np.ndarray, bits: int):
    """Symmetric integer codes per 128-column group: scale = group amax / (2^(bits-1) - 1) (1 for an
    all-zero group), code = round-half-even(w / scale) clipped to +-(2^(bits-1) - 1).  fp32 arithmetic.
    Returns (int8 codes [R, C], fp32 scales [R, C/128])."""
    w = np.ascontiguousarray(w, np.float32)
    R, C = w.shape
    qmax = np.float32(2 ** (bits - 1) - 1)
    g = w.reshape(R, C // 128, 128)
    amax = np.abs(g).max(-1)
    scale = np.where(amax > 0, amax / qmax, np.float32(1.0)).astype(np.float32)
    q = np.clip(np.rint(g / scale[..., None]), -qmax, qmax).astype(np.int8)
    return q.reshape(R, C), scale


def resplit_encode(w13, w_down):
    """Residual-split storage (RapidMoE Alg. 3, own codec): gate/up as 4-bit codes W^Q and 4-bit codes of
    the residual W - W^Q (W^R); down as 4-bit (W^L) and 8-bit (W^H) codes.  W^Q = q * scale in fp32."""
    q13, sq13 = quantize_groups(w13, 4)
    deq = (q13.reshape(q13.shape[0], -1, 128).astype(np.float32) * sq13[..., None]).reshape(q13.shape)
    r13, sr13 = quantize_groups(np.asarray(w13, np.float32) - deq, 4)
    l2, sl2 = quantize_groups(w_down, 4)
    h2, sh2 = quantize_groups(w_down, 8)
    return {"q13": q13, "sq13": sq13, "r13": r13, "sr13": sr13, "l2": l2, "sl2": sl2, "h2": h2, "sh2": sh2}


def pack_int4(q: np.ndarray) -> np.ndarray:
    """int4 codes [R, C] (C even) -> bytes [R, C/2]: element 2j in the low nibble, 2j+1 in the high."""
    u = (np.asarray(q, np.int8).astype(np.uint8) & 0x0F)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def unpack_int4(b: np.ndarray, C: int) -> np.ndarray:
    """Inverse of pack_int4 (two's-complement nibbles)."""
    b = np.asarray(b, np.uint8)
    lo = (b & 0x0F).astype(np.int16)
    hi = (b >> 4).astype(np.int16)
    out = np.empty((b.shape[0], C), np.int16)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    out[out >= 8] -= 16
    return out.astype(np.int8)


def encode_expert(wl: Workload, w_gate, w_up, w_down):
    """Stored form of one expert: dict with w13 [2I,H], w2 [H,I] (+ s13, s2 for fp8)."""
    w13 = np.concatenate([w_gate, w_up], axis=0)
    if wl.weight_dtype == F32:
        return {"w13": w13.astype(np.float32), "w2": np.asarray(w_down, np.float32)}
    if wl.weight_dtype == BF16:
        return {"w13": f32_to_bf16_bits(w13), "w2": f32_to_bf16_bits(w_down)}
    if wl.weight_dtype == RESPLIT_Q4R4:
        return resplit_encode(w13, w_down)
    c13, s13 = quantize_fp8_blocks(w13)
    c2, s2 = quantize_fp8_blocks(w_down)
    return {"w13": c13, "w2": c2, "s13": s13, "s2": s2}


def expert_stored(wl: Workload, layer: int, expert: int, base_seed: int = 0):
    return encode_expert(wl, *expert_fp32(wl, layer, expert, base_seed))


def shared_expert_stored(wl: Workload, layer: int, base_seed: int = 0):
    g = np_rng(seed_for(wl.name, layer, "shared", base_seed))
    w_gate = g.standard_normal((wl.I, wl.H), dtype=np.float32) * np.float32(0.02)
    w_up = g.standard_normal((wl.I, wl.H), dtype=np.float32) * np.float32(0.02)
    w_down = g.standard_normal((wl.H, wl.I), dtype=np.float32) * np.float32(0.02)
    return encode_expert(wl, w_gate, w_up, w_down)


# --- the bf16 record format: 128 x 64 tiles in 128-byte-swizzled order -------
# Element (r, c) of a tile (row r < 128, column c < 64) sits at byte
# r*128 + ((c // 8) ^ (r % 8)) * 16 + (c % 8) * 2: each 128-byte row holds eight
# 16-byte chunks whose order is XOR-permuted by the row index mod 8.  Matrix
# rows/columns beyond the matrix are zero.

def _swz_perm():
    r = np.arange(128)[:, None]
    p = np.arange(8)[None, :]
    return p ^ (r % 8)                      # logical chunk held by physical chunk p of row r


def tile_sw128(w: np.ndarray) -> np.ndarray:
    """uint16 [R, C] -> uint16 [ceil(R/128), ceil(C/64), 128, 64] in swizzled tile order."""
    R, C = w.shape
    mt, kb = -(-R // 128), -(-C // 64)
    pad = np.zeros((mt * 128, kb * 64), np.uint16)
    pad[:R, :C] = w
    t = pad.reshape(mt, 128, kb, 64).transpose(0, 2, 1, 3).reshape(mt, kb, 128, 8, 8)
    idx = np.broadcast_to(_swz_perm()[None, None, :, :, None], t.shape)
    return np.take_along_axis(t, idx, axis=3).reshape(mt, kb, 128, 64)


def untile_sw128(tiles: np.ndarray, R: int, C: int) -> np.ndarray:
    """Inverse of tile_sw128."""
    mt, kb = tiles.shape[:2]
    t = tiles.reshape(mt, kb, 128, 8, 8)
    out = np.empty_like(t)
    perm = _swz_perm()
    for r in range(128):                    # physical chunk p holds logical chunk perm[r, p]
        out[:, :, r, perm[r], :] = t[:, :, r, :, :]
    return out.reshape(mt, kb, 128, 64).transpose(0, 2, 1, 3).reshape(mt * 128, kb * 64)[:R, :C]


def expert_record_bytes(wl: Workload, stored) -> bytes:
    """Pack one stored expert into the host-pool record layout (padded)."""
    o13, o2, os13, os2, rec = wl.expert_layout()
    buf = np.zeros(rec, np.uint8)
    if wl.weight_dtype == RESPLIT_Q4R4:
        o = resplit_offsets(wl.H, wl.I)
        parts = {"q13": pack_int4(stored["q13"]), "r13": pack_int4(stored["r13"]), "l2": pack_int4(stored["l2"]),
                 "h2": np.asarray(stored["h2"], np.int8).view(np.uint8)}
        for key in ("sq13", "sr13", "sl2", "sh2"):
            parts[key] = np.ascontiguousarray(stored[key], np.float32).view(np.uint8)
        for key, raw in parts.items():
            raw = np.ascontiguousarray(raw).reshape(-1)
            buf[o[key]:o[key] + raw.size] = raw
        return buf
    if wl.weight_dtype == BF16:
        I = wl.I
        g = tile_sw128(stored["w13"][:I])
        u = tile_sw128(stored["w13"][I:])
        w13 = np.stack([g, u], axis=2)      # [I/128][H/64][gate, up][128][64]
        w2 = tile_sw128(stored["w2"])       # [H/128][I/64][128][64]
        buf[o13:o13 + w13.nbytes] = w13.view(np.uint8).ravel()
        buf[o2:o2 + w2.nbytes] = w2.view(np.uint8).ravel()
        return buf
    for key, off in (("w13", o13), ("w2", o2), ("s13", os13), ("s2", os2)):
        if key in stored:
            raw = np.ascontiguousarray(stored[key]).view(np.uint8).ravel()
            buf[off:off + raw.size] = raw
    return buf


def zipf_bias(wl: Workload, layer: int, s: float, base_seed: int = 0) -> np.ndarray:
    """b_e = -s * ln(rank_e); rank is a seeded permutation of 1..E."""
    g = np_rng(seed_for(wl.name, layer, "rank", base_seed))
    rank = g.permutation(wl.E) + 1
    return (-s * np.log(rank.astype(np.float64))).astype(np.float32)


def router_stored(wl: Workload, layer: int, s=None, base_seed: int = 0):
    """(W_r stored [E,H] as fp32 or bf16 bits, bias fp32 [E])."""
    g = np_rng(seed_for(wl.name, layer, "router", base_seed))
    w = g.standard_normal((wl.E, wl.H), dtype=np.float32) * np.float32(0.02)
    b = zipf_bias(wl, layer, wl.zipf_s if s is None else s, base_seed)
    if wl.act_dtype == BF16:
        return f32_to_bf16_bits(w), b
    return w, b


def decode_hidden(wl: Workload, layer: int, T: int, steps: int, base_seed: int = 0):
    """AR(1) hidden states [steps, T, H] as drawn in fp32 (store with store_act)."""
    g = np_rng(seed_for(wl.name, layer, f"ar1_T{T}", base_seed))
    rho = np.float32(wl.ar_rho)
    c = np.float32(math.sqrt(1.0 - wl.ar_rho ** 2))
    out = np.empty((steps, T, wl.H), np.float32)
    x = g.standard_normal((T, wl.H), dtype=np.float32)
    for t in range(steps):
        if t > 0:
            x = rho * x + c * g.standard_normal((T, wl.H), dtype=np.float32)
        out[t] = x
    return out


def prefill_hidden(wl: Workload, layer: int, T: int, base_seed: int = 0):
    g = np_rng(seed_for(wl.name, layer, f"prefill_T{T}", base_seed))
    return g.standard_normal((T, wl.H), dtype=np.float32)


def store_act(wl: Workload, x: np.ndarray) -> np.ndarray:
    """Activation storage: fp32 as is, bf16 as uint16 bits."""
    if wl.act_dtype == BF16:
        return f32_to_bf16_bits(x)
    return np.ascontiguousarray(x, np.float32)


def initial_lut(wl: Workload, base_seed: int = 0, S=None) -> np.ndarray:
    """Per layer a seeded random quota(l) experts, slots handed out in draw order."""
    S = wl.S if S is None else S
    lut = np.full((wl.L, wl.E), -1, np.int32)
    nxt = 0
    base, extra = divmod(S, wl.L)
    for l in range(wl.L):
        q = min(base + (1 if l < extra else 0), wl.E)
        g = np_rng(seed_for(wl.name, l, "fill", base_seed))
        for e in g.permutation(wl.E)[:q]:
            lut[l, e] = nxt
            nxt += 1
    return lut


# ----------------------------------------------------------------------------
# device (torch) generators for full-size weights
# ----------------------------------------------------------------------------

def torch_expert_chunk(wl: Workload, layer: int, e0: int, n: int, device, base_seed: int = 0):
    """Draw experts [e0, e0+n) of one layer on `device`; returns (w13 [n,2I,H], w2 [n,H,I]) fp32."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(wl.name, layer, f"dev_experts{e0}_{n}", base_seed))
    w13 = torch.randn((n, 2 * wl.I, wl.H), generator=g, device=device, dtype=torch.float32).mul_(0.02)
    w2 = torch.randn((n, wl.H, wl.I), generator=g, device=device, dtype=torch.float32).mul_(0.02)
    return w13, w2


def torch_quantize_fp8_blocks(w):
    """Device version of quantize_fp8_blocks for [n, R, C] fp32 -> (uint8 [n,R,C], fp32 [n,R/128,C/128])."""
    import torch
    n, R, C = w.shape
    blk = w.view(n, R // 128, 128, C // 128, 128)
    amax = blk.abs().amax(dim=(2, 4))
    scale = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
    q = (blk / scale[:, :, None, :, None]).clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).reshape(n, R, C), scale.contiguous()


def torch_tile_sw128(w):
    """Device version of tile_sw128 for a batch [n, R, C] -> [n, R/128, C/64, 128, 64] (any 16-bit dtype)."""
    import torch
    n, R, C = w.shape
    mt, kb = -(-R // 128), -(-C // 64)
    pad = torch.zeros((n, mt * 128, kb * 64), dtype=w.dtype, device=w.device)
    pad[:, :R, :C] = w
    t = pad.view(n, mt, 128, kb, 64).permute(0, 1, 3, 2, 4).reshape(n, mt, kb, 128, 8, 8)
    perm = torch.from_numpy(_swz_perm()).to(w.device)
    idx = perm.view(1, 1, 1, 128, 8, 1).expand(n, mt, kb, 128, 8, 8)
    return torch.gather(t, 4, idx).reshape(n, mt, kb, 128, 64).contiguous()


def torch_quantize_groups(w, bits):
    """Device version of quantize_groups for [n, R, C] fp32 -> (int8 [n,R,C], fp32 [n,R,C/128])."""
    import torch
    n, R, C = w.shape
    qmax = float(2 ** (bits - 1) - 1)
    g = w.reshape(n, R, C // 128, 128)
    amax = g.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / qmax, torch.ones_like(amax))
    q = torch.round(g / scale[..., None]).clamp(-qmax, qmax).to(torch.int8)
    return q.reshape(n, R, C), scale.contiguous()


def torch_pack_int4(q):
    """[n, R, C] int8 codes -> [n, R, C/2] uint8, element 2j in the low nibble."""
    import torch
    u = q.view(torch.uint8) & 0x0F
    return (u[..., 0::2] | (u[..., 1::2] << 4)).contiguous()


def torch_encode_records(wl: Workload, w13, w2):
    """Stored records [n, record_bytes] uint8 on the device from fp32 w13/w2 chunks."""
    import torch
    n = w13.shape[0]
    o13, o2, os13, os2, rec = wl.expert_layout()
    out = torch.zeros((n, rec), dtype=torch.uint8, device=w13.device)
    if wl.weight_dtype == RESPLIT_Q4R4:
        o = resplit_offsets(wl.H, wl.I)
        q13, sq13 = torch_quantize_groups(w13, 4)
        deq = (q13.reshape(n, 2 * wl.I, -1, 128).float() * sq13[..., None]).reshape(w13.shape)
        r13, sr13 = torch_quantize_groups(w13 - deq, 4)
        l2, sl2 = torch_quantize_groups(w2, 4)
        h2, sh2 = torch_quantize_groups(w2, 8)
        parts = [("q13", torch_pack_int4(q13)), ("r13", torch_pack_int4(r13)), ("l2", torch_pack_int4(l2)),
                 ("h2", h2.view(torch.uint8)), ("sq13", sq13), ("sr13", sr13), ("sl2", sl2), ("sh2", sh2)]
        for key, t in parts:
            raw = t.contiguous().view(n, -1).view(torch.uint8)
            out[:, o[key]:o[key] + raw.shape[1]] = raw
        return out
    if wl.weight_dtype == F32:
        parts = [(o13, w13.contiguous()), (o2, w2.contiguous())]
    elif wl.weight_dtype == BF16:
        I = wl.I
        g = torch_tile_sw128(w13[:, :I].to(torch.bfloat16))
        u = torch_tile_sw128(w13[:, I:].to(torch.bfloat16))
        parts = [(o13, torch.stack([g, u], dim=3)), (o2, torch_tile_sw128(w2.to(torch.bfloat16)))]
    else:
        c13, s13 = torch_quantize_fp8_blocks(w13)
        c2, s2 = torch_quantize_fp8_blocks(w2)
        parts = [(o13, c13), (o2, c2), (os13, s13), (os2, s2)]
    for off, t in parts:
        raw = t.contiguous().view(n, -1).view(torch.uint8)
        out[:, off:off + raw.shape[1]] = raw
    return out


# ----------------------------------------------------------------------------
# whole-workload assembly (format only: record packing, no layer arithmetic)
# ----------------------------------------------------------------------------

def record_to_stored(wl: Workload, rec: np.ndarray):
    """Parse one host-pool record (uint8) back into the stored dict (w13, w2[, s13, s2])."""
    o13, o2, os13, os2, _ = wl.expert_layout()
    H, I = wl.H, wl.I
    if wl.weight_dtype == RESPLIT_Q4R4:
        o = resplit_offsets(H, I)

        def region(key, n, dt=np.uint8):
            return rec[o[key]:o[key] + n].view(dt)
        return {"q13": unpack_int4(region("q13", I * H).reshape(2 * I, H // 2), H),
                "r13": unpack_int4(region("r13", I * H).reshape(2 * I, H // 2), H),
                "l2": unpack_int4(region("l2", I * H // 2).reshape(H, I // 2), I),
                "h2": region("h2", I * H).view(np.int8).reshape(H, I).copy(),
                "sq13": region("sq13", 8 * I * (H // 128), np.float32).reshape(2 * I, H // 128).copy(),
                "sr13": region("sr13", 8 * I * (H // 128), np.float32).reshape(2 * I, H // 128).copy(),
                "sl2": region("sl2", 4 * H * (I // 128), np.float32).reshape(H, I // 128).copy(),
                "sh2": region("sh2", 4 * H * (I // 128), np.float32).reshape(H, I // 128).copy()}
    if wl.weight_dtype == BF16:
        mt_i, kb_h = -(-I // 128), -(-H // 64)
        mt_h, kb_i = -(-H // 128), -(-I // 64)
        w13 = rec[o13:o13 + 2 * mt_i * kb_h * 16384].view(np.uint16).reshape(mt_i, kb_h, 2, 128, 64)
        w2 = rec[o2:o2 + mt_h * kb_i * 16384].view(np.uint16).reshape(mt_h, kb_i, 128, 64)
        gate = untile_sw128(w13[:, :, 0], I, H)
        up = untile_sw128(w13[:, :, 1], I, H)
        return {"w13": np.concatenate([gate, up], axis=0).copy(), "w2": untile_sw128(w2, H, I).copy()}
    if wl.weight_dtype == F32:
        dt, eb = np.float32, 4
    elif wl.weight_dtype == BF16:
        dt, eb = np.uint16, 2
    else:
        dt, eb = np.uint8, 1
    out = {"w13": rec[o13:o13 + 2 * I * H * eb].view(dt).reshape(2 * I, H).copy(),
           "w2": rec[o2:o2 + H * I * eb].view(dt).reshape(H, I).copy()}
    if wl.weight_dtype == FP8_E4M3_B128:
        n13 = (2 * I // 128) * (H // 128)
        n2 = (H // 128) * (I // 128)
        out["s13"] = rec[os13:os13 + 4 * n13].view(np.float32).reshape(2 * I // 128, H // 128).copy()
        out["s2"] = rec[os2:os2 + 4 * n2].view(np.float32).reshape(H // 128, I // 128).copy()
    return out


def fill_host_pool(wl: Workload, host_u8, device=None, base_seed: int = 0, chunk: int = 16):
    """Write all L*E expert records into a host buffer (record (l, e) at (l*E+e)*record_bytes).

    host_u8: numpy uint8 view (device=None: numpy generator, per-expert seeds) or a
    torch uint8 CPU tensor (device given: torch generator on that device, per-chunk seeds).
    """
    rec = wl.expert_layout()[4]
    if device is None:
        for l in range(wl.L):
            for e in range(wl.E):
                off = (l * wl.E + e) * rec
                host_u8[off:off + rec] = expert_record_bytes(wl, expert_stored(wl, l, e, base_seed))
        return
    import torch
    for l in range(wl.L):
        recs = device_layer_records(wl, l, device, base_seed, chunk)
        off = l * wl.E * rec
        host_u8[off:off + wl.E * rec].copy_(recs.view(-1))
        del recs
    torch.cuda.synchronize(device)


def shared_records(wl: Workload, base_seed: int = 0) -> np.ndarray:
    """L shared-expert records, uint8 [L * record_bytes]."""
    return np.concatenate([expert_record_bytes(wl, shared_expert_stored(wl, l, base_seed)) for l in range(wl.L)])


def routers(wl: Workload, zipf_s=None, base_seed: int = 0):
    """(W_r stored [L, E, H], b fp32 [L, E]) for every layer."""
    ws, bs = zip(*(router_stored(wl, l, zipf_s, base_seed) for l in range(wl.L)))
    return np.stack(ws), np.stack(bs)


def device_layer_records(wl: Workload, layer: int, device, base_seed: int = 0, chunk: int = 16):
    """All E expert records of one layer drawn on `device` (same values fill_host_pool writes)."""
    import torch
    rec = wl.expert_layout()[4]
    out = torch.empty((wl.E, rec), dtype=torch.uint8, device=device)
    for e0 in range(0, wl.E, chunk):
        n = min(chunk, wl.E - e0)
        w13, w2 = torch_expert_chunk(wl, layer, e0, n, device, base_seed)
        out[e0:e0 + n] = torch_encode_records(wl, w13, w2)
    return out


def torch_decode_hidden(wl: Workload, T: int, steps: int, device, base_seed: int = 0, layers=None):
    """AR(1) hidden states for every layer on `device`: bf16/fp32 tensor [steps, L, T, H].

    x_0 ~ N(0,1); x_t = rho x_{t-1} + sqrt(1-rho^2) eps_t, one independent stream per (layer, token lane).
    """
    import torch
    L = wl.L if layers is None else layers
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(wl.name, -1, f"dev_ar1_T{T}", base_seed))
    dt = torch.bfloat16 if wl.act_dtype == BF16 else torch.float32
    out = torch.empty((steps, L, T, wl.H), dtype=dt, device=device)
    c = math.sqrt(1.0 - wl.ar_rho ** 2)
    x = torch.randn((L, T, wl.H), generator=g, device=device)
    for t in range(steps):
        if t > 0:
            x = wl.ar_rho * x + c * torch.randn((L, T, wl.H), generator=g, device=device)
        out[t] = x.to(dt)
    return out


def torch_prefill_hidden(wl: Workload, T: int, device, base_seed: int = 0, layers=None):
    """i.i.d. N(0,1) prefill hidden states on `device`: [L, T, H] in the activation dtype."""
    import torch
    L = wl.L if layers is None else layers
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(wl.name, -1, f"dev_prefill_T{T}", base_seed))
    dt = torch.bfloat16 if wl.act_dtype == BF16 else torch.float32
    return torch.randn((L, T, wl.H), generator=g, device=device).to(dt)
