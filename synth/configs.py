"""The five workload shapes of the routed-MoE slot-pool layer.

Each entry fixes the layer shape (layers L, routed experts E, top-k, hidden H,
expert intermediate I), the stored dtypes, the gating form, the slot-pool size
S and the synthetic input recipe (router-bias Zipf exponent, AR(1) drift of
decode hidden states, token counts).  Shapes are those of Qwen3-30B-A3B,
DeepSeek-V3 and Mixtral-8x7B MoE layers plus a tiny fp32 case; weights are
random, never a real checkpoint.
"""
from dataclasses import dataclass, field
from typing import Tuple

# dtype codes shared with the C ABI header (moeslot.h): values only, no logic.
F32, BF16, FP8_E4M3_B128, RESPLIT_Q4R4 = 0, 1, 2, 3
GATE_SOFTMAX_RENORM, GATE_SIGMOID_RENORM = 0, 1
EVICT_CORE, EVICT_MRS, EVICT_LRU = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    L: int                  # MoE layers
    E: int                  # routed experts per layer
    k: int                  # top-k
    H: int                  # hidden size
    I: int                  # expert intermediate size
    weight_dtype: int       # F32 / BF16 / FP8_E4M3_B128
    act_dtype: int          # F32 / BF16
    gating: int             # GATE_*
    residency: float        # fraction of the L*E experts that have a slot
    zipf_s: float           # router bias b_e = -s * ln(rank_e)
    evict: int = EVICT_CORE
    window: int = 16
    shared: bool = False
    decode_T: Tuple[int, ...] = ()
    decode_steps: int = 0
    prefill_T: Tuple[int, ...] = ()
    prefill_zipf_s: float = 0.0
    ar_rho: float = 0.8
    fixed_slots: int = 0    # slot count given outright (overrides residency)
    notes: str = field(default="", compare=False)

    @property
    def S(self) -> int:
        """Slot count: given outright, else round(residency * L * E)."""
        if self.fixed_slots:
            return self.fixed_slots
        return int(round(self.residency * self.L * self.E))

    def quota(self, layer: int) -> int:
        """Initial per-layer share of the pool: floor(S/L), +1 for the first S mod L layers."""
        base, extra = divmod(self.S, self.L)
        return base + (1 if layer < extra else 0)

    @property
    def weight_elt_bytes(self) -> int:
        return {F32: 4, BF16: 2, FP8_E4M3_B128: 1, RESPLIT_Q4R4: 1}[self.weight_dtype]

    @property
    def act_elt_bytes(self) -> int:
        return {F32: 4, BF16: 2}[self.act_dtype]

    def expert_layout(self):
        """Byte offsets of one expert's record.

        Returns (w13_off, w2_off, s13_off, s2_off, record_bytes).  fp32 and fp8
        records hold w13 [2I,H] and w2 [H,I] row-major (fp8 followed by its block
        scales).  bf16 records hold the same matrices cut into 128-row x 64-column
        tiles (see synth.gen.tile_sw128): w13 as [I/128][H/64][gate, up] tiles and
        w2 as [H/128][I/64] tiles, 16 KiB each.  Records are padded to 4096 bytes.
        """
        eb = self.weight_elt_bytes
        if self.weight_dtype == RESPLIT_Q4R4:
            # [q13 | r13 | l2 | h2 | sq13 | sr13 | sl2 | sh2]: 4-bit codes two per byte, 8-bit codes,
            # fp32 scales per 128-column group; (w13_off, w2_off, s13_off, s2_off) = (q13, l2, sq13, sl2)
            o = resplit_offsets(self.H, self.I)
            return o["q13"], o["l2"], o["sq13"], o["sl2"], o["record"]
        if self.weight_dtype == BF16:
            mt_i, kb_h = -(-self.I // 128), -(-self.H // 64)
            mt_h, kb_i = -(-self.H // 128), -(-self.I // 64)
            w13 = 2 * mt_i * kb_h * 16384
            w2 = mt_h * kb_i * 16384
            return 0, w13, w13 + w2, w13 + w2, (w13 + w2 + 4095) // 4096 * 4096
        w13 = 2 * self.I * self.H * eb
        w2 = self.H * self.I * eb
        s13 = s2 = 0
        if self.weight_dtype == FP8_E4M3_B128:
            s13 = (2 * self.I // 128) * (self.H // 128) * 4
            s2 = (self.H // 128) * (self.I // 128) * 4
        off13, off2 = 0, w13
        offs13, offs2 = w13 + w2, w13 + w2 + s13
        raw = w13 + w2 + s13 + s2
        rec = (raw + 4095) // 4096 * 4096
        return off13, off2, offs13, offs2, rec


def resplit_offsets(H, I):
    """Byte offsets of the residual-split record's regions and its padded size."""
    IH = I * H
    sizes = [("q13", IH), ("r13", IH), ("l2", IH // 2), ("h2", IH), ("sq13", 2 * I * (H // 128) * 4),
             ("sr13", 2 * I * (H // 128) * 4), ("sl2", H * (I // 128) * 4), ("sh2", H * (I // 128) * 4)]
    off, out = 0, {}
    for name, n in sizes:
        out[name] = off
        off += n
    out["record"] = (off + 4095) // 4096 * 4096
    return out


WORKLOADS = {
    "tiny": Workload(
        name="tiny", L=1, E=8, k=2, H=256, I=128, weight_dtype=F32, act_dtype=F32,
        gating=GATE_SOFTMAX_RENORM, residency=0.5, fixed_slots=4, zipf_s=0.5,
        decode_T=(4,), decode_steps=8, notes="1 layer, 4 slots holding a seeded random 4 experts"),
    "qwen3_decode": Workload(
        name="qwen3_decode", L=48, E=128, k=8, H=2048, I=768, weight_dtype=BF16, act_dtype=BF16,
        gating=GATE_SOFTMAX_RENORM, residency=0.45, zipf_s=1.0, evict=EVICT_MRS,
        decode_T=(1, 4, 16), decode_steps=256),
    "qwen3_prefill": Workload(
        name="qwen3_prefill", L=48, E=128, k=8, H=2048, I=768, weight_dtype=BF16, act_dtype=BF16,
        gating=GATE_SOFTMAX_RENORM, residency=0.45, zipf_s=0.0, prefill_T=(512, 2048),
        prefill_zipf_s=0.0, notes="router bias 0 so that all 128 experts receive tokens"),
    "dsv3": Workload(
        name="dsv3", L=4, E=256, k=8, H=7168, I=2048, weight_dtype=FP8_E4M3_B128, act_dtype=BF16,
        gating=GATE_SIGMOID_RENORM, residency=0.40, zipf_s=1.2, shared=True, evict=EVICT_MRS,
        decode_T=(1, 8, 32), decode_steps=64, prefill_T=(1024,), prefill_zipf_s=1.2),
    "mixtral": Workload(
        name="mixtral", L=32, E=8, k=2, H=4096, I=14336, weight_dtype=BF16, act_dtype=BF16,
        gating=GATE_SOFTMAX_RENORM, residency=0.25, fixed_slots=64, zipf_s=0.0,
        evict=EVICT_MRS, decode_T=(1,), decode_steps=512, prefill_T=(32, 256, 1024)),
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]
