"""CPU oracle for the routed-MoE slot-pool layer — TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product path (the C-ABI library and its Python
binding) never calls it and shares no code with it.

What it computes, and from where:
  * ``numerics``  — exact decoding of stored weights (bf16, fp8 e4m3 with
    128x128 block scales).
  * ``layer``     — the top-k gated MoE layer: router projection, softmax- or
    sigmoid-renormalised gate, top-k, SwiGLU experts and the weighted combine
    (RapidMoE §2.1 and Eq. 7; CAP §II-A Eq. 1), in float64.  The top-k order is
    decided on float32 logits, the precision the kernels decide it in.
  * ``cache``     — the slot-pool simulator: expert_id -> slot_id lookup table,
    resident/missing detection, victim choice and the two routing-history
    eviction scores (MoE-CORE "Mechanism"; HybriMoE "Mechanism"; SeqMoE
    "Mechanism"), plus the permutation of token rows by expert.  Score
    arithmetic is float32 in a fixed order because it decides integer victim
    choices, exactly as the kernels do it.

Every function is written to be checked by eye against the pages; nothing is
blocked, fused or reordered beyond what the definitions state.
"""
