#!/usr/bin/env python
"""Benchmark of the slot-pool MoE layer on GB300.

Workload (default): the Qwen3-30B-A3B-shaped decode — 48 MoE layers, hidden
2048, 128 experts, top-8, intermediate 768, bf16 weights and activations, a
shared slot pool of round(0.45 * 48 * 128) = 2765 slots, Zipf(s=1.0) router
bias, AR(1) (rho = 0.8) drift of the hidden states, Minus-Recent-Score eviction
(HybriMoE; on this trace it misses less often than the MoE-CORE score or LRU).
Weights are random (seeded), never a checkpoint.

One "step" is one decode step of T tokens through all 48 layers: every stage
of the layer (router, gate/top-k, history, table, victims, device-started miss
copies, permutation, expert FFN, combine) runs in the library's kernels, the
48 moe_forward calls being captured once into a CUDA graph.  The metric is
MoE-layer tokens/s = (steps * T * 48) / elapsed.

Printed (rank 0, one JSON line): value (inputs already in HBM), e2e (same
metric through the C ABI with host buffers: per-step pinned H2D of x and D2H of
the output inside the timed region), roofline of the dominant kernel (the decode
layer kernel, timed per launch with CUDA events in a profiling pass of the same
workload), layer_floor (the layer-step's bound from HBM bytes and miss records
over the measured host link), clocks sampled with nvidia-smi during the timed
region, the other decode batches (sweep) and workload shapes (configs), and the
CPU oracle timed on a bounded sample as cpu_baseline.

--impl reference times the CPU oracle itself on the same workload and prints
the same line with "impl": "reference".
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The CPU oracle's BLAS thread count, fixed before numpy loads: every host core this process may
# run on, unless the caller set it (the one-thread baseline runs in a child with it set to 1).
HOST_CORES = len(os.sched_getaffinity(0))
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(HOST_CORES))
ORACLE_THREADS = int(os.environ["OPENBLAS_NUM_THREADS"])

WORKLOAD_LABEL = {"qwen3_decode": "qwen3-30b-a3b-shaped-decode"}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="qwen3_decode")
    ap.add_argument("--batch", type=int, default=16, help="decode tokens per step (headline)")
    ap.add_argument("--sweep", default="1,4", help="other decode batches reported under 'sweep' ('' for none)")
    ap.add_argument("--prof-steps", type=int, default=32)
    ap.add_argument("--cpu-sample", type=int, default=32, help="oracle layer-steps in cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling only: run the workload's layer shape with fewer layers (0 = all)")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling only: the workload's expert shape with this many routed experts (0 = all)")
    ap.add_argument("--top-k", type=int, default=0, help="profiling only: top-k with --experts (0 = the workload's)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--configs",
                    default="qwen3_hit,s_independence,prefetch,quotas,aes,qwen3_prefill,dsv3,dsv3_resplit,mixtral",
                    help="other workloads measured at N=1 and reported under 'configs' ('' for none)")
    ap.add_argument("--probe-link", action="store_true",
                    help="measure the host->GPU link: device-started record copies vs DMA, then exit")
    ap.add_argument("--prefill", type=int, default=0,
                    help="only a staged prefill of this many tokens through the workload's layers (with --layers: "
                         "fewer layers of the same shape); prints one JSON line of its measurement, then exits")
    ap.add_argument("--cpu-sample-only", type=int, default=0,
                    help="internal: time the oracle on this many layer-steps, print one JSON line, exit")
    return ap.parse_args()


def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce_device():
    import torch.distributed as dist
    return "cuda" if dist.get_backend() == "nccl" else "cpu"


def max_over_ranks(v, world):
    """Slowest rank's value (replicas: the job takes as long as its slowest GPU)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=_reduce_device())
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v, world):
    """Work done by all replicas together."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=_reduce_device())
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        # nvidia-smi numbers GPUs physically; the device's UUID names the one this process uses
        self.idx = gpu_index
        try:
            import torch
            self.idx = "GPU-" + str(torch.cuda.get_device_properties(gpu_index).uuid)
        except Exception:
            pass
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in out.strip().splitlines():
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], "measured"
    return 6800.0, "fallback"


def load_tc_peak():
    """Dense bf16 TFLOP/s: measured burst figure, else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f)["bf16_tflops"]
    return 1900.0


def sources_digest(paths):
    """sha256 over the named source files (relative to the repo root), in the given order."""
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(rel.encode() + b"\0" + f.read())
    return h.hexdigest()


def captured_traffic(kernel):
    """DRAM bytes (read + write) per launch of `kernel` from its committed ncu capture, or None.

    The capture file records a digest of the kernel's sources; once they change the counters no
    longer describe the kernel and the traffic is reported as unknown."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    try:
        if sources_digest(d["sources"]) != d["sources_sha256"]:
            return None
    except OSError:
        return None
    return d["dram_bytes_per_launch"]


# ------------------------------------------------------------------ our arm
def host_chunk(wl):
    """Experts drawn per device chunk when filling a host pool (bounded fp32 temporaries, ~3 GB)."""
    per = 3 * wl.H * wl.I * 4
    return max(1, min(16, (3 << 30) // per))


class PoolBench:
    """One slot pool over a pinned host pool, driven through the C ABI.

    host: an already-filled HostPool to share (its weights are those of `host_wl`), else one is
    allocated and filled with this workload's weights.  slots overrides the slot count (L*E gives the
    all-resident hit path).  staging adds the two layer-sized prefill regions.
    """

    def __init__(self, wl, max_T, device, host=None, slots=None, staging=False, lut=None):
        import numpy as np
        import torch

        import expert_offload_slot_gb300 as moe
        from synth import gen
        self.moe, self.wl, self.device = moe, wl, device
        self.rec = wl.expert_layout()[4]
        self.S = wl.S if slots is None else slots
        self.cfg = moe.make_config(wl.L, wl.E, wl.k, wl.H, wl.I, self.S, wl.weight_dtype, wl.act_dtype, wl.gating,
                                   wl.shared, wl.evict, wl.window, 0.9, (0.25, 0.25, 0.25, 0.25),
                                   2 if staging else 0, max_T)
        t0 = time.time()
        self.own_host = host is None
        if host is None:
            host = moe.HostPool(wl.L * wl.E * self.rec)
            gen.fill_host_pool(wl, host.torch(), device=device, chunk=host_chunk(wl))
        self.host = host
        w_r, b = gen.routers(wl)
        wr = w_r.view(np.int16) if wl.act_dtype == 1 else w_r
        self.w_r = torch.from_numpy(np.ascontiguousarray(wr)).to(device)
        self.b = torch.from_numpy(b).to(device)
        self.shared = torch.from_numpy(gen.shared_records(wl)).to(device) if wl.shared else None
        self.pool = moe.Pool(self.cfg, self.host.ptr, self.host.nbytes, self.w_r, self.b, self.shared,
                             device=torch.cuda.current_device())
        self.pool.set_lut(gen.initial_lut(wl, S=self.S) if lut is None else lut)
        torch.cuda.synchronize()
        self.setup_s = time.time() - t0

    def capture(self, x_in, out, stream):
        import torch
        n0 = self.pool.launch_count()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(self.wl.L):
                self.pool.forward(l, x_in[l], out[l], self.moe.MOE_MODE_DECODE)
        return g, self.pool.launch_count() - n0

    def decode(self, T, W, K, prof_steps, clocks=None, world=1, e2e=True):
        """W warm-up and K timed decode steps (one CUDA graph of L moe_forward calls per step)."""
        import torch
        wl, moe = self.wl, self.moe
        dev = self.device
        # one AR(1) trace: warm-up [0, W), timed [W, W+K), profiling pass after it, then the
        # end-to-end pass on steps of its own (never a replay of steps the pool has already seen)
        P = prof_steps if prof_steps > 0 else 0
        xs = __import__("synth").gen.torch_decode_hidden(wl, T, W + K + P + (K if e2e else 0), dev)
        s = torch.cuda.Stream()
        x_in = torch.empty((wl.L, T, wl.H), dtype=xs.dtype, device=dev)
        out = torch.empty_like(x_in)
        with torch.cuda.stream(s):
            x_in.copy_(xs[0])
            for l in range(wl.L):                    # one eager step before capture
                self.pool.forward(l, x_in[l], out[l], moe.MOE_MODE_DECODE)
        s.synchronize()
        g, launches_per_step = self.capture(x_in, out, s)
        with torch.cuda.stream(s):
            for i in range(W):
                x_in.copy_(xs[i])
                g.replay()
        s.synchronize()
        st0 = self.pool.stats()
        barrier(world)
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nq = 4 if K >= 8 else 1                   # quarters of the timed region, for the spread
        bounds = [j * K // nq for j in range(nq + 1)]
        evq = [torch.cuda.Event(enable_timing=True) for _ in range(nq + 1)]
        if clocks:
            clocks.start()
        with torch.cuda.stream(s):
            ev0.record(s)
            evq[0].record(s)
            for i in range(W, W + K):
                x_in.copy_(xs[i])
                g.replay()
                if i - W + 1 in bounds[1:]:
                    evq[bounds.index(i - W + 1, 1)].record(s)
            ev1.record(s)
        s.synchronize()
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
        q_ms = [(evq[j].elapsed_time(evq[j + 1]), bounds[j + 1] - bounds[j]) for j in range(nq)]
        clk = clocks.stop() if clocks else None
        barrier(world)
        st1 = self.pool.stats()
        res = {"T": T, "ms": ms, "steps": K, "launches_per_step": launches_per_step, "quarter_ms": q_ms,
               "hits": st1["hits"] - st0["hits"], "misses": st1["misses"] - st0["misses"],
               "bytes_copied": st1["bytes_copied"] - st0["bytes_copied"], "clocks": clk,
               "prefetch": {n: st1["prefetch_" + n] - st0["prefetch_" + n]
                            for n in ("issued", "committed", "demanded", "bytes")},
               "critical_entries": st1["critical_entries"] - st0["critical_entries"],
               "aes_substitutions": st1["aes_substitutions"] - st0["aes_substitutions"]}
        res["status"] = self.pool.status()
        # profiling pass: per-stage CUDA-event times of every layer, same workload continued
        res["prof"] = self.profile_decode(xs[W + K:W + K + P], x_in, out, s, T, prof_steps) if prof_steps > 0 else \
            {"launches": 0, "stage_ms": [0.0] * self.moe.MOE_NUM_STAGES, "sum_U": 0, "T": T, "bytes_copied": 0}
        if e2e:
            res["e2e"] = self.run_e2e(xs[W + K + P:], g, x_in, out, s, K)
        del g
        return res

    def _collect(self, stage, n):
        for l in range(self.wl.L):
            v = self.pool.profile_read(l)
            for i in range(len(stage)):
                stage[i] += v[i]
            n += 1
        return n

    def profile_decode(self, xs, x_in, out, s, T, P):
        import torch
        wl = self.wl
        self.pool.profile_enable(True)
        gp, _ = self.capture(x_in, out, s)
        stage = [0.0] * self.moe.MOE_NUM_STAGES
        st0 = self.pool.stats()
        n = 0
        for i in range(P):
            with torch.cuda.stream(s):
                x_in.copy_(xs[i % xs.shape[0]])
                gp.replay()
            s.synchronize()
            n = self._collect(stage, n)
        st1 = self.pool.stats()
        self.pool.profile_enable(False)
        del gp
        U = (st1["hits"] - st0["hits"]) + (st1["misses"] - st0["misses"])
        if wl.shared:
            U += n                              # the shared expert is streamed by every launch
        return {"launches": n, "stage_ms": stage, "sum_U": U, "T": T,
                "bytes_copied": st1["bytes_copied"] - st0["bytes_copied"]}

    def prefill(self, T, W, K, prof_steps=1):
        """Staged prefill of T tokens through all L layers (two swapped layer-sized staging regions,
        layer l+1 copied while l computes), eager launches: W warm-up and K timed steps."""
        import torch
        wl, moe = self.wl, self.moe
        x = __import__("synth").gen.torch_prefill_hidden(wl, T, self.device)
        out = torch.empty_like(x)
        s = torch.cuda.Stream()

        def step():
            for l in range(wl.L):
                self.pool.forward(l, x[l], out[l], moe.MOE_MODE_PREFILL_STAGED, stream=s)

        link_now = {"fresh_buffer_GBps": dma_probe(), "pool_buffer_GBps": dma_probe(self.host)}
        for _ in range(W):
            step()
        s.synchronize()
        st0 = self.pool.stats()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        ev0.record(s)
        for _ in range(K):
            step()
        ev1.record(s)
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
        st1 = self.pool.stats()
        self.pool.profile_enable(True)
        stage, n = [0.0] * moe.MOE_NUM_STAGES, 0
        for _ in range(prof_steps):
            step()
            s.synchronize()
            n = self._collect(stage, n)
        self.pool.profile_enable(False)
        return {"T": T, "ms": ms, "steps": K, "status": self.pool.status(), "link_now": link_now,
                "staged": st1["staged_layers"] - st0["staged_layers"],
                "prof": {"launches": n, "stage_ms": stage}}

    def run_e2e(self, xs, g, x_in, out, s, K):
        """Same metric through the C ABI with host buffers: H2D of x and D2H of out every step, on K
        steps of the trace that follow every step the pool has run so far."""
        import torch
        x_host = xs[:K].cpu().pin_memory()
        out_host = torch.empty_like(x_host).pin_memory()
        torch.cuda.synchronize()
        st0 = self.pool.stats()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            ev0.record(s)
            for i in range(K):
                x_in.copy_(x_host[i], non_blocking=True)
                g.replay()
                out_host[i].copy_(out, non_blocking=True)
            ev1.record(s)
        s.synchronize()
        ms = ev0.elapsed_time(ev1)
        st1 = self.pool.stats()
        nb = x_in.numel() * x_in.element_size()
        hits, misses = st1["hits"] - st0["hits"], st1["misses"] - st0["misses"]
        return {"ms": ms, "h2d": nb, "d2h": nb, "hit_rate": hits / max(1, hits + misses),
                "misses": misses, "steps": K}

    def decode_repeat(self, T, W, K):
        """W + K decode steps that all route the same hidden state (one step of the AR(1) trace):
        after the first step the table holds every expert the step needs, so the timed steps are
        pure hit-path forwards whatever the slot count."""
        import torch
        wl, moe = self.wl, self.moe
        xs = __import__("synth").gen.torch_decode_hidden(wl, T, 1, self.device)
        s = torch.cuda.Stream()
        x_in = xs[0].clone()
        out = torch.empty_like(x_in)
        g, _ = self.capture(x_in, out, s)
        with torch.cuda.stream(s):
            for _ in range(W):
                g.replay()
        s.synchronize()
        st0 = self.pool.stats()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            ev0.record(s)
            for _ in range(K):
                g.replay()
            ev1.record(s)
        s.synchronize()
        st1 = self.pool.stats()
        del g
        hits, misses = st1["hits"] - st0["hits"], st1["misses"] - st0["misses"]
        return {"slots": self.S, "us_per_layer": ev0.elapsed_time(ev1) * 1e3 / (K * wl.L), "steps": K,
                "hit_rate": hits / max(1, hits + misses), "status": moe_status_name(self.pool.status())}

    def close(self, keep_host=False):
        self.pool.close()
        if self.own_host and not keep_host:
            self.host.free()


def dma_probe(host=None, nbytes=1 << 30):
    """Host -> GPU DMA GB/s of one copy of nbytes: from a freshly pinned buffer, or from the start of
    an existing host pool."""
    import torch
    if host is None:
        src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    else:
        nbytes = min(nbytes, host.nbytes)
        src = host.torch()[:nbytes]
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    dst.copy_(src, non_blocking=True)
    ev1.record()
    torch.cuda.synchronize()
    return nbytes / (ev0.elapsed_time(ev1) / 1e3) / 1e9


def expert_bytes(wl):
    """Stored bytes of one expert's three matrices (3*H*I elements, plus fp8 block scales)."""
    be = 3 * wl.H * wl.I * wl.weight_elt_bytes
    if wl.weight_dtype == 2:
        be += 3 * (wl.H // 128) * (wl.I // 128) * 4
    return be


def ffn_algorithmic_bytes(wl, sum_U, bytes_copied, layer_steps, T, router=False):
    """HBM bytes the expert kernel must move: the U expert records it reads, the miss bytes it
    writes into slots, x in / out once per layer-step, and (router=True, when the router runs in
    the same kernel) the router matrix once per layer-step."""
    b = sum_U * expert_bytes(wl) + bytes_copied + layer_steps * 2 * T * wl.H * wl.act_elt_bytes
    if router:
        b += layer_steps * wl.E * wl.H * wl.act_elt_bytes
    return b


def fused_layer(stage_ms):
    """True when the profile attributes the whole layer to the expert stage (one decode layer kernel)."""
    import expert_offload_slot_gb300 as moe
    return stage_ms[moe.STAGES.index("ffn")] > 0 and all(
        stage_ms[moe.STAGES.index(n)] == 0 for n in ("route", "plan", "copy"))


KERNEL_LABEL = {True: "tc_decode_layer_kernel (router, gate, plan, miss copies, gate/up, down, combine)",
                False: "tc_fused_decode_kernel (miss copies + gate/up + down + combine)"}


def kernel_label(wl, fused, T):
    """The decode FFN kernel a call of T tokens runs: fp32 weights take the CUDA-core streaming
    kernels, bf16 single-token decode layer calls the CUDA-core streaming variant of the layer kernel,
    everything else the tensor-core kernels."""
    if wl.weight_dtype == 0:
        return "ffn_gate_up_kernel + ffn_down_combine_kernel"
    if fused and wl.weight_dtype == 1 and T == 1:
        return "tc_decode_layer_kernel, streaming FFN variant (router, gate, plan, miss copies, gate/up, down)"
    return KERNEL_LABEL[fused]


def layer_floor(layer_bytes, miss_bytes, us_per_layer, hbm_gbs, link_gbs):
    """Lower bound on a decode layer-step's time from its two streams, which can overlap: the
    algorithmic HBM bytes at the measured HBM copy peak, and the miss records at the measured host
    link rate (None when the link was not measured).  frac = floor / measured time."""
    hbm_us = layer_bytes / (hbm_gbs * 1e9) * 1e6
    link_us = miss_bytes / (link_gbs * 1e9) * 1e6 if link_gbs else None
    floor = max(hbm_us, link_us or 0.0)
    return {"hbm_us": hbm_us, "link_us": link_us, "floor_us": floor, "us_per_layer": us_per_layer,
            "frac": floor / us_per_layer if us_per_layer > 0 else 0.0, "link_GBps": link_gbs,
            "bound": "link" if link_us is not None and link_us > hbm_us else "hbm"}


def step_bytes(wl, U_per_layer, T):
    """Algorithmic HBM bytes of one layer-step: router + U expert records + x in and out."""
    return wl.E * wl.H * wl.act_elt_bytes + U_per_layer * expert_bytes(wl) + 2 * T * wl.H * wl.act_elt_bytes


def prefill_flops(wl, T):
    """Routed expert FLOPs of one layer (2*T*k*3*H*I), the shared expert's, and the router's."""
    f = 2 * T * wl.k * 3 * wl.H * wl.I + 2 * T * wl.H * wl.E
    if wl.shared:
        f += 2 * T * 3 * wl.H * wl.I
    return f


def prefetch_summary(wl, r, base=None):
    """Per layer-step: demand misses, prefetches issued / committed / demanded before their commit,
    and the bytes over the host link (demand copies + prefetch copies), next to tokens/s."""
    n = r["steps"] * wl.L
    pf = r["prefetch"]
    out = {"tokens_per_s": r["steps"] * r["T"] * wl.L / (r["ms"] / 1e3), "us_per_layer": r["ms"] * 1e3 / n,
           "hit_rate": r["hits"] / max(1, r["hits"] + r["misses"]), "demand_misses_per_layer_step": r["misses"] / n,
           "prefetch_issued_per_layer_step": pf["issued"] / n, "prefetch_committed_per_layer_step": pf["committed"] / n,
           "prefetch_demanded_per_layer_step": pf["demanded"] / n,
           "link_MB_per_layer_step": (r["bytes_copied"] + pf["bytes"]) / 1e6 / n, "status": moe_status_name(r["status"])}
    if base is not None:
        out["vs_no_prefetch"] = out["tokens_per_s"] / base["tokens_per_s"]
    return out


def decode_summary(wl, r, peak):
    """Per-config decode line: tokens/s, us/layer, hit rate, per-stage us, FFN-kernel HBM roofline."""
    import expert_offload_slot_gb300 as moe
    prof = r["prof"]
    n = max(1, prof["launches"])
    ffn_ms = prof["stage_ms"][moe.STAGES.index("ffn")] + prof["stage_ms"][moe.STAGES.index("copy")]
    fused = fused_layer(prof["stage_ms"])
    ffn_b = ffn_algorithmic_bytes(wl, prof["sum_U"], prof["bytes_copied"], prof["launches"], r["T"], router=fused)
    ach = ffn_b / (ffn_ms / 1e3) / 1e9 if ffn_ms > 0 else 0.0
    U = prof["sum_U"] / n
    lay_us = sum(prof["stage_ms"]) * 1e3 / n
    return {"T": r["T"], "tokens_per_s": r["steps"] * r["T"] * wl.L / (r["ms"] / 1e3),
            "us_per_layer": r["ms"] * 1e3 / (r["steps"] * wl.L), "steps": r["steps"],
            "hit_rate": r["hits"] / max(1, r["hits"] + r["misses"]),
            "miss_MB_per_layer": r["bytes_copied"] / 1e6 / (r["steps"] * wl.L),
            "mean_U": U, "stage_us_per_layer": {k: v * 1e3 / n for k, v in zip(moe.STAGES, prof["stage_ms"])},
            "ffn_roofline": {"bound": "hbm", "kernel": kernel_label(wl, fused, r["T"]),
                             "achieved": ach, "unit": "GB/s", "frac": ach / peak,
                             "bytes_per_launch": ffn_b / n, "us_per_launch": ffn_ms * 1e3 / n},
            "layer_frac": step_bytes(wl, U, r["T"]) / (lay_us * 1e-6) / 1e9 / peak if lay_us else 0.0,
            "status": moe_status_name(r["status"]), "clocks": r.get("clocks")}


def prefill_summary(wl, r, U, hbm_peak, tc_peak, link_gbs):
    """Per-config staged-prefill line: the pipeline (bound by the host link: E records per layer)
    and the in-HBM forward of one layer (route + plan + expert kernels) against both rooflines."""
    import expert_offload_slot_gb300 as moe
    T, L = r["T"], wl.L
    prof = r["prof"]
    n = max(1, prof["launches"])
    st = {k: v * 1e3 / n for k, v in zip(moe.STAGES, prof["stage_ms"])}
    us_layer = r["ms"] * 1e3 / (r["steps"] * L)
    ffn_us = st["ffn"]
    fl = prefill_flops(wl, T)
    byt = (U + (1 if wl.shared else 0)) * expert_bytes(wl) + 2 * T * wl.H * wl.act_elt_bytes
    staged_bytes = wl.E * wl.expert_layout()[4]
    inhbm_us = st["route"] + st["plan"] + st["ffn"]
    return {"T": T, "tokens_per_s": r["steps"] * T * L / (r["ms"] / 1e3), "us_per_layer": us_layer,
            "steps": r["steps"], "staged_layers": r["staged"], "experts_with_tokens": U,
            "link": {"bound": "host link", "bytes_per_layer": staged_bytes,
                     "achieved": staged_bytes / (us_layer * 1e-6) / 1e9, "unit": "GB/s",
                     "frac_of_measured_link": staged_bytes / (us_layer * 1e-6) / 1e9 / link_gbs if link_gbs else None},
            "in_hbm": {"us_per_layer": inhbm_us, "tokens_per_s": T / (inhbm_us * 1e-6),
                       "stage_us_per_layer": st,
                       "ffn_tflops": fl / (ffn_us * 1e-6) / 1e12, "ffn_tc_frac": fl / (ffn_us * 1e-6) / 1e12 / tc_peak,
                       "ffn_gbs": byt / (ffn_us * 1e-6) / 1e9, "ffn_hbm_frac": byt / (ffn_us * 1e-6) / 1e9 / hbm_peak,
                       "flops_per_layer": fl, "bytes_per_layer": byt,
                       "bound": "hbm" if fl / byt < tc_peak * 1e12 / (hbm_peak * 1e9) else "tensor"},
            "link_now": r.get("link_now"), "status": moe_status_name(r["status"])}


def moe_status_name(st):
    import expert_offload_slot_gb300 as moe
    return moe.STATUS_NAMES.get(st, st)


def distinct_experts_last_call(bench, T):
    r = bench.pool.routing(T)
    return int(len(set(int(v) for v in r["ids"].reshape(-1))))


def profile_trace(wl, T, steps, dev):
    """A profiling trace of the decode workload's routing (steps of its AR(1) hidden states drawn
    with another seed), routed on the GPU by moe_route_topk_noalloc: ids [steps, L, T, k] int32 and
    probs [steps, L, T, E] float32 on the host."""
    import numpy as np
    import torch

    import expert_offload_slot_gb300 as moe
    from synth import gen
    xs = gen.torch_decode_hidden(wl, T, steps, dev, base_seed=1)
    w_r, b = gen.routers(wl)
    wr = torch.from_numpy(np.ascontiguousarray(w_r.view(np.int16))).to(dev)
    bd = torch.from_numpy(b).to(dev)
    ids = torch.empty((steps, wl.L, T, wl.k), dtype=torch.int32, device=dev)
    probs = torch.empty((steps, wl.L, T, wl.E), dtype=torch.float32, device=dev)
    w = torch.empty((T, wl.k), dtype=torch.float32, device=dev)
    gap = torch.empty(T, dtype=torch.float32, device=dev)
    for st in range(steps):
        for l in range(wl.L):
            moe.moe_route_topk_noalloc(wl.E, wl.k, wl.H, wl.act_dtype, wl.gating, xs[st, l].view(torch.int16), wr[l],
                                       bd[l], ids[st, l], w, probs[st, l], gap)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), probs.cpu().numpy()


def run_configs(names, dev, qwen_host, args, peaks, link_gbs):
    """The other workload shapes at one GPU, each pool built, measured and freed in turn."""
    import dataclasses

    from synth import get_workload
    hbm, tc = peaks
    out = {}
    q = get_workload("qwen3_decode")
    for name in names:
        t0 = time.time()
        if name not in ("qwen3_hit", "s_independence", "quotas", "prefetch", "aes") and qwen_host is not None and \
                qwen_host.ptr:
            qwen_host.free()             # the remaining configs bring host pools of their own
        if name == "qwen3_hit":
            # every expert resident (S = L*E): the hit path alone, no miss copies
            b = PoolBench(q, 16, dev, host=qwen_host, slots=q.L * q.E)
            res = {}
            for T in (1, 16):
                c = Clocks(torch_local())
                res[str(T)] = decode_summary(q, b.decode(T, 8, 64, 8, c, 1, e2e=False), hbm)
            b.close()
            out[name] = {"workload": "qwen3-30b-a3b-shaped-decode, all 6144 experts resident", "decode": res}
        elif name == "s_independence":
            # SeqMoE "Mechanism": a slot count above the expert count leaves the fused kernel's latency
            # unchanged.  Same repeated step (every needed expert resident) at 45 %, 100 % and 200 % of
            # the L*E experts as slots.
            res = []
            for S in (q.S, q.L * q.E, 2 * q.L * q.E):
                b = PoolBench(q, 16, dev, host=qwen_host, slots=S)
                res.append(b.decode_repeat(16, 8, 64))
                b.close()
            us = [r["us_per_layer"] for r in res]
            out[name] = {"workload": "qwen3-30b-a3b-shaped-decode, T=16, one step repeated (hit path only)",
                         "by_slots": res, "max_over_min": max(us) / min(us)}
        elif name == "prefetch":
            # SeqMoE asynchronous prefetch: the headline decode (T = 16) without prefetch, then with one
            # and two prefetches per layer-step (each pool fresh from the same table and trace)
            res = {}
            base = None
            for per in (0, 1, 2):
                b = PoolBench(q, 16, dev, host=qwen_host)
                b.pool.prefetch_enable(per)
                r = b.decode(16, 8, 64, 0, Clocks(torch_local()), 1, e2e=False)
                b.close()
                res[str(per)] = prefetch_summary(q, r, base)
                if per == 0:
                    base = res["0"]
            out[name] = {"workload": "qwen3-30b-a3b-shaped-decode, T=16, 2765 slots, MRS; per_step 0 / 1 / 2",
                         "by_per_step": res}
        elif name == "aes":
            # MoE-CORE approximate expert substitution (off in the page's main numbers): the headline
            # decode with substitution at two logit margins, reported as availability (hit rate,
            # demand misses, time) and as output deviation.  The deviation compares each layer call's
            # output with the exact routing's, which any pool without substitution computes (its
            # output does not depend on its resident set): two pools fed the same inputs eagerly.
            import torch

            import expert_offload_slot_gb300 as moe
            res = {}
            base = None
            for alpha in (None, 0.05, 0.2):
                b = PoolBench(q, 16, dev, host=qwen_host)
                if alpha is not None:
                    b.pool.set_aes(1, alpha)
                r = b.decode(16, 8, 64, 0, Clocks(torch_local()), 1, e2e=False)
                steps = r["steps"] * q.L
                row = {"tokens_per_s": r["steps"] * 16 * q.L / (r["ms"] / 1e3),
                       "us_per_layer": r["ms"] * 1e3 / steps,
                       "hit_rate": r["hits"] / max(1, r["hits"] + r["misses"]),
                       "demand_misses_per_layer_step": r["misses"] / steps,
                       "substitutions_per_layer_step": r["aes_substitutions"] / steps,
                       "status": moe_status_name(r["status"])}
                if alpha is not None:
                    # output deviation over 4 eager steps of a continued trace (all 48 layers each)
                    ex = PoolBench(q, 16, dev, host=qwen_host)
                    xs = __import__("synth").gen.torch_decode_hidden(q, 16, 4, dev, base_seed=977)
                    o1 = torch.empty_like(xs[0][0])
                    o2 = torch.empty_like(o1)
                    rel = []
                    s_ = torch.cuda.Stream()
                    with torch.cuda.stream(s_):
                        for st in range(4):
                            for l in range(q.L):
                                b.pool.forward(l, xs[st][l], o1, moe.MOE_MODE_DECODE)
                                ex.pool.forward(l, xs[st][l], o2, moe.MOE_MODE_DECODE)
                                a_ = o1.float()
                                e_ = o2.float()
                                rel.append((torch.linalg.vector_norm(a_ - e_) / torch.linalg.vector_norm(e_)).item())
                    ex.close()
                    row["alpha"] = alpha
                    row["output_rel_l2_mean"] = sum(rel) / len(rel)
                    row["output_rel_l2_max"] = max(rel)
                    row["vs_exact_time"] = base["us_per_layer"] / row["us_per_layer"]
                b.close()
                res["off" if alpha is None else "alpha_%g" % alpha] = row
                if alpha is None:
                    base = row
            out[name] = {"workload": "qwen3-30b-a3b-shaped-decode, T=16, 2765 slots, MRS; substitution off / "
                                     "logit margin 0.05 / 0.2",
                         "by_alpha": res,
                         "deviation": "relative L2 norm of (output - exact-routing output) per layer call"}
        elif name == "dsv3_resplit":
            # RapidMoE residual-split experts on the DeepSeek-V3 expert shape (4-bit W^Q + 4-bit
            # residual for gate/up, 4- or 8-bit down, own codec), UMIA deciding each step's precision:
            # every expert high (theta 0), every expert low, and a mixed threshold
            from synth.configs import RESPLIT_Q4R4
            wl = dataclasses.replace(get_workload("dsv3"), name="dsv3_resplit", weight_dtype=RESPLIT_Q4R4)
            o = wl.expert_layout()
            IH = wl.I * wl.H
            b = PoolBench(wl, max(wl.decode_T), dev)
            res = {}
            for label, theta in (("all_high", 0.0), ("mixed_theta_0.8", 0.8), ("all_low", 10.0)):
                b.pool.set_umia(theta)
                per_T = {}
                for T in wl.decode_T:
                    r = b.decode(T, 3, 24, 0, Clocks(torch_local()), 1, e2e=False)
                    n_ent = (r["hits"] + r["misses"]) + r["steps"] * wl.L      # routed + shared entries
                    crit = r["critical_entries"]
                    # HBM bytes the expert kernels read: W^Q + W^R + W^H_down (+ scales) for a critical
                    # entry, W^Q + W^L_down (+ scales) for the others
                    b_hi = IH + IH + IH + (2 * 2 * wl.I * (wl.H // 128) + wl.H * (wl.I // 128)) * 4
                    b_lo = IH + IH // 2 + (2 * wl.I * (wl.H // 128) + wl.H * (wl.I // 128)) * 4
                    byt = crit * b_hi + (n_ent - crit) * b_lo
                    per_T[str(T)] = {"tokens_per_s": r["steps"] * T * wl.L / (r["ms"] / 1e3),
                                     "us_per_layer": r["ms"] * 1e3 / (r["steps"] * wl.L),
                                     "hit_rate": r["hits"] / max(1, r["hits"] + r["misses"]),
                                     "critical_fraction": crit / max(1, n_ent),
                                     "expert_GB_per_s_whole_layer": byt / (r["ms"] / 1e3) / 1e9,
                                     "status": moe_status_name(r["status"])}
                res[label] = per_T
            b.close()
            out[name] = {"workload": "deepseek-v3-shaped, residual-split records (%d B), 4 layers, 410 slots, MRS"
                                     % o[4], "decode_by_umia": res,
                         "note": "expert_GB_per_s_whole_layer counts the expert bytes read over the whole "
                                 "layer call (router, plan and miss copies included)"}
        elif name == "quotas":
            # MoE-CORE cache shaping: the headline decode (T = 16, 2765 slots) with the table filled
            # from a profiling trace, uniform quotas and the replayed nonuniform ones
            import numpy as np

            import expert_offload_slot_gb300 as moe
            ids, probs = profile_trace(q, 16, 64, dev)
            cfg = moe.make_config(q.L, q.E, q.k, q.H, q.I, q.S, q.weight_dtype, q.act_dtype, q.gating, False,
                                  q.evict, q.window)
            uniform = np.array([q.quota(l) for l in range(q.L)], np.int32)
            t_plan = time.time()
            planned, hit = moe.moe_plan_quotas(cfg, ids, probs, q.S, 4, 0.01)
            t_plan = time.time() - t_plan
            res = {}
            for label, quotas in (("uniform_profile_fill", uniform), ("planned_profile_fill", planned)):
                b = PoolBench(q, 16, dev, host=qwen_host, lut=moe.moe_profile_lut(cfg, probs, quotas))
                r = decode_summary(q, b.decode(16, 8, 64, 8, Clocks(torch_local()), 1, e2e=False), hbm)
                b.close()
                res[label] = {"tokens_per_s": r["tokens_per_s"], "us_per_layer": r["us_per_layer"],
                              "hit_rate": r["hit_rate"], "quota_min": int(quotas.min()), "quota_max": int(quotas.max())}
            out[name] = {"workload": "qwen3-30b-a3b-shaped-decode, T=16, 2765 slots; profile: 64 steps of another "
                                     "seed routed by moe_route_topk_noalloc",
                         "plan": {"delta_k": 4, "tau_low": 0.01, "replayed_hit_rate_min": float(hit.min()),
                                  "replayed_hit_rate_max": float(hit.max()), "layers_changed":
                                  int((planned != uniform).sum()), "seconds": t_plan},
                         "decode": res}
        elif name == "qwen3_prefill":
            # the decode workload's expert weights and router matrix (same shapes and law) with the
            # prefill router bias 0, so that all 128 experts receive tokens
            # a fresh host pool of its own: inside one long run the staged copies from the decode
            # workload's host pool ran at half the link rate, fresh pools at the full rate
            p = dataclasses.replace(get_workload("qwen3_prefill"), name="qwen3_decode")
            pr = get_workload("qwen3_prefill")
            b = PoolBench(p, max(pr.prefill_T), dev, staging=True)
            res = {}
            for T in pr.prefill_T:
                r = b.prefill(T, 3, 3)
                res[str(T)] = prefill_summary(p, r, distinct_experts_last_call(b, T), hbm, tc, link_gbs)
            b.close()
            out[name] = {"workload": "qwen3-30b-a3b-shaped-prefill, staged (2 layer-sized regions), fresh host pool",
                         "prefill": res}
        elif name in ("dsv3", "mixtral"):
            wl = get_workload(name)
            max_T = max(wl.decode_T + wl.prefill_T)
            b = PoolBench(wl, max_T, dev, staging=True)
            dec = {}
            for T in wl.decode_T:
                K = 32 if name == "dsv3" else 24
                dec[str(T)] = decode_summary(wl, b.decode(T, 3, K, 4, Clocks(torch_local()), 1, e2e=False), hbm)
            pf = None
            if name == "mixtral":
                # the link-bound decode with one prefetch per layer-step (same pool, continued trace)
                r0 = b.decode(1, 3, 24, 0, None, 1, e2e=False)
                b.pool.prefetch_enable(1)
                r1 = b.decode(1, 3, 24, 0, None, 1, e2e=False)
                b.pool.prefetch_enable(0)
                b.pool.prefetch_drain()
                base = prefetch_summary(wl, r0)
                pf = {"0": base, "1": prefetch_summary(wl, r1, base)}
            pre = {}
            for T in wl.prefill_T:
                r = b.prefill(T, 3, 3)
                pre[str(T)] = prefill_summary(wl, r, distinct_experts_last_call(b, T), hbm, tc, link_gbs)
            b.close()
            lbl = {"dsv3": "deepseek-v3-shaped (fp8 e4m3, 128x128 block scales, shared expert, MRS eviction)",
                   "mixtral": "mixtral-8x7b-shaped (64 slots, MRS eviction)"}[name]
            out[name] = {"workload": lbl, "layers": wl.L, "slots": wl.S, "decode": dec, "prefill": pre}
            if pf:
                out[name]["decode_prefetch_T1"] = pf
        out[name]["seconds"] = time.time() - t0
    return out


def torch_local():
    import torch
    return torch.cuda.current_device()


# ------------------------------------------------------------------ oracle arm
class OracleSample:
    """The CPU oracle as it stands, on the first layer-steps of the same workload."""

    def __init__(self, wl, T, n_layers, n_steps, device):
        import numpy as np

        from synth import gen
        self.wl, self.T = wl, T
        self.rec = wl.expert_layout()[4]
        self.n_layers, self.n_steps = n_layers, n_steps
        self.records = {l: gen.device_layer_records(wl, l, device).cpu().numpy() for l in range(n_layers)}
        self.w_r, self.b = gen.routers(wl)
        xs = gen.torch_decode_hidden(wl, T, n_steps, device)
        self.xs = xs.view(__import__("torch").int16).cpu().numpy().view(np.uint16) if wl.act_dtype == 1 \
            else xs.cpu().numpy()
        self.lut = gen.initial_lut(wl)

    def run(self, max_layer_steps):
        import numpy as np

        from oracle.cache import SlotPoolSim
        from oracle.layer import layer_from_stored
        from synth import gen
        wl = self.wl
        sim = SlotPoolSim(wl.L, wl.E, wl.S, wl.evict, wl.window)
        sim.set_lut(self.lut)
        done = 0
        t0 = time.perf_counter()
        for t in range(self.n_steps):
            for l in range(self.n_layers):
                if done >= max_layer_steps:
                    break
                recs = self.records[l]
                out, r = layer_from_stored(self.xs[t, l], wl.act_dtype, self.w_r[l], self.b[l],
                                           lambda e: gen.record_to_stored(wl, recs[e]), wl.weight_dtype, wl.I,
                                           wl.k, wl.gating)
                sim.update_scores(l, r["ids"], r["probs"].astype(np.float32))
                sim.plan(l, r["ids"])
                done += 1
        el = time.perf_counter() - t0
        return done, el


def oracle_sample(wl, T, n_layer_steps, device):
    n_layers = min(4, wl.L)
    n_steps = (n_layer_steps + n_layers - 1) // n_layers
    o = OracleSample(wl, T, n_layers, n_steps, device)
    done, el = o.run(n_layer_steps)
    return {"value": done * T / el, "unit": "MoE-layer tokens/s", "threads": ORACLE_THREADS,
            "us_per_layer": el * 1e6 / done,
            "sample": f"{done} layer-steps (layers 0-{n_layers - 1} x first {n_steps} decode steps, T={T}) "
                      f"of the same workload, numpy float64, {el:.1f} s"}


def cpu_baseline(wl, T, n_layer_steps, device, n_single):
    """The oracle on every host core (BLAS threads = the affinity mask's cores), and on one thread in
    a child process started with the BLAS thread count set to 1 before numpy loads."""
    allt = oracle_sample(wl, T, n_layer_steps, device)
    single = None
    if n_single > 0:
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-sample-only", str(n_single),
                            "--batch", str(T), "--workload", wl.name], env=env, capture_output=True, text=True)
        try:
            single = json.loads(r.stdout.strip().splitlines()[-1])
        except (IndexError, ValueError):
            single = {"error": (r.stderr or r.stdout)[-300:]}
    return {"value": allt["value"], "unit": allt["unit"], "cores": HOST_CORES, "threads": allt["threads"],
            "kind": "oracle", "sample": allt["sample"], "us_per_layer": allt["us_per_layer"],
            "single_thread": single}


def probe_link(wl):
    """Host -> GPU bandwidth of the library's device-started record copy (moe_load_slot) and of DMA."""
    import numpy as np
    import torch

    import expert_offload_slot_gb300 as moe
    from synth import gen
    one = __import__("dataclasses").replace(wl, L=1)
    rec = one.expert_layout()[4]
    cfg = moe.make_config(1, one.E, one.k, one.H, one.I, 16, one.weight_dtype, one.act_dtype, max_tokens=16)
    host = moe.HostPool(one.E * rec)
    wr = torch.zeros((one.E, one.H), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(one.E, dtype=torch.float32, device="cuda")
    pool = moe.Pool(cfg, host.ptr, host.nbytes, wr, b)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in range(4):
        pool.load_slot(0, e, e % 16)
    torch.cuda.synchronize()
    n = 64
    ev0.record()
    for i in range(n):
        pool.load_slot(0, 4 + i % (one.E - 4), i % 16)
    ev1.record()
    torch.cuda.synchronize()
    kern = n * rec / (ev0.elapsed_time(ev1) / 1e3) / 1e9
    src = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    dst = torch.empty_like(src, device="cuda")
    dst.copy_(src, non_blocking=True)
    torch.cuda.synchronize()
    ev0.record()
    dst.copy_(src, non_blocking=True)
    ev1.record()
    torch.cuda.synchronize()
    dma = src.numel() / (ev0.elapsed_time(ev1) / 1e3) / 1e9
    pool.close()
    host.free()
    return {"probe": "link", "record_bytes": rec, "device_started_copy_GBps": kern, "dma_h2d_GBps": dma,
            "us_per_record": rec / kern / 1e3}


def main():
    args = parse_args()
    import torch

    import dataclasses

    from synth import get_workload
    wl = get_workload(args.workload)
    if args.layers:
        # a reduced case for profiler captures: same layer shape, fewer layers, same residency
        wl = dataclasses.replace(wl, L=args.layers)
    if args.experts:
        # a reduced case for profiler captures: same expert matrices (H, I, dtype), fewer experts
        k = args.top_k or min(wl.k, args.experts)
        wl = dataclasses.replace(wl, E=args.experts, k=k, fixed_slots=0)
    if args.cpu_sample_only:
        print(json.dumps(oracle_sample(wl, args.batch, args.cpu_sample_only, "cuda")))
        return
    rank, world, local = dist_setup(args.gpus)
    if args.prefill:
        import expert_offload_slot_gb300 as moe  # noqa: F401  (fails loudly without the library)
        hbm, _ = load_peaks()
        # the decode pool is not used by staged calls: one slot per expert at most
        b = PoolBench(wl, args.prefill, torch.device("cuda", torch.cuda.current_device()), staging=True,
                      slots=max(1, min(wl.S, wl.E)))
        r = b.prefill(args.prefill, max(1, args.warmup), max(1, args.steps))
        out = prefill_summary(wl, r, distinct_experts_last_call(b, args.prefill), hbm, load_tc_peak(), None)
        b.close()
        if rank == 0:
            print(json.dumps(dict(out, workload=wl.name, layers=wl.L)))
        return
    if args.probe_link:
        if rank == 0:
            print(json.dumps(probe_link(wl)))
        return
    label = WORKLOAD_LABEL.get(args.workload, args.workload)
    T = args.batch
    base_cfg = {"workload": label, "layers": wl.L, "experts": wl.E, "top_k": wl.k, "hidden": wl.H,
                "inter": wl.I, "slots": wl.S, "residency": wl.residency, "batch_tokens": T,
                "evict": ["moe-core", "mrs", "lru"][wl.evict], "router_bias_zipf_s": wl.zipf_s,
                "ar1_rho": wl.ar_rho, "graph": "48 moe_forward calls captured once per step",
                "l2": "no flush: a step streams ~48*U expert records (GBs) >> 129 MB L2"}

    if args.impl == "reference":
        if rank != 0:
            return
        n = min(args.steps, 24)
        o = OracleSample(wl, T, min(4, wl.L), (n + 3) // 4, "cuda")
        warm = min(args.warmup, 4)      # untimed oracle layer-steps (~0.4 s each)
        o.run(warm)
        done, el = o.run(n)
        v = done * T / el
        line = {"impl": "reference", "metric": "MoE-layer tokens/s (decode)", "value": v,
                "unit": "MoE-layer tokens/s", "n_gpus": 1, "steps": done, "warmup": warm,
                "ms_per_step": el * 1e3 / done, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic (seeded random weights, AR(1) hidden states)",
                "config": dict(base_cfg, reference_step="one layer-step of the oracle (T tokens, one layer)"),
                "cpu_baseline": {"value": v, "unit": "MoE-layer tokens/s", "cores": HOST_CORES,
                                 "threads": ORACLE_THREADS, "us_per_layer": el * 1e6 / done,
                                 "kind": "oracle", "sample": f"{done} layer-steps of the requested {args.steps}"},
                "e2e": {"value": v, "unit": "MoE-layer tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import expert_offload_slot_gb300 as moe  # noqa: F401  (fails loudly without the library)
    dev = torch.device("cuda", torch.cuda.current_device())
    sweep_T = [int(v) for v in args.sweep.split(",") if v.strip()] if args.sweep else []
    max_T = max([T] + sweep_T)
    peak, peak_kind = load_peaks()
    tc_peak = load_tc_peak()
    bench = PoolBench(wl, max_T, dev)
    sweep = {}
    for t in sweep_T:
        r = bench.decode(t, args.warmup, args.steps, max(4, args.prof_steps // 2), None, world, e2e=False)
        sweep[str(t)] = decode_summary(wl, r, peak)
    clocks = Clocks(local) if rank == 0 else None
    r = bench.decode(T, args.warmup, args.steps, args.prof_steps, clocks, world, e2e=not args.no_e2e)
    ms = max_over_ranks(r["ms"], world)
    tokens = sum_over_ranks(r["steps"] * T * wl.L, world)
    value = tokens / (ms / 1e3)
    e2e_ms = max_over_ranks(r["e2e"]["ms"], world) if "e2e" in r else float("nan")
    e2e_value = tokens / (e2e_ms / 1e3)

    prof = r["prof"]
    ffn_ms = prof["stage_ms"][moe.STAGES.index("ffn")] + prof["stage_ms"][moe.STAGES.index("copy")]
    layer_steps = prof["launches"]
    U_mean = prof["sum_U"] / max(1, layer_steps)
    fused = fused_layer(prof["stage_ms"])
    ffn_bytes = ffn_algorithmic_bytes(wl, prof["sum_U"], prof["bytes_copied"], layer_steps, T, router=fused)
    achieved = ffn_bytes / (ffn_ms / 1e3) / 1e9 if ffn_ms > 0 else 0.0
    prof_layer_us = sum(prof["stage_ms"]) * 1e3 / max(1, layer_steps)
    layer_bytes = step_bytes(wl, U_mean, T)
    if rank != 0:
        bench.close()
        return
    bench.close(keep_host=True)
    configs = {}
    names = [v.strip() for v in args.configs.split(",") if v.strip()]
    if world == 1 and names and args.workload == "qwen3_decode" and not args.layers:
        link = probe_link(wl)
        configs["link"] = link
        configs.update(run_configs(names, dev, bench.host, args, (peak, tc_peak), link["dma_h2d_GBps"]))
    bench.host.free()
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, T, args.cpu_sample, dev, max(2, args.cpu_sample // 8))
    us_layer = ms * 1e3 / (r["steps"] * wl.L)
    try:
        floor = layer_floor(layer_bytes, r["bytes_copied"] / (r["steps"] * wl.L), us_layer, peak,
                            configs.get("link", {}).get("dma_h2d_GBps"))
    except (KeyError, TypeError, ZeroDivisionError):
        floor = None
    line = {
        "metric": "MoE-layer tokens/s (decode)", "value": value, "unit": "MoE-layer tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / r["steps"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded random N(0,0.02) weights, Zipf router bias, AR(1) hidden states)",
        "config": dict(base_cfg, parallelism=f"replicas x{world}" if world > 1 else "single GPU"),
        "us_per_layer": ms * 1e3 / (r["steps"] * wl.L),
        "hit_rate": r["hits"] / max(1, r["hits"] + r["misses"]),
        "miss_copy_GB": r["bytes_copied"] / 1e9,
        "e2e": {"value": e2e_value, "unit": "MoE-layer tokens/s",
                "h2d_bytes_per_step": r.get("e2e", {}).get("h2d"), "d2h_bytes_per_step": r.get("e2e", {}).get("d2h"),
                "hit_rate": r.get("e2e", {}).get("hit_rate"), "misses": r.get("e2e", {}).get("misses"),
                "steps": "the K decode steps that follow the timed and profiling passes in the same trace"},
        "spread": {"quarter_tokens_per_s": [n * T * wl.L / (q / 1e3) for q, n in r["quarter_ms"]],
                   "timed_misses": r["misses"]},
        "roofline": {"bound": "hbm", "kernel": KERNEL_LABEL[fused],
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": captured_traffic(KERNEL_LABEL[fused].split()[0]),
                     "peak_source": f"{peak_kind} hbm_gbs", "launches_timed": prof["launches"],
                     "bytes_per_launch": ffn_bytes / max(1, prof["launches"]),
                     "us_per_launch": ffn_ms * 1e3 / max(1, prof["launches"])},
        "layer_roofline": {"algorithmic_bytes_per_layer": layer_bytes, "mean_U": U_mean,
                           "us_per_layer_profiled": prof_layer_us,
                           "frac": layer_bytes / (prof_layer_us * 1e-6) / 1e9 / peak if prof_layer_us else 0.0},
        "layer_floor": floor,
        "stage_us_per_layer": {n: v * 1e3 / max(1, layer_steps) for n, v in zip(moe.STAGES, prof["stage_ms"])},
        "clocks": r["clocks"],
        "gpu_launches": r["launches_per_step"] * r["steps"],
        "status": moe.STATUS_NAMES.get(r["status"], r["status"]),
        "sweep": sweep,
        "setup_s": bench.setup_s,
        "cpu_baseline": cpu,
        "configs": configs,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
