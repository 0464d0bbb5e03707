"""Benchmark of the MoE FFN layer forward on GB300: tokens/s per layer.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]

A step is one pass of the whole layer (route -> permute -> gather -> gate/up
GEMM + SwiGLU -> down GEMM -> combine) over one batch of seeded synthetic
tokens.  The default workload is the Mixtral-8x7B-shaped decode layer (T=16,
d_model=4096, d_ff=14336, E=8, top-2, int4 group-128 weights).  Prints one JSON
line (rank 0).

--impl ours       the CUDA library (inputs resident in HBM for `value`; `e2e`
                  adds the pinned host<->device copies of x, logits and out).
--impl reference  the CPU oracle (test infrastructure) on the host cores, one
                  thread per token slice (the C oracle releases the GIL), on the
                  same workload; no GPU work.
N > 1 (torchrun): independent replicas, one per GPU, no data-path collective
("scaling": "weak"); a barrier brackets the timed region and the max time over
ranks is used.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import moe_synth as ms  # noqa: E402

STAGES = ("route", "permute", "gather", "gate_up", "down", "combine")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mixtral_decode", choices=list(ms.CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="time only --config, not the other workloads as well")
    return ap.parse_args()


L2_BYTES = 129 * 2 ** 20   # GB300 L2


def describe(cfg: ms.LayerConfig, n_gpus: int = 1) -> dict:
    """The workload's config dict, identical for both arms."""
    w = {"bf16": "bf16", "int4": "int4 asymmetric group-128 (fp16 scale + zero)",
         "fp8": "fp8 E4M3 group-128 (fp16 scale)"}[cfg.fmt]
    route = {"normal": "i.i.d. N(0,1) logits", "zipf": f"Zipf(s={cfg.zipf_s}) routing",
             "reuse": f"{int(cfg.reuse_p * 100)}% of tokens reuse the previous token's experts"}[cfg.logits]
    lg = ms.make_logits(cfg)
    n_active = len(needed_experts(cfg, lg, list(range(cfg.T)))) + (1 if cfg.shared else 0)
    wbytes = n_active * ms.active_expert_bytes(cfg)
    l2 = (f"inputs larger than L2: every step streams the {n_active} active experts' weights "
          f"({wbytes / 1e6:.0f} MB) from HBM, above the 129 MB L2" if wbytes > L2_BYTES else
          f"weights ({wbytes / 1e6:.1f} MB) fit in L2 and stay resident across steps (no flush): "
          f"a launch-bound workload")
    return {"workload": f"{cfg.name}: MoE FFN layer forward, T={cfg.T}, d_model={cfg.d}, "
                        f"d_ff={cfg.F}, E={cfg.E}, top-{cfg.k}, SwiGLU, {w} weights, {route}"
                        + (", + 1 shared expert" if cfg.shared else ""),
            "T": cfg.T, "d_model": cfg.d, "d_ff": cfg.F, "experts": cfg.E, "top_k": cfg.k,
            "weights": cfg.fmt, "shared_expert": cfg.shared, "active_experts": n_active,
            "parallelism": "single GPU" if n_gpus == 1 else f"{n_gpus} independent replicas, one per GPU",
            "l2": l2}


# ----------------------------------------------------------------------------- distributed
def dist_init(n: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(mx)) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- oracle timing
def oracle_refs(cfg, weights_cpu: dict):
    import oracle
    refs = {e: oracle.ExpertRef(w, cfg.fmt) for e, w in weights_cpu.items()}
    return refs


def time_oracle(cfg, x_cpu, logits_np, refs: dict, tokens: list[int], threads: int) -> float:
    """Wall time of the oracle forward of `tokens`, split over `threads` threads."""
    import oracle
    first = next(iter(refs))
    ex = [refs.get(e, refs[first]) for e in range(cfg.E)]
    sh = refs.get("shared")
    chunks = [tokens[i::threads] for i in range(threads) if tokens[i::threads]]

    def run(ch):
        return oracle.layer_forward(x_cpu, logits_np, cfg.k, ex, sh, cfg.d, cfg.F, tokens=ch)

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=len(chunks)) as pool:
        list(pool.map(run, chunks))
    return time.perf_counter() - t0


def needed_experts(cfg, logits_np, tokens) -> list[int]:
    top = np.argsort(-logits_np[tokens], axis=1, kind="stable")[:, :cfg.k]
    return sorted(set(int(e) for e in top.ravel()))


# ----------------------------------------------------------------------------- reference arm
def slice_weights(w: dict, fmt: str, f0: int, f1: int) -> dict:
    """Expert weights restricted to the d_ff columns [f0, f1) (multiples of 128):
    gate/up keep those rows, down keeps those K columns with their groups."""
    out = {}
    for m in ("gate", "up"):
        out[m] = {key: t[f0:f1].contiguous() for key, t in w[m].items()}
    dn = w["down"]
    if fmt == "bf16":
        out["down"] = {"w": dn["w"][:, f0:f1].contiguous()}
    elif fmt == "fp8":
        out["down"] = {"q": dn["q"][:, f0:f1].contiguous(), "scale": dn["scale"][:, f0 // 128:f1 // 128].contiguous()}
    else:
        out["down"] = {"q": dn["q"][:, f0 // 2:f1 // 2].contiguous(),
                       "scale": dn["scale"][:, f0 // 128:f1 // 128].contiguous(),
                       "zero": dn["zero"][:, f0 // 128:f1 // 128].contiguous()}
    return out


def run_reference(args, cfg):
    rank, world, _ = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0
    if rank != 0:
        return
    import oracle
    oracle.build()
    x = ms.make_x(cfg)
    lg = ms.make_logits(cfg)
    toks = list(range(cfg.T))
    used = needed_experts(cfg, lg, toks)
    w = {e: ms.expert_weights(cfg, e, "cpu") for e in used}
    if cfg.shared:
        w["shared"] = ms.expert_weights(cfg, "shared", "cpu")
    refs = oracle_refs(cfg, w)
    cores = os.cpu_count() or 1
    threads = max(1, min(cfg.T, cores))
    runs = args.steps + args.warmup
    budget = 180.0   # seconds for the whole --steps + --warmup run
    # one step = the whole layer on the T tokens when that fits the budget;
    # else fewer tokens per step; and when even one token per step (on one
    # thread) would overrun it, a unit of work is one token's FFN over 1/S of
    # d_ff (gate/up rows and down columns of those features), `threads` units
    # per step on as many threads: the sample shrinks, the oracle is unchanged
    wave = time_oracle(cfg, x, lg, refs, toks[:threads], threads)   # `threads` tokens at once
    waves = (cfg.T + threads - 1) // threads
    S = 1
    if wave * waves * runs <= budget:
        n_tok = cfg.T
    elif wave * runs <= budget:
        n_tok = max(1, min(cfg.T, threads * int(budget / (wave * runs))))
    else:
        n_tok = threads
        G = cfg.F // 128
        need = wave * runs / budget
        S = next((c for c in range(2, G + 1) if G % c == 0 and c >= need), G)
    if S == 1:
        step_toks = toks[:n_tok]
        step = lambda: time_oracle(cfg, x, lg, refs, step_toks, min(threads, n_tok))
        tok_per_step = n_tok
        sample = f"{n_tok} of {cfg.T} tokens per step, all their experts, one host thread per token slice"
        used_threads = min(threads, n_tok)
    else:
        Fs = cfg.F // S
        # unit i: token i % T, feature slice i % S (every unit a different slice
        # or token), the slice's experts built once
        units = [(i % cfg.T, i % S) for i in range(threads)]
        srefs = {}
        for _, sl in units:
            if sl not in srefs:
                srefs[sl] = {e: oracle.ExpertRef(slice_weights(w[e], cfg.fmt, sl * Fs, (sl + 1) * Fs), cfg.fmt)
                             for e in w}
        first = next(iter(w))

        def run_unit(u):
            t, sl = u
            r = srefs[sl]
            ex = [r.get(e, r[first]) for e in range(cfg.E)]
            return oracle.layer_forward(x, lg, cfg.k, ex, r.get("shared"), cfg.d, Fs, tokens=[t])

        def step():
            t0 = time.perf_counter()
            with cf.ThreadPoolExecutor(max_workers=len(units)) as pool:
                list(pool.map(run_unit, units))
            return time.perf_counter() - t0

        tok_per_step = len(units) / S
        sample = (f"{len(units)} units per step, each one token's FFN over 1/{S} of d_ff "
                  f"({tok_per_step:g} token equivalents), one host thread per unit")
        used_threads = len(units)
    for _ in range(args.warmup):
        step()
    total = 0.0
    for _ in range(args.steps):
        total += step()
    value = tok_per_step * args.steps / total
    line = {
        "impl": "reference", "metric": "moe_layer_tokens_per_s", "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": describe(cfg, args.gpus),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": used_threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm
def gateup_bytes(cfg, n_active: int, rows: int) -> int:
    if cfg.fmt == "int4":
        wb = 2 * (cfg.d * cfg.F // 2 + cfg.F * (cfg.d // 128) * 4)
    elif cfg.fmt == "fp8":
        wb = 2 * (cfg.d * cfg.F + cfg.F * (cfg.d // 128) * 2)
    else:
        wb = 2 * cfg.d * cfg.F * 2
    return n_active * wb + rows * cfg.d * 2 + rows * cfg.F * 2


def layer_bytes(cfg, n_active: int) -> int:
    return n_active * ms.active_expert_bytes(cfg) + cfg.T * cfg.d * 2 * 2 + cfg.T * cfg.E * 4


def load_peaks() -> tuple[float, float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return float(j["hbm_gbs"]), float(j.get("bf16_tflops", 1900.0)), "measured"
    return 6800.0, 1900.0, "fallback"


GEMM_SOURCES = ("gemm.cu", "gemm_group.cu", "gemm_common.cuh", "ptx.cuh", "kernels.cuh")


def gemm_sources_sha256() -> str:
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        h.update(open(os.path.join(ROOT, "moe_expert_layer_03_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def kernel_traffic(key: str):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu summary,
    valid only while the GEMM sources are unchanged (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    j = json.load(open(p))
    ent = j.get(key)
    if not ent or ent.get("gemm_sources_sha256") != gemm_sources_sha256():
        return None
    return ent.get("dram_bytes_per_launch")


def layer_roofline(cfg, rows, lb, ms_step, hbm, tflops) -> dict:
    """Whole-step roofline: HBM (the active experts' bytes) for decode-sized
    batches, the bf16 tensor peak (3 GEMMs, 2 flops per MAC) once the step's
    arithmetic intensity exceeds the ridge point."""
    flops = 2.0 * 3 * cfg.d * cfg.F * rows
    ent = {"algorithmic_bytes_per_step": lb, "algorithmic_flops_per_step": flops}
    if flops / lb > tflops * 1e12 / (hbm * 1e9):
        ach = flops / (ms_step / 1e3) / 1e12
        ent.update(bound="tensor", achieved=ach, peak=tflops, unit="TFLOP/s", frac=ach / tflops)
    else:
        ach = lb / (ms_step / 1e3) / 1e9
        ent.update(bound="hbm", achieved=ach, peak=hbm, unit="GB/s", frac=ach / hbm)
    return ent


def dominant_roofline(cfg, n_active, rows, gu_bytes, gu_ms, hbm, tflops, peak_kind) -> dict:
    """Roofline of the gate/up GEMM launch: HBM for decode-sized batches, the bf16
    tensor peak when its arithmetic intensity exceeds the ridge point."""
    flops = 2.0 * 2 * cfg.d * cfg.F * rows               # gate and up, 2 flops per MAC
    kname = "grouped gate/up GEMM + SwiGLU (tcgen05" + (", int4 dequant in the main loop)"
                                                       if cfg.fmt == "int4" else
                                                       ", fp8 E4M3 weights read by the MMA)" if cfg.fmt == "fp8"
                                                       else ")")
    ent = {"kernel": kname, "peak_source": peak_kind, "algorithmic_bytes_per_launch": gu_bytes,
           "algorithmic_flops_per_launch": flops, "traffic": kernel_traffic(cfg.name)}
    if flops / gu_bytes > tflops * 1e12 / (hbm * 1e9):
        ach = flops / (gu_ms / 1e3) / 1e12
        ent.update(bound="tensor", achieved=ach, peak=tflops, unit="TFLOP/s", frac=ach / tflops)
    else:
        ach = gu_bytes / (gu_ms / 1e3) / 1e9
        ent.update(bound="hbm", achieved=ach, peak=hbm, unit="GB/s", frac=ach / hbm)
    return ent


class Layer:
    """One workload's layer, resident on the device: seeded inputs, the expert
    pool (prepacked through the library) and its routed / shared views."""

    def __init__(self, moe, cfg, dev, keep_cpu: bool):
        self.cfg = cfg
        self.x = ms.make_x(cfg).to(dev)
        self.logits_np = ms.make_logits(cfg)
        self.logits = torch.from_numpy(self.logits_np).to(dev)
        e2s = ms.make_slot_table(cfg)
        self.e2s = e2s
        self.pool = moe.ExpertPool(cfg.E + (1 if cfg.shared else 0), cfg.d, cfg.F, cfg.fmt, device=dev)
        used = set(needed_experts(cfg, self.logits_np, list(range(cfg.T))))
        self.weights_cpu = {}
        for e in range(cfg.E):
            w = ms.expert_weights(cfg, e, dev)
            self.pool.load_expert(int(e2s[e]), w)
            if keep_cpu and e in used:
                self.weights_cpu[e] = {m: {k: v.cpu() for k, v in w[m].items()} for m in w}
            del w
        self.routed = self.pool.view(torch.from_numpy(e2s).to(dev))
        self.shared = None
        if cfg.shared:
            w = ms.expert_weights(cfg, "shared", dev)
            self.pool.load_expert(cfg.E, w)
            if keep_cpu:
                self.weights_cpu["shared"] = {m: {k: v.cpu() for k, v in w[m].items()} for m in w}
            self.shared = self.pool.view(torch.tensor([cfg.E], dtype=torch.int32, device=dev))
            del w
        torch.cuda.synchronize()
        self.n_active = len(used) + (1 if cfg.shared else 0)
        self.rows = cfg.A + (cfg.T if cfg.shared else 0)


def time_layer(moe, L: Layer, args, world: int, local: int, dev) -> dict:
    """K graph replays of the layer timed with CUDA events (inputs resident),
    clocks sampled meanwhile, then the per-stage split of an eager run."""
    cfg = L.cfg
    stream = torch.cuda.current_stream()
    ws = moe.workspace(moe.layer_workspace_bytes(cfg.T, cfg.k, L.routed, L.shared), dev)
    out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=dev)
    # the step as a user runs it: the layer captured once as a CUDA graph over
    # fixed input/output buffers, replayed per step
    lg = moe.LayerGraph(cfg.T, cfg.k, L.routed, L.shared, device=dev)
    lg.x.copy_(L.x)
    lg.logits.copy_(L.logits)
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(max(args.warmup, 3)):
        if i == 1:
            w0.record(stream)
        lg.replay()
    w1.record(stream)
    moe.layer_forward(L.x, L.logits, cfg.k, L.routed, L.shared, out=out, ws=ws)
    torch.cuda.synchronize()
    code = moe.last_device_error(lg.ws) or moe.last_device_error(ws)
    if code:
        raise SystemExit(f"{cfg.name}: device error code {code} during warm-up")
    per_replay_s = max(w0.elapsed_time(w1) / 1e3 / max(max(args.warmup, 3) - 1, 1), 1e-6)

    # ---- timed region: K steps (graph replays).  The clock sampler runs from
    # before an untimed ~0.25 s stretch of replays (the GPU under load when the
    # samples are taken) until after the timed steps.
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.2)
    for _ in range(int(min(0.25 / per_replay_s, 20000))):
        lg.replay()
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        lg.replay()
    stop.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = clk.stop()
    total_ms = max_over_ranks(start.elapsed_time(stop), world)
    if moe.last_device_error(lg.ws):
        raise SystemExit(f"{cfg.name}: device error during the timed region")

    # ---- per-stage breakdown: the same step run eagerly with CUDA events
    # between the kernels (the events add gaps and turn off the dependent
    # launches, so this run only apportions time; it is not the headline)
    n_ev = min(args.steps, 50)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(STAGES) + 1)] for _ in range(n_ev)]
    for i in range(n_ev):
        moe.layer_forward(L.x, L.logits, cfg.k, L.routed, L.shared, out=out, ws=ws, events=ev[i])
    torch.cuda.synchronize()
    stage_ms = {s_: float(np.mean([ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(n_ev)]))
                for j, s_ in enumerate(STAGES)}
    return {"total_ms": total_ms, "stage_ms": stage_ms, "clocks": clocks, "graph": lg,
            "launches": moe.layer_launch_count(cfg.T, cfg.k, L.routed, L.shared)}


def summarize(L: Layer, t: dict, args, world: int, hbm, tflops, peak_kind) -> dict:
    cfg = L.cfg
    ms_step = t["total_ms"] / args.steps
    gu_bytes = gateup_bytes(cfg, L.n_active, L.rows)
    lb = layer_bytes(cfg, L.n_active)
    return {
        "value": world * cfg.T * args.steps / (t["total_ms"] / 1e3), "unit": "tokens/s",
        "ms_per_step": ms_step, "steps": args.steps, "warmup": args.warmup,
        "dtype": dtype_of(cfg), "config": describe(cfg, world),
        "roofline": dominant_roofline(cfg, L.n_active, L.rows, gu_bytes, t["stage_ms"]["gate_up"], hbm,
                                      tflops, peak_kind),
        "layer_roofline": layer_roofline(cfg, L.rows, lb, ms_step, hbm, tflops),
        "stage_ms": t["stage_ms"], "gpu_launches": t["launches"] * args.steps, "clocks": t["clocks"],
    }


def dtype_of(cfg) -> str:
    """The arithmetic the layer's GEMMs run in for this workload."""
    bn = 16
    mean = -(-cfg.A // cfg.E)
    while bn < 2 * mean and bn < 256:
        bn <<= 1
    if cfg.fmt == "bf16":
        return "bf16 (tensor cores bf16 x bf16 -> fp32)"
    w = "int4 codes" if cfg.fmt == "int4" else "fp8 E4M3 codes"
    if bn <= 32:   # the decode kernel
        return (f"{w} x bf16 activations carried as two e4m3 terms (hi + lo, per-row power-of-two "
                f"scale), tensor cores e4m3 x e4m3 -> fp32, scales applied in fp32")
    return (f"{w} dequantised to fp16 x fp16 activations (per-row power-of-two scale), tensor cores "
            f"fp16 x fp16 -> fp32")


def run_ours(args, cfg):
    import moe_expert_layer_03_gb300 as moe
    rank, world, local = dist_init(args.gpus)
    moe.build()
    dev = f"cuda:{local}"
    torch.cuda.set_device(local)
    hbm, tflops, peak_kind = load_peaks()
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline

    # ---- the headline workload
    L = Layer(moe, cfg, dev, keep_cpu=want_cpu)
    t = time_layer(moe, L, args, world, local, dev)
    head = summarize(L, t, args, world, hbm, tflops, peak_kind)
    lgraph = t["graph"]
    stream = torch.cuda.current_stream()
    x, logits, routed, shared = L.x, L.logits, L.routed, L.shared

    # ---- the optional router GEMM (logits = x . w_router) that can stand in front
    # of the gating; not part of the step (the step takes logits as input).
    # RG launches captured in one CUDA graph (no host launch gaps), replayed and
    # timed with CUDA events
    RG = 20
    wr = ms.make_router_weight(cfg).to(dev)
    rl = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        moe.router_logits(x, wr, logits=rl)
        side.synchronize()
        rgraph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(rgraph, stream=side):
            for _ in range(RG):
                moe.router_logits(x, wr, logits=rl)
    stream.wait_stream(side)
    for _ in range(3):
        rgraph.replay()
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    r0.record(stream)
    n_rg = max(args.steps // 10, 3)
    for _ in range(n_rg):
        rgraph.replay()
    r1.record(stream)
    torch.cuda.synchronize()
    router_us = r0.elapsed_time(r1) / (n_rg * RG) * 1e3
    router_bytes = x.numel() * 2 + wr.numel() * 2 + rl.numel() * 4

    # ---- the step from the token rows alone (router GEMM + layer, one call;
    # for T <= 64 the router runs inside the routing launch): captured and
    # replayed like the headline step
    router_step = {}
    try:
        rg_graph = moe.LayerGraph(cfg.T, cfg.k, routed, shared, device=dev, router_weight=wr)
        rg_graph.x.copy_(x)
        for _ in range(max(args.warmup, 3)):
            rg_graph.replay()
        q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        for _ in range(args.steps):
            rg_graph.replay()
        q1.record(stream)
        torch.cuda.synchronize()
        if moe.last_device_error(rg_graph.ws):
            raise SystemExit("device error in the router step")
        same = torch.equal(rg_graph.logits, moe.router_logits(x, wr)) and torch.equal(
            rg_graph.out.view(torch.int16),
            moe.layer_forward(x, rg_graph.logits, cfg.k, routed, shared)[0].view(torch.int16))
        # the same work as two calls (router GEMM, then the layer on its logits),
        # captured and replayed the same way
        two_lg = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
        two_out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device=dev)
        two_ws = moe.workspace(moe.layer_workspace_bytes(cfg.T, cfg.k, routed, shared), dev)
        side2 = torch.cuda.Stream(device=dev)
        side2.wait_stream(stream)
        with torch.cuda.stream(side2):
            moe.router_logits(x, wr, logits=two_lg)
            moe.layer_forward(x, two_lg, cfg.k, routed, shared, out=two_out, ws=two_ws)
            side2.synchronize()
            two_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(two_graph, stream=side2):
                moe.router_logits(x, wr, logits=two_lg)
                moe.layer_forward(x, two_lg, cfg.k, routed, shared, out=two_out, ws=two_ws)
        stream.wait_stream(side2)
        for _ in range(max(args.warmup, 3)):
            two_graph.replay()
        q2, q3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        q2.record(stream)
        for _ in range(args.steps):
            two_graph.replay()
        q3.record(stream)
        torch.cuda.synchronize()
        lg_np = rg_graph.logits.cpu().numpy()
        router_step = {"us_per_step": q0.elapsed_time(q1) / args.steps * 1e3,
                       "us_per_step_two_calls": q2.elapsed_time(q3) / args.steps * 1e3,
                       "gpu_launches_per_step": moe.layer_router_launch_count(cfg.T, cfg.k, routed, shared),
                       "gpu_launches_per_step_two_calls": moe.layer_launch_count(cfg.T, cfg.k, routed, shared) + 1,
                       "router_fused_into_routing_launch": cfg.T <= 64,
                       "topk_fused_into_router_launch": cfg.T > 64 and cfg.E <= 16 and cfg.d % 64 == 0
                                                        and cfg.T * max(cfg.E, 8) >= 8192,
                       "active_experts": len(needed_experts(cfg, lg_np, list(range(cfg.T))))
                                         + (1 if cfg.shared else 0),
                       "matches_router_then_layer": bool(same),
                       "note": "graph replays of moe_layer_forward_router against moe_router_logits + "
                               "moe_layer_forward on the same router logits (random router weight: "
                               "the routing, and so the active experts, differ from the headline step's)"}
        del rg_graph, two_graph
    except (RuntimeError, moe.MoeError) as e:
        router_step = {"error": str(e)[:200]}

    # ---- expert streaming (pools larger than HBM): expert images in pinned host
    # memory copied on demand into 2 HBM slots by the LRU cache; timed as
    # alternating pairs of cold experts, 2 copies per ensure(), once with the
    # DMA engines and once with the SM copy kernel (when the images are mapped)
    pool, e2s = L.pool, L.e2s
    sb = pool.slot_bytes
    streaming = {}
    for mode_name, mode in (("dma", moe.ExpertCache.COPY_ENGINE), ("sm", moe.ExpertCache.COPY_SM)):
        hot = moe.ExpertPool(2, cfg.d, cfg.F, cfg.fmt, device=dev)
        try:
            cache = moe.ExpertCache(hot, cfg.E, copy_mode=mode)
        except moe.MoeError:
            streaming[mode_name] = None   # images not mapped into the device address space
            continue
        n_img = min(cfg.E, 4)
        for e in range(n_img):
            s_e = int(e2s[e])
            cache.load_image(e, pool.buf[s_e * sb:(s_e + 1) * sb])
        pairs = [[0, 1], [2, 3]] if n_img >= 4 else [[0], [1 % n_img]]
        cache.ensure(pairs[0])
        torch.cuda.synchronize()
        c0 = cache.stats()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for i in range(6):
            cache.ensure(pairs[(i + 1) % 2])
        s1.record(stream)
        torch.cuda.synchronize()
        copied = cache.stats()["bytes_copied"] - c0["bytes_copied"]
        streaming[mode_name] = copied / (s0.elapsed_time(s1) / 1e3) / 1e9
        del cache, hot

    # ---- overlapped streaming: a one-token decode loop over the headline
    # workload's token rows, each step's two experts served from a 4-slot hot
    # pool whose other experts live in pinned host memory.  Overlapped: the next
    # step's experts are prefetched on a copy stream while the current step
    # computes, then committed on the compute stream.  Serial: ensure() and the
    # forward on one stream.  Both over the same steps; the all-resident
    # forwards of the same steps give the compute time alone.
    overlap = None
    if cfg.E >= 4 and cfg.k <= 2:
        caches = []
        for _ in range(2):   # one cache per mode (ensure and prefetch/commit do not mix)
            hot = moe.ExpertPool(4, cfg.d, cfg.F, cfg.fmt, device=dev)
            cache = moe.ExpertCache(hot, cfg.E)
            for e in range(cfg.E):
                s_e = int(e2s[e])
                cache.load_image(e, pool.buf[s_e * sb:(s_e + 1) * sb])
            caches.append((hot, cache))
        cache, cache_serial = caches[0][1], caches[1][1]
        steps = list(range(min(cfg.T, 12)))
        xs = [x[t:t + 1].contiguous() for t in steps]
        lgs = [logits[t:t + 1].contiguous() for t in steps]
        act = [needed_experts(cfg, L.logits_np, [t]) for t in steps]
        wsz = moe.workspace(moe.layer_workspace_bytes(1, cfg.k, cache.view), dev)
        outo = torch.empty(1, cfg.d, dtype=torch.bfloat16, device=dev)
        copy_s = torch.cuda.Stream(device=dev)

        def run_overlap():
            cache.prefetch(act[0], copy_s)
            cache.commit(act[0], stream)
            for i in range(len(steps)):
                if i + 1 < len(steps):
                    cache.prefetch(act[i + 1], copy_s)
                moe.layer_forward(xs[i], lgs[i], cfg.k, cache.view, out=outo, ws=wsz)
                if i + 1 < len(steps):
                    cache.commit(act[i + 1], stream)

        def run_serial():
            for i in range(len(steps)):
                cache_serial.ensure(act[i], stream)
                moe.layer_forward(xs[i], lgs[i], cfg.k, cache_serial.view, out=outo, ws=wsz)

        def run_resident():
            for i in range(len(steps)):
                moe.layer_forward(xs[i], lgs[i], cfg.k, routed, out=outo, ws=wsz)

        def timed(fn, c):
            torch.cuda.synchronize()
            c0 = c.stats()["bytes_copied"]
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / len(steps), c.stats()["bytes_copied"] - c0

        for fn in (run_overlap, run_serial, run_resident):   # warm-up
            fn()
        torch.cuda.synchronize()
        t_ov, b_ov = timed(run_overlap, cache)
        t_se, b_se = timed(run_serial, cache_serial)
        t_re, _ = timed(run_resident, cache)
        if moe.last_device_error(wsz):
            raise SystemExit("device error in the streaming loop")
        overlap = {"steps": len(steps), "tokens_per_step": 1, "hot_slots": 4,
                   "overlapped_ms_per_step": t_ov, "serial_ms_per_step": t_se,
                   "compute_only_ms_per_step": t_re,
                   "bytes_copied_per_step_overlapped": b_ov / len(steps),
                   "bytes_copied_per_step_serial": b_se / len(steps),
                   "note": "one-token decode steps of the headline workload; overlapped = prefetch of "
                           "the next step's experts on a copy stream during the current forward, "
                           "commit on the compute stream; serial = ensure + forward on one stream"}
        del cache, cache_serial, caches

    # ---- end to end through the public API: pinned host in, pinned host out.
    # Every step copies its inputs in from pinned host buffers and its output
    # back to a pinned host buffer, inside the timed region; LayerPipeline runs
    # those copies on a second stream under the neighbouring steps' compute.
    eg = moe.LayerPipeline(cfg.T, cfg.k, routed, shared, device=dev)
    for sl in range(2):
        eg.x_host[sl].copy_(x.cpu())
        eg.logits_host[sl].copy_(logits.cpu())

    def e2e_run(n):
        eg.start()
        for i in range(n):
            eg.step(i)
        eg.finish(n - 1)

    e2e_run(max(args.warmup, 3))
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    if not torch.equal(eg.out_host[(args.steps - 1) % 2].view(torch.int16), lgraph.out.cpu().view(torch.int16)):
        raise SystemExit("end-to-end output differs from the device-resident step")

    ms_step = head["ms_per_step"]
    line = {
        "metric": "moe_layer_tokens_per_s", "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic (seeded), random-init weights of the configured shape",
        "config": head["config"],
        "roofline": head["roofline"], "layer_roofline": head["layer_roofline"],
        "stage_ms": head["stage_ms"],
        "e2e": {"value": world * cfg.T * args.steps / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": x.numel() * 2 + logits.numel() * 4,
                "d2h_bytes_per_step": cfg.T * cfg.d * 2},
        "gpu_launches": head["gpu_launches"],
        "router_gemm": {"us_per_launch": router_us, "algorithmic_bytes": router_bytes,
                        "achieved_gbs": router_bytes / (router_us / 1e6) / 1e9,
                        "kernel": ("tensor cores (tcgen05, 8-CTA cluster per 128 tokens)"
                                   if cfg.E <= 16 and cfg.d % 64 == 0 and cfg.T * max(cfg.E, 8) >= 8192
                                   else "CUDA cores"),
                        "note": "back-to-back launches in one CUDA graph; x and the router weight stay in L2"},
        "router_step": router_step,
        "expert_streaming": {"h2d_gbs_dma": streaming["dma"], "h2d_gbs_sm": streaming["sm"],
                             "expert_image_bytes": sb,
                             "cold_step_ms": L.n_active * sb / (max(v for v in streaming.values() if v) * 1e9)
                                             * 1e3 + ms_step,
                             "note": "LRU expert cache, pinned host images -> 2 HBM slots, 12 images "
                                     "copied per mode; cold_step_ms = every active expert copied in at "
                                     "the faster mode's rate, then the step",
                             "overlapped_decode": overlap},
        "clocks": head["clocks"],
    }
    if want_cpu:
        import oracle
        oracle.build()
        refs = oracle_refs(cfg, L.weights_cpu)
        cores = os.cpu_count() or 1
        toks = list(range(cfg.T))
        n_all = min(cfg.T, cores)
        t_all = time_oracle(cfg, x.cpu(), L.logits_np, refs, toks[:n_all], n_all)
        t_one = time_oracle(cfg, x.cpu(), L.logits_np, refs, toks[:1], 1)
        line["cpu_baseline"] = {
            "value": n_all / t_all, "unit": "tokens/s", "cores": n_all, "nproc": cores, "kind": "oracle",
            "sample": f"{n_all} of {cfg.T} tokens (their {cfg.k} experts each, full d_model x d_ff), "
                      f"one host thread per token on {n_all} of {cores} cores",
            "single_thread": {"value": 1.0 / t_one, "unit": "tokens/s", "cores": 1,
                              "sample": "token 0 on one host thread"}}
    del lgraph, eg, t, L
    torch.cuda.empty_cache()

    # ---- every other workload, same steps and warm-up, each under its own clocks
    workloads = {}
    if not args.no_workloads:
        for name, c in ms.CONFIGS.items():
            if name == cfg.name:
                continue
            Lw = Layer(moe, c, dev, keep_cpu=False)
            tw = time_layer(moe, Lw, args, world, local, dev)
            workloads[name] = summarize(Lw, tw, args, world, hbm, tflops, peak_kind)
            del Lw, tw
            torch.cuda.empty_cache()
        line["workloads"] = workloads
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse()
    cfg = ms.CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_ours(args, cfg)


if __name__ == "__main__":
    main()
