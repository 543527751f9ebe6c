"""Benchmark of the routed-MoE expert stage (and the dense quantised GEMMs).

One step = one moe_expert_stage_w4_iq4 call over the 5268-token prompt
workload (T=5268, D=2048, F=768, E=128, top-8): routing, grouping, W4 gate/up +
SwiGLU + q8_1, IQ4_NL down and the weighted combine.  The dense W4A16
(M=2048, K=5120, N=17408) and FP8 block-128 (M=2048, K=5120, N=5120) products
are timed in the same run and reported under "quant_gemm".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mine|reference]

Multi-GPU (torchrun, one rank per GPU): every rank runs the stage on its own
prompt (independent problems, no collective); value = tokens of all ranks /
max time over ranks ("scaling": "weak").

--impl reference times the CPU oracle (the plain fp64 C implementation the
tests check against) on the host cores, on bounded token samples of the same
workload; rank 0 alone runs it.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synthetic import workloads as wl  # noqa: E402

STAGE = "moe_t5268_d2048_f768_e128_k8"
GEMM_W4 = "w4a16_m2048_k5120_n17408"
GEMM_FP8 = "fp8blk128_m2048_k5120_n5120"
GEMM_ROUTER = "w4a16_router_m2048_k2560_n512"
METRIC = "MoE expert-stage prefill tokens/s; quant-GEMM TFLOP/s vs GB300 tensor peak"
GEMM_TINY = "w4a16_m64_k512_n512"
STAGE_LARGE = "moe_t21504_d2560_f1024_e256_k8_zipf"
# the dense Q8_0 x q8_1 projection: a latent layer's D projection at M = 2048
# (41.3M multiply-adds per row: K = 5120, N = 8064)
Q8_SHAPE = (2048, 5120, 8064)
# DRAM bytes (read + write) per launch of a stage kernel on the 5268-token
# workload, from one ncu capture (profiles/), with the SHA-256 of the kernel's
# sources at the time of the capture: the figure is reported only while the
# sources are unchanged (else null).
DRAM_TRAFFIC = {
    "down": {"bytes": 242750976 + 28232704, "sources_sha": "e0ea5ba104808a9f"},
    "gate_up": {"bytes": 399353088 + 62938368, "sources_sha": "b35d5c0eaaecac4d"},
}
KERNEL_SOURCES = {
    "down": ["csrc/down_iq4.cuh", "csrc/gemm_down.cu", "csrc/qgemm.cuh", "csrc/ptx.cuh"],
    "gate_up": ["csrc/qgemm.cuh", "csrc/gemm_w4.cu", "csrc/ptx.cuh"],
}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def sources_sha(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, "block_quantized_weight_route_gb300", rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str):
    """The captured per-launch DRAM bytes of `kernel`, or None if its sources changed since."""
    t = DRAM_TRAFFIC.get(kernel)
    if not t or t["sources_sha"] != sources_sha(kernel):
        return None
    return t["bytes"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            out = {}
            for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                v = d.get(key)
                if isinstance(v, dict):
                    v = v.get("value")
                if v is not None:
                    out[key] = float(v)
            if "hbm_gbs" in out and "bf16_tflops" in out:
                out.setdefault("bf16_tflops_sustained", out["bf16_tflops"])
                return out, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"qmm_clocks_{os.getpid()}_{gpu_index}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[4:8]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.remove(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def setup_dist(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("QMM_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float, device) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- oracle timing

def time_oracle_stage(g: dict, k: int, ntok: int, cores: int) -> tuple[float, int]:
    """Seconds the CPU oracle takes for the stage on the first `ntok` tokens
    (routing over all tokens, then the full chain for the sample)."""
    os.environ["OMP_NUM_THREADS"] = str(cores)
    import oracle
    toks = np.arange(ntok, dtype=np.int32)
    t0 = time.perf_counter()
    oracle.moe_expert_stage(g["X"], g["logits"], g["Wgu_c"], g["Wgu_s"], g["gu_scale2"], g["Wd_idx"], g["Wd_s"],
                            k, tokens=toks)
    return time.perf_counter() - t0, ntok


def cpu_baseline_sample(g: dict, k: int, target_s: float = 15.0) -> dict:
    cores = os.cpu_count() or 1
    dt, n = time_oracle_stage(g, k, 16, cores)                 # calibration
    ntok = int(max(16, min(4096, target_s / max(dt / n, 1e-6))))
    dt, n = time_oracle_stage(g, k, ntok, cores)
    return {"value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {n} of {g['X'].shape[0]} tokens of {STAGE} (routing over all tokens), "
                      f"{dt:.1f} s, fp32 dequant + fp64 accumulation, OpenMP over outputs"}


# --------------------------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    if rank != 0:
        return
    w = wl.WORKLOADS[STAGE]
    g = wl.generate(w)
    cores = os.cpu_count() or 1
    dt, n = time_oracle_stage(g, w.k, 2, cores)
    per_tok = dt / n
    # each step a bounded sample: the whole --steps/--warmup run stays within ~3 minutes
    ntok = int(max(2, min(256, 150.0 / max(args.steps + args.warmup, 1) / max(per_tok, 1e-6))))
    for _ in range(args.warmup):
        time_oracle_stage(g, w.k, ntok, cores)
    times = []
    for _ in range(args.steps):
        dt, _ = time_oracle_stage(g, w.k, ntok, cores)
        times.append(dt)
    total = sum(times)
    value = ntok * args.steps / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": STAGE, "T": w.T, "D": w.D, "F": w.F, "E": w.E, "k": w.k,
                   "sample_tokens_per_step": ntok},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {ntok} tokens of {STAGE} per step (routing over all {w.T} tokens)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# --------------------------------------------------------------------------- GPU arm

def stage_work(w):
    """Algorithmic work of one expert-stage call: the two grouped GEMMs' flops, the
    down product's fold (one multiply and one FMA per output and 32-K block, on
    the FP32 lanes), the bytes the stage must move (every expert's weights, X, the
    logits, the q8_1 H written and read once, Y), and per-phase bytes of the
    data-movement kernels."""
    P = w.T * w.k
    flops = {"gate_up": 2.0 * P * w.D * 2 * w.F, "down": 2.0 * P * w.F * w.D}
    fold_ops = 2.0 * P * w.D * (w.F // 32)
    weights = w.E * (2 * w.F * w.D // 2 + 2 * w.F * w.D // 16 + w.D * w.F // 2 + w.D * (w.F // 32) * 2 + 4)
    h_bytes = P * w.F + P * (w.F // 32) * 4
    total = weights + w.T * w.D * 2 + w.T * w.E * 4 + 2 * h_bytes + w.T * w.D * 4
    phase_bytes = {
        "route": w.T * w.E * 4 + 4 * P * 4 + P * 4 + w.T * w.D * 4,   # logits in; ids, w, src, row, wrow out; Y zeroed
        "gather": w.T * w.D * 2 + P * w.D * 2,                       # X read once, X_perm written
        "combine": P * w.D * 4 + w.T * w.D * 4 + P * 8,              # (per-slot form) Yslot read, Y written
    }
    return flops, fold_ops, total, phase_bytes


def fp32_lane_ops_peak(sm_mhz: float, sms: int = 152) -> float:
    """FP32 lane operations per second (one FMA or multiply per lane per clock):
    128 lanes per SM at the sampled SM clock, in T/s."""
    return sms * 128 * sm_mhz * 1e6 / 1e12


def stage_roofline(w, ms: float, peaks: dict, sm_mhz: float, sms: int) -> dict:
    """Roofline time of the stage = max(tensor flops / bf16 peak + fold ops / FP32
    lane peak, bytes / HBM bandwidth); fraction = roofline time / measured time."""
    flops, fold_ops, total, _ = stage_work(w)
    t_tensor = sum(flops.values()) / (peaks["bf16_tflops"] * 1e12) * 1e3
    t_fold = fold_ops / (fp32_lane_ops_peak(sm_mhz, sms) * 1e12) * 1e3
    t_hbm = total / (peaks["hbm_gbs"] * 1e9) * 1e3
    roof = max(t_tensor + t_fold, t_hbm)
    return {"measured_ms": ms, "roofline_ms": roof, "frac": roof / ms, "tensor_ms": t_tensor, "fold_ms": t_fold,
            "hbm_ms": t_hbm, "flops": sum(flops.values()), "fold_ops": fold_ops, "bytes": total,
            "peaks": "bf16 burst and HBM copy of MEASURED_PEAKS.json; FP32 lanes 152 x 128 x sampled SM clock"}


def phase_rooflines(w, phases: dict, peaks: dict, peak_src: str, sm_mhz: float, sms: int) -> dict:
    flops, fold_ops, _, pbytes = stage_work(w)
    pk_t = peaks["bf16_tflops"]
    out = {}
    for name, ms in phases.items():
        if name in flops:
            ach = flops[name] / (ms * 1e-3) / 1e12
            r = {"ms": ms, "bound": "tensor", "achieved": ach, "peak": pk_t, "unit": "TFLOP/s", "frac": ach / pk_t,
                 "peak_source": f"{peak_src} (burst bf16)"}
            if name == "down":
                # the exact integer block dots run on the f16 tensor pipe; the fp32 fold
                # of every 32-K block's dot runs on the FP32 lanes beside it
                pk_f = fp32_lane_ops_peak(sm_mhz, sms)
                fa = fold_ops / (ms * 1e-3) / 1e12
                r["fold"] = {"ops": fold_ops, "achieved": fa, "peak": pk_f, "unit": "T lane-ops/s", "frac": fa / pk_f}
            out[name] = r
        elif ms > 0.005:
            ach = pbytes[name] / (ms * 1e-3) / 1e9
            out[name] = {"ms": ms, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"]}
        else:
            out[name] = {"ms": ms, "note": "empty: the combine runs inside the down product"}
    return out


def expert_histogram(q, ws, w) -> dict:
    """Rows per expert of the last stage call (the workspace's counts region)."""
    import torch
    lay = q.moe_expert_stage_workspace_layout(w.T, w.D, w.F, w.E, w.k)
    c = q.workspace_view(ws, lay, "counts", torch.int32, (w.E,)).cpu().numpy()
    return {"max": int(c.max()), "mean": float(c.mean()), "min": int(c.min()), "max_over_mean": float(c.max() / c.mean()),
            "experts_under_128_rows": int((c < 128).sum()), "empty_experts": int((c == 0).sum())}


def run_gpu(args, world, rank, local):
    import torch
    import block_quantized_weight_route_gb300 as q

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    q.build_library()
    peaks, peak_src = load_peaks()

    w = wl.WORKLOADS[STAGE]
    g = wl.generate(w)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
    X = d(g["X"].view(np.int16))
    logits = d(g["logits"])
    Wgu_c, Wgu_s, s2 = d(g["Wgu_c"]), d(g["Wgu_s"]), d(g["gu_scale2"])
    Wd_idx, Wd_s = d(g["Wd_idx"]), d(g["Wd_s"].view(np.int16))
    ws = torch.empty(q.moe_expert_stage_workspace_size(w.T, w.D, w.F, w.E, w.k), dtype=torch.uint8, device=device)
    Y = torch.empty((w.T, w.D), dtype=torch.float32, device=device)

    def step():
        q.moe_expert_stage_w4_iq4(X, logits, Wgu_c, Wgu_s, s2, Wd_idx, Wd_s, w.k, ws=ws, Y=Y)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    q.qmm_check_status()

    # ---- timed region: K steps, inputs (340 MB of weights per step) larger than L2
    q.qmm_profile_enable(True)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    phase_ms = []
    t_wall = time.perf_counter()
    for i in range(args.steps):          # no host wait between steps: phases are read afterwards
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    phase_ms = [q.qmm_profile_read_call(i) for i in range(max(0, args.steps - 256), args.steps)]
    barrier(world)
    wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    q.qmm_profile_enable(False)
    q.qmm_check_status()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_s = max_over_ranks(world, sum(step_ms) / 1e3, device)
    value = w.T * world * args.steps / total_s

    phases = {k: statistics.mean(p[k] for p in phase_ms) for k in q.PROFILE_PHASES}
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    sm_mhz = clk.get("sm_mhz") or 2070.0
    phase_roof = phase_rooflines(w, phases, peaks, peak_src, sm_mhz, sms)
    # the dominant kernel: on the tensor pipe against the burst bf16 peak (a kernel
    # of a ~1 ms step), the down product's fold beside it
    dom = max((n for n in phases if "bound" in phase_roof[n]), key=phases.get)
    roof = {k: v for k, v in phase_roof[dom].items() if k != "ms"}
    roof["kernel"] = dom
    roof["traffic"] = dram_traffic(dom)
    roof["traffic_note"] = ("DRAM read + write bytes per launch from the ncu capture of these sources"
                            if roof["traffic"] is not None else "no ncu capture of the kernel's current sources")
    stage_roof = stage_roofline(w, 1e3 * total_s / (args.steps * world), peaks, sm_mhz, sms)
    hist = expert_histogram(q, ws, w)

    # the per-slot form of the stage (QMM_STAGE_SLOTS: separate j-ordered combine,
    # reproducible bit for bit), timed the same way as context
    for _ in range(2):
        q.moe_expert_stage_w4_iq4(X, logits, Wgu_c, Wgu_s, s2, Wd_idx, Wd_s, w.k, ws=ws, Y=Y, slots=True)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nsl = max(3, min(20, args.steps))
    a.record(stream)
    for _ in range(nsl):
        q.moe_expert_stage_w4_iq4(X, logits, Wgu_c, Wgu_s, s2, Wd_idx, Wd_s, w.k, ws=ws, Y=Y, slots=True)
    b.record(stream)
    torch.cuda.synchronize()
    slots_ms = a.elapsed_time(b) / nsl
    step()                         # leave the default form's Y for the end-to-end check
    torch.cuda.synchronize()

    # ---- end to end through the public API: every step copies its own inputs in
    # from pinned host memory and its Y back out.  Double-buffered the way a
    # serving loop runs it: step i+1's inputs go in (H2D stream) and step i-1's Y
    # comes out (D2H stream) while step i computes, ordered by events.
    nb = 2
    Xh = [torch.from_numpy(g["X"].view(np.int16)).pin_memory() for _ in range(nb)]
    Lh = [torch.from_numpy(g["logits"]).pin_memory() for _ in range(nb)]
    Yh = [torch.empty((w.T, w.D), dtype=torch.float32).pin_memory() for _ in range(nb)]
    Xd = [torch.empty_like(X) for _ in range(nb)]
    Ld = [torch.empty_like(logits) for _ in range(nb)]
    Yd = [torch.empty_like(Y) for _ in range(nb)]
    h2d, d2h = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready = [ev() for _ in range(args.steps)]
    done = [ev() for _ in range(args.steps)]
    out_done = [ev() for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d.wait_stream(stream)
    d2h.wait_stream(stream)
    for i in range(args.steps):
        b = i % nb
        with torch.cuda.stream(h2d):
            if i >= nb:
                h2d.wait_event(done[i - nb])              # step i-nb has finished reading these buffers
            Xd[b].copy_(Xh[b], non_blocking=True)
            Ld[b].copy_(Lh[b], non_blocking=True)
            in_ready[i].record(h2d)
        stream.wait_event(in_ready[i])
        if i >= nb:
            stream.wait_event(out_done[i - nb])           # Yd[b] has been copied out
        q.moe_expert_stage_w4_iq4(Xd[b], Ld[b], Wgu_c, Wgu_s, s2, Wd_idx, Wd_s, w.k, ws=ws, Y=Yd[b])
        done[i].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(done[i])
            Yh[b].copy_(Yd[b], non_blocking=True)
            out_done[i].record(d2h)
    stream.wait_event(out_done[args.steps - 1])
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(world, e0.elapsed_time(e1) / 1e3, device)
    # the last step's Y, checked against the device-timed run's Y (same inputs; the
    # fused combine adds each token's k terms in no fixed order, so up to rounding)
    Yl, Yr = Yh[(args.steps - 1) % nb], Y.cpu()
    assert float((Yl - Yr).abs().max()) <= 1e-6 * float(Yr.abs().max()), \
        "end-to-end output differs from the device-timed output"
    e2e = {"value": w.T * world * args.steps / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": int(Xh[0].numel() * 2 + Lh[0].numel() * 4), "d2h_bytes_per_step": int(Yh[0].numel() * 4),
           "overlap": "double-buffered: H2D of step i+1 and D2H of step i-1 on their own streams while step i computes"}
    del Xd, Ld, Yd
    del ws, Y, X, Wgu_c, Wgu_s, Wd_idx, Wd_s
    torch.cuda.empty_cache()

    quant = {} if args.no_gemm else bench_dense(q, torch, device, args, peaks, peak_src)
    other = {} if args.no_gemm else bench_other_stage(q, torch, device, args, peaks, peak_src, sms)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16/f16 operands, f32 accumulate", "data": "synthetic",
        "config": {"workload": STAGE, "T": w.T, "D": w.D, "F": w.F, "E": w.E, "k": w.k,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (340 MB of expert weights read per step)",
                   "timing": "CUDA events per step; phase events between the stage's kernels inside the timed steps "
                             "(the e2e loop records none)"},
        "roofline": roof, "stage_roofline": stage_roof, "phases": phase_roof, "expert_counts": hist,
        "stage_slots_ms": slots_ms, "quant_gemm": quant, "other_stage": other, "e2e": e2e, "clocks": clk,
        # per step: top-k, histogram, scan, permutation, gather, gate/up, down (combine fused)
        "gpu_launches": 7 * args.steps, "wall_s": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_sample(g, w.k)
    if rank == 0:
        print(json.dumps(line))


def bench_other_stage(q, torch, device, args, peaks, peak_src, sms):
    """The larger stage configuration (T=21504, D=2560, F=1024, E=256, Zipf(1.1)
    expert popularity: load imbalance and tail experts), timed like the headline
    stage: CUDA events per step, phase events, roofline, per-expert counts."""
    w = wl.WORKLOADS[STAGE_LARGE]
    g = wl.generate(w)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
    X, L = d(g["X"].view(np.int16)), d(g["logits"])
    args_ = (d(g["Wgu_c"]), d(g["Wgu_s"]), d(g["gu_scale2"]), d(g["Wd_idx"]), d(g["Wd_s"].view(np.int16)))
    ws = torch.empty(q.moe_expert_stage_workspace_size(w.T, w.D, w.F, w.E, w.k), dtype=torch.uint8, device=device)
    Y = torch.empty((w.T, w.D), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        q.moe_expert_stage_w4_iq4(X, L, *args_, w.k, ws=ws, Y=Y)
    torch.cuda.synchronize()
    n = max(3, min(20, args.steps))
    q.qmm_profile_enable(True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    for i in range(n):
        ev[i][0].record(stream)
        q.moe_expert_stage_w4_iq4(X, L, *args_, w.k, ws=ws, Y=Y)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ph = [q.qmm_profile_read_call(i) for i in range(n)]
    q.qmm_profile_enable(False)
    q.qmm_check_status()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    phases = {k: statistics.mean(p[k] for p in ph) for k in q.PROFILE_PHASES}
    sm_mhz = clk.get("sm_mhz") or 2070.0
    out = {STAGE_LARGE: {"ms": ms, "tokens_per_s": w.T / (ms * 1e-3), "tflops": w.flops() / (ms * 1e-3) / 1e12,
                         "steps": n, "stage_roofline": stage_roofline(w, ms, peaks, sm_mhz, sms),
                         "phases": phase_rooflines(w, phases, peaks, peak_src, sm_mhz, sms),
                         "expert_counts": expert_histogram(q, ws, w), "clocks": clk}}
    del ws, Y, X, L, args_
    torch.cuda.empty_cache()
    return out


def bench_dense(q, torch, device, args, peaks, peak_src):
    """Dense W4A16 and FP8 block-128 GEMMs: per-launch CUDA events, L2 flushed before each launch."""
    out = {}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    for name in (GEMM_TINY, GEMM_W4, GEMM_FP8, GEMM_ROUTER):
        w = wl.WORKLOADS[name]
        g = wl.generate(w)
        d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
        X = d(g["X"].view(np.int16))
        # the K-split workspace, allocated once outside the timed launches
        nws = q.qmm_dense_workspace_size(w.M, w.K, w.N)
        dws = torch.empty(max(nws, 1), dtype=torch.uint8, device=device)
        if w.kind == "w4a16":
            Wc, Ws = d(g["Wc"]), d(g["Ws"])
            odt = torch.bfloat16 if w.out == "bf16" else torch.float32
            Y = torch.empty((w.M, w.N), dtype=odt, device=device)
            call = lambda: q.qmm_w4a16(X, Wc, Ws, float(g["scale2"]), out_dtype=odt, Y=Y, ws=dws)  # noqa: E731
        else:
            W, S = d(g["W"]), d(g["S"])
            Y = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=device)
            call = lambda: q.qmm_fp8_blk128(X, W, S, Y=Y, ws=dws)  # noqa: E731
        for _ in range(max(3, args.warmup)):
            call()
        torch.cuda.synchronize()
        times = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        q.qmm_check_status()
        ms = statistics.mean(times)
        tfl = w.flops() / (ms * 1e-3) / 1e12
        out[name] = {"ms": ms, "tflops": tfl, "peak": peaks["bf16_tflops"], "frac": tfl / peaks["bf16_tflops"],
                     "peak_source": f"{peak_src} (burst bf16)", "l2": "flushed before each launch"}
        if name == GEMM_TINY:
            # latency-bound: also the bytes it must move (X, codes, scales, Y) against HBM
            nbytes = w.M * w.K * 2 + w.N * w.K // 2 + w.N * w.K // 16 + w.M * w.N * 4
            out[name].update({"us": ms * 1e3, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
                              "bound": "latency (reported, not targeted)"})
        del X, Y, dws
        torch.cuda.empty_cache()
    # the dense Q8_0 x q8_1 projection re-quantised to q8_1 (a latent layer's D)
    M, K, N = Q8_SHAPE
    g = wl.gen_q8_0_q8_1(M, K, N, seed=6)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)  # noqa: E731
    Xq, Xd, Wq, Wd = d(g["Xq"]), d(g["Xd"].view(np.int16)), d(g["Wq"]), d(g["Wd"].view(np.int16))
    qws = torch.empty(q.qmm_q8_0_q8_1_workspace_size(M, K, N), dtype=torch.uint8, device=device)
    for _ in range(max(3, args.warmup)):
        q.qmm_q8_0_q8_1(Xq, Xd, Wq, Wd, ws=qws)
    torch.cuda.synchronize()
    times = []
    for _ in range(args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        q.qmm_q8_0_q8_1(Xq, Xd, Wq, Wd, ws=qws)
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    q.qmm_check_status()
    ms = statistics.mean(times)
    tfl = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    out[f"q8_0_q8_1_m{M}_k{K}_n{N}"] = {"ms": ms, "tflops": tfl, "peak": peaks["bf16_tflops"],
                                          "frac": tfl / peaks["bf16_tflops"], "peak_source": f"{peak_src} (burst bf16)",
                                          "l2": "flushed before each launch",
                                          "note": "exact int8 block dots on the f16 tensor path + fp32 fold"}
    del Xq, Xd, Wq, Wd, qws
    torch.cuda.empty_cache()
    return out


def run_case(args):
    """Run one op `--steps` times after `--warmup` runs (no JSON line): a small,
    fixed command for profiler captures of a single kernel family."""
    import torch
    import block_quantized_weight_route_gb300 as q
    q.build_library()
    dev = torch.device("cuda", 0)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    if args.case in ("stage", "stage_large"):
        w = wl.WORKLOADS[STAGE if args.case == "stage" else STAGE_LARGE]
        g = wl.generate(w)
        X, L = d(g["X"].view(np.int16)), d(g["logits"])
        args_ = (d(g["Wgu_c"]), d(g["Wgu_s"]), d(g["gu_scale2"]), d(g["Wd_idx"]), d(g["Wd_s"].view(np.int16)))
        ws = torch.empty(q.moe_expert_stage_workspace_size(w.T, w.D, w.F, w.E, w.k), dtype=torch.uint8, device=dev)
        call = lambda: q.moe_expert_stage_w4_iq4(X, L, *args_, w.k, ws=ws)  # noqa: E731
    elif args.case == "w4a16":
        w = wl.WORKLOADS[GEMM_W4]
        g = wl.generate(w)
        X, Wc, Ws = d(g["X"].view(np.int16)), d(g["Wc"]), d(g["Ws"])
        call = lambda: q.qmm_w4a16(X, Wc, Ws, float(g["scale2"]), out_dtype=torch.bfloat16)  # noqa: E731
    elif args.case == "q8":
        M, K, N = Q8_SHAPE
        g = wl.gen_q8_0_q8_1(M, K, N, seed=6)
        Xq, Xd, Wq, Wd = d(g["Xq"]), d(g["Xd"].view(np.int16)), d(g["Wq"]), d(g["Wd"].view(np.int16))
        call = lambda: q.qmm_q8_0_q8_1(Xq, Xd, Wq, Wd)  # noqa: E731
    else:
        w = wl.WORKLOADS[GEMM_FP8]
        g = wl.generate(w)
        X, W, S = d(g["X"].view(np.int16)), d(g["W"]), d(g["S"])
        call = lambda: q.qmm_fp8_blk128(X, W, S)  # noqa: E731
    for _ in range(args.warmup_case):
        call()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        call()
    torch.cuda.synchronize()
    q.qmm_check_status()
    print(f"case {args.case}: {args.steps} runs, {1e3 * (time.perf_counter() - t0) / args.steps:.3f} ms/run (wall)")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["mine", "reference"], default="mine")
    ap.add_argument("--no-gemm", action="store_true", help="skip the dense GEMM measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["stage", "stage_large", "w4a16", "fp8", "q8"], default=None,
                    help="run one op only (for profiler captures); prints no JSON line")
    ap.add_argument("--warmup-case", type=int, default=1, help="untimed runs before --steps in --case mode")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = setup_dist(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
