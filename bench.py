"""Benchmark of the LatentMoE layer forward (one JSON line on rank 0).

Default workload: the MAI-Base-1-shaped layer (T=16384 tokens, hidden 6656,
latent 3072, 512 experts, top-8, SwiGLU FFN 10240, bf16, ~97 GB of expert
weights resident). A step is one full forward through the C ABI. Inputs are
larger than L2 (every step streams all touched expert weights from HBM).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--fp8]
  python bench.py --impl reference ...   # the float64 CPU oracle, rank 0 only

--fp8 runs the expert GEMMs in FP8 E4M3 with delayed scaling (a separate
metric; the default line is the bf16 forward).

Multi-GPU runs are independent replicas (one process per GPU, weak scaling);
the only collectives are the timing barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "LatentMoE bf16 fwd tokens/s at MAI-Base-1 shape; % of tensor-core roofline"
METRIC_FP8 = ("LatentMoE fwd tokens/s at MAI-Base-1 shape with FP8 E4M3 expert GEMMs; "
              "% of tensor-core roofline")
METRIC_FP8_DENSE = ("LatentMoE fwd tokens/s at MAI-Base-1 shape with FP8 E4M3 GEMMs (router "
                    "fp32); % of tensor-core roofline")
# dense E4M3 tensor rate over dense bf16 (nominal 4.5 vs 2.25 PFLOP/s)
FP8_OVER_BF16 = 2.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DOMINANT = "expert_gate_up"
GEMM_SRC = [os.path.join(ROOT, "mixture_experts_layer_router_gb300", "csrc", f)
            for f in ("gemm_grouped.cuh", "gemm_grouped2.cuh", "ptx.cuh", "ptx_pair.cuh",
                      "fp8.cuh")]


# ---------------------------------------------------------------- arithmetic

def layer_flops_per_token(c) -> int:
    """Router, latent down, k expert SwiGLU FFNs, latent up, shared expert."""
    return 2 * c.d * c.E + 2 * c.d * c.l + 6 * c.k * c.l * c.F + 2 * c.l * c.d + 6 * c.d * c.Fs


def expert_flops_per_token(c) -> int:
    return 6 * c.k * c.l * c.F


def layer_bytes(c, touched_experts: int, eb: int = 2, db: int = 2) -> int:
    """Algorithmic bytes: weights read once (experts that got tokens only,
    eb bytes per expert weight, db per latent-projection and shared-expert
    weight; the router's weights in bf16), x read once, y written once;
    intermediates excluded as avoidable."""
    w = touched_experts * 3 * c.l * c.F * eb + c.E * c.d * 2 + \
        (2 * c.l * c.d + 3 * c.d * c.Fs) * db
    return w + c.T * c.d * 2 * 2


def gate_up_work(c, touched_experts: int, eb: int = 2):
    """Per launch of the grouped gate+up GEMM: FLOPs, algorithmic bytes (the
    gate and up weights of the experts that got tokens, eb bytes each: 2 for
    bf16, 1 for E4M3; the z rows it reads and the h rows it writes are
    intermediates a fused design avoids, so they are not counted) and the
    as-built bytes (weights + z rows read + h rows written)."""
    S = c.T * c.k
    flops = 2 * S * c.l * 2 * c.F
    nbytes = touched_experts * 2 * c.F * c.l * eb
    built = nbytes + S * c.l * eb + S * c.F * eb
    return flops, nbytes, built


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
            "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def profiled_traffic(workload: str, fp8: bool = False):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    kernel = DOMINANT + ("_e4m3" if fp8 else "")
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.txt")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    m_tr = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_sha and m_tr):
        return None
    h = hashlib.sha256()
    for f in GEMM_SRC:
        h.update(open(f, "rb").read())
    cur = h.hexdigest()
    return float(m_tr.group(1)) if m_sha.group(1) == cur else None


def max_over_ranks(value: float, dist, device="cpu") -> float:
    """The largest value over all ranks (the job's time is its slowest rank's);
    the value itself on one process."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,clocks.mem,clocks.max.mem")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(1.0)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.seek(0)
        rows = [r.split(", ") for r in self.file.read().strip().splitlines() if r.count(",") >= 9]
        os.unlink(self.file.name)
        samples = []
        for r in rows:
            try:
                whole, _, frac = r[0].partition(".")
                ts = time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + float("0." + (frac or "0"))
                samples.append((ts, float(r[1]), float(r[2]), r[4:8], float(r[3]), float(r[8]),
                                float(r[9])))
            except Exception:
                continue
        inside = [s for s in samples if t0 <= s[0] <= t1]
        if len(inside) < 3:
            inside = [s for s in samples if t0 - 0.5 <= s[0] <= t1 + 0.5] or samples
        if not inside:
            return None
        mhz = sorted(s[1] for s in inside)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i, v in enumerate(s[3])
                          if v.strip().lower() == "active"})
        mem = sorted(s[5] for s in inside)
        watts = sorted(s[4] for s in inside)
        return {"sm_mhz": mhz[len(mhz) // 2], "sm_max_mhz": max(s[2] for s in inside),
                "reasons": reasons, "samples": len(inside),
                "mem_mhz": mem[len(mem) // 2], "mem_max_mhz": max(s[6] for s in inside),
                "power_w": watts[len(watts) // 2]}


# ---------------------------------------------------------------- oracle legs

def oracle_tokens_per_s(cfg, x_rows, logits_rows, fetch, repeats=1, fp8_scales=None):
    """Time the float64 oracle on given token rows; returns (tokens/s, s).
    With fp8_scales (s_z, s_h) the oracle's E4M3 expert layer is timed; with
    (s_z, s_h, s_x, s_c, s_sh) the all-E4M3 layer."""
    from oracle import latentmoe_ref as ref
    from oracle import fp8 as ofp8
    import numpy as np
    W = ref.OracleWeights(fetch["w_r"], fetch["w_dn"], fetch["w_up"], fetch["expert"],
                          b_r=fetch["b_r"], w_gs=fetch["w_gs"], w_us=fetch["w_us"],
                          w_ds=fetch["w_ds"])
    t0 = time.perf_counter()
    for _ in range(repeats):
        xr = np.asarray(x_rows, dtype=np.float64)
        if fp8_scales is None:
            ref.forward(xr, W, cfg.k, logits=logits_rows)
        else:
            dense = None if len(fp8_scales) == 2 else \
                {"s_x": fp8_scales[2], "s_c": fp8_scales[3], "s_sh": fp8_scales[4]}
            ofp8.forward_fp8(xr, W, cfg.k, s_z=fp8_scales[0], s_h=fp8_scales[1],
                             logits=logits_rows, dense=dense)
    dt = time.perf_counter() - t0
    return x_rows.shape[0] * repeats / dt, dt


def host_weights(cfg, w, experts):
    """bf16 weights as host float32 arrays (exact), with the experts needed."""
    import numpy as np

    def h(t):
        return None if t is None else t.detach().float().cpu().numpy()
    ex = {}
    for e in experts:
        if w.get("w_g") is not None:
            ex[e] = (h(w["w_g"][e]), h(w["w_u"][e]), h(w["w_d"][e]))
        else:
            from mixture_experts_layer_router_gb300 import synth
            dev = "cuda" if _cuda_ok() else "cpu"
            ex[e] = tuple(h(t) for t in synth.make_expert(cfg, e, 0, dev))

    def expert(e):
        return tuple(a.astype(np.float64) for a in ex[e])
    return {"w_r": h(w["w_r"]), "b_r": h(w["b_r"]), "w_dn": h(w["w_dn"]), "w_up": h(w["w_up"]),
            "w_gs": h(w["w_gs"]), "w_us": h(w["w_us"]), "w_ds": h(w["w_ds"]), "expert": expert}


def _cuda_ok():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def cores_used():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- arms

def run_reference(args, cfg, rank, world):
    """The oracle on the host cores: each step is a bounded token sample."""
    if rank != 0:
        return None
    import numpy as np
    import torch
    from mixture_experts_layer_router_gb300 import synth
    from oracle import latentmoe_ref as ref
    dev = "cuda" if _cuda_ok() else "cpu"
    n_steps = args.warmup + args.steps
    per_step = args.ref_tokens
    toks = synth.sample_tokens(cfg.T, n_steps * per_step, seed=1).numpy()
    w = synth.make_weights(cfg, 0, dev, experts=False)
    x = synth.make_x(cfg, 0, dev)
    xs = x[torch.from_numpy(toks).to(dev)].float().cpu().numpy().astype(np.float64)
    L = ref.router_logits(xs, w["w_r"].float().cpu().numpy().astype(np.float64),
                          None if w["b_r"] is None else w["b_r"].cpu().numpy().astype(np.float64))
    need = sorted(set(ref.top_k_stable(L, cfg.k).ravel().tolist()))
    fetch = host_weights(cfg, w, need)
    del w, x
    times = []
    for i in range(n_steps):
        rows = slice(i * per_step, (i + 1) * per_step)
        _, dt = oracle_tokens_per_s(cfg, xs[rows], None, fetch)
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = args.steps * per_step / total
    line = {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores_used(),
                         "kind": "oracle",
                         "sample": f"{per_step} seeded token(s) of the {cfg.name} workload per "
                                   "step, float64 NumPy oracle with its expert weights upcast "
                                   "from host bf16 inside the timed work"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


def workload_config(cfg):
    return {"workload": f"{cfg.name} LatentMoE layer forward: T={cfg.T} d={cfg.d} l={cfg.l} "
                        f"E={cfg.E} top-{cfg.k} F={cfg.F}" + (f" shared F={cfg.Fs}" if cfg.Fs else ""),
            "T": cfg.T, "d": cfg.d, "l": cfg.l, "E": cfg.E, "k": cfg.k, "F": cfg.F, "Fs": cfg.Fs,
            "l2": "inputs larger than L2 (all touched expert weights stream from HBM every step)",
            "parallelism": "replicas"}


def layer_roofline(cfg, touched, ms_step, peaks, peak_src, f8, fp8_dense, capped):
    """FLOPs, algorithmic bytes and the layer's roofline fraction. The tensor
    peak is the measured sustained one for a run the power cap held down,
    the burst one otherwise; E4M3 FLOPs count at the nominal E4M3/bf16 ratio."""
    flops_tok = layer_flops_per_token(cfg)
    eb = 1 if f8 else 2
    lbytes = layer_bytes(cfg, touched, eb, 1 if fp8_dense else 2)
    peak_key = "bf16_tflops_sustained" if capped else "bf16_tflops"
    bf16_peak = peaks[peak_key] * 1e12
    router_flops = cfg.T * 2 * cfg.d * cfg.E
    x_flops = cfg.T * expert_flops_per_token(cfg)
    if fp8_dense:
        x_flops = cfg.T * flops_tok - router_flops
    o_flops = cfg.T * flops_tok - x_flops
    tc_ms = (o_flops / bf16_peak + x_flops / (bf16_peak * (FP8_OVER_BF16 if f8 else 1.0))) * 1e3
    hbm_ms = lbytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    return {"flops": cfg.T * flops_tok, "bytes": lbytes, "tc_ms": tc_ms, "hbm_ms": hbm_ms,
            "roofline_ms": max(tc_ms, hbm_ms), "frac": max(tc_ms, hbm_ms) / ms_step,
            "touched_experts": touched,
            "tensor_peak": f"{peak_src} {'sustained' if capped else 'burst'} bf16 "
                           f"({peaks[peak_key]:.1f} TFLOP/s)",
            "peaks": {**peaks, "source": peak_src}}


def cpu_oracle_baseline(cfg, r, x, w, n, f8_scales=None, fp8_dense=False):
    """The oracle on n seeded tokens of the workload (all T when n >= T),
    routed from the GPU logits; tokens/s, with the full-T time extrapolated
    where n < T."""
    import numpy as np
    from mixture_experts_layer_router_gb300 import synth
    n = min(n, cfg.T)
    toks = synth.sample_tokens(cfg.T, n, seed=1)
    tsel = toks.cuda()
    L = r["logits"][tsel].double().cpu().numpy()
    need = sorted(set(r["idx"][tsel].cpu().numpy().ravel().tolist()))
    fetch = host_weights(cfg, w, need)
    xs = x[tsel].float().cpu().numpy().astype(np.float64)
    tps, dt = oracle_tokens_per_s(cfg, xs, L, fetch, fp8_scales=f8_scales)
    what = "all tokens" if n == cfg.T else f"{n} seeded tokens"
    out = {"value": tps, "unit": "tokens/s", "cores": cores_used(), "kind": "oracle",
           "sample": f"{what} of the {cfg.name} workload ({dt:.1f} s), float64 NumPy oracle" +
                     ((" (E4M3 layer at the GPU's scales)" if f8_scales is not None else "")) +
                     " routed from the GPU logits, expert weights upcast from host bf16 inside "
                     "the timed work"}
    if n < cfg.T:
        out["extrapolated_s_per_forward"] = dt * cfg.T / n
        out["extrapolation"] = (f"x T/n = x {cfg.T / n:.0f}: overstates the per-expert fixed "
                                "costs (weight upcast), which a full-T run pays once")
    return out


def measure_small(cfg, args, peaks, peak_src, local, cpu_tokens):
    """One extra workload at N = 1: the same forward through the C ABI, each
    timed step bracketed by CUDA events after an L2 flush (a 512 MiB write),
    then a profiled pass for the stage times; its own clock record and CPU
    baseline. Returns the entry of the line's "configs"."""
    import torch
    from mixture_experts_layer_router_gb300 import capi, synth
    w = synth.make_weights(cfg, 0, "cuda")
    x = synth.make_x(cfg, 0, "cuda")
    layer = capi.LatentMoE(cfg.d, cfg.l, cfg.E, cfg.k, cfg.F, cfg.Fs, max_tokens=cfg.T,
                           router_bias=w["b_r"] is not None)
    layer.load_weights(w)
    if args.no_pdl:
        layer.set_pdl(False)
    if args.no_fusion:
        layer.set_expert_fusion(0)
    elif args.fusion:
        layer.set_expert_fusion(1)
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        layer.forward(x, y)
    torch.cuda.synchronize()
    assert layer.status() == 0, f"device status set during the {cfg.name} warm-up"
    t0 = time.perf_counter()
    for _ in range(5):
        layer.forward(x, y)
    torch.cuda.synchronize()
    est_ms = (time.perf_counter() - t0) * 1e3 / 5
    # enough steps for the clock sampler (>= 0.6 s of timed work)
    steps = max(args.steps, int(600.0 / max(est_ms, 0.02)) + 1)
    steps = min(steps, 20000)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    clocks = ClockSampler(local)
    clocks.start()
    launches0 = layer.launch_count()
    torch.cuda.synchronize()
    wall0 = time.time()
    for a, b in evs:
        flush.fill_(1)
        a.record(stream)
        layer.forward(x, y)
        b.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    launches = layer.launch_count() - launches0
    clk = clocks.stop(wall0, wall1)
    ms = sorted(a.elapsed_time(b) for a, b in evs)
    ms_mean = sum(ms) / len(ms)
    prof = min(steps, 200)
    layer.set_profiling(prof)
    for _ in range(prof):
        flush.fill_(1)
        layer.forward(x, y)
    torch.cuda.synchronize()
    stage_ms = {}
    for s in range(prof):
        for name, v in layer.stage_times(s).items():
            stage_ms[name] = stage_ms.get(name, 0.0) + v / prof
    layer.set_profiling(0)
    status = layer.status()
    r = layer.get_routing(cfg.T, "cuda")
    touched = int((r["counts"] > 0).sum().item())
    capped = bool(clk and "sw_power_cap" in clk.get("reasons", []))
    roof = layer_roofline(cfg, touched, ms_mean, peaks, peak_src, False, False, capped)
    cpu = cpu_oracle_baseline(cfg, r, x, w, cpu_tokens) if not args.no_cpu_baseline else None
    out = {"workload": workload_config(cfg)["workload"], "steps": steps,
           "ms_per_step": ms_mean, "ms_per_step_median": ms[len(ms) // 2],
           "tokens_per_s": cfg.T / (ms_mean / 1e3),
           "tflops": roof["flops"] / (ms_mean / 1e3) / 1e12,
           "roofline_frac": roof["frac"], "layer_roofline": roof,
           "l2": "flushed before every timed step (512 MiB write outside the events)",
           "stage_ms": stage_ms, "gpu_launches_per_step": launches / steps,
           "clocks": clk, "cpu_baseline": cpu, "device_status": status}
    layer.close()
    del layer, w, x, y, flush
    torch.cuda.empty_cache()
    return out


EXTRA_CONFIGS = (("tiny", 128), ("mid", 4096), ("imbalanced", 4096), ("mai-base-2", 12))


def run_ours(args, cfg, rank, world, dist):
    import numpy as np  # noqa: F401
    import torch
    from mixture_experts_layer_router_gb300 import build, capi, synth

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    # one rank builds (a no-op when the library is current); the others wait
    if rank == 0:
        build.build()
    if dist is not None:
        dist.barrier()
    capi.load()
    w = synth.make_weights(cfg, 0, "cuda")
    x = synth.make_x(cfg, 0, "cuda")
    f8 = args.fp8 or args.fp8_dense
    layer = capi.LatentMoE(cfg.d, cfg.l, cfg.E, cfg.k, cfg.F, cfg.Fs, max_tokens=cfg.T,
                           router_bias=w["b_r"] is not None, fp8=f8, fp8_dense=args.fp8_dense)
    layer.load_weights(w)
    if args.no_sm_pairs:
        layer.set_sm_pairs(False)
    if args.no_pdl:
        layer.set_pdl(False)
    if args.no_fusion:
        layer.set_expert_fusion(0)
    elif args.fusion:
        layer.set_expert_fusion(1)
    if args.capacity > 0:
        layer.set_capacity(args.capacity, args.group_size, args.max_rounds)
    # the library holds its own (packed) copy; the expert weights the CPU
    # baseline needs are regenerated from their per-expert seeds
    for key in ("w_g", "w_u", "w_d"):
        w[key] = None
    torch.cuda.empty_cache()
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        layer.forward(x, y)
    torch.cuda.synchronize()
    assert layer.status() == 0, "device status set during warm-up"
    fp8_state = layer.fp8_state() if f8 else None
    rounds_info = None
    if args.capacity > 0:
        ri = layer.rounds()
        rounds_info = {"needed": ri["needed"], "launched": ri["launched"],
                       "left_over": ri["left_over"]}
    r = layer.get_routing(cfg.T, "cuda")
    counts = r["counts"].cpu().numpy()
    touched = int((counts > 0).sum())
    layer.set_profiling(args.steps)

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    launches0 = layer.launch_count()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        layer.forward(x, y)
    e1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if dist is not None:
        dist.barrier()
    ms_total = e0.elapsed_time(e1)
    launches = layer.launch_count() - launches0
    clk = clocks.stop(wall0, wall1) if rank == 0 else None
    stage_ms = {}
    for s in range(args.steps):
        for name, v in layer.stage_times(s).items():
            stage_ms[name] = stage_ms.get(name, 0.0) + v / args.steps
    status = layer.status()
    layer.set_profiling(0)

    ms_total = max_over_ranks(ms_total, dist, "cuda")

    # end to end through the host-buffer entry points: pinned x in, y out, every
    # step. The headline uses the pipelined entry (step i+1's input copy and
    # step i-1's output copy run during step i's forward); the synchronous
    # entry (copy in, forward, copy out, wait) is reported beside it.
    e2e = None
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        yh = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16).pin_memory()
        layer.forward_host(xh, yh)
        for _ in range(2):
            layer.forward_host_async(xh, yh)
        layer.host_wait()
        n_e2e = max(3, min(args.steps, 20))
        # its own clock record: this region runs at whatever clock the power
        # cap allows by then, which can differ from the device-timed region's
        e2e_clocks = ClockSampler(local)
        e2e_clocks.start()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e2e_wall0 = time.time()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            layer.forward_host_async(xh, yh)
        layer.host_wait()
        e2e_wall1 = time.time()
        dt = max_over_ranks(time.perf_counter() - t0, dist, "cuda")
        e2e_clk = e2e_clocks.stop(e2e_wall0, e2e_wall1)
        if dist is not None:
            dist.barrier()
        t1 = time.perf_counter()
        for _ in range(n_e2e):
            layer.forward_host(xh, yh)
        dt_sync = max_over_ranks(time.perf_counter() - t1, dist, "cuda")
        e2e = {"value": world * cfg.T * n_e2e / dt, "unit": "tokens/s",
               "h2d_bytes_per_step": cfg.T * cfg.d * 2, "d2h_bytes_per_step": cfg.T * cfg.d * 2,
               "steps": n_e2e, "clocks": e2e_clk,
               "entry": "latentmoe_forward_host_async (copies overlap the neighbouring "
                        "steps' forwards), then latentmoe_host_wait",
               "synchronous": {"value": world * cfg.T * n_e2e / dt_sync, "unit": "tokens/s",
                               "entry": "latentmoe_forward_host (copy in, forward, copy out, "
                                        "wait, per step)"}}

    # CPU baseline: the oracle on a bounded token sample, rank 0 at N=1 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        scales = (layer.fp8_state()["scales"] if args.fp8_dense else
                  layer.fp8_state()["scales"][:2]) if f8 else None
        cpu = cpu_oracle_baseline(cfg, r, x, w, args.cpu_tokens, f8_scales=scales,
                                  fp8_dense=args.fp8_dense)

    peaks, peak_src = load_peaks()
    ms_step = ms_total / args.steps
    value = world * cfg.T * args.steps / (ms_total / 1e3)
    capped = clk is None or "sw_power_cap" in clk.get("reasons", [])
    lroof = layer_roofline(cfg, touched, ms_step, peaks, peak_src, f8, args.fp8_dense, True)
    lroof_now = layer_roofline(cfg, touched, ms_step, peaks, peak_src, f8, args.fp8_dense,
                               capped)
    eb = 1 if f8 else 2
    g_flops, g_bytes, g_built = gate_up_work(cfg, touched, eb)
    g_ms = stage_ms.get(DOMINANT, float("nan"))
    g_peak = peaks["bf16_tflops_sustained"] * (FP8_OVER_BF16 if f8 else 1.0)
    g_tc = g_flops / (g_peak * 1e12) * 1e3
    g_hbm = g_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3
    if g_hbm >= g_tc:
        roof = {"bound": "hbm", "achieved": g_bytes / (g_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": g_flops / (g_ms / 1e3) / 1e12,
                "peak": g_peak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    traffic = profiled_traffic(cfg.name, f8)
    roof["traffic"] = traffic
    peak_kind = ("sustained bf16 x 2 for E4M3" if f8 else "sustained bf16") \
        if roof["bound"] == "tensor" else "HBM copy"
    roof.update({"kernel": DOMINANT + ("_e4m3" if f8 else ""), "ms_per_launch": g_ms,
                 "algorithmic_bytes": g_bytes,
                 "algorithmic": "gate and up weights of the experts that got tokens",
                 "as_built_bytes": g_built,
                 "as_built_gbs": g_built / (g_ms / 1e3) / 1e9,
                 "flops": g_flops,
                 "tensor_tflops": g_flops / (g_ms / 1e3) / 1e12,
                 "peak_source": f"{peak_src} ({peak_kind})"})

    line = {
        "metric": METRIC_FP8_DENSE if args.fp8_dense else (METRIC_FP8 if f8 else METRIC),
        "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 GEMMs, fp32 router" if args.fp8_dense else
                  "e4m3 experts, bf16 elsewhere") if f8 else "bf16",
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) bf16 weights)",
        "config": workload_config(cfg),
        "variant": {"expert_gemm": "single-SM" if args.no_sm_pairs else
                    "SM pairs where shapes allow",
                    "launch": "stream order" if args.no_pdl else
                    "programmatic dependent launch",
                    "expert_launches": "two (gate+up, down)" if args.no_fusion or
                    args.no_sm_pairs or args.capacity > 0 else
                    ("one fused launch where shapes allow" if args.fusion else
                     "automatic: one fused launch for small layers, else two"),
                    **({"capacity": args.capacity, "group_size": args.group_size,
                        "rounds": rounds_info} if args.capacity > 0 else {})},
        "tflops": cfg.T * layer_flops_per_token(cfg) / (ms_step / 1e3) / 1e12,
        "tc_roofline_frac": lroof["tc_ms"] / ms_step,
        "layer_roofline": {**lroof, "frac_at_this_runs_clock_peak": lroof_now["frac"]},
        "roofline": roof,
        "stage_ms": stage_ms,
        "gpu_launches": int(launches),
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clk,
        "device_status": status,
    }
    if f8:
        names = ("z", "h", "x", "c", "shared_hidden") if args.fp8_dense else ("z", "h")
        line["fp8_scales"] = {**dict(zip(names, fp8_state["scales"])),
                              "history_steps": fp8_state["steps"]}

    # the other workloads, at N = 1 only (a scaling run times the headline alone)
    if world == 1 and not args.no_extra_configs and not f8 and cfg.name == "mai-base-1" \
            and args.capacity == 0 and not args.no_sm_pairs:
        layer.close()
        del layer, w, x, y, r
        torch.cuda.empty_cache()
        extra = {}
        for name, n_cpu in EXTRA_CONFIGS:
            extra[name] = measure_small(synth.CONFIGS[name], args, peaks, peak_src, local, n_cpu)
        line["configs"] = extra
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="mai-base-1")
    ap.add_argument("--cpu-tokens", type=int, default=None,
                    help="oracle sample for cpu_baseline (default 48 tokens; 2 with --fp8, "
                         "whose oracle quantizes each touched expert's weights)")
    ap.add_argument("--ref-tokens", type=int, default=1)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="time the headline workload only (by default an N=1 bf16 run at the "
                         "MAI-Base-1 shape also times tiny, mid, imbalanced and MAI-Base-2)")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 E4M3 expert GEMMs with delayed scaling")
    ap.add_argument("--fp8-dense", action="store_true",
                    help="with --fp8: the latent projections and the shared expert in E4M3 too")
    ap.add_argument("--no-pdl", action="store_true",
                    help="the forward's kernels in plain stream order (comparison runs)")
    ap.add_argument("--no-fusion", action="store_true",
                    help="run the two expert GEMMs as two launches")
    ap.add_argument("--fusion", action="store_true",
                    help="run the two expert GEMMs as one fused launch where the shapes allow "
                         "(default: automatic, fused for small layers only)")
    ap.add_argument("--no-sm-pairs", action="store_true",
                    help="expert GEMMs on single SMs instead of SM pairs (comparison runs)")
    ap.add_argument("--capacity", type=int, default=0,
                    help="multi-round fixed-capacity schedule: slots per expert per round "
                         "(0: one dropless pass)")
    ap.add_argument("--group-size", type=int, default=8,
                    help="experts per borrowing group for --capacity")
    ap.add_argument("--max-rounds", type=int, default=0,
                    help="rounds launched per forward for --capacity (0: worst case)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.cpu_tokens is None:
        args.cpu_tokens = 2 if (args.fp8 or args.fp8_dense) else 48

    from mixture_experts_layer_router_gb300 import synth
    cfg = synth.CONFIGS[args.config]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        if args.impl == "ours":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
            tdist.init_process_group("nccl")
        else:
            tdist.init_process_group("gloo")
        dist = tdist
    if args.impl == "reference":
        line = run_reference(args, cfg, rank, world)
    else:
        line = run_ours(args, cfg, rank, world, dist)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
