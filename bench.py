"""Benchmark of the masked, block-scaled NVFP4 grouped GEMM-NT on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config c4] [--impl ours|reference]

One step = one call of nvfp4_grouped_gemm_nt_masked over one batch of the
synthetic workload (default: the largest single-GPU workload, the prefill
GEMM2 of a 256-expert MoE layer: G=256, masked_m from top-8 routing of 4096
tokens, M_max=256, N=7168, K=2048, 962 GFLOP and 2.6 GB per call).  The same
run also times the other four workloads (decode GEMM1 at 32 and 256 experts,
the compute-bound G=8 M=2048 shape and the small masked case) and the fused
MoE GEMM1 epilogue (SwiGLU + NVFP4 output, the same shape taken as GEMM1)
and reports them under "per_config", with sampled parity against the oracle.  Each timed step is bracketed by
CUDA events on the launching stream; between steps L2 is flushed by writing a
256 MB buffer and then reading it back, so the next step starts with an L2
that holds none of its inputs and no dirty lines.  Prints one JSON line (rank 0).  Under torchrun every rank runs an
independent replica (the GEMM has no exchange step): value = all ranks' work /
the slowest rank's time.

--impl reference times the CPU oracle (the plain C fp64 reference) on the
host cores instead, each step a bounded random sample of the same workload's
outputs.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_block_scaled_masked_gb300 import workloads as W  # noqa: E402

METRIC = "grouped NVFP4 GEMM TFLOP/s and weight GB/s, % of roofline, vs oracle"
UNIT = "TFLOP/s"
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25    # dense nominal ratio (fp4 13.5 PF, bf16 2.25 PF)
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.txt")


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    src="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# Sources each kernel family is compiled from: a change to any of them makes
# that family's recorded traffic stale.
KERNEL_SOURCES = {
    "gemm": ("ptx.cuh", "quant.cuh", "gemm.cuh", "gemm_pair.cuh", "gemm_tok_pair.cuh", "nvfp4gg.cu"),
    "gemv": ("gemv.cuh", "nvfp4gg.cu"),
}


def kernel_source_hash(family: str = "gemm") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_block_scaled_masked_gb300", "csrc")
    for name in KERNEL_SOURCES[family]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config_key: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the workload's kernel family; else None."""
    try:
        text = open(PROFILE_TRAFFIC).read()
    except OSError:
        return None
    src = kernel_source_hash("gemv" if W.lookup(config_key).kind == "gemv_w4a16" else "gemm")
    for line in text.splitlines():
        m = re.match(r"\s*(\w+)\s+source=(\w+)\s+dram_bytes_per_launch=(\d+)", line)
        if m and m.group(1) == config_key and m.group(2) == src:
            return int(m.group(3))
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons every 100 ms in a thread."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.dev = device_index
        self.t_on = None
        self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._reader, daemon=True).start()

    def _reader(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        rows = []
        for t, line in self.samples:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        inside = [r for r in rows if self.t_on and self.t_on - 0.05 <= r[0] <= (self.t_off or 1e30) + 0.05]
        note = "samples inside the timed region"
        if not inside:
            inside = rows[-3:]
            note = "timed region shorter than the sampling period: nearest samples"
        mhz = [float(p[1]) for _, p in inside if p[1].replace(".", "").isdigit()]
        mx = [float(p[2]) for _, p in inside if p[2].replace(".", "").isdigit()]
        power = [float(p[3]) for _, p in inside if re.match(r"^[\d.]+$", p[3])]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in inside:
            for name, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(inside), "note": note}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args, cfg, ws, rank):
    """The oracle (plain C, fp64, all host cores) on bounded random samples of
    the workload's valid outputs: one sample per step."""
    if rank != 0:
        return
    from oracle import oracle
    d = W.generate(cfg)
    counts = W.algorithmic_counts(cfg, d["masked_m"])
    mm = d["masked_m"]
    valid_g = np.flatnonzero(mm > 0)
    rng = np.random.default_rng(1)
    cores = oracle.max_threads()

    def sample(n):
        g = rng.choice(valid_g, n)
        m = (rng.random(n) * mm[g]).astype(np.int64)
        nn = rng.integers(0, cfg.N, n)
        return np.stack([g, m, nn], 1)

    # calibrate: outputs per second, then size each step so that the whole
    # run stays within ~60 s of CPU time
    t = time.perf_counter()
    oracle.gemm_sampled(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], sample(4096),
                        cfg.G, cfg.M_max, cfg.N, cfg.K)
    rate = 4096 / max(time.perf_counter() - t, 1e-6)
    per_step = int(max(256, min(rate * 60.0 / max(1, args.steps + args.warmup), rate * 2)))
    for _ in range(args.warmup):
        oracle.gemm_sampled(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], sample(per_step),
                            cfg.G, cfg.M_max, cfg.N, cfg.K)
    times = []
    for _ in range(args.steps):
        idx = sample(per_step)
        t = time.perf_counter()
        oracle.gemm_sampled(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], idx,
                            cfg.G, cfg.M_max, cfg.N, cfg.K)
        times.append(time.perf_counter() - t)
    tot = sum(times)
    flops = 2.0 * per_step * cfg.K * args.steps
    value = flops / tot / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_block(cfg, counts),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} random valid outputs (g,m,n) per step, "
                                   f"K={cfg.K} fp64 terms each"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(cfg, counts):
    return {"workload": cfg.name, "G": cfg.G, "M_max": cfg.M_max, "N": cfg.N, "K": cfg.K,
            "masked_rows": counts["rows"], "nonempty_experts": counts["nonempty"],
            "seed": hex(cfg.seed), "parallelism": "replicas",
            "l2": "flushed between steps: 256 MB written, then read back (clean L2)"}


def replica_seconds(local_seconds: float, world_size: int) -> float:
    """Max over ranks of the device time of the timed steps (the slowest
    replica sets the job's time); identity on one rank."""
    if world_size <= 1:
        return local_seconds
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def torch_int64():
    import torch
    return torch.int64


def flush_l2(buf, i):
    """Evict L2: write a buffer larger than L2, then read it back so the
    evicted lines are clean when the timed step starts."""
    buf.fill_(i & 0xFF)
    return buf.view(torch_int64()).sum()


def time_steps(run_step, steps, flush, stream):
    """Device time of `steps` calls, each after an L2 flush, CUDA events on
    the launching stream; returns the per-step milliseconds."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        flush_l2(flush, i)
        starts[i].record(stream)
        run_step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


PER_CONFIG_KEYS = ("c1", "c2", "c3", "c4", "c5")


def roofline_fracs(cfg, counts, ms, peaks, probe_best):
    """Achieved rates of one call and its fractions of the HBM and NVFP4
    tensor roofs (measured HBM copy bandwidth; the higher MMA-probe rate)."""
    tflops = counts["flops"] / (ms / 1e3) / 1e12
    gbs = counts["bytes"] / (ms / 1e3) / 1e9
    return dict(tflops=tflops, gbs=gbs, frac_hbm=gbs / peaks["hbm"],
                frac_tensor=(tflops / probe_best) if probe_best else None,
                bound="tensor" if cfg.key == "c5" else ("launch" if cfg.key == "c1" else "hbm"))


def per_config_block(args, peaks, probe_best, main_key, main_ms, main_d, main_C, flush, stream):
    """Device-timed ms and roofline fractions of every workload in one run;
    the data and C of each are kept for the sampled parity check of the
    CPU-baseline leg."""
    import torch
    from nvfp4_block_scaled_masked_gb300 import binding
    from nvfp4_block_scaled_masked_gb300.device import Problem
    out, kept = {}, {}
    for key in PER_CONFIG_KEYS:
        cfg = W.CONFIGS[key]
        if key == main_key:
            d, C_bits, ms_list = main_d, main_C, None
            ms = main_ms
        else:
            d = W.generate(cfg)
            prob = Problem(d)
            for _ in range(3):
                prob.run()
            prob.reset_C()
            prob.run()                       # the output kept for the parity check
            C_bits = prob.C_bits()
            if binding.nvfp4_gg_check_error() != 0:
                raise RuntimeError(f"device error on {key}")
            ms_list = time_steps(prob.run, args.per_config_steps, flush, stream)
            if binding.nvfp4_gg_check_error() != 0:
                raise RuntimeError(f"device error on {key}")
            ms = statistics.median(ms_list)
            del prob
            torch.cuda.empty_cache()
        counts = W.algorithmic_counts(cfg, d["masked_m"])
        r = roofline_fracs(cfg, counts, ms, peaks, probe_best)
        out[key] = {"workload": cfg.name, "ms": ms, "TFLOP/s": r["tflops"],
                    "algorithmic_GB/s": r["gbs"], "bound": r["bound"],
                    "frac_of_hbm": r["frac_hbm"], "frac_of_nvfp4_probe": r["frac_tensor"],
                    "traffic": profiled_traffic(key), "algorithmic_bytes": counts["bytes"],
                    "flops": counts["flops"],
                    "steps": args.steps if ms_list is None else len(ms_list),
                    "timing": "median of steps, CUDA events, L2 flushed before each"}
        kept[key] = (d, C_bits)
    return out, kept


SWIGLU_QUANT_KEY = "c4_swiglu_quant"
SWIGLU_QUANT_QSCALE = 2.0 ** -9


def swiglu_quant_entry(args, peaks, probe_best, d, flush, stream):
    """GEMM1 + SwiGLU + NVFP4 output (nvfp4_grouped_gemm_nt_masked_swiglu_quant)
    on the prefill workload's shape taken as GEMM1 (N = 2I gate and up rows):
    device time and HBM fraction over its algorithmic bytes (weights and
    activations once, the bf16 SwiGLU output, the e2m1 codes and e4m3
    scales).  The outputs are kept for the sampled parity check."""
    import torch
    from nvfp4_block_scaled_masked_gb300 import binding
    from nvfp4_block_scaled_masked_gb300.device import Problem
    cfg = d["cfg"]
    prob = Problem(d, keep_raw_weights=True)
    binding.nvfp4_prepare_weights_swiglu(prob.raw_B, prob.raw_Bsf, cfg.G, cfg.N, cfg.K,
                                         prob.B_prep, prob.B_sf_prep)
    prob.raw_B = prob.raw_Bsf = prob.C = None
    I = cfg.N // 2
    C_half = torch.full((cfg.G, cfg.M_max, I), W.SENTINEL_BF16, dtype=torch.int16, device="cuda")
    A2 = torch.zeros((cfg.G, cfg.M_max, I // 2), dtype=torch.uint8, device="cuda")
    A2_sf = torch.zeros((cfg.G, cfg.M_max, I // 16), dtype=torch.uint8, device="cuda")
    qscale = torch.full((cfg.G,), SWIGLU_QUANT_QSCALE, dtype=torch.float32, device="cuda")

    def step():
        binding.nvfp4_grouped_gemm_nt_masked_swiglu_quant(
            prob.A, prob.A_sf, prob.B_prep, prob.B_sf_prep, prob.alpha, prob.masked_m, C_half,
            qscale, A2, A2_sf, cfg.G, cfg.M_max, cfg.N, cfg.K)

    for _ in range(3):
        step()
    if binding.nvfp4_gg_check_error() != 0:
        raise RuntimeError("device error on the SwiGLU + NVFP4 entry")
    ms_list = time_steps(step, args.per_config_steps, flush, stream)
    if binding.nvfp4_gg_check_error() != 0:
        raise RuntimeError("device error on the SwiGLU + NVFP4 entry")
    ms = statistics.median(ms_list)
    counts = W.algorithmic_counts(cfg, d["masked_m"])
    counts["bytes"] -= counts["out_bytes"] // 2            # N/2 bf16 columns per valid row
    counts["bytes"] += counts["rows"] * (cfg.N // 4 + cfg.N // 32)   # codes and scales
    r = roofline_fracs(cfg, counts, ms, peaks, probe_best)
    entry = {"workload": f"GEMM1 + SwiGLU + NVFP4 output on the shape of {cfg.name} "
                         f"(N = {cfg.N} gate and up rows, {I} outputs per row)",
             "entry_point": "nvfp4_grouped_gemm_nt_masked_swiglu_quant",
             "ms": ms, "TFLOP/s": r["tflops"], "algorithmic_GB/s": r["gbs"], "bound": "hbm",
             "frac_of_hbm": r["frac_hbm"], "frac_of_nvfp4_probe": r["frac_tensor"],
             "traffic": None, "algorithmic_bytes": counts["bytes"], "flops": counts["flops"],
             "steps": len(ms_list),
             "timing": "median of steps, CUDA events, L2 flushed before each"}
    kept = (d, C_half.cpu().numpy().view(np.uint16), A2.cpu().numpy(), A2_sf.cpu().numpy(),
            SWIGLU_QUANT_QSCALE)
    del prob, C_half, A2, A2_sf, qscale
    torch.cuda.empty_cache()
    return entry, kept


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="c4", choices=sorted(W.CONFIGS) + sorted(W.EXTRA))
    ap.add_argument("--per-config-steps", type=int, default=100,
                    help="timed steps per workload in the per_config block (0: no per_config)")
    ap.add_argument("--splitk", type=int, default=-1,
                    help="time nvfp4_grouped_gemm_nt_masked_splitk with this split (0 = automatic)")
    ap.add_argument("--swiglu", action="store_true",
                    help="time the fused GEMM1 + SwiGLU entry point (output N/2 columns)")
    ap.add_argument("--swiglu-quant", action="store_true",
                    help="time the fused GEMM1 + SwiGLU entry point that also writes GEMM2's "
                         "NVFP4 activations (codes + scales of the N/2 columns)")
    ap.add_argument("--pair-mode", default="auto", choices=["auto", "on", "off", "token"],
                    help="prefill kernel family: CTA pairs (on), single CTAs (off), token-major "
                         "CTA pairs (token), or the library's automatic choice")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    cfg = W.lookup(args.config)
    ws, rank, local = dist_setup()

    if args.impl == "reference":
        if cfg.kind != "gemm":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable":
                                  "the reference arm times the grouped GEMM workloads only"}))
            return
        run_reference(args, cfg, ws, rank)
        return
    if cfg.kind == "gemv_w4a16":
        bench_gemv(args, cfg, ws, rank, local)
        return

    import torch
    from nvfp4_block_scaled_masked_gb300 import binding, build
    from nvfp4_block_scaled_masked_gb300.device import Problem

    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    build.build()
    binding.load()
    peaks = load_peaks()

    d = W.generate(cfg)
    counts = W.algorithmic_counts(cfg, d["masked_m"])
    if args.swiglu_quant:
        args.swiglu = True
    if args.swiglu:   # the fused epilogue writes N/2 bf16 columns per valid row
        counts["bytes"] -= counts["out_bytes"] // 2
        counts["out_bytes"] //= 2
    if args.swiglu_quant:   # + N/2 e2m1 codes and N/32 e4m3 scales per valid row
        q_bytes = counts["rows"] * (cfg.N // 4 + cfg.N // 32)
        counts["bytes"] += q_bytes
        counts["out_bytes"] += q_bytes
    stream = torch.cuda.current_stream()

    # one-time weight re-layout, timed separately (median of 5)
    binding.nvfp4_gg_set_pair_mode({"off": 0, "on": 1, "auto": 2, "token": 3}[args.pair_mode])
    prob = Problem(d, keep_raw_weights=True)
    prep_ms = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        prepare = (binding.nvfp4_prepare_weights_swiglu if args.swiglu
                   else binding.nvfp4_prepare_weights)
        prepare(prob.raw_B, prob.raw_Bsf, cfg.G, cfg.N, cfg.K, prob.B_prep, prob.B_sf_prep)
        e1.record()
        e1.synchronize()
        prep_ms.append(e0.elapsed_time(e1))
    prob.raw_B = prob.raw_Bsf = None
    torch.cuda.empty_cache()   # the device then holds only what the timed call uses

    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    if args.splitk >= 0:
        splitk_bytes = binding.nvfp4_splitk_workspace_bytes(cfg.G, cfg.M_max, cfg.N, cfg.K,
                                                            args.splitk)
        splitk_ws = torch.empty(splitk_bytes, dtype=torch.uint8, device="cuda")

        def run_step():
            binding.nvfp4_grouped_gemm_nt_masked_splitk(
                prob.A, prob.A_sf, prob.B_prep, prob.B_sf_prep, prob.alpha, prob.masked_m, prob.C,
                cfg.G, cfg.M_max, cfg.N, cfg.K, args.splitk, splitk_ws, splitk_bytes)
    elif args.swiglu_quant:
        C_half = torch.empty((cfg.G, cfg.M_max, cfg.N // 2), dtype=torch.int16, device="cuda")
        A2 = torch.empty((cfg.G, cfg.M_max, cfg.N // 4), dtype=torch.uint8, device="cuda")
        A2_sf = torch.empty((cfg.G, cfg.M_max, cfg.N // 32), dtype=torch.uint8, device="cuda")
        qscale = torch.full((cfg.G,), 2.0 ** -9, dtype=torch.float32, device="cuda")

        def run_step():
            binding.nvfp4_grouped_gemm_nt_masked_swiglu_quant(
                prob.A, prob.A_sf, prob.B_prep, prob.B_sf_prep, prob.alpha, prob.masked_m, C_half,
                qscale, A2, A2_sf, cfg.G, cfg.M_max, cfg.N, cfg.K)
    elif args.swiglu:
        C_half = torch.empty((cfg.G, cfg.M_max, cfg.N // 2), dtype=torch.int16, device="cuda")

        def run_step():
            binding.nvfp4_grouped_gemm_nt_masked_swiglu(
                prob.A, prob.A_sf, prob.B_prep, prob.B_sf_prep, prob.alpha, prob.masked_m, C_half,
                cfg.G, cfg.M_max, cfg.N, cfg.K)
    else:
        run_step = prob.run
    for i in range(args.warmup):
        run_step()
    if binding.nvfp4_gg_check_error() != 0:
        raise RuntimeError("device error during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark_on()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush_l2(flush, i)
        starts[i].record(stream)
        run_step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    wall = time.perf_counter() - t_wall
    sampler.mark_off()
    sampler.stop()
    rc = binding.nvfp4_gg_check_error()
    if rc != 0:
        raise RuntimeError(f"device error in the timed region: {binding.status_string(rc)}")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    dev_s = replica_seconds(sum(step_ms) / 1e3, ws)
    ms = 1e3 * dev_s / args.steps
    tflops = counts["flops"] * ws / (ms / 1e3) / 1e12
    gbs = counts["bytes"] / (ms / 1e3) / 1e9
    wgbs = counts["weight_bytes"] / (ms / 1e3) / 1e9

    # end to end through the host-buffer entry point: pinned inputs copied in,
    # valid rows of C copied out, every step
    h = {k: torch.from_numpy(np.ascontiguousarray(d[k])).pin_memory()
         for k in ("A", "A_sf", "alpha", "masked_m")}
    h["masked_m"] = torch.from_numpy(d["masked_m"].astype(np.int32)).pin_memory()
    hC = torch.empty((cfg.G, cfg.M_max, cfg.N), dtype=torch.int16).pin_memory()
    staging_bytes = binding.nvfp4_host_staging_bytes(cfg.G, cfg.M_max, cfg.N, cfg.K)
    staging = torch.empty(staging_bytes, dtype=torch.uint8, device="cuda")

    def e2e_step():
        binding.nvfp4_grouped_gemm_nt_masked_host(
            h["A"], h["A_sf"], h["alpha"], h["masked_m"], prob.B_prep, prob.B_sf_prep, hC,
            cfg.G, cfg.M_max, cfg.N, cfg.K, staging, staging_bytes)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(args.e2e_steps):
        flush_l2(flush, i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step()
        stream.synchronize()         # the host reads the result
        e2e_ms.append(1e3 * (time.perf_counter() - t0))
    if binding.nvfp4_gg_check_error() != 0:
        raise RuntimeError("device error in the end-to-end leg")
    e2e_med = statistics.median(e2e_ms)
    h2d = sum(h[k].numel() * h[k].element_size() for k in h)
    d2h = int(d["masked_m"].sum()) * cfg.N * 2

    line = {
        "metric": METRIC, "value": tflops, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e2m1, e4m3 block-16 scales, f32 accumulate, bf16 out)",
        "data": "synthetic", "config": config_block(cfg, counts),
        "algorithmic_gbs": gbs, "weight_gbs": wgbs,
        "prepare_weights_ms": statistics.median(prep_ms),
        "gpu_launches": args.steps,
        "entry_point": ("nvfp4_grouped_gemm_nt_masked_splitk(split_k=%d)" % args.splitk
                        if args.splitk >= 0 else "nvfp4_grouped_gemm_nt_masked_swiglu_quant"
                        if args.swiglu_quant else "nvfp4_grouped_gemm_nt_masked_swiglu"
                        if args.swiglu else "nvfp4_grouped_gemm_nt_masked"),
        "pair_mode": args.pair_mode,
        "wall_s_timed_region": wall,
        "step_ms_min": min(step_ms), "step_ms_median": statistics.median(step_ms),
    }
    # dense NVFP4 tensor rate, measured by the library's probes (single-CTA
    # M = 128 MMAs at N = 256 and 192, CTA-pair M = 256 MMAs at N = 256)
    probe = {"cta1_N256": mma_peak_tflops(256), "cta1_N192": mma_peak_tflops(192),
             "pair_N256": mma_peak_tflops(256, pair=True)}
    probe_best = max(probe.values())
    line["mma_probe_tflops"] = probe
    if cfg.key == "c5":
        peak = peaks["bf16"] * NOMINAL_FP4_OVER_BF16
        line["roofline"] = {"bound": "tensor", "achieved": tflops / ws, "peak": peak,
                            "unit": "TFLOP/s", "frac": tflops / ws / peak,
                            "traffic": profiled_traffic(cfg.key),
                            "peak_note": f"nvfp4 = bf16 {peaks['src']} burst x {NOMINAL_FP4_OVER_BF16:g} (nominal ratio)",
                            "frac_of_probe": tflops / ws / probe_best,
                            "probe_note": "the higher of the library's MMA-probe rates (mma_probe_tflops)"}
    else:
        line["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                            "frac": gbs / peaks["hbm"], "traffic": profiled_traffic(cfg.key),
                            "algorithmic_bytes": counts["bytes"],
                            "peak_note": f"HBM copy bandwidth, {peaks['src']}"}
    if args.splitk >= 0 or args.swiglu:
        # the recorded DRAM traffic is the plain GEMM kernel's, not this entry point's
        line["roofline"]["traffic"] = None
    kept, kept_sq = {}, None
    if args.per_config_steps > 0 and ws == 1:
        plain = args.splitk < 0 and not args.swiglu
        main_key = cfg.key if (plain and cfg.key in PER_CONFIG_KEYS) else None
        line["per_config"], kept = per_config_block(
            args, peaks, probe_best, main_key, ms, d, prob.C_bits() if main_key else None,
            flush, stream)
        if plain:
            d_sq = d if cfg.key == "c4" else W.generate(W.CONFIGS["c4"])
            line["per_config"][SWIGLU_QUANT_KEY], kept_sq = swiglu_quant_entry(
                args, peaks, probe_best, d_sq, flush, stream)
    line["e2e"] = {"value": counts["flops"] / (e2e_med / 1e3) / 1e12, "unit": UNIT,
                   "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                   "ms_per_step": e2e_med, "steps": args.e2e_steps,
                   "how": ("(plain GEMM: the host-buffer entry point has no SwiGLU variant) "
                           if args.swiglu else "") +
                          "nvfp4_grouped_gemm_nt_masked_host on pinned host buffers: A and A_sf "
                          "copied to the device (prefill-sized calls in up to four expert chunks "
                          "on a side stream, each chunk's GEMM after its own copy), alpha and "
                          "masked_m read and the valid rows of C written by the kernel in host "
                          "memory, stream sync; wall clock per step (Python call included)"}
    line["clocks"] = sampler.summary()

    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, d, prob)
        for key, (dk, Ck) in kept.items():
            line["per_config"][key]["parity"] = sampled_parity(dk, Ck)
        if kept_sq is not None:
            line["per_config"][SWIGLU_QUANT_KEY]["parity"] = sampled_parity_swiglu(*kept_sq)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def bench_gemv(args, cfg, ws, rank, local):
    """The W4A16 decode GEMV (nvfp4_gemv_w4a16): same timing rules and JSON
    line as the GEMM; HBM roofline over its algorithmic bytes (weights and
    scales once, the bf16 tokens and outputs)."""
    import torch
    from nvfp4_block_scaled_masked_gb300 import binding, build
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    build.build()
    binding.load()
    peaks = load_peaks()
    d = W.generate_gemv(cfg)
    M, N, K = cfg.M_max, cfg.N, cfg.K
    flops = 2.0 * M * N * K
    nbytes = N * (K // 2 + K // 16) + M * K * 2 + M * N * 2
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    x, B, Bsf, al = dev(d["x"].view(np.int16)), dev(d["B"]), dev(d["B_sf"]), dev(d["alpha"])
    y = torch.empty((M, N), dtype=torch.int16, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        binding.nvfp4_gemv_w4a16(x, B, Bsf, al, y, M, N, K)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        step()
    if binding.nvfp4_gg_check_error() != 0:
        raise RuntimeError("device error during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.mark_on()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2(flush, i)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    wall = time.perf_counter() - t0
    sampler.mark_off()
    sampler.stop()
    if binding.nvfp4_gg_check_error() != 0:
        raise RuntimeError("device error in the timed region")
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = 1e3 * replica_seconds(sum(step_ms) / 1e3, ws) / args.steps
    gbs = nbytes / (ms / 1e3) / 1e9
    # end to end: pinned tokens in, GEMV, outputs back, every step
    hx = torch.from_numpy(d["x"].view(np.int16).copy()).pin_memory()
    hy = torch.empty((M, N), dtype=torch.int16).pin_memory()

    def e2e_step():
        x.copy_(hx, non_blocking=True)
        step()
        hy.copy_(y, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(args.e2e_steps):
        flush_l2(flush, i)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        e2e_step()
        stream.synchronize()
        e2e_ms.append(1e3 * (time.perf_counter() - t1))
    e2e_med = statistics.median(e2e_ms)
    line = {
        "metric": METRIC, "value": flops * ws / (ms / 1e3) / 1e12, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "nvfp4 weights (e2m1, e4m3 block-16 scales) x bf16 activations, f32 accumulate, bf16 out",
        "data": "synthetic",
        "config": {"workload": cfg.name, "M": M, "N": N, "K": K, "seed": hex(cfg.seed),
                   "parallelism": "replicas",
                   "l2": "flushed between steps: 256 MB written, then read back (clean L2)"},
        "algorithmic_gbs": gbs, "gpu_launches": args.steps, "entry_point": "nvfp4_gemv_w4a16",
        "wall_s_timed_region": wall,
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm"], "traffic": profiled_traffic(cfg.key),
                     "algorithmic_bytes": nbytes, "peak_note": f"HBM copy bandwidth, {peaks['src']}"},
        "e2e": {"value": flops / (e2e_med / 1e3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": M * K * 2, "d2h_bytes_per_step": M * N * 2,
                "ms_per_step": e2e_med, "steps": args.e2e_steps,
                "how": "pinned tokens copied in, nvfp4_gemv_w4a16, outputs copied back, stream "
                       "sync; wall clock per step (Python call included)"},
        "clocks": sampler.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        from oracle import oracle
        t1 = time.perf_counter()
        _, ref = oracle.gemv_w4a16(d["x"], d["B"], d["B_sf"], d["alpha"][0], K)
        el = time.perf_counter() - t1
        vals = (y.cpu().numpy().view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        ok = oracle.tolerance_ok(vals, ref, np.abs(ref).max())
        line["cpu_baseline"] = {"value": flops / el / 1e12, "unit": UNIT, "cores": os.cpu_count(),
                                "kind": "oracle", "sample": f"the whole GEMV (M={M}, N={N}, K={K}), fp64",
                                "seconds": el,
                                "parity": {"outputs": int(ok.size), "within_tolerance": int(ok.sum())}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def mma_peak_tflops(n: int, iters: int = 1 << 16, pair: bool = False) -> float:
    """Dense NVFP4 tensor rate from the library's MMA probes: all SMs issue
    back-to-back block-scaled MMAs of K=64, M=128 per CTA (pair=False) or
    M=256 per 2-CTA cluster (pair=True), N=n; median of 5 launches."""
    import torch
    from nvfp4_block_scaled_masked_gb300 import binding
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    probe = binding.nvfp4_gg_mma_peak_probe_pair if pair else binding.nvfp4_gg_mma_peak_probe
    probe(iters // 16, n)
    times = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        probe(iters, n)
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    if binding.nvfp4_gg_check_error() != 0:
        raise RuntimeError("device error in the MMA probe")
    flops = (sms // 2 if pair else sms) * iters * 4 * 2.0 * (256 if pair else 128) * n * 64
    return flops / statistics.median(times) / 1e12


def sampled_parity(d, C_bits, outputs: int = 20000, seed: int = 3):
    """Part of the CPU-baseline leg: random valid outputs of one call against
    the oracle (fp64, sampled), and every row m >= masked_m[g] compared with
    the 0x7FC0 prefill."""
    from oracle import oracle
    cfg = d["cfg"]
    mm = d["masked_m"]
    untouched = all(bool(np.all(C_bits[g, mm[g]:] == W.SENTINEL_BF16)) for g in range(cfg.G))
    rng = np.random.default_rng(seed)
    valid_g = np.flatnonzero(mm > 0)
    g = rng.choice(valid_g, outputs)
    m = (rng.random(outputs) * mm[g]).astype(np.int64)
    n = rng.integers(0, cfg.N, outputs)
    idx = np.stack([g, m, n], 1).astype(np.int64)
    ref = oracle.gemm_sampled(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], idx,
                              cfg.G, cfg.M_max, cfg.N, cfg.K)
    vals = (C_bits[g, m, n].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok = oracle.tolerance_ok(vals, ref, np.abs(ref).max())
    return {"outputs": int(ok.size), "within_tolerance": int(ok.sum()),
            "masked_rows_untouched": untouched,
            "sample": f"{outputs} random valid (g, m, n), fp64 oracle; max|ref| over the sample"}


def sampled_parity_swiglu(d, C_bits, A2, A2_sf, q, outputs: int = 20000, rows: int = 64,
                          seed: int = 5):
    """Part of the CPU-baseline leg, for the SwiGLU + NVFP4 entry: random valid
    SwiGLU outputs against silu(gate) * up from the oracle's sampled fp64 GEMM
    (gate column j, up column I + j), the GEMM tolerance; rows m >= masked_m
    compared with the prefill; and random valid rows' NVFP4 codes and scales
    against the oracle's encoder applied to the GPU's own bf16 row, bit for
    bit."""
    from oracle import oracle
    cfg = d["cfg"]
    mm = d["masked_m"]
    I = cfg.N // 2
    untouched = all(bool(np.all(C_bits[g, mm[g]:] == W.SENTINEL_BF16)) for g in range(cfg.G))
    rng = np.random.default_rng(seed)
    valid_g = np.flatnonzero(mm > 0)
    g = rng.choice(valid_g, outputs)
    m = (rng.random(outputs) * mm[g]).astype(np.int64)
    j = rng.integers(0, I, outputs)
    args = (d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"])
    gate = oracle.gemm_sampled(*args, np.stack([g, m, j], 1).astype(np.int64),
                               cfg.G, cfg.M_max, cfg.N, cfg.K)
    up = oracle.gemm_sampled(*args, np.stack([g, m, I + j], 1).astype(np.int64),
                             cfg.G, cfg.M_max, cfg.N, cfg.K)
    ref = oracle.silu(gate) * up
    vals = (C_bits[g, m, j].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ok = oracle.tolerance_ok(vals, ref, np.abs(ref).max())
    gr = rng.choice(valid_g, rows)
    mr = (rng.random(rows) * mm[gr]).astype(np.int64)
    want_c, want_sf = oracle.quantize_nvfp4(C_bits[gr, mr], np.full(rows, q, np.float32))
    same = np.all(A2[gr, mr] == want_c, axis=1) & np.all(A2_sf[gr, mr] == want_sf, axis=1)
    return {"outputs": int(ok.size), "within_tolerance": int(ok.sum()),
            "masked_rows_untouched": untouched,
            "nvfp4_rows": int(rows), "nvfp4_rows_bit_identical": int(same.sum()),
            "sample": f"{outputs} random valid (g, m, j) SwiGLU outputs against the fp64 "
                      f"oracle (max|ref| over the sample); {rows} random valid rows' codes and "
                      "scales against the oracle's encoder on the GPU's bf16 row"}


def cpu_baseline(cfg, d, prob):
    """The oracle as it stands, all host cores, on the full workload when that
    is small (decode configs) or on a bounded set of experts; the GPU output of
    the last timed step is checked against it on the same outputs."""
    from oracle import oracle
    mm = d["masked_m"]
    cores = oracle.max_threads()
    G = cfg.G
    # choose experts until ~2e10 fp64 multiply-adds (10-30 s of CPU work)
    budget = 2e10
    chosen, work = [], 0.0
    for g in np.flatnonzero(mm > 0):
        w = float(mm[g]) * cfg.N * cfg.K + cfg.N * cfg.K
        if chosen and work + w > budget:
            break
        chosen.append(int(g))
        work += w
    sub_mm = np.zeros_like(mm)
    sub_mm[chosen] = mm[chosen]
    t = time.perf_counter()
    Cref, ref = oracle.gemm(d["A"], d["A_sf"], d["B"], d["B_sf"], d["alpha"], sub_mm, d["C_init"],
                            G, cfg.M_max, cfg.N, cfg.K)
    el = time.perf_counter() - t
    rows = int(sub_mm.sum())
    flops = 2.0 * rows * cfg.N * cfg.K
    Cg = prob.C_bits()
    valid = np.zeros((G, cfg.M_max), bool)
    for g in chosen:
        valid[g, :mm[g]] = True
    vals = (Cg[valid].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    r = ref[valid]
    ok = oracle.tolerance_ok(vals, r, np.abs(r).max()) if r.size else np.array([True])
    return {"value": flops / el / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"experts {chosen[0]}..{chosen[-1]} ({len(chosen)} of {int((mm > 0).sum())} "
                       f"non-empty), all {rows} valid rows x N={cfg.N}, K={cfg.K}, fp64"),
            "seconds": el,
            "parity": {"outputs": int(ok.size), "within_tolerance": int(ok.sum())}}


if __name__ == "__main__":
    main()
