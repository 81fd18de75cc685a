"""Benchmark of one verify step (paged KV append + paged GQA verify attention +
fused rejection sampling) on the LLaMA-3-70B layer-shaped workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3_70b] [--sigma 1.5] [--no-configs]

Prints ONE JSON line on rank 0. `value` is verify steps/s of the whole job
(inputs resident in HBM); `e2e` is the same metric through the public API with
every step's inputs copied from pinned host memory and its outputs read back
inside the timed region (two device copies of the inputs: a step's copy, on
its own stream, overlaps the previous step's compute). The reference arm (`--impl reference`) times the CPU
oracle on a bounded sample of the same workload and scales it to steps/s.
`configs` holds one object per other workload of the verify step (the
LLaMA-3-8B layer, the 128K-token context, the fp8 cache with fp32 logits, and
the 70B layer at the other draft-noise levels of its sweep), each timed the
same way with its own attention and sampling rooflines and oracle baseline.
Multi-GPU runs are independent replicas (one batch per GPU, no collective);
--gpus must equal the number of ranks the launcher started.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify steps/sec & tokens/sec; HBM GB/s vs 8 TB/s roofline (1×GB300)"
UNIT = "verify steps/s"
NOMINAL_HBM_GBS = 8000.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_70b")
    ap.add_argument("--sigma", type=float, default=None)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end pass")
    ap.add_argument("--mla-only", action="store_true",
                    help="time only the MLA verify attention (prints its JSON object; for profiling)")
    ap.add_argument("--mla-batch", type=int, default=64, help="sequences of the --mla-only workload")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' objects")
    ap.add_argument("--config-steps", type=int, default=40, help="timed steps per object of `configs`")
    return ap.parse_args()


def check_world(args, world):
    """--gpus N is the number of ranks the launcher started (torchrun for N > 1):
    a disagreement would print a line for a job that did not run."""
    if args.gpus != world:
        raise SystemExit("bench.py: --gpus %d but WORLD_SIZE is %d; for N > 1 launch one rank per GPU with "
                         "python -m torch.distributed.run --nproc-per-node N bench.py --gpus N" % (args.gpus, world))


def pct(xs, q):
    """q-th percentile (0..100) of a list, linear interpolation."""
    ys = sorted(xs)
    if not ys:
        return None
    k = (len(ys) - 1) * q / 100.0
    lo = int(math.floor(k))
    hi = min(lo + 1, len(ys) - 1)
    return ys[lo] + (ys[hi] - ys[lo]) * (k - lo)


def dist_summary(xs_ms):
    """median, p10 and p90 of per-step event times, in microseconds."""
    us = [1e3 * x for x in xs_ms]
    return {"median_us": pct(us, 50), "p10_us": pct(us, 10), "p90_us": pct(us, 90)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(seed, rank):
    """Each rank verifies its own batch of sequences (weak scaling): the
    inputs of rank r are those of seed + r."""
    return seed + rank


def max_over_ranks(x, device, world):
    """The slowest rank's time: the job is done when every rank is."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_steps_per_sec(steps, world, total_ms):
    """Whole-job throughput: every rank ran `steps` steps in total_ms."""
    return world * steps / (total_ms / 1e3)


def workload_config(cfg, sigma, lens, world, step_bytes):
    """The `config` object of the JSON line (the same for both arms)."""
    return {"workload": "%s: B=%d H_q=%d H_kv=%d d_head=%d %s KV, ctx %s, block 16, K=%d, V=%d %s logits, "
                        "draft sigma %.2g" % (cfg.name, cfg.B, cfg.H_q, cfg.H_kv, cfg.d_head, cfg.kv_dtype,
                                             cfg.ctx, cfg.K, cfg.V, cfg.logit_dtype, sigma),
            "global_batch": cfg.B * world, "seq_len": int(sum(lens) / len(lens)),
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "inputs larger than L2 (%.2f GB touched per step)" % (step_bytes / 1e9)}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def attn_traffic_from_profile():
    """DRAM bytes per attention launch from the committed ncu summary, if the
    kernel source is unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "attn_tc5_llama3_70b.md")
    src = os.path.join(ROOT, "speculative_verify_paged_gb300", "csrc", "attn.cu")
    if not (os.path.exists(p) and os.path.exists(src)):
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    text = open(p).read()
    src_line = [l for l in text.splitlines() if l.startswith("source_sha256_16:")]
    val_line = [l for l in text.splitlines() if l.startswith("dram_bytes_per_launch_full_workload:")]
    if not src_line or not val_line or src_line[0].split(":", 1)[1].strip() != digest:
        return None
    return int(float(val_line[0].split(":", 1)[1].strip()))


class ClockSampler:
    """SM clock and clock-event reasons sampled every 2 ms during the timed
    region through NVML (read-only queries), falling back to nvidia-smi at
    its 200 ms period when NVML cannot be loaded."""

    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, period_s=0.002):
        self.index = index
        self.period = period_s
        self.samples = []      # (sm_mhz, reason bits)
        self.max_mhz = None
        self.proc = None
        self.lines = []
        self.thread = None
        self.stop_flag = threading.Event()
        self.nvml = self._open_nvml()

    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            idx = self.index
            if vis and vis.split(",")[0].strip().isdigit():
                idx = int(vis.split(",")[self.index].strip())
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(idx), ctypes.byref(h)) != 0:
                return None
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            return (lib, h, reasons)
        except (OSError, AttributeError):
            return None

    def _poll_nvml(self):
        import ctypes
        lib, h, reasons = self.nvml
        clk = ctypes.c_uint()
        bits = ctypes.c_ulonglong()
        while True:
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = int(bits.value) if reasons(h, ctypes.byref(bits)) == 0 else 0
                self.samples.append((float(clk.value), r))
            if self.stop_flag.wait(self.period):
                break

    def start(self):
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.nvml is not None:
            self.stop_flag.set()
            self.thread.join(timeout=2)
            if not self.samples:
                return None
            reasons = sorted({n for _, r in self.samples for bit, n in self.REASONS.items() if r & bit})
            return {"sm_mhz": statistics.median(s for s, _ in self.samples), "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(self.samples), "source": "nvml, 2 ms"}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi, 200 ms"}


# ------------------------------------------------------------ our arm -----

class StepSetup:
    """Inputs, outputs and workspaces of one verify step (append, attention,
    sampling) of a workload on the device, and the step itself."""

    def __init__(self, sv, cfg, sigma, seed, dev, stream):
        import torch

        import workloads
        self.sv, self.cfg, self.stream = sv, cfg, stream
        a = self.a = workloads.make_attention_inputs(cfg, seed=seed, device=dev)
        self.n = workloads.make_append_inputs(cfg, seed=seed, device=dev)
        self.s = workloads.make_sampling_inputs(cfg, seed=seed, device=dev, sigma=sigma)
        self.lens = a["seq_lens"].tolist()
        self.attn_bytes = workloads.attention_bytes(cfg, self.lens)
        self.samp_bytes = workloads.sampling_bytes(cfg)
        self.app_bytes = workloads.append_bytes(cfg)
        self.step_bytes = self.attn_bytes + self.samp_bytes + self.app_bytes
        self.k_cache, self.v_cache = a["k_cache"], a["v_cache"]
        self.out = torch.empty_like(a["q"])
        self.attn_ws = sv.alloc_workspace(sv.attn_workspace_size(cfg.B, cfg.n_new, cfg.H_q, cfg.H_kv, cfg.d_head,
                                                                 a["block_table"].shape[1]), dev)
        self.samp_ws = sv.alloc_workspace(sv.sample_workspace_size(cfg.B, cfg.K, cfg.V), dev)
        self.toks = torch.empty((cfg.B, cfg.K + 1), dtype=torch.int32, device=dev)
        self.nacc = torch.empty((cfg.B,), dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def step(self, ev=None):
        sv, a, n, s, stream = self.sv, self.a, self.n, self.s, self.stream
        if ev is not None:
            ev[0].record(stream)
        sv.kv_block_append(n["k_new"], n["v_new"], self.k_cache, self.v_cache, a["block_table"], a["seq_lens"],
                           a["k_scale"], a["v_scale"], status=self.status)
        if ev is not None:
            ev[1].record(stream)
        sv.spec_verify_attn(a["q"], self.k_cache, self.v_cache, a["block_table"], a["seq_lens"], None,
                            a["k_scale"], a["v_scale"], out=self.out, workspace=self.attn_ws, status=self.status)
        if ev is not None:
            ev[2].record(stream)
        sv.spec_verify_sample(s["target_logits"], s["draft_logits"], s["draft_tokens"], s["uniforms"],
                              out_tokens=self.toks, num_accepted=self.nacc, workspace=self.samp_ws,
                              status=self.status, want_probs=False)
        if ev is not None:
            ev[3].record(stream)


def other_configs(headline, sigma):
    """The workloads of the verify step other than the headline line's: every
    other configuration, and the 70B layer at the sweep's other noise levels."""
    import workloads
    out = [(name, workloads.CONFIGS[name].sigma) for name in ("llama3_8b", "long", "fp8") if name != headline]
    if headline == "llama3_70b":
        out += [("llama3_70b", sg) for sg in workloads.SIGMA_SWEEP_70B if sg != sigma]
    else:
        out += [("llama3_70b", sg) for sg in workloads.SIGMA_SWEEP_70B]
    return out


def measure_config(sv, cfg, sigma, seed, dev, stream, steps, warmup=5, cpu=True):
    """One object of `configs`: the verify step of this workload timed like the
    headline (per-op CUDA events on the launching stream over `steps` steps,
    each step's working set above twice the L2), with the median, p10 and
    p90 of each op, the attention and sampling rooflines, and the oracle on a
    bounded sample of the same inputs."""
    import torch

    import workloads
    st = StepSetup(sv, cfg, sigma, seed, dev, stream)
    for _ in range(warmup):
        st.step()
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0, "device status %d (%s)" % (int(st.status.item()), cfg.name)
    emitted = int((st.nacc.long() + 1).sum().item())
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        st.step(evs[k])
    t1.record(stream)
    torch.cuda.synchronize()
    assert int(st.status.item()) == 0
    total_ms = t0.elapsed_time(t1)
    app = [e[0].elapsed_time(e[1]) for e in evs]
    att = [e[1].elapsed_time(e[2]) for e in evs]
    smp = [e[2].elapsed_time(e[3]) for e in evs]
    peak, peak_kind = measured_peaks()
    a_us, s_us = 1e3 * pct(att, 50), 1e3 * pct(smp, 50)
    a_gbs, s_gbs = st.attn_bytes / (a_us * 1e-6) / 1e9, st.samp_bytes / (s_us * 1e-6) / 1e9
    res = {"workload": workload_config(cfg, sigma, st.lens, 1, st.step_bytes)["workload"],
           "sigma": sigma, "steps": steps, "stat": "median of per-step CUDA events",
           "steps_per_sec": steps / (total_ms / 1e3), "ms_per_step": total_ms / steps,
           "tokens_per_sec": emitted * steps / (total_ms / 1e3), "emitted_tokens_per_step": emitted,
           "append": dist_summary(app), "attn": dist_summary(att), "sample": dist_summary(smp),
           "step": dist_summary([x + y + z for x, y, z in zip(app, att, smp)]),
           "bytes": {"attn": st.attn_bytes, "sample": st.samp_bytes, "append": st.app_bytes},
           "roofline_attn": {"bound": "hbm", "kernel": "spec_verify_attn", "achieved": a_gbs, "peak": peak,
                             "peak_kind": peak_kind, "unit": "GB/s", "frac": a_gbs / peak,
                             "frac_of_8tbs": a_gbs / NOMINAL_HBM_GBS},
           "roofline_sample": {"bound": "hbm", "kernel": "spec_verify_sample", "achieved": s_gbs, "peak": peak,
                               "peak_kind": peak_kind, "unit": "GB/s", "frac": s_gbs / peak,
                               "frac_of_8tbs": s_gbs / NOMINAL_HBM_GBS},
           "l2": "inputs larger than twice the L2 (%.2f GB touched per step)" % (st.step_bytes / 1e9)}
    if cpu:
        res["cpu_baseline"] = cpu_baseline_bounded(cfg, st.a, st.n, st.s)
    del st
    torch.cuda.empty_cache()
    return res


def cpu_baseline_bounded(cfg, a, n, s, budget_s=6.0):
    """The oracle on the first sequences of the workload, sized from a
    one-sequence probe to about budget_s seconds, scaled to the full step."""
    _, t_one, _ = oracle_sample_time(cfg, a, n, s, 1, 1)
    k = max(1, min(cfg.B, int(budget_s / max(t_one, 1e-3))))
    full, spent, desc = oracle_sample_time(cfg, a, n, s, k, k) if k > 1 else oracle_sample_time(cfg, a, n, s, 1, 1)
    return {"value": 1.0 / full, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": desc + "; %.1f s of CPU work; numpy fp64 (BLAS threads = cores)" % spent}

def run_ours(args, rank, world, local):
    import torch
    import torch.distributed as dist

    import speculative_verify_paged_gb300 as sv
    import workloads

    check_world(args, world)
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sv.build()
    cfg = workloads.CONFIGS[args.workload]
    sigma = cfg.sigma if args.sigma is None else args.sigma
    seed = rank_seed(args.seed, rank)
    stream = torch.cuda.current_stream()
    st = StepSetup(sv, cfg, sigma, seed, dev, stream)
    a, n, s = st.a, st.n, st.s
    lens, attn_bytes, samp_bytes, app_bytes, step_bytes = st.lens, st.attn_bytes, st.samp_bytes, st.app_bytes, \
        st.step_bytes
    k_cache, v_cache, out, attn_ws, samp_ws = st.k_cache, st.v_cache, st.out, st.attn_ws, st.samp_ws
    toks, nacc, status = st.toks, st.nacc, st.status
    step = st.step

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "device status %d" % int(status.item())
    emitted_per_step = int((nacc.long() + 1).sum().item())

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches0 = sv.kernel_launches()
    t0.record(stream)
    for k in range(args.steps):
        step(evs[k])
    t1.record(stream)
    timed_launches = sv.kernel_launches() - launches0
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    app_ms = [e[0].elapsed_time(e[1]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    samp_ms = [e[2].elapsed_time(e[3]) for e in evs]
    total_ms = max_over_ranks(total_ms, dev, world)

    # ---- end to end through the public API with host buffers -------------
    host = {k: v.cpu().pin_memory() for k, v in
            {"q": a["q"], "k_new": n["k_new"], "v_new": n["v_new"], "target_logits": s["target_logits"],
             "draft_logits": s["draft_logits"], "draft_tokens": s["draft_tokens"],
             "uniforms": s["uniforms"], "seq_lens": a["seq_lens"], "block_table": a["block_table"]}.items()}
    # two device copies of the inputs: step i's copy (on its own stream)
    # overlaps step i-1's compute, and waits until step i-2 released the copy
    devbufs = [{k: torch.empty_like(v, device=dev) for k, v in host.items()} for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)   # (a second copy stream gained nothing: the link is the limit)
    copied = [torch.cuda.Event() for _ in range(2)]
    released = [torch.cuda.Event() for _ in range(2)]
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    toks_h = torch.empty(toks.shape, dtype=toks.dtype).pin_memory()
    nacc_h = torch.empty(nacc.shape, dtype=nacc.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(x.numel() * x.element_size() for x in (out_h, toks_h, nacc_h))

    def e2e_step(i):
        devbuf = devbufs[i % 2]
        copy_stream.wait_event(released[i % 2])
        with torch.cuda.stream(copy_stream):
            for k, v in host.items():
                devbuf[k].copy_(v, non_blocking=True)
        copied[i % 2].record(copy_stream)
        stream.wait_event(copied[i % 2])
        o, tk, na = sv.verify_step(devbuf["q"], devbuf["k_new"], devbuf["v_new"], k_cache, v_cache,
                                   devbuf["block_table"], devbuf["seq_lens"], devbuf["target_logits"],
                                   devbuf["draft_logits"], devbuf["draft_tokens"], devbuf["uniforms"],
                                   a["k_scale"], a["v_scale"], attn_out=out, attn_workspace=attn_ws,
                                   sample_workspace=samp_ws, status=status)
        released[i % 2].record(stream)
        out_h.copy_(o, non_blocking=True)
        toks_h.copy_(tk, non_blocking=True)
        nacc_h.copy_(na, non_blocking=True)

    e2e_steps = 0 if args.no_e2e else max(5, args.steps // 2)
    for i in range(3 if e2e_steps else 0):
        e2e_step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)   # the first copy starts inside the timed region
    for i in range(e2e_steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    e2e_ms = max_over_ranks(e2e_ms, dev, world)
    if world > 1:
        dist.barrier()
    assert int(status.item()) == 0

    nxt = None
    others = None
    if rank == 0:
        nxt = measure_next_rows(sv, cfg, a, s, dev, stream, status)
        nxt["mla"] = measure_mla(sv, dev, stream, status)
        nxt["multi_layer"] = measure_multi_layer(sv, cfg, a, n, s, dev, stream, status)
        if not args.no_configs:
            others = []
            for name, sg in other_configs(args.workload, sigma):
                others.append(measure_config(sv, workloads.CONFIGS[name], sg, seed, dev, stream,
                                             args.config_steps, cpu=not args.no_cpu_baseline))

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    ms_step = total_ms / args.steps
    value = job_steps_per_sec(args.steps, world, total_ms)
    # per-op times: medians of the per-step events (p10 / p90 beside them)
    attn_us = 1e3 * pct(attn_ms, 50)
    samp_us = 1e3 * pct(samp_ms, 50)
    app_us = 1e3 * pct(app_ms, 50)
    peak, peak_kind = measured_peaks()
    attn_gbs = attn_bytes / (attn_us * 1e-6) / 1e9
    samp_gbs = samp_bytes / (samp_us * 1e-6) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(cfg, sigma, lens, world, step_bytes),
        "tokens_per_sec": world * emitted_per_step * args.steps / (total_ms / 1e3),
        "hbm_gbs_step": step_bytes / (ms_step * 1e-3) / 1e9,
        "frac_of_8tbs_step": step_bytes / (ms_step * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
        "ops": {"stat": "median of per-step CUDA events", "append_us": app_us, "attn_us": attn_us,
                "sample_us": samp_us, "append": dist_summary(app_ms), "attn": dist_summary(attn_ms),
                "sample": dist_summary(samp_ms),
                "step": dist_summary([x + y + z for x, y, z in zip(app_ms, attn_ms, samp_ms)]),
                "attn_bytes": attn_bytes, "sample_bytes": samp_bytes, "append_bytes": app_bytes,
                "attn_gbs": attn_gbs, "sample_gbs": samp_gbs,
                "attn_frac_of_8tbs": attn_gbs / NOMINAL_HBM_GBS, "sample_frac_of_8tbs": samp_gbs / NOMINAL_HBM_GBS,
                "emitted_tokens_per_step": emitted_per_step},
        "roofline": {"bound": "hbm", "kernel": "spec_verify_attn (attn_tc5_kernel + attn_merge_kernel)",
                     "achieved": attn_gbs, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": attn_gbs / peak, "traffic": attn_traffic_from_profile()},
        "roofline_sample": {"bound": "hbm", "kernel": "spec_verify_sample (stats + draw + finish)",
                            "achieved": samp_gbs, "peak": peak, "unit": "GB/s", "frac": samp_gbs / peak},
        "e2e": ({"value": job_steps_per_sec(e2e_steps, world, e2e_ms), "unit": UNIT,
                 "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h} if e2e_steps else None),
        "gpu_launches": timed_launches,
        "clocks": clk,
        "next": nxt,
        "configs": others,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(cfg, a, n, s, sigma)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------- oracle -----

def measure_next_rows(sv, cfg, a, s, dev, stream, status, reps=20):
    """The opt-in parts beyond the timed step, each timed alone with CUDA
    events on the launching stream (outside the step's timed region):
    sampling at top_p = 0.9 with the draft rows filtered too, the top-p
    filter alone over those target and draft rows (HBM-bound: every row read
    once and written once), the copy-on-write page copy of one page per
    sequence in this layer's K and V pools, and tree verification (attention
    and sampling) with a five-node draft tree in place of the chain."""
    import torch

    import workloads

    def timed(fn):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return 1e3 * e0.elapsed_time(e1) / reps

    B, K, V = cfg.B, cfg.K, cfg.V
    peak, _ = measured_peaks()
    ws = sv.alloc_workspace(sv.load_library().spec_verify_sample_topp_workspace_size(
        B, K, V, sv.SV_BF16 if s["target_logits"].dtype == torch.bfloat16 else sv.SV_F32, 1), dev)
    toks = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    nacc = torch.empty((B,), dtype=torch.int32, device=dev)
    samp_us = timed(lambda: sv.spec_verify_sample(s["target_logits"], s["draft_logits"], s["draft_tokens"],
                                                  s["uniforms"], out_tokens=toks, num_accepted=nacc,
                                                  workspace=ws, status=status, want_probs=False, top_p=0.9,
                                                  draft_top_p=True))
    rows = torch.cat([s["target_logits"].reshape(-1, V), s["draft_logits"].reshape(-1, V)])
    filt = torch.empty_like(rows)
    filt_us = timed(lambda: sv.topp_filter(rows, 0.9, out=filt, status=status))
    filt_bytes = 2 * rows.numel() * rows.element_size()
    kc, vc = a["k_cache"], a["v_cache"]
    pages = [(int(b), int(b)) for b in a["block_table"][:, 0].tolist()]     # one page per sequence, onto itself
    page_bytes = kc.stride(0) * kc.element_size()
    idx = torch.tensor(pages, dtype=torch.int32).t().contiguous().to(dev)
    lib = sv.load_library()
    import ctypes
    pools = (ctypes.c_void_p * 2)(kc.data_ptr(), vc.data_ptr())

    def cow():
        rc = lib.sv_copy_blocks(pools, 2, page_bytes, page_bytes, ctypes.c_void_p(idx[0].data_ptr()),
                                ctypes.c_void_p(idx[1].data_ptr()), len(pages), kc.shape[0],
                                ctypes.c_void_p(status.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0
    cow_us = timed(cow)
    cow_bytes = 2 * 2 * len(pages) * page_bytes

    # draft tree of K + 1 = 5 nodes per sequence: root, two children, one
    # grandchild under each (the same positions and bytes as the chain)
    n = K + 1
    parents = [-1, 0, 0, 1, 2][:n] if n <= 5 else [-1] + list(range(n - 1))
    par = torch.tensor(parents, dtype=torch.int32, device=dev).repeat(B, 1)
    q_t, kc_t, vc_t = a["q"], a["k_cache"], a["v_cache"]
    attn_out = torch.empty_like(q_t)
    tws = sv.alloc_workspace(sv.load_library().spec_verify_attn_tree_workspace_size(
        B, n, cfg.H_q, cfg.H_kv, cfg.d_head, a["block_table"].shape[1], cfg.block_size), dev)
    tattn_us = timed(lambda: sv.spec_verify_attn(q_t, kc_t, vc_t, a["block_table"], a["seq_lens"], None,
                                                a["k_scale"], a["v_scale"], out=attn_out, workspace=tws,
                                                status=status, tree_parent=par))
    attn_bytes = workloads.attention_bytes(cfg, a["seq_lens"].tolist())
    drafts = torch.zeros((B, n, V), dtype=s["draft_logits"].dtype, device=dev)
    drafts[:, :K] = s["draft_logits"]
    ttok = torch.zeros((B, n), dtype=torch.int32, device=dev)
    ttok[:, 1:] = s["draft_tokens"]
    t_out = torch.empty((B, n), dtype=torch.int32, device=dev)
    t_acc = torch.empty((B,), dtype=torch.int32, device=dev)
    t_path = torch.empty((B, n), dtype=torch.int32, device=dev)
    t_ws = sv.alloc_workspace(sv.load_library().spec_verify_sample_tree_workspace_size(B, n), dev)
    tsamp_us = timed(lambda: sv.spec_verify_sample_tree(s["target_logits"], drafts, par, ttok, s["uniforms"],
                                                        out_tokens=t_out, num_accepted=t_acc, path_nodes=t_path,
                                                        status=status, workspace=t_ws))
    # rows the walk needs: p_u of every node it visits, q_u of those with children
    has_child = [any(p == u for p in parents) for u in range(n)]
    tree_rows = 0
    for b_, acc in enumerate(t_acc.tolist()):
        for u in [0] + t_path[b_, :acc].tolist():
            tree_rows += 1 + (1 if has_child[u] else 0)
    tsamp_bytes = tree_rows * V * s["target_logits"].element_size()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return {
        "tree": {"parents": parents,
                 "attn_us": tattn_us,
                 "attn_roofline": {"bound": "hbm", "kernel": "attn_tc5_kernel (tree mask)",
                                   "achieved": attn_bytes / (tattn_us * 1e-6) / 1e9, "peak": peak, "unit": "GB/s",
                                   "frac": attn_bytes / (tattn_us * 1e-6) / 1e9 / peak, "bytes": attn_bytes},
                 "sample_us": tsamp_us, "rows_read": tree_rows,
                 "sample_roofline": {"bound": "hbm", "kernel": "sample_tree_kernel",
                                     "achieved": tsamp_bytes / (tsamp_us * 1e-6) / 1e9, "peak": peak,
                                     "unit": "GB/s", "frac": tsamp_bytes / (tsamp_us * 1e-6) / 1e9 / peak,
                                     "bytes": tsamp_bytes}},
        "top_p": {"top_p": 0.9, "draft_top_p": True, "sample_topp_us": samp_us,
                  "filter_us": filt_us, "filter_rows": rows.shape[0],
                  "roofline": {"bound": "hbm",
                               "kernel": "topp_bin_kernel" if rows.shape[1] <= 188000 else "topp_row_kernel",
                               "achieved": filt_bytes / (filt_us * 1e-6) / 1e9,
                               "peak": peak, "unit": "GB/s",
                               "frac": filt_bytes / (filt_us * 1e-6) / 1e9 / peak, "bytes": filt_bytes}},
        "cow_copy": {"pairs": len(pages), "pools": 2, "page_bytes": page_bytes, "us": cow_us,
                     "roofline": {"bound": "hbm", "kernel": "copy_blocks_kernel",
                                  "achieved": cow_bytes / (cow_us * 1e-6) / 1e9, "peak": peak, "unit": "GB/s",
                                  "frac": cow_bytes / (cow_us * 1e-6) / 1e9 / peak, "bytes": cow_bytes}},
    }


def measure_mla(sv, dev, stream, status, reps=10, B=64, n_new=5, H=128, ctx=(1024, 8192), seed=0):
    """MLA verify attention on a DeepSeek-V2 layer shape: 128 heads, latent rows
    of d_c + d_r = 512 + 64 bf16 values, K = 4 drafts (5 query positions), the
    70B config's batch and ragged context lengths, 16-token blocks in a
    random permutation. The cache (about 340 MB) is larger than L2. Work is
    counted as the algorithm's multiply-adds (Q K^T over 576 values and P V
    over 512 per visible key and query row), not the kernel's own (it
    computes Q K^T once per output half)."""
    import torch
    g = torch.Generator(device="cpu").manual_seed(seed)
    lens = torch.randint(ctx[0], ctx[1] + 1, (B,), generator=g).tolist()
    nblk = [(L + 15) // 16 for L in lens]
    nb = sum(nblk) + 8
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    table = torch.full((B, max(nblk)), -1, dtype=torch.int32)
    off = 0
    for b, k in enumerate(nblk):
        table[b, :k] = perm[off:off + k]
        off += k
    gd = torch.Generator(device=dev).manual_seed(seed)
    cache = torch.randn((nb, 16, 576), generator=gd, device=dev).to(torch.bfloat16)
    q = torch.randn((B, n_new, H, 576), generator=gd, device=dev).to(torch.bfloat16)
    table, seq = table.to(dev), torch.tensor(lens, dtype=torch.int32, device=dev)
    out = torch.empty((B, n_new, H, 512), dtype=torch.bfloat16, device=dev)
    ws = sv.alloc_workspace(sv.mla_workspace_size(B, n_new, H, table.shape[1]), dev)
    scale = 1.0 / math.sqrt(128 + 64)
    fn = lambda: sv.spec_verify_attn_mla(q, cache, table, seq, scale, out=out, workspace=ws, status=status)
    for _ in range(3):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / reps
    assert int(status.item()) == 0
    vis = sum(H * (L - n_new + j + 1) for L in lens for j in range(n_new))
    flops = 2.0 * vis * (576 + 512)
    nbytes = sum(lens) * 1152 + q.numel() * 2 + out.numel() * 2
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        tpeak = float(json.load(f)["bf16_tflops"])
    cpu = mla_oracle_time(q, cache, table, lens, nblk, scale)
    return {"workload": "DeepSeek-V2 MLA layer shape: B=%d, H=%d, d_c=512, d_r=64, K=%d, ctx uniform [%d, %d], "
                        "block_size 16, bf16" % (B, H, n_new - 1, ctx[0], ctx[1]),
            "us": us, "flops": flops, "bytes": nbytes, "cpu_baseline": cpu,
            "roofline": {"bound": "tensor", "kernel": "attn_mla_kernel", "achieved": flops / (us * 1e-6) / 1e12,
                         "peak": tpeak, "unit": "TFLOP/s", "frac": flops / (us * 1e-6) / 1e12 / tpeak,
                         "hbm_gbs": nbytes / (us * 1e-6) / 1e9}}


def mla_oracle_time(q, cache, table, lens, nblk, scale):
    """The fp64 oracle on the host cores for the sequence of median length,
    scaled to the whole batch by visible keys (its work is linear in them)."""
    import numpy as np
    import torch

    from oracle import mla as omla
    b = int(np.argsort(lens)[len(lens) // 2])
    rows = cache[table[b, :nblk[b]].long()].reshape(-1, cache.shape[-1])[: lens[b]].cpu()
    qb = q[b].cpu()
    n_new = q.shape[1]
    t0 = time.perf_counter()
    omla.latent_attention(qb, rows, scale, 512)
    dt = time.perf_counter() - t0
    keys = lambda L: sum(L - n_new + j + 1 for j in range(n_new))
    full = dt * sum(keys(L) for L in lens) / keys(lens[b])
    return {"value": full * 1e6, "unit": "us per call", "cores": cpu_cores(), "kind": "oracle",
            "sample": "oracle.mla.latent_attention (numpy fp64) on sequence %d (%d tokens), %.2f s, scaled to all "
                      "%d sequences by visible keys" % (b, lens[b], dt, len(lens))}


def measure_multi_layer(sv, cfg, a, n, s, dev, stream, status, n_layers=8, reps=5):
    """One verify round over n_layers layers (append + attention per layer, one
    sampling pass) launched directly and as a replayed CUDA graph. The layers
    share this layer's pools (each layer's working set is far above L2, so a
    layer reads its KV from HBM either way) and have their own queries."""
    import torch
    layers = [{"q": a["q"].clone(), "k_new": n["k_new"], "v_new": n["v_new"], "k_cache": a["k_cache"],
               "v_cache": a["v_cache"], "k_scale": a["k_scale"], "v_scale": a["v_scale"]} for _ in range(n_layers)]
    mv = sv.MultiLayerVerify(layers, a["block_table"], a["seq_lens"], s["target_logits"], s["draft_logits"],
                             s["draft_tokens"], s["uniforms"], block_size=cfg.block_size)

    def timed(fn):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(torch.cuda.current_stream())
        for _ in range(reps):
            fn()
        e1.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        return 1e3 * e0.elapsed_time(e1) / reps
    direct_us = timed(mv.run)
    mv.capture()
    graph_us = timed(mv.replay)
    assert int(mv.status.item()) == 0
    return {"layers": n_layers, "direct_us": direct_us, "graph_us": graph_us,
            "per_layer_us_graph": graph_us / n_layers}


def oracle_sample_time(cfg, a, n, s, n_attn, n_samp):
    """Seconds the oracle takes for the append + attention of sequences
    [0, n_attn) and the sampling of sequences [0, n_samp); returns the time
    scaled to one full step and a description of the sample."""
    import numpy as np

    from oracle import attention as oatt
    from oracle import kv_append as oapp
    from oracle import sampling as osamp
    cpu = lambda d: {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in d.items()}
    a, n, s = cpu(a), cpu(n), cpu(s)
    lens = a["seq_lens"].tolist()
    idx = list(range(n_attn))
    t0 = time.perf_counter()
    sub_lens = a["seq_lens"][idx]
    oapp.kv_block_append(a["k_cache"], a["v_cache"], n["k_new"][idx], n["v_new"][idx],
                         a["block_table"][idx], sub_lens, cfg.block_size, cfg.kv_dtype,
                         a["k_scale"], a["v_scale"])
    t1 = time.perf_counter()
    oatt.verify_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["seq_lens"],
                          1 / math.sqrt(cfg.d_head), cfg.block_size, cfg.kv_dtype, a["k_scale"],
                          a["v_scale"], batch_indices=idx)
    t2 = time.perf_counter()
    osamp.rejection_sample_chunked(s["target_logits"], s["draft_logits"], s["draft_tokens"],
                                   s["uniforms"], batch_indices=list(range(n_samp)))
    t3 = time.perf_counter()
    key_frac = sum(lens[:n_attn]) / sum(lens)
    full = (t1 - t0) * cfg.B / n_attn + (t2 - t1) / key_frac + (t3 - t2) * cfg.B / n_samp
    desc = ("oracle append+attention on sequences 0..%d (%d of %d keys) and sampling on sequences "
            "0..%d of %d, scaled to the full batch" % (n_attn - 1, sum(lens[:n_attn]), sum(lens),
                                                      n_samp - 1, cfg.B))
    return full, t3 - t0, desc


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(cfg, a, n, s, sigma, min_seconds=10.0, max_reps=5):
    """The oracle on the whole step (every sequence), repeated until at least
    min_seconds of CPU work have been timed."""
    reps, spent, desc = 0, 0.0, ""
    while reps < max_reps and (reps == 0 or spent < min_seconds):
        _, t, desc = oracle_sample_time(cfg, a, n, s, cfg.B, cfg.B)
        spent += t
        reps += 1
    return {"value": reps / spent, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": "the full step (append, attention and sampling of all %d sequences), %d time(s), "
                      "%.1f s of CPU work; numpy fp64 (BLAS threads = cores)" % (cfg.B, reps, spent)}


def run_reference(args, rank, world):
    check_world(args, world)
    if rank != 0:
        return
    import torch

    import workloads
    cfg = workloads.CONFIGS[args.workload]
    sigma = cfg.sigma if args.sigma is None else args.sigma
    a = workloads.make_attention_inputs(cfg, seed=args.seed)
    n = workloads.make_append_inputs(cfg, seed=args.seed)
    s = workloads.make_sampling_inputs(cfg, seed=args.seed, sigma=sigma)
    lens = a["seq_lens"].tolist()
    step_bytes = (workloads.attention_bytes(cfg, lens) + workloads.sampling_bytes(cfg)
                  + workloads.append_bytes(cfg))
    # size each step's sample so the whole run stays near 90 s of CPU work
    _, t_one, _ = oracle_sample_time(cfg, a, n, s, 1, 1)
    per_step = 90.0 / max(1, args.steps + args.warmup)
    n_attn = n_samp = max(1, min(cfg.B, int(per_step / max(t_one, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample_time(cfg, a, n, s, n_attn, n_samp)
    fulls = []
    desc = ""
    t0 = time.perf_counter()
    for _ in range(args.steps):
        full, _, desc = oracle_sample_time(cfg, a, n, s, n_attn, n_samp)
        fulls.append(full)
    wall = time.perf_counter() - t0
    value = 1.0 / statistics.mean(fulls)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(fulls),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(cfg, sigma, lens, world, step_bytes),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": desc + "; each step is this sample (%.1f s wall for %d steps)"
                             % (wall, args.steps)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    del torch


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.mla_only:
        import torch
        import speculative_verify_paged_gb300 as sv
        sv.build()
        sv.load_library()
        dev = torch.device("cuda:0")
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        print(json.dumps(measure_mla(sv, dev, torch.cuda.current_stream(), status, B=args.mla_batch)))
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
