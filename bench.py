"""ChunkKV compression throughput on GB300: HBM GB/s and tokens/s of the full path.

One step = one chunkkv_compress_layers call over every layer of the workload
(score + select on the scoring layers of Algorithm 2, gather on every layer),
inputs resident in HBM.  value = algorithmic bytes / device time, where the
algorithmic bytes are the keys read by every scoring layer plus the kept K and
V rows read and written on every layer (plus the window queries).

The default workload is the largest single-GPU configuration, the Qwen2-7B-
shaped 28-layer model with T = 131072 (qwen_128k); the LLaMA-3-8B-shaped
32-layer model with T = 32768 is measured in the same run and reported as a
secondary line object.

--impl reference times the CPU oracle, single-threaded, on the host on a
bounded sample of the same workload (whole heads of the first scoring layer
per step) and reports the same metric.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)


def _oracle_process() -> bool:
    """Whether this process only times the CPU oracle (the reference arm, or the child process of the
    cpu_baseline leg): those run the oracle single-threaded, so every BLAS / OpenMP pool is held to one
    thread before numpy loads."""
    argv = sys.argv[1:]
    ref = any(a == "--impl=reference" or (a == "--impl" and i + 1 < len(argv) and argv[i + 1] == "reference")
              for i, a in enumerate(argv))
    return ref or "--cpu-baseline-child" in argv


if _oracle_process():
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
               "NUMEXPR_NUM_THREADS", "VECLIB_MAXIMUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np  # noqa: E402
import torch  # noqa: E402

from synthetic import configs, generator as gen  # noqa: E402

METRIC = "chunkkv_compress_hbm_gbps"
UNIT = "GB/s"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in self.rows:
            if len(r) >= 9:
                for n, v in zip(names, r[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows)}


def slowest_rank(step_ms: float, ws_n: int) -> float:
    """The job's step time: the maximum over the ranks of the default process group (all_reduce MAX;
    on the GPU for NCCL, on the host for gloo)."""
    if ws_n <= 1:
        return step_ms
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([step_ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def job_rate(units_per_rank: float, ws_n: int, step_ms: float) -> float:
    """Whole-job throughput: the units every rank processed (replicas: the same per rank) per second
    of the slowest rank's step."""
    return units_per_rank * ws_n / (step_ms * 1e-3)


def algorithmic_bytes(wl, counts) -> int:
    """K read by the scoring layers + kept K, V rows read and written on every layer + Q_w."""
    elt = 2 if wl.dtype == "bf16" else 4
    n_score = -(-wl.n_layers // wl.n_reuse)
    k_read = n_score * wl.T_total * wl.Hkv * wl.d * elt
    q_read = n_score * wl.B * wl.w * wl.Hq * wl.d * elt
    kept = 0
    cnt = counts.to("cpu").numpy().astype(np.int64)         # [groups, B, Hkv]
    for layer in range(wl.n_layers):
        kept += int(cnt[layer // wl.n_reuse].sum())
    return k_read + q_read + 4 * kept * wl.d * elt


def sources_digest(paths) -> str:
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_record(workload: str, kernel: str):
    """DRAM read + write bytes per full launch of `kernel` on `workload`, from the committed one-pass
    ncu capture (profiles/traffic.json), or None if the kernel's sources changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)["workloads"][workload][kernel]
        if sources_digest(rec["sources"]) != rec["sources_sha256"]:
            return None
        return int(rec["dram_read_bytes"]) + int(rec["dram_write_bytes"])
    except Exception:
        return None


def head_path(wl, groups) -> bool:
    """Whether the library runs log-sum-exp, finalisation and selection as one kernel per head: the
    same rule as the library's planner (window rows present, at most 16384 chunks per sequence, and
    the (group, sequence, head) CTAs, one per SM, making one wave over at least 3/4 of the SMs)."""
    c_max = max(-(-(wl.cu_seqlens[b + 1] - wl.cu_seqlens[b]) // wl.c) for b in range(wl.B)) if wl.B else 0
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    heads = wl.B * wl.Hkv * groups
    return wl.w * wl.G > 0 and c_max <= 16384 and heads <= sms and 4 * heads >= 3 * sms


def phase_rooflines(wl, counts, phase_ms, peaks, peak_src, path, ex2_rate=None):
    """Roofline of the scoring, finalisation and gather launches of one compress step.

    Algorithmic amounts per launch (all layers / reuse groups of the step):
      score:    K of every scoring layer read once (T_total*Hkv*d*elt per group),
                2*w*G*T_total*Hkv*d flops and one base-2 exponential per logit
                (w*G*T_total*Hkv per group); the roof is whichever takes longest at peak:
                HBM copy bandwidth, the sustained bf16 tensor rate, or the exponential rate
                that chunkkv_probe_ex2 measured on this GPU (ex2_rate, exponentials/s);
      finalize: one 16-bit bin per (chunk, window row, KV head) per group read once (the phase is
                one kernel with the log-sum-exp and the selection when head_path() holds);
      gather:   kept K and V rows read and written (4*kept*d*elt per layer).
    Returns (rooflines of the three phases, every roof of the scoring phase).
    """
    elt = 2 if wl.dtype == "bf16" else 4
    groups = -(-wl.n_layers // wl.n_reuse)
    cnt = counts.to("cpu").numpy().astype(np.int64)
    kept_all = sum(int(cnt[layer // wl.n_reuse].sum()) for layer in range(wl.n_layers))
    chunks = sum(-(-(wl.cu_seqlens[b + 1] - wl.cu_seqlens[b]) // wl.c) for b in range(wl.B))
    hbm = peaks["hbm_gbs"]
    tensor = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])

    def hbm_roof(phase, kernel, nbytes):
        ms = phase_ms[phase]
        ach = nbytes / (ms * 1e-3) / 1e9
        return {"phase": phase, "kernel": kernel, "bound": "hbm", "achieved": round(ach, 2), "peak": hbm,
                "unit": "GB/s", "frac": round(ach / hbm, 4), "traffic": traffic_record(wl.name, kernel),
                "algorithmic_bytes": int(nbytes), "avg_launch_ms": round(ms, 5),
                "peak_source": f"{peak_src} hbm_gbs"}

    score_bytes = groups * wl.T_total * wl.Hkv * wl.d * elt
    score_flops = 2.0 * groups * wl.w * wl.G * wl.T_total * wl.Hkv * wl.d
    score_exps = float(groups * wl.w * wl.G * wl.T_total * wl.Hkv)
    kernel = "score_tc_kernel" if path == 1 else "score_simt_kernel"
    ms = phase_ms["score"]
    score_roofs = [dict(hbm_roof("score", kernel, score_bytes), ideal_ms=round(score_bytes / (hbm * 1e9) * 1e3, 5))]
    if path == 1:
        ach = score_flops / (ms * 1e-3) / 1e12
        score_roofs.append({"phase": "score", "kernel": kernel, "bound": "tensor", "achieved": round(ach, 2),
                            "peak": tensor, "unit": "TFLOP/s", "frac": round(ach / tensor, 4),
                            "traffic": traffic_record(wl.name, kernel), "algorithmic_flops": score_flops,
                            "algorithmic_bytes": int(score_bytes), "avg_launch_ms": round(ms, 5),
                            "ideal_ms": round(score_flops / (tensor * 1e12) * 1e3, 5),
                            "peak_source": f"{peak_src} bf16_tflops_sustained"})
    if ex2_rate:
        ach = score_exps / (ms * 1e-3) / 1e9
        peak = ex2_rate["exp_per_s"] / 1e9
        score_roofs.append({"phase": "score", "kernel": kernel, "bound": "sfu", "achieved": round(ach, 2),
                            "peak": round(peak, 2), "unit": "Gexp/s", "frac": round(ach / peak, 4),
                            "traffic": traffic_record(wl.name, kernel), "algorithmic_exps": score_exps,
                            "algorithmic_bytes": int(score_bytes), "avg_launch_ms": round(ms, 5),
                            "ideal_ms": round(score_exps / ex2_rate["exp_per_s"] * 1e3, 5),
                            "peak_source": "measured here: chunkkv_probe_ex2 (ex2.approx.ftz.f32)"})
    out = [max(score_roofs, key=lambda r: r["ideal_ms"])]         # the roof that takes longest binds
    fin_kernel = "head_kernel" if head_path(wl, groups) else "finalize_kernel"
    out.append(hbm_roof("finalize", fin_kernel, groups * chunks * wl.Hkv * wl.w * wl.G * 2))
    out.append(hbm_roof("gather", "gather_kernel", 4 * kept_all * wl.d * elt))
    return out, score_roofs


def ex2_probe(ckv, dev, gpu_index: int):
    """Exponential rate of this GPU: chunkkv_probe_ex2 over 8 CTAs of 256 threads per SM, launches back
    to back for about half a second (median of the per-launch event times), with the SM clock sampled
    meanwhile."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, iters = 8 * sms, 2048
    sink = torch.empty(blocks * 256, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    n_exp = ckv.chunkkv_probe_ex2(sink, blocks, iters)
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_index)
    sampler.start()
    time.sleep(0.3)
    evs = []
    t_end = time.perf_counter() + 0.6
    while time.perf_counter() < t_end or len(evs) < 20:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ckv.chunkkv_probe_ex2(sink, blocks, iters)
        e1.record(stream)
        evs.append((e0, e1))
        if len(evs) % 50 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    rate = n_exp / (ms * 1e-3)
    out = {"exp_per_s": rate, "launch_ms": round(ms, 5), "exps_per_launch": n_exp, "launches": len(evs),
           "sm_mhz": clocks.get("sm_mhz"), "reasons": clocks.get("reasons")}
    if clocks.get("sm_mhz"):
        out["exp_per_clk_per_sm"] = round(rate / (clocks["sm_mhz"] * 1e6) / sms, 2)
    return out


def link_probe(dev, nbytes: int = 1 << 30):
    """Host link bandwidth with pinned host memory: one 1 GiB cudaMemcpyAsync each way (best of 3)."""
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    res = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        best = None
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        res[f"{name}_GBps"] = round(nbytes / (best * 1e-3) / 1e9, 1)
    del h, d
    return res


def workload_of(args):
    """The workload named on the command line, with the sweep point (--chunk, --budget) and the
    layer count (--layers) applied."""
    wl = configs.ALL[args.workload]()
    c = getattr(args, "chunk", 0) or wl.c
    L = getattr(args, "budget", 0) or wl.L_max
    if (c, L) != (wl.c, wl.L_max):
        base = wl.name.split("_c")[0] if wl.name.startswith("mistral") else wl.name
        wl = wl.with_params(c=c, L_max=L, name=f"{base}_c{c}_L{L}")
    if args.layers:
        wl = wl.with_params(n_layers=args.layers, name=f"{wl.name}_first{args.layers}L")
    if getattr(args, "causal", False):
        wl = wl.with_params(name=f"{wl.name}_causal")
    return wl


def device_timing(ckv, wl, args, dev, local, ws_n, peaks, peak_src, ex2_rate):
    """Warm-up, then K timed compress steps (CUDA events on the launching stream, inputs resident in
    HBM), then K more steps with the library's phase events.  Returns the inputs, outputs and the
    measured figures of the workload."""
    qs, ks, vs, _ = gen.make_all_layers(wl, dev)
    p, keep = ckv.params_for(next(q for q in qs if q is not None), ks[0], wl.cu_seqlens, Hkv=wl.Hkv, w=wl.w,
                             c=wl.c, L_max=wl.L_max, causal_window=getattr(args, "causal", False))
    n_cap, C_max = ckv.chunkkv_out_capacity(p)
    groups = -(-wl.n_layers // wl.n_reuse)
    ko = [torch.empty(wl.B, wl.Hkv, n_cap, wl.d, dtype=ks[0].dtype, device=dev) for _ in range(wl.n_layers)]
    vo = [torch.empty_like(x) for x in ko]
    idx = torch.empty(groups, wl.B, wl.Hkv, n_cap, dtype=torch.int32, device=dev)
    cnt = torch.empty(groups, wl.B, wl.Hkv, dtype=torch.int32, device=dev)
    ws = torch.zeros(ckv.chunkkv_workspace_size(p, wl.n_layers, wl.n_reuse), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ckv.chunkkv_compress_layers(p, wl.n_reuse, qs, ks, vs, ko, vo, idx, cnt, None, ws)

    for _ in range(args.warmup):
        step()
    ckv.chunkkv_status_check(ws)
    in_bytes = sum(x.numel() * x.element_size() for x in ks + vs) + \
        sum(q.numel() * q.element_size() for q in qs if q is not None)
    l2_note = "inputs larger than L2 (no flush)" if in_bytes > 2 * 129e6 else "L2 flushed between steps"
    flush = torch.empty(int(2 * 129e6) // 4, dtype=torch.float32, device=dev) if in_bytes <= 2 * 129e6 else None

    sampler = ClockSampler(local)
    if ws_n > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    launches0 = ckv.chunkkv_launch_count()
    times = []
    for _ in range(args.steps):
        if flush is not None:
            flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        times.append((e0, e1))
    torch.cuda.synchronize()
    launches = ckv.chunkkv_launch_count() - launches0        # library kernels in the timed region
    if ws_n > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms = [a.elapsed_time(b) for a, b in times]
    ckv.chunkkv_status_check(ws)
    step_ms = slowest_rank(sum(ms) / len(ms), ws_n)
    nbytes = algorithmic_bytes(wl, cnt)

    # ---- device time of each phase inside the same compress call: K more steps with the library's
    # phase events recorded on its stream (a record between two launches ends their overlap, so these
    # steps are not the headline ones)
    path = ckv.chunkkv_score_path(p)
    n_ev = len(ckv.PHASES) + 1
    phase_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    for evs in phase_evs:
        if flush is not None:
            flush.fill_(1.0)
        ckv.chunkkv_set_phase_events(evs)
        step()
    ckv.chunkkv_set_phase_events(None)
    torch.cuda.synchronize()
    phase_ms = {name: sum(evs[i].elapsed_time(evs[i + 1]) for evs in phase_evs) / len(phase_evs)
                for i, name in enumerate(ckv.PHASES)}
    roofs, score_roofs = phase_rooflines(wl, cnt, phase_ms, peaks, peak_src, path, ex2_rate)
    dominant = max(roofs, key=lambda r: phase_ms[r["phase"]])
    value = job_rate(nbytes, ws_n, step_ms) / 1e9
    return {"wl": wl, "p": p, "keep": keep, "qs": qs, "ks": ks, "vs": vs, "ko": ko, "vo": vo, "idx": idx,
            "cnt": cnt, "ws": ws, "n_cap": n_cap, "step": step, "stream": stream, "l2_note": l2_note,
            "launches": launches, "clocks": clocks, "step_ms": step_ms, "nbytes": nbytes, "value": value,
            "tokens_s": job_rate(wl.T_total, ws_n, step_ms), "phase_ms": phase_ms, "roofs": roofs,
            "score_roofs": score_roofs, "dominant": dominant}


def parse_cpulist(text: str) -> set:
    """CPU numbers of a Linux cpulist ("0-3,8,10-11")."""
    cpus = set()
    for part in text.strip().split(","):
        if not part:
            continue
        lo, _, hi = part.partition("-")
        cpus.update(range(int(lo), int(hi or lo) + 1))
    return cpus


def bind_to_gpu_cpus(gpu_index: int):
    """Restrict this process to the host CPUs that the PCI topology lists as local to the GPU (its
    NUMA node), before any host buffer is allocated, so that pinned host memory lands next to the
    GPU.  Returns the CPUs kept, or None when the topology gives nothing usable."""
    try:
        bus = subprocess.run(["nvidia-smi", f"--id={gpu_index}", "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=30).stdout.strip().lower()
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{int(dom, 16):04x}:{rest}/local_cpulist"
        with open(path) as f:
            local = parse_cpulist(f.read()) & os.sched_getaffinity(0)
        if local:
            os.sched_setaffinity(0, local)
            return sorted(local)
    except Exception:
        pass
    return None


def run_gpu(args):
    import chunk_level_kv_gb300 as ckv
    ws_n, rank, local = dist_env()
    host_cpus = bind_to_gpu_cpus(local)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peak_src = measured_peaks()
    ex2_rate = ex2_probe(ckv, dev, local)

    secondary = None
    if args.secondary != "none" and args.secondary != args.workload:
        sec_args = argparse.Namespace(**vars(args))
        sec_args.workload, sec_args.chunk, sec_args.budget = args.secondary, 0, 0
        t = device_timing(ckv, workload_of(sec_args), args, dev, local, ws_n, peaks, peak_src, ex2_rate)
        secondary = {"workload": t["wl"].name, "value": round(t["value"], 3), "unit": UNIT,
                     "ms_per_step": round(t["step_ms"], 4), "hbm_roof_frac": round(t["value"] / ws_n / peaks["hbm_gbs"], 4),
                     "tokens_per_s": round(t["tokens_s"], 1), "algorithmic_bytes_per_step": t["nbytes"],
                     "phases_ms": {k: round(v, 5) for k, v in t["phase_ms"].items()}, "roofline": t["dominant"],
                     "roofline_score": t["score_roofs"], "gpu_launches": int(t["launches"]), "clocks": t["clocks"],
                     "config": {"B": t["wl"].B, "T_total": t["wl"].T_total, "layers": t["wl"].n_layers,
                                "n_reuse": t["wl"].n_reuse, "Hq": t["wl"].Hq, "Hkv": t["wl"].Hkv, "w": t["wl"].w,
                                "c": t["wl"].c, "L_max": t["wl"].L_max, "l2": t["l2_note"]}}
        del t
        torch.cuda.empty_cache()

    t = device_timing(ckv, workload_of(args), args, dev, local, ws_n, peaks, peak_src, ex2_rate)
    wl, p, qs, ks, vs, ko, vo = t["wl"], t["p"], t["qs"], t["ks"], t["vs"], t["ko"], t["vo"]
    idx, cnt, ws, n_cap, step, stream = t["idx"], t["cnt"], t["ws"], t["n_cap"], t["step"], t["stream"]
    step_ms, nbytes, value, phase_ms = t["step_ms"], t["nbytes"], t["value"], t["phase_ms"]

    # ---- §4.2 observation behind Algorithm 2: adjacent-layer overlap of the kept lists with every layer
    # scored (n_reuse = 1), and the device time of the overlap kernel
    overlap = None
    if wl.n_layers > 1 and not args.no_diagnostics:
        idx1 = torch.empty(wl.n_layers, wl.B, wl.Hkv, n_cap, dtype=torch.int32, device=dev)
        cnt1 = torch.empty(wl.n_layers, wl.B, wl.Hkv, dtype=torch.int32, device=dev)
        ws1 = torch.zeros(ckv.chunkkv_workspace_size(p, wl.n_layers, 1), dtype=torch.uint8, device=dev)
        q_all = [x if x is not None else gen.gen_q_window(wl, i, dev) for i, x in enumerate(qs)]   # every layer's own
        ckv.chunkkv_compress_layers(p, 1, q_all, ks, vs, ko, vo, idx1, cnt1, None, ws1)
        del ws1
        inter, uni = ckv.chunkkv_layer_overlap(p, idx1, cnt1)
        torch.cuda.synchronize()
        reps = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ckv.chunkkv_layer_overlap(p, idx1, cnt1)
            e1.record(stream)
            reps.append((e0, e1))
        torch.cuda.synchronize()
        ov_ms = statistics.median(a.elapsed_time(b) for a, b in reps)
        read = int(cnt1.sum()) * 4 + cnt1.numel() * 4
        u = uni.double()
        jac = torch.where(u > 0, inter.double() / u.clamp(min=1), torch.ones_like(u))
        overlap = {"lists": wl.n_layers, "mean_adjacent_jaccard": round(float(jac.mean()), 4),
                   "min_adjacent_jaccard": round(float(jac.min()), 4), "kernel_ms": round(ov_ms, 5),
                   "index_bytes_read": read, "achieved_GBps": round(read / (ov_ms * 1e-3) / 1e9, 2)}

    # ---- end to end through the C-ABI with host buffers (pinned), transfers inside the timed region
    e2e = e2e_staged = None
    if not args.no_e2e:
        # pinned host buffers allocated directly (no pageable copy in between) and filled from the device
        def pinned_like(x, fill=True):
            h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
            if fill:
                h.copy_(x)
            return h
        hq = [pinned_like(q) if q is not None else None for q in qs]
        hk = [pinned_like(x) for x in ks]
        hv = [pinned_like(x) for x in vs]
        hko = [pinned_like(x, False) for x in ko]
        hvo = [pinned_like(x, False) for x in vo]
        hidx = pinned_like(idx, False)
        hcnt = pinned_like(cnt, False)
        nbytes_of = lambda ts: sum(x.numel() * x.element_size() for x in ts if x is not None)
        cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def pipelined(sets, copies_out, n_steps, start=None):
            """Steps pipelined the way a serving loop would run them.  sets[j] = (copies_in, run) is
            the input buffer set of steps j, j + len(sets), ...: the host->device copies of step i+1
            (copy-in stream) overlap the compression of step i when there are two sets, and the
            device->host copies of step i (copy-out stream) in any case.  A step's copies into a set
            wait for the compression that last read that set, and its compression waits for the
            previous step's outputs to be copied out."""
            done_of = [start] * len(sets)
            prev_out = None
            for i in range(n_steps):
                copies_in, run = sets[i % len(sets)]
                with torch.cuda.stream(cin):
                    if done_of[i % len(sets)] is not None:
                        cin.wait_event(done_of[i % len(sets)])
                    for dst, src in copies_in:
                        dst.copy_(src, non_blocking=True)
                    loaded = torch.cuda.Event()
                    loaded.record(cin)
                stream.wait_event(loaded)
                if prev_out is not None:
                    stream.wait_event(prev_out)
                run()
                done = torch.cuda.Event()
                done.record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(done)
                    for dst, src in copies_out:
                        dst.copy_(src, non_blocking=True)
                    out_done = torch.cuda.Event()
                    out_done.record(cout)
                done_of[i % len(sets)], prev_out = done, out_done
            stream.wait_stream(cout)

        def timed(sets, copies_out):
            pipelined(sets, copies_out, len(sets))
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n_e2e = max(2, min(args.steps, 4))
            e0.record(stream)
            pipelined(sets, copies_out, n_e2e, start=e0)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / n_e2e

        # (1) The layers' K and V stay in pinned host memory.  Each step copies in the window queries
        # and the keys of the scoring layers (the tensor-core kernel reads them through TMA, so they
        # must be in device memory), into one of two device buffer sets so that the copies of step
        # i+1 run beside the compression of step i; the gather reads the kept rows of the other
        # layers' K and of every layer's V from host memory itself and writes K' and V' straight into
        # host memory, so only the kept rows cross the host link.  Indices and counts are copied out.
        elt = ks[0].element_size()
        cnt_h = cnt.to("cpu")
        kept = [int(cnt_h[layer // wl.n_reuse].sum()) for layer in range(wl.n_layers)]
        row = wl.d * elt
        scoring = [layer for layer in range(wl.n_layers) if layer % wl.n_reuse == 0]
        sets = []
        for j in range(2):
            dq = [(q if j == 0 else torch.empty_like(q)) if q is not None else None for q in qs]
            dk = {layer: ks[layer] if j == 0 else torch.empty_like(ks[layer]) for layer in scoring}
            k_args = [dk[layer] if layer in dk else hk[layer] for layer in range(wl.n_layers)]
            copies_in = [(dq[layer], hq[layer]) for layer in scoring if dq[layer] is not None] + \
                        [(dk[layer], hk[layer]) for layer in scoring]
            sets.append((copies_in, functools.partial(ckv.chunkkv_compress_layers, p, wl.n_reuse, dq, k_args, hv,
                                                      hko, hvo, idx, cnt, None, ws)))
        copies_out = [(hidx, idx), (hcnt, cnt)]
        e2e_ms = timed(sets, copies_out)
        h2d = nbytes_of([d for d, _ in sets[0][0]]) + \
            row * (sum(kept) + sum(n for layer, n in enumerate(kept) if layer % wl.n_reuse != 0))
        d2h = nbytes_of([hidx, hcnt]) + 2 * row * sum(kept)
        e2e = {"value": round(nbytes * ws_n / (e2e_ms * 1e-3) / 1e9, 3), "unit": UNIT,
               "link_probe": link_probe(dev),
               "host_cpus": (f"{len(host_cpus)} CPUs local to the GPU ({host_cpus[0]}-{host_cpus[-1]}), "
                             f"pinned buffers allocated after binding") if host_cpus else "not bound",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4),
               "transfers": "window queries and scoring-layer keys copied in (two device buffer sets); "
                            "kept K/V rows read from and K'/V' written to pinned host memory by the gather "
                            "kernel; indices and counts copied out"}
        # (2) For comparison: every layer's Q_w, K and V copied in and every output copied out.
        staged_in = [(d, h) for d, h in zip(qs, hq) if d is not None] + list(zip(ks, hk)) + list(zip(vs, hv))
        staged_out = list(zip(hko, ko)) + list(zip(hvo, vo)) + [(hidx, idx), (hcnt, cnt)]
        staged_ms = timed([(staged_in, step)], staged_out)
        e2e_staged = {"value": round(nbytes * ws_n / (staged_ms * 1e-3) / 1e9, 3), "unit": UNIT,
                      "h2d_bytes_per_step": int(nbytes_of([h for _, h in staged_in])),
                      "d2h_bytes_per_step": int(nbytes_of([h for h, _ in staged_out])),
                      "ms_per_step": round(staged_ms, 4)}

    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline and not args.causal:   # the oracle sample has no causal window
        cpu = cpu_baseline(args, budget_s=args.cpu_seconds)

    if ws_n > 1:
        torch.distributed.barrier()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded, needles planted)",
        "config": {"workload": wl.name, "B": wl.B, "T": list(wl.seqlens) if wl.B <= 4 else "ragged",
                   "T_total": wl.T_total, "layers": wl.n_layers, "n_reuse": wl.n_reuse, "Hq": wl.Hq,
                   "Hkv": wl.Hkv, "d": wl.d, "w": wl.w, "c": wl.c, "L_max": wl.L_max,
                   "causal_window": bool(args.causal), "l2": t["l2_note"], "parallelism": f"replicas x{ws_n}"},
        "tokens_per_s": round(t["tokens_s"], 1),
        "token_layers_per_s": round(t["tokens_s"] * wl.n_layers, 1),
        "algorithmic_bytes_per_step": nbytes,
        "hbm_roof_frac": round(value / ws_n / peaks["hbm_gbs"], 4),
        "roofline": t["dominant"],
        "roofline_score": t["score_roofs"],
        "ex2_probe": ex2_rate,
        "phases_ms": {k: round(v, 5) for k, v in phase_ms.items()},
        "secondary": secondary,
        "layer_overlap": overlap,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "e2e_staged": e2e_staged,
        "gpu_launches": int(t["launches"]),
        "clocks": t["clocks"],
    }
    print(json.dumps(line), flush=True)


def tail_case(base, n_new: int):
    """The caches of an incremental pass over workload `base`: (workload of the caches, kept prefix per
    sequence, the tail's budget).  A prefill pass keeps at most k c + w positions of a prompt (k =
    L_max // c chunks and the window), so each cache is that prefix followed by n_new decoded tokens; the
    tail's budget keeps the prefill's ratio L_max / T over the longest prompt, at least one chunk."""
    n_prev = [min(T, base.L_max // base.c * base.c + base.w) for T in base.seqlens]
    L_tail = max(base.c, base.L_max * n_new // max(base.seqlens))
    wl = base.with_params(seqlens=tuple(x + n_new for x in n_prev), B=len(n_prev), name=f"{base.name}_tail{n_new}")
    return wl, n_prev, L_tail


def run_tail(args):
    """Incremental pass during decoding (chunkkv_compress_tail): every cache of the workload holds the
    positions a prefill pass kept (min(T_b, k c + w) of its prompt) followed by args.tail decoded
    tokens; each pass re-scores that tail against the whole cache on the scoring layers and gathers the
    kept tail rows of every layer.  The tail's budget keeps the prefill's ratio (L_max / T_b).  Device
    time per pass with the inputs resident in HBM; bytes counted as for the prefill path (the whole
    cache's keys on each scoring layer, Q_w, and the kept rows' K and V read and written)."""
    import chunk_level_kv_gb300 as ckv
    ws_n, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peak_src = measured_peaks()
    n_new = args.tail
    wl, n_prev, L_tail = tail_case(workload_of(args), n_new)
    qs, ks, vs, _ = gen.make_all_layers(wl, dev)
    p, keep = ckv.params_for(next(q for q in qs if q is not None), ks[0], wl.cu_seqlens, Hkv=wl.Hkv, w=wl.w,
                             c=wl.c, L_max=L_tail)
    n_cap, c_max, ws_bytes = ckv.chunkkv_tail_sizes(p, n_prev, wl.n_layers, wl.n_reuse)
    groups = -(-wl.n_layers // wl.n_reuse)
    ko = [torch.empty(wl.B, wl.Hkv, max(n_cap, 1), wl.d, dtype=ks[0].dtype, device=dev) for _ in range(wl.n_layers)]
    vo = [torch.empty_like(x) for x in ko]
    idx = torch.empty(groups, wl.B, wl.Hkv, max(n_cap, 1), dtype=torch.int32, device=dev)
    cnt = torch.empty(groups, wl.B, wl.Hkv, dtype=torch.int32, device=dev)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        ckv.chunkkv_compress_tail(p, n_prev, wl.n_reuse, qs, ks, vs, ko, vo, idx, cnt, None, ws)

    for _ in range(args.warmup):
        step()
    ckv.chunkkv_status_check(ws)
    timed = step
    if args.graph:
        # the pass captured once in a CUDA graph and replayed: no host work between passes (a decode
        # loop with fixed cache sizes can do the same)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step()
        stream.wait_stream(side)
        n0 = ckv.chunkkv_launch_count()
        with torch.cuda.graph(graph):
            step()
        per_replay = ckv.chunkkv_launch_count() - n0                 # kernels each replay launches
        torch.cuda.synchronize()
        timed = graph.replay
    in_bytes = sum(x.numel() * x.element_size() for x in ks + vs)
    l2_note = "inputs larger than L2 (no flush)" if in_bytes > 2 * 129e6 else "L2 flushed between steps"
    flush = torch.empty(int(2 * 129e6) // 4, dtype=torch.float32, device=dev) if in_bytes <= 2 * 129e6 else None
    sampler = ClockSampler(local)
    if ws_n > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    launches0 = ckv.chunkkv_launch_count()
    times = []
    t_host = time.perf_counter()
    for _ in range(args.steps):
        if flush is not None:
            flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        timed()
        e1.record(stream)
        times.append((e0, e1))
    t_host = (time.perf_counter() - t_host) / args.steps * 1e3           # host time to issue one pass
    torch.cuda.synchronize()
    launches = ckv.chunkkv_launch_count() - launches0
    if args.graph:
        launches = per_replay * args.steps        # replays bypass the library's host-side launch count
    if ws_n > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms = [a.elapsed_time(b) for a, b in times]
    ckv.chunkkv_status_check(ws)
    step_ms = slowest_rank(sum(ms) / len(ms), ws_n)
    nbytes = algorithmic_bytes(wl, cnt)
    value = job_rate(nbytes, ws_n, step_ms) / 1e9
    # device time of each phase: K more passes with the library's phase events
    n_ev = len(ckv.PHASES) + 1
    phase_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    for evs in phase_evs:
        if flush is not None:
            flush.fill_(1.0)
        ckv.chunkkv_set_phase_events(evs)
        step()
    ckv.chunkkv_set_phase_events(None)
    torch.cuda.synchronize()
    phase_ms = {name: sum(evs[i].elapsed_time(evs[i + 1]) for evs in phase_evs) / len(phase_evs)
                for i, name in enumerate(ckv.PHASES)}
    del keep
    if rank != 0:
        return
    hbm = peaks["hbm_gbs"]
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded, needles planted)",
        "config": {"workload": wl.name, "mode": "incremental pass during decoding", "B": wl.B, "n_prev": n_prev,
                   "tail": n_new, "layers": wl.n_layers, "n_reuse": wl.n_reuse, "Hq": wl.Hq, "Hkv": wl.Hkv,
                   "d": wl.d, "w": wl.w, "c": wl.c, "L_tail": L_tail, "l2": l2_note,
                   "parallelism": f"replicas x{ws_n}"},
        "tail_tokens_per_s": round(job_rate(n_new * wl.B, ws_n, step_ms), 1),
        "cuda_graph": bool(args.graph), "host_ms_per_pass": round(t_host, 4),
        "phases_ms": {k: round(v, 5) for k, v in phase_ms.items()},
        "algorithmic_bytes_per_step": nbytes,
        "hbm_roof_frac": round(value / ws_n / hbm, 4),
        "roofline": {"bound": "hbm", "achieved": round(value / ws_n, 2), "peak": hbm, "unit": "GB/s",
                     "frac": round(value / ws_n / hbm, 4), "traffic": None, "kernel": "whole pass",
                     "peak_source": f"{peak_src} hbm_gbs"},
        "cpu_baseline": None, "e2e": None,
        "gpu_launches": int(launches),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def pin_one_core() -> int:
    """Restrict this process to the first core it may run on; returns that core."""
    if not hasattr(os, "sched_getaffinity"):
        return -1
    core = min(os.sched_getaffinity(0))
    os.sched_setaffinity(0, {core})
    return core


def oracle_sample(wl, q, k, budget_s: float) -> dict:
    """The oracle as it stands, in this process: Algorithm 1 for whole (sequence, KV head) pairs of the
    first scoring layer (q: [B, w, Hq, d], k: [T_total, Hkv, d] torch CPU tensors), until budget_s."""
    import oracle
    qf = q.detach().to("cpu", torch.float32).numpy().astype(np.float64)
    cu = wl.cu_seqlens
    elt = 2 if wl.dtype == "bf16" else 4
    done_bytes, done_tokens, heads = 0, 0, 0
    t0 = time.perf_counter()
    for b in range(wl.B):
        kb = k[cu[b]:cu[b + 1]].detach().to("cpu", torch.float32).numpy().astype(np.float64)
        T = cu[b + 1] - cu[b]
        for h in range(wl.Hkv):
            A, sel, idx = oracle.chunkkv_head(oracle.group_window_rows(qf[b], h, wl.G), kb[:, h], wl.c, wl.w,
                                              wl.L_max)
            oracle.gather(kb[:, h], idx)
            done_bytes += T * wl.d * elt + 2 * len(idx) * wl.d * elt
            done_tokens += T
            heads += 1
            if time.perf_counter() - t0 > budget_s:
                break
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": round(done_bytes / dt / 1e9, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"Algorithm 1 on {heads} (sequence, KV head) pairs of scoring layer 0 "
                      f"({done_tokens} tokens, {dt:.1f} s), fp64 numpy, K read + kept K/V counted "
                      f"like the GPU metric",
            "threads": 1, "cpu_model": cpu_model()}


def cpu_baseline(args, budget_s: float = 15.0) -> dict:
    """The oracle timed on one host core: a child process of this script (BLAS and OpenMP pools at one
    thread, affinity to one core) generates the first scoring layer of the same workload on the CPU and
    runs oracle_sample on it."""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-child", "--workload", args.workload,
           "--cpu-seconds", str(budget_s)]
    if args.chunk:
        cmd += ["--chunk", str(args.chunk)]
    if args.budget:
        cmd += ["--budget", str(args.budget)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=budget_s * 4 + 300)
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    if r.returncode != 0 or not lines:
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle",
                "error": (r.stderr or r.stdout)[-400:]}
    return json.loads(lines[-1])


def run_cpu_baseline_child(args):
    core = pin_one_core()
    wl = workload_of(args)
    q, k, v = gen.make_layer(wl, 0, "cpu")
    res = oracle_sample(wl, q, k, args.cpu_seconds)
    res["core"] = core
    print(json.dumps(res), flush=True)


def run_reference(args):
    """The reference arm: the oracle, single-threaded on one host core, timed step by step on a bounded
    sample of the workload (whole heads of the first scoring layer)."""
    ws_n, rank, local = dist_env()
    if rank != 0:
        return
    core = pin_one_core()
    wl = workload_of(args)
    q, k, v = gen.make_layer(wl, 0, "cpu")
    per_step = min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup))   # whole run ~ 2.5 min
    for _ in range(args.warmup):
        oracle_sample(wl, q, k, budget_s=per_step / 4)
    vals = []
    t0 = time.perf_counter()
    last = None
    for _ in range(args.steps):
        last = oracle_sample(wl, q, k, budget_s=per_step)
        vals.append(last["value"])
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / max(1, args.steps) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "T_total": wl.T_total, "layers": wl.n_layers,
                   "n_reuse": wl.n_reuse, "w": wl.w, "c": wl.c, "L_max": wl.L_max},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "threads": 1, "kind": "oracle",
                         "sample": last["sample"], "cpu_model": last["cpu_model"], "core": core},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=sorted(configs.ALL), default="qwen_128k")
    ap.add_argument("--secondary", default="llama_model",
                    help="a second workload timed in the same run (device time only); 'none' to skip")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-diagnostics", action="store_true", help="skip the adjacent-layer overlap measurement")
    ap.add_argument("--layers", type=int, default=0, help="keep only the first N layers (profiling)")
    ap.add_argument("--chunk", type=int, default=0, help="chunk size c instead of the workload's (a sweep point)")
    ap.add_argument("--budget", type=int, default=0, help="L_max instead of the workload's (a sweep point)")
    ap.add_argument("--causal", action="store_true", help="causal window (chunkkv_params.causal_window)")
    ap.add_argument("--tail", type=int, default=0,
                    help="time the incremental pass during decoding with this many new tokens per cache instead")
    ap.add_argument("--graph", action="store_true", help="with --tail: replay the pass from a CUDA graph")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.cpu_baseline_child:
        run_cpu_baseline_child(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.tail > 0:
        run_tail(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
