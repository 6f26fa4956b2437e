"""Benchmark of the DeepSeek-V4 attention O-projection on GB300.

One step = the whole hot path over one batch of synthetic input:
inverse RoPE + FP8 quantisation -> grouped wo_a GEMM (with the fused per-128
re-quantisation of z) -> wo_b GEMM, through the C ABI (dsv4_o_proj).
Default workload: T = 4096 tokens, 128 heads of 512 (16 groups x 8),
o_lora_rank 1024, hidden 7168.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  Under torchrun each rank runs its own T tokens
(weak scaling, replicated weights, no collective on the data path); the
timing is the max over ranks.  --impl reference times the CPU oracle on a
bounded token sample of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import dsv4_inputs as di  # noqa: E402

METRIC = "O-proj tokens/s"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--tokens", type=int, default=None, help="tokens per GPU (default 4096)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other synthetic workloads (decode, prefill, quant sweep) that "
                         "the default run times after the full O-projection")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--summarize-traffic", metavar="CSV", default=None,
                    help="print the per-launch DRAM lines of profiles/dram_traffic_full_T4096.txt "
                         "from an ncu --csv launch list (no GPU needed) and exit")
    ap.add_argument("--workload", default="full",
                    choices=["full", "tiny", "decode", "prefill", "quant1k", "quant8k", "quant32k",
                             "decode_bf16", "prefill_bf16"],
                    help="full: the O-projection (default); decode / prefill: quant + grouped "
                         "wo_a; quantNk: the quantiser alone (timed by CUDA-graph replay over "
                         "rotating input sets)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def workload(args) -> di.Workload:
    w = di.WORKLOADS["full"]
    if args.tokens:
        w = w.with_tokens(args.tokens)
    return w


def rank_workload(w: di.Workload, rank: int) -> di.Workload:
    """Token shard of one rank: the same shapes and weights, its own T tokens."""
    import dataclasses
    return dataclasses.replace(w, seed=w.seed + 1000 * rank,
                               weight_seed=w.seed if w.weight_seed is None else w.weight_seed)


def reduce_max(x: float, device) -> float:
    """Max of a per-rank scalar over all ranks (the slowest rank's time)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, steps: int, ms_total: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * world * steps / (ms_total / 1e3)


def config_of(w: di.Workload, n_gpus: int) -> dict:
    return {
        "workload": f"full O-projection: T={w.T} tokens/GPU, {w.H} heads x 512 "
                    f"({w.n_groups} groups x {w.heads_per_group}), o_lora_rank {w.o_lora_rank}, "
                    f"hidden {w.hidden}, positions U[0,{w.max_pos})",
        "tokens_per_gpu": w.T, "n_groups": w.n_groups, "heads_per_group": w.heads_per_group,
        "head_dim": w.head_dim, "o_lora_rank": w.o_lora_rank, "hidden": w.hidden,
        "global_tokens": w.T * n_gpus, "parallelism": f"replicas x{n_gpus} (token shards)",
        "l2": "inputs larger than L2 (o 537 MB + weights 184 MB streamed per step)",
    }


# ---------------------------------------------------------------- clocks --
class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU sampled every
    INTERVAL_MS while the `with` block (the timed region) runs: read through
    NVML (the library nvidia-smi itself uses) from a background thread, or,
    where NVML cannot be loaded, by an nvidia-smi loop.  Nothing is set, only
    read."""
    INTERVAL_MS = 2
    # clock-event reason bits of NVML's public API
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []          # (sm_mhz, power_w or None, reason names)
        self.max_mhz = None
        self.source = None
        self._nvml = None
        self._thread = None
        self._proc = None

    def _nvml_handle(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit")
        p = torch.cuda.get_device_properties(self.gpu)
        bus = "%08x:%02x:%02x.0" % (getattr(p, "pci_domain_id", 0), getattr(p, "pci_bus_id", 0),
                                    getattr(p, "pci_device_id", 0))
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
            if nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
                raise OSError("nvml handle")
        reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        return nv, h, reasons

    def __enter__(self):
        import ctypes
        import threading
        try:
            nv, h, reasons = self._nvml_handle()
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # 1: SM clock
                self.max_mhz = float(mx.value)
            self._stop = threading.Event()

            def loop():
                mhz, mw, bits = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
                while not self._stop.is_set():
                    if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(mhz)) == 0:
                        pw = mw.value / 1e3 if nv.nvmlDeviceGetPowerUsage(
                            h, ctypes.byref(mw)) == 0 else None
                        rs = [n for b, n in self.REASONS.items() if bits.value & b] \
                            if reasons(h, ctypes.byref(bits)) == 0 else []
                        self.samples.append((float(mhz.value), pw, rs))
                    self._stop.wait(self.INTERVAL_MS / 1e3)

            self._thread = threading.Thread(target=loop, daemon=True)
            self._thread.start()
            self.source = f"nvml, every {self.INTERVAL_MS} ms"
        except (OSError, AttributeError):
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "20"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi, every 20 ms"
            except OSError:
                self._proc = None
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        if self._proc is not None:
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
                out, _ = self._proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for ln in out.splitlines():
                f = [x.strip() for x in ln.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm, self.max_mhz = float(f[1]), float(f[2])
                    pw = float(f[3])
                except ValueError:
                    continue
                self.samples.append((sm, pw, [n for n, v in zip(names, f[5:9])
                                              if v.lower().startswith("active")]))

    def summary(self) -> dict:
        sm = [s[0] for s in self.samples]
        pw = [s[1] for s in self.samples if s[1] is not None]
        reasons = sorted({r for s in self.samples for r in s[2]})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(sm),
                "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": max(pw) if pw else None, "source": self.source}


def recorded_traffic(kernel: str) -> float | None:
    """DRAM bytes per launch of `kernel` from the committed ncu summary of the
    full workload, or None when the kernel sources changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic_full_T4096.txt")
    if not os.path.exists(path):
        return None
    csrc = os.path.join(ROOT, "deepseek_v4_attention_gb300", "csrc")
    vals = []
    with open(path) as f:
        for line in f:
            tok = line.split()
            if not tok or tok[0].startswith("#"):
                continue
            if tok[0] == "source":
                with open(os.path.join(csrc, tok[1]), "rb") as g:
                    if hashlib.sha256(g.read()).hexdigest() != tok[2]:
                        return None
            elif tok[0] == kernel:
                vals.append(float(tok[1]) + float(tok[2]))
    return sum(vals) / len(vals) if vals else None


TRAFFIC_SOURCES = ("dsv4_gemm.cu", "dsv4_gemm_pair.cu", "dsv4_gemm_common.cuh", "dsv4_quant.cu",
                   "dsv4_device.cuh")


def summarize_traffic(csv_path: str) -> str:
    """The body of profiles/dram_traffic_full_T4096.txt from an ncu launch list
    (--csv with gpu__time_duration.sum, dram__bytes_read.sum and
    dram__bytes_write.sum): the sha256 of the kernel sources, then one line per
    launch, grouped by kernel.  recorded_traffic() reads it back."""
    import csv
    import hashlib
    launches: dict[str, tuple[str, dict]] = {}
    header = None
    with open(csv_path, newline="") as f:
        for row in csv.reader(f):
            if "Kernel Name" in row:
                header = row
                continue
            if header is None or len(row) != len(header):
                continue
            rec = dict(zip(header, row))
            name, metrics = launches.setdefault(rec["ID"], (rec["Kernel Name"], {}))
            metrics[rec["Metric Name"]] = float(rec["Metric Value"].replace(",", ""))

    def kernel_of(name: str) -> str:
        if "inv_rope" in name:
            return "quant"
        # the re-quantising epilogue (kEpi = 1) is wo_a's: the first template
        # argument of the CTA-pair kernel, the second of the one-SM kernel
        pair_quant = "pair_kernel<1>" in name or "pair_kernel<1," in name
        return "wo_a" if (pair_quant or "<256, 1," in name) else "wo_b"

    csrc = os.path.join(ROOT, "deepseek_v4_attention_gb300", "csrc")
    lines = []
    for src in TRAFFIC_SOURCES:
        with open(os.path.join(csrc, src), "rb") as g:
            lines.append(f"source {src} {hashlib.sha256(g.read()).hexdigest()}")
    lines.append("# kernel  read_bytes  write_bytes  duration_us (one line per captured launch)")
    for k in ("quant", "wo_a", "wo_b"):
        for name, m in launches.values():
            if kernel_of(name) == k:
                lines.append(f"{k} {m['dram__bytes_read.sum'] / 1e6:.1f}e6 "
                             f"{m['dram__bytes_write.sum'] / 1e6:.1f}e6 "
                             f"{m['gpu__time_duration.sum'] / 1e3:.1f}")
    return "\n".join(lines)


def measured_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# Dense tensor-core work per SM and clock of the MMAs the kernels issue
# (tcgen05.mma): kind::mxf8f6f4 with e4m3 operands, 128 x 256 x 32
# multiply-adds per SM in 128 cycles (one SM's tile, or its half of a CTA
# pair's 256 x 256 x 32) = 16384 flop per clock; kind::f16 with bf16 operands
# half of that.  152 SMs at 1.81 GHz give the nominal 4.5 PFLOP/s FP8.
MMA_FLOP_PER_CLK_SM = {"e4m3": 16384.0, "bf16": 8192.0}
SUSTAINED_REGION_S = 1.0   # timed regions at least this long use the sustained peak


def tensor_peak(peaks: dict, src: str, timed_s: float, dtype: str) -> tuple[float, str]:
    """The measured tensor peak for a contraction of `dtype` timed inside a
    region of timed_s seconds: the burst cuBLAS bf16 figure for a short region,
    the sustained one for a region of a second or more; FP8 = 2 x bf16 (the
    nominal dense ratio)."""
    ratio = 2.0 if dtype == "e4m3" else 1.0
    if timed_s >= SUSTAINED_REGION_S and "bf16_tflops_sustained" in peaks:
        base, which = peaks["bf16_tflops_sustained"], "bf16_tflops_sustained"
    else:
        base, which = peaks["bf16_tflops"], "bf16_tflops (burst)"
    rule = f"{src}: {which}" + (" x 2 (fp8 = 2 x bf16)" if ratio == 2.0 else "") + \
        f", timed region {timed_s * 1e3:.1f} ms"
    return ratio * base, rule


def add_roofline(stage: dict, peaks: dict, src: str, timed_s: float, clocks: dict,
                 num_sms: int, dtype: str = "e4m3") -> dict:
    """Fills peak / frac of one stage; for a tensor-bound stage also the
    clock-matched MMA peak (per-SM rate x SMs x the median sampled SM clock)
    and the achieved TFLOP/s per GHz of that clock."""
    if stage["bound"] == "hbm":
        stage["peak"], stage["peak_rule"] = peaks["hbm_gbs"], f"{src}: hbm_gbs"
    else:
        stage["peak"], stage["peak_rule"] = tensor_peak(peaks, src, timed_s, dtype)
        mhz = clocks.get("sm_mhz") or clocks.get("sm_max_mhz")
        if mhz:
            cm = MMA_FLOP_PER_CLK_SM[dtype] * num_sms * mhz * 1e6 / 1e12
            stage["clock_matched"] = {"peak": cm, "frac": stage["achieved"] / cm,
                                      "sm_mhz": mhz, "unit": "TFLOP/s"}
            stage["tflops_per_ghz"] = stage["achieved"] / (mhz / 1e3)
    stage["frac"] = stage["achieved"] / stage["peak"]
    return stage


def gpu_local_cpus(local_rank: int) -> set[int] | None:
    """CPUs on the NUMA node the GPU is attached to (sysfs of its PCI device),
    or None when that cannot be read."""
    try:
        bus = subprocess.run(["nvidia-smi", "-i", str(local_rank), "--query-gpu=pci.bus_id",
                              "--format=csv,noheader"], capture_output=True, text=True,
                             timeout=20).stdout.strip()
        with open(f"/sys/bus/pci/devices/{bus[-12:].lower()}/local_cpulist") as f:
            text = f.read().strip()
    except (OSError, subprocess.SubprocessError):
        return None
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    cpus &= os.sched_getaffinity(0)
    return cpus or None


def copy_gbs(dst: torch.Tensor, src: torch.Tensor, dev, reps: int = 5) -> float:
    """GB/s of one cudaMemcpyAsync of src into dst (pinned host <-> device),
    timed with CUDA events on the copying stream after one untimed copy."""
    s = torch.cuda.Stream(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        dst.copy_(src, non_blocking=True)
        e0.record(s)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        e1.record(s)
    torch.cuda.synchronize(dev)
    return src.numel() * src.element_size() * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9


# ------------------------------------------------------------- our arm --
def run_ours(args, ws, rank, local):
    import deepseek_v4_attention_gb300 as k

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    w = rank_workload(workload(args), rank)                 # each rank its own tokens
    host = di.make_inputs(w)
    d = {n: t.to(dev) for n, t in host.items()}
    need = k.dsv4_o_proj_workspace_bytes(w.T, w.n_groups, w.heads_per_group, w.head_dim,
                                         w.o_lora_rank)
    wsp = torch.empty(need, dtype=torch.uint8, device=dev)
    out = torch.empty(w.T, w.hidden, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    kw = dict(n_groups=w.n_groups, heads_per_group=w.heads_per_group, o_lora_rank=w.o_lora_rank,
              out=out, workspace=wsp)
    args_dev = [d[n] for n in ("o", "positions", "cache", "wo_a", "wo_a_scale", "wo_b",
                               "wo_b_scale")]

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, dev)

    # per-kernel events, recorded by the library between its three launches
    n_ev = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_ev)]
    for e in evs:                      # create the events outside the timed region
        for ev in e:
            ev.record(stream)
    for _ in range(args.warmup):
        k.dsv4_o_proj(*args_dev, **kw)
    torch.cuda.synchronize(dev)
    if k.dsv4_device_status(clear=True) != 0:
        raise RuntimeError("device status error during warm-up")

    launches = 0
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t0.record(stream)
        for i in range(args.steps):
            k.dsv4_o_proj(*args_dev, **kw, stage_events=evs[i])
            launches += k.dsv4_last_launch_count()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    ms_total = max_over_ranks(t0.elapsed_time(t1))
    if k.dsv4_device_status(clear=True) != 0:
        raise RuntimeError("device status error in the timed region")
    ms_step = ms_total / args.steps
    value = job_throughput(w.T, ws, args.steps, ms_total)

    stage_ms = [0.0, 0.0, 0.0]
    for e in evs:
        for j in range(3):
            stage_ms[j] += e[j].elapsed_time(e[j + 1])
    stage_ms = [x / n_ev for x in stage_ms]

    # The library launches each GEMM to overlap the kernel before it, which
    # per-kernel events would prevent: the step is timed again without them
    # (same barrier / synchronize / max-over-ranks rules), and that is the
    # reported value; the events above give the breakdown.
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t0.record(stream)
        for i in range(args.steps):
            k.dsv4_o_proj(*args_dev, **kw)
            launches += k.dsv4_last_launch_count()
        t1.record(stream)
        torch.cuda.synchronize(dev)
    barrier()
    ms_events = ms_total
    ms_total = max_over_ranks(t0.elapsed_time(t1))
    if k.dsv4_device_status(clear=True) != 0:
        raise RuntimeError("device status error in the timed region")
    ms_step = ms_total / args.steps
    value = job_throughput(w.T, ws, args.steps, ms_total)
    step_timing = (f"launches overlapped, no events (with per-kernel events: "
                   f"{ms_events / args.steps:.4f} ms per step)")
    launches //= 2

    # --- e2e: host buffers in, host result out, through the same C-ABI call.
    # Every step copies its own o and positions from pinned host memory and
    # reads its own result back; steps are pipelined as a serving loop would
    # run them: the input copy of step i+1 (copy stream) and the read-back of
    # step i-1 (read-back stream) overlap the compute of step i, with two
    # device input buffers and two device output buffers.
    e2e = None
    if not args.no_e2e:
        nbuf = 2
        # Pinned host buffers on the NUMA node the GPU is attached to (pages
        # are placed where the allocating thread runs), as a serving process
        # bound to its GPU's CPUs would hold them.
        saved_affinity = os.sched_getaffinity(0)
        local_cpus = gpu_local_cpus(local)
        if local_cpus:
            os.sched_setaffinity(0, local_cpus)
        try:
            o_h = [host["o"].pin_memory() for _ in range(nbuf)]
            p_h = [host["positions"].pin_memory() for _ in range(nbuf)]
            out_h = [torch.empty(w.T, w.hidden, dtype=torch.bfloat16).pin_memory()
                     for _ in range(nbuf)]
        finally:
            os.sched_setaffinity(0, saved_affinity)
        o_d = [torch.empty_like(d["o"]) for _ in range(nbuf)]
        p_d = [torch.empty_like(d["positions"]) for _ in range(nbuf)]
        out_d = [torch.empty_like(out) for _ in range(nbuf)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        e2e_steps = max(3, min(args.steps, 50))
        ev = lambda: torch.cuda.Event()  # noqa: E731
        loaded = [ev() for _ in range(nbuf)]      # input copy of a buffer done
        computed = [ev() for _ in range(nbuf)]    # compute of a buffer done
        drained = [ev() for _ in range(nbuf)]     # read-back of a buffer done
        consumed = [ev() for _ in range(nbuf)]    # compute finished reading the inputs
        kw_e = dict(kw)

        def run(n):
            for i in range(n):
                b = i % 2
                with torch.cuda.stream(s_in):           # H2D of step i
                    s_in.wait_event(consumed[b])
                    o_d[b].copy_(o_h[b], non_blocking=True)
                    p_d[b].copy_(p_h[b], non_blocking=True)
                    loaded[b].record(s_in)
                stream.wait_event(loaded[b])            # compute of step i
                stream.wait_event(drained[b])
                kw_e["out"] = out_d[b]
                k.dsv4_o_proj(o_d[b], p_d[b], *args_dev[2:], **kw_e)
                consumed[b].record(stream)
                computed[b].record(stream)
                with torch.cuda.stream(s_out):          # D2H of step i
                    s_out.wait_event(computed[b])
                    out_h[b].copy_(out_d[b], non_blocking=True)
                    drained[b].record(s_out)

        for e in loaded + computed + drained + consumed:
            e.record(stream)
        run(2)
        torch.cuda.synchronize(dev)
        # five timed regions, the median reported (stalls of the host side of
        # the pipeline have hit single regions)
        e_runs = []
        for _ in range(5):
            barrier()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            run(e2e_steps)
            stream.wait_stream(s_out)                   # the last read-back is inside
            a1.record(stream)
            torch.cuda.synchronize(dev)
            barrier()
            e_runs.append(max_over_ranks(a0.elapsed_time(a1)))
        e_ms = statistics.median(e_runs)
        h2d_bytes = o_h[0].numel() * 2 + p_h[0].numel() * 8
        d2h_bytes = out_h[0].numel() * 2
        # the host link measured on this machine in this run: one copy of the
        # step's o in, one of its out back, from/to the same pinned buffers
        h2d_gbs = copy_gbs(o_d[0], o_h[0], dev)
        d2h_gbs = copy_gbs(out_h[0], out_d[0], dev)
        bound_ms = max(h2d_bytes / (h2d_gbs * 1e9) * 1e3, d2h_bytes / (d2h_gbs * 1e9) * 1e3,
                       ms_step)
        value_e2e = job_throughput(w.T, ws, e2e_steps, e_ms)
        bound = job_throughput(w.T, ws, 1, bound_ms)
        e2e = {"value": value_e2e, "unit": UNIT,
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "steps": e2e_steps, "regions": 5,
               "region_values": [job_throughput(w.T, ws, e2e_steps, x) for x in e_runs],
               "pipeline": "input copy / compute / read-back of consecutive steps overlap "
                           "(two buffers, three streams)",
               "link": {"h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
                        "pinned_on_gpu_numa_node": bool(local_cpus),
                        "bound": bound, "frac_of_bound": value_e2e / bound,
                        "bound_rule": "T / max(h2d bytes / h2d GB/s, d2h bytes / d2h GB/s, "
                                      "device step time)"}}
        del o_h, p_h, out_h, o_d, p_d, out_d

    # --- roofline of the dominant kernel (the largest stage time)
    peaks, src = measured_peaks()
    clocks = clk.summary()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    timed_s = ms_total / 1e3
    T, G, R, D, Hd = w.T, w.n_groups, w.o_lora_rank, w.D, w.hidden
    fl_a = 2.0 * T * G * R * D
    fl_b = 2.0 * T * Hd * G * R
    quant_bytes = T * w.H * (1024 + 512 + 4) + T * (8 + 256)
    stages = {
        "quant": {"ms": stage_ms[0], "bound": "hbm", "algorithmic": quant_bytes,
                  "achieved": quant_bytes / (stage_ms[0] * 1e-3) / 1e9, "unit": "GB/s"},
        "wo_a": {"ms": stage_ms[1], "bound": "tensor", "algorithmic": fl_a,
                 "achieved": fl_a / (stage_ms[1] * 1e-3) / 1e12, "unit": "TFLOP/s"},
        "wo_b": {"ms": stage_ms[2], "bound": "tensor", "algorithmic": fl_b,
                 "achieved": fl_b / (stage_ms[2] * 1e-3) / 1e12, "unit": "TFLOP/s"},
    }
    for s_ in stages.values():
        add_roofline(s_, peaks, src, timed_s, clocks, num_sms)
    dom = max(stages, key=lambda n: stages[n]["ms"])
    ds = stages[dom]
    roofline = {"kernel": dom, "bound": ds["bound"], "achieved": ds["achieved"],
                "peak": ds["peak"], "unit": ds["unit"], "frac": ds["frac"],
                "traffic": recorded_traffic(dom) if w.T == 4096 else None,
                "peak_source": ds["peak_rule"]}
    if "clock_matched" in ds:
        roofline["clock_matched"] = ds["clock_matched"]

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic (seeded; FP8 block-scaled weights drawn in stored form)",
        "config": config_of(w, ws), "clocks": clocks, "e2e": e2e,
        "gpu_launches": launches, "roofline": roofline, "step_timing": step_timing,
        "stages": {n: {kk: v for kk, v in s.items()} for n, s in stages.items()},
    }
    if rank == 0 and not args.no_configs and ws == 1:
        result["configs"] = {}
        for name in CONFIG_WORKLOADS:
            r = run_workload(name, max(args.steps, 200), max(args.warmup, 3), local)
            result["configs"][name] = r
            result["gpu_launches_configs"] = result.get("gpu_launches_configs", 0) + \
                r["gpu_launches"]
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result if rank == 0 else None


# ------------------------------------------------------ oracle (CPU) --
def _oracle_tokens(w: di.Workload, host: dict, idx, oracle):
    ti = torch.as_tensor(idx)
    oracle.o_proj(host["o"][ti], host["positions"][ti], host["cache"], host["wo_a"],
                  host["wo_a_scale"], host["wo_b"], host["wo_b_scale"], n_groups=w.n_groups,
                  heads_per_group=w.heads_per_group, o_lora_rank=w.o_lora_rank, hidden=w.hidden)


def _oracle_stages(w: di.Workload, host: dict, idx, oracle) -> dict:
    """The same O-projection as _oracle_tokens, stage by stage (O-1 quant, O-2
    grouped wo_a, O-3 z re-quant + wo_b); returns each stage's seconds."""
    ti = torch.as_tensor(idx)
    T = len(idx)
    G, R, D = w.n_groups, w.o_lora_rank, w.D
    t0 = time.perf_counter()
    x, xs = oracle.inv_rope_fp8_quant(host["o"][ti], host["positions"][ti], host["cache"],
                                      G, w.heads_per_group)
    t1 = time.perf_counter()
    z = oracle.grouped_gemm(x, xs, host["wo_a"], host["wo_a_scale"], T, G, D, R)
    t2 = time.perf_counter()
    zq, zs = oracle.block_quant_rows(z.reshape(T, G * R))
    oracle.grouped_gemm(zq, zs, host["wo_b"], host["wo_b_scale"], T, 1, G * R, w.hidden)
    t3 = time.perf_counter()
    return {"quant": t1 - t0, "wo_a": t2 - t1, "wo_b": t3 - t2}


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


def cpu_baseline(w: di.Workload, seconds: float, host: dict | None = None) -> dict:
    """The oracle as it stands, on a bounded token sample of the same workload:
    the whole O-projection on all host threads (the reported value), its stages
    separately, and a one-thread run on a small sub-sample."""
    import oracle
    host = host or di.make_inputs(w)
    threads = oracle.num_threads()
    n = max(1, threads)
    t = time.perf_counter()
    _oracle_tokens(w, host, list(range(n)), oracle)
    per_tok = (time.perf_counter() - t) / n
    m = max(n, min(w.T, int(seconds / max(per_tok, 1e-9))))
    m = max(threads, m // threads * threads)
    t = time.perf_counter()
    _oracle_tokens(w, host, list(range(m)), oracle)
    el = time.perf_counter() - t
    # stage by stage on a quarter of the sample, then one thread on 8 tokens
    ms_ = max(threads, m // 4 // threads * threads)
    st = _oracle_stages(w, host, list(range(ms_)), oracle)
    quant_bytes = w.H * (2 * w.head_dim + w.head_dim + 4) + 8 + 4 * w.rope_dim
    work = {"quant": (quant_bytes * ms_ / 1e9, "GB/s"),
            "wo_a": (2.0 * ms_ * w.n_groups * w.o_lora_rank * w.D / 1e9, "GFLOP/s"),
            "wo_b": (2.0 * ms_ * w.hidden * w.n_groups * w.o_lora_rank / 1e9, "GFLOP/s")}
    stages = {k: {"s": round(v, 3), "tokens_per_s": ms_ / v,
                  work[k][1]: work[k][0] / v} for k, v in st.items()}
    one = min(8, w.T)
    oracle.set_num_threads(1)
    try:
        t = time.perf_counter()
        _oracle_tokens(w, host, list(range(one)), oracle)
        el1 = time.perf_counter() - t
    finally:
        oracle.set_num_threads(threads)
    return {"value": m / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{m} of the workload's {w.T} tokens through the whole O-projection "
                      f"(plain C, fp64 GEMMs), {el:.1f} s; stages on {ms_} tokens; "
                      f"one thread on {one} tokens",
            "cpu_model": _cpu_model(), "stages": stages,
            "one_thread": {"value": one / el1, "unit": UNIT}}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    import oracle
    w = workload(args)
    host = di.make_inputs(w)
    threads = oracle.num_threads()
    # size one step so that warmup + steps take ~90 s in all
    t = time.perf_counter()
    _oracle_tokens(w, host, list(range(threads)), oracle)
    per_tok = (time.perf_counter() - t) / threads
    budget = 90.0 / max(1, args.steps + args.warmup)
    n = max(1, min(w.T, int(budget / max(per_tok, 1e-9))))
    rng = list(range(w.T))
    for i in range(args.warmup):
        _oracle_tokens(w, host, rng[(i * n) % w.T:][:n] or rng[:n], oracle)
    t = time.perf_counter()
    for i in range(args.steps):
        s0 = (i * n) % w.T
        _oracle_tokens(w, host, (rng[s0:] + rng[:s0])[:n], oracle)
    el = time.perf_counter() - t
    value = n * args.steps / el
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; FP8 block-scaled weights drawn in stored form)",
        "config": config_of(w, ws),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{n} tokens per step of the workload's {w.T}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------- per-workload reports --
def _graph_ms(fn, steps: int, stream) -> dict:
    """Device time per call of fn over `steps` calls, captured in a CUDA graph of
    10 calls and replayed (no host launch overhead in the measurement).  Each
    replay is timed on its own: the mean over all calls, and the median, p10 and
    p90 of the per-replay times per call."""
    chunk = min(steps, 10)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(chunk):
            fn(i)
    reps = max(1, steps // chunk)
    with torch.cuda.stream(stream):          # replay on the stream the events are on
        g.replay()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
        ev[0].record(stream)
        for r in range(reps):
            g.replay()
            ev[r + 1].record(stream)
    torch.cuda.synchronize()
    per = sorted(ev[r].elapsed_time(ev[r + 1]) / chunk for r in range(reps))
    q = lambda f: per[min(reps - 1, int(f * reps))]
    return {"ms": ev[0].elapsed_time(ev[reps]) / (reps * chunk), "p10_ms": q(0.1),
            "p50_ms": q(0.5), "p90_ms": q(0.9)}


# The other synthetic workloads the default run times after the full
# O-projection, each by CUDA-graph replay: tiny (correctness-sized), decode
# (weight-read bound wo_a), prefill (FP8 tensor bound wo_a) and the quantiser
# sweep.
CONFIG_WORKLOADS = ("tiny", "decode", "prefill", "quant1k", "quant8k", "quant32k")


def run_workload(name: str, steps: int, warmup: int, local: int, tokens: int | None = None) -> dict:
    """One of the smaller synthetic workloads: quant (+ grouped wo_a).  Each step
    uses the next of several rotating input sets whose total exceeds 3x L2, so
    that weights and activations come from HBM, not from the previous step.
    The quantiser sweep's large o tensors are drawn on the device (same recipe,
    the device's random stream) to keep the host's generation time short."""
    import deepseek_v4_attention_gb300 as k

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    bf16 = name.endswith("_bf16")
    w = di.WORKLOADS[name.replace("_bf16", "")]
    if tokens:                 # the same shapes at another token count
        w = w.with_tokens(tokens)
    gemm = not w.name.startswith("quant")
    on_device = w.name in ("quant8k", "quant32k")
    host = di.make_inputs(w, with_wo_b=False, o_device=dev if on_device else None)
    if bf16:   # the model served without FP8: bf16 wo_a, quantize=False
        host["wo_a"] = di.bf16_weight(w.n_groups * w.o_lora_rank, w.D, w.seed + 303)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    esz = 2 if bf16 else 1
    set_bytes = host["o"].numel() * 2 + (host["wo_a"].numel() * esz if gemm else 0) + \
        w.n_groups * w.T * w.D * esz + (w.T * w.n_groups * w.o_lora_rank * 2 if gemm else 0)
    nsets = max(1, min(32, -(-3 * l2 // set_bytes)))
    T_al = k.tma_aligned_tokens(w.T)
    sets = []
    for i in range(nsets):
        st = {n: host[n].to(dev) for n in ("o", "positions", "cache")}
        st["x"] = torch.empty(w.n_groups, w.T, w.D, dtype=torch.bfloat16 if bf16
                              else torch.float8_e4m3fn, device=dev)
        st["xs"] = torch.empty(w.n_groups, (w.D // 128 + 3) // 4, T_al, dtype=torch.int32,
                               device=dev)
        if gemm:
            st["wo_a"] = host["wo_a"].to(dev)
            st["wo_a_scale"] = host["wo_a_scale"].to(dev)
            st["z"] = torch.empty(w.T, w.n_groups, w.o_lora_rank, dtype=torch.bfloat16,
                                  device=dev)
        sets.append(st)
    del host
    stream = torch.cuda.Stream(dev)

    def quant(i):
        st = sets[i % nsets]
        if bf16:
            return k.dsv4_inv_rope_bf16(st["o"], st["positions"], st["cache"], w.n_groups,
                                        w.heads_per_group, out=st["x"], stream=stream)
        return k.dsv4_inv_rope_fp8_quant(st["o"], st["positions"], st["cache"], w.n_groups,
                                         w.heads_per_group, out_fp8=st["x"], out_scale=st["xs"],
                                         stream=stream)

    # The step launches wo_a to overlap the kernel before it (the quantiser,
    # which does not write the weights): the GEMM's prologue and weight reads
    # run under it.  Timed alone, wo_a is measured both ways: back to back with
    # the same overlap (the previous call writes only its own z) and serialised.
    def wo_a(i, overlap=True):
        st = sets[i % nsets]
        if bf16:
            k.dsv4_grouped_wo_a_bf16(st["x"].transpose(0, 1), st["wo_a"], w.n_groups,
                                     w.o_lora_rank, z=st["z"], stream=stream)
            return
        k.dsv4_grouped_wo_a(st["x"].transpose(0, 1), st["xs"].permute(2, 0, 1)[:w.T],
                            st["wo_a"], st["wo_a_scale"], w.n_groups, w.o_lora_rank, z=st["z"],
                            overlap_previous=overlap, stream=stream)

    def wo_a_serial(i):
        wo_a(i, overlap=False)

    # decode sizes: the quantiser fused into wo_a is timed beside the step (the
    # step is the two separate launches, the faster of the two at these sizes)
    fused = gemm and not bf16 and w.T <= k.FUSED_MAX_TOKENS

    def wo_a_fused(i):
        st = sets[i % nsets]
        k.dsv4_inv_rope_grouped_wo_a(st["o"], st["positions"], st["cache"], st["wo_a"],
                                     st["wo_a_scale"], w.n_groups, w.heads_per_group,
                                     w.o_lora_rank, z=st["z"], stream=stream)

    def step(i):
        quant(i)
        if gemm:
            wo_a(i)

    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            step(i)
    torch.cuda.synchronize()
    launches_per_step = 2 if gemm else 1
    with ClockSampler(local) as clk:
        t_step = _graph_ms(step, steps, stream)
        t_q = _graph_ms(quant, steps, stream)
        t_a = _graph_ms(wo_a, steps, stream) if gemm else None
        t_as = _graph_ms(wo_a_serial, steps, stream) if gemm and not bf16 else None
        t_f = _graph_ms(wo_a_fused, steps, stream) if fused else None
    ms_step, ms_q = t_step["ms"], t_q["ms"]
    ms_a = t_a["ms"] if gemm else 0.0
    spread = lambda t: {k_: round(v, 5) for k_, v in t.items() if k_ != "ms"}
    if k.dsv4_device_status(clear=True) != 0:
        raise RuntimeError("device status error")
    peaks, src = measured_peaks()
    clocks = clk.summary()
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    dtype = "bf16" if bf16 else "e4m3"
    qbytes = w.T * w.H * (1024 + (1024 if bf16 else 512 + 4)) + w.T * (8 + 256)
    stages = {"quant": {"ms": ms_q, "bound": "hbm", "algorithmic": qbytes,
                        "achieved": qbytes / (ms_q * 1e-3) / 1e9, "unit": "GB/s", **spread(t_q)}}
    if gemm:
        fl = 2.0 * w.T * w.n_groups * w.o_lora_rank * w.D
        by = (w.n_groups * w.o_lora_rank * w.D + w.n_groups * w.T * w.D) * esz + \
            w.T * w.n_groups * w.o_lora_rank * 2
        if w.name in ("decode", "tiny"):      # weight-read bound: bytes against HBM
            stages["wo_a"] = {"ms": ms_a, "bound": "hbm", "algorithmic": by,
                              "achieved": by / (ms_a * 1e-3) / 1e9, "unit": "GB/s",
                              **spread(t_a)}
        else:
            stages["wo_a"] = {"ms": ms_a, "bound": "tensor", "algorithmic": fl,
                              "achieved": fl / (ms_a * 1e-3) / 1e12, "unit": "TFLOP/s",
                              **spread(t_a)}
    if t_as is not None:   # the same GEMM launched without overlap (not part of the step)
        bound = stages["wo_a"]["bound"]
        work = by if bound == "hbm" else fl
        scale = 1e9 if bound == "hbm" else 1e12
        stages["wo_a_serial"] = {"ms": t_as["ms"], "bound": bound, "algorithmic": work,
                                 "achieved": work / (t_as["ms"] * 1e-3) / scale,
                                 "unit": stages["wo_a"]["unit"], **spread(t_as)}
    if fused:   # one kernel: o and the weights in, z out (not part of the step)
        fb = w.T * w.H * 1024 + w.T * (8 + 256) + w.n_groups * w.o_lora_rank * w.D + \
            w.T * w.n_groups * w.o_lora_rank * 2
        stages["fused_quant_wo_a"] = {"ms": t_f["ms"], "bound": "hbm", "algorithmic": fb,
                                      "achieved": fb / (t_f["ms"] * 1e-3) / 1e9, "unit": "GB/s",
                                      **spread(t_f)}
    for n_, s_ in stages.items():
        region_s = {"quant": t_q, "wo_a": t_a, "wo_a_serial": t_as,
                    "fused_quant_wo_a": t_f}[n_]["ms"] * steps / 1e3
        add_roofline(s_, peaks, src, region_s, clocks, num_sms, dtype)
    dom = max((n for n in stages if n not in ("fused_quant_wo_a", "wo_a_serial")),
              key=lambda n: stages[n]["ms"])
    ds = stages[dom]
    roofline = {"kernel": dom, "bound": ds["bound"], "achieved": ds["achieved"],
                "peak": ds["peak"], "unit": ds["unit"], "frac": ds["frac"],
                "traffic": None, "peak_source": ds["peak_rule"]}
    if "clock_matched" in ds:
        roofline["clock_matched"] = ds["clock_matched"]
    return {
        "metric": METRIC, "value": w.T / (ms_step * 1e-3), "unit": UNIT, "n_gpus": 1,
        "steps": steps, "warmup": warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype,
        "data": "synthetic (seeded; " + ("bf16 weights" if bf16 else
                                         "FP8 block-scaled weights drawn in stored form") +
                ("; o drawn on the device" if on_device else "") + ")",
        "launch": "wo_a launched to overlap the kernel before it (its prologue and weight "
                  "reads under that kernel; wo_a_serial: the same GEMM without overlap)"
                  if gemm and not bf16 else None,
        "config": {"workload": f"{name}: T={w.T}, {w.H} heads x 512 ({w.n_groups} "
                               f"groups x {w.heads_per_group})" +
                               (f", o_lora_rank {w.o_lora_rank}, " + ("bf16 inverse RoPE + bf16 "
                                "grouped wo_a" if bf16 else "quant + grouped wo_a")
                                if gemm else ", quantiser alone"),
                   "timing": "CUDA-graph replay, graphs of 10 calls; p10/p50/p90 over the "
                             "replays", "input_sets": nsets,
                   "l2": f"{nsets} rotating input sets of {set_bytes / 1e6:.1f} MB (>= 3x L2)"},
        "clocks": clocks, "gpu_launches": launches_per_step * steps,
        "roofline": roofline, "stages": stages, "step_spread": spread(t_step),
    }


def main():
    args = parse()
    if args.summarize_traffic:
        print(summarize_traffic(args.summarize_traffic))
        return
    ws, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
    elif args.workload != "full":
        if ws > 1:
            raise SystemExit("--workload other than full runs on one GPU")
        res = run_workload(args.workload, args.steps, args.warmup, local, args.tokens)
    else:
        res = run_ours(args, ws, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
