"""Benchmark of the MHLA forward pass on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--variant auto|simt|multipass|fused] [--impl mine|reference]
                    [--no-per-config] [--no-cpu-baseline] [--pass forward|backward]
                    [--feature-map elu1|relu|exp] [--causal] [--layout bhnd|bnhd] [--mc-per-head]

A step is one full forward (block summaries, mixing, output) over one batch
of the workload's seeded synthetic inputs, already resident in HBM.  The
metric is tokens*heads per second (B*H*N / step time).  The default workload
is the video-shaped 3D grid (B=2, H=16, d=64, 16x64x64 tokens, 2x8x8 blocks,
M=512): its 403 MB of inputs exceed the 126 MB L2, so no flush runs between
timed steps.  The default run also times every other configuration (each
with its own warm-up, an L2 flush between steps where its inputs fit in L2,
outside the per-step events) and lists them under "per_config".

Rooflines: "roofline" is the dominant kernel of the step, "kernels" every
kernel, each with the method's own bytes (or FLOPs) per launch divided by the
kernel's average launch time; "path_roofline" is the whole step against
max(bytes / HBM, FLOPs / tensor peak) with bytes = read Q, K, V, write O, read
Mc and FLOPs = 4 N d^2 + 2 M^2 d^2 per unit.

--pass backward times mhla_backward instead (one step = dQ, dK, dV and dMc of
the same workload for a seeded dO, the forward summaries recomputed inside);
its line has the same keys, with the backward's own roofline.

--impl reference times the float64 CPU oracle (the only reference there is)
on the same workload: each step is one (batch, head) unit.

Multi-GPU (torchrun): every rank runs an independent replica of the workload
(units are independent, no collective on the data path); value = all ranks'
tokens*heads / the slowest rank's time ("scaling": "weak").
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from token_level_head_phi_gb300 import workloads as wl  # noqa: E402

METRIC = "MHLA fwd tokens*heads/sec (d=64) and % of GB300 HBM/tensor roofline"
UNIT = "tokens*heads/s"
PHASES = ["prep", "summary", "scale", "mix", "output"]
L2_BYTES = 126 * 1024 * 1024


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def job_throughput(local_ms: float, steps: int, units_per_step: int, world: int, dist, device):
    """Whole-job throughput of N replicas: every rank ran `steps` steps of
    `units_per_step` token-heads in `local_ms`; the job took as long as its
    slowest rank (max over ranks), and did `world` times the work.  Returns
    (max ms over ranks, units per second)."""
    import torch
    t = torch.tensor([float(local_ms)], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    max_ms = float(t.item())
    return max_ms, world * units_per_step * steps / (max_ms / 1e3)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="mhla_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                rows.append(parts)
        os.unlink(self.path)
        # keep samples taken inside [t0, t1] (wall clock); nvidia-smi stamps are local time
        def stamp(p):
            try:
                return time.mktime(time.strptime(p[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + \
                    float("0." + p[0].split(".")[1]) if "." in p[0] else 0.0
            except Exception:
                return None
        inside = [r for r in rows if stamp(r) is not None and t0 - 0.15 <= stamp(r) <= t1 + 0.15]
        use = inside if inside else rows
        sm = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        smax = [float(r[3]) for r in use if r[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for name, val in zip(names, r[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(use), "samples_in_region": len(inside)}


# ------------------------------------------------------------ my arm

def phase_kernels(w: wl.Workload, info, fmap: str, causal: bool):
    """Kernel that runs in each phase of one forward (None: the phase is
    absent from this variant), as ncu names it, with its source file."""
    import token_level_head_phi_gb300.binding as mb
    C = "token_level_head_phi_gb300/csrc/"
    if info.variant == mb.VARIANT_SIMT:
        return {"prep": ("mc_rowsum_kernel", C + "simt.cu"), "summary": ("simt_summary_kernel", C + "simt.cu"),
                "scale": None, "mix": ("simt_mix_kernel", C + "simt.cu"),
                "output": ("causal_output_kernel", C + "simt_causal.cu") if causal else
                ("simt_output_kernel", C + "simt.cu")}
    if info.variant == mb.VARIANT_FUSED:
        return {"prep": ("tc_prep_kernel", C + "tc_mix.cu"), "summary": None, "scale": None, "mix": None,
                "output": ("tc_fused_kernel", C + "tc_fused.cu")}
    f16 = w.norm != "mala" and fmap != "exp" and not causal
    q = w.n_blocks * info.summary_splits
    small = not causal and w.n_blocks <= 16 and q <= 256          # CUDA-core mixing of few blocks
    mixt = f16 and w.n_blocks <= 128 and 2 * ((q + 63) // 64) * 32 <= 256
    mix = ("tc_mixs_kernel", C + "tc_mixs.cu") if small else \
        ("tc_mixt_kernel", C + "tc_mix.cu") if mixt else ("tc_mix_kernel", C + "tc_mix.cu")
    return {"prep": None if (f16 and small) else ("tc_prep_kernel", C + "tc_mix.cu"),
            "summary": ("tc_summary_kernel", C + "tc_summary.cu"),
            "scale": ("tc_scale_kernel", C + "tc_scale.cu") if f16 and not small else None,
            "mix": mix,
            "output": ("tc_causal_kernel", C + "tc_causal.cu") if causal else ("tc_output_kernel", C + "tc_output.cu")}


def kernel_table(w: wl.Workload, info, fmap: str, causal: bool, avg_phase: dict, peaks, sm_mhz=None):
    """One row per kernel of the forward: its average launch time and, for the
    kernels that do the method's work, the method's own bytes or FLOPs per
    launch (read K and V for the summaries; read Q and write O for the output
    step, plus K and V for the causal one; the mixing's 2 M^2 d^2 FLOPs per
    unit; Q, K, V, O for the fused launch) against the measured peak, and the
    ncu DRAM bytes per launch where the committed table has them for the
    current sources.  Preparation and exponent folding move only
    intermediates: their time is reported, no fraction."""
    import token_level_head_phi_gb300.binding as mb
    hbm, tf_burst, tf_sust, peak_kind = peaks
    el = 2 if w.dtype == "bf16" else 4
    io = w.units * w.n_tokens * w.head_dim * el
    mix_flops = 2 * w.units * w.n_blocks ** 2 * w.head_dim ** 2
    kernels = phase_kernels(w, info, fmap, causal)
    tt = traffic_table()
    rows = {}
    for ph, kern in kernels.items():
        if kern is None:
            continue
        name, src = kern
        ms = avg_phase.get(ph, 0.0)
        row = {"kernel": name, "avg_launch_ms": ms}
        if ph == "summary":
            row.update(bound="hbm", algorithmic_bytes_per_launch=2 * io)
        elif ph == "output":
            if name == "tc_fused_kernel":
                nb = 4 * io + 4 * w.n_blocks ** 2   # the whole forward in one launch
            else:
                nb = (4 if causal else 2) * io      # Q in, O out (the causal step also reads K, V)
            row.update(bound="hbm", algorithmic_bytes_per_launch=nb)
        elif ph == "mix":
            row.update(bound="tensor" if info.variant != mb.VARIANT_SIMT else "alu", flops_per_launch=mix_flops)
        else:
            row.update(bound="overhead")
        if ms > 0 and row["bound"] == "hbm":
            row["achieved"] = row["algorithmic_bytes_per_launch"] / (ms / 1e3) / 1e9
            row.update(peak=hbm, unit="GB/s", peak_source=peak_kind)
        elif ms > 0 and row["bound"] == "tensor":
            row["achieved"] = mix_flops / (ms / 1e3) / 1e12
            row.update(peak=tf_burst, unit="TFLOP/s", peak_source=peak_kind + " bf16 dense burst (fp16 runs at the same rate)")
        elif ms > 0 and row["bound"] == "alu":
            mhz = sm_mhz or 2070.0
            peak = SM_COUNT * FP32_LANES_PER_SM * 2 * mhz * 1e6 / 1e12
            row["achieved"] = mix_flops / (ms / 1e3) / 1e12
            row.update(peak=peak, unit="TFLOP/s",
                       peak_source="fp32 FMA lanes x 2 x max SM clock: %d x %d x 2 x %.0f MHz" % (SM_COUNT, FP32_LANES_PER_SM, mhz))
        if "achieved" in row:
            row["frac"] = row["achieved"] / row["peak"]
        t = tt.get((name, w.name))
        row["traffic"] = t[0] if (t and t[1] == source_hash(src)) else None
        if row["traffic"] is not None and row.get("algorithmic_bytes_per_launch"):
            row["traffic_over_algorithmic"] = row["traffic"] / row["algorithmic_bytes_per_launch"]
        rows[ph] = row
    return rows


def traffic_table():
    """Per-launch DRAM bytes from the committed ncu summary, keyed by
    (kernel, workload); each entry carries the hash of the kernel source it
    was captured from and is ignored once that source changes."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    table = {}
    if not os.path.exists(path):
        return table
    for line in open(path):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        parts = line.split()
        if len(parts) != 4:
            continue
        kernel, workload, nbytes, src_hash = parts
        table[(kernel, workload)] = (float(nbytes), src_hash)
    return table


KERNEL_HEADERS = ["token_level_head_phi_gb300/csrc/tc_common.cuh", "token_level_head_phi_gb300/csrc/common.cuh",
                  "token_level_head_phi_gb300/csrc/plan.h", "token_level_head_phi_gb300/csrc/tc_host.h",
                  "token_level_head_phi_gb300/csrc/tc_summary.cuh", "token_level_head_phi_gb300/csrc/tc_mix.cuh",
                  "token_level_head_phi_gb300/csrc/tc_mixt.cuh", "token_level_head_phi_gb300/csrc/tc_output.cuh"]


def source_hash(relpath: str) -> str:
    """Hash of a kernel's source file and the headers every kernel includes."""
    h = hashlib.sha256()
    for path in [relpath] + KERNEL_HEADERS:
        with open(os.path.join(ROOT, path), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


def run_mine(args, w: wl.Workload, world: int, rank: int, local: int, dist, sample_clocks: bool = True):
    import torch
    import token_level_head_phi_gb300.binding as mb
    from token_level_head_phi_gb300 import build as mbuild

    if rank == 0 or world == 1:
        mbuild.build()
    if dist is not None:
        dist.barrier()
    mb.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)

    qn, kn, vn = wl.all_device_inputs(w)
    mcn = wl.make_mc(w)

    def to_dev(a):
        t = torch.from_numpy(a)
        if w.dtype == "bf16":
            t = t.view(torch.bfloat16)
        return t.to(dev)

    q, k, v = to_dev(qn), to_dev(kn), to_dev(vn)
    if args.layout == "bnhd":
        # token-major [B, N, H, d], as a fused QKV projection writes it
        q, k, v = (t.permute(0, 2, 1, 3).contiguous() for t in (q, k, v))
    if args.mc_per_head:
        # one matrix per head: the workload's recipe with a different noise seed per head
        mcn = np.stack([wl.make_mc(w.with_(seed=w.seed + 101 * h)) for h in range(w.heads)]).astype(np.float32)
    mc = torch.from_numpy(mcn).to(dev)
    out = torch.empty_like(q)
    p = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, w.dtype, args.feature_map, w.norm, args.variant,
                       args.causal, args.layout, args.mc_per_head)
    info = mb.mhla_plan(p)
    ws = torch.empty(max(info.workspace_bytes, 1), dtype=torch.uint8, device=dev)
    ws_bytes = ws.numel()
    handle = stream.cuda_stream
    io_bytes = q.numel() * q.element_size()
    flush = None
    if io_bytes * 3 < 2 * L2_BYTES:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        st = mb.mhla_forward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), mc.data_ptr(), p, out.data_ptr(),
                                 ws.data_ptr(), ws_bytes, handle)
        if st != 0:
            raise mb.MhlaError(st, "mhla_forward")

    for _ in range(args.warmup):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    code, detail = mb.mhla_device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} during warm-up (detail {detail})")

    # timed region: K steps back to back (the kernels of consecutive launches
    # may overlap their set-up with the previous kernel's tail), no flush
    # when inputs exceed L2; with a flush, per-step events bracket each step
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local) if rank == 0 and sample_clocks else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    t0 = time.time()
    start.record(stream)
    host_s = 0.0
    for i in range(K):
        if flush is not None:
            flush.zero_()
            step_ev[i][0].record(stream)
        h0 = time.perf_counter()
        step()
        host_s += time.perf_counter() - h0
        if flush is not None:
            step_ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop(t0, t1) if sampler else None
    code, detail = mb.mhla_device_status()
    if code != 0:
        raise RuntimeError(f"device status {code} in timed region (detail {detail})")
    if flush is None:
        total_ms = start.elapsed_time(end)
    else:
        total_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    # inputs that fit in L2: the same steps back to back without the flush
    # (warm L2), reported beside the cold-L2 number
    warm = None
    if flush is not None:
        wa, wb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        step()
        wa.record(stream)
        for _ in range(K):
            step()
        wb.record(stream)
        torch.cuda.synchronize()
        wms = wa.elapsed_time(wb) / K
        warm = {"ms_per_step": wms, "value": w.units * w.n_tokens / (wms / 1e3), "unit": UNIT,
                "l2": "warm: no flush, steps back to back"}

    # per-phase breakdown (for the dominant kernel's roofline): a separate
    # run with events between the kernels, which serialise them
    KP = max(10, min(K, 50))
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(mb.NUM_PHASE_EVENTS)] for _ in range(KP)]
    for i in range(KP):
        if flush is not None:
            flush.zero_()
        mb.mhla_set_phase_events(ev_sets[i])
        step()
    mb.mhla_set_phase_events(None)
    torch.cuda.synchronize()
    phase_ms = {ph: [] for ph in PHASES}
    for evs in ev_sets:
        for j, ph in enumerate(PHASES):
            phase_ms[ph].append(evs[j].elapsed_time(evs[j + 1]))
    max_ms, value = job_throughput(total_ms, K, w.units * w.n_tokens, world, dist, dev)
    ms_per_step = max_ms / K

    peaks = load_peaks()
    hbm, tf_burst, tf_sust, peak_kind = peaks
    avg_phase = {ph: statistics.mean(v) for ph, v in phase_ms.items()}
    kernels = kernel_table(w, info, args.feature_map, bool(args.causal), avg_phase, peaks,
                           (clocks or {}).get("sm_max_mhz"))
    # the dominant kernel: the longest of those that do the method's work
    work = {ph: r for ph, r in kernels.items() if r["bound"] != "overhead" and "frac" in r}
    dom = max(work, key=lambda ph: work[ph]["avg_launch_ms"])
    roof = dict(work[dom], phase=dom)
    roof_bytes = wl.roofline_bytes(w)
    roof_flops = wl.roofline_flops(w)
    t_hbm = roof_bytes / (hbm * 1e9)
    # a whole step is a long run of kernels: the sustained tensor peak
    t_tc = roof_flops / (tf_sust * 1e12)
    t_roof = max(t_hbm, t_tc)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic (seeded normals, locality-biased Mc; no dataset, no weights)",
        "config": dict(wl.describe(w), feature_map=args.feature_map, causal=bool(args.causal), layout=args.layout,
                       mc_per_head=bool(args.mc_per_head),
                       variant=info.variant,
                       variant_name={1: "simt", 2: "multipass", 3: "fused"}.get(info.variant, str(info.variant)),
                       l2="no flush: inputs exceed L2" if flush is None else "L2 flushed (256 MB write) between steps, outside per-step events",
                       parallelism=f"replicas{world}" if world > 1 else "single GPU"),
        "roofline": roof,
        "kernels": kernels,
        "path_roofline": {"bytes": roof_bytes, "flops": roof_flops, "t_hbm_us": t_hbm * 1e6, "t_tc_us": t_tc * 1e6,
                          "bound": "hbm" if t_hbm >= t_tc else "tensor", "frac": t_roof / (ms_per_step / 1e3),
                          "peak_hbm_gbs": hbm, "peak_bf16_tflops_sustained": tf_sust, "peak_source": peak_kind},
        "phase_ms": avg_phase,
        "warm_l2": warm,
        "phase_note": "per-kernel times from a separate run with events between the kernels (which serialises "
                      "the launches the timed steps overlap)",
        "gpu_launches": info.kernels_per_call * K,
        "host_us_per_call": host_s / K * 1e6,
        "clocks": clocks,
    }
    return result, (q, k, v, mc, out, p, info, stream)


# The other configurations of the default run: (label, workload).  The
# video-shaped workload is the headline line itself.
PER_CONFIG = [("C0 tiny fp32", "tiny_f32"), ("C1 DeiT-T-shaped", "deit_t"), ("C2 high-res image", "image_64x64"),
              ("C4 1D 32k divisive", "seq_32k"), ("C4 1D 32k MALA", "seq_32k_mala"),
              ("C4 1D 32k M=1 divisive", "seq_32k_m1"), ("C4 1D 32k M=1 MALA", "seq_32k_m1_mala"),
              ("Wan-shaped 3D (21x30x50, 300-token blocks)", "wan_21x30x50")]


def run_per_config(args, world, rank, local, dist):
    """Each other configuration with its own warm-up and timed steps (an L2
    flush between steps where its inputs fit in L2), as the headline: step
    time, tokens*heads/s, whole-path roofline fraction and the per-kernel
    table with the dominant kernel."""
    import torch
    out = {}
    for label, name in PER_CONFIG:
        w = wl.WORKLOADS[name]
        if args.variant in ("multipass", "fused") and (w.dtype != "bf16" or w.head_dim != 64):
            continue  # the tensor-core launches take bf16 with d = 64
        sub = argparse.Namespace(**vars(args))
        sub.steps = max(10, min(args.steps, 30))
        sub.causal = False
        r, st = run_mine(sub, w, world, rank, local, dist, sample_clocks=False)
        del st
        torch.cuda.empty_cache()
        out[name] = {
            "label": label, "ms_per_step": r["ms_per_step"], "value": r["value"], "unit": UNIT,
            "path_roofline_frac": r["path_roofline"]["frac"], "path_bound": r["path_roofline"]["bound"],
            "t_roofline_us": max(r["path_roofline"]["t_hbm_us"], r["path_roofline"]["t_tc_us"]),
            "dominant": {k: r["roofline"].get(k) for k in ("kernel", "phase", "bound", "frac", "achieved", "unit",
                                                           "avg_launch_ms")},
            "kernels": {ph: {k: v for k, v in row.items() if k in ("kernel", "avg_launch_ms", "bound", "frac",
                                                                   "traffic_over_algorithmic")}
                        for ph, row in r["kernels"].items()},
            "variant_name": r["config"]["variant_name"], "dtype": w.dtype, "norm": w.norm,
            "host_us_per_call": r["host_us_per_call"],
            "steps": sub.steps, "warmup": sub.warmup, "l2": r["config"]["l2"],
            "warm_l2": r.get("warm_l2"),
        }
    return out


def run_e2e(w: wl.Workload, state, steps: int):
    """Same metric through mhla_forward_host: pinned host inputs copied in,
    result copied out, every step."""
    import torch
    import token_level_head_phi_gb300.binding as mb
    q, k, v, mc, out, p, info, stream = state
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    hmc = mc.cpu().pin_memory()
    hout = torch.empty_like(hq).pin_memory()
    need = mb.mhla_host_buffer_bytes(p)
    del q, k, v, out
    torch.cuda.empty_cache()
    buf = torch.empty(need, dtype=torch.uint8, device=mc.device)
    lib = mb.load()
    import ctypes

    def step():
        st = lib.mhla_forward_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), hmc.data_ptr(), ctypes.byref(p),
                                   hout.data_ptr(), buf.data_ptr(), need, stream.cuda_stream)
        if st != 0:
            raise mb.MhlaError(st, "mhla_forward_host")

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    t1 = time.perf_counter()
    io = hq.numel() * hq.element_size()
    return {"value": w.units * w.n_tokens * steps / (t1 - t0), "unit": UNIT,
            "h2d_bytes_per_step": 3 * io + hmc.numel() * 4, "d2h_bytes_per_step": io,
            "steps": steps, "ms_per_step": (t1 - t0) * 1e3 / steps}


# ------------------------------------------------------------ backward

BWD_METRIC = "MHLA bwd tokens*heads/sec (dQ, dK, dV, dMc; d=64) and % of GB300 HBM/tensor roofline"
BWD_PHASES = ["recompute", "output", "mix", "mc", "summary"]
# phase -> (kernel name in ncu, source, engine that bounds it when not HBM)
BWD_PHASE_KERNEL = {
    "simt": {
        "recompute": ("simt_summary_kernel", "token_level_head_phi_gb300/csrc/simt.cu", "alu"),
        "output": ("bwd_output_kernel", "token_level_head_phi_gb300/csrc/backward.cu", "alu"),
        "mix": ("bwd_mix_kernel", "token_level_head_phi_gb300/csrc/backward.cu", "alu"),
        "mc": ("bwd_mc_kernel", "token_level_head_phi_gb300/csrc/backward.cu", "alu"),
        "summary": ("bwd_summary_kernel", "token_level_head_phi_gb300/csrc/backward.cu", "alu"),
    },
    "simt_causal": {
        "recompute": ("simt_summary_kernel", "token_level_head_phi_gb300/csrc/simt.cu", "alu"),
        "output": ("causal_bwd_fwd_kernel", "token_level_head_phi_gb300/csrc/simt_causal_bwd.cu", "alu"),
        "mix": ("bwd_mix_kernel", "token_level_head_phi_gb300/csrc/backward.cu", "alu"),
        "mc": ("bwd_mc_kernel", "token_level_head_phi_gb300/csrc/backward.cu", "alu"),
        "summary": ("bwd_summary_kernel", "token_level_head_phi_gb300/csrc/backward.cu", "alu"),
    },
    "tc": {
        "recompute": ("tc_summary_kernel", "token_level_head_phi_gb300/csrc/tc_summary.cu", "tensor"),
        "output": ("tc_bwd_output_kernel", "token_level_head_phi_gb300/csrc/tc_bwd_output.cu", "tensor"),
        "mix": ("tc_mix_kernel", "token_level_head_phi_gb300/csrc/tc_mix.cu", "tensor"),
        "mc": ("tc_bwd_mc_kernel", "token_level_head_phi_gb300/csrc/tc_bwd_mc.cu", "tensor"),
        "summary": ("tc_bwd_summary_kernel", "token_level_head_phi_gb300/csrc/tc_bwd_summary.cu", "tensor"),
    },
}
BWD_LAUNCHES = {"simt": 7, "simt_causal": 9, "tc": 10}


def simt_mc_reduce_launches(w, mc_heads):
    """1 when the CUDA-core dMc kernel splits its units over groups (then a
    reduce kernel follows): fewer tiles than about four CTAs per SM."""
    tiles = ((w.n_blocks + 63) // 64) ** 2 * mc_heads
    units = w.units if mc_heads == 1 else w.batch
    return int(min(-(-608 // tiles), units, 64) > 1)
FP32_LANES_PER_SM = 128  # FP32 FMA lanes per SM (4 partitions x 32)
SM_COUNT = 152


def bwd_phase_cost(w: wl.Workload, splits: int, causal: bool = False):
    """Compulsory bytes and dense FLOPs of each backward phase.  Records take
    4 bytes per entry on both paths (float32, or bf16 high + low planes); the
    FLOPs are those of the float32 contractions (the tensor cores run each
    split product three times).  Causal form: the in-block step reads Q, K, V,
    dO and the prefix records and writes dQ, and runs the per-token state
    products forwards and backwards (16 d^2 FLOPs per token); the summary
    step also reads the in-block parts of dK, dV (float32)."""
    el = 2 if w.dtype == "bf16" else 4
    U, N, d, M = w.units, w.n_tokens, w.head_dim, w.n_blocks
    R = d * d + 2 * d
    Q = M * splits
    io = U * N * d * el
    stack, mixed, mc = U * Q * R * 4, U * M * R * 4, 4 * M * M
    nd2, m2 = U * N * d * d, U * M * M * d * d
    cost = {
        "recompute": (2 * io + 2 * stack + mixed + mc, 2 * nd2 + 2 * U * M * Q * R),
        "output": (2 * io + mixed + io + stack, 6 * nd2),
        "mix": (stack + mixed + mc, 2 * U * M * Q * R),
        "mc": (2 * stack + mc, 2 * U * Q * Q * R),
        "summary": (2 * io + mixed + 2 * io, 4 * nd2),
    }
    if causal:
        cost["output"] = (5 * io + mixed, 16 * nd2)
        cost["summary"] = (2 * io + mixed + 2 * io + 2 * U * N * d * 4, 4 * nd2)
    return cost


def run_backward(args, w: wl.Workload, world: int, rank: int, local: int, dist):
    """One step = one mhla_backward over the workload (the forward summaries
    and mixing recomputed inside it), inputs and dO resident in HBM."""
    import torch
    import token_level_head_phi_gb300.binding as mb
    from token_level_head_phi_gb300 import build as mbuild

    if rank == 0 or world == 1:
        mbuild.build()
    if dist is not None:
        dist.barrier()
    mb.load()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    qn, kn, vn = wl.all_device_inputs(w)
    _, gn = wl.output_grad(w)

    def to_dev(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if w.dtype == "bf16":
            t = t.view(torch.bfloat16)
        return t.to(dev)

    q, k, v, g = to_dev(qn), to_dev(kn), to_dev(vn), to_dev(gn)
    del qn, kn, vn, gn
    if args.layout == "bnhd":
        q, k, v, g = (t.permute(0, 2, 1, 3).contiguous() for t in (q, k, v, g))
    if args.mc_per_head:
        mc = torch.from_numpy(np.stack([wl.make_mc(w.with_(seed=w.seed + 101 * h))
                                        for h in range(w.heads)]).astype(np.float32)).to(dev)
    else:
        mc = torch.from_numpy(wl.make_mc(w)).to(dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    dmc = torch.empty_like(mc)
    path = "tc" if (w.dtype == "bf16" and w.head_dim == 64 and args.variant != "simt") else "simt"
    if args.causal:
        path = "simt_causal"  # the causal form's gradients run on the CUDA cores
    variant = "auto" if path == "tc" else "simt"
    p = mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, w.dtype, args.feature_map, w.norm, variant,
                       bool(args.causal), args.layout, args.mc_per_head)
    splits = mb.mhla_plan(mb.make_params(w.batch, w.heads, w.head_dim, w.grid, w.block, w.dtype, args.feature_map, w.norm,
                                         "multipass" if path == "tc" else "simt")).summary_splits
    need = mb.mhla_backward_workspace_bytes(p)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    handle = stream.cuda_stream
    io_bytes = q.numel() * q.element_size()
    flush = None
    if io_bytes * 4 < 2 * L2_BYTES:
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        st = mb.mhla_backward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), mc.data_ptr(), g.data_ptr(), p,
                                  dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dmc.data_ptr(), ws.data_ptr(), need,
                                  handle)
        if st != 0:
            raise mb.MhlaError(st, "mhla_backward")

    for _ in range(args.warmup):
        if flush is not None:
            flush.zero_()
        step()
    torch.cuda.synchronize()
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local) if rank == 0 else None
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    t0 = time.time()
    start.record(stream)
    host_s = 0.0
    for i in range(K):
        if flush is not None:
            flush.zero_()
            step_ev[i][0].record(stream)
        h0 = time.perf_counter()
        step()
        host_s += time.perf_counter() - h0
        if flush is not None:
            step_ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop(t0, t1) if sampler else None
    total_ms = start.elapsed_time(end) if flush is None else sum(a.elapsed_time(b) for a, b in step_ev)

    KP = max(3, min(K, 20))
    ev_sets = [[torch.cuda.Event(enable_timing=True) for _ in range(mb.NUM_BWD_PHASE_EVENTS)] for _ in range(KP)]
    for i in range(KP):
        if flush is not None:
            flush.zero_()
        mb.mhla_set_backward_phase_events(ev_sets[i])
        step()
    mb.mhla_set_backward_phase_events(None)
    torch.cuda.synchronize()
    avg_phase = {ph: statistics.mean(evs[j].elapsed_time(evs[j + 1]) for evs in ev_sets)
                 for j, ph in enumerate(BWD_PHASES)}
    max_ms, value = job_throughput(total_ms, K, w.units * w.n_tokens, world, dist, dev)
    ms_per_step = max_ms / K

    hbm, tf_burst, tf_sust, peak_kind = load_peaks()
    cost = bwd_phase_cost(w, splits, bool(args.causal))
    dom = max(avg_phase, key=avg_phase.get)
    kname, ksrc, engine = BWD_PHASE_KERNEL[path][dom]
    nbytes, nflops = cost[dom]
    sec = avg_phase[dom] / 1e3
    sm_mhz = (clocks or {}).get("sm_max_mhz") or 2070.0
    alu_peak = SM_COUNT * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12  # TFLOP/s
    peak_flops = alu_peak if engine == "alu" else tf_sust
    if nbytes / (hbm * 1e9) >= nflops / (peak_flops * 1e12):
        roof = {"bound": "hbm", "achieved": nbytes / sec / 1e9, "peak": hbm, "unit": "GB/s",
                "peak_source": peak_kind}
    else:
        roof = {"bound": engine, "achieved": nflops / sec / 1e12, "peak": peak_flops, "unit": "TFLOP/s",
                "peak_source": ("fp32 FMA lanes x 2 x max SM clock: %d x %d x 2 x %.0f MHz"
                                % (SM_COUNT, FP32_LANES_PER_SM, sm_mhz)) if engine == "alu" else peak_kind}
    roof.update({"frac": roof["achieved"] / roof["peak"], "kernel": kname, "phase": dom, "traffic": None,
                 "algorithmic_bytes_per_launch": nbytes, "flops_per_launch": nflops, "avg_launch_ms": avg_phase[dom]})
    rb, rf = wl.backward_roofline_bytes(w), wl.backward_roofline_flops(w)
    t_hbm, t_tc = rb / (hbm * 1e9), rf / (tf_sust * 1e12)

    # end to end: pinned host Q, K, V, dO, Mc in, dQ, dK, dV, dMc out, every step
    hin = [t.cpu().pin_memory() for t in (q, k, v, g, mc)]
    hout = [torch.empty_like(t, device="cpu").pin_memory() for t in (dq, dk, dv, dmc)]
    dins, douts = (q, k, v, g, mc), (dq, dk, dv, dmc)

    def e2e_step():
        for d_, h_ in zip(dins, hin):
            d_.copy_(h_, non_blocking=True)
        step()
        for h_, d_ in zip(hout, douts):
            h_.copy_(d_, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    e2e_step()
    E = max(3, min(args.e2e_steps, 10))
    te0 = time.perf_counter()
    for _ in range(E):
        e2e_step()
    te1 = time.perf_counter()
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    return {
        "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if path == "tc" else "f32",
        "data": "synthetic (seeded normals, locality-biased Mc, seeded normal dO)",
        "config": dict(wl.describe(w), pass_="backward", feature_map=args.feature_map, layout=args.layout,
                       mc_per_head=bool(args.mc_per_head), causal=bool(args.causal),
                       input_dtype=w.dtype,
                       path="tensor cores (split bf16)" if path == "tc" else "CUDA cores (float32)",
                       l2="no flush: inputs exceed L2" if flush is None else "L2 flushed (256 MB write) between steps, outside per-step events",
                       parallelism=f"replicas{world}" if world > 1 else "single GPU"),
        "roofline": roof,
        "path_roofline": {"bytes": rb, "flops": rf, "t_hbm_us": t_hbm * 1e6, "t_tc_us": t_tc * 1e6,
                          "bound": "hbm" if t_hbm >= t_tc else "tensor",
                          "frac": max(t_hbm, t_tc) / (ms_per_step / 1e3)},
        "phase_ms": avg_phase,
        "gpu_launches": (BWD_LAUNCHES[path] + (0 if path == "tc" else simt_mc_reduce_launches(
            w, w.heads if args.mc_per_head else 1))) * K,
        "host_us_per_call": host_s / K * 1e6,
        "clocks": clocks,
        "e2e": {"value": w.units * w.n_tokens * E / (te1 - te0), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": E, "ms_per_step": (te1 - te0) * 1e3 / E},
    }


# ------------------------------------------------------ oracle baseline

ORACLE_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, {root!r})
from token_level_head_phi_gb300 import workloads as wl
from oracle import mhla_oracle as orc
from oracle import mhla_backward_oracle as orb
from oracle import mhla_causal_oracle as oca
from oracle import mhla_causal_backward_oracle as ocb
w = wl.WORKLOADS[{name!r}]
mc = wl.make_mc(w)
budget, max_units, per_step, backward, fmap = {budget}, {max_units}, {per_step}, {backward}, {fmap!r}
causal = {causal}
times = []
units = 0
t_all = time.perf_counter()
for step in range(max_units):
    u = step % w.units
    q, k, v = wl.head_inputs(w, u)
    g = wl.head_output_grad(w, u) if backward else None
    t0 = time.perf_counter()
    if backward:
        (ocb.mhla_causal_head_backward64 if causal else orb.mhla_head_backward64)(q, k, v, mc, w.grid, w.block, g,
                                                                                 fmap, w.norm)
    else:
        (oca.mhla_causal_head64 if causal else orc.mhla_head64)(q, k, v, mc, w.grid, w.block, fmap, w.norm)
    times.append(time.perf_counter() - t0)
    units += 1
    if not per_step and sum(times) >= budget:
        break
print(json.dumps({{"times": times, "units": units}}))
"""


def oracle_run(w: wl.Workload, budget_s: float, max_units: int, per_step: bool, backward: bool = False,
               fmap: str = "elu1", causal: bool = False, threads: int = 0):
    """Runs the oracle in a fresh process (BLAS threads = available cores,
    or `threads`)."""
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    if threads > 0:
        cores = threads
    env = dict(os.environ)
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(cores)
    code = ORACLE_SNIPPET.format(root=ROOT, name=w.name, budget=budget_s, max_units=max_units, per_step=per_step,
                               backward=backward, fmap=fmap, causal=causal)
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=1800)
    if res.returncode != 0:
        raise RuntimeError(f"oracle run failed: {res.stderr[-2000:]}")
    d = json.loads(res.stdout.strip().splitlines()[-1])
    return d["times"], d["units"], cores


def cpu_baseline(w: wl.Workload, budget_s: float = 15.0, backward: bool = False, fmap: str = "elu1",
                 causal: bool = False):
    times, units, cores = oracle_run(w, budget_s, max_units=10 ** 6, per_step=False, backward=backward, fmap=fmap,
                                     causal=causal)
    total = sum(times)
    what = ("causal " if causal else "") + ("backward" if backward else "forward")
    # the same oracle on one BLAS thread, on a shorter sample
    t1, u1, _ = oracle_run(w, budget_s / 3, max_units=10 ** 6, per_step=False, backward=backward, fmap=fmap,
                           causal=causal, threads=1)
    return {"value": units * w.n_tokens / total, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{units} of {w.units} (batch, head) units of {w.name}, float64 NumPy {what} oracle, "
                      f"{total:.1f} s of CPU time; input generation excluded",
            "one_thread": {"value": u1 * w.n_tokens / sum(t1), "unit": UNIT, "cores": 1,
                           "sample": f"{u1} units, {sum(t1):.1f} s"}}


def run_reference(args, w: wl.Workload):
    """--impl reference: the float64 oracle, each step one (batch, head) unit."""
    K, W = args.steps, args.warmup
    backward = getattr(args, "pass_", "forward") == "backward"
    times, units, cores = oracle_run(w, 0.0, max_units=W + K, per_step=True, backward=backward,
                                     fmap=getattr(args, "feature_map", "elu1"), causal=bool(getattr(args, "causal", 0)))
    timed = times[W:W + K]
    total = sum(timed)
    value = K * w.n_tokens / total
    return {
        "impl": "reference", "metric": BWD_METRIC if backward else METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": K,
        "warmup": W, "ms_per_step": total * 1e3 / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded normals, locality-biased Mc)",
        "config": dict(wl.describe(w), feature_map=getattr(args, "feature_map", "elu1"), parallelism="host cores"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step one (batch, head) unit of {w.name} ({w.n_tokens} tokens)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=wl.BENCH_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--variant", default="auto", choices=["auto", "simt", "multipass", "fused"])
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other configurations (listed under per_config by default)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--pass", dest="pass_", default="forward", choices=["forward", "backward"])
    ap.add_argument("--feature-map", default="elu1", choices=["elu1", "relu", "exp"])
    ap.add_argument("--causal", action="store_true", help="block-ordered causal form (forward or backward)")
    ap.add_argument("--layout", default="bhnd", choices=["bhnd", "bnhd"], help="q/k/v/out memory layout")
    ap.add_argument("--mc-per-head", action="store_true", help="one mixing matrix per head")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_env()
    w = wl.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        return

    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    import torch
    if args.pass_ == "backward":
        result = run_backward(args, w, world, rank, local, dist)
        if rank == 0 and not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(w, backward=True, fmap=args.feature_map, causal=bool(args.causal))
        if rank == 0:
            print(json.dumps(result), flush=True)
        if dist is not None:
            dist.barrier()
            dist.destroy_process_group()
        return
    result, state = run_mine(args, w, world, rank, local, dist)
    result["e2e"] = run_e2e(w, state, args.e2e_steps)
    del state
    torch.cuda.empty_cache()
    if not args.no_per_config and args.workload == wl.BENCH_WORKLOAD:
        result["per_config"] = run_per_config(args, world, rank, local, dist)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, fmap=args.feature_map, causal=bool(args.causal))
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
