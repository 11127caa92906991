#!/usr/bin/env python3
"""Throughput of the attention hot path on GB300, one JSON line on stdout.

One step is one pass of every step of the path over one batch of seeded
synthetic inputs, all on one CUDA stream:

* the YOLO C2PSA block: QKV [8, 512, 20, 20] fp16 -> psa_pack_qkv ->
  psa_fa2_forward (HEAD_DIM 32 on Q, K with V_lo and with V_hi, N = 400, one
  pass over the scores for both) -> psa_merge_attn_nchw -> [8, 256, 20, 20],
  three few-microsecond kernels replayed as one CUDA graph;
* attention forward + backward, bf16, B=2 H=16 (BH = 32), N_q = N_k = 8192,
  HEAD_DIM 128: fa2_forward, then fa2_backward_preprocess (the row sums D) and
  fa2_backward_passes (the dK/dV and dQ passes in one grid) - the two launches
  fa2_backward makes at this head size, called as stages so that each is timed.

``value`` = algorithmic FLOPs of a step / device time of a step, in TFLOP/s:
forward 4*BH*N_q*N_k*d, backward 2.5x the forward (recomputed products are not
counted), for both attention problems of the step.  Inputs are resident in HBM
when the timed region starts; the per-step working set (Q, K, V, dO, O, dQ, dK,
dV: 512 MiB) is larger than the 129 MB L2, so no flush is inserted.

``--impl reference`` times the float64 CPU oracle instead (on a bounded sample
of the same workload per step); it is a deliberately slow baseline.

Multi-GPU (torchrun, one process per GPU): each rank runs its own batch (weak
scaling, no collective on the data path); the step time is the maximum over
ranks and ``value`` counts the work of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from attention_fa2_forward_02_gb300 import synth  # noqa: E402

# ---------------------------------------------------------------------------- workload
BH, N, D = 32, 8192, 128            # B=2, H=16
PSA_B, PSA_NH, PSA_KD, PSA_H, PSA_W = 8, 4, 32, 20, 20
PSA_N = PSA_H * PSA_W
PSA_BH = PSA_B * PSA_NH
FWD_FLOPS = 4.0 * BH * N * N * D
BWD_FLOPS = 2.5 * FWD_FLOPS
PSA_FLOPS = 2 * 4.0 * PSA_BH * PSA_N * PSA_N * PSA_KD
STEP_FLOPS = FWD_FLOPS + BWD_FLOPS + PSA_FLOPS
# algorithmic FLOPs of each timed call: the backward's 10*d per (query, key) pair is
# S, dP, dV, dK (8*d, the key-tile pass) and dQ (2*d; the dQ pass's recomputed S and
# dP are not counted)
KERNEL_FLOPS = {"fa2_fwd": FWD_FLOPS, "fa2_bwd_passes": BWD_FLOPS}
KERNEL_SOURCES = {
    "fa2_fwd": ["fa2_fwd_tc.cu", "common.cuh"],
    "fa2_bwd_passes": ["fa2_bwd_tc.cu", "bwd_common.cuh", "common.cuh"],
}
LAUNCHES_PER_STEP = 6  # pack, fused PSA fwd (V_lo and V_hi), merge, fwd, bwd preprocess, bwd passes
WORKLOAD = ("C2PSA block (QKV [8,512,20,20] fp16, 4 heads, KEY_DIM 32) + attention fwd+bwd "
            "bf16 B=2 H=16 N=8192 HEAD_DIM=128")


def set_heads(bh: int):
    """Resize the attention problem to `bh` (batch*head) slices; 32 (B=2, H=16) is the headline workload.
    Smaller values serve profiler captures of the same complete step."""
    global BH, FWD_FLOPS, BWD_FLOPS, STEP_FLOPS, KERNEL_FLOPS, WORKLOAD
    BH = bh
    FWD_FLOPS = 4.0 * BH * N * N * D
    BWD_FLOPS = 2.5 * FWD_FLOPS
    STEP_FLOPS = FWD_FLOPS + BWD_FLOPS + PSA_FLOPS
    KERNEL_FLOPS = {"fa2_fwd": FWD_FLOPS, "fa2_bwd_passes": BWD_FLOPS}
    if bh != 32:
        WORKLOAD = WORKLOAD.replace("B=2 H=16", f"BH={bh}")
METRIC = "FA2 fwd+bwd TFLOP/s (bf16, B=2 H=16 N=8192 d=128, with the C2PSA pack/attention/merge block)"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16": p["bf16_tflops"], "bf16_sustained": p["bf16_tflops_sustained"],
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def env_rank():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                name = line.split(":", 1)[1].strip()
                if name and not name.isdigit():
                    vendor = next((ln.split(":", 1)[1].strip() for ln in out.splitlines()
                                   if ln.split(":")[0].strip() == "Vendor ID"), "")
                    return f"{vendor} {name}".strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 20 ms; only those stamped inside the timed region count.

    `begin()` and `end()` bracket the timed region on the host clock (the GPU work of the
    region runs between them: its launches follow begin() and end() follows the final
    synchronize). nvidia-smi stamps each sample with its local wall-clock time; the offset
    of that clock from the host's epoch time (its time zone, a whole number of quarter
    hours) is taken from when the samples arrive. A region shorter than the sampling
    interval may hold no sample: the record then says so and gives no clock. power.draw
    is an average over a window longer than a short region, so its maximum there
    understates the draw."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMED = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    INTERVAL_MS = 20

    def __init__(self, device_id: str, start: bool = True):
        self.lines = []  # (host time received, line)
        self.proc = None
        self.t_begin = self.t_end = None
        if not start:
            return
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", device_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def begin(self):
        self.t_begin = time.time()

    def end(self):
        self.t_end = time.time()

    def stop(self):
        if self.proc is None and not self.lines:
            return {"unavailable": "nvidia-smi not found"}
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)
        return self.summary()

    @staticmethod
    def _stamp(text):
        import datetime
        return datetime.datetime.strptime(text, "%Y/%m/%d %H:%M:%S.%f").timestamp()

    def summary(self):
        rows = []  # (received, stamped, sm, sm max, power, reasons)
        for received, line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append((received, self._stamp(f[0]), float(f[2]), float(f[3]), float(f[4]),
                             [n for n, v in zip(self.NAMED, f[6:10]) if v.lower() == "active"]))
            except ValueError:
                continue
        if not rows:
            return {"unavailable": "no samples"}
        offsets = sorted(r[0] - r[1] for r in rows)
        zone = round(offsets[len(offsets) // 2] / 900.0) * 900.0  # the stamps' time-zone offset
        t0 = self.t_begin if self.t_begin is not None else -math.inf
        t1 = self.t_end if self.t_end is not None else math.inf
        inside = [r for r in rows if t0 <= r[1] + zone <= t1]
        out = {"sm_max_mhz": max(r[3] for r in rows), "samples": len(inside), "samples_total": len(rows),
               "interval_ms": self.INTERVAL_MS, "region_s": (round(t1 - t0, 4) if self.t_begin is not None
                                                            and self.t_end is not None else None)}
        if not inside:
            out.update({"sm_mhz": None, "reasons": [], "power_w_max": None,
                        "note": "no sample fell inside the timed region (shorter than the sampling interval)"})
            return out
        out.update({"sm_mhz": statistics.median(r[2] for r in inside), "sm_min_mhz": min(r[2] for r in inside),
                    "reasons": sorted({n for r in inside for n in r[5]}),
                    "power_w_max": max(r[4] for r in inside)})
        return out


# ---------------------------------------------------------------------------- ncu traffic
def _sources_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "attention_fa2_forward_02_gb300", "csrc", n), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel source is unchanged since."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_bf16_d128_n8192.md")
    if BH != 32:
        return None
    try:
        text = open(path).read()
    except OSError:
        return None
    m_t = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    m_h = re.search(r"source_hash:\s*([0-9a-f]+)", text)
    if not m_t or not m_h or m_h.group(1) != _sources_hash(KERNEL_SOURCES[kernel]):
        return None
    return float(m_t.group(1))


# ---------------------------------------------------------------------------- inputs
def make_inputs(seed):
    q = synth.tensor("bench/attn/q", (BH, N, D), "bf16", seed=seed)
    k = synth.tensor("bench/attn/k", (BH, N, D), "bf16", seed=seed)
    v = synth.tensor("bench/attn/v", (BH, N, D), "bf16", seed=seed)
    d_o = synth.tensor("bench/attn/do", (BH, N, D), "bf16", seed=seed)
    qkv = synth.tensor("bench/c2psa/qkv", (PSA_B, PSA_NH * 4 * PSA_KD, PSA_H, PSA_W), "f16", seed=seed)
    return q, k, v, d_o, qkv


def cpu_oracle_sample(q, k, v, d_o, budget_s: float, block_rows: int = 1024):
    """The float64 oracle (as it stands) on blocks of query rows of head 0 until the budget is spent."""
    from oracle import attention as A
    w = synth.widen
    kb, vb = w(k[0:1], "bf16"), w(v[0:1], "bf16")
    scale = 1 / math.sqrt(D)
    t0 = time.perf_counter()
    blocks = 0
    head = 0
    while True:
        r0 = (blocks * block_rows) % N
        if blocks and r0 == 0:  # next head once a head's query rows are all done
            head = (head + 1) % BH
            kb, vb = w(k[head:head + 1], "bf16"), w(v[head:head + 1], "bf16")
        A.backward(w(q[head:head + 1, r0:r0 + block_rows], "bf16"), kb, vb,
                   w(d_o[head:head + 1, r0:r0 + block_rows], "bf16"), scale)
        blocks += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    flops = 3.5 * 4.0 * blocks * block_rows * N * D
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": host_cores(), "cpu_model": cpu_model(),
            "kind": "oracle", "sample": f"{blocks} block(s) of {block_rows} query rows x {N} keys (HEAD_DIM {D}, {head + 1} head(s)): "
                      f"forward+backward in float64 numpy ({dt:.1f} s); FLOPs counted as for the GPU step"}


# ---------------------------------------------------------------------------- reference arm
def run_reference(args):
    rank, world, _ = env_rank()
    if rank != 0:
        return 0
    from oracle import attention as A
    block = 256
    heads = {n: synth.normal(synth.BASE_SEED, f"bench/attn/{n}", N * D).reshape(1, N, D) for n in ("q", "k", "v", "do")}
    w = {n: synth.widen(synth.to_storage(x, "bf16"), "bf16") for n, x in heads.items()}
    scale = 1 / math.sqrt(D)

    def ref_step(i):
        r0 = (i * block) % N
        A.backward(w["q"][:, r0:r0 + block], w["k"], w["v"], w["do"][:, r0:r0 + block], scale)

    for i in range(args.warmup):
        ref_step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        ref_step(i)
    dt = time.perf_counter() - t0
    flops = 3.5 * 4.0 * block * N * D * args.steps
    value = flops / dt / 1e12
    sample = (f"each step: {block} query rows x {N} keys of one head (HEAD_DIM {D}), forward+backward in float64 "
              f"numpy; the C2PSA block is not sampled")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": host_cores(), "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- our arm
def reduce_max(x: float, dist=None, device=None) -> float:
    """The maximum of `x` over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, step_flops: float, ms_step: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own batch (weak scaling) in the max-over-ranks step time."""
    return world * step_flops / (ms_step * 1e-3) / 1e12


def roofline_peak(elapsed_ms: float, clocks: dict):
    """Which measured peak the roofline fraction divides by, and the rule that chose it.

    The burst figure (a cuBLAS GEMM timed alone, at full clock) fits a timed region shorter
    than a second or one whose SM clock stayed at its maximum; the sustained figure (the same
    GEMM looped for seconds under the power cap, at a lower clock) fits a long region that
    ran below the maximum clock."""
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    at_max = sm is not None and smax is not None and sm >= 0.99 * smax
    if elapsed_ms < 1000.0:
        return "burst", f"timed region {elapsed_ms:.0f} ms < 1 s: burst peak"
    if at_max:
        return "burst", f"median SM clock {sm:.0f} MHz = maximum {smax:.0f} MHz: burst peak"
    if sm is None:
        return "sustained", f"timed region {elapsed_ms:.0f} ms >= 1 s, no clock samples: sustained peak"
    return "sustained", (f"timed region {elapsed_ms:.0f} ms >= 1 s at median SM clock {sm:.0f} MHz "
                         f"< maximum {smax:.0f} MHz: sustained peak")


def run_ours(args):
    import torch
    rank, world, local = env_rank()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from attention_fa2_forward_02_gb300 import binding as B
    from attention_fa2_forward_02_gb300 import build as build_mod
    build_mod.build()
    B.library()

    q_h, k_h, v_h, do_h, qkv_h = make_inputs(synth.BASE_SEED + rank)

    def pinned(arr, dtype):
        if dtype == torch.bfloat16:
            t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
        else:
            t = torch.from_numpy(np.ascontiguousarray(arr))
        return t.pin_memory()

    host_in = {"q": pinned(q_h, torch.bfloat16), "k": pinned(k_h, torch.bfloat16), "v": pinned(v_h, torch.bfloat16),
               "do": pinned(do_h, torch.bfloat16), "qkv": pinned(qkv_h, torch.float16)}
    dev = torch.device("cuda", local)

    def alloc_set(fill: bool):
        """One set of device buffers for a step: inputs (copied from the host when `fill`) and outputs."""
        b = {n: (h.to(dev) if fill else torch.empty(h.shape, dtype=h.dtype, device=dev)) for n, h in host_in.items()}
        b["o"] = torch.empty_like(b["q"])
        b["lse"] = torch.empty((BH, N), dtype=torch.float32, device=dev)
        b["dq"], b["dk"], b["dv"] = torch.empty_like(b["q"]), torch.empty_like(b["k"]), torch.empty_like(b["v"])
        b["ws"] = torch.empty(B.fa2_backward_workspace_size(BH, N, N, D, B.DTYPE_BF16), dtype=torch.uint8, device=dev)
        b["packed"] = torch.empty((4, PSA_BH, PSA_N, PSA_KD), dtype=torch.float16, device=dev)
        b["o_lo"] = torch.empty((PSA_BH, PSA_N, PSA_KD), dtype=torch.float16, device=dev)
        b["o_hi"] = torch.empty_like(b["o_lo"])
        b["lse_lo"] = torch.empty((PSA_BH, PSA_N), dtype=torch.float32, device=dev)
        b["lse_hi"] = torch.empty_like(b["lse_lo"])
        b["merged"] = torch.empty((PSA_B, PSA_NH * 2 * PSA_KD, PSA_H, PSA_W), dtype=torch.float16, device=dev)
        return b

    sets = [alloc_set(True)]
    s128, s32 = 1 / math.sqrt(D), 1 / math.sqrt(PSA_KD)
    stream = torch.cuda.current_stream()

    def c2psa_calls(b):
        B.psa_pack_qkv(b["qkv"], b["packed"], PSA_NH)
        B.psa_fa2_forward(b["packed"], b["o_lo"], b["o_hi"], b["lse_lo"], s32)
        B.psa_merge_attn_nchw(b["o_lo"], b["o_hi"], b["merged"], PSA_NH)

    c2psa_graphs = {}

    def c2psa_graph(b):
        """The C2PSA block's three few-microsecond kernels as one CUDA graph per buffer set
        (captured before any timed region; a replay launches the same three kernels)."""
        if id(b) not in c2psa_graphs:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                c2psa_calls(b)  # first-call set-up outside the capture
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                c2psa_calls(b)
            c2psa_graphs[id(b)] = g
        return c2psa_graphs[id(b)]

    c2psa_graph(sets[0])

    def step(b=None, ev=None):
        b = b or sets[0]
        if ev is not None:
            ev[0].record(stream)
        c2psa_graph(b).replay()
        if ev is not None:
            ev[1].record(stream)
        B.fa2_forward(b["q"], b["k"], b["v"], b["o"], b["lse"], s128)
        if ev is not None:
            ev[2].record(stream)
        B.fa2_backward_preprocess(b["o"], b["do"], b["lse"], b["ws"], N)
        if ev is not None:
            ev[3].record(stream)
        B.fa2_backward_passes(b["q"], b["k"], b["v"], b["do"], b["ws"], b["dq"], b["dk"], b["dv"], s128)
        if ev is not None:
            ev[4].record(stream)

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(x: float) -> float:
        return reduce_max(x, dist, dev)

    for _ in range(args.warmup):
        step()
    B.fa2_device_status()
    barrier()

    # ------------------------------------------------------------------ timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    e_begin, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        dev_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:  # noqa: BLE001
        dev_id = str(local)
    sampler = ClockSampler(dev_id)
    time.sleep(0.3)
    sampler.begin()
    e_begin.record(stream)
    for s in range(args.steps):
        step(ev=evs[s])
    e_end.record(stream)
    torch.cuda.synchronize()
    sampler.end()
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(e_begin.elapsed_time(e_end))
    B.fa2_device_status()
    barrier()

    ms_step = elapsed_ms / args.steps

    # ------------------------------------------------------------------ end to end, host buffers
    # Every step copies its inputs in from pinned host memory and all of its
    # results (O, LSE, dQ, dK, dV, the merged C2PSA output) back.  Two buffer sets
    # and copy streams (two per direction: together they move more than one stream
    # per direction when both directions run at once) let the copies of steps s+2 (in)
    # and s (out) run while step s+1 computes.  Timed right after the main region,
    # before the component timings: later, after seconds of tensor-core load, the
    # power cap holds the SM clock lower, and the two numbers would compare clocks
    # rather than copies.
    e2e_steps = max(30, args.steps // 5)
    sets.append(alloc_set(False))
    c2psa_graph(sets[1])
    out_names = ["o", "lse", "dq", "dk", "dv", "merged"]
    host_out = {n: torch.empty(sets[0][n].shape, dtype=sets[0][n].dtype).pin_memory() for n in out_names}
    h2d = sum(h.numel() * h.element_size() for h in host_in.values())
    d2h = sum(h.numel() * h.element_size() for h in host_out.values())
    n_copy = 2
    in_lanes = [["q", "v", "qkv"], ["k", "do"]]                # tensors per host-to-device stream
    out_lanes = [["o", "dq", "lse"], ["dk", "dv", "merged"]]   # tensors per device-to-host stream
    h2d_streams = [torch.cuda.Stream() for _ in range(n_copy)]
    d2h_streams = [torch.cuda.Stream() for _ in range(n_copy)]
    in_ready = [[torch.cuda.Event() for _ in range(n_copy)] for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    out_read = [[torch.cuda.Event() for _ in range(n_copy)] for _ in range(2)]
    barrier()
    e2e_sampler = ClockSampler(dev_id)
    time.sleep(0.3)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_sampler.begin()
    a.record(stream)
    for hs in h2d_streams:
        hs.wait_event(a)

    def copy_in(i):
        for c, hs in enumerate(h2d_streams):
            with torch.cuda.stream(hs):
                for n in in_lanes[c]:
                    sets[i][n].copy_(host_in[n], non_blocking=True)
                in_ready[i][c].record(hs)

    copy_in(0)
    copy_in(1)
    for s in range(e2e_steps):
        i = s % 2
        for c in range(n_copy):
            stream.wait_event(in_ready[i][c])
            if s >= 2:
                stream.wait_event(out_read[i][c])  # outputs of step s-2 copied out before they are overwritten
        step(sets[i])
        computed[i].record(stream)
        for c, ds in enumerate(d2h_streams):
            ds.wait_event(computed[i])
            with torch.cuda.stream(ds):
                for n in out_lanes[c]:
                    host_out[n].copy_(sets[i][n], non_blocking=True)
                out_read[i][c].record(ds)
        if s + 2 < e2e_steps:
            for hs in h2d_streams:
                hs.wait_event(computed[i])  # step s has finished reading set i's inputs
            copy_in(i)
    for ds in d2h_streams:
        stream.wait_stream(ds)
    b.record(stream)
    torch.cuda.synchronize()
    e2e_sampler.end()
    e2e_clocks = e2e_sampler.stop()
    e2e_ms = max_over_ranks(a.elapsed_time(b)) / e2e_steps
    e2e = {"value": job_throughput(world, STEP_FLOPS, e2e_ms), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
           "copies": "pinned host buffers, H2D and D2H on two copy streams each, overlapping the neighbouring steps",
           "clocks": e2e_clocks}
    B.fa2_device_status()

    value = job_throughput(world, STEP_FLOPS, ms_step)
    names = ["c2psa_block", "fa2_fwd", "fa2_bwd_preprocess", "fa2_bwd_passes"]
    per = {n: statistics.fmean(evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(args.steps))
           for i, n in enumerate(names)}
    pk = peaks()
    dominant = max(KERNEL_FLOPS, key=lambda n: per[n])
    achieved = KERNEL_FLOPS[dominant] / (per[dominant] * 1e-3) / 1e12
    traffic = load_traffic(dominant)
    peak_kind, peak_rule = roofline_peak(elapsed_ms, clocks)
    peak = pk["bf16"] if peak_kind == "burst" else pk["bf16_sustained"]
    roofline = {"kernel": dominant, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "peak_kind": f"bf16 dense, {peak_kind} ({pk['source']})", "peak_rule": peak_rule,
                "frac_burst": achieved / pk["bf16"], "frac_sustained": achieved / pk["bf16_sustained"],
                "flops_per_launch": KERNEL_FLOPS[dominant]}
    bwd_ms = per["fa2_bwd_preprocess"] + per["fa2_bwd_passes"]
    components = {
        "fa2_fwd_ms": per["fa2_fwd"], "fa2_fwd_tflops": FWD_FLOPS / per["fa2_fwd"] / 1e9,
        "fa2_fwd_frac_burst_peak": FWD_FLOPS / per["fa2_fwd"] / 1e9 / pk["bf16"],
        "fa2_bwd_ms": bwd_ms, "fa2_bwd_tflops": BWD_FLOPS / bwd_ms / 1e9,
        "fa2_bwd_frac_burst_peak": BWD_FLOPS / bwd_ms / 1e9 / pk["bf16"],
        "fa2_bwd_preprocess_ms": per["fa2_bwd_preprocess"], "fa2_bwd_passes_ms": per["fa2_bwd_passes"],
        # the preprocess reads O, dO (16-bit) and LSE and writes D and LSE2 (float32): HBM-bound
        "fa2_bwd_preprocess_gbs": (2 * BH * N * D * 2 + BH * N * 4 + 2 * BH * N * 4) / (per["fa2_bwd_preprocess"] * 1e-3) / 1e9,
        "fa2_bwd_preprocess_frac_hbm": (2 * BH * N * D * 2 + BH * N * 4 + 2 * BH * N * 4) / (per["fa2_bwd_preprocess"] * 1e-3)
        / 1e9 / pk["hbm_gbs"],
        "c2psa_block_us": per["c2psa_block"] * 1e3,
        "peak_bf16_burst_tflops": pk["bf16"], "peak_source": pk["source"],
    }
    components.update(separate_passes(torch, B, sets[0], stream, s128))
    components.update(other_configs(torch, B, dev, pk))

    # ------------------------------------------------------------------ PSA pack / merge bandwidth
    components.update(psa_bandwidth(torch, B, dev, pk))
    components.update(c2psa_graph_timings(torch, B, dev))

    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world * BH, "seq_len": N, "head_dim": D,
                   "parallelism": f"replicas x{world} (independent batches per GPU, no collective)",
                   "l2": "inputs larger than L2 (512 MiB attention working set per step), no flush"},
        "components": components, "roofline": roofline, "e2e": e2e, "clocks": clocks,
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(q_h, k_h, v_h, do_h, budget_s=args.cpu_budget)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def separate_passes(torch, B, b, stream, scale, reps=50):
    """The backward's stages launched one by one (fa2_backward_preprocess, _dkdv, _dq), outside
    the timed region: how the one-grid fa2_backward_passes splits between the passes."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
    for r in range(reps):
        evs[r][0].record(stream)
        B.fa2_backward_preprocess(b["o"], b["do"], b["lse"], b["ws"], N)
        evs[r][1].record(stream)
        B.fa2_backward_dkdv(b["q"], b["k"], b["v"], b["do"], b["ws"], b["dk"], b["dv"], scale)
        evs[r][2].record(stream)
        B.fa2_backward_dq(b["q"], b["k"], b["v"], b["do"], b["ws"], b["dq"], scale)
        evs[r][3].record(stream)
    torch.cuda.synchronize()
    t = [statistics.fmean(evs[r][j].elapsed_time(evs[r][j + 1]) for r in range(reps)) for j in range(3)]
    B.fa2_device_status()
    return {"bwd_stages_separately_ms": sum(t), "bwd_preprocess_ms": t[0], "bwd_dkdv_pass_ms": t[1],
            "bwd_dq_pass_ms": t[2], "bwd_dkdv_pass_tflops": 0.8 * BWD_FLOPS / t[1] / 1e9}


def _batched_ms(torch, fn, reps=50, batch=8):
    """Device time of one fn() call: `batch` calls back to back between two events (the host
    queues them ahead of the GPU, so no launch cost falls inside), median over `reps` after
    10 warm-up calls."""
    for _ in range(10):
        fn()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(batch):
            fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b) / batch)
    return statistics.median(ts)


def other_configs(torch, B, dev, pk, reps=50):
    """The other attention shapes of the workload list, timed after the main region (seeded
    N(0,1) inputs; median of `reps` timings of 8 back-to-back calls each):
    forward B=4 H=16 N=4096 d=64, and cross attention B=1 H=32 N_q=1024 N_k=32768 d=128
    with K scaled by 8 (peaked rows), forward and backward; then two head counts too small
    to fill the SMs, cross attention either way at d=128: B*H=2, N_q=128, N_k=32768 (the
    forward's and the dQ pass's key ranges) and B*H=2, N_q=32768, N_k=128 (the dK/dV
    pass's query ranges)."""
    out = {}
    for tag, bh, nq, nk, d, kscale, with_bwd in (("fwd_b4h16_n4096_d64", 64, 4096, 4096, 64, 1.0, True),
                                                 ("cross_b1h32_nq1024_nk32768_d128", 32, 1024, 32768, 128, 8.0, True),
                                                 ("few_heads_bh2_nq128_nk32768_d128", 2, 128, 32768, 128, 1.0, True),
                                                 ("few_heads_bh2_nq32768_nk128_d128", 2, 32768, 128, 128, 1.0, True)):
        g = torch.Generator(device=dev).manual_seed(synth.BASE_SEED)
        q = torch.randn((bh, nq, d), device=dev, generator=g).to(torch.bfloat16)
        k = (kscale * torch.randn((bh, nk, d), device=dev, generator=g)).to(torch.bfloat16)
        v = torch.randn((bh, nk, d), device=dev, generator=g).to(torch.bfloat16)
        o = torch.empty_like(q)
        lse = torch.empty((bh, nq), dtype=torch.float32, device=dev)
        scale = 1 / math.sqrt(d)
        fl = 4.0 * bh * nq * nk * d

        def med(fn):
            return _batched_ms(torch, fn, reps)
        f_ms = med(lambda: B.fa2_forward(q, k, v, o, lse, scale))
        out[f"{tag}_fwd_ms"] = f_ms
        out[f"{tag}_fwd_tflops"] = fl / f_ms / 1e9
        out[f"{tag}_fwd_frac_burst_peak"] = fl / f_ms / 1e9 / pk["bf16"]
        if with_bwd:
            d_o = torch.randn((bh, nq, d), device=dev, generator=g).to(torch.bfloat16)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws = torch.empty(B.fa2_backward_workspace_size(bh, nq, nk, d, B.DTYPE_BF16), dtype=torch.uint8, device=dev)
            b_ms = med(lambda: B.fa2_backward(q, k, v, o, d_o, lse, dq, dk, dv, ws, scale))
            out[f"{tag}_bwd_ms"] = b_ms
            out[f"{tag}_bwd_tflops"] = 2.5 * fl / b_ms / 1e9
            out[f"{tag}_bwd_frac_burst_peak"] = 2.5 * fl / b_ms / 1e9 / pk["bf16"]
        B.fa2_device_status()
        del q, k, v, o, lse
    torch.cuda.empty_cache()
    return out


def c2psa_graph_timings(torch, B, dev):
    """GPU time of the C2PSA block (QKV [8, 512, 20, 20] fp16) as CUDA graphs, replayed 200 times:
    the forward (pack, fused attention, merge) and the training step (forward, then merge^T, fused
    attention backward, pack^T, and extract_v / extract_v^T for the V path).  At this size every
    kernel takes a few microseconds, so a graph removes the per-launch host cost."""
    nh, kd, n, bh = PSA_NH, PSA_KD, PSA_N, PSA_BH
    c = nh * 2 * kd
    qkv = torch.randn((PSA_B, nh * 4 * kd, PSA_H, PSA_W), device=dev).to(torch.float16)
    d_out = torch.randn((PSA_B, c, PSA_H, PSA_W), device=dev).to(torch.float16)
    d_vpe = torch.randn_like(d_out)
    packed = torch.empty((4, bh, n, kd), dtype=torch.float16, device=dev)
    o_lo, o_hi = torch.empty((bh, n, kd), dtype=torch.float16, device=dev), torch.empty((bh, n, kd), dtype=torch.float16, device=dev)
    lse = torch.empty((bh, n), dtype=torch.float32, device=dev)
    merged, v_nchw = torch.empty_like(d_out), torch.empty_like(d_out)
    d_lo, d_hi = torch.empty_like(o_lo), torch.empty_like(o_hi)
    d_packed = torch.empty_like(packed)
    d_qkv = torch.empty_like(qkv)
    ws = torch.empty(B.fa2_backward_workspace_size(bh, n, n, kd, B.DTYPE_F16), dtype=torch.uint8, device=dev)
    s32 = 1 / math.sqrt(kd)

    def fwd():
        B.psa_pack_qkv(qkv, packed, nh)
        B.psa_fa2_forward(packed, o_lo, o_hi, lse, s32)
        B.psa_merge_attn_nchw(o_lo, o_hi, merged, nh)

    def train():
        fwd()
        B.psa_extract_v_nchw(qkv, v_nchw, nh)
        B.psa_merge_attn_backward(d_out, d_lo, d_hi, nh)
        B.psa_fa2_backward(packed, o_lo, o_hi, d_lo, d_hi, lse, d_packed, ws, s32)
        B.psa_pack_qkv_backward(d_packed, d_qkv, nh)
        B.psa_extract_v_backward(d_vpe, d_qkv, nh)

    out = {}
    for name, fn, launches in (("c2psa_fwd_graph_us", fwd, 3), ("c2psa_train_graph_us", train, 8)):
        try:
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                for _ in range(3):
                    fn()  # warm-up outside capture: first-call set-up (smem limits, symbol lookups)
            torch.cuda.current_stream().wait_stream(side)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            for _ in range(5):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(200):
                g.replay()
            e1.record()
            torch.cuda.synchronize()
            out[name] = e0.elapsed_time(e1) / 200 * 1e3
            out[name.replace("_us", "_kernels")] = launches
        except Exception as exc:  # noqa: BLE001
            out[name] = f"unavailable: {type(exc).__name__}: {exc}"[:200]
    B.fa2_device_status()
    return out


def _graph_ms_per_call(torch, fn, calls=50, replays=20):
    """Device time of one fn() call: `calls` back-to-back calls captured in a CUDA graph,
    replayed `replays` times between two events (no per-launch host cost in the figure)."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(calls):
            fn()
    for _ in range(3):
        g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (calls * replays)


def psa_bandwidth(torch, B, dev, pk):
    """psa_pack_qkv / psa_merge_attn_nchw GB/s: at the C2PSA shape (3.3 MB per tensor,
    L2-resident; a CUDA graph of 50 back-to-back calls, so that the few-microsecond kernels
    and not the host's launch cost are timed) and at B=1024 (419 MB per tensor, larger than
    L2: every call reads from and writes to HBM; median of 50 timings of 4 back-to-back calls)."""
    out = {}
    for label, b in (("c2psa", PSA_B), ("hbm_b1024", 1024)):
        qkv = torch.randn((b, PSA_NH * 4 * PSA_KD, PSA_H, PSA_W), device=dev).to(torch.float16)
        packed = torch.empty((4, b * PSA_NH, PSA_N, PSA_KD), dtype=torch.float16, device=dev)
        merged = torch.empty((b, PSA_NH * 2 * PSA_KD, PSA_H, PSA_W), dtype=torch.float16, device=dev)
        calls = {"pack": lambda: B.psa_pack_qkv(qkv, packed, PSA_NH),
                 "merge": lambda: B.psa_merge_attn_nchw(packed[2], packed[3], merged, PSA_NH)}
        ms = {}
        if label == "c2psa":
            for name, fn in calls.items():
                ms[name] = _graph_ms_per_call(torch, fn)
        else:
            for name, fn in calls.items():
                ms[name] = _batched_ms(torch, fn, reps=50, batch=4)
        nbytes = {"pack": 2 * qkv.numel() * 2, "merge": 2 * merged.numel() * 2}
        for name in ("pack", "merge"):
            out[f"psa_{name}_{label}_gbs"] = nbytes[name] / (ms[name] * 1e-3) / 1e9
            if label != "c2psa":
                out[f"psa_{name}_{label}_frac_hbm"] = out[f"psa_{name}_{label}_gbs"] / pk["hbm_gbs"]
        del qkv, packed, merged
    B.fa2_device_status()
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--bh", type=int, default=32, help="attention batch*heads (32 = B=2 H=16, the headline workload)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    set_heads(args.bh)
    return run_reference(args) if args.impl == "reference" else run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
