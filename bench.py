#!/usr/bin/env python
"""Benchmark of the routed-MoE layer (ds4moe) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one ds4moe_forward over one batch of the workload's synthetic tokens
(all of router, grouping, experts, shared expert and combine). The default
workload is decode batch 1 on the H=4096, E=384, top-6 layer; a rotating pool
of 64 tokens makes consecutive steps pick different experts, and L2 is flushed
(a 2x-L2 device write) between steps, outside the timed events.

Prints one JSON line. ``value`` is whole-job tokens/s with inputs resident in
HBM; ``e2e`` is the same metric through ds4moe_forward_host with pinned host
buffers (host->device copy of x and device->host copy of y inside each step).
``roofline`` is for the dominant kernel, timed live with CUDA events recorded
by the library on its stream. ``cpu_baseline`` times the CPU oracle on a
bounded sample of the same workload. ``--impl reference`` times that oracle
alone as the reference arm.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE-layer tokens/sec (decode T=1..8, prefill T=1024); % HBM / tensor roofline"
UNIT = "tokens/s"
POOL = 64


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode_t1",
                    choices=["decode_t1", "decode_t8", "batch_t64", "prefill_t1024", "prefill_t4096_zipf4", "tiny",
                             "prefill_profile", "decode_profile", "prefill_hot_profile", "batch_profile"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-steps", type=int, default=20)
    ap.add_argument("--headline-only", action="store_true",
                    help="with the default decode_t1 workload, skip the other full-size workloads")
    ap.add_argument("--crossover", action="store_true",
                    help="time the decode and the prefill path on the decode layer for T = 1..64 and print "
                         "one JSON line of the per-T medians (not a bench line)")
    ap.add_argument("--routed-format", default="q2", choices=["q2", "mx4", "vq12", "vq13"],
                    help="routed experts in the 2-bit format, in MXFP4 (Q8 activations) or VQ with 12/13-bit indices")
    ap.add_argument("--gains", type=int, default=0, choices=[0, 1, 2],
                    help="per-expert down-gain tables (sidecar, post-training) on every layer")
    return ap.parse_args()


# ---- algorithmic work --------------------------------------------------------

Q2_BPW = 84 / 256  # bytes per 2-bit weight
Q8_BPW = 34 / 32


GAIN_BPC = 17 / 32  # bytes per output channel of one down-gain table
BATCH_MERGE_MAX_T = 4  # the batch kernels run the shared expert's items in the same launch up to this T
MX4_BPW = 17 / 32  # bytes per MXFP4 weight
VQ_BITS = {"vq12": 12, "vq13": 13}  # index bits per 8 weights


def layer_bytes(shape, T, U, gains=0, fmt="q2"):
    """Bytes the layer must move per call: selected experts (and their down-gain
    blocks), shared expert, router, x in, y out."""
    H, I, E, Ish = shape.hidden, shape.inter, shape.n_experts, shape.shared_inter
    bpw = {"mx4": MX4_BPW, "vq12": 12 / 64, "vq13": 13 / 64}.get(fmt, Q2_BPW)
    return (U * 3 * H * I * bpw + gains * U * H * GAIN_BPC + 3 * H * Ish * Q8_BPW + 4 * E * H + 2 * T * H
            + 4 * T * H)


def layer_flops(shape, T):
    H, I, K, Ish, E = shape.hidden, shape.inter, shape.top_k, shape.shared_inter, shape.n_experts
    return T * (2 * K * 3 * H * I + 2 * 3 * H * Ish + 2 * E * H)


def kernel_bytes(name, shape, T, U, gains=0, fmt="q2"):
    """Algorithmic bytes of one launch of a library kernel (weights it must read plus its activations)."""
    H, I, E, K, Ish = shape.hidden, shape.inter, shape.n_experts, shape.top_k, shape.shared_inter
    P = T * K
    table = {
        "router_logits": 4 * E * H + 4 * T * H + 4 * T * E,
        "router_logits_tc": 2 * 3 * E * H + 2 * T * H + 4 * T * E,
        "prefill_gateup_q2": U * 2 * I * H * Q2_BPW + 2 * T * H + 2 * P * I,
        "prefill_down_q2": U * H * I * Q2_BPW + 2 * P * I + 4 * P * H,
        "prefill_gateup_q8": 2 * Ish * H * Q8_BPW + 2 * T * H + 2 * T * Ish,
        "prefill_down_q8": H * Ish * Q8_BPW + 2 * T * Ish + 4 * T * H,
        "combine": 4 * P * H + 4 * T * H + 4 * T * H + gains * U * H * GAIN_BPC,
        # batch path (each product over the distinct experts' 2-bit rows and the shared expert's
        # 8-bit rows): weights, activation rows in, results out
        "batch_gateup": U * 2 * I * H * Q2_BPW + 2 * T * H + 4 * P * I
        + (2 * Ish * H * Q8_BPW + 4 * T * Ish if T <= BATCH_MERGE_MAX_T else 0),
        "batch_down": U * H * I * Q2_BPW + 4 * P * I + 4 * P * H
        + (H * Ish * Q8_BPW + 4 * T * Ish + 4 * T * H if T <= BATCH_MERGE_MAX_T else 0),
        "batch_gateup_shared": 2 * Ish * H * Q8_BPW + 2 * T * H + 4 * T * Ish,
        "batch_down_shared": H * Ish * Q8_BPW + 4 * T * Ish + 4 * T * H,
        # one launch of the fused decode kernel does the whole layer for up to 8 tokens
        "decode_fused": layer_bytes(shape, T, U, gains),
        # MXFP4 experts: weights of the distinct experts, fp32 activation rows in, results out
        "mx4_gateup": U * 2 * I * H * MX4_BPW + 4 * T * H + 4 * P * I,
        "mx4_down": U * H * I * MX4_BPW + 4 * P * I + 4 * P * H,
        # MXFP4 prefill form: grouped GEMMs on the MXFP4 tile records, binary16 activation rows
        "prefill_gateup_mx4": U * 2 * I * H * MX4_BPW + 2 * T * H + 2 * P * I,
        "prefill_down_mx4": U * H * I * MX4_BPW + 2 * P * I + 4 * P * H,
        # VQ experts: index streams (+ bit planes) and row gains of the distinct experts
        "vq_gateup": U * 2 * I * H * VQ_BITS.get(fmt, 12) / 64 + U * 2 * I * 2 + 4 * T * H + 4 * P * I,
        "vq_down": U * H * I * VQ_BITS.get(fmt, 12) / 64 + U * H * 2 + 4 * P * I + 4 * P * H,
        # VQ tensor-core form: index bits (and plane), row gains, codebook, binary16 activation rows
        "prefill_gateup_vq": U * 2 * I * H * VQ_BITS.get(fmt, 12) / 64 + U * 2 * I * 2 + (8 << VQ_BITS.get(fmt, 12))
        + 2 * T * H + 2 * P * I,
        "prefill_down_vq": U * H * I * VQ_BITS.get(fmt, 12) / 64 + U * H * 2 + (8 << VQ_BITS.get(fmt, 12))
        + 2 * P * I + 4 * P * H,
    }
    return table.get(name)


# dram__bytes_read.sum + dram__bytes_write.sum per launch of the dominant
# kernel, from one ncu capture of this workload (summaries under profiles/),
# with the SHA-1 of the kernel's source file at capture time: the figure is
# reported only while that source is unchanged.
TRAFFIC = {
    ("prefill_gateup_q2", "prefill_t1024"): (2188350208, "prefill_gemm.cuh", "c4d8d4b85ae902ac97cf5595672432168c7c5ec7"),
    ("prefill_down_q2", "prefill_t1024"): (1174632192, "prefill_gemm.cuh", "c4d8d4b85ae902ac97cf5595672432168c7c5ec7"),
    # mean of the four Zipf layers' launches
    ("prefill_gateup_q2", "prefill_t4096_zipf4"): (2425953536, "prefill_gemm.cuh",
                                                   "c4d8d4b85ae902ac97cf5595672432168c7c5ec7"),
    # mean of two launches
    ("decode_fused", "decode_t1"): (83569152, "decode_fused.cuh", "e72c292f502930ae0475e19e48ff689409d3a399"),
    # one launch, a batch of the pool with about 46 distinct experts (the traffic follows the batch's experts)
    ("batch_gateup", "decode_t8"): (256490752, "batch_experts.cuh", "03b7b0fabb2eb84ea263c524d2264b2f9fa4a45c"),
    ("batch_gateup", "batch_t64"): (1363641344, "batch_experts.cuh", "03b7b0fabb2eb84ea263c524d2264b2f9fa4a45c"),
}


def kernel_traffic(name, workload, gains=0, fmt="q2"):
    """The recorded DRAM bytes per launch, for the plain 2-bit layer the capture ran on."""
    import hashlib
    rec = TRAFFIC.get((name, workload)) if gains == 0 and fmt == "q2" else None
    if rec is None:
        return None
    path = os.path.join(ROOT, "quantized_moe_expert_gb300", "csrc", rec[1])
    try:
        with open(path, "rb") as f:
            digest = hashlib.sha1(f.read()).hexdigest()
    except OSError:
        return None
    return rec[0] if digest == rec[2] else None


def kernel_flops(name, shape, T):
    """Tensor-core flops of one launch (dense contractions only)."""
    H, I, K, Ish, E = shape.hidden, shape.inter, shape.top_k, shape.shared_inter, shape.n_experts
    P = T * K
    table = {
        "router_logits_tc": 2 * T * E * 3 * H,
        "prefill_gateup_q2": 2 * P * 2 * I * H,
        "prefill_down_q2": 2 * P * H * I,
        "prefill_gateup_mx4": 2 * P * 2 * I * H,
        "prefill_down_mx4": 2 * P * H * I,
        "prefill_gateup_vq": 2 * P * 2 * I * H,
        "prefill_down_vq": 2 * P * H * I,
        "prefill_gateup_q8": 2 * T * 2 * Ish * H,
        "prefill_down_q8": 2 * T * H * Ish,
    }
    return table.get(name)


# ---- clocks --------------------------------------------------------------------

class ClockSampler:
    """SM clock and throttle reasons sampled during the timed region.

    Reads NVML through ctypes every 2 ms (read-only queries); falls back to
    `nvidia-smi -lms 100` when the NVML library cannot be loaded.
    """
    # clock event reason bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.sw_power_cap",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown"]

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.sm, self.mx, self.reasons = [], [], set()
        self.lines = []
        self.proc = None
        self.stop = threading.Event()
        self.thread = None
        self.nvml = self._nvml_handle()

    def _nvml_handle(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            if not self.gpu_id or lib.nvmlDeviceGetHandleByUUID(self.gpu_id.encode(), ctypes.byref(h)) != 0:
                return None
            get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            return lib, h, get_reasons
        except (OSError, AttributeError):
            return None

    def _poll_nvml(self):
        import ctypes
        lib, h, get_reasons = self.nvml
        clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.sm.append(float(clk.value))
                self.mx.append(float(mx.value))
            if get_reasons(h, ctypes.byref(rs)) == 0:
                for bit, name in self.REASONS.items():
                    if rs.value & bit:
                        self.reasons.add(name)
            self.stop.wait(0.002)

    def __enter__(self):
        if self.nvml:
            self.thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self.thread.start()
            return self
        cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        self.stop.set()
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = list(self.sm), list(self.mx), set(self.reasons)
        names = ["sw_power_cap", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvml" if self.nvml else "nvidia-smi"}


# ---- the workload ----------------------------------------------------------------

def workload_layers(name, gains=0, fmt="q2"):
    import synth
    wl = synth.WORKLOADS[name]
    kind = "vq" if fmt in VQ_BITS else fmt
    return wl, [synth.make_layer(wl.shape, s, zipf=wl.zipf, gains=gains, routed_format=kind,
                                 vq_bits=VQ_BITS.get(fmt, 12)) for s in wl.layer_seeds]


def workload_batches(name):
    """List of bf16 token batches (host uint16 [T, H]) cycled through by the steps."""
    import synth
    wl = synth.WORKLOADS[name]
    if name == "decode_t1":
        pool = synth.make_tokens(name, T=POOL)
        return [pool[i:i + 1] for i in range(POOL)]
    if name == "decode_t8":
        import synth as s
        H = wl.shape.hidden
        batches = []
        for b in range(POOL // 8):
            batches.append(np.stack([s.normal_bf16(H, s.token_seed("decode_t8", 8 * b + t), s.S_X)
                                     for t in range(8)]))
        return batches
    return [synth.make_tokens(name)]


def cpu_oracle_rate(name, layers, batches, budget_tokens=None, min_seconds=0.0):
    """Time the oracle on a bounded sample; returns (tokens/s, threads used, sample text, seconds).

    The sample is run again until min_seconds of CPU time have passed (whole passes)."""
    import oracle
    import synth
    wl = synth.WORKLOADS[name]
    cores = oracle.max_threads()
    if wl.tokens <= 8:
        n = budget_tokens or min(16, POOL if name == "decode_t1" else 16)
        flat = np.concatenate(batches)[:n]
        sample = f"{len(flat)} tokens of the {name} pool through all {len(layers)} layer(s), oracle.forward"
    else:
        n = budget_tokens or 16
        flat = batches[0][:n]
        sample = f"first {len(flat)} of the {wl.tokens} tokens through all {len(layers)} layer(s), oracle.forward"
    t0 = time.perf_counter()
    passes = 0
    while True:
        for layer in layers:
            oracle.forward(wl.shape, layer, np.ascontiguousarray(flat), act=mx4_act(layer, wl.tokens))
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    if passes > 1:
        sample += f", {passes} passes"
    return passes * len(flat) / dt, cores, sample, dt


def mx4_act(layer, T):
    """The activation arithmetic of an MXFP4 layer's expert products at T tokens
    (the library's automatic form: Q8 for decode, FP4 for prefill); None for
    other layers."""
    if layer.get("routed_format") != "mx4":
        return None
    import quantized_moe_expert_gb300 as ds4
    return "mx4" if T >= ds4.AUTO_MX4_PREFILL_MIN_T else "q8"


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(value, world, device=None):
    """The maximum of a per-rank float over all ranks (the slowest rank's time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, tokens_per_rank_step, steps, total_ms):
    """Whole-job tokens/s: every rank processes its own batches (weak scaling)."""
    return world * tokens_per_rank_step * steps / (total_ms / 1000.0)


def run_reference(args, world, rank):
    import synth
    if rank != 0:
        return
    wl, layers = workload_layers(args.workload, args.gains, args.routed_format)
    batches = workload_batches(args.workload)
    times = []
    n_tok = None
    for i in range(args.warmup + args.steps):
        rate, cores, sample, dt = cpu_oracle_rate(args.workload, layers, batches)
        n_tok = rate * dt
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = n_tok * len(times) / total
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total / len(times),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_config(wl, args.workload, None, args.gains, args.routed_format),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def workload_config(wl, name, l2_note, gains=0, fmt="q2"):
    s = wl.shape
    cfg = {"workload": name, "description": wl.description, "hidden": s.hidden, "inter": s.inter,
           "n_experts": s.n_experts, "top_k": s.top_k, "shared_inter": s.shared_inter,
           "tokens_per_step": wl.tokens, "layers_per_step": wl.n_layers,
           "weights": {"mx4": "routed MXFP4 17B/32 blocks on " + (
                           "FP4 activations (tensor cores)" if mx4_act({"routed_format": "mx4"}, wl.tokens) == "mx4"
                           else "Q8 activations"),
                       "vq12": "routed VQ, 12-bit indices per 8 weights into a 4096 x 8 E4M3 codebook, f16 row gains",
                       "vq13": "routed VQ, 13-bit indices per 8 weights into an 8192 x 8 E4M3 codebook, f16 row gains"
                       }.get(fmt, "routed 2-bit 84B/256 blocks") + ", shared 8-bit 34B/32 blocks, router fp32"}
    if gains:
        cfg["down_gain_tables"] = gains
        cfg["weights"] += f", {gains} down-gain table(s) of 17B/32-channel FP4 blocks"
    if l2_note:
        cfg["l2"] = l2_note
    return cfg


CROSSOVER_T = (1, 2, 4, 6, 8, 9, 12, 16, 24, 32, 48, 64)


def run_crossover(args):
    """Every path (decode, prefill, and batch up to its token limit) on the
    H=4096, E=384 decode layer for each T of CROSSOVER_T:
    tokens ~N(0,1) bf16 from seed SEED_BASE + 0x100 + T, L2 flushed before every
    call, median of 15 calls after 3 warm-up calls (CUDA events)."""
    import torch

    import quantized_moe_expert_gb300 as ds4
    import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fmt = args.routed_format
    wl, layers = workload_layers("decode_t1", args.gains, fmt)
    shape = wl.shape
    stream = torch.cuda.current_stream(dev)
    T_list = CROSSOVER_T if fmt == "q2" else tuple(sorted(set(CROSSOVER_T + (3, 5, 128, 256))))
    moe = make_handles(layers[:1], shape, dev, max(T_list), fmt, stream)[0]
    flush = torch.empty(2 * torch.cuda.get_device_properties(dev).L2_cache_size, dtype=torch.uint8, device=dev)
    gpu_id = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    gpu_id = ("GPU-" + str(gpu_id)) if gpu_id is not None and not str(gpu_id).startswith("GPU-") else gpu_id
    rows = {}
    with ClockSampler(gpu_id) as clk:
        for T in T_list:
            xb = synth.normal_bf16(T * shape.hidden, synth.SEED_BASE + 0x100 + T, synth.S_X)
            x = torch.from_numpy(xb.reshape(T, shape.hidden).view(np.int16)).to(dev)
            y = torch.empty((T, shape.hidden), dtype=torch.float32, device=dev)
            idx, _, _, _ = moe.route(x)
            row = {"unique_experts": int(torch.unique(idx).numel())}
            paths = [("decode_us", ds4.PATH_DECODE), ("prefill_us", ds4.PATH_PREFILL)]
            if T <= ds4.BATCH_MAX_T and fmt == "q2":
                paths.append(("batch_us", ds4.PATH_BATCH))
            for name, path in paths:
                ts = []
                for it in range(18):
                    flush.zero_()
                    a = torch.cuda.Event(enable_timing=True)
                    b = torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    ds4.ds4moe_forward_path(moe.handle, x, T, path, y)
                    b.record(stream)
                    torch.cuda.synchronize()
                    if it >= 3:
                        ts.append(1000.0 * a.elapsed_time(b))
                row[name] = float(np.median(ts))
            row["fastest"] = min((row[n], n[:-3]) for n, _ in paths)[1]
            rows[T] = row
    if moe.status() != 0:
        raise RuntimeError("device error during the crossover sweep")
    moe.close()
    print(json.dumps({"crossover": rows, "routed_format": fmt, "auto_decode_max_t": ds4.AUTO_DECODE_MAX_T,
                      "auto_batch_max_t": ds4.AUTO_BATCH_MAX_T, "auto_mx4_prefill_min_t": ds4.AUTO_MX4_PREFILL_MIN_T,
                      "config": workload_config(wl, "decode_t1", "flushed before every call", args.gains),
                      "clocks": clk.summary()}))


# The full-size configurations besides the headline, measured in the same run
# (same L2 flush between steps): workload -> (steps, warmup, profiled steps,
# end-to-end steps, seconds of CPU baseline).
SIDE_WORKLOADS = {
    "decode_t8": (20, 3, 10, 10, 5.0),
    "batch_t64": (10, 3, 5, 5, 5.0),
    "prefill_t1024": (8, 3, 4, 4, 5.0),
    "prefill_t4096_zipf4": (4, 3, 2, 2, 5.0),
}


def peaks_table():
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peaks = {}
    if os.path.exists(pk_path):
        with open(pk_path) as f:
            peaks = json.load(f)
    return peaks


def measure(ctx, name, handles, layers, steps, warmup, profile_steps, e2e_steps, cpu_seconds):
    """Time one workload on its handles: the step loop (device-resident inputs),
    the per-kernel pass, the end-to-end pass through host memory and the CPU
    baseline. Returns the fields of a bench line."""
    import torch

    import quantized_moe_expert_gb300 as ds4
    import synth

    args, world, rank, dev, stream, flush, gpu_id = (ctx[k] for k in ("args", "world", "rank", "dev", "stream",
                                                                        "flush", "gpu_id"))
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    batches = workload_batches(name)
    T = wl.tokens
    xs = [torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(dev) for b in batches]
    y = torch.empty((T, shape.hidden), dtype=torch.float32, device=dev)

    def step(i):
        x = xs[i % len(xs)]
        for m in handles:
            ds4.ds4moe_forward(m.handle, x, T, y)

    # distinct experts per batch, from the library's own routing
    uniq = []
    for x in xs[:min(len(xs), 64)]:
        uniq.append([len(torch.unique(m.route(x)[0])) for m in handles])
    U_mean = float(np.mean(uniq))

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for i in range(warmup):
        flush.zero_()
        step(i)
    torch.cuda.synchronize()
    launches_per_step = handles[0].stats().kernel_count * len(handles)
    path_taken = handles[0].stats().path

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id) as clk:
        for i in range(steps):
            flush.zero_()
            evs[i][0].record(stream)
            step(warmup + i)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = job_rate(world, T, steps, total_ms)
    ms_per_step = total_ms / steps

    # per-kernel device times, recorded by the library around each launch
    for m in handles:
        ds4.ds4moe_profile(m.handle, True)
    for i in range(profile_steps):
        flush.zero_()
        step(i)
    ktimes = {}
    for m in handles:
        for kname, (n, ms) in ds4.ds4moe_profile_read(m.handle).items():
            a = ktimes.setdefault(kname, [0, 0.0])
            a[0] += n
            a[1] += ms
        ds4.ds4moe_profile(m.handle, False)
    dom = max(ktimes, key=lambda k: ktimes[k][1])
    if launches_per_step == 1:
        # the step is this one launch: its time is the timed region's own
        dom_avg_ms = ms_per_step
        time_source = "timed region (the step is one launch of this kernel)"
    else:
        dom_avg_ms = ktimes[dom][1] / ktimes[dom][0]
        time_source = ("per-launch CUDA events in a pass of %d steps right after the timed region; the profiled "
                       "kernels sum to %.4f ms per step against %.4f ms timed" % (
                           profile_steps, sum(v[1] for v in ktimes.values()) / profile_steps, ms_per_step))
    dom_bytes = kernel_bytes(dom, shape, T, U_mean, args.gains, args.routed_format)
    peaks = peaks_table()
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    tf_peak = peaks.get("bf16_tflops", 1900.0)
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"
    roofline = None
    dom_flops = kernel_flops(dom, shape, T)
    if dom_bytes is not None:
        sec = dom_avg_ms / 1000.0
        t_hbm = dom_bytes / (hbm_peak * 1e9)
        t_tc = dom_flops / (tf_peak * 1e12) if dom_flops else 0.0
        traffic = kernel_traffic(dom, name, args.gains, args.routed_format)
        if t_tc > t_hbm:
            ach = dom_flops / sec / 1e12
            roofline = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": tf_peak, "unit": "TFLOP/s",
                        "frac": ach / tf_peak, "traffic": traffic, "peak_source": peak_src + " bf16 burst",
                        "flops_per_launch": dom_flops, "bytes_per_launch": dom_bytes,
                        "hbm_frac": dom_bytes / sec / 1e9 / hbm_peak, "avg_launch_us": 1000 * dom_avg_ms,
                        "kernel_time_source": time_source}
        else:
            ach = dom_bytes / sec / 1e9
            roofline = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                        "frac": ach / hbm_peak, "traffic": traffic, "peak_source": peak_src,
                        "bytes_per_launch": dom_bytes, "avg_launch_us": 1000 * dom_avg_ms,
                        "kernel_time_source": time_source}
            if dom_flops:
                roofline["flops_per_launch"] = dom_flops
                roofline["tensor_frac"] = dom_flops / sec / 1e12 / tf_peak
    lay_bytes = layer_bytes(shape, T, U_mean, args.gains, args.routed_format) * len(handles)
    layer_gbs = lay_bytes / (ms_per_step / 1000.0) / 1e9
    lay_flops = layer_flops(shape, T) * len(handles)
    layer_tf = lay_flops / (ms_per_step / 1000) / 1e12

    # end to end through host memory
    xh = [torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).pin_memory() for b in batches]
    yh = torch.empty((T, shape.hidden), dtype=torch.float32).pin_memory()
    e2e_ms = []
    for i in range(warmup + e2e_steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for m in handles:
            ds4.ds4moe_forward_host(m.handle, xh[i % len(xh)].data_ptr(), T, yh.data_ptr())
        b.record(stream)
        b.synchronize()
        if i >= warmup:
            e2e_ms.append(a.elapsed_time(b))
    e2e_total = max_over_ranks(sum(e2e_ms), world, dev)
    e2e = {"value": job_rate(world, T, e2e_steps, e2e_total), "unit": UNIT, "steps": e2e_steps,
           "h2d_bytes_per_step": 2 * T * shape.hidden * len(handles),
           "d2h_bytes_per_step": 4 * T * shape.hidden * len(handles)}
    for m in handles:
        if m.status() != 0:
            raise RuntimeError("device error reported by the library")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # whole passes over a bounded sample until cpu_seconds of CPU work
        rate, cores, sample, dt = cpu_oracle_rate(name, layers, batches, min_seconds=cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cores, "host_cores": os.cpu_count(), "kind": "oracle",
               "sample": sample, "seconds": dt}
    l2_note = "flushed between steps: %d MiB device write outside the timed events" % (
        flush.numel() // (1 << 20))
    return {"value": value, "ms_per_step": ms_per_step, "steps": steps, "warmup": warmup,
            # decode and batch paths: exact products, fp32 accumulation; prefill: bf16 tensor cores
            "dtype": "bf16" if path_taken == ds4.PATH_PREFILL else "f32",
            "config": workload_config(wl, name, l2_note, args.gains, args.routed_format),
            "roofline": roofline,
            "layer_roofline": {"bound": "tensor" if lay_flops / (tf_peak * 1e12) > lay_bytes / (hbm_peak * 1e9)
                               else "hbm",
                               "bytes_per_step": lay_bytes, "achieved_gbs": layer_gbs,
                               "frac_hbm": layer_gbs / hbm_peak, "tflops": layer_tf, "frac_tensor": layer_tf / tf_peak,
                               "unique_experts_mean": U_mean},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * steps,
            "clocks": clk.summary(),
            "kernels_us": {k: round(1000 * v[1] / v[0], 2) for k, v in ktimes.items()}}


def make_handles(layers, shape, dev, max_tokens, fmt, stream):
    import torch

    import quantized_moe_expert_gb300 as ds4
    handles = []
    for layer in layers:
        w = {k: (None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(dev)) for k, v in layer.items()
             if v is None or isinstance(v, np.ndarray)}
        flags = {"mx4": ds4.FLAG_MXFP4, "vq12": ds4.FLAG_VQ12, "vq13": ds4.FLAG_VQ13}.get(fmt, 0)
        handles.append(ds4.MoELayer(shape, w, max_tokens=max_tokens, flags=flags))
        del w
    torch.cuda.empty_cache()
    for m in handles:
        m.set_stream(stream)
    return handles


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.crossover:
        if rank == 0:
            run_crossover(args)
        return

    import torch

    import synth

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    gpu_id = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    gpu_id = ("GPU-" + str(gpu_id)) if gpu_id is not None and not str(gpu_id).startswith("GPU-") else gpu_id
    ctx = {"args": args, "world": world, "rank": rank, "dev": dev, "stream": stream, "flush": flush,
           "gpu_id": gpu_id}

    head = args.workload
    side = [w for w in SIDE_WORKLOADS if head == "decode_t1" and not args.headline_only]
    wl, layers = workload_layers(head, args.gains, args.routed_format)
    # decode_t1, decode_t8 and prefill_t1024 share one layer: one handle sized for all of them
    shares = [w for w in side if synth.WORKLOADS[w].layer_seeds == wl.layer_seeds]
    max_t = max([wl.tokens, 8] + [synth.WORKLOADS[w].tokens for w in shares])
    handles = make_handles(layers, wl.shape, dev, max_t, args.routed_format, stream)
    out = measure(ctx, head, handles, layers, args.steps, args.warmup, args.profile_steps, args.steps, 10.0)
    extra = {}
    for name in side:
        steps, warmup, prof, e2e_steps, cpu_s = SIDE_WORKLOADS[name]
        if name in shares:
            extra[name] = measure(ctx, name, handles, layers, steps, warmup, prof, e2e_steps, cpu_s)
            continue
        for m in handles:
            m.close()
        handles = []
        torch.cuda.empty_cache()
        swl, slayers = workload_layers(name, args.gains, args.routed_format)
        handles = make_handles(slayers, swl.shape, dev, swl.tokens, args.routed_format, stream)
        extra[name] = measure(ctx, name, handles, slayers, steps, warmup, prof, e2e_steps, cpu_s)
        del slayers
    for m in handles:
        m.close()

    if rank == 0:
        line = {"metric": METRIC, "value": out["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": out["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": out["dtype"], "data": "synthetic",
                "config": out["config"], "roofline": out["roofline"], "layer_roofline": out["layer_roofline"],
                "cpu_baseline": out["cpu_baseline"], "e2e": out["e2e"], "gpu_launches": out["gpu_launches"],
                "clocks": out["clocks"], "kernels_us": out["kernels_us"]}
        if extra:
            line["workloads"] = {k: dict(v, metric=METRIC, unit=UNIT, higher_is_better=True, vs_baseline=None)
                                 for k, v in extra.items()}
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
