"""Benchmark of the NVFP4 weight path on one GB300 (or N replicas).

One step = one pass of every operation of the path over the Qwen2.5-7B-shaped
decode workload (MLP up 18944 x 3584 and down 3584 x 18944, bf16 weights
~N(0, 0.02^2) with 0.1% outliers x20, LoRA r = 32, noise sigma 5e-4):
  1. quantise both weight matrices with a dynamic (amax) tensor scale;
  2. decode GEMM Y = s_t X' deq(W)^T + s (X' A^T) B^T for M = 1, 4, 8, 16 on
     both matrices (8 GEMMs), FP32 output;
  3. scale-only update (round trained block-scale parameters to E4M3) for
     both matrices.
Inputs are resident in HBM before the timed region; the GEMMs read quantised
weights from a ring of replicas (>4x L2 in total) so that no GEMM reads
codes another operation just wrote to L2, and the bf16 weights (272 MB) are
larger than L2.

value  = algorithmic bytes of the step / device time of the step (GB/s).
e2e    = the same through the public API with pinned host inputs copied in
         and the outputs copied back inside the timed region.
--impl reference times the CPU oracle on a bounded sample of the same step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MS = (1, 4, 8, 16)
R_LORA = 32
SIGMA = 5e-4
LORA_SCALE = 2.0
UP = (18944, 3584)
DOWN = (3584, 18944)
WORKLOAD = "qwen2.5-7b-mlp-decode"


# ----------------------------------------------------------------- byte counts
def quant_bytes(N, K):
    return 2.5625 * N * K + 4


def gemm_bytes(M, N, K, r):
    return N * K * 0.5625 + 2 * M * K + 4 * M * N + 2 * r * K + 2 * N * r + 4 * K + 4


def gemm_flops(M, N, K, r):
    return 2.0 * M * N * K + 2.0 * M * r * (K + N)


def round_bytes(N, K):
    return 5.0 * N * K / 16 + 4


def step_bytes():
    b = sum(quant_bytes(*s) for s in (UP, DOWN))
    b += sum(gemm_bytes(M, *s, R_LORA) for M in MS for s in (UP, DOWN))
    b += sum(round_bytes(*s) for s in (UP, DOWN))
    return b


# ----------------------------------------------------------------- helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


# The sources each profiled kernel is built from: a committed DRAM-traffic
# figure counts only while none of them has changed since it was taken.
KERNEL_SOURCES = {
    "decode_stream": ("gemm_stream.cu", "common.cuh", "sm100.cuh", "internal.h"),
    "quantize_fused": ("quantize.cu", "common.cuh", "internal.h"),
}


def source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_weight_only_02_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def traffic_record(kernel):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    rec = d.get(kernel)
    if not rec or kernel not in KERNEL_SOURCES or rec.get("source_hash") != source_hash(kernel):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- ranks
def max_over_ranks(torch, dist, ms, device, world):
    """The slowest rank's time: every rank gets the maximum (one all-reduce)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, bytes_per_step, ms_per_step):
    """Whole-job throughput in GB/s: every rank moves bytes_per_step per step."""
    return world * bytes_per_step / (ms_per_step * 1e-3) / 1e9


# ----------------------------------------------------------------- GPU arm
class Workload:
    def __init__(self, torch, nv, synth, device, replicas):
        self.torch = torch
        self.nv = nv
        dev = device
        t = torch

        def to_dev(bits):
            return t.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(t.bfloat16).to(dev)

        self.host = {}
        self.w = {}
        self.lora = {}
        self.z = {}
        self.x = {}
        for name, shape, seed in (("up", UP, 0), ("down", DOWN, 100)):
            wb = synth.normal_weight(shape, 0.02, seed, outlier_frac=1e-3, outlier_mult=20.0)
            a, b = synth.lora_pair(shape[0], shape[1], R_LORA, 0.01, seed + 2)
            z = synth.noise_vector(shape[1], SIGMA, seed + 3)
            self.host[name] = (wb, a, b, z)
            self.w[name] = to_dev(wb)
            self.lora[name] = (to_dev(a), to_dev(b))
            self.z[name] = t.from_numpy(z).to(dev)
            for M in MS:
                self.x[(name, M)] = to_dev(synth.activations(M, shape[1], seed + 10 + M))
        self.ws = nv.new_workspace(max(nv.nvfp4_workspace_bytes(16, *s, R_LORA) for s in (UP, DOWN)), dev)
        # outputs and workspace of the projection lists (32 up + 32 down per list)
        self.ylist = {(n, M, k): t.empty((M, (UP if n == "up" else DOWN)[0]), dtype=t.float32, device=dev)
                      for n in ("up", "down") for M in MS for k in range(32)}
        # replicas of the quantised weights for the GEMMs
        self.rep = []
        for i in range(replicas):
            self.rep.append({n: nv.quantize(self.w[n], workspace=self.ws) for n in ("up", "down")})
        q0 = self.rep[0]
        ents = [(self.x[(n, 16)], q0[n].codes, q0[n].scales, q0[n].tensor_scale, *self.lora[n], LORA_SCALE,
                 self.z[n], self.ylist[(n, 16, k)]) for k in range(32) for n in ("up", "down")]
        self.wsl = nv.new_workspace(nv.nvfp4_gemm_list_workspace_bytes(ents), dev)
        self.y = {(n, M): t.empty((M, (UP if n == "up" else DOWN)[0]), dtype=t.float32, device=dev)
                  for n in ("up", "down") for M in MS}
        # trained block-scale parameters for the scale-only update
        self.param = {}
        for n in ("up", "down"):
            q = self.rep[0][n]
            dec = q.scales.view(t.float8_e4m3fn).float()
            g = t.Generator(device="cpu").manual_seed(7)
            jitter = (t.rand(dec.shape, generator=g) * 0.2 - 0.1).to(dev)
            self.param[n] = (dec * q.tensor_scale * (1 + jitter)).contiguous()
        self.new_scales = {n: t.empty_like(self.rep[0][n].scales) for n in ("up", "down")}
        self.qbuf = {n: (t.empty_like(self.rep[0][n].codes), t.empty_like(self.rep[0][n].scales),
                         t.zeros(1, dtype=t.float32, device=dev)) for n in ("up", "down")}
        # kernels per call and 16-token group: two for either decode GEMM path
        # (activation preparation, then the GEMM); quantiser and scale update one each
        per_gemm = {"decode_stream": 2, "decode_registers": 2}
        self.launches_per_step = 2 + 2 + sum(
            per_gemm[nv.gemm_kernel(M, *shape, R_LORA)] * ((M + 15) // 16) for M in MS for shape in (UP, DOWN))

    def op_quantize(self, frozen=False):
        for n in ("up", "down"):
            codes, scales, ts = self.qbuf[n]
            if frozen:  # the tensor scale of the resident replica, used as given
                ts = self.rep[0][n].tensor_scale
            self.nv.nvfp4_quantize(self.w[n], codes, scales, ts, frozen, self.ws)

    def op_gemm(self, M, i):
        R = len(self.rep)
        for j, n in enumerate(("up", "down")):
            q = self.rep[(i * 2 + j) % R][n]
            a, b = self.lora[n]
            self.nv.nvfp4_w4a16_lora_gemm(self.x[(n, M)], q.codes, q.scales, q.tensor_scale, a, b,
                                          LORA_SCALE, self.z[n], self.y[(n, M)], self.ws)

    def op_gemm_list(self, M, i, L=64):
        """One projection list: the up and down weights of L/2 consecutive
        replicas from replica i on (independent projections, one token count)."""
        R = len(self.rep)
        ents = []
        for k in range(L // 2):
            for n in ("up", "down"):
                q = self.rep[(i + k) % R][n]
                a, b = self.lora[n]
                ents.append((self.x[(n, M)], q.codes, q.scales, q.tensor_scale, a, b, LORA_SCALE, self.z[n],
                             self.ylist[(n, M, k)]))
        self.nv.nvfp4_w4a16_lora_gemm_list(ents, self.wsl)

    def op_round(self):
        for n in ("up", "down"):
            q = self.rep[0][n]
            self.nv.nvfp4_round_scales(self.param[n], q.tensor_scale, self.new_scales[n], self.ws)

    def step(self, i, ev=None):
        """One pass of the path.  ev: optional dict of (start, end) event lists
        per kernel kind for per-launch timing."""
        nv, t = self.nv, self.torch

        def timed(kind, fn):
            if ev is None:
                fn()
                return
            s = t.cuda.Event(enable_timing=True)
            e = t.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            ev.setdefault(kind, []).append((s, e))

        for n in ("up", "down"):
            codes, scales, ts = self.qbuf[n]
            timed("quantize", lambda: nv.nvfp4_quantize(self.w[n], codes, scales, ts, False, self.ws))
        R = len(self.rep)
        j = 0
        for M in MS:
            for n in ("up", "down"):
                q = self.rep[(i * 8 + j) % R][n]
                j += 1
                a, b = self.lora[n]
                timed(f"gemm_M{M}", lambda: nv.nvfp4_w4a16_lora_gemm(
                    self.x[(n, M)], q.codes, q.scales, q.tensor_scale, a, b, LORA_SCALE, self.z[n],
                    self.y[(n, M)], self.ws))
        for n in ("up", "down"):
            q = self.rep[0][n]
            timed("round_scales", lambda: nv.nvfp4_round_scales(self.param[n], q.tensor_scale,
                                                                self.new_scales[n], self.ws))


def capture(torch, fn):
    """CUDA graph of fn() (None if capture is not possible here)."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            fn()  # warm path on the capture stream
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=side):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        return g
    except Exception as exc:  # noqa: BLE001 - report and fall back to eager launches
        print(f"graph capture unavailable: {exc}", file=sys.stderr)
        return None


def time_replays(torch, runs, reps):
    """Mean device time (ms) of runs[i % len(runs)]() over reps calls."""
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for i in range(reps):
        runs[i % len(runs)]()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from nvfp4_weight_only_02_gb300 import binding as nv
    from nvfp4_weight_only_02_gb300 import synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    nv.load()
    R = 9
    wl = Workload(torch, nv, synth, dev, replicas=R)
    torch.cuda.synchronize()
    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()
    st = nv.nvfp4_get_device_status(wl.ws)
    if st != nv.OK:
        raise RuntimeError(f"device status after warm-up: {nv.status_string(st)}")

    # one graph per replica-rotation index: step i replays graph i % R
    graphs = None if args.eager else [capture(torch, lambda i=i: wl.step(i)) for i in range(R)]
    if graphs is not None and any(g is None for g in graphs):
        graphs = None
    runs = [g.replay for g in graphs] if graphs else [lambda i=i: wl.step(i) for i in range(R)]
    for i in range(args.warmup):
        runs[i % R]()
    torch.cuda.synchronize()

    props = torch.cuda.get_device_properties(dev)
    uuid = "GPU-" + str(props.uuid) if not str(props.uuid).startswith("GPU-") else str(props.uuid)
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)

    # timed region: K steps, device time by events on the launch stream
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(args.steps):
        runs[i % R]()
    end.record()
    torch.cuda.synchronize()
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(torch, dist, total_ms, dev, world)
    clocks = sampler.stop()

    # per-operation device times: each operation kind repeated over the whole
    # replica ring in one graph (back to back, as the calls of a decode step
    # run), time per call
    def op_time(fn_of_i, calls_per_i):
        seq = lambda: [fn_of_i(i) for i in range(R)]
        g = capture(torch, seq) if graphs else None
        run = g.replay if g is not None else seq
        reps = max(3, args.steps // 4)
        return time_replays(torch, [run], reps) / (R * calls_per_i)

    kb = {}
    kb["quantize"] = op_time(lambda i: wl.op_quantize(), 2)
    kb["quantize_frozen"] = op_time(lambda i: wl.op_quantize(frozen=True), 2)
    for M in MS:
        kb[f"gemm_M{M}"] = op_time(lambda i, M=M: wl.op_gemm(M, i), 2)
    for M in MS:
        kb[f"gemm_list_M{M}"] = op_time(lambda i, M=M: wl.op_gemm_list(M, i), 64)
    kb["round_scales"] = op_time(lambda i: wl.op_round(), 2)
    st = nv.nvfp4_get_device_status(wl.ws)
    if st != nv.OK:
        raise RuntimeError(f"device status after timing: {nv.status_string(st)}")

    # end-to-end: pinned host inputs in, outputs back, through the public API
    e2e = run_e2e(torch, nv, wl, dev, args)

    bytes_step = step_bytes()
    ms_step = total_ms / args.steps
    value = job_value(world, bytes_step, ms_step)
    peak_hbm, peak_tf, peak_kind = load_peaks()

    # roofline of the dominant operation kind (time per step)
    gemm_ms = sum(kb[f"gemm_M{M}"] for M in MS) * 2
    quant_ms = kb["quantize"] * 2
    if gemm_ms >= quant_ms:
        alg = sum(gemm_bytes(M, *s, R_LORA) for M in MS for s in (UP, DOWN)) / (2 * len(MS))
        dur = gemm_ms / (2 * len(MS)) * 1e-3
        kern, tkey = "decode_gemm", "decode_stream"
    else:
        alg = sum(quant_bytes(*s) for s in (UP, DOWN)) / 2
        dur = kb["quantize"] * 1e-3
        kern, tkey = "quantize", "quantize_fused"
    achieved = alg / dur / 1e9
    roof = {"kernel": kern, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak_hbm,
            "peak_source": peak_kind, "unit": "GB/s", "frac": round(achieved / peak_hbm, 4),
            "traffic": traffic_record(tkey), "alg_bytes_per_launch": alg,
            "timing": "CUDA events around graph replays of the operation (all of its kernels)"}

    per_kernel = {}
    for M in MS:
        b = sum(gemm_bytes(M, *s, R_LORA) for s in (UP, DOWN)) / 2
        f = sum(gemm_flops(M, *s, R_LORA) for s in (UP, DOWN)) / 2
        us = kb[f"gemm_M{M}"] * 1e3
        per_kernel[f"gemm_M{M}"] = {"mean_us": round(us, 2), "GB/s": round(b / us / 1e3, 1),
                                    "TFLOP/s": round(f / us / 1e6, 2),
                                    "frac_hbm": round(b / us / 1e3 / peak_hbm, 4)}
    for M in MS:  # per projection, inside lists of 64 (nvfp4_w4a16_lora_gemm_list)
        b = sum(gemm_bytes(M, *s, R_LORA) for s in (UP, DOWN)) / 2
        us = kb[f"gemm_list_M{M}"] * 1e3
        per_kernel[f"gemm_list_M{M}"] = {"mean_us_per_projection": round(us, 2), "GB/s": round(b / us / 1e3, 1),
                                         "frac_hbm": round(b / us / 1e3 / peak_hbm, 4),
                                         "projections_per_call": 64}
    qb = sum(quant_bytes(*s) for s in (UP, DOWN)) / 2
    for key in ("quantize", "quantize_frozen"):
        q_us = kb[key] * 1e3
        per_kernel[key] = {"mean_us": round(q_us, 2), "GB/s": round(qb / q_us / 1e3, 1),
                           "frac_hbm": round(qb / q_us / 1e3 / peak_hbm, 4)}
    r_us = kb["round_scales"] * 1e3
    rb = sum(round_bytes(*s) for s in (UP, DOWN)) / 2
    per_kernel["round_scales"] = {"mean_us": round(r_us, 2), "GB/s": round(rb / r_us / 1e3, 1)}

    line = {
        "metric": "nvfp4 weight path: quantise + W4A16+LoRA decode GEMM + scale update, algorithmic HBM bytes per second",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e2m1/e4m3 weights, bf16->f16 activations, f32 accumulate",
        "data": "synthetic (seeded Qwen2.5-7B-shaped weights and activations)",
        "config": {"workload": WORKLOAD, "layers": {"up": list(UP), "down": list(DOWN)}, "M": list(MS),
                   "lora_rank": R_LORA, "noise_sigma": SIGMA, "bytes_per_step": bytes_step,
                   "l2": "inputs larger than L2 (272 MB bf16 weights; GEMMs read a 9-replica ring, 0.69 GB)",
                   "launch": "CUDA graph replay of each step" if graphs else "eager launches",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "kernels": per_kernel, "clocks": clocks, "e2e": e2e,
        "gpu_launches": wl.launches_per_step * args.steps,
    }
    if rank == 0:
        if not args.no_configs:
            line["configs"] = {
                "single_layer_512x2048": run_single_layer(torch, nv, synth),
                "qwen2.5-32b-mlp-decode": run_qwen32b(torch, nv, synth, peak_hbm),
                "qwen2.5-7b-whole-stack-M8": run_whole_stack(torch, nv, synth, peak_hbm),
            }
        if not args.no_prefill:
            line["prefill"] = run_prefill_case(torch, nv, synth, peak_tf)
            line["dgrad"] = run_dgrad_case(torch, nv, synth, peak_tf)
            line["lora_grads"] = run_lora_grads_case(torch, nv, synth, peak_hbm)
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def graph_time_per_call(torch, seq, ncalls, reps=5):
    """Device time per call of seq() (ncalls calls) replayed as one CUDA graph."""
    g = capture(torch, seq)
    run = g.replay if g is not None else seq
    run()
    torch.cuda.synchronize()
    return time_replays(torch, [run], reps) / ncalls


def run_single_layer(torch, nv, synth):
    """The 512 x 2048 layer, 4 tokens, LoRA r = 16, s = 2, noise sigma 1e-2: its
    0.59 MB of weights stay in L2, so the call is launch-bound: microseconds
    per call, no roofline."""
    c = synth.single_layer_case()
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    q = nv.quantize(dev(c.w))
    M, K = c.x.shape
    N = c.w.shape[0]
    x, a, b = dev(c.x), dev(c.a), dev(c.b)
    z = torch.from_numpy(c.z).cuda()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    ws = nv.new_workspace(nv.nvfp4_workspace_bytes(M, N, K, 16))
    n = 64
    seq = lambda: [nv.nvfp4_w4a16_lora_gemm(x, q.codes, q.scales, q.tensor_scale, a, b, c.lora_scale, z, y, ws)
                   for _ in range(n)]
    ms = graph_time_per_call(torch, seq, n)
    return {"M": M, "N": N, "K": K, "lora_rank": 16, "us_per_call": round(ms * 1e3, 2),
            "kernel": nv.gemm_kernel(M, N, K, 16), "timing": f"graph of {n} back-to-back calls"}


def _student_t_device(torch, shape, scale, nu, seed):
    """Seeded Student-t(nu) * scale drawn on the device (normal / sqrt(chi2_nu / nu)),
    rounded to bf16; nu is an integer here (4)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    zz = torch.randn(shape, generator=g, device="cuda")
    chi2 = torch.zeros(shape, device="cuda")
    for _ in range(int(nu)):
        chi2 += torch.randn(shape, generator=g, device="cuda") ** 2
    return (zz / torch.sqrt(chi2 / nu) * scale).to(torch.bfloat16)


def run_qwen32b(torch, nv, synth, peak_hbm):
    """Qwen2.5-32B-shaped MLP decode: W 27648 x 5120 and 5120 x 27648 =
    0.02 Student-t(4), M in {1, 8}, LoRA r = 64, noise sigma 5e-4.  Each
    projection is quantised into 4 replicas (0.64 GB in all, > 2x L2) and the
    calls rotate through them, up and down alternating, in one graph."""
    r, R = 64, 4
    up, down = synth.QWEN32B_UP, synth.QWEN32B_DOWN
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    ws = nv.new_workspace(max(nv.nvfp4_workspace_bytes(16, *sh, r) for sh in (up, down)))
    reps, lora, zs = {}, {}, {}
    for name, sh, seed in (("up", up, 300), ("down", down, 400)):
        w = _student_t_device(torch, sh, 0.02, 4, seed)
        reps[name] = [nv.quantize(w, workspace=ws) for _ in range(R)]
        del w
        a, b = synth.lora_pair(sh[0], sh[1], r, 0.01, seed + 2)
        lora[name] = (dev(a), dev(b))
        zs[name] = torch.from_numpy(synth.noise_vector(sh[1], SIGMA, seed + 3)).cuda()
    out = {"layers": {"up": list(up), "down": list(down)}, "lora_rank": r, "replicas": R}
    for M in (1, 8):
        xs = {n: dev(synth.activations(M, sh[1], 500 + M)) for n, sh in (("up", up), ("down", down))}
        ys = {n: torch.empty((M, sh[0]), dtype=torch.float32, device="cuda") for n, sh in (("up", up), ("down", down))}

        def seq():
            for i in range(R):
                for n in ("up", "down"):
                    q = reps[n][i]
                    a, b = lora[n]
                    nv.nvfp4_w4a16_lora_gemm(xs[n], q.codes, q.scales, q.tensor_scale, a, b, LORA_SCALE, zs[n],
                                             ys[n], ws)
        ms = graph_time_per_call(torch, seq, 2 * R)
        nbytes = sum(gemm_bytes(M, *sh, r) for sh in (up, down)) / 2
        flops = sum(gemm_flops(M, *sh, r) for sh in (up, down)) / 2
        out[f"gemm_M{M}"] = {"mean_us": round(ms * 1e3, 2), "GB/s": round(nbytes / ms / 1e6, 1),
                             "TFLOP/s": round(flops / ms / 1e9, 2),
                             "frac_hbm": round(nbytes / ms / 1e6 / peak_hbm, 4),
                             "alg_bytes_per_call": nbytes}
        # the same 8 projections as one list call
        yl = {(n, i): torch.empty_like(ys[n]) for n in ("up", "down") for i in range(R)}  # no shared outputs
        ents = [(xs[n], reps[n][i].codes, reps[n][i].scales, reps[n][i].tensor_scale, *lora[n], LORA_SCALE, zs[n],
                 yl[(n, i)]) for i in range(R) for n in ("up", "down")]
        wsl = nv.new_workspace(nv.nvfp4_gemm_list_workspace_bytes(ents))
        ms_l = graph_time_per_call(torch, lambda: nv.nvfp4_w4a16_lora_gemm_list(ents, wsl), 2 * R)
        out[f"gemm_list_M{M}"] = {"mean_us_per_projection": round(ms_l * 1e3, 2),
                                  "GB/s": round(nbytes / ms_l / 1e6, 1),
                                  "frac_hbm": round(nbytes / ms_l / 1e6 / peak_hbm, 4),
                                  "projections_per_call": 2 * R}
        if nv.nvfp4_get_device_status(wsl) != nv.OK:
            raise RuntimeError("device status after the 32B list")
    st = nv.nvfp4_get_device_status(ws)
    if st != nv.OK:
        raise RuntimeError(f"device status after the 32B decode: {nv.status_string(st)}")
    return out


STACK_SHAPES = [("q", 3584, 3584), ("k", 512, 3584), ("v", 512, 3584), ("o", 3584, 3584),
                ("gate", 18944, 3584), ("up", 18944, 3584), ("down", 3584, 18944)]


def run_whole_stack(torch, nv, synth, peak_hbm, layers=28, M=8):
    """28 Qwen2.5-7B-shaped layers (196 matrices, bf16 ~N(0, 0.02^2) drawn on
    the device, seed 1000 * layer + matrix), each quantised with its own
    dynamic tensor scale (3.67 GB of codes and scales), then one decode sweep
    of the 196 W4A16 GEMMs with the same 8 tokens (no LoRA, no noise), as one
    graph.  The sweep reads 3.67 GB, far more than L2."""
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    ws = nv.new_workspace(max(nv.nvfp4_workspace_bytes(M, N, K, 0) for _, N, K in STACK_SHAPES))
    xs = {K: dev(synth.activations(M, K, 70 + K)) for K in (3584, 18944)}
    gen = torch.Generator(device="cuda")
    qs, ys = [], []
    qbytes = 0.0
    quant_ms = 0.0
    for layer in range(layers):
        for j, (name, N, K) in enumerate(STACK_SHAPES):
            gen.manual_seed(1000 * layer + j)
            w = (torch.randn((N, K), generator=gen, device="cuda") * 0.02).to(torch.bfloat16)
            codes = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
            scales = torch.empty((N, K // 16), dtype=torch.uint8, device="cuda")
            ts = torch.zeros(1, dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            nv.nvfp4_quantize(w, codes, scales, ts, False, ws)
            e1.record()
            torch.cuda.synchronize()
            quant_ms += e0.elapsed_time(e1)
            qbytes += quant_bytes(N, K)
            qs.append((nv.QuantizedWeight(codes, scales, ts), K))
            ys.append(torch.empty((M, N), dtype=torch.float32, device="cuda"))
            del w

    def seq():
        for (q, K), y in zip(qs, ys):
            nv.nvfp4_w4a16_lora_gemm(xs[K], q.codes, q.scales, q.tensor_scale, None, None, 0.0, None, y, ws)
    ms = graph_time_per_call(torch, seq, 1, reps=3)
    st = nv.nvfp4_get_device_status(ws)
    if st != nv.OK:
        raise RuntimeError(f"device status after the whole-stack sweep: {nv.status_string(st)}")

    # the same sweep grouped as a decoder layer's dependencies allow: q, k and
    # v read one input, so do gate and up; o and down wait for their inputs
    groups = [("q", "k", "v"), ("o",), ("gate", "up"), ("down",)]
    names = [n for n, _, _ in STACK_SHAPES]
    lists = []
    for layer in range(layers):
        for grp in groups:
            ents = []
            for n in grp:
                (q, K), y = qs[layer * len(STACK_SHAPES) + names.index(n)], ys[layer * len(STACK_SHAPES) + names.index(n)]
                ents.append((xs[K], q.codes, q.scales, q.tensor_scale, None, None, 0.0, None, y))
            lists.append(ents)
    wsl = nv.new_workspace(max(nv.nvfp4_gemm_list_workspace_bytes(e) for e in lists))

    def seq_lists():
        for ents in lists:
            nv.nvfp4_w4a16_lora_gemm_list(ents, wsl)
    ms_l = graph_time_per_call(torch, seq_lists, 1, reps=3)
    st = nv.nvfp4_get_device_status(wsl)
    if st != nv.OK:
        raise RuntimeError(f"device status after the layer-list sweep: {nv.status_string(st)}")

    # the sweep as it is defined here (196 GEMMs on synthetic inputs that do not
    # depend on one another): lists of 32, then of 64, in sweep order
    flat = [e for ents in lists for e in ents]
    ms_chunked = {}
    for L in (32, 64):
        chunks = [flat[i:i + L] for i in range(0, len(flat), L)]
        wsc = nv.new_workspace(max(nv.nvfp4_gemm_list_workspace_bytes(c) for c in chunks))

        def seq_chunks(chunks=chunks, wsc=wsc):
            for c in chunks:
                nv.nvfp4_w4a16_lora_gemm_list(c, wsc)
        ms_chunked[L] = graph_time_per_call(torch, seq_chunks, 1, reps=3)
        st = nv.nvfp4_get_device_status(wsc)
        if st != nv.OK:
            raise RuntimeError(f"device status after the {L}-list sweep: {nv.status_string(st)}")
        del wsc
    ms_32, ms_64 = ms_chunked[32], ms_chunked[64]
    nbytes = sum(gemm_bytes(M, N, K, 0) for _ in range(layers) for _, N, K in STACK_SHAPES)
    return {"layers": layers, "matrices": len(qs), "M": M,
            "sweep_ms": round(ms, 4), "sweep_GB/s": round(nbytes / ms / 1e6, 1),
            "sweep_frac_hbm": round(nbytes / ms / 1e6 / peak_hbm, 4), "sweep_alg_bytes": nbytes,
            "layer_lists_ms": round(ms_l, 4), "layer_lists_GB/s": round(nbytes / ms_l / 1e6, 1),
            "layer_lists_frac_hbm": round(nbytes / ms_l / 1e6 / peak_hbm, 4),
            "layer_lists": "per layer [q, k, v], [o], [gate, up], [down]: 112 list calls",
            "lists32_ms": round(ms_32, 4), "lists32_GB/s": round(nbytes / ms_32 / 1e6, 1),
            "lists32_frac_hbm": round(nbytes / ms_32 / 1e6 / peak_hbm, 4),
            "lists32": "the 196 independent GEMMs of the sweep as 7 list calls of up to 32, in sweep order",
            "lists64_ms": round(ms_64, 4), "lists64_GB/s": round(nbytes / ms_64 / 1e6, 1),
            "lists64_frac_hbm": round(nbytes / ms_64 / 1e6 / peak_hbm, 4),
            "lists64": "the same as 4 list calls of up to 64",
            "quantize_all_ms": round(quant_ms, 3), "quantize_GB/s": round(qbytes / quant_ms / 1e6, 1),
            "timing": "one graph each of the 196 GEMM calls, the 112 layer-list calls, the 7 32-lists and "
                      "the 4 64-lists; "
                      "quantisation timed per matrix (events)"}


def timed_op(torch, op, reps=10):
    """Device ms per call of op(), as CUDA-graph replays like every other line
    (eager launches when capture is not possible), and how it was timed."""
    op()
    torch.cuda.synchronize()
    g = capture(torch, op)
    if g is None:
        return time_replays(torch, [op], reps), f"eager, {reps} calls"
    return time_replays(torch, [g.replay], reps), f"CUDA-graph replays, {reps} calls"


def run_prefill_case(torch, nv, synth, peak_tf):
    """16384 tokens x 7B-shaped up projection (tensor-core path), bf16 output."""
    M, (N, K) = 16384, UP
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    w = dev(synth.normal_weight((N, K), 0.02, 0, outlier_frac=1e-3))
    ws = nv.new_workspace(nv.nvfp4_workspace_bytes(M, N, K, R_LORA))
    q = nv.quantize(w, workspace=ws)
    a, b = synth.lora_pair(N, K, R_LORA, 0.01, 2)
    a, b = dev(a), dev(b)
    z = torch.from_numpy(synth.noise_vector(K, SIGMA, 3)).cuda()
    x = dev(synth.activations(M, K, 10))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    op = lambda: nv.nvfp4_w4a16_lora_gemm(x, q.codes, q.scales, q.tensor_scale, a, b, LORA_SCALE, z, y, ws)
    ms, timing = timed_op(torch, op)
    f = gemm_flops(M, N, K, R_LORA)
    return {"workload": "16384 x 18944 x 3584 + LoRA r=32, bf16 out", "ms": round(ms, 3),
            "TFLOP/s": round(f / ms / 1e9, 1), "peak_bf16_tflops": peak_tf,
            "frac": round(f / ms / 1e9 / peak_tf, 4), "timing": timing}


def run_dgrad_case(torch, nv, synth, peak_tf):
    """Input gradient of the same layer for 16384 tokens: dY (16384 x 18944)
    -> dX (16384 x 3584), LoRA r=32, noise, bf16 out (tensor-core path)."""
    M, (N, K) = 16384, UP
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    w = dev(synth.normal_weight((N, K), 0.02, 0, outlier_frac=1e-3))
    q = nv.quantize(w)
    ws = nv.new_workspace(nv.nvfp4_dgrad_workspace_bytes(M, N, K, R_LORA))
    a, b = synth.lora_pair(N, K, R_LORA, 0.01, 2)
    a, b = dev(a), dev(b)
    z = torch.from_numpy(synth.noise_vector(K, SIGMA, 3)).cuda()
    dy = dev(synth.activations(M, N, 11, std=1e-3))
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    op = lambda: nv.nvfp4_w4a16_lora_gemm_dgrad(dy, q.codes, q.scales, q.tensor_scale, a, b, LORA_SCALE, z,
                                                dx, ws)
    ms, timing = timed_op(torch, op)
    st = nv.nvfp4_get_device_status(ws)
    if st != nv.OK:
        raise RuntimeError(nv.status_string(st))
    f = gemm_flops(M, N, K, R_LORA)
    return {"workload": "dX 16384 x 3584 from dY 16384 x 18944 (7B up, transposed) + LoRA r=32, bf16 out",
            "ms": round(ms, 3), "TFLOP/s": round(f / ms / 1e9, 1), "peak_bf16_tflops": peak_tf,
            "frac": round(f / ms / 1e9 / peak_tf, 4), "timing": timing}


def run_lora_grads_case(torch, nv, synth, peak_hbm):
    """LoRA factor gradients for 16384 tokens of the 7B up shape: dA (32 x 3584)
    and dB (18944 x 32) from X, z, dY, A, B.  HBM-bound: the algorithmic bytes
    are one read of X and of dY (and of A, B) plus the two outputs."""
    M, (N, K) = 16384, UP
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    a, b = synth.lora_pair(N, K, R_LORA, 0.01, 2)
    a, b = dev(a), dev(b)
    z = torch.from_numpy(synth.noise_vector(K, SIGMA, 3)).cuda()
    x = dev(synth.activations(M, K, 10))
    dy = dev(synth.activations(M, N, 11, std=1e-3))
    ga = torch.empty((R_LORA, K), dtype=torch.float32, device="cuda")
    gb = torch.empty((N, R_LORA), dtype=torch.float32, device="cuda")
    ws = nv.new_workspace(nv.nvfp4_lora_grads_workspace_bytes(M, N, K, R_LORA))
    op = lambda: nv.nvfp4_lora_grads(x, z, dy, a, b, LORA_SCALE, ga, gb, ws)
    ms, timing = timed_op(torch, op)
    nbytes = 2.0 * M * (K + N) + 2.0 * R_LORA * (K + N) + 4.0 * K + 4.0 * R_LORA * (K + N)
    return {"workload": "dA 32 x 3584, dB 18944 x 32 from X 16384 x 3584 (noise) and dY 16384 x 18944",
            "ms": round(ms, 3), "GB/s": round(nbytes / ms / 1e6, 1), "peak_hbm_gbs": peak_hbm,
            "frac": round(nbytes / ms / 1e6 / peak_hbm, 4), "timing": timing}


def run_e2e(torch, nv, wl, dev, args):
    """Public-API step with host buffers: pinned inputs copied in, outputs back."""
    t = torch
    host_in = {}
    for n in ("up", "down"):
        wb, a, b, z = wl.host[n]
        host_in[("w", n)] = t.from_numpy(wb.view(np.int16)).view(t.bfloat16).pin_memory()
        host_in[("p", n)] = wl.param[n].cpu().pin_memory()
        for M in MS:
            host_in[("x", n, M)] = wl.x[(n, M)].cpu().pin_memory()
        host_in[("z", n)] = wl.z[n].cpu().pin_memory()
        host_in[("a", n)] = wl.lora[n][0].cpu().pin_memory()
        host_in[("b", n)] = wl.lora[n][1].cpu().pin_memory()
    dev_in = {k: t.empty_like(v, device=dev) for k, v in host_in.items()}
    host_out = {k: t.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in wl.y.items()}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    steps = max(1, args.steps)

    # The copies go in on the timing stream in the order the work needs them
    # (the small operands, W up, W down, then the trained scales); a second
    # stream quantises and multiplies each matrix as soon as its weights have
    # arrived, so the compute hides under the copies of the next inputs.
    comp = t.cuda.Stream(device=dev)
    small = [k for k in host_in if k[0] not in ("w", "p")]

    def one(i):
        cur = t.cuda.current_stream()
        for k in small:
            dev_in[k].copy_(host_in[k], non_blocking=True)
        arrived = {}
        for n in ("up", "down"):
            dev_in[("w", n)].copy_(host_in[("w", n)], non_blocking=True)
            arrived[n] = t.cuda.Event()
            arrived[n].record(cur)
        for n in ("up", "down"):
            dev_in[("p", n)].copy_(host_in[("p", n)], non_blocking=True)
        arrived["p"] = t.cuda.Event()
        arrived["p"].record(cur)
        with t.cuda.stream(comp):
            for n in ("up", "down"):
                comp.wait_event(arrived[n])
                codes, scales, ts = wl.qbuf[n]
                nv.nvfp4_quantize(dev_in[("w", n)], codes, scales, ts, False, wl.ws)
                for M in MS:  # the GEMMs multiply by the weights just quantised
                    nv.nvfp4_w4a16_lora_gemm(dev_in[("x", n, M)], codes, scales, ts,
                                             dev_in[("a", n)], dev_in[("b", n)], LORA_SCALE,
                                             dev_in[("z", n)], wl.y[(n, M)], wl.ws)
            comp.wait_event(arrived["p"])
            for n in ("up", "down"):
                nv.nvfp4_round_scales(dev_in[("p", n)], wl.rep[0][n].tensor_scale, wl.new_scales[n], wl.ws)
            for k, v in wl.y.items():
                host_out[k].copy_(v, non_blocking=True)
        cur.wait_stream(comp)  # the next step's copies wait for this step's reads

    one(0)
    torch.cuda.synchronize()
    s = t.cuda.Event(enable_timing=True)
    e = t.cuda.Event(enable_timing=True)
    s.record()
    for i in range(steps):
        one(i + 1)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / steps
    # the host->device copies of a step alone, for comparison
    s.record()
    for _ in range(steps):
        for k, v in host_in.items():
            dev_in[k].copy_(v, non_blocking=True)
    e.record()
    torch.cuda.synchronize()
    copy_ms = s.elapsed_time(e) / steps
    return {"value": round(step_bytes() / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "h2d_GB/s_alone": round(h2d / (copy_ms * 1e-3) / 1e9, 1),
            "overlap": "each matrix is quantised and multiplied on a second stream once its weights "
                       "have arrived, while the next copies run"}


# ----------------------------------------------------------------- CPU oracle
def oracle_sample_inputs(synth, rows_up, rows_down):
    """Seeded inputs of the step restricted to a sample of weight rows."""
    out = []
    for shape, rows, seed in ((UP, rows_up, 0), (DOWN, rows_down, 100)):
        N, K = shape
        wb = synth.normal_weight((rows, K), 0.02, seed, outlier_frac=1e-3, outlier_mult=20.0)
        a, b = synth.lora_pair(rows, K, R_LORA, 0.01, seed + 2)
        z = synth.noise_vector(K, SIGMA, seed + 3)
        xs = {M: synth.activations(M, K, seed + 10 + M) for M in MS}
        out.append((rows, K, wb, a, b, z, xs))
    return out


def oracle_sample_step(oracle, inputs, nthreads):
    """The step on a row sample: quantise the sampled rows of each matrix,
    GEMM at every M on them, scale update on them.  Returns algorithmic bytes."""
    total = 0.0
    for rows, K, wb, a, b, z, xs in inputs:
        rc, codes, scales, st = oracle.quantize(wb, nthreads=nthreads)
        total += quant_bytes(rows, K)
        for M in MS:
            oracle.gemm(xs[M], codes, scales, st, a, b, LORA_SCALE, z, nthreads=nthreads)
            total += gemm_bytes(M, rows, K, R_LORA)
        param = (np.float32(st) * np.ones(scales.shape, np.float32)).astype(np.float32)
        oracle.round_scales(param, st)
        total += round_bytes(rows, K)
    return total


def nproc():
    """Cores this process may run on (what `nproc` prints)."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(seconds=15.0):
    import oracle
    from nvfp4_weight_only_02_gb300 import synth
    oracle.build()
    cores = nproc()
    # calibrate on a small sample, then size the sample to about `seconds`
    small = oracle_sample_inputs(synth, 64, 12)
    t0 = time.perf_counter()
    oracle_sample_step(oracle, small, cores)
    dt = time.perf_counter() - t0
    scale = max(1, int(seconds / max(dt, 1e-3)))
    rows_up, rows_down = min(UP[0], 64 * scale), min(DOWN[0], 12 * scale)
    inputs = oracle_sample_inputs(synth, rows_up, rows_down)
    t0 = time.perf_counter()
    b = oracle_sample_step(oracle, inputs, cores)
    dt = time.perf_counter() - t0
    return {"value": round(b / dt / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "hardware_concurrency": os.cpu_count(), "nproc": nproc(),
            "seconds": round(dt, 2),
            "sample": f"every step operation on {rows_up} of {UP[0]} up rows and {rows_down} of "
                      f"{DOWN[0]} down rows (all M, same K, r, noise)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from nvfp4_weight_only_02_gb300 import synth
    oracle.build()
    cores = nproc()
    rows_up, rows_down = 256, 48
    inputs = oracle_sample_inputs(synth, rows_up, rows_down)
    for _ in range(args.warmup):
        oracle_sample_step(oracle, inputs, cores)
    t0 = time.perf_counter()
    b = 0.0
    for _ in range(args.steps):
        b += oracle_sample_step(oracle, inputs, cores)
    dt = time.perf_counter() - t0
    value = b / dt / 1e9
    sample = (f"every step operation on {rows_up} of {UP[0]} up rows and {rows_down} of {DOWN[0]} "
              f"down rows per step")
    line = {
        "impl": "reference",
        "metric": "nvfp4 weight path: quantise + W4A16+LoRA decode GEMM + scale update, algorithmic HBM bytes per second",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded Qwen2.5-7B-shaped weights and activations)",
        "config": {"workload": WORKLOAD, "layers": {"up": list(UP), "down": list(DOWN)}, "M": list(MS),
                   "lora_rank": R_LORA, "noise_sigma": SIGMA},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "hardware_concurrency": os.cpu_count(), "nproc": nproc(), "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_kernel_case(case, reps):
    """One operation, repeated and timed with CUDA events: a small,
    self-contained target for ncu (quantize_up, gemm_up_M8, gemm_down_M16,
    prefill, ...)."""
    import torch

    from nvfp4_weight_only_02_gb300 import binding as nv
    from nvfp4_weight_only_02_gb300 import synth
    nv.load()
    if case.startswith("list_M"):  # one projection list: 8 up + 8 down replicas, r = 32, noise
        return run_list_case(torch, nv, synth, int(case[6:]), reps)
    if case.startswith("list64_M"):  # one launch of the longest list: 32 up + 32 down replicas
        return run_list_case(torch, nv, synth, int(case[8:]), reps, R=32)
    parts = case.split("_")
    kind = parts[0]
    which = parts[1] if len(parts) > 1 else "up"
    shape = UP if which == "up" else DOWN
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    wb = synth.normal_weight(shape, 0.02, 0, outlier_frac=1e-3, outlier_mult=20.0)
    w = dev(wb)
    M = int(parts[2][1:]) if kind == "gemm" else (16384 if kind in ("prefill", "dgrad", "loragrads") else 0)
    ws = nv.new_workspace(max(nv.nvfp4_workspace_bytes(max(M, 1), *shape, R_LORA),
                              nv.nvfp4_dgrad_workspace_bytes(max(M, 1), *shape, R_LORA)))
    q = nv.quantize(w, workspace=ws)
    if kind == "quantize":
        frozen = len(parts) > 2 and parts[2] == "frozen"
        op = lambda: nv.nvfp4_quantize(w, q.codes, q.scales, q.tensor_scale, frozen, ws)
        nbytes, flops = quant_bytes(*shape), 0.0
    elif kind == "loragrads":
        a, b = synth.lora_pair(shape[0], shape[1], R_LORA, 0.01, 2)
        a, b = dev(a), dev(b)
        z = torch.from_numpy(synth.noise_vector(shape[1], SIGMA, 3)).cuda()
        x = dev(synth.activations(M, shape[1], 10))
        dy = dev(synth.activations(M, shape[0], 11, std=1e-3))
        ga = torch.empty((R_LORA, shape[1]), dtype=torch.float32, device="cuda")
        gb = torch.empty((shape[0], R_LORA), dtype=torch.float32, device="cuda")
        ws = nv.new_workspace(nv.nvfp4_lora_grads_workspace_bytes(M, *shape, R_LORA))
        op = lambda: nv.nvfp4_lora_grads(x, z, dy, a, b, LORA_SCALE, ga, gb, ws)
        nbytes, flops = 2.0 * M * (shape[0] + shape[1]), 0.0
    elif kind == "dgrad":
        a, b = synth.lora_pair(shape[0], shape[1], R_LORA, 0.01, 2)
        a, b = dev(a), dev(b)
        z = torch.from_numpy(synth.noise_vector(shape[1], SIGMA, 3)).cuda()
        dy = dev(synth.activations(M, shape[0], 11, std=1e-3))
        dx = torch.empty((M, shape[1]), dtype=torch.bfloat16, device="cuda")
        op = lambda: nv.nvfp4_w4a16_lora_gemm_dgrad(dy, q.codes, q.scales, q.tensor_scale, a, b, LORA_SCALE, z,
                                                    dx, ws)
        nbytes, flops = gemm_bytes(M, *shape, R_LORA), gemm_flops(M, *shape, R_LORA)
    else:
        a, b = synth.lora_pair(shape[0], shape[1], R_LORA, 0.01, 2)
        a, b = dev(a), dev(b)
        z = torch.from_numpy(synth.noise_vector(shape[1], SIGMA, 3)).cuda()
        x = dev(synth.activations(M, shape[1], 10))
        ydt = torch.bfloat16 if kind == "prefill" else torch.float32
        y = torch.empty((M, shape[0]), dtype=ydt, device="cuda")
        op = lambda: nv.nvfp4_w4a16_lora_gemm(x, q.codes, q.scales, q.tensor_scale, a, b, LORA_SCALE, z, y, ws)
        nbytes, flops = gemm_bytes(M, *shape, R_LORA), gemm_flops(M, *shape, R_LORA)
    op()
    torch.cuda.synchronize()
    us_eager = time_replays(torch, [op], reps) * 1e3
    g = capture(torch, op)
    us = time_replays(torch, [g.replay], reps) * 1e3 if g is not None else us_eager
    st = nv.nvfp4_get_device_status(ws)
    if st != nv.OK:
        raise RuntimeError(nv.status_string(st))
    print(f"kernel case {case}: {reps} reps, graph {us:.2f} us/call (eager {us_eager:.2f}), "
          f"{nbytes / us / 1e3:.1f} GB/s, {flops / us / 1e6:.1f} TFLOP/s")


def run_list_case(torch, nv, synth, M, reps, R=8):
    """Kernel case for ncu: one nvfp4_w4a16_lora_gemm_list call over R up and R
    down replicas of the 7B MLP weights (R = 8: 0.61 GB, > 4x L2), repeated."""
    dev = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).cuda()
    ws = nv.new_workspace(max(nv.nvfp4_workspace_bytes(16, *sh, R_LORA) for sh in (UP, DOWN)))
    ents = []
    for name, sh, seed in (("up", UP, 0), ("down", DOWN, 100)):
        w = dev(synth.normal_weight(sh, 0.02, seed, outlier_frac=1e-3, outlier_mult=20.0))
        a, b = synth.lora_pair(sh[0], sh[1], R_LORA, 0.01, seed + 2)
        a, b = dev(a), dev(b)
        z = torch.from_numpy(synth.noise_vector(sh[1], SIGMA, seed + 3)).cuda()
        x = dev(synth.activations(M, sh[1], seed + 10 + M))
        for _ in range(R):
            q = nv.quantize(w, workspace=ws)
            ents.append((x, q.codes, q.scales, q.tensor_scale, a, b, LORA_SCALE, z,
                         torch.empty((M, sh[0]), dtype=torch.float32, device="cuda")))
        del w
    ents = [ents[(k % 2) * R + k // 2] for k in range(2 * R)]  # up, down alternating
    wsl = nv.new_workspace(nv.nvfp4_gemm_list_workspace_bytes(ents))
    op = lambda: nv.nvfp4_w4a16_lora_gemm_list(ents, wsl)
    op()
    torch.cuda.synchronize()
    us_eager = time_replays(torch, [op], reps) * 1e3
    g = capture(torch, op)
    us = time_replays(torch, [g.replay], reps) * 1e3 if g is not None else us_eager
    if nv.nvfp4_get_device_status(wsl) != nv.OK:
        raise RuntimeError("device status after the list case")
    nbytes = sum(gemm_bytes(M, *sh, R_LORA) for sh in (UP, DOWN)) * R
    name = f"list_M{M}" if R == 8 else f"list{2 * R}_M{M}"
    print(f"kernel case {name}: {reps} reps, graph {us:.2f} us/call (eager {us_eager:.2f}), "
          f"{2 * R} projections, {us / (2 * R):.2f} us/projection, {nbytes / us / 1e3:.1f} GB/s")


def free_port():
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def replica_command(argv, n, port):
    """The command that runs this benchmark as n single-GPU ranks on 127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel-case", default=None,
                    help="run one operation repeatedly (quantize_up, gemm_up_M8, gemm_down_M16, ...)")
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of CUDA graphs")
    ap.add_argument("--no-prefill", action="store_true", help="skip the 16384-token tensor-core GEMM line")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the single-layer, 32B-decode and whole-stack lines")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and not args.kernel_case:
        # N replicas: one process per GPU, started the way the driver does
        sys.exit(subprocess.call(replica_command(sys.argv[1:], args.gpus, free_port())))
    if args.kernel_case:
        run_kernel_case(args.kernel_case, args.reps)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
