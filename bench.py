"""Throughput of the FP8 MoE expert-FFN forward on GB300.

One step = one pass of the whole forward path (activation quantisation,
ragged sort + gather, gmm wi_0|wi_1, SwiGLU + requantisation, gmm wo, ragged
gather-reduce) over one batch of synthetic tokens.  Default workload: the
DeepSeek-V3-shaped layer (T=16384, d_model=7168, 256 experts, top-8,
d_ff=2048), per-token-per-128-channel activation scales and blockwise
[E, K/128, N] weight scales, the largest of the five layers on every axis.
Timed in the same run and reported as sub-objects of the same line
(`secondary`, `secondaries`):
- the Mixtral-shaped layer (T=8192, d_model=4096, 8 experts, top-2,
  d_ff=14336, per-token / per-channel scales);
- the serving prefill chunk (T=2048, d_model=2048, 128 experts, top-8,
  d_ff=768, pre-quantised blockwise weights);
- the MXFP8 variant of the DeepSeek-V3-shaped layer;
- the int8-weight variants of the Mixtral-shaped layer and the prefill chunk.

Prints one JSON line (rank 0).  Launch with torchrun for several GPUs: every
rank runs its own batch (data parallel over tokens, no collective on the data
path), the timing is the max over ranks, and `value` counts the tokens of all
ranks.  `--impl reference` times the CPU oracle instead, on a bounded sample.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE FFN fwd tokens/s & gmm_fp8 TFLOP/s as % of GB300 FP8 dense peak"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="dsv3", choices=list(synth.CONFIGS))
    ap.add_argument("--secondary", default="mixtral,prefill,dsv3_mx,mixtral_w8,prefill_w8",
                    help="comma-separated configs timed in the same run after the main one (at most 50 steps "
                         "each), reported as sub-objects: 'secondary' (the first) and 'secondaries' (all); "
                         "'' for none")
    ap.add_argument("--tokens", type=int, default=0, help="override T (small cases for profiling)")
    ap.add_argument("--experts", type=int, default=0, help="override E (small cases for profiling)")
    ap.add_argument("--cpu-sample-tokens", type=int, default=0, help="oracle sample size (0 = auto)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--suite", action="store_true",
                    help="time every call of the path alone, for every config (one JSON line per call)")
    ap.add_argument("--suite-configs", default="mixtral,dsv3,prefill,fwdbwd,tiny")
    ap.add_argument("--train-passes", type=int, default=0,
                    help="run this many forward + backward passes of --config (for profiling the backward "
                         "kernels; prints one timing line instead of the benchmark line)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_name(cfg) -> str:
    modes = {0: "per-token", 1: "per-token-per-128", 2: "static", 4: "MXFP8 (E8M0 per 32 columns)"}
    wmodes = {0: "per-channel", 1: "blockwise [E, K/128, N]", 2: "static", 4: "MXFP8 (E8M0 per 32 of K)"}
    return (f"{cfg.name} MoE expert FFN fwd: T={cfg.T} d_model={cfg.D} E={cfg.E} top-k={cfg.k} d_ff={cfg.F} SwiGLU; "
            f"e4m3 {modes[cfg.act_mode]} activation scales, {wmodes[cfg.w_mode]} weight scales"
            + ("; int8 weight codes" if cfg.w_int8 else ""))


def fwd_flops(cfg) -> dict:
    R = cfg.T * cfg.k
    return {"gmm_in": 2.0 * R * cfg.D * 2 * cfg.F, "gmm_out": 2.0 * R * cfg.F * cfg.D}


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def kernel_source_hash() -> str:
    """Hash of the contraction kernels' sources: recorded DRAM traffic is only
    reported while the kernels are the ones it was measured on."""
    import hashlib
    h = hashlib.sha256()
    for f in ("gmm.cu", "common.cuh"):
        with open(os.path.join(ROOT, "fp8_quantized_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kname: str, cfg):
    """DRAM bytes (read + write) per call of `kname` on this workload, from the
    ncu record in profiles/traffic.json, or None when there is no record or
    the contraction kernels changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        recs = json.load(f)
    src = kernel_source_hash()
    for rec in recs:
        if (rec.get("call") == kname and rec.get("config") == cfg.name and rec.get("T") == cfg.T
                and rec.get("source") == src):
            return rec["bytes_per_call"]
    return None


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

CPU_SAMPLE_EXPERTS = 16


def sample_experts(cfg):
    """The experts whose (token, expert) pairs the CPU sample takes: all of
    them for small E, else a seeded choice of 16."""
    if cfg.E <= CPU_SAMPLE_EXPERTS:
        return list(range(cfg.E))
    rng = np.random.default_rng(12345)
    return sorted(int(e) for e in rng.choice(cfg.E, CPU_SAMPLE_EXPERTS, replace=False))


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def omp_threads(n: int) -> bool:
    """Thread count of the oracle's OpenMP regions (libgomp, already loaded
    with the oracle library)."""
    try:
        ctypes.CDLL("libgomp.so.1").omp_set_num_threads(int(n))
        return True
    except (OSError, AttributeError):
        return False


class OracleSample:
    """The oracle forward on a bounded sample of one workload.

    The sample is a seeded selection of the (token, expert) pairs routed to
    the experts of `sample_experts` (every expert when E <= 16).  Each pair is
    one row of the oracle's forward: its token's activation quantised, the
    row gathered, both contractions with its expert's weights, SwiGLU with the
    requantisation, and the weighted combine; a token's output is the sum of
    k such rows, so `pairs / k` is the number of tokens of work done.  Only
    the sampled experts' weights are quantised (beforehand, untimed)."""

    def __init__(self, cfg, x_bits, ids, w, w_in_bits, w_out_bits, experts, static):
        import oracle
        self.oracle = oracle
        self.cfg, self.x, self.static = cfg, x_bits, static
        self.mx = cfg.act_mode == synth.MX32
        if self.mx:
            self.wq = oracle.prepare_weights_mx(w_in_bits, w_out_bits)
        elif cfg.w_int8:
            self.wq = oracle.prepare_weights_w8(w_in_bits, w_out_bits, cfg.w_mode)
        else:
            self.wq = oracle.prepare_weights(w_in_bits, w_out_bits, cfg.w_mode, static)
        remap = -np.ones(cfg.E, np.int64)
        remap[np.asarray(experts)] = np.arange(len(experts))
        loc = remap[ids]
        t, j = np.nonzero(loc >= 0)
        perm = np.random.default_rng(7).permutation(len(t))
        self.t, self.j = t[perm], j[perm]
        self.local = loc[self.t, self.j].astype(np.int32)
        self.w = w[self.t, self.j].astype(np.float32)
        self.nE = len(experts)
        self.npairs = len(self.t)

    def time(self, n: int, offset: int = 0) -> float:
        idx = (offset + np.arange(n)) % self.npairs
        xs = np.ascontiguousarray(self.x[self.t[idx]])
        ids = self.local[idx].reshape(-1, 1)
        w = self.w[idx].reshape(-1, 1)
        t0 = time.perf_counter()
        if self.mx:
            self.oracle.ffn_forward_mx(xs, ids, w, self.wq, self.nE)
        else:
            self.oracle.ffn_forward(xs, ids, w, self.wq, self.nE, self.cfg.act_mode, self.static)
        return time.perf_counter() - t0

    def aim(self, target_s: float, start: int = 64) -> tuple:
        """(pairs, seconds) of a sample grown towards target_s seconds."""
        n = min(start, self.npairs)
        dt = self.time(n)
        for _ in range(2):
            if dt >= 0.6 * target_s or n >= self.npairs:
                break
            n = int(min(self.npairs, max(n + 1, n * target_s / max(dt, 1e-3))))
            dt = self.time(n)
        return n, dt


def host_bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def host_inputs(cfg, seed=0):
    x = synth.activations(cfg, seed)
    ids, w = synth.routing(cfg, seed)
    return x, ids, w


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_ours(args, cfg, rank, world, local, secondary=False):
    """Time `args.steps` forward steps of `cfg`.  A secondary run (a second
    workload in the same process) skips the end-to-end loop and the CPU
    baseline and times at most 50 steps."""
    import fp8_quantized_moe_gb300 as moe

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group("nccl", device_id=dev)
    steps = min(args.steps, 50) if secondary else args.steps
    static = synth.calibration_scales(cfg, 0) if cfg.act_mode == synth.PER_TENSOR else None
    sx = sh = None
    if static:
        sx = torch.tensor([static["x"]], dtype=torch.float32, device=dev)
        sh = torch.tensor([static["h"]], dtype=torch.float32, device=dev)

    # inputs: each rank its own batch (seed = rank)
    x_host, ids_np, w_np = host_inputs(cfg, seed=rank)
    w_in, w_out = synth.expert_weights(cfg, 0, device=dev)
    W = (moe.prepare_weights_w8(w_in, w_out, cfg.w_mode) if cfg.w_int8 else
         moe.prepare_weights(w_in, w_out, cfg.w_mode, static))
    torch.cuda.synchronize()
    cpu_sample = None
    if rank == 0 and not args.no_cpu_baseline and not secondary:
        # the oracle leg quantises its own copy of the sampled experts' bf16 weights
        ex = sample_experts(cfg)
        sel = torch.tensor(ex, device=dev)
        cpu_sample = (ex, host_bits(w_in.index_select(0, sel)), host_bits(w_out.index_select(0, sel)))
    # only the fp8 copies stay resident
    w_in = w_out = None
    torch.cuda.empty_cache()
    x = x_host.to(dev)
    ids = torch.from_numpy(ids_np).to(dev)
    w = torch.from_numpy(w_np).to(dev)
    buf = moe.FFNBuffers(cfg.T, cfg.D, cfg.E, cfg.k, cfg.F, cfg.act_mode, dev)
    stream = torch.cuda.current_stream()

    mx = cfg.act_mode == synth.MX32
    w8 = cfg.w_int8

    def step(ev=None):
        if ev is None:
            return moe.ffn_forward(x, ids, w, W, cfg.act_mode, buf, sx, sh)
        # the same calls as ffn_forward, with events around the two gmms
        E = W.w_in.shape[0]
        if mx:
            s = moe.quantize_sort_mx(x, ids, E, out=buf.sort)
            ev[0].record(stream)
            moe.gmm_mx_swiglu(s["xs_q"], s["xs_scale"], W.w_in, W.s_in, s["group_sizes"], h_q=buf.h_q, h_sf=buf.h_s)
            ev[1].record(stream)
            ev[2].record(stream)
            moe.gmm_mx(buf.h_q, buf.h_s, W.w_out, W.s_out, s["group_sizes"], out=buf.o)
            ev[3].record(stream)
            moe.ragged_gather_reduce(buf.o, s["pos"], w, cfg.k, out=buf.y)
            return buf.y
        s = moe.quantize_sort(x, ids, E, cfg.act_mode, sx, out=buf.sort)
        xs_s = s["xs_scale"] if cfg.act_mode != 2 else sx
        ev[0].record(stream)
        if w8:
            ws = buf.w8_workspace()
            moe.gmm_w8(s["xs_q"], xs_s, cfg.act_mode, W.w_in, W.s_in, W.in_mode, s["group_sizes"], out=buf.a,
                       workspace=ws)
            ev[1].record(stream)
            moe.swiglu_quant(buf.a, cfg.act_mode, sh, h_q=buf.h_q, h_scale=buf.h_s)
            h_s = buf.h_s if cfg.act_mode != 2 else sh
            ev[2].record(stream)
            moe.gmm_w8(buf.h_q, h_s, cfg.act_mode, W.w_out, W.s_out, W.out_mode, s["group_sizes"], out=buf.o,
                       workspace=ws)
            ev[3].record(stream)
            moe.ragged_gather_reduce(buf.o, s["pos"], w, cfg.k, out=buf.y)
            return buf.y
        if moe.swiglu_fuse_pays(cfg.act_mode, W.in_mode, cfg.F):
            moe.gmm_swiglu(s["xs_q"], xs_s, cfg.act_mode, W.w_in, W.s_in, W.in_mode, s["group_sizes"], cfg.act_mode,
                           sh, h=buf.h, h_q=buf.h_q, h_scale=buf.h_s)
            ev[1].record(stream)
        else:
            moe.gmm(s["xs_q"], xs_s, cfg.act_mode, W.w_in, W.s_in, W.in_mode, s["group_sizes"], out=buf.a)
            ev[1].record(stream)
            moe.swiglu_quant(buf.a, cfg.act_mode, sh, h_q=buf.h_q, h_scale=buf.h_s)
        h_s = buf.h_s if cfg.act_mode != 2 else sh
        ev[2].record(stream)
        moe.gmm(buf.h_q, h_s, cfg.act_mode, W.w_out, W.s_out, W.out_mode, s["group_sizes"], out=buf.o)
        ev[3].record(stream)
        moe.ragged_gather_reduce(buf.o, s["pos"], w, cfg.k, out=buf.y)
        return buf.y

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if moe.device_error():
        raise RuntimeError("device error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    start.record(stream)
    for i in range(steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    ms = start.elapsed_time(end) / steps
    gmm_ms = [(e[0].elapsed_time(e[1]), e[2].elapsed_time(e[3])) for e in evs]
    if world > 1:
        t = torch.tensor([ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    if moe.device_error():
        raise RuntimeError("device error during the timed steps")

    # end to end through the public API: every step copies its inputs in from
    # pinned host memory and its y out, double-buffered so that the copies of
    # step i+1 (in) and i-1 (out) run on their own streams beside step i
    e2e = None
    if not args.no_e2e and not secondary:
        xh = x_host.pin_memory()
        idh = torch.from_numpy(ids_np).pin_memory()
        wh = torch.from_numpy(w_np).pin_memory()
        bufs = [buf, moe.FFNBuffers(cfg.T, cfg.D, cfg.E, cfg.k, cfg.F, cfg.act_mode, dev)]
        xd, idd, wd = [x, torch.empty_like(x)], [ids, torch.empty_like(ids)], [w, torch.empty_like(w)]
        yh = [torch.empty(cfg.T, cfg.D, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def e2e_step(i):
            j = i % 2
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(ev_done[j])  # step i-2 is done reading these inputs
                xd[j].copy_(xh, non_blocking=True)
                idd[j].copy_(idh, non_blocking=True)
                wd[j].copy_(wh, non_blocking=True)
                ev_in[j].record(h2d)
            stream.wait_event(ev_in[j])
            if i >= 2:
                stream.wait_event(ev_out[j])  # step i-2's y has left this buffer
            y = moe.ffn_forward(xd[j], idd[j], wd[j], W, cfg.act_mode, bufs[j], sx, sh)
            ev_done[j].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_done[j])
                yh[j].copy_(y, non_blocking=True)
                ev_out[j].record(d2h)

        def e2e_run(n):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            h2d.wait_stream(stream)
            for i in range(n):
                e2e_step(i)
            stream.wait_stream(d2h)
            stream.wait_stream(h2d)
            s1.record(stream)
            torch.cuda.synchronize()
            return s0.elapsed_time(s1)

        e2e_run(3)
        ems = e2e_run(args.steps) / args.steps
        if world > 1:
            t = torch.tensor([ems], device=dev)
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            ems = float(t.item())
        if moe.device_error():
            raise RuntimeError("device error during the end-to-end steps")
        h2d_bytes = xh.numel() * 2 + idh.numel() * 4 + wh.numel() * 4
        e2e = {"value": cfg.T * world / (ems / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d_bytes,
               "d2h_bytes_per_step": yh[0].numel() * 2, "ms_per_step": ems,
               "note": "public ffn_forward per step; inputs copied in from pinned host memory and y copied out "
                       "every step, on their own streams, double-buffered across steps"}

    fused = mx or (not w8 and moe.swiglu_fuse_pays(cfg.act_mode, W.in_mode, cfg.F))
    # quantise + sort (histogram, scan, scatter, quantise-gather) + (fused gmm+SwiGLU 1, +1 code
    # pass for per-row h scales | gmm 1 + SwiGLU 1) + gmm 1 + combine 1; the int8-weight gmms each
    # add their f16 decode of the activations where they take the 256-token tile (groups of 256
    # rows or more on average)
    # the sort's index kernels run as one CTA for up to 32768 pairs and 64 experts
    sort_launches = 1 if (cfg.T * cfg.k <= 32768 and cfg.E <= 64) else 3
    launches_per_step = (sort_launches + 1 + ((1 + (1 if cfg.act_mode == 0 else 0)) if fused else 2) + 1 + 1
                         + (2 if w8 and cfg.T * cfg.k >= 256 * cfg.E else 0))
    fl = fwd_flops(cfg)
    g_in = float(np.mean([a for a, _ in gmm_ms]))
    g_out = float(np.mean([b for _, b in gmm_ms]))
    pk, pk_kind = peaks()
    # the timed region is well under a second of GPU time: the burst figure
    # applies; the int8-weight contractions run on the f16 MMA, whose dense
    # rate is the bf16 one
    fp8_peak = 2.0 * pk["bf16_tflops"]
    tc_peak = pk["bf16_tflops"] if w8 else fp8_peak
    # the dominant call of the step is the wi_0 | wi_1 contraction; it is
    # bound by whichever of its flops (fp8 peak) and its bytes (HBM) takes
    # longer: the weight stream binds the small prefill batch
    R = cfg.T * cfg.k
    if mx:
        nbytes = (R * cfg.D + cfg.E * 2 * cfg.F * cfg.D + R * cfg.F) * 33 // 32
    else:
        # codes, the weights, the output, and the fp32 scales the call reads
        sa = {synth.PER_ROW: 4 * R, synth.PER_ROW_BLOCK128: 4 * R * (cfg.D // 128)}.get(cfg.act_mode, 0)
        sw = {synth.PER_ROW: 4 * cfg.E * 2 * cfg.F,
              synth.PER_ROW_BLOCK128: 4 * cfg.E * (cfg.D // 128) * 2 * cfg.F}.get(cfg.w_mode, 0)
        out = (5 if cfg.act_mode == synth.PER_ROW else 1) * R * cfg.F if fused else 4 * R * cfg.F
        nbytes = R * cfg.D + cfg.E * 2 * cfg.F * cfg.D + out + sa + sw
    hbm_bound = nbytes / (pk["hbm_gbs"] * 1e9) > fl["gmm_in"] / (tc_peak * 1e12)
    if hbm_bound:
        achieved, peak, unit = nbytes / (g_in / 1e3) / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = fl["gmm_in"] / (g_in / 1e3) / 1e12, tc_peak, "TFLOP/s"
    both = (fl["gmm_in"] + fl["gmm_out"]) / ((g_in + g_out) / 1e3) / 1e12
    kname = ("gmm_fp8_mx_swiglu" if mx else "gmm_fp8_w8 (wi_0|wi_1)" if w8 else
             "gmm_fp8_swiglu" if fused else "gmm_fp8 (wi_0|wi_1)")
    result = {
        "metric": METRIC,
        "value": cfg.T * world / (ms / 1e3),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("e4m3 with E8M0 block scales (MXFP8), fp32 accumulate, bf16 in/out" if mx else
                  "e4m3 activations x int8 weights on the f16 tensor-core MMA (both exact in f16), fp32 "
                  "accumulate, bf16 in/out" if w8 else "e4m3 (fp32 accumulate, bf16 in/out)"),
        "data": "synthetic (seeded N(0,1) activations, N(0,0.02) weights, random-init)",
        "config": {"workload": workload_name(cfg), "tokens_per_gpu": cfg.T, "parallelism": f"dp{world} (replicas)",
                   "l2": "inputs larger than L2: fp8 expert weights %.2f GB streamed every step"
                         % ((2 * cfg.F * cfg.D + cfg.D * cfg.F) * cfg.E / 1e9)},
        "roofline": {"bound": "hbm" if hbm_bound else "tensor", "kernel": kname, "achieved": achieved,
                     "peak": peak, "unit": unit, "frac": achieved / peak,
                     "traffic": recorded_traffic(kname, cfg) if not (args.tokens or args.experts) else None,
                     "peak_note": (f"of {pk_kind}: STREAM-style copy" if hbm_bound else
                                   f"of {pk_kind}: f16 = burst bf16 cuBLAS ({pk['bf16_tflops']} TFLOP/s; the "
                                   "nominal dense f16 and bf16 rates are equal)" if w8 else
                                   f"of {pk_kind}: fp8 = 2 x burst bf16 cuBLAS ({pk['bf16_tflops']} TFLOP/s; "
                                   "the nominal dense fp8 / bf16 ratio is 2)"),
                     "flops_per_call": fl["gmm_in"], "algorithmic_bytes_per_call": nbytes, "ms_per_call": g_in,
                     "note": ("one gmm_fp8_mx_swiglu call per step: the block-scaled tcgen05 contraction with the "
                              "SwiGLU and MXFP8 requantisation epilogue") if mx else
                             ("one gmm_fp8_w8 call per step: the e4m3 activations "
                              + ("decoded to f16 in a workspace (256-token tiles)" if cfg.T * cfg.k >= 256 * cfg.E
                                 else "converted to f16 on the SM (128-token tiles)")
                              + ", the int8 weights converted to f16 into tensor memory, tcgen05 kind::f16") if w8 else
                             ("one gmm_fp8_swiglu call per step: the tcgen05 contraction with the SwiGLU and "
                              "requantisation epilogue, plus the h code pass of the per-token scales") if fused else
                             "one gmm_fp8 call per step"},
        "gmm_fp8_both": {"achieved": both, "frac": both / tc_peak, "unit": "TFLOP/s", "gmm_in_ms": g_in,
                         "gmm_out_ms": g_out, "note": "both contractions of the step, timed with events"},
        "gpu_launches": launches_per_step * steps,
        "clocks": clk,
    }
    if e2e:
        result["e2e"] = e2e
    del buf, W
    torch.cuda.empty_cache()
    if cpu_sample is not None:
        result["cpu_baseline"] = cpu_baseline(args, cfg, x_host, ids_np, w_np, cpu_sample, static)
    return result


def cpu_baseline(args, cfg, x_host, ids_np, w_np, cpu_sample, static):
    """The oracle, as it stands, on a bounded sample of the workload: ~15 s on
    all host cores, then ~8 s on one core."""
    ex, w_in_b, w_out_b = cpu_sample
    smp = OracleSample(cfg, host_bits(x_host), ids_np, w_np, w_in_b, w_out_b, ex, static)
    cores = os.cpu_count()
    omp_threads(cores)
    if args.cpu_sample_tokens:
        n = min(smp.npairs, args.cpu_sample_tokens * cfg.k)
        dt = smp.time(n)
    else:
        n, dt = smp.aim(15.0)
    rate = n / cfg.k / dt
    res = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
           "sample": f"{n} (token, expert) pairs of {cfg.T * cfg.k} ({n / cfg.k:.0f} tokens of work), routed to "
                     f"{len(ex)} of the {cfg.E} experts, through the oracle forward (fp64, OpenMP); weights "
                     f"quantised beforehand", "seconds": dt, "cpu_model": cpu_model()}
    if omp_threads(1):
        n1 = max(1, min(smp.npairs, int(n * 8.0 / max(dt * cores, 1e-3))))
        dt1 = smp.time(n1, offset=n)
        res["single_thread"] = {"value": n1 / cfg.k / dt1, "unit": "tokens/s", "cores": 1,
                                "sample": f"{n1} pairs", "seconds": dt1}
        omp_threads(cores)
    return res


def run_reference(args, cfg, rank, world):
    """The reference arm: the oracle, as it stands, on the host's cores.  Each
    step is a bounded sample of the workload (16 tokens of work: 16 k
    (token, expert) pairs of the sampled experts, see OracleSample).  Only
    the sampled experts' weights are drawn and quantised (beforehand)."""
    if rank != 0:
        return None
    import oracle
    oracle.build()
    x_host, ids_np, w_np = host_inputs(cfg, seed=0)
    ex = sample_experts(cfg)
    w_in, w_out = synth.expert_weights(cfg, 0, experts=ex)
    static = synth.calibration_scales(cfg, 0) if cfg.act_mode == synth.PER_TENSOR else None
    smp = OracleSample(cfg, host_bits(x_host), ids_np, w_np, host_bits(w_in), host_bits(w_out), ex, static)
    del w_in, w_out
    cores = os.cpu_count()
    omp_threads(cores)
    n = min(smp.npairs, (args.cpu_sample_tokens or 16) * cfg.k)
    for i in range(args.warmup):
        smp.time(max(1, n // 4), offset=i * n)
    times = [smp.time(n, offset=i * n) for i in range(args.steps)]
    sec = float(np.sum(times))
    value = n / cfg.k * args.steps / sec
    return {
        "metric": METRIC, "impl": "reference", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": workload_name(cfg)},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} (token, expert) pairs per step ({n / cfg.k:.0f} tokens of work) routed to "
                                   f"{len(ex)} of the {cfg.E} experts", "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ---------------------------------------------------------------------------
# Per-call suite: every step of the path timed alone against its roofline
# ---------------------------------------------------------------------------

def mx_calls(moe, cfg, x, ids, w, W, buf):
    """The MXFP8 variant's calls: (label, fn, bound, work), E8M0 codes one
    byte per 32 values (1/32 of the codes' bytes)."""
    T, D, E, k, F = cfg.T, cfg.D, cfg.E, cfg.k, cfg.F
    R = T * k
    s = buf.sort
    return [
        ("quantize_sort_mx (steps 1 + 2 fused)", lambda: moe.quantize_sort_mx(x, ids, E, out=s),
         "hbm", 2 * T * D + R * D + R * D // 32 + 16 * R),
        ("gmm_fp8_mx_swiglu (wi_0|wi_1 + SwiGLU + MX requant)",
         lambda: moe.gmm_mx_swiglu(s["xs_q"], s["xs_scale"], W.w_in, W.s_in, s["group_sizes"], h_q=buf.h_q,
                                   h_sf=buf.h_s),
         "tensor", (2.0 * R * D * 2 * F, (R * D + E * 2 * F * D + R * F) * 33 // 32)),
        ("gmm_fp8_mx wi_0|wi_1", lambda: moe.gmm_mx(s["xs_q"], s["xs_scale"], W.w_in, W.s_in, s["group_sizes"],
                                                    out=buf.a),
         "tensor", (2.0 * R * D * 2 * F, (R * D + E * 2 * F * D) * 33 // 32 + 4 * R * F)),
        ("moe_swiglu_quant_mx", lambda: moe.swiglu_quant_mx(buf.a, h_q=buf.h_q, h_sf=buf.h_s),
         "hbm", 4 * R * F + R * F * 33 // 32),
        ("gmm_fp8_mx wo", lambda: moe.gmm_mx(buf.h_q, buf.h_s, W.w_out, W.s_out, s["group_sizes"], out=buf.o),
         "tensor", (2.0 * R * F * D, (R * F + E * D * F) * 33 // 32 + 2 * R * D)),
    ]


def run_suite(args):
    import fp8_quantized_moe_gb300 as moe

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pk, pk_kind = peaks()
    hbm = pk["hbm_gbs"]
    fp8 = 2.0 * pk["bf16_tflops"]  # calls timed alone: burst figure
    # L2 flush by reading 512 MB (> 129 MB of L2): the lines left behind are
    # clean, so the timed call pays no write-back of someone else's data
    flush = torch.ones(64 * 1024 * 1024, dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream()
    lines = []

    def timed(fn, reps=10):
        fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            flush.sum()  # evict the previous call's data from L2
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    for name in args.suite_configs.split(","):
        cfg = synth.CONFIGS[name]
        T, D, E, k, F = cfg.T, cfg.D, cfg.E, cfg.k, cfg.F
        R = T * k
        static = synth.calibration_scales(cfg, 0) if cfg.act_mode == synth.PER_TENSOR else None
        sx = sh = None
        if static:
            sx = torch.tensor([static["x"]], dtype=torch.float32, device=dev)
            sh = torch.tensor([static["h"]], dtype=torch.float32, device=dev)
        x_host, ids_np, w_np = host_inputs(cfg, 0)
        w_in, w_out = synth.expert_weights(cfg, 0, device=dev)
        W = (moe.prepare_weights_w8(w_in, w_out, cfg.w_mode) if cfg.w_int8 else
             moe.prepare_weights(w_in, w_out, cfg.w_mode, static, for_backward=cfg.backward))
        del w_in, w_out
        torch.cuda.empty_cache()
        x = x_host.to(dev)
        ids = torch.from_numpy(ids_np).to(dev)
        w = torch.from_numpy(w_np).to(dev)
        buf = moe.FFNBuffers(T, D, E, k, F, cfg.act_mode, dev, backward=cfg.backward)
        am = cfg.act_mode
        w8 = cfg.w_int8
        fused = not w8 and moe.swiglu_fuse_pays(am, W.in_mode, F)
        fusable = not w8 and moe.swiglu_fusable(am, W.in_mode, F)
        moe.ffn_forward(x, ids, w, W, am, buf, sx, sh)  # fills every intermediate
        torch.cuda.synchronize()
        nb = lambda c: (c + 127) // 128
        sbytes = lambda rows, cols: 0 if am == 2 else 4 * rows * (1 if am == 0 else nb(cols))
        xs_s = buf.sort["xs_scale"] if am != 2 else sx
        h_s = buf.h_s if am != 2 else sh
        if am == synth.MX32:
            calls = mx_calls(moe, cfg, x, ids, w, W, buf)
            fused, fusable = True, True
        else:
            calls = []
        calls += [] if am == synth.MX32 else [
            ("quantize_sort (steps 1 + 2 fused)", lambda: moe.quantize_sort(x, ids, E, am, sx, out=buf.sort),
             "hbm", 2 * T * D + R * D + 16 * R + sbytes(R, D)),
            ("quantize_rows x", lambda: moe.quantize_rows(x, am, sx, q=buf.x_q, scale=buf.x_s),
             "hbm", 3 * T * D + sbytes(T, D)),
            ("ragged_sort (+ gather)", lambda: moe.ragged_sort(ids, E, buf.x_q, buf.x_s if am != 2 else sx, am,
                                                               out=buf.sort),
             "hbm", T * D + R * D + 16 * R + 2 * sbytes(T, D)),
        ]
        if fusable and am != synth.MX32:
            calls.append(("gmm_fp8_swiglu (wi_0|wi_1 + SwiGLU + requant)",
                          lambda: moe.gmm_swiglu(buf.sort["xs_q"], xs_s, am, W.w_in, W.s_in, W.in_mode,
                                                 buf.sort["group_sizes"], am, sh, h=buf.h, h_q=buf.h_q,
                                                 h_scale=buf.h_s, a_out=buf.a if buf.keep_a else None),
                          "tensor", (2.0 * R * D * 2 * F, R * D + E * 2 * F * D + (5 if am == 0 else 1) * R * F)))
        if w8:
            # the weight scales: per channel [E, N] or blockwise [E, K/128, N]
            ws = lambda N_, K_: 4 * E * N_ * (1 if cfg.w_mode == synth.PER_ROW else nb(K_))
            w8ws = buf.w8_workspace()
            calls.append(("gmm_fp8_w8 wi_0|wi_1", lambda: moe.gmm_w8(buf.sort["xs_q"], xs_s, am, W.w_in, W.s_in,
                                                                    W.in_mode, buf.sort["group_sizes"], out=buf.a,
                                                                    workspace=w8ws),
                          "tensor_f16", (2.0 * R * D * 2 * F, R * D + E * 2 * F * D + 4 * R * F + sbytes(R, D)
                                         + ws(2 * F, D))))
            calls.append(("moe_swiglu_quant", lambda: moe.swiglu_quant(buf.a, am, sh, h_q=buf.h_q,
                                                                       h_scale=buf.h_s),
                          "hbm", 5 * R * F + sbytes(R, F)))
            calls.append(("gmm_fp8_w8 wo", lambda: moe.gmm_w8(buf.h_q, h_s, am, W.w_out, W.s_out, W.out_mode,
                                                             buf.sort["group_sizes"], out=buf.o, workspace=w8ws),
                          "tensor_f16", (2.0 * R * F * D, R * F + E * D * F + 2 * R * D + sbytes(R, F) + ws(D, F))))
            calls.append(("gmm_fp8_w8 wi_0|wi_1 (activations converted on the SM)",
                          lambda: moe.gmm_w8(buf.sort["xs_q"], xs_s, am, W.w_in, W.s_in, W.in_mode,
                                             buf.sort["group_sizes"], out=buf.a),
                          "tensor_f16", (2.0 * R * D * 2 * F, R * D + E * 2 * F * D + 4 * R * F + sbytes(R, D)
                                         + ws(2 * F, D))))
        elif am != synth.MX32:
            calls.append(("gmm_fp8 wi_0|wi_1", lambda: moe.gmm(buf.sort["xs_q"], xs_s, am, W.w_in, W.s_in,
                                                               W.in_mode, buf.sort["group_sizes"], out=buf.a),
                          "tensor", (2.0 * R * D * 2 * F, R * D + E * 2 * F * D + 4 * R * F)))
            calls.append(("moe_swiglu_quant", lambda: moe.swiglu_quant(buf.a, am, sh, h_q=buf.h_q,
                                                                       h_scale=buf.h_s),
                          "hbm", 5 * R * F + sbytes(R, F)))
            calls.append(("gmm_fp8 wo", lambda: moe.gmm(buf.h_q, h_s, am, W.w_out, W.s_out, W.out_mode,
                                                        buf.sort["group_sizes"], out=buf.o),
                          "tensor", (2.0 * R * F * D, R * F + E * D * F + 2 * R * D)))
        calls.append(("ragged_gather_reduce", lambda: moe.ragged_gather_reduce(buf.o, buf.sort["pos"], w, k,
                                                                                out=buf.y),
                      "hbm", 2 * R * D + 2 * T * D + 8 * R))
        if cfg.backward:
            G = synth.output_grad(cfg, 0, device=dev)
            src, sizes = buf.sort["sorted_src"], buf.sort["group_sizes"]
            wflat = w.reshape(-1)
            dO, dO_q, dO_s = moe.gather_scale_quant(G, wflat, src, k)
            dA, dA_q, dA_s = moe.swiglu_bwd_quant(buf.dH, buf.a)
            calls += [
                ("bwd moe_gather_scale_quant", lambda: moe.gather_scale_quant(G, wflat, src, k),
                 "hbm", 2 * T * D + 3 * R * D + 4 * R),
                ("bwd gmm_fp8 dH = dO wo", lambda: moe.gmm(dO_q, dO_s, 0, W.w_out_t, W.s_out, 2, sizes, out=buf.dH),
                 "tensor", (2.0 * R * D * F, R * D + E * D * F + 2 * R * F)),
                ("bwd moe_swiglu_bwd_quant", lambda: moe.swiglu_bwd_quant(buf.dH, buf.a),
                 "hbm", 2 * R * F + 4 * R * F + 6 * R * F + 4 * R),
                ("bwd gmm_fp8_ksplit dXs = dA [wi_0|wi_1]",
                 lambda: moe.gmm_ksplit(dA_q, dA_s, 0, W.w_in_t, W.s_in_split, F, sizes, out=buf.dXs),
                 "tensor", (2.0 * R * 2 * F * D, 2 * R * F + E * 2 * F * D + 2 * R * D)),
                ("bwd ragged_gather_reduce dX", lambda: moe.ragged_gather_reduce(buf.dXs, buf.sort["pos"], None, k,
                                                                                 out=buf.dX),
                 "hbm", 2 * R * D + 2 * T * D + 4 * R),
                ("bwd moe_quantize_group_cols dA (scales)",
                 lambda: moe.quantize_group_cols(dA, sizes, scales_only=True), "hbm", 2 * R * 2 * F),
                ("bwd moe_quantize_group_cols dO (scales)",
                 lambda: moe.quantize_group_cols(dO, sizes, scales_only=True), "hbm", 2 * R * D),
            ]
            _, dAg_s = moe.quantize_group_cols(dA, sizes, scales_only=True)
            _, dOg_s = moe.quantize_group_cols(dO, sizes, scales_only=True)
            ws = torch.empty(moe.lib().tgmm_fp8_workspace_bytes(R, D, 2 * F, E), dtype=torch.uint8, device=dev)
            calls += [
                ("bwd tgmm_fp8_gcq dW_in (with the operand layouts)",
                 lambda: moe.tgmm_gcq(buf.sort["xs_q"], sx, 2, dA, dAg_s, sizes, workspace=ws),
                 "tensor", (2.0 * R * D * 2 * F, 4 * E * D * 2 * F + R * D + 2 * R * 2 * F)),
                ("bwd tgmm_fp8_gcq dW_out (with the operand layouts)",
                 lambda: moe.tgmm_gcq(buf.h_q, sh, 2, dO, dOg_s, sizes, workspace=ws),
                 "tensor", (2.0 * R * F * D, 4 * E * F * D + R * F + 2 * R * D)),
            ]
        # the router (gate contraction + softmax top-k, and its gradient): off the FFN step
        gwg = torch.Generator(device=dev)
        gwg.manual_seed(3)
        w_gate = (torch.randn(E, D, generator=gwg, device=dev) * (1.5 / np.sqrt(D))).to(torch.bfloat16)
        rlog, rids, _ = moe.router_topk(x, w_gate, k)
        G_r = torch.randn(T, D, generator=gwg, device=dev).to(torch.bfloat16)
        rws = torch.empty(moe.lib().moe_router_backward_workspace_bytes(T, D, E), dtype=torch.uint8, device=dev)
        calls += [
            ("router_topk (gate + softmax top-k)", lambda: moe.router_topk(x, w_gate, k),
             "tensor_bf16", (2.0 * T * D * E, 2 * T * D + 2 * E * D + 4 * T * E + 8 * T * k)),
            ("router_backward (dw, dlogits, grad_gate, state_grad)",
             lambda: moe.router_backward(G_r, buf.o, buf.sort["pos"], x, w_gate, rlog, rids, workspace=rws),
             "tensor_bf16", (4.0 * T * D * E, 2 * T * D + 2 * R * D + 3 * 2 * T * D + 2 * T * D + 4 * E * D)),
        ]
        total = 0.0
        for label, fn, bound, work in calls:
            ms = timed(fn)
            if bound == "hbm":
                ach, peak, unit = work / (ms / 1e3) / 1e9, hbm, "GB/s"
            elif bound in ("tensor_bf16", "tensor_f16"):  # the f16 and bf16 MMAs have one dense rate
                flops, nbytes = work
                if nbytes / (hbm * 1e9) > flops / (pk["bf16_tflops"] * 1e12):
                    bound, ach, peak, unit = "hbm", nbytes / (ms / 1e3) / 1e9, hbm, "GB/s"
                else:
                    bound, ach, peak, unit = "tensor", flops / (ms / 1e3) / 1e12, pk["bf16_tflops"], "TFLOP/s"
            else:
                # a contraction is bound by whichever of its flops and its bytes takes longer
                flops, nbytes = work
                if nbytes / (hbm * 1e9) > flops / (fp8 * 1e12):
                    bound, ach, peak, unit = "hbm", nbytes / (ms / 1e3) / 1e9, hbm, "GB/s"
                else:
                    ach, peak, unit = flops / (ms / 1e3) / 1e12, fp8, "TFLOP/s"
            if am == synth.MX32:
                on_path = label.startswith(("quantize_sort_mx", "gmm_fp8_mx_swiglu", "gmm_fp8_mx wo",
                                            "ragged_gather_reduce"))
            elif label.startswith("gmm_fp8_swiglu"):
                on_path = fused
            elif label.startswith("router") or label.endswith("(activations converted on the SM)"):
                on_path = False  # routing is an input of the FFN step; the variant is the slower form
            else:
                on_path = not ((fused and label in ("gmm_fp8 wi_0|wi_1", "moe_swiglu_quant")) or
                               label in ("quantize_rows x", "ragged_sort (+ gather)"))
            if on_path:
                total += ms
            line = {"suite": cfg.name, "call": label, "ms": round(ms, 4), "bound": bound,
                    "achieved": round(ach, 1), "peak": peak, "unit": unit, "frac": round(ach / peak, 3),
                    "on_step": on_path, "peak_kind": pk_kind}
            print(json.dumps(line), flush=True)
        step = {"suite": cfg.name, "call": "sum of the step's calls (timed alone, L2 flushed)",
                "ms": round(total, 4), "tokens_per_s": round(T / (total / 1e3), 1),
                "workload": workload_name(cfg) + (" + backward" if cfg.backward else "")}
        print(json.dumps(step), flush=True)
        assert moe.device_error() == 0
        del buf, W, x
        torch.cuda.empty_cache()


def run_train_passes(args):
    """Forward + backward passes of one config (the static-scale training layer by
    default); a profiling aid for the backward kernels, timed with CUDA events."""
    import fp8_quantized_moe_gb300 as moe

    cfg = synth.CONFIGS[args.config if args.config != "mixtral" else "fwdbwd"]
    if args.tokens:
        cfg = synth.scaled(cfg, T=args.tokens)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    static = synth.calibration_scales(cfg, 0) if cfg.act_mode == synth.PER_TENSOR else None
    sx = sh = None
    if static:
        sx = torch.tensor([static["x"]], dtype=torch.float32, device=dev)
        sh = torch.tensor([static["h"]], dtype=torch.float32, device=dev)
    x = synth.activations(cfg, 0).to(dev)
    ids, w = synth.routing(cfg, 0)
    w_in, w_out = synth.expert_weights(cfg, 0, device=dev)
    W = moe.prepare_weights(w_in, w_out, cfg.w_mode, static, for_backward=True)
    del w_in, w_out
    torch.cuda.empty_cache()
    G = synth.output_grad(cfg, 0).to(dev)
    buf = moe.FFNBuffers(cfg.T, cfg.D, cfg.E, cfg.k, cfg.F, cfg.act_mode, dev, backward=True)
    idd, wd = torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev)
    ms = []
    for _ in range(args.train_passes):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        moe.ffn_forward(x, idd, wd, W, cfg.act_mode, buf, sx, sh)
        moe.ffn_backward(G, wd.reshape(-1), W, buf, sx, sh)
        e1.record()
        torch.cuda.synchronize()
        ms.append(e0.elapsed_time(e1))
    if moe.device_error():
        raise RuntimeError("device error during the training passes")
    print(json.dumps({"train_passes": args.train_passes, "config": workload_name(cfg),
                      "ms_per_pass": ms, "tokens_per_s_last": cfg.T / (ms[-1] / 1e3)}), flush=True)


def main():
    args = parse()
    if args.suite:
        run_suite(args)
        return
    if args.train_passes:
        run_train_passes(args)
        return
    cfg = synth.CONFIGS[args.config]
    if args.tokens:
        cfg = synth.scaled(cfg, T=args.tokens)
    if args.experts:
        cfg = synth.scaled(cfg, E=args.experts)
    rank, world, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, cfg, rank, world)
    else:
        res = run_ours(args, cfg, rank, world, local)
        names = [n for n in (args.secondary or "").split(",") if n and n != cfg.name]
        if names and not (args.tokens or args.experts):
            subs = []
            for n in names:
                r2 = run_ours(args, synth.CONFIGS[n], rank, world, local, secondary=True)
                subs.append({k: r2[k] for k in ("value", "unit", "ms_per_step", "steps", "config", "roofline",
                                                "gmm_fp8_both", "gpu_launches", "clocks", "dtype")})
            res["secondary"] = subs[0]
            res["secondaries"] = subs
        if world > 1:
            torch.distributed.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
