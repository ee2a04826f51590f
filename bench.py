#!/usr/bin/env python
"""Throughput of the routed-expert MoE layer (libmoe) on GB300.

Default workload: single-token decode of the guide's layer (H 4096, I 2048,
256 MXFP4 experts, top-6 sqrt-softplus router, w_scale 1.5): every step is
one T = 1 layer call (route + permute + quantise + gate/up + down + combine)
on a fresh token with fresh logits, so the experts touched vary and the
3.4 GB expert set is far larger than L2.  --config 2/3/4 time the batched
decode, pp512 and 8192-token prefill workloads instead.

One JSON line on rank 0.  Under torchrun every rank runs an independent
replica on its own GPU (no collective in the layer); the time is the max over
ranks and `value` counts the tokens of all ranks.

--impl reference times the fp64 CPU oracle on the host cores on the same
workload (time-bounded; rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "routed-MoE layer tokens/s"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, choices=[1, 2, 3, 4])
    ap.add_argument("--path", choices=["auto", "cc", "tc"], default="auto")
    ap.add_argument("--graph-chunk", type=int, default=256, help="steps per CUDA graph")
    ap.add_argument("--decode-kernel", type=int, default=0, choices=[0, 1, 2],
                    help="one-token calls: 0 automatic, 1 the CUDA-core GEMV kernel, 2 the tcgen05 kernel")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the time-boxed records of the other workloads (default run only)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--trace", action="store_true",
                    help="after timing, trace one more call of the GEMM kernels (stderr)")
    ap.add_argument("--experts", type=int, default=None,
                    help="a smaller expert set with the same per-token work (for profiler captures)")
    ap.add_argument("--prune", default=None, metavar="KEEP[,MIN_W[,RHO]]",
                    help="tail pruning of the learned router (moe_set_route_prune), e.g. 5 or 6,0.11")
    args = ap.parse_args()
    args.prune_t = None
    if args.prune:
        v = args.prune.split(",")
        args.prune_t = (int(v[0]), float(v[1]) if len(v) > 1 else 0.0, float(v[2]) if len(v) > 2 else 0.0)
    return args


def default_steps(cfg):
    # long enough (~1 s) for the clock samples to fall inside the timed region
    return {1: 32768, 2: 1024, 3: 256, 4: 32}[cfg.index]


# ------------------------------------------------------------------ ranks --
# Replicas: every rank runs its own layer on its own tokens (no exchange);
# the job's time is the slowest rank's and its rate counts every rank's tokens.
def rank_seed(cfg, rank):
    """Token seed of a rank: each replica draws its own tokens."""
    return cfg.default_seed + 7919 * rank


def max_over_ranks(ms, world, dev):
    """The slowest rank's time (all ranks get it)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    tm = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(tm, op=dist.ReduceOp.MAX)
    return float(tm.item())


def chunk_spread(ms_per_step):
    """Median, min, max and std of the per-step time over the timed region's
    graph chunks; spread_pct = (max - min) / median (above 15 % is flagged)."""
    a = np.asarray(ms_per_step, dtype=np.float64)
    med = float(np.median(a))
    spread = float((a.max() - a.min()) / med * 100.0) if med > 0 else 0.0
    return {"chunks": int(a.size), "median_ms": round(med, 6), "min_ms": round(float(a.min()), 6),
            "max_ms": round(float(a.max()), 6), "std_ms": round(float(a.std()), 6),
            "spread_pct": round(spread, 2), "spread_over_15pct": spread > 15.0}


def job_rate(world, tokens_per_rank, ms):
    """Tokens per second of the whole job: every rank's tokens over the slowest rank's time."""
    return round(world * tokens_per_rank / (ms * 1e-3), 1)


def config_json(cfg, args, world):
    return {"workload": cfg.name, "hidden": cfg.H, "inter": cfg.I, "experts": cfg.E,
            "top_k": cfg.k, "tokens_per_step": cfg.T, "router": cfg.router,
            "shared_expert": cfg.shared, "weights": "MXFP4 e2m1 + UE8M0 /32",
            "activations": "MXFP8 e4m3 + UE8M0 /32", "gemm_path": args.path,
            **({"decode_kernel": {0: "auto", 1: "gemv", 2: "tcgen05"}[args.decode_kernel]}
               if cfg.T == 1 else {}),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "inputs larger than L2 (3.4 GB expert set; fresh tokens each step)",
            **({"route_prune": {"keep": args.prune_t[0], "min_w": args.prune_t[1], "rho": args.prune_t[2]}}
               if args.prune_t else {})}


def algorithmic_bytes(cfg, touched, rows):
    """Bytes one layer call must move at least: the touched experts' MXFP4
    weights (payload + scales) and the activation rows in and out."""
    H, I = cfg.H, cfg.I
    blk = 16 if getattr(cfg, "wfmt", "mxfp4") == "nvfp4" else 32  # elements per block scale byte
    w_gu = 2 * (I * H // 2 + I * H // blk)
    w_dn = H * I // 2 + H * I // blk
    act_gu = rows * (H + H // 32) + rows * (I + I // 32)
    act_dn = rows * (I + I // 32) + rows * H * 4
    return {"gateup": touched * w_gu + act_gu, "down": touched * w_dn + act_dn}


# ------------------------------------------------------------------ clocks --
def gpu_uuid(dev):
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


class ClockSampler:
    FIELDS = ("timestamp,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = []
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 10:
                continue
            if self.uuid and parts[1] != self.uuid:
                continue
            rows.append(parts)
        os.unlink(self.f.name)
        return rows

    @staticmethod
    def summary(rows):
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- our path --
def _upload_weights(w, dev):
    import torch
    return {n: torch.from_numpy(np.array(getattr(w, n))).to(dev)
            for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s",
                      "sh_gate_q", "sh_gate_s", "sh_up_q", "sh_up_s", "sh_down_q", "sh_down_s",
                      "gate_g", "up_g", "down_g")
            if getattr(w, n, None) is not None}


def make_layer(bqe, cfg, w, dev, max_tokens, path="auto", prune=None, decode_kernel=0):
    import torch
    dw = _upload_weights(w, dev)
    mc = bqe.MoeConfig(cfg.H, cfg.I, cfg.E, cfg.k, max_tokens, cfg.shared, cfg.w_scale,
                       bqe.MOE_WEIGHTS_NVFP4 if cfg.wfmt == "nvfp4" else bqe.MOE_WEIGHTS_MXFP4)
    layer = bqe.moe_create(mc, dw)
    torch.cuda.synchronize(dev)
    del dw
    bqe.moe_set_gemm_path(layer, {"auto": 0, "cc": 1, "tc": 2}[path])
    if decode_kernel:
        bqe.moe_set_decode_kernel(layer, decode_kernel)
    if prune:
        bqe.moe_set_route_prune(layer, *prune)
    return layer


class Workload:
    """Device inputs of S distinct batches of one configuration and the call
    that runs the layer on batch i (route + layer)."""

    def __init__(self, bqe, cfg, layer, dev, S, seed, router=None):
        import torch
        from workloads import make_hash_table, make_tokens
        self.bqe, self.cfg, self.layer, self.S = bqe, cfg, layer, S
        self.router = router or cfg.router
        tk = make_tokens(cfg, seed=seed, n=S * cfg.T)
        self.tokens = tk
        self.x = torch.from_numpy(tk.x_bits.view(np.int16).reshape(S, cfg.T, cfg.H).copy()).to(dev)
        self.lg = torch.from_numpy(tk.logits.reshape(S, cfg.T, cfg.E).copy()).to(dev)
        if self.router == "hash":
            self.tab = torch.from_numpy(make_hash_table(cfg)).to(dev)
            self.tok = torch.from_numpy(tk.token_ids.reshape(S, cfg.T).copy()).to(dev)
        self.ids = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
        self.wt = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
        self.out = torch.empty((cfg.T, cfg.H), dtype=torch.float32, device=dev)

    def step(self, i):
        j = i % self.S
        b = self.bqe
        if self.router == "hash":
            b.moe_route_hash(self.layer, self.tok[j], self.tab, self.ids, self.wt)
            b.moe_forward(self.layer, self.x[j], self.ids, self.wt, self.out)
        else:
            b.moe_route_forward(self.layer, self.lg[j], self.x[j], self.ids, self.wt, self.out)

    def touched(self, n=64):
        """Mean experts touched and mean kept (routed) rows per batch."""
        touched, kept = [], []
        for j in range(min(self.S, n)):
            self.step(j)
            idn = self.ids.cpu().numpy()
            touched.append(len(np.unique(idn[idn >= 0])))  # -1: a pruned slot
            kept.append(int((idn >= 0).sum()))
        return float(np.mean(touched)), int(round(np.mean(kept)))


def capture(step, first, n, chunk, stream, before_step=None):
    """CUDA graphs of n steps (chunk steps each) starting at step `first`."""
    import torch
    graphs = []
    with torch.cuda.stream(stream):
        for c0 in range(0, n, chunk):
            g = torch.cuda.CUDAGraph()
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for i in range(c0, min(n, c0 + chunk)):
                    if before_step is not None:
                        before_step(i)
                    step(first + i)
            graphs.append(g)
    return graphs


def timed_replay(graphs, K, chunk, stream, dev, world):
    """Replay the graphs (K steps) between two events on their stream,
    bracketed by a barrier and a device synchronisation on both sides; an
    event after each graph gives the per-step time of every chunk.  Returns
    (slowest rank's ms, per-chunk ms per step, wall start, wall end)."""
    import torch
    import torch.distributed as dist
    for g in graphs[:2]:
        g.replay()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    chunk_ev = [torch.cuda.Event(enable_timing=True) for _ in graphs]
    wall0 = time.time()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for g, ce in zip(graphs, chunk_ev):
            g.replay()
            ce.record(stream)
        t1.record(stream)
    torch.cuda.synchronize(dev)
    wall1 = time.time()
    if world > 1:
        dist.barrier()
    chunk_ms, prev = [], t0
    for ci, ce in enumerate(chunk_ev):
        n_steps = min(chunk, K - ci * chunk)
        chunk_ms.append(prev.elapsed_time(ce) / n_steps)
        prev = ce
    return max_over_ranks(t0.elapsed_time(t1), world, dev), chunk_ms, wall0, wall1


STAGES = ["permute", "quantize", "gateup", "down", "combine"]


def stage_times(bqe, layer, step, first, n, stream):
    """Per-stage device times (ms) from a separate, untimed pass: n more
    steps captured with the library's stage events on every step (the
    events sit between the stage kernels, so this pass is not the timed one)."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n)]
    with torch.cuda.stream(stream):
        for e6 in evs:  # events must exist on the stream before the capture
            for e in e6:
                e.record(stream)
    graphs = capture(step, first, n, n, stream, before_step=lambda i: bqe.moe_set_stage_events(layer, evs[i]))
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    st = np.array([[e6[i].elapsed_time(e6[i + 1]) for i in range(5)] for e6 in evs])
    return dict(zip(STAGES, st.mean(0).tolist()))


def clocked(fn):
    """Run fn() with nvidia-smi sampling the SM clocks; returns (fn(), clocks)."""
    import torch
    sampler = ClockSampler(gpu_uuid(torch.cuda.current_device()))
    time.sleep(0.3)
    r = fn()
    rows = sampler.stop()
    wall0, wall1 = r[2], r[3]
    in_region = [row for row in rows if _ts_in(row[0], wall0, wall1)]
    clocks = ClockSampler.summary(in_region if in_region else rows)
    clocks["window"] = "timed region" if in_region else "around the timed region"
    return r, clocks


def gemv_alu(cfg, touched, kernel_ms, clocks):
    """The CUDA-core decode kernel against its arithmetic ceiling: weight
    elements per SM clock (the touched experts' 3 H I elements over the
    kernel's duration at the median SM clock of the timed region) beside the
    e2m1 dot-product rate measured here (libmoe_peaks)."""
    import torch
    from block_quantized_expert_gb300 import peaks as pk
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = clocks.get("sm_mhz") or 2070.0
    elems = touched * 3.0 * cfg.H * cfg.I
    achieved = elems / (kernel_ms * 1e-3 * mhz * 1e6 * sms)
    peak = pk.dot_e2m1_el_per_clk()
    return {"unit": "weight elements per SM clock", "achieved": round(achieved, 1), "peak": round(peak, 1),
            "frac": round(achieved / peak, 4), "sm_mhz": mhz,
            "peak_source": "e2m1 x f16 -> fp32 block dot products on the CUDA cores (libmoe_peaks "
                           "peak_dot_e2m1) measured in this run, of measured"}


def load_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except OSError:
        return {}


def roofline(cfg, dom, kernel_ms, byts, rows, peaks, mma_peak=None):
    """Roofline of the dominant kernel: algorithmic bytes (or flops) per
    launch over its measured duration, against the measured peak."""
    hbm = peaks.get("hbm_gbs", 6800.0)
    achieved = byts[dom] / (kernel_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 4), "kernel_ms": round(kernel_ms, 6),
            "algorithmic_bytes_per_launch": int(byts[dom]),
            "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs), of measured" if "hbm_gbs" in peaks
            else "fallback 6.8 TB/s, of fallback"}
    if dom in ("gateup", "down"):
        H, I = cfg.H, cfg.I
        flops = {"gateup": rows * 4.0 * H * I, "down": rows * 2.0 * H * I}[dom]
        if cfg.shared and dom == "down":  # the down stage also runs the shared expert's two GEMMs
            flops += cfg.T * 6.0 * H * I
        tflops = flops / (kernel_ms * 1e-3) / 1e12
        # the recipe's figure: the fp8-class block-scaled MMA at twice the
        # measured bf16 rate (sustained: the kernel runs inside a long step)
        tpeak = 2.0 * peaks.get("bf16_tflops_sustained", 1700.0)
        tensor = {"tflops": round(tflops, 1), "algorithmic_flops_per_launch": flops,
                  "peak_2x_bf16_sustained": round(tpeak, 1),
                  "frac_2x_bf16_sustained": round(tflops / tpeak, 4)}
        if mma_peak:
            tensor.update({"peak_mxf8f6f4_measured": round(mma_peak, 1),
                           "frac_mxf8f6f4_measured": round(tflops / mma_peak, 4)})
        roof["tensor"] = tensor
        ref = mma_peak or tpeak
        if tflops / ref > achieved / hbm:
            roof.update({"bound": "tensor", "achieved": round(tflops, 1), "peak": round(ref, 1),
                         "unit": "TFLOP/s", "frac": round(tflops / ref, 4),
                         "peak_source": ("block-scaled MMA loop (libmoe_peaks, kind::mxf8f6f4, M128 N256 "
                                         "K32) measured in this run, of measured") if mma_peak else
                                        "measured bf16_tflops_sustained x 2 (fp8 / bf16 nominal ratio), of measured"})
    return roof


def run_ours(args, cfg, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import block_quantized_expert_gb300 as bqe
    from workloads import make_weights

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    K = args.steps if args.steps is not None else default_steps(cfg)
    W = args.warmup if args.warmup is not None else (64 if cfg.T == 1 else 3)
    W = max(W, 3)

    w = make_weights(cfg)
    layer = make_layer(bqe, cfg, w, dev, cfg.T, args.path, args.prune_t, args.decode_kernel)
    decode_kind = bqe.moe_decode_info(layer) if cfg.T == 1 else 0
    # distinct inputs: one token per step for decode, else a few batches cycled
    S = (K + W) if cfg.T == 1 else min(K + W, 4)
    wl = Workload(bqe, cfg, layer, dev, S, rank_seed(cfg, rank))
    avg_touched, rows = wl.touched()
    for i in range(W):
        wl.step(i)
    bqe.moe_check(layer)

    # the timed region: K steps as chunked CUDA graphs, nothing else inside
    stream = torch.cuda.Stream(device=dev)
    launches0 = bqe.moe_kernel_launches(layer)
    graphs = capture(wl.step, W, K, args.graph_chunk, stream)
    launches = bqe.moe_kernel_launches(layer) - launches0   # kernels per replay of all graphs
    (ms, chunk_ms, wall0, wall1), clocks = clocked(lambda: timed_replay(graphs, K, args.graph_chunk, stream,
                                                                         dev, world))
    bqe.moe_check(layer)
    del graphs

    if args.trace:
        trace_report(bqe, layer, wl.step, K + W, dev)

    byts = algorithmic_bytes(cfg, avg_touched, rows)
    step_bytes = byts["gateup"] + byts["down"]
    peaks = load_peaks()
    if launches == K:
        # one kernel per call (the whole-layer decode kernel): its average
        # duration is the timed region over the K calls
        dom, kernel_ms, stage_ms = "layer", ms / K, None
        byts["layer"] = step_bytes
        kernel = DECODE_KERNELS[decode_kind]
    else:
        stage_ms = stage_times(bqe, layer, wl.step, W + K, min(K, 32), stream)
        dom = max(("gateup", "down"), key=lambda n: stage_ms[n])
        kernel_ms, kernel = stage_ms[dom], f"{dom} GEMM"
    roof = roofline(cfg, dom, kernel_ms, byts, rows, peaks)
    roof["kernel"] = kernel
    roof["traffic"] = profiled_traffic(cfg, dom, decode_kind) if not args.prune_t else None
    if dom == "layer" and decode_kind == 1:
        roof["alu"] = gemv_alu(cfg, avg_touched, roof["kernel_ms"], clocks)
    roof["hbm_frac_whole_step"] = round(step_bytes / (ms / K * 1e-3) / 1e9 / roof["peak"], 4) \
        if roof["unit"] == "GB/s" else None

    res = {"metric": METRIC, "value": job_rate(world, K * cfg.T, ms), "unit": UNIT, "n_gpus": world,
           "steps": K, "warmup": W, "ms_per_step": ms / K, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None,
           "dtype": "mxfp4 x mxfp8 -> f32 accumulate", "data": "synthetic (seeded)",
           "config": config_json(cfg, args, world),
           "gpu_launches": int(launches),
           "per_step_spread": chunk_spread(chunk_ms),
           "experts_touched_per_step": avg_touched,
           "roofline": roof,
           "clocks": clocks}
    if stage_ms:
        res["stage_ms_untimed_pass"] = {k: round(v, 5) for k, v in stage_ms.items()}

    if not args.no_e2e:
        res["e2e"] = run_e2e(args, cfg, layer, wl.tokens, S, K, W, world, dev)
    layer.close()
    del wl
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and cfg.index == 1 and not args.no_per_config and not args.prune_t:
        res["per_config"] = per_config(args, bqe, dev, peaks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(cfg, w, wl_tokens_for_cpu(cfg, rank), args.cpu_seconds, args.prune_t)
    if world > 1:
        dist.destroy_process_group()
    return res


def wl_tokens_for_cpu(cfg, rank):
    from workloads import make_tokens
    # enough tokens for the oracle's time budget (~60 tokens/s per 16 cores)
    return make_tokens(cfg, seed=rank_seed(cfg, rank), n=max(cfg.T, 2048))


PER_CONFIG = [  # (config, router, timed steps)
    (2, "hash", 128), (2, "learned", 128), (3, None, 48), (4, None, 16),
    (6, None, 32), (7, None, 4)]  # the NVFP4-style weight variant (CUDA-core GEMMs)


def per_config(args, bqe, dev, peaks):
    """One time-boxed record per other workload (batched decode with the hash
    and the learned router, pp512, prefill 8192 with the shared expert):
    tokens/s over the timed steps, the dominant GEMM's time from an untimed
    instrumented pass and its roofline fraction (prefill 8192 against the
    block-scaled MMA peak measured here, right after its timed region)."""
    import torch
    from block_quantized_expert_gb300 import peaks as pk
    from workloads import CONFIGS, make_weights

    recs = []
    layer = None
    layer_for = None
    for ci, router, K in PER_CONFIG:
        cfg = CONFIGS[ci]
        t_start = time.time()
        key = (cfg.shared, cfg.T if cfg.shared else 512, cfg.wfmt)
        if layer_for != key:
            if layer is not None:
                layer.close()
                torch.cuda.empty_cache()
            layer = make_layer(bqe, cfg, make_weights(cfg), dev, key[1], args.path if cfg.wfmt == "mxfp4" else "auto")
            layer_for = key
        W = 3
        wl = Workload(bqe, cfg, layer, dev, min(K + W, 4), cfg.default_seed, router=router)
        avg_touched, rows = wl.touched(4)
        for i in range(W):
            wl.step(i)
        bqe.moe_check(layer)
        stream = torch.cuda.Stream(device=dev)
        launches0 = bqe.moe_kernel_launches(layer)
        graphs = capture(wl.step, W, K, K, stream)
        launches = bqe.moe_kernel_launches(layer) - launches0
        (ms, _, w0, w1), clocks = clocked(lambda: timed_replay(graphs, K, K, stream, dev, 1))
        del graphs
        mma_peak = None
        if cfg.index == 4:
            mma_peak = pk.mma_mx_tflops(iters=60000, reps=3)
        byts = algorithmic_bytes(cfg, avg_touched, rows)
        if launches == K:
            # one whole-layer decode kernel per step: its average duration is the
            # timed region over the K steps
            stage_ms = None
            byts["layer"] = byts["gateup"] + byts["down"]
            roof = roofline(cfg, "layer", ms / K, byts, rows, peaks, mma_peak)
            roof["kernel"] = DECODE_KERNELS[bqe.moe_decode_info(layer)]
            if bqe.moe_decode_info(layer) == 1:
                roof["alu"] = gemv_alu(cfg, avg_touched, ms / K, clocks)
        else:
            stage_ms = stage_times(bqe, layer, wl.step, W + K, min(K, 16), stream)
            dom = max(("gateup", "down"), key=lambda n: stage_ms[n])
            roof = roofline(cfg, dom, stage_ms[dom], byts, rows, peaks, mma_peak)
            roof["kernel"] = f"{dom} GEMM ({'k_gemm_cc, CUDA cores' if cfg.wfmt == 'nvfp4' else 'k_gemm_tc'})"
        bqe.moe_check(layer)
        recs.append({"workload": cfg.name if router is None else f"{cfg.name.rsplit('_', 1)[0]}_{router}",
                     "tokens_per_step": cfg.T, "router": router or cfg.router, "shared_expert": cfg.shared,
                     "weights": "NVFP4-style e2m1 + e4m3 /16 + fp32 per matrix (CUDA cores)"
                     if cfg.wfmt == "nvfp4" else "MXFP4 e2m1 + UE8M0 /32",
                     "value": job_rate(1, K * cfg.T, ms), "unit": UNIT, "steps": K, "warmup": W,
                     "ms_per_step": round(ms / K, 6), "experts_touched_per_step": avg_touched,
                     **({"stage_ms_untimed_pass": {k: round(v, 5) for k, v in stage_ms.items()}} if stage_ms else {}),
                     "gpu_launches": int(launches),
                     "roofline": roof, "clocks": clocks,
                     "l2": "weights of the touched experts larger than L2; 4 input batches cycled",
                     "wall_s": round(time.time() - t_start, 1)})
        del wl
    if layer is not None:
        layer.close()
    torch.cuda.empty_cache()
    return recs


# The whole-layer decode kernels (moe_decode_info codes), and for each the
# committed ncu capture of its DRAM bytes per launch with the sources it is
# valid for
DECODE_KERNELS = {1: "whole-layer decode kernel, CUDA-core GEMV (k_decode_gemv)",
                  2: "whole-layer decode kernel, tcgen05 (k_decode)"}
PROFILE_COUNTERS = {1: ("decode_t1_k_decode_gemv_counters.json",
                        ["decode_gemv.cu", "common.cuh", "tc_ptx.cuh", "route.cuh", "layer.h"]),
                    2: ("decode_t1_k_decode_counters.json",
                        ["gemm_tc.cu", "common.cuh", "tc_ptx.cuh", "route.cuh", "layer.h"])}


def kernel_sources_sha256(sources):
    import hashlib
    h = hashlib.sha256()
    for name in sorted(sources):
        with open(os.path.join(ROOT, "block_quantized_expert_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(cfg, dom, decode_kind):
    if dom != "layer" or cfg.index != 1 or decode_kind not in PROFILE_COUNTERS:
        return None
    fname, sources = PROFILE_COUNTERS[decode_kind]
    try:
        rec = json.load(open(os.path.join(ROOT, "profiles", fname)))
    except (OSError, ValueError):
        return None
    if rec.get("kernel_sources_sha256") != kernel_sources_sha256(sources):
        return None  # the kernel changed since the counters were taken
    return int(rec["dram_bytes_per_launch"])


def trace_report(bqe, layer, step, i, dev):
    """Timeline of one more call: front kernel and GEMM launches (stderr)."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n_tr = 3  # the last three calls of the graph are traced
    bufs = [torch.zeros(max(48 * sms + 4, 8 * sms + 1024), dtype=torch.int64, device=dev) for _ in range(n_tr)]
    stream = torch.cuda.Stream(device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for k in range(4):
            step(i + k)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):  # as in the timed region: graph replay
            for k in range(8):
                if k >= 8 - n_tr:
                    bqe.moe_set_trace(layer, bufs[k - 8 + n_tr])
                step(i + k)
        g.replay()
        stream.synchronize()
    # call to call: first entry of each traced call after the first
    ent = [b.cpu().numpy().astype(np.float64)[: sms * 12].reshape(sms, 12) for b in bufs]
    if all(e[:, 0].max() > 0 for e in ent):
        print("TRACE", json.dumps({"launch": "call_to_call", "entry_gap_us": [
            round((ent[j + 1][:, 0].min() - ent[j][:, 0].min()) / 1e3, 2) for j in range(n_tr - 1)],
            "exit_to_next_entry_us": [round((ent[j + 1][:, 0].min() - ent[j][:, 1].max()) / 1e3, 2)
                                      for j in range(n_tr - 1)]}), file=sys.stderr, flush=True)
    buf = bufs[-1]
    raw = buf.cpu().numpy().astype(np.float64)
    t = raw[: 4 * sms * 12].reshape(4, sms, 12)
    fr = raw[4 * sms * 12:]
    t0 = fr[0] if fr[0] > 0 else t[0, :, 0].min()
    if fr[0] > 0:
        print("TRACE", json.dumps({"launch": "front", "entry_us": 0.0, "wait_end_us": round((fr[1] - t0) / 1e3, 2),
                                   "exit_us": round((fr[2] - t0) / 1e3, 2)}), file=sys.stderr, flush=True)
    if t[0, :, 9].max() > 0:  # the whole-layer decode kernel
        e0 = t[0, :, 0].min()
        rep = {"launch": "decode", "percentiles": [0, 50, 100]}
        for key, c in (("entry", 0), ("wait_end", 8), ("routed", 9), ("producer_start", 2),
                       ("first_weights", 3), ("gateup_issued", 4), ("gateup_written", 10),
                       ("h_flags_seen", 5), ("h_landed", 6), ("down_issued", 7), ("down_written", 11),
                       ("exit", 1)):
            v = t[0, :, c]
            v = v[v > 0]
            if v.size:
                rep[key] = [round((np.percentile(v, p) - e0) / 1e3, 2) for p in (0, 50, 100)]
        print("TRACE", json.dumps(rep), file=sys.stderr, flush=True)
        if t[0, :, 11].max() <= 0:  # the phase stamps are not compiled in
            return
        # the CTAs that finish last: their stamps (us from the first entry)
        last = np.argsort(-t[0, :, 11])[:8]
        slow = {int(b): [round((t[0, b, c] - e0) / 1e3, 2) if t[0, b, c] > 0 else None
                         for c in (2, 3, 4, 10, 5, 6, 7, 11)] for b in last}
        print("TRACE", json.dumps({"launch": "decode_last_ctas", "columns": [
            "producer_start", "first_weights", "gateup_issued", "gateup_written", "down_loads_start",
            "h_landed", "down_issued", "down_written"], "ctas": slow}), file=sys.stderr, flush=True)
        return
    names = ["gateup", "down", "shared_gateup", "shared_down"]
    for j in range(4):
        if t[j, :, 0].max() == 0:
            continue
        dur = (t[j, :, 1] - t[j, :, 0]) / 1e3
        rep = {"launch": names[j], "first_entry_us": round((t[j, :, 0].min() - t0) / 1e3, 2),
               "wait_end_us": round((t[j, :, 8].min() - t0) / 1e3, 2),
               "last_exit_us": round((t[j, :, 1].max() - t0) / 1e3, 2),
               "cta_us_mean": round(dur.mean(), 2),
               "producer_wait_free_us": round(t[j, :, 2].mean() / 1e3, 2),
               "mma_wait_data_us": round(t[j, :, 3].mean() / 1e3, 2),
               "mma_wait_acc_us": round(t[j, :, 4].mean() / 1e3, 2),
               "epi_wait_acc_us": round(t[j, :, 5].mean() / 1e3, 2),
               "epi_work_us": round(t[j, :, 6].mean() / 1e3, 2),
               "stages_per_cta": round(t[j, :, 7].mean(), 1)}
        print("TRACE", json.dumps(rep), file=sys.stderr, flush=True)


def _ts_in(ts, a, b):
    try:
        t = time.mktime(time.strptime(ts.split(".")[0], "%Y/%m/%d %H:%M:%S"))
        return a - 1.0 <= t <= b + 1.0
    except Exception:
        return False


def run_e2e(args, cfg, layer, tk, S, K, W, world, dev):
    """Same steps through moe_forward_host: each step copies its x and logits
    from page-locked host memory and reads the layer output back."""
    import torch
    import torch.distributed as dist

    import block_quantized_expert_gb300 as bqe

    if cfg.router == "hash":
        return {"value": None, "unit": UNIT, "note": "host entry covers the learned router only"}
    xh = torch.from_numpy(tk.x_bits.view(np.int16).reshape(S, cfg.T, cfg.H).copy()).pin_memory()
    lh = torch.from_numpy(tk.logits.reshape(S, cfg.T, cfg.E).copy()).pin_memory()
    oh = torch.empty((cfg.T, cfg.H), dtype=torch.float32).pin_memory()
    stream = torch.cuda.Stream(device=dev)
    graphs = []
    with torch.cuda.stream(stream):
        for i in range(W):
            bqe.moe_forward_host(layer, xh[i % S], lh[i % S], oh)
        stream.synchronize()
        for c0 in range(0, K, args.graph_chunk):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(c0, min(K, c0 + args.graph_chunk)):
                    j = (W + i) % S
                    bqe.moe_forward_host(layer, xh[j], lh[j], oh)
            graphs.append(g)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for g in graphs:
            g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    return {"value": job_rate(world, K * cfg.T, ms), "unit": UNIT,
            "h2d_bytes_per_step": cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4,
            "d2h_bytes_per_step": cfg.T * cfg.H * 4,
            "path": ("moe_forward_host (pinned host in/out, CUDA graphs; one token: the decode kernel "
                     "reads x and logits and writes out in mapped host memory, no copy nodes)"
                     if cfg.T == 1 else "moe_forward_host (pinned host in/out, CUDA graphs)")}


# ------------------------------------------------------------- CPU oracle --
def oracle_rate(cfg, w, tk, seconds, prune=None, max_tokens=None, warmup_calls=1):
    """Tokens/s of the fp64 oracle (route + layer) on the host cores, on a
    sample sized to about `seconds` of work and at most `max_tokens` tokens,
    after `warmup_calls` untimed calls on one token each."""
    from oracle import oracle as orc

    for n in ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s"):
        np.asarray(getattr(w, n)).sum()   # page the weights in before timing
    T = cfg.T
    n_all = tk.logits.shape[0]

    def run(n):
        tok = min(n, n_all)
        lg, xb = tk.logits[:tok], tk.x_bits[:tok]
        t = time.perf_counter()
        ids, wt = orc.route_learned(lg, cfg.k, cfg.w_scale)
        if prune:
            ids, wt = orc.route_prune(ids, wt, *prune)
        orc.layer_forward(w, xb, ids, wt)
        return tok, time.perf_counter() - t

    # calibrate on two tokens per thread (the oracle runs tokens in parallel),
    # after the warm-up calls (the first loads the library and its tables)
    for _ in range(max(1, warmup_calls)):
        run(1)
    cap = n_all if max_tokens is None else max(1, min(n_all, max_tokens))
    n0, t0 = run(min(2 * orc.max_threads(), cap))
    per = t0 / n0
    n = int(max(min(4, cap), min(cap, seconds / max(per, 1e-9))))
    n, t = run(n)
    return n, t, orc.max_threads(), T


def cpu_baseline(cfg, w, tk, seconds, prune=None):
    n, t, cores, T = oracle_rate(cfg, w, tk, seconds, prune)
    return {"value": round(n / t, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} tokens of the {cfg.name} workload (tokens are independent; "
                      f"route + layer per token), {t:.1f} s"}


def run_reference(args, cfg, rank, world):
    if rank != 0:
        return None
    from workloads import make_tokens, make_weights

    K = args.steps if args.steps is not None else default_steps(cfg)
    W = args.warmup if args.warmup is not None else 3
    w = make_weights(cfg)
    tk = make_tokens(cfg, n=min(cfg.T * (K + W), 4096) if cfg.T == 1 else cfg.T)
    budget = 60.0
    # W untimed warm-up steps (one token each), then at most K steps' tokens,
    # bounded to about `budget` seconds (tokens are independent; the oracle
    # runs them in parallel over the host cores)
    n, t, cores, T = oracle_rate(cfg, w, tk, budget, args.prune_t, max_tokens=K * cfg.T, warmup_calls=W)
    value = n / t
    steps_done = max(1, n // cfg.T)
    res = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
           "steps": steps_done, "warmup": W, "ms_per_step": 1e3 * t * cfg.T / n,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded)", "config": config_json(cfg, args, world),
           "impl": "reference",
           "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": cores,
                            "kind": "oracle",
                            "sample": f"{n} tokens (of the {K * cfg.T} in {K} steps; time-bounded "
                                      f"~{budget:.0f} s) of the {cfg.name} workload after {W} "
                                      f"warm-up tokens"},
           "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    return res


def main():
    args = parse()
    from workloads import CONFIGS

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    cfg = CONFIGS[args.config]
    if args.experts is not None:
        import dataclasses
        cfg = dataclasses.replace(cfg, E=args.experts, name=f"{cfg.name}_e{args.experts}")
    if args.impl == "reference":
        res = run_reference(args, cfg, rank, world)
    else:
        res = run_ours(args, cfg, rank, world, local_rank)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
