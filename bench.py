"""Benchmark of the low-rank bottleneck sublayer on GB300.

One step = forward + backward of one low-rank SwiGLU MLP block (T 16384 tokens,
d 2048, f 5632, r 512, bf16 storage, fp32 accumulation) with low-rank activation
checkpointing: online-RMSNorm grouped gate/up GEMM, SwiGLU dual GEMM, down pair
with residual, and the whole backward including the re-forward of the [T, f]
tensors from the saved [T, r] pre-activations.  Inputs are resident in HBM; L2
is flushed (a 512 MB write) before every timed step, outside the timed events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--mode ckpt|full] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica on its own GPU (the path needs no exchange between GPUs): value is the
tokens of all ranks over the slowest rank's time.  Besides the headline (the
single block above), the line carries records of the metric's other workloads
at full size, timed after the headline on the same GPU: ``attn_proj`` (q/k/v
group + o-projection, d 4096, r 1024), ``stack24`` (24 blocks + MSE, with and
without checkpointing, peak device memory of each), ``sweep`` (144 shapes), and the
widening workloads ``block`` (the low-rank transformer block at LLaMA-7B widths) and
``attention`` (its causal attention alone); ``--no-extras`` leaves them out.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "low-rank block fwd+bwd tokens/s on 1 GB300; % of per-shape roofline"
NOMINAL = {"tflops": 2250.0, "hbm_gbs": 8000.0}
FALLBACK = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, averaged over the launches of
# one step) from an ncu capture of the named kernel.  A figure holds only for the kernel sources it was
# taken on: TRAFFIC_SOURCES are hashed at run time and a mismatch reports traffic as null.
TRAFFIC_SOURCES = ["common.cuh", "epilogues.cuh", "gemm.h", "umma_gemm.cuh", "umma_launch.cuh", "lowrank_api.cu"]
NCU_TRAFFIC = {
    "umma_swiglu_rebwd_bn256": {"bytes_per_launch": 105.1e6 + 498.5e6,
                                "sources_sha256": "cb44c26bd0a709158dd92d7e717b74d34f2b6601324d51bc176e09e4c61851c5",
                                "profile": "profiles/mlp_block_T16384_d2048_f5632_r512_launches.md"},
    "umma_f32_bn256": {"bytes_per_launch": 402.7e6 + 9.8e6,
                       "sources_sha256": "cb44c26bd0a709158dd92d7e717b74d34f2b6601324d51bc176e09e4c61851c5",
                       "profile": "profiles/mlp_block_T16384_d2048_f5632_r512_launches.md"},
}


# Algorithmic bytes per launch of a dominant kernel: the operands it must read and the outputs the
# method defines, without the [T, f] intermediates (h, a, b) this design materialises (a fully fused
# implementation need not store them).
ALG_BYTES = {
    "umma_swiglu_bn256": lambda s: 2.0 * (2 * s.T * s.r + 2 * s.f * s.r),
    # three-accumulator re-forward + SwiGLU backward: z_g, z_u, du_down [T, r]; B_gate, B_up, A_down
    "umma_swiglu_rebwd_bn256": lambda s: 2.0 * (3 * s.T * s.r + 3 * s.f * s.r),
    # weight gradients, the mean of the step's two launches: the grouped one reads da, db, h [T, f],
    # z_g, z_u, du_down, z_down [T, r] and dout [T, d] and writes dB_gate, dB_up, dA_down, dB_down (fp32);
    # the split-K one reads s du [T, 2r] and x [T, d] and writes dA'_gate;up [2r, d] (fp32)
    "umma_f32_bn256": lambda s: 0.5 * (2.0 * (3 * s.T * s.f + 4 * s.T * s.r + s.T * s.d) + 4.0 * (3 * s.f * s.r + s.d * s.r)
                                       + 2.0 * (2 * s.T * s.r + s.T * s.d) + 4.0 * (2 * s.r * s.d)),
}


def kernel_sources_sha256() -> str:
    import hashlib

    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "rank_bottleneck_block_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ncu_traffic(kernel: str):
    rec = NCU_TRAFFIC.get(kernel)
    if rec is None or rec["sources_sha256"] != kernel_sources_sha256():
        return None, "no ncu capture of the current kernel sources"
    return rec["bytes_per_launch"], rec["profile"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d["bf16_tflops_sustained"],
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return dict(FALLBACK, source="fallback")


# ----------------------------------------------------------------- workload
def workload(mode: str):
    from rank_bottleneck_block_gb300 import inputs as I

    s = I.MLP_BLOCK_BF16
    T, d, f, r = s.T, s.d, s.f, s.r
    fwd = 2.0 * T * (2 * r * d + 2 * f * r + r * f + d * r)  # K1 (gate;up), K2 (dual), A_down, B_down
    flops = 3.0 * fwd + (4.0 * T * r * f if mode == "ckpt" else 0.0)
    params = 2 * r * d + 2 * f * r + r * f + d * r
    act = 2.0 * T * d * 4  # read x and dout, write out and dx
    saved = (3 * r * 2 + 4) * T * 2.0 if mode == "ckpt" else (3 * r * 2 * 2 + 3 * f * 2 + 4) * T * 2.0
    nbytes = act + 2.0 * params + 4.0 * params + 2.0 * d + 4.0 * d + saved
    cfg = {"workload": f"low-rank SwiGLU MLP block fwd+bwd, T={T} d={d} f={f} r={r}, "
                       f"{'low-rank activation checkpointing' if mode == 'ckpt' else 'no checkpointing'}",
           "tokens": T, "d": d, "f": f, "r": r, "mode": mode, "seed": 0,
           "l2": "flushed before every timed step (512 MB write, outside the timed events)"}
    return s, cfg, flops, nbytes


# ------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_uuid=None):
        self.p = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if dev_uuid:
            cmd += ["-i", dev_uuid]
        try:
            self.p = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, smax, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None, "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------ CPU baseline
def oracle_tokens_per_s(shape, rows: int, min_seconds: float, mode: str):
    """The fp64 oracle's fwd+bwd of the block on `rows` tokens of the workload (same d, f, r), repeated
    until at least min_seconds; returns (tokens/s, reps, seconds)."""
    import oracle.lowrank_oracle as O
    from rank_bottleneck_block_gb300 import inputs as I

    sub = I.MlpShape(T=rows, d=shape.d, f=shape.f, r=shape.r, dtype=shape.dtype)
    case = I.make_mlp_case(sub, seed=0)
    om = O.CKPT if mode == "ckpt" else O.FULL
    reps, t0 = 0, time.perf_counter()
    while True:
        _, saved = O.mlp_block_fwd(case["x"], case["g"], case, sub.eps, om)
        O.mlp_block_bwd(case["g"], case, saved, case["G"], sub.eps)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            return rows * reps / el, reps, el


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# ------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo", rank=rank, world_size=ws)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(tokens_per_rank: int, ws: int, seconds_max: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return tokens_per_rank * ws / seconds_max


# --------------------------------------------------------------- our arm
def run_ours(a, ws, rank, local):
    import torch

    from rank_bottleneck_block_gb300 import build as B

    if rank == 0 or ws == 1:
        B.build()
    barrier(ws)
    from rank_bottleneck_block_gb300 import inputs as I
    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import MlpBlock

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shape, cfg, flops, nbytes = workload(a.mode)
    mode = L.LR_SAVE_CKPT if a.mode == "ckpt" else L.LR_SAVE_FULL
    case = I.make_mlp_case(shape, seed=0)
    blk = MlpBlock(shape, case, mode, device=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    for _ in range(a.warmup):
        blk.step()
    torch.cuda.synchronize()
    L.lr_check_device_error()

    # ------------------------------------------------ per-kernel pass (untimed)
    # Events around every launch break the overlap of each kernel's start with the
    # previous kernel's tail, so the per-kernel table comes from a pass of its own and
    # the timed steps carry events around the dominant kernel only.
    prof_steps = max(3, min(a.steps, 20))
    L.lr_profile_filter(None)
    L.lr_profile_start()
    for i in range(prof_steps):
        flush.fill_(i & 0xFF)
        blk.step()
    torch.cuda.synchronize()
    prof_all = L.lr_profile_stop()
    gemms = {k: v for k, v in prof_all.items() if v["flops"] > 0}
    dom_name = max(gemms.items(), key=lambda kv: kv[1]["ms"])[0]

    # ------------------------------------------------ device-resident timing
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(a.steps)]
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    clk = ClockSampler(uuid)
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    n0 = L.lr_launch_count()
    L.lr_profile_filter(dom_name)
    L.lr_profile_start()
    for i in range(a.steps):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        blk.step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    prof = L.lr_profile_stop()
    L.lr_profile_filter(None)
    launches = L.lr_launch_count() - n0
    L.lr_check_device_error()
    step_ms = [s.elapsed_time(e) for s, e in evs]
    total_s = sum(step_ms) / 1e3
    total_s_max = max_over_ranks(total_s, ws)
    ms_per_step = total_s_max * 1e3 / a.steps
    value = aggregate(shape.T * a.steps, ws, total_s_max)

    # ------------------------------------------------ end to end (host buffers)
    # Inputs x and dout come from pinned host memory and out, dx go back every step; the
    # copies of neighbouring steps run on two copy streams and overlap the compute.
    from rank_bottleneck_block_gb300.runner import HostPipeline

    xh = case["x"].pin_memory()
    gh = case["G"].pin_memory()
    outh = torch.empty_like(xh).pin_memory()
    dxh = torch.empty_like(xh).pin_memory()
    pipe = HostPipeline(blk)
    pipe.run([xh], [gh], outh, dxh, 3, stream)  # warm-up of the copy path
    e2e_steps = max(3, min(a.steps, 200))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    ev0.record(stream)
    pipe.run([xh], [gh], outh, dxh, e2e_steps, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    L.lr_check_device_error()
    # The clock record spans the timed steps and these end-to-end steps (a timed region of a few tens of
    # milliseconds alone holds at most one sample of nvidia-smi's loop).
    clocks = clk.stop()
    clocks["window"] = "timed steps, then the end-to-end steps"
    e2e_s = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, ws)
    h2d, d2h = pipe.bytes_per_step()
    e2e = {"value": aggregate(shape.T * e2e_steps, ws, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "api": "lr_mlp_fwd + lr_mlp_bwd on device copies of pinned host x and dout, out and dx copied back, "
                  "every step; copies on two side streams overlap the neighbouring steps' compute"}

    # ------------------------------------------------ rooflines
    pk = peaks()
    dom = prof[dom_name]
    achieved_tf = dom["flops"] / (dom["ms"] / 1e3) / 1e12
    # The dominant kernel runs for well under a millisecond inside a step of about a millisecond:
    # the burst figure of the measured peaks is its denominator.
    roofline = {"kernel": dom_name, "bound": "tensor", "achieved": round(achieved_tf, 1),
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": round(achieved_tf / pk["bf16_tflops"], 4),
                "peak_kind": f"bf16 dense, burst ({pk['source']})",
                "frac_nominal": round(achieved_tf / NOMINAL["tflops"], 4),
                "launches": dom["launches"], "avg_launch_us": round(1e3 * dom["ms"] / dom["launches"], 2),
                "flops_per_launch": dom["flops"] / dom["launches"],
                "share_of_step": round(dom["ms"] / a.steps / ms_per_step, 4),
                "traffic": None}
    alg = ALG_BYTES.get(dom_name)
    if alg:
        roofline["algorithmic_bytes"] = alg(shape)
    traffic, tsrc = ncu_traffic(dom_name)
    roofline["traffic"] = traffic
    roofline["traffic_source"] = tsrc
    if traffic:
        roofline["traffic_gbs"] = round(traffic / (dom["ms"] / dom["launches"] / 1e3) / 1e9, 1)
        if alg:
            roofline["traffic_over_algorithmic"] = round(traffic / roofline["algorithmic_bytes"], 2)
    ms_step_s = ms_per_step / 1e3
    t_nom = max(flops / (NOMINAL["tflops"] * 1e12), nbytes / (NOMINAL["hbm_gbs"] * 1e9))
    t_meas = max(flops / (pk["bf16_tflops"] * 1e12), nbytes / (pk["hbm_gbs"] * 1e9))
    block = {"frac_nominal": round(t_nom / ms_step_s, 4),
             "peak_nominal": "2.25 PFLOP/s dense bf16, 8 TB/s HBM (the per-shape roofline of the metric)",
             "frac_measured": round(t_meas / ms_step_s, 4),
             "peak_measured": f"{pk['bf16_tflops']} TFLOP/s bf16 burst, {pk['hbm_gbs']} GB/s ({pk['source']})",
             "flops_per_step": flops, "bytes_per_step": nbytes, "tflops": round(flops / ms_step_s / 1e12, 1),
             "roofline_ms_nominal": round(t_nom * 1e3, 4), "roofline_ms_measured": round(t_meas * 1e3, 4)}
    kernels = {k: {"launches": v["launches"], "ms_per_step": round(v["ms"] / prof_steps, 4),
                   "share": round(v["ms"] / sum(w["ms"] for w in prof_all.values()), 4),
                   **({"tflops": round(v["flops"] / (v["ms"] / 1e3) / 1e12, 1)} if v["flops"] else
                      {"gbs": round(v["bytes"] / (v["ms"] / 1e3) / 1e9, 1)})}
               for k, v in sorted(prof_all.items(), key=lambda kv: -kv[1]["ms"])}
    kernels["_pass"] = (f"{prof_steps} untimed steps with events around every launch (they serialise "
                        f"launches, so the sum exceeds the timed step)")

    res = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws, "steps": a.steps,
           "warmup": a.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) "
                                                           "weights, g=1+N(0,0.1))",
           "config": dict(cfg, parallelism=f"replicas x{ws}" if ws > 1 else "single GPU"),
           "roofline": roofline, "block_roofline": block, "e2e": e2e, "gpu_launches": int(launches),
           "clocks": clocks, "kernels": kernels}
    # The other workloads of the metric at their full sizes, each with its own roofline fraction: the
    # attention projections, the 24-block stack in both save modes (with peak device memory), and the
    # 144-shape sweep.  The headline value above is the single-block workload alone.
    if rank == 0 and not a.no_extras:
        del pipe
        res["attn_proj"] = measure_attn_proj(pk, flush, stream, a.extra_steps, 3)
        res["stack24"] = measure_stack(pk, flush, stream, a.extra_steps, 3, dev)
        res["sweep"] = measure_sweep(pk, flush, stream, a.sweep_steps, 3)
        res["block"] = measure_block(pk, flush, stream, a.extra_steps, 3, dev)
        res["attention"] = measure_attention(pk, flush, stream, a.extra_steps, 3, dev)
        L.lr_check_device_error()
    if ws == 1 and not a.no_cpu_baseline:
        tps, reps, el = oracle_tokens_per_s(shape, a.cpu_rows, a.cpu_seconds, a.mode)
        res["cpu_baseline"] = {"value": round(tps, 2), "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                               "sample": f"fp64 numpy oracle fwd+bwd of the same block on {a.cpu_rows} of the "
                                         f"{shape.T} tokens, {reps} repetition(s) in {el:.1f} s; numpy BLAS "
                                         f"default threading"}
    if rank == 0:
        print(json.dumps(res), flush=True)


# ---------------------------------------------------- other workloads
def _time_steps(step, steps, warmup, flush, stream):
    import torch

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush.fill_(i & 0xFF)
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(s.elapsed_time(e) for s, e in evs) / steps


def _kernel_table(step, flush, stream, steps: int = 10):
    """Per-kernel device time from an untimed pass with CUDA events around every launch."""
    import torch

    from rank_bottleneck_block_gb300 import lowrank as L

    L.lr_profile_filter(None)
    L.lr_profile_start()
    for i in range(steps):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize()
    prof = L.lr_profile_stop()
    return {k: {"launches": v["launches"], "ms_per_step": round(v["ms"] / steps, 4),
                **({"tflops": round(v["flops"] / (v["ms"] / 1e3) / 1e12, 1)} if v["flops"] else
                   {"gbs": round(v["bytes"] / (v["ms"] / 1e3) / 1e9, 1)})}
            for k, v in sorted(prof.items(), key=lambda kv: -kv[1]["ms"])}


def _proj_flops_bytes(T, d_in, d_out, r, group, norm):
    f = 3.0 * 2.0 * T * r * (d_in + d_out) * group
    params = group * r * (d_in + d_out)
    b = 2.0 * T * d_in * 2 + 2.0 * T * d_out * group * 2  # x read, dx written; outs written, douts read
    b += 2.0 * params + 4.0 * params + (6.0 * d_in if norm else 0.0)
    b += (2.0 * T * group * r * 2 + (4.0 * T if norm else 0.0)) * 2  # saved u, z written and read
    return f, b


def _roofline(flops, nbytes, ms, pk):
    t_nom = max(flops / (NOMINAL["tflops"] * 1e12), nbytes / (NOMINAL["hbm_gbs"] * 1e9))
    t_meas = max(flops / (pk["bf16_tflops"] * 1e12), nbytes / (pk["hbm_gbs"] * 1e9))
    return {"tflops": round(flops / (ms / 1e3) / 1e12, 1), "roofline_ms_nominal": round(t_nom * 1e3, 4),
            "frac_nominal": round(t_nom / (ms / 1e3), 4), "frac_measured": round(t_meas / (ms / 1e3), 4),
            "bound": "tensor" if flops / (NOMINAL["tflops"] * 1e12) >= nbytes / (NOMINAL["hbm_gbs"] * 1e9) else "hbm"}


def measure_attn_proj(pk, flush, stream, steps, warmup, with_kernels=False):
    """The attention projections at LLaMA-7B width: q/k/v group (3 pairs, r 1024, d 4096, RMSNorm) and the
    o-projection (1 pair, no norm) on T 16384 tokens, fwd+bwd."""
    from rank_bottleneck_block_gb300 import inputs as I
    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import ProjGroup

    qkv = ProjGroup(I.ATTN_PROJ_BF16, I.make_proj_case(I.ATTN_PROJ_BF16, seed=0, device="cuda"))
    o = ProjGroup(I.ATTN_OPROJ_BF16, I.make_proj_case(I.ATTN_OPROJ_BF16, seed=1, device="cuda"))

    def step():
        qkv.step()
        o.step()

    ms = _time_steps(step, steps, warmup, flush, stream)
    L.lr_check_device_error()
    s1, s2 = I.ATTN_PROJ_BF16, I.ATTN_OPROJ_BF16
    f1, b1 = _proj_flops_bytes(s1.T, s1.d_in, s1.d_out, s1.r, s1.group, True)
    f2, b2 = _proj_flops_bytes(s2.T, s2.d_in, s2.d_out, s2.r, s2.group, False)
    res = {"workload": f"low-rank attention projections fwd+bwd: q/k/v group (3 pairs, r {s1.r}, d {s1.d_in}, "
                       f"RMSNorm) + o-projection (1 pair, no norm), T {s1.T}", "steps": steps,
           "ms_per_step": round(ms, 4), "tokens_per_s": round(s1.T / (ms / 1e3), 1),
           **_roofline(f1 + f2, b1 + b2, ms, pk)}
    if with_kernels:
        res["kernels"] = _kernel_table(step, flush, stream)
    del qkv, o
    return res


def measure_stack(pk, flush, stream, steps, warmup, dev):
    """24 residual low-rank SwiGLU MLP blocks + MSE, one training step, with low-rank activation
    checkpointing and without; peak device memory of each mode's buffers."""
    import torch

    from rank_bottleneck_block_gb300 import inputs as I
    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import BlockStack

    shape, nb = I.MLP_BLOCK_BF16, 24
    case = I.make_stack_case(shape, blocks=nb, seed=0, device="cuda")
    out = {"workload": f"{nb} residual low-rank SwiGLU MLP blocks (T {shape.T}, d {shape.d}, f {shape.f}, "
                       f"r {shape.r}) + MSE, one training step", "steps": steps}
    T, d, f, r = shape.T, shape.d, shape.f, shape.r
    for mode, name in ((L.LR_SAVE_CKPT, "ckpt"), (L.LR_SAVE_FULL, "full")):
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats(dev)
        base = torch.cuda.memory_allocated(dev)
        st = BlockStack(shape, case, mode, device=dev)
        ms = _time_steps(st.step, steps, warmup, flush, stream)
        L.lr_check_device_error()
        peak = torch.cuda.max_memory_allocated(dev) - base
        wsb = L.lr_stack_workspace_bytes(L.LR_BF16, mode, nb, T, d, f, r)
        fl = nb * (3.0 * 2.0 * T * (2 * r * d + 2 * f * r + r * f + d * r) +
                   (4.0 * T * r * f if name == "ckpt" else 0.0))
        params = 2 * r * d + 2 * f * r + r * f + d * r
        saved = (3 * r * 2 + 4) * T * 2.0 if name == "ckpt" else (3 * r * 2 * 2 + 3 * f * 2 + 4) * T * 2.0
        nbytes = nb * (2.0 * T * d * 2 + 6.0 * params + 6.0 * d + saved) + 2.0 * T * d * 3
        out[name] = {"ms_per_step": round(ms, 3), "tokens_per_s": round(T / (ms / 1e3), 1),
                     "workspace_bytes": wsb, "peak_hbm_bytes": int(peak), "loss": st.loss.item(),
                     **_roofline(fl, nbytes, ms, pk)}
        del st
        torch.cuda.empty_cache()
    del case
    torch.cuda.empty_cache()
    return out


def measure_sweep(pk, flush, stream, steps, warmup, emit=None, eager=False):
    """The 144-shape grouped GEMM-pair sweep (d x r x T x group, no norm, d_out = d), fwd+bwd per shape,
    each step replayed from a CUDA graph."""
    import torch

    from rank_bottleneck_block_gb300 import inputs as I
    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import GraphStep, ProjGroup

    rows = []
    for shp in I.sweep_shapes():
        pg = ProjGroup(shp, I.make_proj_case(shp, seed=0, device="cuda"))
        row = {"d": shp.d_in, "r": shp.r, "T": shp.T, "group": shp.group}
        if eager:
            row["ms_eager"] = round(_time_steps(pg.step, steps, warmup, flush, stream), 4)
        gs = GraphStep(pg.step)  # the same launches replayed from a CUDA graph
        ms = _time_steps(gs, steps, warmup, flush, stream)
        L.lr_check_device_error()
        fl, nbytes = _proj_flops_bytes(shp.T, shp.d_in, shp.d_out, shp.r, shp.group, False)
        row.update({"ms": round(ms, 4), **_roofline(fl, nbytes, ms, pk)})
        rows.append(row)
        if emit:
            emit(row)
        del gs, pg
        torch.cuda.empty_cache()
    fr = [r["frac_nominal"] for r in rows]
    fm = [r["frac_measured"] for r in rows]
    worst = min(rows, key=lambda r: r["frac_nominal"])
    t2k = [r["frac_nominal"] for r in rows if r["T"] == 2048]
    return {"workload": "grouped low-rank GEMM-pair sweep, 144 shapes (d 2048-8192, r d/8-d/2, T 2048-65536, "
                        "group 1-3), fwd+bwd, each step replayed from a CUDA graph", "steps": steps,
            "shapes": len(rows), "frac_nominal_min": min(fr), "frac_nominal_median": statistics.median(fr),
            "frac_nominal_max": max(fr), "shapes_at_or_above_0.6_nominal": sum(x >= 0.6 for x in fr),
            "frac_measured_min": min(fm), "frac_measured_median": statistics.median(fm),
            "shapes_at_or_above_0.6_measured": sum(x >= 0.6 for x in fm),
            "frac_nominal_median_T2048": statistics.median(t2k) if t2k else None,
            "worst_shape": {k: worst[k] for k in ("d", "r", "T", "group", "ms", "frac_nominal")},
            "per_shape": [[r["d"], r["r"], r["T"], r["group"], r["ms"], r["frac_nominal"]] for r in rows],
            "per_shape_fields": ["d", "r", "T", "group", "ms", "frac_nominal"]}


def measure_block(pk, flush, stream, steps, warmup, dev, with_kernels=False):
    """The full low-rank transformer block at LLaMA-7B widths: q/k/v group, causal attention,
    o-projection with residual, checkpointed MLP block; fwd+bwd."""
    from rank_bottleneck_block_gb300 import inputs as I
    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import TransformerBlock

    shape = I.BLOCK_7B
    T, d, f, ra, rm = shape.T, shape.d, shape.f, shape.ra, shape.rm
    blk = TransformerBlock(shape, I.make_block_case(shape, seed=0, device="cuda"), device=dev)
    ms = _time_steps(blk.step, steps, warmup, flush, stream)
    L.lr_check_device_error()

    def pair(din, dout, r):  # one pair's forward FLOPs
        return 2.0 * T * r * (din + dout)

    proj = 4 * pair(d, d, ra)  # q, k, v, o
    mlp = 2 * pair(d, f, rm) + pair(f, d, rm)
    causal = 2.0 * shape.b * shape.H * shape.s * shape.s * shape.dh  # QK^T and PV over the causal half
    flops = 3 * (proj + mlp) + 2.0 * 2 * T * rm * f + causal * (1 + 2.5)  # bwd 2x; MLP re-forward
    params = 4 * 2 * d * ra + 2 * (d + f) * rm + (f + d) * rm
    nbytes = 4.0 * T * d * 2 + params * (2 + 4) + 2.0 * T * (3 * ra + 3 * rm + 8 * d) * 2
    res = {"workload": f"low-rank transformer block fwd+bwd (q/k/v group, causal attention, o-projection + "
                       f"residual, checkpointed SwiGLU MLP), b={shape.b} s={shape.s} H={shape.H} dh={shape.dh} "
                       f"d={d} f={f} ranks {ra}/{rm}, bf16", "steps": steps,
           "ms_per_step": round(ms, 4), "tokens_per_s": round(T / (ms / 1e3), 1), "params": params,
           "flops_note": "algorithmic: attention counted over the causal half",
           **_roofline(flops, nbytes, ms, pk)}
    if with_kernels:
        res["kernels"] = _kernel_table(blk.step, flush, stream)
    del blk
    return res


def measure_attention(pk, flush, stream, steps, warmup, dev, b=8, with_kernels=False):
    """Causal multi-head attention alone at LLaMA-7B widths (32 heads of 128, 2048 tokens per sequence),
    fwd+bwd over b sequences."""
    import torch

    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import Attention

    s, H, dh = 2048, 32, 128
    g = torch.Generator().manual_seed(0)
    q, k, v, dout = (torch.randn(b * s, H * dh, generator=g).to(torch.bfloat16) for _ in range(4))
    at = Attention(b, s, H, dh, q, k, v, device=dev)
    at.dout.copy_(dout.to(dev))
    ms = _time_steps(at.step, steps, warmup, flush, stream)
    L.lr_check_device_error()
    half = 1.0 * b * H * s * s * dh  # one causal product: 2 (s^2 / 2) dh per head
    flops = 7 * half  # fwd Q K^T, P V; bwd Q K^T, dO V^T, P^T dO, dS K, dS^T Q
    # compulsory bytes: q, k, v read and o written (forward); q, k, v, o, dO read and dq, dk, dv written
    # (backward); the row log-sum-exp (the scores themselves are intermediates)
    nbytes = 12.0 * b * s * H * dh * 2 + 2 * 4.0 * b * H * s
    res = {"workload": f"causal attention fwd+bwd, b={b} s={s} H={H} dh={dh}, bf16 (forward without stored scores, "
                       f"backward with only dS^T in HBM, for the dQ GEMM)", "steps": steps,
           "ms_per_step": round(ms, 4), "tokens_per_s": round(b * s / (ms / 1e3), 1),
           "flops_note": "algorithmic: the causal half of the seven s x s x dh products",
           **_roofline(flops, nbytes, ms, pk)}
    if with_kernels:
        res["kernels"] = _kernel_table(at.step, flush, stream)
    del at
    return res


def run_other(a):
    """Non-default workloads (one JSON line each): attn_proj, stack, sweep, dense, block, attention."""
    import torch

    from rank_bottleneck_block_gb300 import build as B

    B.build()
    from rank_bottleneck_block_gb300 import inputs as I
    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import DenseBlock, MlpBlock

    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    pk = peaks()
    if a.workload == "attn_proj":
        print(json.dumps(measure_attn_proj(pk, flush, stream, a.steps, a.warmup, with_kernels=True)), flush=True)
    elif a.workload == "stack":
        print(json.dumps(measure_stack(pk, flush, stream, a.steps, a.warmup, dev)), flush=True)
    elif a.workload == "dense":
        # The low-rank block against the full-rank block it replaces, same d, f, T, same kernels, one box.
        shape = I.MLP_BLOCK_BF16
        T, d, f, r = shape.T, shape.d, shape.f, shape.r
        res = {"workload": f"low-rank vs dense SwiGLU MLP block fwd+bwd, T={T} d={d} f={f} (low-rank r={r}), bf16"}
        lr_blk = MlpBlock(shape, I.make_mlp_case(shape, seed=0, device="cuda"), L.LR_SAVE_CKPT, device=dev)
        ms_lr = _time_steps(lr_blk.step, a.steps, a.warmup, flush, stream)
        L.lr_check_device_error()
        _, _, fl_lr, nb_lr = workload("ckpt")
        res["lowrank_ckpt"] = {"ms_per_step": round(ms_lr, 4), "tokens_per_s": round(T / (ms_lr / 1e3), 1),
                               "params": 2 * r * d + 2 * f * r + r * f + d * r, **_roofline(fl_lr, nb_lr, ms_lr, pk)}
        del lr_blk
        torch.cuda.empty_cache()
        dn = DenseBlock(shape, I.make_dense_case(shape, seed=0, device="cuda"), device=dev)
        ms_dn = _time_steps(dn.step, a.steps, a.warmup, flush, stream)
        L.lr_check_device_error()
        fl_dn = 18.0 * T * d * f  # fwd 6 T d f, bwd twice that
        nb_dn = 2.0 * T * d * 4 + 3 * d * f * (2 + 4) + 3.0 * T * f * 2 * 2 + 2.0 * d * 6
        res["dense"] = {"ms_per_step": round(ms_dn, 4), "tokens_per_s": round(T / (ms_dn / 1e3), 1),
                        "params": 3 * d * f, **_roofline(fl_dn, nb_dn, ms_dn, pk)}
        res["lowrank_speedup"] = round(ms_dn / ms_lr, 3)
        print(json.dumps(res), flush=True)
    elif a.workload == "block":
        print(json.dumps(measure_block(pk, flush, stream, a.steps, a.warmup, dev, with_kernels=True)), flush=True)
    elif a.workload == "attention":
        print(json.dumps(measure_attention(pk, flush, stream, a.steps, a.warmup, dev, a.attn_batch,
                                           with_kernels=True)), flush=True)
    elif a.workload == "sweep":
        res = measure_sweep(pk, flush, stream, a.steps, a.warmup,
                            emit=lambda row: print(json.dumps(row), flush=True), eager=True)
        print(json.dumps(res), flush=True)


# --------------------------------------------------------- reference arm
def run_reference(a, ws, rank):
    if rank != 0:
        return
    shape, cfg, _, _ = workload(a.mode)
    budget = 90.0
    # calibrate the oracle's per-token cost, then size each step's sample so the run stays bounded
    tps, _, _ = oracle_tokens_per_s(shape, 64, 0.0, a.mode)
    rows = int(budget / max(1, a.steps + a.warmup) * tps) // 8 * 8
    rows = max(8, min(rows, 4096))
    for _ in range(a.warmup):
        oracle_tokens_per_s(shape, rows, 0.0, a.mode)
    t0 = time.perf_counter()
    for _ in range(a.steps):
        oracle_tokens_per_s(shape, rows, 0.0, a.mode)
    el = time.perf_counter() - t0
    value = rows * a.steps / el
    sample = (f"fp64 numpy oracle fwd+bwd of the block on {rows} of the {shape.T} tokens per step "
              f"(same d, f, r, seed); numpy BLAS default threading")
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws,
           "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(el * 1e3 / a.steps, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": dict(cfg, parallelism="host cores"),
           "cpu_baseline": {"value": round(value, 2), "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--mode", choices=["ckpt", "full"], default="ckpt")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=1024)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--attn-batch", type=int, default=8, help="sequences of the attention workload")
    ap.add_argument("--no-extras", action="store_true",
                    help="leave the attention-projection, stack and sweep records out of the benchmark line")
    ap.add_argument("--extra-steps", type=int, default=10, help="timed steps of the attn_proj and stack records")
    ap.add_argument("--sweep-steps", type=int, default=5, help="timed steps per shape of the sweep record")
    ap.add_argument("--workload", choices=["mlp_block", "attn_proj", "stack", "sweep", "dense", "block", "attention"],
                    default="mlp_block",
                    help="mlp_block is the benchmark line; the others print their own measurement lines")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_setup()
    if a.impl == "reference":
        run_reference(a, ws, rank)
    elif a.workload != "mlp_block":
        if rank == 0:
            run_other(a)
    else:
        run_ours(a, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
