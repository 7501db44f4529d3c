#!/usr/bin/env python
"""Throughput of one GPT-2 training iteration (forward + backward + clip +
AdamW) on B300 through the library's C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload gpt2_124m|gpt2_24l_1024d|char] [--no-cpu-baseline]

Prints one JSON line on rank 0. A step is one pass of the whole hot path over
one synthetic batch (Zipf(1.1) token ids, seeded) with inputs resident in HBM;
`value` is whole-job tokens/s. Under torchrun (N > 1) every rank runs an
independent replica on its own GPU and batch (no collective on the data path:
the gradient exchange of data parallelism is not part of this single-GPU
build); timing is the max over ranks.

`--impl reference` times the CPU oracle (plain fp64 numpy) on a bounded sample
of the same workload on the host cores, as the comparison arm.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synthdata  # noqa: E402

METRIC = "tokens/s and MFU, GPT-2 124M fwd+bwd+AdamW step, B=16 T=1024, 1 B300"
# B300 dense bf16 tensor peak: NVIDIA's HGX B300 specification lists 36
# PFLOPS FP16/BF16 for eight GPUs with 2:4 sparsity, i.e. 18 dense, 2.25 per GPU
NOMINAL_BF16_DENSE = 2.25e15

WORKLOADS = {
    # name: (n_layer, n_head, d_model, vocab, padded, T, B, stream kind)
    "gpt2_124m": (12, 12, 768, 50257, 50304, 1024, 16, "zipf"),
    "gpt2_124m_accum32": (12, 12, 768, 50257, 50304, 1024, 16, "zipf"),
    "gpt2_24l_1024d": (24, 16, 1024, 50257, 50304, 1024, 8, "zipf"),
    "char": (6, 6, 384, 65, 0, 256, 64, "markov"),
}
# micro-steps per optimizer step (gradient accumulation; sotaaz Section 3:
# 32 micro-batches of 16 x 1024 = 524,288 tokens per step)
ACCUM = {"gpt2_124m_accum32": 32}
# the oracle's bounded sample for both CPU arms: one sequence of this many tokens
ORACLE_SAMPLE_TOKENS = 256


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    max_mhz=d.get("sm_max_mhz", 2032.0), source="measured")
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, max_mhz=2032.0, source="fallback")


def tensor_peak(peaks, clocks):
    """The bf16 peak for a kernel timed at the clocks this run saw: the burst
    figure (measured at full clock) when the run's median SM clock is within
    5% of the maximum, else the burst figure scaled by median / maximum. The
    sustained figure was taken at a lower clock under the power cap, so it
    would overstate the fraction of a kernel that runs at full clock."""
    mhz = (clocks or {}).get("sm_mhz")
    mx = (clocks or {}).get("sm_max_mhz") or peaks["max_mhz"]
    if mhz and mhz < 0.95 * mx:
        return peaks["bf16"] * mhz / mx, (f"{peaks['source']} bf16_tflops (burst) x median SM clock "
                                          f"{mhz:.0f} / {mx:.0f} MHz of this run")
    return peaks["bf16"], (f"{peaks['source']} bf16_tflops (burst): this run's median SM clock "
                           f"{mhz if mhz else 'unknown'} MHz is at the maximum")


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def flops_per_token(L, C, V_padded, T, block):
    """6N + 12 L T d with N the non-position parameters, padded vocabulary
    (nanoGPT guide Part IV Stage 6, estimate_mfu)."""
    n = V_padded * C + L * (12 * C * C + 13 * C) + 2 * C
    return 6 * n + 12 * L * T * C


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, regions=None):
        """Median SM clock, its maximum and the throttle reasons seen over all
        samples; with regions ({name: (t0, t1)} in time.time() seconds) also
        the median SM clock of the samples taken inside each region."""
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return self.summarize(lines, regions)

    @staticmethod
    def summarize(lines, regions=None):
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 10:
                rows.append(parts)
        if not rows:
            return None

        def mhz(r, i):
            return float(r[i]) if r[i].replace(".", "").isdigit() else None

        sm = [v for v in (mhz(r, 2) for r in rows) if v is not None]
        mx = [v for v in (mhz(r, 3) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
               "samples": len(rows)}
        if regions:
            # nvidia-smi stamps each sample in the host's local time
            stamped = []
            for r in rows:
                try:
                    t = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    continue
                v = mhz(r, 2)
                if v is not None:
                    stamped.append((t, v))
            by_region = {}
            for name, (t0, t1) in regions.items():
                inside = [v for t, v in stamped if t0 <= t <= t1]
                by_region[name] = {"sm_mhz": statistics.median(inside) if inside else None,
                                   "samples": len(inside)}
            out["by_region"] = by_region
        return out


# ----------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def barrier_max(x: float, world: int, torch):
    """Max of x over the ranks (a barrier as a side effect); the tensor lives
    where the process group's backend wants it (CUDA for NCCL, host for gloo)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- CPU oracle
def cpu_oracle_time(workload: str, tokens: int, steps: int = 1):
    """Time the oracle's fwd+bwd+AdamW on a bounded sample: one sequence of
    `tokens` tokens of the workload's model (all parameters, real vocabulary).
    Returns (seconds per step, threads used, sample description)."""
    from oracle import gpt2_oracle as O
    L, H, C, V, Vp, T, B, kind = WORKLOADS[workload]
    c = O.Config(n_layer=L, n_head=H, d_model=C, vocab_size=V, padded_vocab=Vp, block_size=T,
                 batch_size=1, seq_len=tokens)
    tr = O.Trainer(c, 1337)
    x, y = synthdata.batch_for(kind, V, 1, tokens, 1337)
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        tr.forward(x, y)
        tr.backward()
        tr.step(lr=6e-4)
        tr.zero_grad()
        times.append(time.perf_counter() - t0)
    try:
        from threadpoolctl import threadpool_info
        cores = max(i.get("num_threads", 1) for i in threadpool_info()) or os.cpu_count()
    except Exception:
        cores = os.cpu_count()
    sample = (f"oracle (fp64 numpy) fwd+bwd+AdamW of the full {workload} model on 1 sequence x "
              f"{tokens} tokens (of the {B}x{T} batch), {steps} step(s); CPU {cpu_model()}, "
              f"{os.cpu_count()} logical cores")
    return times, cores, sample


def workload_config(workload: str, B: int, world: int) -> dict:
    """The bench line's `config`, the same for both arms."""
    L, H, C, V, Vp, T, _, _ = WORKLOADS[workload]
    return {"workload": workload, "global_batch": B * world, "seq_len": T,
            "n_layer": L, "n_head": H, "d_model": C, "vocab": V, "padded_vocab": Vp,
            "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
            "l2": "inputs larger than L2: a step's weights, optimizer state and activations far exceed the 126 MB L2"}


def run_reference(args):
    world, rank, _ = dist_env()
    L, H, C, V, Vp, T, B, kind = WORKLOADS[args.workload]
    if args.batch:
        B = args.batch
    if rank != 0:
        return
    n = args.steps + args.warmup
    # the same bounded sample as the GPU arm's cpu_baseline (one sequence of
    # ORACLE_SAMPLE_TOKENS tokens), one oracle step per bench step
    tokens = min(T, ORACLE_SAMPLE_TOKENS)
    times, cores, sample = cpu_oracle_time(args.workload, tokens, n)
    timed = times[args.warmup:] if len(times) > args.warmup else times
    sec = sum(timed) / len(timed)
    value = tokens / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * sec, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        # the workload timed is ours; the oracle runs a bounded sample of it
        # (cpu_baseline.sample says which)
        "config": workload_config(args.workload, B, world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- GPU arm
def traffic_ratio_from_profiles(kernel_src: str):
    """DRAM bytes per algorithmic byte of the dominant kernel, from the
    committed ncu summary, if that summary was taken on the current kernel
    source (single-kernel captures on a smaller case; see the file)."""
    path = os.path.join(ROOT, "profiles", "gemm_tc_gpt2_124m_traffic.txt")
    if not os.path.exists(path) or not os.path.exists(kernel_src):
        return None
    with open(kernel_src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    vals = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != h:
        return None
    try:
        return float(vals["dram_to_algorithmic_ratio"])
    except (KeyError, ValueError):
        return None


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from decoder_only_transformer_06_b300 import gpt2

    L, H, C, V, Vp, T, B, kind = WORKLOADS[args.workload]
    if args.batch:
        B = args.batch
    accum = ACCUM.get(args.workload, 1)
    cfg = gpt2.Config(n_layer=L, n_head=H, d_model=C, vocab_size=V, padded_vocab=Vp,
                      block_size=T, batch_size=B, seq_len=T, grad_accum_steps=accum,
                      precision=gpt2.GPT2_BF16)
    stream = torch.cuda.Stream()
    model = gpt2.GPT2(cfg, seed=1337, stream=stream)
    # one synthetic batch per micro-step; with accumulation a bounded pool of
    # distinct batches is cycled (the step's arithmetic does not depend on it)
    nb = min((args.warmup + args.steps) * accum, 64)
    host = [synthdata.batch_for(kind, V, B, T, 1337 + 1000 * rank + i) for i in range(nb)]
    toks = [torch.from_numpy(x.reshape(-1)).cuda() for x, _ in host]
    tgts = [torch.from_numpy(y.reshape(-1)).cuda() for _, y in host]
    lr = lambda it: gpt2.lr_schedule(it, 715, 19073, 6e-4, 6e-5)

    def train_step(i, it):
        # one optimizer step: `accum` micro-steps of forward + backward, then
        # clip + AdamW and zero_grad (nanoGPT guide Part IV Stages 4-5)
        for a in range(accum):
            j = (i * accum + a) % nb
            model.forward(toks[j], tgts[j], sync_loss=False)
            model.backward()
        model.step(lr(it), sync_norm=False)
        model.zero_grad()

    # the clock sampler (an nvidia-smi process polling every 200 ms) starts
    # before the warm-up steps, so that its start-up lands outside the timed
    # regions
    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        train_step(i, i)
    model.sync()
    if world > 1:
        torch.distributed.barrier()
    # the library counts its launches even with event timing off: clear the
    # counters here and read them right after the timed region
    model.profile(False)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_dev0 = time.time()
    e0.record(stream)
    for k in range(args.steps):
        train_step(args.warmup + k, args.warmup + k)
    # the last step's AdamW and zero_grad run on the library's second stream:
    # join it before the closing event
    model.join()
    e1.record(stream)
    torch.cuda.synchronize()
    t_dev1 = time.time()
    launches_timed = sum(r["kernels"] for r in model.profile_report())
    if world > 1:
        torch.distributed.barrier()
    ms = e0.elapsed_time(e1)
    model.sync()
    ms = barrier_max(ms, world, torch)
    ms_step = ms / args.steps
    tokens_step = B * T * accum * world
    value = tokens_step / (ms_step / 1000.0)

    # ---- end to end through the public API with host buffers, right after the
    # device-timed region and with as many steps (the same clock conditions)
    pin_t = [torch.from_numpy(x.reshape(-1)).pin_memory() for x, _ in host]
    pin_y = [torch.from_numpy(y.reshape(-1)).pin_memory() for _, y in host]
    dt, dy = torch.empty_like(toks[0]), torch.empty_like(tgts[0])
    e2e_steps = args.steps
    # every step's loss is copied to pinned host memory on the stream (read
    # after the final sync), as a training loop that logs its loss would do
    # without stalling the device each step
    h_loss = torch.zeros(e2e_steps + 2, dtype=torch.float32).pin_memory()

    def e2e_step(i, it):
        for a in range(accum):
            j = (i * accum + a) % nb
            with torch.cuda.stream(stream):
                dt.copy_(pin_t[j], non_blocking=True)
                dy.copy_(pin_y[j], non_blocking=True)
            model.forward(dt, dy, sync_loss=False)
            model.backward()
        model.loss_async(h_loss[i:i + 1])   # device -> host copy of the step's (last micro-step's) loss
        model.step(lr(it), sync_norm=False)
        model.zero_grad()

    # as many warm-up steps as the device-timed region had: the power cap sets
    # the clock from recent power draw, and the host set-up above idled the GPU
    for i in range(args.warmup):
        e2e_step(i, i)
    model.sync()
    if world > 1:
        torch.distributed.barrier()
    t_e2e0 = time.time()
    t0 = time.perf_counter()
    for k in range(e2e_steps):
        e2e_step(k, k)
    model.sync()                     # the last step's update and loss copy have landed
    t_e2e1 = time.time()
    e2e_s = barrier_max(time.perf_counter() - t0, world, torch)
    # the clock sampler (nvidia-smi polling) ran through both timed regions,
    # so that whatever it perturbs, it perturbs both alike; the power cap moves
    # the clock between them, so each region's own median is reported too
    clk = clocks.stop({"device_timed": (t_dev0, t_dev1), "e2e": (t_e2e0, t_e2e1)})
    if not all(math.isfinite(v) for v in h_loss[:e2e_steps].tolist()):
        raise RuntimeError("non-finite loss in the end-to-end loop")
    e2e_value = tokens_step * e2e_steps / e2e_s

    # ---- per-kernel measurement: CUDA events around every launch site, same
    # workload, a few steps after the timed regions
    model.profile(True)
    psteps = max(1, min(3, args.steps))
    for k in range(psteps):
        train_step(k % nb, args.warmup + args.steps + k)
    rep = model.profile_report()
    model.profile(False)
    per_step = {r["name"]: r for r in rep}
    peaks = load_peaks()
    gemm = [r for r in rep if r["name"].startswith("gemm_")]
    # the split-K reduce completes the weight-gradient GEMMs that write fp32
    # partials: its time counts toward the GEMMs' (it adds no FLOPs)
    reduce_ms = sum(r["ms"] for r in rep if r["name"] == "splitk_reduce")
    g_ms = sum(r["ms"] for r in gemm) + reduce_ms
    g_flops = sum(r["flops"] for r in gemm)
    g_launch = sum(r["calls"] for r in gemm)
    achieved_tf = g_flops / (g_ms / 1000.0) / 1e12 if g_ms > 0 else None
    total_ms = sum(r["ms"] for r in rep)
    # DRAM traffic per GEMM launch: the step's algorithmic GEMM bytes per launch
    # times the DRAM/algorithmic ratio of the committed single-kernel capture
    ratio = traffic_ratio_from_profiles(os.path.join(ROOT, "decoder_only_transformer_06_b300", "csrc",
                                                     "k_gemm_tc.cu"))
    g_bytes = sum(r["bytes"] for r in gemm)
    traffic = ratio * g_bytes / g_launch if (ratio and g_launch) else None
    peak_tf, peak_src = tensor_peak(peaks, clk)
    roofline = {
        "bound": "tensor",
        "kernel": "gemm_tc_kernel (tcgen05; every Linear fwd/dX/dW) + splitk_reduce of its dW partials",
        "achieved": achieved_tf, "peak": peak_tf, "unit": "TFLOP/s",
        "frac": (achieved_tf / peak_tf) if achieved_tf else None,
        "traffic": traffic,
        "peak_source": peak_src,
        "launches_per_step": g_launch / psteps,
        "gemm_flops_per_step": g_flops / psteps,
        "gemm_plus_reduce_ms_per_step": g_ms / psteps,
        "share_of_step": g_ms / total_ms if total_ms else None,
    }
    mem_kernels = {}
    for name in ("layernorm_fwd", "layernorm_bwd", "cross_entropy", "adamw", "grad_norm",
                 "embed_fwd", "embed_bwd", "bias_colsum", "splitk_reduce"):
        r = per_step.get(name)
        if r and r["ms"] > 0:
            gbs = r["bytes"] / (r["ms"] / 1000.0) / 1e9
            mem_kernels[name] = {"GB/s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peaks["hbm"], 3),
                                 "frac_of_8TBs": round(gbs / 8000.0, 3),
                                 "ms_per_step": round(r["ms"] / psteps, 4)}
    attn = {}
    for name in ("attention_fwd", "attention_bwd"):
        r = per_step.get(name)
        if r and r["ms"] > 0:
            attn[name] = {"TFLOP/s": round(r["flops"] / (r["ms"] / 1000.0) / 1e12, 1),
                          "ms_per_step": round(r["ms"] / psteps, 4)}
    sites = {r["name"]: round(r["ms"] / psteps, 4) for r in sorted(rep, key=lambda r: -r["ms"])}

    fpt = flops_per_token(L, C, Vp, T, T)
    step_flops = fpt * tokens_step
    achieved = step_flops / (ms_step / 1000.0)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic Zipf(1.1) token ids (seeded), random-init weights",
        "config": workload_config(args.workload, B, world),
        "mfu": {"flops_per_token": fpt, "achieved_tflops": achieved / 1e12,
                "vs_nominal_2.25PF": achieved / NOMINAL_BF16_DENSE / world,
                "vs_measured_burst": achieved / (peaks["bf16"] * 1e12) / world},
        "roofline": roofline,
        "memory_bound_kernels": mem_kernels,
        "attention": attn,
        "site_ms_per_step": sites,
        "gpu_launches": int(launches_timed),
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": int(2 * B * T * 4 * accum), "d2h_bytes_per_step": 4,
                "steps": e2e_steps},
    }
    if accum > 1:
        line["config"]["grad_accum_steps"] = accum
        line["config"]["tokens_per_step"] = tokens_step
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tokens = min(T, ORACLE_SAMPLE_TOKENS)
        times, cores, sample = cpu_oracle_time(args.workload, tokens, 3)
        line["cpu_baseline"] = {"value": tokens / (sum(times) / len(times)), "unit": "tokens/s",
                                "cores": cores, "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    model.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def run_op_workload(args):
    """Four rounds of one block's op-level kernels at the workload's shapes,
    for ncu captures of a single kernel (no timing, no JSON bench line):
      attention  causal attention forward, then backward (dQ, then dK/dV)
      mlp_gemms  the MLP's c_fc GEMM with the GELU epilogue, then the c_proj
                 input-gradient GEMM with the GELU-backward epilogue"""
    import torch
    from decoder_only_transformer_06_b300 import gpt2
    L, H, C, V, Vp, T, B, kind = WORKLOADS[args.workload]
    if args.batch:
        B = args.batch
    M = B * T
    g = torch.Generator(device="cuda").manual_seed(0)
    rnd = lambda *shape, scale=1.0: (scale * torch.randn(*shape, device="cuda", generator=g)).bfloat16()
    if args.op_workload == "attention":
        hs = C // H
        qkv, dout = rnd(M, 3 * C), rnd(M, C)
        out = torch.empty(M, C, dtype=torch.bfloat16, device="cuda")
        dqkv = torch.empty(M, 3 * C, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B * H * T, device="cuda")
        scratch = torch.empty(B * H * T, device="cuda")
        for _ in range(4):
            gpt2.op_attention_fwd(gpt2.GPT2_BF16, B, T, H, hs, qkv, out, lse)
            gpt2.op_attention_bwd(gpt2.GPT2_BF16, B, T, H, hs, qkv, out, lse, dout, dqkv, scratch)
    else:
        F = 4 * C
        u, w_fc, b_fc = rnd(M, C), rnd(F, C, scale=0.02), torch.zeros(F, device="cuda")
        dy, w_mp = rnd(M, C), rnd(C, F, scale=0.02)
        dgelu = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
        h = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
        dh = torch.empty(M, F, dtype=torch.bfloat16, device="cuda")
        for _ in range(4):
            gpt2.op_gemm_bf16_gelu(M, F, C, u, C, 1, w_fc, C, 1, dgelu, h, bias=b_fc)
            gpt2.op_gemm_bf16_gelu(M, F, C, dy, C, 1, w_mp, F, 0, dh, dgelu, backward=True)
    torch.cuda.synchronize()
    gpt2.op_sync()
    print(json.dumps({"op_workload": args.op_workload, "workload": args.workload, "batch": B,
                      "rounds": 4}), flush=True)


def run_generate_workload(args):
    """Generation throughput of the workload's model (bf16, random-init
    weights, batch B): new tokens per second of the library's loop with the
    key/value cache (one position per step after the first forward) and
    without it (the full [B, T] forward per token, as the pages' loop does),
    from a short and from a long synthetic prompt. Prints one JSON line."""
    import torch
    from decoder_only_transformer_06_b300 import gpt2
    from decoder_only_transformer_06_b300.generate import generate
    L, H, C, V, Vp, T, B, kind = WORKLOADS[args.workload]
    if args.batch:
        B = args.batch
    cfg = gpt2.Config(n_layer=L, n_head=H, d_model=C, vocab_size=V, padded_vocab=Vp, block_size=T,
                      batch_size=B, seq_len=T, precision=gpt2.GPT2_BF16)
    stream = torch.cuda.Stream()
    model = gpt2.GPT2(cfg, seed=1337, stream=stream)
    new = 64
    res = {}
    for t0 in (32, T - new):
        prompt, _ = synthdata.batch_for(kind, V, B, t0, 7)
        for cache in (True, False):
            generate(model, prompt, 4, temperature=1.0, top_k=50, seed=1, kv_cache=cache)   # warm-up
            torch.cuda.synchronize()
            t_start = time.perf_counter()
            generate(model, prompt, new, temperature=1.0, top_k=50, seed=2, kv_cache=cache)
            torch.cuda.synchronize()
            dt = time.perf_counter() - t_start
            res[f"prompt{t0}_{'kv_cache' if cache else 'full_forward'}"] = {
                "tokens_per_s": round(B * new / dt, 1), "ms_per_token_step": round(1e3 * dt / new, 3)}
    # per-site device time of the cached steps (library profiling mode)
    prompt, _ = synthdata.batch_for(kind, V, B, T - new, 7)
    model.profile(True)
    generate(model, prompt, 9, temperature=1.0, top_k=50, seed=3, kv_cache=True)
    rep = model.profile_report()
    model.profile(False)
    sites = {r["name"]: round(r["ms"] / 8, 4) for r in rep if r["name"].startswith("decode_")}
    model.close()
    print(json.dumps({"op_workload": "generate", "workload": args.workload, "batch": B,
                      "new_tokens": new, "sampling": "temperature 1.0, top-k 50", "results": res,
                      f"decode_site_ms_per_step_at_prompt{T - new}": sites}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="gpt2_124m")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (small profiling captures)")
    ap.add_argument("--op-workload", choices=["attention", "mlp_gemms", "generate"], default=None,
                    help="only run one block's op-level kernels (for ncu captures), or time generation")
    args = ap.parse_args()
    if args.op_workload == "generate":
        run_generate_workload(args)
        return
    if args.op_workload:
        run_op_workload(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
