#!/usr/bin/env python
"""Throughput of the block-diffusion draft step on GB300, one JSON line.

A step is one pass of the whole hot path over one batch of synthetic input:
the L-way mix + RMSNorm of every draft layer, D draft layers (dual-source
projections, block attention, output projection), the LM head with argmax
and the acceptance epilogue (greedy, or K-draft sampling + streak-score
self-selection).  value = drafted block-tokens (N * B per step, all ranks)
per second of device time.

  python bench.py [--workload qwen3_8b_drafter] [--steps K] [--warmup W]
  python bench.py --impl reference      # the fp64 CPU oracle on the same workload
  torchrun --nproc-per-node N bench.py --gpus N   # one replica per GPU (weak scaling)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "drafted block-tokens/sec on 1 GB300 (+accept epilogue); % of HBM/tensor roofline"
UNIT = "block-tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp32 FMA on the CUDA cores (the fp32 path's GEMMs): 152 SMs x 128 lanes x 2 flop x 2.07 GHz, nominal
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Between timed steps: write one buffer larger than L2, then read another.

    The read evicts the written (dirty) lines, so their write-back to HBM
    happens here, outside the timed region, and the next step starts with an
    L2 that holds none of its inputs and nothing left to write back."""

    def __init__(self) -> None:
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

    def __call__(self) -> None:
        self.w.zero_()
        self.r.amax()   # a plain read of the whole buffer (no dtype promotion)
PREFILL_ROWS = 512   # context rows per sequence and step while a cached workload's caches are filled


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="qwen3_8b_drafter")
    p.add_argument("--batch", type=int, default=0,
                   help="override sequences per GPU (a smaller case of the same kernels, e.g. for ncu)")
    p.add_argument("--context", type=int, default=0, help="override the context length (smaller case, e.g. for ncu)")
    p.add_argument("--tv", action="store_true", help="self-selection workloads: add the TV acceptance proxy")
    p.add_argument("--accept-rule", choices=["greedy", "stochastic", "sampled"], default="greedy",
                   help="self-selection workloads: acceptance of the selected draft (argmax greedy, lossless "
                        "stochastic, or greedy against the verifier's samples)")
    p.add_argument("--kernel", choices=["mix", "attn", "fc_fuse"], default=None,
                   help="time one operation alone at the workload's shape (one JSON line of kernel timings, "
                        "not the benchmark line; for profiling)")
    p.add_argument("--rows", type=int, default=0, help="--kernel mix / fc_fuse: context rows (default N * C)")
    p.add_argument("--iters", type=int, default=10, help="--kernel: timed launches")
    p.add_argument("--no-graph", action="store_true", help="time eager launches instead of a CUDA graph of the step")
    p.add_argument("--e2e-steps", type=int, default=7)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args(argv)


# ------------------------------------------------------------------ ranks --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_scalar(x: float, world: int, op: str, device=None) -> float:
    """MAX or SUM of a host scalar over ranks (identity on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(units_per_rank: float, seconds_max: float, world: int) -> float:
    """Whole-job throughput: units all ranks processed / slowest rank's time."""
    return units_per_rank * world / seconds_max


# ---------------------------------------------------------------- helpers --

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "block_diffusion_speculative_dfl_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# kernel trace name -> source files its code lives in (for the traffic record):
# the kernel's own files, then the device helpers every kernel uses
_GEMM_SRC = ["gemm_tc.cuh", "gemm_tc.cu"]
KERNEL_SOURCES = {k: v + ["common.cuh"] for k, v in {
    "gemm_ctx_kv": _GEMM_SRC, "gemm_block_qkv": _GEMM_SRC, "gemm_kv_qkv": _GEMM_SRC, "gemm_kv_qkv_append": _GEMM_SRC,
    "gemm_o_proj": _GEMM_SRC, "gemm_lm_head": _GEMM_SRC,
    "mix_rmsnorm_bf16": ["mix_rmsnorm.cu"], "attn_bf16": ["block_attn.cu"], "attn_tc": ["block_attn_tc.cu"],
    "verifier_row_stats": ["self_select.cu"],
}.items()}


def ncu_traffic(kernel, workload):
    """DRAM bytes per launch from profiles/ncu_traffic.txt, if taken on the current source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    cur = source_hash(KERNEL_SOURCES[kernel])
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
                return float(parts[2]) if parts[3] == cur else None
    return None


def kernel_work(w, ctx_lens=None):
    """Algorithmic work per launch: {kernel: (flops, bytes)} (bf16 operands, 2 B).

    For a cached-context workload (w.R > 0) ``ctx_lens`` holds each
    sequence's attended context length; the mix and the context projection
    then cover the N*R new-row slots of one step.
    """
    N, C, B, d, Hq, Hkv, hd, D, L, V = w.N, w.C, w.B, w.d, w.Hq, w.Hkv, w.hd, w.D, w.L, w.V
    kv, qd = Hkv * hd, Hq * hd
    rows_c, rows_b = N * (w.R if w.R > 0 else C), N * B
    keys = float(np.sum(np.asarray(ctx_lens) + B)) if w.R > 0 else float(N * (C + B))   # keys over all sequences
    ctx = "gemm_ctx_kv_append" if w.R > 0 else "gemm_ctx_kv"
    work = {
        "mix_rmsnorm_bf16": (2.0 * D * L * rows_c * d, 2.0 * (L + D) * rows_c * d),
        ctx: (2.0 * rows_c * 2 * kv * d, 2.0 * (rows_c * d + 2 * kv * d + rows_c * 2 * kv)),
        "gemm_block_qkv": (2.0 * rows_b * (qd + 2 * kv) * d,
                           2.0 * (rows_b * d + (qd + 2 * kv) * d + rows_b * (qd + 2 * kv))),
        "attn_bf16": (4.0 * B * Hq * keys * hd, 2.0 * (2 * keys * kv + 2 * rows_b * qd)),
        "attn_tc": (4.0 * B * Hq * keys * hd, 2.0 * (2 * keys * kv + 2 * rows_b * qd)),
        "gemm_o_proj": (2.0 * rows_b * d * qd, 2.0 * (rows_b * qd + d * qd) + 8.0 * rows_b * d),
    }
    # the context and block projections of a layer run as one grouped launch
    both = "gemm_kv_qkv_append" if w.R > 0 else "gemm_kv_qkv"
    work[both] = tuple(a + b for a, b in zip(work[ctx], work["gemm_block_qkv"]))
    if w.fc:   # DFlash fusion: one FC over the concatenated L slabs, fp32 pre-norm features out
        work["gemm_fc_fuse"] = (2.0 * rows_c * d * L * d, 2.0 * (L * rows_c * d + d * L * d) + 4.0 * rows_c * d)
    if w.F > 0:
        M = rows_b
        work["gemm_ffn_gate_up"] = (2.0 * M * 2 * w.F * d, 2.0 * (M * d + 2 * w.F * d + M * w.F))
        work["gemm_ffn_down"] = (2.0 * M * d * w.F, 2.0 * (M * w.F + d * w.F) + 8.0 * M * d)
    if V > 0:
        M = N * (B - 1)
        work["gemm_lm_head"] = (2.0 * M * V * d, 2.0 * (M * d + V * d) + (4.0 * M * V if w.K > 0 else 0.0))
    if w.dtype == "f32":   # CUDA-core path: the average fp32 GEMM launch of a step, and the attention
        M = N * (B - 1)
        gemm = D * (2.0 * rows_b * (qd + 2 * kv) * d + 2.0 * rows_c * 2 * kv * d + 2.0 * rows_b * d * qd)
        gemm += 2.0 * D * rows_b * 3 * w.F * d + (2.0 * M * V * d if V > 0 else 0.0)
        n_gemm = D * (6 + (3 if w.F > 0 else 0)) + (1 if V > 0 else 0)
        work["gemm_f32"] = (gemm / n_gemm, 0.0)
        work["attn_f32"] = (4.0 * B * Hq * keys * hd, 4.0 * (2 * keys * kv + 2 * rows_b * qd))
    if w.K > 0:
        G = B - 1
        work["verifier_row_stats"] = (0.0, 2.0 * N * w.K * B * V)
        work["tv_alpha"] = (0.0, 4.0 * N * G * V + 2.0 * N * w.K * G * V)
    return work


def tensor_peak_key(clk):
    """Which measured bf16 peak a tensor-bound kernel of this run is held to.

    The burst figure is cuBLAS at full clock; the sustained one the same GEMM
    held at the power cap for seconds.  A timed region that saw the power cap,
    or whose median SM clock sat below 97% of the maximum, ran at the
    sustained level; otherwise at burst."""
    reasons = clk.get("reasons") or []
    sm, mx = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    if "sw_power_cap" in reasons:
        return "bf16_tflops_sustained", "sw_power_cap active during the timed steps"
    if sm and mx and sm < 0.97 * mx:
        return "bf16_tflops_sustained", f"median SM clock {sm:.0f} of {mx:.0f} MHz"
    if not sm:
        return "bf16_tflops", "no clock samples: burst assumed"
    return "bf16_tflops", f"no power cap, median SM clock {sm:.0f} of {mx:.0f} MHz"


def kernel_table(prof, work, peaks, tkey):
    """Per traced kernel: launches, time, share and (when its work is known)
    bound, achieved rate and fraction of the chosen peak."""
    traced = sum(t for _, t in prof.values()) or 1.0
    kernels = {}
    for name, (n_l, tot) in sorted(prof.items(), key=lambda kv: -kv[1][1]):
        per = tot / n_l
        ent = {"launches": n_l, "ms_per_launch": round(per, 5), "share": round(tot / traced, 4)}
        if name in work:
            fl, by = work[name]
            if name.endswith("_f32") and by == 0.0:   # fp32 FMA on the CUDA cores
                ent["bound"] = "alu"
                ent["achieved"] = round(fl / (per / 1e3) / 1e12, 3)
                ent["frac"] = round(ent["achieved"] / FP32_ALU_TFLOPS, 4)
                kernels[name] = ent
                continue
            tensor = fl / (peaks[tkey] * 1e12) >= by / (peaks["hbm_gbs"] * 1e9)
            ent["bound"] = "tensor" if tensor else "hbm"
            ent["achieved"] = round(fl / (per / 1e3) / 1e12, 2) if tensor else round(by / (per / 1e3) / 1e9, 1)
            ent["frac"] = round(ent["achieved"] / (peaks[tkey] if tensor else peaks["hbm_gbs"]), 4)
        kernels[name] = ent
    return kernels


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# -------------------------------------------------------------- workloads --

def workload(name, rank=0, batch=0, context=0):
    import dataclasses
    from dfl_synth import WORKLOADS
    w = WORKLOADS[name]
    if batch:
        w = dataclasses.replace(w, N=batch)
    if context:
        w = dataclasses.replace(w, C=context)
    if rank:   # every rank drafts its own batch of sequences (weak scaling)
        w = dataclasses.replace(w, seed=w.seed + 1000 * rank)
    return w


def host_params(w):
    from dfl_synth import gen_fc_weights, gen_ffn_gains, gen_gains, gen_layer_weights, gen_lm_head, gen_mix_logits
    g_mix, g_blk, g_fin = gen_gains(w)
    W_fc, g_fc = gen_fc_weights(w) if w.fc else (None, None)
    return {"mix": gen_mix_logits(w), "g_mix": g_mix, "g_blk": g_blk, "g_fin": g_fin, "g_ffn": gen_ffn_gains(w),
            "layers": [gen_layer_weights(w, l) for l in range(w.D)],
            # W_lm in the working dtype: bf16 storage bits, or fp32 values for an fp32 workload
            "W_lm": gen_lm_head(w, as_bits=w.dtype == "bf16") if w.V > 0 else None, "W_fc": W_fc, "g_fc": g_fc}


def lm_head_f32(w, p):
    """The LM head as fp32 values (the oracle's input)."""
    from dfl_synth import bits_to_f32
    if w.V == 0:
        return None
    return bits_to_f32(p["W_lm"]) if w.dtype == "bf16" else p["W_lm"]


def oracle_step(w, p, n, W_lm_f32, vlog_n=None):
    """The fp64 oracle's draft step for sequence n (test infrastructure, CPU)."""
    import oracle as orc
    from dfl_synth import gen_block_init, gen_hidden, plant_targets  # noqa: F401
    Hn = gen_hidden(w, seqs=[n])
    Xb0 = gen_block_init(w)[n]
    t0 = time.perf_counter()
    layers = [dict(W, g_ffn=p["g_ffn"][l]) if w.F > 0 else W for l, W in enumerate(p["layers"])]
    out = orc.draft_forward(Xb0, Hn, p["mix"], p["g_mix"], p["g_blk"], layers,
                            {"Hq": w.Hq, "Hkv": w.Hkv, "hd": w.hd}, w.eps, w.rope_theta,
                            fused=(p["W_fc"], p["g_fc"]) if w.fc else None)
    if w.V > 0:
        z = orc.lm_head_logits(out["Xb"][1:], p["g_fin"], w.eps, W_lm_f32)
        drafts = orc.argmax_lowest(z)
        if w.K > 0:
            samples = np.array([[orc.sample_inverse_cdf(z[j], w.T, orc.draw_uniform(w.philox_seed, n, j, k))[0]
                                 for j in range(w.gamma)] for k in range(w.K)])
            orc.self_select(vlog_n, samples)
        else:
            orc.greedy_accept(drafts, np.concatenate([drafts, [0]]))
    return time.perf_counter() - t0


def oracle_step_cached(w, p, n, W_lm_f32, vlog_n=None):
    """The fp64 oracle's cached draft step for sequence n (test infrastructure, CPU).

    The caches of the sequence's c0 positions are built first (not timed);
    the timed part appends its n_new rows, runs the block and the LM head and
    takes the argmax and greedy acceptance.
    """
    import oracle as orc
    from dfl_synth import gen_block_init, gen_cache_state, gen_hidden_rows
    c0, m = (int(x[n]) for x in gen_cache_state(w))
    shape = {"Hq": w.Hq, "Hkv": w.Hkv, "hd": w.hd}
    layers = [dict(W, g_ffn=p["g_ffn"][l]) if w.F > 0 else W for l, W in enumerate(p["layers"])]
    Hc = gen_hidden_rows(w, n, 0, c0)
    cache = [orc.context_kv_rows(Hc, p["mix"][l], p["g_mix"][l], W["Wkc"], W["Wvc"], np.arange(c0), shape, w.eps,
                                 w.rope_theta) for l, W in enumerate(layers)]
    H_new = gen_hidden_rows(w, n, c0, c0 + m)
    Xb0 = gen_block_init(w)[n]
    t0 = time.perf_counter()
    Xb, _ = orc.draft_step_cached(Xb0, H_new, cache, p["mix"], p["g_mix"], p["g_blk"], layers, shape, w.eps,
                                  w.rope_theta)
    z = orc.lm_head_logits(Xb[1:], p["g_fin"], w.eps, W_lm_f32)
    drafts = orc.argmax_lowest(z)
    orc.greedy_accept(drafts, np.concatenate([drafts, [0]]))
    return time.perf_counter() - t0


def cpu_baseline(w, p, seqs):
    from dfl_synth import gen_verifier_logits
    W_lm = lm_head_f32(w, p)
    step = oracle_step_cached if w.R > 0 else oracle_step
    total = 0.0
    for n in seqs:
        vl = gen_verifier_logits(w, seqs=[n])[0] if w.K > 0 else None
        total += step(w, p, n, W_lm, vl)
    return total


def cached_rows(w, starts, counts, R):
    """bf16 bits [L][N*R][d]: positions starts[n] .. starts[n]+counts[n]-1 of each sequence, zero-padded."""
    from dfl_synth import gen_hidden_rows
    H = np.zeros((w.L, w.N * R, w.d), np.uint16)
    for n in range(w.N):
        if counts[n] > 0:
            H[:, n * R:n * R + counts[n]] = gen_hidden_rows(w, n, int(starts[n]), int(starts[n] + counts[n]),
                                                            as_bits=True)
    return H


def prefill_cache(model, w, lengths, X0, chunk):
    """Fill every sequence's context caches to lengths[n] with cached steps of up to `chunk` rows."""
    import torch
    cur = np.zeros(w.N, np.int64)
    while (cur < lengths).any():
        m = np.minimum(lengths - cur, chunk)
        H = torch.from_numpy(cached_rows(w, cur, m, chunk).view(np.int16)).view(torch.bfloat16).cuda()
        model.step(H, X0, torch.from_numpy(m.astype(np.int32)).cuda(), R=chunk)
        cur += m
    torch.cuda.synchronize()
    if not np.array_equal(model.ctx_len.cpu().numpy(), lengths):
        raise RuntimeError("cache prefill did not reach the requested lengths")


def describe_sample(w, seqs):
    parts = "all D draft layers, LM head and " + ("K-draft sampling + self-selection" if w.K > 0 else
                                                  "greedy acceptance" if w.V > 0 else "no head")
    if w.R > 0:
        parts = "cached step: append of the new rows, " + parts
    return f"{len(seqs)} of {w.N} sequences of {w.name} ({parts}), fp64 NumPy"


# -------------------------------------------------------------- our arm --

def run_ours(args, rank, world, local):
    import torch

    import block_diffusion_speculative_dfl_gb300 as dfl
    from dfl_synth import gen_block_init, gen_cache_state, gen_hidden, gen_verifier_logits, plant_targets

    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    dfl.build()
    dfl.load()
    w = workload(args.workload, rank, args.batch, args.context)
    p = host_params(w)
    shape = dfl.DraftShape(N=w.N, d=w.d, Hq=w.Hq, Hkv=w.Hkv, hd=w.hd, D=w.D, L=w.L, B=w.B, C=w.C, V=w.V,
                           dtype=w.dtype, K=w.K, T=w.T, seed=w.philox_seed, eps=w.eps, rope_theta=w.rope_theta,
                           F=w.F, fc=w.fc)
    W_lm = None
    if w.V > 0:
        W_lm = (torch.from_numpy(p["W_lm"].view(np.int16)).view(torch.bfloat16) if w.dtype == "bf16"
                else torch.from_numpy(p["W_lm"]))
    cached = w.R > 0
    rule = {"greedy": 0, "stochastic": 1, "sampled": 2}[args.accept_rule] if w.K > 0 else 0
    kw = dict(tv=args.tv and w.K > 0, accept_rule=rule, accept_seed=w.philox_seed ^ 0xACCE97, ffn_gain=p["g_ffn"],
              W_fc=p["W_fc"], fc_gain=p["g_fc"])
    X_host = torch.from_numpy(gen_block_init(w))
    X0 = X_host.cuda()
    n_host = n_new = None
    ctx_lens = None
    if cached:
        # steady-state decoding: caches prefilled to the ragged lengths c0, then
        # each timed step appends n_new rows (lengths held, so every step is alike)
        model = dfl.CachedDraftModel(shape, PREFILL_ROWS, p["mix"], p["g_mix"], p["g_blk"], p["g_fin"],
                                     p["layers"], W_lm, **kw)
        c0, m_new = gen_cache_state(w)
        prefill_cache(model, w, c0.astype(np.int64), X0, PREFILL_ROWS)
        ctx_lens = c0 + m_new
        H_host = torch.from_numpy(cached_rows(w, c0, m_new, w.R).view(np.int16)).view(torch.bfloat16)
        n_host = torch.from_numpy(m_new)
        n_new = n_host.cuda()
    else:
        model = dfl.DraftModel(shape, p["mix"], p["g_mix"], p["g_blk"], p["g_fin"], p["layers"], W_lm, **kw)
        H_host = (torch.from_numpy(gen_hidden(w, as_bits=True).view(np.int16)).view(torch.bfloat16)
                  if w.dtype == "bf16" else torch.from_numpy(gen_hidden(w)))
    H = H_host.cuda()
    vlog_host = vlog = None
    if w.K > 0:
        vlog_host = (torch.from_numpy(gen_verifier_logits(w, as_bits=True).view(np.int16)).view(torch.bfloat16)
                     if w.dtype == "bf16" else torch.from_numpy(gen_verifier_logits(w)))
        vlog = vlog_host.cuda()

    def run_step(target=None):
        if cached:
            model.step(H, X0, n_new, target=target, vlog=vlog, R=w.R, advance=False)
        else:
            model.step(H, X0, target=target, vlog=vlog)

    target_host = target = None
    if w.V > 0 and w.K == 0:   # plant the target's argmax against this step's drafts
        run_step()
        torch.cuda.synchronize()
        target_host = torch.from_numpy(plant_targets(w, model.draft.cpu().numpy()))
        target = target_host.cuda()

    def step():
        run_step(target)

    flush = L2Flush()
    for _ in range(max(args.warmup, 0)):
        step()
        flush()
    torch.cuda.synchronize()
    # The timed steps replay one CUDA graph of the step (a call allocates and
    # synchronises nothing, so a captured step replays bit for bit), with no
    # per-launch trace events in them; a traced pass of the same steps, eager,
    # follows and gives each kernel's time (the roofline) and the launch count.
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("bench_timed")   # profilers can select the timed steps' kernels by this range
    for a, b in evs:
        a.record()
        run()
        b.record()
        flush()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    barrier(world)
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    dfl.dfl_profile_enable(True)
    for _ in range(args.steps):
        step()
        flush()
    torch.cuda.synchronize()
    dfl.dfl_profile_enable(False)
    clk = clocks.stop()
    prof, launches = dfl.dfl_profile_report()
    launches -= prof.get("copy_block_init", (0, 0.0))[0]   # a device-to-device copy, not a kernel
    err = dfl.dfl_get_device_error()
    if err:
        raise RuntimeError(f"device error {err} during the timed steps")
    ms_max = reduce_scalar(ms, world, "max", device="cuda")
    units = w.N * w.B
    value = aggregate(units, ms_max / 1e3, world)

    # roofline of the dominant kernel (largest share of traced time)
    peaks, peak_src = load_peaks()
    tkey, why = tensor_peak_key(clk)
    work = kernel_work(w, ctx_lens)
    kernels = kernel_table(prof, work, peaks, tkey)
    dom = next(k for k in kernels if k in work)
    de = kernels[dom]
    peak_of = {"tensor": peaks[tkey], "hbm": peaks["hbm_gbs"], "alu": FP32_ALU_TFLOPS}
    roofline = {"kernel": dom, "bound": de["bound"], "achieved": de["achieved"],
                "peak": round(peak_of[de["bound"]], 1),
                "unit": "GB/s" if de["bound"] == "hbm" else "TFLOP/s", "frac": de["frac"],
                "traffic": ncu_traffic(dom, w.name),
                "peak_source": (f"{peak_src} ({'bf16 dense ' + ('burst' if tkey == 'bf16_tflops' else 'sustained')}"
                                f": {why})" if de["bound"] == "tensor" else
                                "nominal fp32 FMA rate: 152 SMs x 128 lanes x 2 flop x 2.07 GHz"
                                if de["bound"] == "alu" else f"{peak_src} (HBM copy)"),
                "algorithmic_per_launch": work[dom][1] if de["bound"] == "hbm" else work[dom][0]}
    if de["bound"] == "tensor":   # both fractions, the chosen one in "frac"
        roofline["frac_burst"] = round(de["achieved"] / peaks["bf16_tflops"], 4)
        roofline["frac_sustained"] = round(de["achieved"] / peaks["bf16_tflops_sustained"], 4)

    # end to end through the public API: pinned host inputs in, results out
    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        H_pin, X_pin = H_host.pin_memory(), X_host.pin_memory()
        t_pin = target_host.pin_memory() if target_host is not None else None
        v_pin = vlog_host.pin_memory() if vlog_host is not None else None
        n_pin = n_host.pin_memory() if n_host is not None else None
        dev_in = {}

        def e2e_step(dev_in):
            if cached:
                return model.step_from_host(H_pin, X_pin, n_pin, t_pin, v_pin, dev_in, R=w.R, advance=False)
            return model.step_from_host(H_pin, X_pin, t_pin, v_pin, dev_in)

        for _ in range(2):   # allocate device buffers, touch the pinned pages
            out, dev_in = e2e_step(dev_in)
        times = []
        for _ in range(args.e2e_steps):
            t0 = time.perf_counter()
            out, dev_in = e2e_step(dev_in)
            times.append(time.perf_counter() - t0)
        # median: the host link shows occasional 2-3x slow copies on some boxes
        e2e_s = reduce_scalar(statistics.median(times), world, "max", device="cuda")
        h2d = sum(t.numel() * t.element_size() for t in (H_pin, X_pin, n_pin, t_pin, v_pin) if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in out.values())
        e2e = {"value": round(aggregate(units, e2e_s, world), 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 3), "statistic": "median",
               "steps": len(times), "ms_mean": round(statistics.mean(times) * 1e3, 3),
               "ms_min": round(min(times) * 1e3, 3), "ms_max": round(max(times) * 1e3, 3)}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        seqs = [0] if w.N > 1 else [0]
        t_cpu = cpu_baseline(w, p, seqs)
        cpu = {"value": round(len(seqs) * w.B / t_cpu, 3), "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
               "kind": "oracle", "sample": describe_sample(w, seqs), "seconds": round(t_cpu, 2)}

    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms_max, 4), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
                "data": "synthetic (seeded NumPy PCG64; shapes and distributions of the workload)",
                "config": {"workload": w.name, "N_per_gpu": w.N, "d": w.d, "Hq": w.Hq, "Hkv": w.Hkv, "hd": w.hd,
                           "draft_layers": w.D, "target_layers": w.L, "block": w.B, "context": w.C, "vocab": w.V,
                           "ffn": w.F, "new_rows_per_step": w.R or None,
                           "K": w.K, "T": w.T, "parallelism": f"replicas x{world}",
                           "context_features": "DFlash FC fusion" if w.fc else "per-layer mixtures",
                           "epilogue": ("self-selection" + (" + TV proxy" if args.tv else "") +
                                        {"greedy": " + greedy acceptance",
                                         "stochastic": " + stochastic acceptance",
                                         "sampled": " + sampled-greedy acceptance"}[args.accept_rule])
                           if w.K > 0 else "greedy acceptance",
                           "l2": "inputs larger than L2; between timed steps a 256 MB buffer is written, then another read, so the dirty lines are written back before the next step"},
                "timing": ("CUDA graph of the step, replayed; per-kernel times from a traced eager pass of the "
                           "same steps" if graph is not None else "eager launches; per-kernel times from a traced "
                           "eager pass of the same steps"),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clk, "kernels": kernels}
        print(json.dumps(line), flush=True)
    barrier(world)


# ------------------------------------------------------- one operation --

def run_kernel(args):
    """One operation alone at a workload's shape (profiling aid): random bf16
    inputs on the device, two untimed launches (so that a profiler's
    ``-s 2 -c 1`` selects a warm one), then ``--iters`` launches each after an
    L2 flush, timed by the library's own trace.  Prints one JSON line."""
    import torch

    import block_diffusion_speculative_dfl_gb300 as dfl
    torch.cuda.set_device(0)
    dfl.build()
    dfl.load()
    w = workload(args.workload, 0, args.batch, args.context)
    peaks, _ = load_peaks()
    g = torch.Generator(device="cuda").manual_seed(1)
    rnd = lambda *sh: torch.randn(*sh, device="cuda", generator=g).to(torch.bfloat16)   # noqa: E731
    rows = args.rows or w.N * w.C
    if args.kernel == "mix":
        H, Xc = rnd(w.L, rows, w.d), torch.empty(w.D, rows, w.d, device="cuda", dtype=torch.bfloat16)
        mix, gain = torch.randn(w.D, w.L, device="cuda"), torch.ones(w.D, w.d, device="cuda")
        call = lambda: dfl.dfl_layer_mix_rmsnorm(H, rows * w.d, w.L, rows, w.d, dfl.DFL_BF16, w.D, mix, gain,  # noqa
                                                 w.eps, Xc, rows * w.d)
        main, work = "mix_rmsnorm_bf16", (0.0, 2.0 * (w.L + w.D) * rows * w.d)
    elif args.kernel == "fc_fuse":
        H, Xc = rnd(w.L, rows, w.d), torch.empty(rows, w.d, device="cuda", dtype=torch.bfloat16)
        W, gain = (rnd(w.d, w.L * w.d) * (w.L * w.d) ** -0.5).to(torch.bfloat16), torch.ones(w.d, device="cuda")
        wsb = dfl.workspace_size(dfl.DFL_OP_FC_FUSE, N=rows, C=1, d=w.d, dtype=dfl.DFL_BF16)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        call = lambda: dfl.dfl_fc_fuse(H, rows * w.d, w.L, rows, w.d, dfl.DFL_BF16, W, gain, w.eps, Xc, ws,  # noqa
                                       wsb)
        main = "gemm_fc_fuse"
        work = (2.0 * rows * w.d * w.L * w.d, 2.0 * (w.L * rows * w.d + w.d * w.L * w.d) + 4.0 * rows * w.d)
    else:
        N, C, B, Hq, Hkv, hd, d = w.N, w.C, w.B, w.Hq, w.Hkv, w.hd, w.d
        Q, Kc, Vc, Kb, Vb = rnd(N * B, Hq, hd), rnd(N * C, Hkv, hd), rnd(N * C, Hkv, hd), rnd(N * B, Hkv, hd), \
            rnd(N * B, Hkv, hd)
        Wo = (rnd(d, Hq * hd) * (Hq * hd) ** -0.5).to(torch.bfloat16)
        Xb = torch.zeros(N * B, d, device="cuda")
        wsb = dfl.workspace_size(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, dtype=dfl.DFL_BF16)
        ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
        call = lambda: dfl.dfl_block_attn(Q, Kc, Vc, Kb, Vb, N, C, B, Hq, Hkv, hd, dfl.DFL_BF16, Wo, d, Xb, ws,  # noqa
                                          wsb)
        keys = N * (C + B)
        main, work = "attn_tc", (4.0 * B * Hq * keys * hd, 2.0 * (2 * keys * Hkv * hd + 2 * N * B * Hq * hd))
    flush = L2Flush()
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    dfl.dfl_profile_enable(True)
    for _ in range(args.iters):
        flush()
        call()
    torch.cuda.synchronize()
    dfl.dfl_profile_enable(False)
    prof, _ = dfl.dfl_profile_report()
    if dfl.dfl_get_device_error():
        raise RuntimeError("device error during the timed launches")
    if main not in prof:
        main = next(iter(sorted(prof, key=lambda k: -prof[k][1])))
    kernels = kernel_table(prof, {main: work}, peaks, "bf16_tflops")
    print(json.dumps({"kernel_only": args.kernel, "workload": w.name, "rows": rows if args.kernel != "attn" else None,
                      "us_per_launch": {k: round(v[1] / v[0] * 1e3, 2) for k, v in prof.items()},
                      "main": main, "roofline": kernels[main]}), flush=True)


# -------------------------------------------------------- reference arm --

def run_reference(args, rank, world):
    """The fp64 CPU oracle on the same workload, one sequence per step."""
    if rank != 0:
        return
    from dfl_synth import gen_verifier_logits
    w = workload(args.workload, 0, args.batch, args.context)
    p = host_params(w)
    W_lm = lm_head_f32(w, p)
    times = []
    step = oracle_step_cached if w.R > 0 else oracle_step
    for i in range(args.warmup + args.steps):
        n = i % w.N
        vl = gen_verifier_logits(w, seqs=[n])[0] if w.K > 0 else None
        t = step(w, p, n, W_lm, vl)
        if i >= args.warmup:
            times.append(t)
    total = sum(times)
    value = w.B * len(times) / total
    cores = len(os.sched_getaffinity(0))
    sample = f"one sequence of {w.name} per step (" + describe_sample(w, [0]).split("(", 1)[1]
    line = {"metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * total / len(times), 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "impl": "reference",
            "data": "synthetic (seeded NumPy PCG64; shapes and distributions of the workload)",
            "config": {"workload": w.name, "N": w.N, "B": w.B, "context": w.C, "draft_layers": w.D},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.kernel:
        run_kernel(args)
        return
    run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
