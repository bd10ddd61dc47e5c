"""Kernel-level timing of one operation at a workload's shape (profiling aid).

    python -m block_diffusion_speculative_dfl_gb300.kernel_bench mix  qwen3_8b_drafter [--rows R] [--iters K]
    python -m block_diffusion_speculative_dfl_gb300.kernel_bench attn qwen3_8b_drafter [--iters K]

`mix` runs dfl_layer_mix_rmsnorm on H[L][rows][d] (rows = N * C unless
--rows is given); `attn` runs dfl_block_attn (attention and output
projection) on the workload's N, C, B, heads and head dim.  Inputs are
random bf16 tensors on the device; between launches a 256 MB buffer is
written and another read, so the inputs come from HBM and no dirty line of
the flush is written back during the timed launch.  Prints one JSON line with the
library's own per-kernel trace (CUDA events around each launch), in µs per
launch, and the achieved bandwidth of the main kernel.  Two untimed launches
come first, so under a profiler `-s 2 -c 1` selects a warm launch.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import _lib as dfl
from ._build import build


def _peak_gbs() -> float:
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"])
    except (OSError, KeyError, ValueError):
        return 6800.0


def _flush(w: torch.Tensor, r: torch.Tensor) -> None:
    # write one buffer larger than L2, then read another: the read evicts the
    # dirty lines, so their write-back does not land in the timed launch
    w.zero_()
    r.amax()


def _timed(call, iters: int) -> dict:
    w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    r = torch.ones(64 << 20, dtype=torch.int32, device="cuda")
    for _ in range(2):
        call()
    torch.cuda.synchronize()
    dfl.dfl_profile_enable(True)
    for _ in range(iters):
        _flush(w, r)
        call()
    torch.cuda.synchronize()
    dfl.dfl_profile_enable(False)
    prof, _ = dfl.dfl_profile_report()
    if dfl.dfl_get_device_error():
        raise RuntimeError("device error during the timed launches")
    return {k: v[1] / v[0] * 1000.0 for k, v in prof.items()}


def bench_mix(w, rows: int, iters: int) -> dict:
    rows = rows or w.N * w.C
    H = torch.randn(w.L, rows, w.d, device="cuda").to(torch.bfloat16)
    Xc = torch.empty(w.D, rows, w.d, device="cuda", dtype=torch.bfloat16)
    mix = torch.randn(w.D, w.L, device="cuda")
    gain = torch.ones(w.D, w.d, device="cuda")
    us = _timed(lambda: dfl.dfl_layer_mix_rmsnorm(H, rows * w.d, w.L, rows, w.d, dfl.DFL_BF16, w.D, mix, gain, w.eps,
                                                  Xc, rows * w.d), iters)
    byts = 2.0 * (w.L + w.D) * rows * w.d
    t = us["mix_rmsnorm_bf16"]
    return {"op": "mix", "workload": w.name, "rows": rows, "us": {k: round(v, 2) for k, v in us.items()},
            "GBs": round(byts / t / 1e3, 1), "frac_of_hbm": round(byts / t / 1e3 / _peak_gbs(), 3)}


def bench_attn(w, iters: int) -> dict:
    N, C, B, Hq, Hkv, hd, d = w.N, w.C, w.B, w.Hq, w.Hkv, w.hd, w.d
    g = torch.Generator(device="cuda").manual_seed(1)
    r = lambda *s: torch.randn(*s, device="cuda", generator=g).to(torch.bfloat16)   # noqa: E731
    Q, Kc, Vc, Kb, Vb = r(N * B, Hq, hd), r(N * C, Hkv, hd), r(N * C, Hkv, hd), r(N * B, Hkv, hd), r(N * B, Hkv, hd)
    Wo = (r(d, Hq * hd) * (Hq * hd) ** -0.5).to(torch.bfloat16)
    Xb = torch.zeros(N * B, d, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, dtype=dfl.DFL_BF16)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    us = _timed(lambda: dfl.dfl_block_attn(Q, Kc, Vc, Kb, Vb, N, C, B, Hq, Hkv, hd, dfl.DFL_BF16, Wo, d, Xb, ws, wsb),
                iters)
    keys = N * (C + B)
    byts = 2.0 * (2 * keys * Hkv * hd + 2 * N * B * Hq * hd)
    name = "attn_tc" if "attn_tc" in us else "attn_bf16"
    return {"op": "attn", "workload": w.name, "us": {k: round(v, 2) for k, v in us.items()},
            "GBs": round(byts / us[name] / 1e3, 1), "frac_of_hbm": round(byts / us[name] / 1e3 / _peak_gbs(), 3)}


def main(argv=None) -> None:
    from dfl_synth import WORKLOADS
    p = argparse.ArgumentParser()
    p.add_argument("op", choices=["mix", "attn"])
    p.add_argument("workload", choices=sorted(WORKLOADS))
    p.add_argument("--rows", type=int, default=0, help="mix: context rows (default N * C)")
    p.add_argument("--iters", type=int, default=10)
    a = p.parse_args(argv)
    w = WORKLOADS[a.workload]
    build()
    dfl.load()
    out = bench_mix(w, a.rows, a.iters) if a.op == "mix" else bench_attn(w, a.iters)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
