"""Programmatic dependent launch changes no result (GPU).

Every kernel of the library is launched with programmatic stream
serialisation and waits for its predecessor inside the kernel; DFL_PDL=0 in
the environment launches plainly.  The launch mode is read once per process,
so two child processes run the same two draft steps (plant targets from the
drafts, then step again) with the mode off and on, and every output -- the
residual stream, the logits, the drafts and the acceptance -- must agree bit
for bit.  The second workload (d = 4096, 160 LM-head rows) runs the 256x512
pair tiles of the grouped projection and of the greedy LM head and the
output projection split along K.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WIDE = dict(N=10, d=4096, Hq=32, Hkv=8, hd=128, D=2, L=3, B=17, C=512, V=8192, dtype="bf16", seed=2024,
            geom_p=0.3)


def _child(kind: str, out: str) -> None:
    """Runs in the child process: two steps of one workload (no logits kept,
    so the greedy LM head takes its widest tiles), outputs to `out`."""
    sys.path.insert(0, ROOT)
    import torch

    import __graft_entry__ as ge
    import block_diffusion_speculative_dfl_gb300 as dfl
    from dfl_synth import Workload, plant_targets
    torch.cuda.set_device(0)
    w = Workload("pdl_" + kind, **(ge.SMOKE_BF16 if kind == "smoke" else WIDE))
    inp = ge._smoke_inputs(w)
    shape = dfl.DraftShape(N=w.N, d=w.d, Hq=w.Hq, Hkv=w.Hkv, hd=w.hd, D=w.D, L=w.L, B=w.B, C=w.C, V=w.V,
                           dtype=w.dtype, eps=w.eps, rope_theta=w.rope_theta)
    W_lm = torch.from_numpy(inp["W_lm_bits"].view(np.int16)).view(torch.bfloat16)
    H = torch.from_numpy(inp["H"]).cuda().to(torch.bfloat16)
    model = dfl.DraftModel(shape, inp["mix"], inp["g_mix"], inp["g_blk"], inp["g_fin"], inp["layers"], W_lm)
    X0 = torch.from_numpy(inp["Xb0"]).cuda()
    model.step(H, X0)
    torch.cuda.synchronize()
    first = model.draft.cpu().numpy()
    target = plant_targets(w, first)
    model.step(H, X0, target=torch.from_numpy(target).cuda())
    torch.cuda.synchronize()
    assert dfl.dfl_get_device_error() == 0
    np.savez(out, first_draft=first, Xb=model.Xb.cpu().numpy(), draft=model.draft.cpu().numpy(),
             accept_len=model.accept_len.cpu().numpy(), bonus=model.bonus.cpu().numpy())


@pytest.mark.parametrize("kind", ["smoke", "wide"])
def test_dependent_launch_changes_no_result(kind, tmp_path):
    outs = {}
    for mode in ("0", "1"):
        out = str(tmp_path / f"{kind}_{mode}.npz")
        env = dict(os.environ, DFL_PDL=mode)
        code = f"import sys; sys.path.insert(0, 'tests'); import test_gpu_pdl as t; t._child({kind!r}, {out!r})"
        r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                           timeout=900)
        assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-3000:]
        outs[mode] = np.load(out)
    for k in outs["0"].files:
        a, b = outs["0"][k], outs["1"][k]
        assert a.shape == b.shape and np.array_equal(a.view(np.uint8), b.view(np.uint8)), k
