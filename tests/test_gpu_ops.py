"""Per-operation parity of the CUDA path against the fp64 oracle (GPU).

Sizes span several tiles with ragged tails; every call goes through the C ABI.
"""
import numpy as np
import pytest
import torch

import block_diffusion_speculative_dfl_gb300 as dfl
import oracle as orc
from gpu_util import (BF16_MEAN_REL, assert_bf16_close, assert_f32_close, check_samples, dev, host,
                      rel_rms_err, rng_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dfl.build()
    dfl.load()
    torch.cuda.set_device(0)
    yield
    assert dfl.dfl_get_device_error() == 0


def _ws(nbytes):
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")


# ------------------------------------------------------------------- mix --

@pytest.mark.parametrize("rows,d,L,D", [
    (300, 512, 9, 7), (200, 2880, 7, 8), (5, 4096, 9, 1), (149, 256, 3, 2),
    (3000, 512, 9, 7),    # ~20 rows per CTA: both teams, the stage ring wraps many times
    (1000, 2880, 7, 8),   # more draft layers than target layers: an output-only slab per stage
    (40, 4096, 16, 8),    # one stage fits: a single team
    (7, 5120, 9, 8),      # the widest rows (20 groups per warp)
])
def test_mix_rmsnorm_bf16(rows, d, L, D):
    rng = np.random.default_rng(rows + d)
    H = rng_bf16(rng, (L, rows, d)) * rng.uniform(0.5, 2, (L, 1, 1)).astype(np.float32)
    from dfl_synth import round_bf16
    H = round_bf16(H)
    mix = rng.standard_normal((D, L)).astype(np.float32)
    gain = rng.uniform(0.5, 1.5, (D, d)).astype(np.float32)
    Xc = torch.empty((D, rows, d), dtype=torch.bfloat16, device="cuda")
    dfl.dfl_layer_mix_rmsnorm(dev(H, "bf16"), rows * d, L, rows, d, dfl.DFL_BF16, D, dev(mix), dev(gain), 1e-6,
                              Xc, rows * d)
    got = host(Xc)
    for l in range(D):
        ref = orc.mix_rmsnorm(H, mix[l], gain[l], 1e-6)
        assert_bf16_close(got[l], ref, f"Xc[{l}]")


def test_mix_rmsnorm_f32():
    rng = np.random.default_rng(3)
    rows, d, L, D = 37, 256, 3, 2
    H = rng.standard_normal((L, rows, d)).astype(np.float32)
    mix = rng.standard_normal((D, L)).astype(np.float32)
    gain = rng.uniform(0.5, 1.5, (D, d)).astype(np.float32)
    Xc = torch.empty((D, rows, d), dtype=torch.float32, device="cuda")
    dfl.dfl_layer_mix_rmsnorm(dev(H), rows * d, L, rows, d, dfl.DFL_F32, D, dev(mix), dev(gain), 1e-6, Xc,
                              rows * d)
    got = host(Xc)
    for l in range(D):
        assert_f32_close(got[l], orc.mix_rmsnorm(H, mix[l], gain[l], 1e-6), f"Xc[{l}]")


# ------------------------------------------------------- DFlash fusion --

@pytest.mark.parametrize("rows,d,L,pad", [
    (300, 256, 3, 0),      # ragged last M tile
    (1000, 512, 9, 64),    # nine slabs, slab stride beyond the rows
    (129, 128, 1, 0),      # one slab: a plain GEMM
    (2048, 4096, 9, 0),    # the Qwen3-8B shape (K = 36,864), one sequence's context
    (77, 2880, 7, 0),      # the GPT-OSS shape (d = 45 * 64)
])
def test_fc_fuse_bf16(rows, d, L, pad):
    rng = np.random.default_rng(rows + d + L)
    stride = rows * d + pad
    Hs = np.zeros((L, stride), np.float32)
    H = rng_bf16(rng, (L, rows, d)) * rng.uniform(0.5, 2, (L, 1, 1)).astype(np.float32)
    from dfl_synth import round_bf16
    H = round_bf16(H)
    Hs[:, :rows * d] = H.reshape(L, -1)
    W = rng_bf16(rng, (d, L * d), (L * d) ** -0.5)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    Xc = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_FC_FUSE, N=rows, C=1, d=d, dtype=dfl.DFL_BF16)
    dfl.dfl_fc_fuse(dev(Hs, "bf16"), stride, L, rows, d, dfl.DFL_BF16, dev(W, "bf16"), dev(g), 1e-6, Xc, _ws(wsb),
                    wsb)
    ref = orc.fc_fuse(H, W, g, 1e-6)
    assert_bf16_close(host(Xc), ref, "Xc")


def test_fc_fuse_f32():
    rng = np.random.default_rng(5)
    rows, d, L = 45, 96, 4
    H = rng.standard_normal((L, rows, d)).astype(np.float32)
    W = (rng.standard_normal((d, L * d)) * (L * d) ** -0.5).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    Xc = torch.empty((rows, d), dtype=torch.float32, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_FC_FUSE, N=rows, C=1, d=d, dtype=dfl.DFL_F32)
    dfl.dfl_fc_fuse(dev(H), rows * d, L, rows, d, dfl.DFL_F32, dev(W), dev(g), 1e-6, Xc, _ws(wsb), wsb)
    assert_f32_close(host(Xc), orc.fc_fuse(H, W, g, 1e-6), "Xc")


# --------------------------------------------------------- dual projection --

def _proj_case(N, C, B, d, Hq, Hkv, hd, dtype, seed):
    rng = np.random.default_rng(seed)
    mk = (lambda s, sc=1.0: rng_bf16(rng, s, sc)) if dtype == "bf16" else \
        (lambda s, sc=1.0: (rng.standard_normal(s) * sc).astype(np.float32))
    W = {"Wq": mk((Hq * hd, d), d ** -0.5), "Wkc": mk((Hkv * hd, d), d ** -0.5), "Wvc": mk((Hkv * hd, d), d ** -0.5),
         "Wkb": mk((Hkv * hd, d), d ** -0.5), "Wvb": mk((Hkv * hd, d), d ** -0.5)}
    return dict(Xc=mk((N * C, d)), Xb=rng.standard_normal((N * B, d)).astype(np.float32),
                g=rng.uniform(0.5, 1.5, d).astype(np.float32), W=W)


def _proj_ref(c, N, C, B, Hq, Hkv, hd, rope, theta=1e6):
    d = c["Xb"].shape[1]
    Xn = orc.rmsnorm(c["Xb"], c["g"], 1e-6)
    W = {k: v.astype(np.float64) for k, v in c["W"].items()}
    Q = (Xn @ W["Wq"].T).reshape(N, B, Hq, hd)
    Kb = (Xn @ W["Wkb"].T).reshape(N, B, Hkv, hd)
    Vb = (Xn @ W["Wvb"].T).reshape(N, B, Hkv, hd)
    Xc = c["Xc"].astype(np.float64)
    Kc = (Xc @ W["Wkc"].T).reshape(N, C, Hkv, hd)
    Vc = (Xc @ W["Wvc"].T).reshape(N, C, Hkv, hd)
    if rope:
        cos, sin = orc.rope_cos_sin(np.arange(C + B), hd, theta)
        for n in range(N):
            Q[n] = orc.apply_rope(Q[n], cos[C:], sin[C:])
            Kb[n] = orc.apply_rope(Kb[n], cos[C:], sin[C:])
            Kc[n] = orc.apply_rope(Kc[n], cos[:C], sin[:C])
    return {"Q": Q, "Kb": Kb, "Vb": Vb, "Kc": Kc, "Vc": Vc}


@pytest.mark.parametrize("N,C,B,d,Hq,Hkv,hd,rope", [
    (2, 200, 16, 512, 8, 2, 128, True),    # ctx BN=256, ragged M (400 rows)
    (2, 200, 16, 520, 8, 2, 128, False),   # K tail (520 = 8 * 65), no rotary
    (3, 150, 8, 256, 16, 2, 64, True),     # hd 64: ctx BN=128, GQA group 8
    (1, 64, 33, 256, 4, 2, 128, True),     # 33-row block (anchor + 32 masks)
    # 256x512 pair tiles (the width the full-size drafters take): rotary split by
    # pairs (hd 128) and by heads (hd 64), V without rotary, ragged context rows
    # (16,000 = 62.5 pair tiles), a 128-row block whose pairs' odd CTA has no rows
    (8, 2000, 16, 1024, 8, 4, 128, True),
    (8, 2000, 16, 1024, 16, 8, 64, True),
])
def test_dual_kv_proj_bf16(N, C, B, d, Hq, Hkv, hd, rope):
    c = _proj_case(N, C, B, d, Hq, Hkv, hd, "bf16", seed=N * 1000 + C + d)
    kv, qd = Hkv * hd, Hq * hd
    out = {k: torch.empty(s, dtype=torch.bfloat16, device="cuda") for k, s in
           {"Q": (N * B, qd), "Kc": (N * C, kv), "Vc": (N * C, kv), "Kb": (N * B, kv), "Vb": (N * B, kv)}.items()}
    table = None
    if rope:
        table = torch.empty((C + B, hd // 2, 2), dtype=torch.float32, device="cuda")
        dfl.dfl_rope_table(table, C + B, hd, 1e6)
    wsb = dfl.workspace_size(dfl.DFL_OP_DUAL_KV_PROJ, N=N, B=B, d=d, dtype=dfl.DFL_BF16)
    ws = _ws(wsb)
    Wd = {k: dev(v, "bf16") for k, v in c["W"].items()}
    dfl.dfl_dual_kv_proj(dev(c["Xc"], "bf16"), dev(c["Xb"]), N, C, B, d, dfl.DFL_BF16, dev(c["g"]), 1e-6,
                         Wd["Wq"], Wd["Wkc"], Wd["Wvc"], Wd["Wkb"], Wd["Wvb"], Hq, Hkv, hd, table,
                         out["Q"], out["Kc"], out["Vc"], out["Kb"], out["Vb"], ws, wsb)
    ref = _proj_ref(c, N, C, B, Hq, Hkv, hd, rope)
    for k in ("Q", "Kb", "Vb", "Kc", "Vc"):
        assert_bf16_close(host(out[k]).reshape(ref[k].shape), ref[k], k)


def test_dual_kv_proj_f32():
    N, C, B, d, Hq, Hkv, hd = 1, 64, 16, 256, 4, 4, 64
    c = _proj_case(N, C, B, d, Hq, Hkv, hd, "f32", seed=5)
    kv, qd = Hkv * hd, Hq * hd
    out = {k: torch.empty(s, dtype=torch.float32, device="cuda") for k, s in
           {"Q": (N * B, qd), "Kc": (N * C, kv), "Vc": (N * C, kv), "Kb": (N * B, kv), "Vb": (N * B, kv)}.items()}
    table = torch.empty((C + B, hd // 2, 2), dtype=torch.float32, device="cuda")
    dfl.dfl_rope_table(table, C + B, hd, 1e6)
    wsb = dfl.workspace_size(dfl.DFL_OP_DUAL_KV_PROJ, N=N, B=B, d=d, dtype=dfl.DFL_F32)
    ws = _ws(wsb)
    Wd = {k: dev(v) for k, v in c["W"].items()}
    dfl.dfl_dual_kv_proj(dev(c["Xc"]), dev(c["Xb"]), N, C, B, d, dfl.DFL_F32, dev(c["g"]), 1e-6, Wd["Wq"],
                         Wd["Wkc"], Wd["Wvc"], Wd["Wkb"], Wd["Wvb"], Hq, Hkv, hd, table, out["Q"], out["Kc"],
                         out["Vc"], out["Kb"], out["Vb"], ws, wsb)
    ref = _proj_ref(c, N, C, B, Hq, Hkv, hd, True)
    for k in ("Q", "Kb", "Vb", "Kc", "Vc"):
        assert_f32_close(host(out[k]).reshape(ref[k].shape), ref[k], k)


def test_rope_table_matches_oracle():
    P, hd = 300, 128
    t = torch.empty((P, hd // 2, 2), dtype=torch.float32, device="cuda")
    dfl.dfl_rope_table(t, P, hd, 1e6)
    cos, sin = orc.rope_cos_sin(np.arange(P), hd, 1e6)
    g = host(t)
    assert np.max(np.abs(g[..., 0] - cos)) < 1e-7 and np.max(np.abs(g[..., 1] - sin)) < 1e-7


# ------------------------------------------------------------- attention --

@pytest.mark.parametrize("N,C,B,Hq,Hkv,hd,d", [
    (2, 200, 16, 8, 2, 128, 512),     # 4 units -> several key splits, ragged last tile
    (40, 48, 16, 16, 8, 128, 256),    # 320 units -> one split, keys < one tile + block
    (2, 130, 8, 16, 2, 64, 320),      # hd 64, GQA group 8
    (1, 100, 33, 16, 4, 128, 256),    # 132 query rows per unit (9 warps)
    (1, 70, 64, 32, 2, 64, 256),      # 1024 query rows per unit -> rows split over CTAs
    (3, 0, 16, 8, 2, 128, 256),       # no context: the block's own keys only
    (1, 300, 64, 4, 2, 128, 256),     # 128 query rows per unit (the padded MMA tile full)
    (2, 1000, 8, 8, 4, 64, 256),      # hd 64, several items per sequence
    (32, 2048, 16, 32, 8, 128, 512),  # the Qwen3-8B drafter's attention shape
    (16, 1024, 33, 32, 8, 128, 512),  # the self-selection window: 132 rows per K/V head, two head subsets
    (3, 500, 24, 48, 4, 64, 256),     # 288 rows per K/V head: three head subsets of 96 rows
    (3, 150, 12, 4, 2, 128, 256),     # M = 64 with 24 rows: a quadrant with 8 rows and 8 padding rows
    (2, 90, 16, 6, 2, 64, 192),       # M = 64, hd 64, group 3: 48 rows, one padding warp
])
def test_block_attn_bf16(N, C, B, Hq, Hkv, hd, d):
    rng = np.random.default_rng(N * 7 + C)
    Q = rng_bf16(rng, (N * B, Hq, hd))
    Kc, Vc = rng_bf16(rng, (N * C, Hkv, hd)), rng_bf16(rng, (N * C, Hkv, hd))
    Kb, Vb = rng_bf16(rng, (N * B, Hkv, hd)), rng_bf16(rng, (N * B, Hkv, hd))
    Wo = rng_bf16(rng, (d, Hq * hd), (Hq * hd) ** -0.5)
    Xb = rng.standard_normal((N * B, d)).astype(np.float32)
    Xb_d = dev(Xb)
    wsb = dfl.workspace_size(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, dtype=dfl.DFL_BF16)
    ws = _ws(wsb)
    dfl.dfl_block_attn(dev(Q, "bf16"), dev(Kc, "bf16"), dev(Vc, "bf16"), dev(Kb, "bf16"), dev(Vb, "bf16"), N, C, B,
                       Hq, Hkv, hd, dfl.DFL_BF16, dev(Wo, "bf16"), d, Xb_d, ws, wsb)
    ref = np.empty((N * B, d))
    for n in range(N):
        K = np.concatenate([Kc[n * C:(n + 1) * C], Kb[n * B:(n + 1) * B]])
        V = np.concatenate([Vc[n * C:(n + 1) * C], Vb[n * B:(n + 1) * B]])
        O = orc.attention(Q[n * B:(n + 1) * B], K, V, orc.block_visibility(C, B))
        ref[n * B:(n + 1) * B] = Xb[n * B:(n + 1) * B] + O.reshape(B, Hq * hd) @ Wo.astype(np.float64).T
    got = host(Xb_d)
    assert_bf16_close(got - Xb, ref - Xb, "O Wo^T")


@pytest.mark.parametrize("N,C,B,Hq,Hkv,hd,d", [
    (1, 1024, 16, 32, 8, 128, 4096),   # the single-layer (batch 1) shape: Wo split over 4 K-ranges
    (3, 200, 16, 16, 2, 128, 2048),    # 48 block rows, 4 splits
    (2, 90, 16, 8, 2, 64, 1056),       # d not a multiple of the tile: ragged last N-tile
])
def test_output_projection_k_split(N, C, B, Hq, Hkv, hd, d):
    # With at most 128 block rows and room in the workspace (a size asked for
    # with d), the output projection is split along K into fp32 partials that
    # a fixed-order sum adds to the residual: the same result as the unsplit
    # projection within bf16 arithmetic, bit-reproducible from run to run.
    rng = np.random.default_rng(N * 11 + d)
    Q = rng_bf16(rng, (N * B, Hq, hd))
    Kc, Vc = rng_bf16(rng, (N * C, Hkv, hd)), rng_bf16(rng, (N * C, Hkv, hd))
    Kb, Vb = rng_bf16(rng, (N * B, Hkv, hd)), rng_bf16(rng, (N * B, Hkv, hd))
    Wo = rng_bf16(rng, (d, Hq * hd), (Hq * hd) ** -0.5)
    Xb = rng.standard_normal((N * B, d)).astype(np.float32)
    args = [dev(Q, "bf16"), dev(Kc, "bf16"), dev(Vc, "bf16"), dev(Kb, "bf16"), dev(Vb, "bf16")]
    base = dfl.workspace_size(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, dtype=dfl.DFL_BF16)
    full = dfl.workspace_size(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, d=d, dtype=dfl.DFL_BF16)
    assert full > base
    out = {}
    for name, nbytes in (("unsplit", base), ("split", full), ("split again", full)):
        Xd = dev(Xb)
        dfl.dfl_block_attn(*args, N, C, B, Hq, Hkv, hd, dfl.DFL_BF16, dev(Wo, "bf16"), d, Xd, _ws(nbytes), nbytes)
        out[name] = host(Xd)
    ref = np.empty((N * B, d))
    for n in range(N):
        K = np.concatenate([Kc[n * C:(n + 1) * C], Kb[n * B:(n + 1) * B]])
        V = np.concatenate([Vc[n * C:(n + 1) * C], Vb[n * B:(n + 1) * B]])
        O = orc.attention(Q[n * B:(n + 1) * B], K, V, orc.block_visibility(C, B))
        ref[n * B:(n + 1) * B] = Xb[n * B:(n + 1) * B] + O.reshape(B, Hq * hd) @ Wo.astype(np.float64).T
    for name in ("unsplit", "split"):
        assert_bf16_close(out[name] - Xb, ref - Xb, name)
    assert np.array_equal(out["split"].view(np.uint32), out["split again"].view(np.uint32))


@pytest.mark.parametrize("N,C,B,Hq,Hkv,hd,d", [
    (1, 64, 16, 32, 8, 128, 4096),    # 16 rows, one M-tile: single-CTA tiles
    (3, 64, 16, 16, 2, 128, 2048),    # 48 rows, 32 k-blocks
    (4, 64, 16, 16, 2, 128, 1056),    # ragged last N-tile (1056 = 4 x 256 + 32)
    (2, 64, 16, 64, 8, 64, 2880),     # the GPT-OSS width: 2880 = 11 x 256 + 64
    (10, 64, 17, 32, 8, 128, 4096),   # 170 rows: pair tiles whose odd CTA holds 42 rows
    (16, 64, 33, 32, 8, 128, 4096),   # 528 rows (the self-selection batch): a third pair tile of 16 rows
])
def test_output_projection_few_tiles(N, C, B, Hq, Hkv, hd, d):
    # Output projections of few tiles with ragged edges (single-CTA and pair
    # tiles, a pair tile whose odd CTA holds few or no rows, a last N-tile of
    # 32 or 64 columns), run with a workspace that holds no split partials:
    # the projection's result within bf16 arithmetic, bit-identical from run
    # to run.
    rng = np.random.default_rng(N * 13 + d)
    Q = rng_bf16(rng, (N * B, Hq, hd))
    Kc, Vc = rng_bf16(rng, (N * C, Hkv, hd)), rng_bf16(rng, (N * C, Hkv, hd))
    Kb, Vb = rng_bf16(rng, (N * B, Hkv, hd)), rng_bf16(rng, (N * B, Hkv, hd))
    Wo = rng_bf16(rng, (d, Hq * hd), (Hq * hd) ** -0.5)
    Xb = rng.standard_normal((N * B, d)).astype(np.float32)
    args = [dev(Q, "bf16"), dev(Kc, "bf16"), dev(Vc, "bf16"), dev(Kb, "bf16"), dev(Vb, "bf16")]
    wsb = dfl.workspace_size(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, dtype=dfl.DFL_BF16)
    outs = []
    for _ in range(2):
        Xd = dev(Xb)
        dfl.dfl_block_attn(*args, N, C, B, Hq, Hkv, hd, dfl.DFL_BF16, dev(Wo, "bf16"), d, Xd, _ws(wsb), wsb)
        outs.append(host(Xd))
    ref = np.empty((N * B, d))
    for n in range(N):
        K = np.concatenate([Kc[n * C:(n + 1) * C], Kb[n * B:(n + 1) * B]])
        V = np.concatenate([Vc[n * C:(n + 1) * C], Vb[n * B:(n + 1) * B]])
        O = orc.attention(Q[n * B:(n + 1) * B], K, V, orc.block_visibility(C, B))
        ref[n * B:(n + 1) * B] = Xb[n * B:(n + 1) * B] + O.reshape(B, Hq * hd) @ Wo.astype(np.float64).T
    assert_bf16_close(outs[0] - Xb, ref - Xb, "O Wo^T")
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert dfl.dfl_get_device_error() == 0


@pytest.mark.parametrize("N,C,B,Hq,Hkv,hd", [
    (32, 2048, 16, 32, 8, 128),   # the Qwen3-8B drafter's attention
    (16, 1024, 33, 32, 8, 128),   # the self-selection window (two head subsets per K/V head)
    (32, 3072, 8, 64, 8, 64),     # the GPT-OSS-20B drafter's attention
    (1, 700, 16, 32, 8, 128),     # key ranges split over items and combined
    (3, 150, 12, 4, 2, 128),      # M = 64 products with padding rows
])
def test_block_attn_output_elementwise(N, C, B, Hq, Hkv, hd):
    # With Wo = I (d = Hq*hd, exact in bf16) and a zero residual stream the
    # call's output is the attention output O itself, compared element by
    # element (a wrong key tile or head is not diluted by a random Wo).
    d = Hq * hd
    rng = np.random.default_rng(N * 31 + C)
    Q = rng_bf16(rng, (N * B, Hq, hd))
    Kc, Vc = rng_bf16(rng, (N * C, Hkv, hd)), rng_bf16(rng, (N * C, Hkv, hd))
    Kb, Vb = rng_bf16(rng, (N * B, Hkv, hd)), rng_bf16(rng, (N * B, Hkv, hd))
    Wo = torch.eye(d, dtype=torch.bfloat16, device="cuda")
    Xb_d = torch.zeros((N * B, d), dtype=torch.float32, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, dtype=dfl.DFL_BF16)
    ws = _ws(wsb)
    dfl.dfl_block_attn(dev(Q, "bf16"), dev(Kc, "bf16"), dev(Vc, "bf16"), dev(Kb, "bf16"), dev(Vb, "bf16"), N, C, B,
                       Hq, Hkv, hd, dfl.DFL_BF16, Wo, d, Xb_d, ws, wsb)
    got = host(Xb_d).reshape(N, B, Hq, hd)
    for n in range(N):
        K = np.concatenate([Kc[n * C:(n + 1) * C], Kb[n * B:(n + 1) * B]])
        V = np.concatenate([Vc[n * C:(n + 1) * C], Vb[n * B:(n + 1) * B]])
        vis = orc.block_visibility(C, B)
        O = orc.attention(Q[n * B:(n + 1) * B], K, V, vis)
        # Element-wise bound from the arithmetic: the probabilities enter the
        # PV product rounded to bf16 (relative error <= 2^-9 each, so at most
        # 2^-9 sum_i p_i |V_i| / l, which is attention over |V|) and O is
        # stored in bf16 (2^-9 |O|), with 10% for the fp32 exponentials and
        # accumulation.
        A = orc.attention(Q[n * B:(n + 1) * B], K, np.abs(V), vis)
        bound = 2.0 ** -9 * (A + 2 * np.abs(O)) * 1.1 + 1e-6
        err = np.abs(got[n] - O)
        assert np.all(err <= bound), (n, float((err / bound).max()), np.unravel_index(np.argmax(err / bound), err.shape))
        for h in range(Hq):   # per head: the typical element as well
            _, mean = rel_rms_err(got[n, :, h], O[:, h])
            assert mean <= BF16_MEAN_REL, (n, h, mean)


@pytest.mark.parametrize("N,C,B,Hq,Hkv,hd,d", [
    (8, 2048, 16, 32, 8, 128, 512),   # M = 64, hd 128, one item per pipeline
    (8, 1500, 8, 64, 8, 64, 256),     # M = 64, hd 64, three S buffers
    (4, 1024, 33, 32, 8, 128, 512),   # M = 128, two head subsets
    (1, 700, 16, 32, 8, 128, 512),    # key ranges split over items, combine kernel
])
def test_block_attn_bitwise_reproducible(N, C, B, Hq, Hkv, hd, d):
    # Items are taken from a global counter in whatever order the CTAs get to
    # it, but each item's arithmetic and the combine's order are fixed: every
    # launch must produce the same bits.
    rng = np.random.default_rng(N * 13 + C)
    Q = dev(rng_bf16(rng, (N * B, Hq, hd)), "bf16")
    Kc, Vc = dev(rng_bf16(rng, (N * C, Hkv, hd)), "bf16"), dev(rng_bf16(rng, (N * C, Hkv, hd)), "bf16")
    Kb, Vb = dev(rng_bf16(rng, (N * B, Hkv, hd)), "bf16"), dev(rng_bf16(rng, (N * B, Hkv, hd)), "bf16")
    Wo = dev(rng_bf16(rng, (d, Hq * hd), (Hq * hd) ** -0.5), "bf16")
    wsb = dfl.workspace_size(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, d=d, dtype=dfl.DFL_BF16)
    ws = _ws(wsb)
    first = None
    for _ in range(8):
        Xb_d = dev(np.zeros((N * B, d), np.float32))
        dfl.dfl_block_attn(Q, Kc, Vc, Kb, Vb, N, C, B, Hq, Hkv, hd, dfl.DFL_BF16, Wo, d, Xb_d, ws, wsb)
        got = host(Xb_d)
        assert np.all(np.isfinite(got))
        if first is None:
            first = got
        else:
            assert np.array_equal(got.view(np.uint32), first.view(np.uint32))


def test_block_attn_f32():
    N, C, B, Hq, Hkv, hd, d = 1, 64, 16, 4, 4, 64, 256
    rng = np.random.default_rng(11)
    f = lambda s, sc=1.0: (rng.standard_normal(s) * sc).astype(np.float32)
    Q, Kc, Vc, Kb, Vb = f((B, Hq, hd)), f((C, Hkv, hd)), f((C, Hkv, hd)), f((B, Hkv, hd)), f((B, Hkv, hd))
    Wo, Xb = f((d, Hq * hd), (Hq * hd) ** -0.5), f((B, d))
    Xb_d = dev(Xb)
    wsb = dfl.workspace_size(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, dtype=dfl.DFL_F32)
    ws = _ws(wsb)
    dfl.dfl_block_attn(dev(Q), dev(Kc), dev(Vc), dev(Kb), dev(Vb), N, C, B, Hq, Hkv, hd, dfl.DFL_F32, dev(Wo), d,
                       Xb_d, ws, wsb)
    O = orc.attention(Q, np.concatenate([Kc, Kb]), np.concatenate([Vc, Vb]), orc.block_visibility(C, B))
    assert_f32_close(host(Xb_d), Xb + O.reshape(B, -1) @ Wo.astype(np.float64).T, "Xb")


# --------------------------------------------------------------- LM head --

def _lm_case(N, B, d, V, seed, dtype="bf16"):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, B, d)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    W = rng_bf16(rng, (V, d), d ** -0.5) if dtype == "bf16" else \
        (rng.standard_normal((V, d)) * d ** -0.5).astype(np.float32)
    return X, g, W


@pytest.mark.parametrize("N,B,row0,d,V", [(3, 16, 1, 512, 1000), (2, 9, 1, 256, 5003), (1, 16, 0, 256, 256),
                                            (10, 16, 1, 256, 3000), (20, 16, 1, 256, 1000)])
def test_lm_head_argmax_bf16(N, B, row0, d, V):
    X, g, W = _lm_case(N, B, d, V, seed=V)
    nr = B - row0
    am = torch.empty((N, nr), dtype=torch.int32, device="cuda")
    lg = torch.empty((N * nr, V), dtype=torch.float32, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_LM_HEAD, N=N, B=B, row0=row0, d=d, V=V, dtype=dfl.DFL_BF16)
    ws = _ws(wsb)
    dfl.dfl_lm_head_argmax(dev(X), N, B, row0, d, dfl.DFL_BF16, dev(g), 1e-6, dev(W, "bf16"), V, am, lg, None, None,
                           ws, wsb)
    z = host(lg)
    ref = orc.lm_head_logits(X[:, row0:].reshape(-1, d), g, 1e-6, W)
    assert_bf16_close(z, ref, "logits")
    # argmax is bit-exact against the oracle's argmax of the same fp32 buffer
    assert np.array_equal(host(am).reshape(-1), orc.argmax_lowest(z))


@pytest.mark.parametrize("N,B,row0,d,V", [(12, 16, 1, 4096, 5003), (12, 16, 1, 4096, 4700),
                                            (40, 16, 1, 4096, 3000)])
def test_lm_head_argmax_wide_tiles(N, B, row0, d, V):
    """Greedy heads of more than 128 rows and K >= 4096 take 512-wide pair tiles, whose two
    epilogue warps per lane quadrant each write a 256-column partial; the
    argmax must equal the one of the 256-wide path (logits stored) and the
    oracle's lowest-index argmax of those logits.  V = 4700 leaves the last
    512-wide tile's second half without columns; V = 5003 a partial last one."""
    X, g, W = _lm_case(N, B, d, V, seed=V + N)
    nr = B - row0
    wsb = dfl.workspace_size(dfl.DFL_OP_LM_HEAD, N=N, B=B, row0=row0, d=d, V=V, dtype=dfl.DFL_BF16)
    ws = _ws(wsb)
    am_wide = torch.full((N, nr), -1, dtype=torch.int32, device="cuda")
    dfl.dfl_lm_head_argmax(dev(X), N, B, row0, d, dfl.DFL_BF16, dev(g), 1e-6, dev(W, "bf16"), V, am_wide, None,
                           None, None, ws, wsb)
    am = torch.empty((N, nr), dtype=torch.int32, device="cuda")
    lg = torch.empty((N * nr, V), dtype=torch.float32, device="cuda")
    dfl.dfl_lm_head_argmax(dev(X), N, B, row0, d, dfl.DFL_BF16, dev(g), 1e-6, dev(W, "bf16"), V, am, lg, None,
                           None, ws, wsb)
    z = host(lg)
    assert np.array_equal(host(am_wide), host(am))
    assert np.array_equal(host(am_wide).reshape(-1), orc.argmax_lowest(z))


def test_lm_head_argmax_ties_take_lowest_index():
    N, B, d, V = 1, 4, 256, 1000
    rng = np.random.default_rng(21)
    x = rng.standard_normal(d).astype(np.float32)
    X = np.broadcast_to(x, (N, B, d)).copy()
    g = np.ones(d, np.float32)
    W = rng_bf16(rng, (V, d), 1e-3)
    from dfl_synth import round_bf16
    u = round_bf16(x / np.linalg.norm(x) * 4)
    for v in (300, 301, 900):         # tie inside a 256-column tile and across tiles
        W[v] = u
    am = torch.empty((N, B), dtype=torch.int32, device="cuda")
    lg = torch.empty((N * B, V), dtype=torch.float32, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_LM_HEAD, N=N, B=B, row0=0, d=d, V=V, dtype=dfl.DFL_BF16)
    ws = _ws(wsb)
    dfl.dfl_lm_head_argmax(dev(X), N, B, 0, d, dfl.DFL_BF16, dev(g), 1e-6, dev(W, "bf16"), V, am, lg, None, None,
                           ws, wsb)
    z = host(lg)
    assert np.all(z[:, 300] == z[:, 900]) and np.all(z[:, 300] == z[:, 301])
    assert np.all(host(am) == 300)
    # all-zero head: every logit ties at 0 -> index 0
    dfl.dfl_lm_head_argmax(dev(X), N, B, 0, d, dfl.DFL_BF16, dev(g), 1e-6, dev(np.zeros((V, d), np.float32), "bf16"),
                           V, am, None, None, None, ws, wsb)
    assert np.all(host(am) == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_lm_head_sampling(dtype):
    N, B, d, V, K, T, seed = 2, 9, 256, 1000, 8, 1.5, 0x5EEDD1F5
    X, g, W = _lm_case(N, B, d, V, seed=77, dtype=dtype)
    dt = dfl.DFL_BF16 if dtype == "bf16" else dfl.DFL_F32
    nr = B - 1
    am = torch.empty((N, nr), dtype=torch.int32, device="cuda")
    lg = torch.empty((N * nr, V), dtype=torch.float32, device="cuda")
    sm = torch.empty((N, K, nr), dtype=torch.int32, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_LM_HEAD, N=N, B=B, row0=1, d=d, V=V, dtype=dt)
    ws = _ws(wsb)
    dfl.dfl_lm_head_argmax(dev(X), N, B, 1, d, dt, dev(g), 1e-6, dev(W, dtype if dtype == "bf16" else None), V, am,
                           lg, (K, T, seed), sm, ws, wsb)
    z = host(lg)
    check_samples(host(sm), lambda n, j: z[n * nr + j], seed, K, T, [(n, j) for n in range(N) for j in range(nr)])
    assert np.array_equal(host(am).reshape(-1), orc.argmax_lowest(z))


# ------------------------------------------------------------- acceptance --

def _golden_greedy():
    import os
    rows = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "greedy_cases.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                d_, t_, a_, b_ = [p.split() for p in line.split("|")]
                rows.append(([int(x) for x in d_], [int(x) for x in t_], int(a_[0]), int(b_[0])))
    return rows


def test_greedy_accept_golden_and_planted():
    for d_, t_, a_, b_ in _golden_greedy():
        n = len(d_)
        al = torch.empty(1, dtype=torch.int32, device="cuda")
        bo = torch.empty(1, dtype=torch.int32, device="cuda")
        dfl.dfl_greedy_accept(dev(np.array([d_], np.int32)), dev(np.array([t_], np.int32)), 1, n, al, bo)
        assert (int(al.item()), int(bo.item())) == (a_, b_)
    from dfl_synth import Workload, geometric_prefix, plant_targets
    w = Workload("p", N=500, d=1, Hq=1, Hkv=1, hd=2, D=1, L=1, B=40, C=1, V=50, dtype="f32", seed=9, geom_p=0.1)
    rng = np.random.default_rng(2)
    drafts = rng.integers(0, w.V, (w.N, w.B - 1)).astype(np.int32)
    t = plant_targets(w, drafts)
    al = torch.empty(w.N, dtype=torch.int32, device="cuda")
    bo = torch.empty(w.N, dtype=torch.int32, device="cuda")
    dfl.dfl_greedy_accept(dev(drafts), dev(t), w.N, w.B - 1, al, bo)
    G = geometric_prefix(w)
    assert np.array_equal(host(al), G)
    assert np.array_equal(host(bo), t[np.arange(w.N), G])


@pytest.mark.parametrize("N,K,G,V", [(3, 4, 5, 1000), (2, 8, 32, 2048), (1, 64, 1, 96), (2, 3, 40, 1001)])
def test_self_select(N, K, G, V):
    rng = np.random.default_rng(N * K + G)
    vlog = rng_bf16(rng, (N, K, G + 1, V), 4.0)
    drafts = rng.integers(0, V, (N, K, G)).astype(np.int32)
    # make some drafts follow the verifier's argmax for a while, so acceptance is non-trivial
    for n in range(N):
        for k in range(K):
            p = rng.integers(0, G + 1)
            drafts[n, k, :p] = np.argmax(vlog[n, k, :p], axis=-1)
    sc = torch.empty((N, K), dtype=torch.float32, device="cuda")
    se, al, bo = (torch.empty(N, dtype=torch.int32, device="cuda") for _ in range(3))
    wsb = dfl.workspace_size(dfl.DFL_OP_SELF_SELECT, N=N, K=K, G=G)
    ws = _ws(wsb)
    dfl.dfl_self_select(dev(vlog, "bf16"), dfl.DFL_BF16, dev(drafts), N, K, G, V, sc, se, al, bo, ws, wsb)
    for n in range(N):
        scores, ks, a, b = orc.self_select(vlog[n], drafts[n])
        g_sc = host(sc)[n]
        assert np.allclose(g_sc, scores, rtol=1e-4, atol=0), (g_sc, scores)
        top = np.sort(scores)[::-1]
        k_gpu = int(host(se)[n])
        if K > 1 and (top[0] - top[1]) <= 1e-5 * top[0]:
            assert scores[k_gpu] >= top[1]      # near-tie: either top draft is correct
        else:
            assert k_gpu == ks
        t = [int(np.argmax(vlog[n, k_gpu, j])) for j in range(G + 1)]
        assert (int(host(al)[n]), int(host(bo)[n])) == orc.greedy_accept(drafts[n, k_gpu], t)


def test_bounded_wait_times_out_and_context_survives():
    st = torch.empty(1, dtype=torch.int32, device="cuda")
    dfl.dfl_selftest_bounded_wait(20_000_000, st)   # 20 ms on a barrier nothing arrives at
    torch.cuda.synchronize()
    assert int(st.item()) == 6                       # DFL_ERR_TIMEOUT
    al = torch.empty(1, dtype=torch.int32, device="cuda")
    bo = torch.empty(1, dtype=torch.int32, device="cuda")
    dfl.dfl_greedy_accept(dev(np.array([[1, 2]], np.int32)), dev(np.array([[1, 5, 7]], np.int32)), 1, 2, al, bo)
    assert (int(al.item()), int(bo.item())) == (1, 5)



# --------------------------------------------------------- feed-forward --

@pytest.mark.parametrize("N,B,d,F", [(3, 16, 256, 384), (20, 16, 512, 1024), (2, 33, 256, 192),
                                     (4, 16, 1024, 4096)])   # a down projection of 4 tiles over 64 k-blocks
def test_block_ffn_bf16(N, B, d, F):
    rng = np.random.default_rng(N * F)
    Xb = rng.standard_normal((N * B, d)).astype(np.float32)
    g = rng.uniform(0.5, 1.5, d).astype(np.float32)
    W1, W3 = rng_bf16(rng, (F, d), d ** -0.5), rng_bf16(rng, (F, d), d ** -0.5)
    W2 = rng_bf16(rng, (d, F), F ** -0.5)
    Xd = dev(Xb)
    wsb = dfl.workspace_size(dfl.DFL_OP_BLOCK_FFN, N=N, B=B, d=d, F=F, dtype=dfl.DFL_BF16)
    ws = _ws(wsb)
    dfl.dfl_block_ffn(Xd, N, B, d, dfl.DFL_BF16, dev(g), 1e-6, dev(W1, "bf16"), dev(W3, "bf16"), dev(W2, "bf16"), F,
                      ws, wsb)
    ref = orc.swiglu_ffn(Xb, g, W1, W3, W2, 1e-6)
    assert_bf16_close(host(Xd) - Xb, ref - Xb, "ffn")


def test_block_ffn_f32():
    rng = np.random.default_rng(3)
    N, B, d, F = 1, 16, 128, 200
    f = lambda s, sc=1.0: (rng.standard_normal(s) * sc).astype(np.float32)
    Xb, g = f((N * B, d)), rng.uniform(0.5, 1.5, d).astype(np.float32)
    W1, W3, W2 = f((F, d), d ** -0.5), f((F, d), d ** -0.5), f((d, F), F ** -0.5)
    Xd = dev(Xb)
    wsb = dfl.workspace_size(dfl.DFL_OP_BLOCK_FFN, N=N, B=B, d=d, F=F, dtype=dfl.DFL_F32)
    ws = _ws(wsb)
    dfl.dfl_block_ffn(Xd, N, B, d, dfl.DFL_F32, dev(g), 1e-6, dev(W1), dev(W3), dev(W2), F, ws, wsb)
    assert_f32_close(host(Xd), orc.swiglu_ffn(Xb, g, W1, W3, W2, 1e-6), "Xb")
