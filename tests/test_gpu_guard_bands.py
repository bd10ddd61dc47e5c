"""Guard bands around every output and workspace buffer (GPU).

compute-sanitizer is closed on this machine, so out-of-bounds writes are looked
for this way instead: each buffer a call writes (its outputs and its
workspace of exactly dfl_workspace_size() bytes) sits between two 4 KiB bands
of a known byte, and after the call the bands must be unchanged.  Shapes are
ragged in every tile dimension.
"""
import numpy as np
import pytest
import torch

import block_diffusion_speculative_dfl_gb300 as dfl
from dfl_synth import (Workload, gen_block_init, gen_fc_weights, gen_gains, gen_hidden, gen_layer_weights,
                       gen_lm_head, gen_mix_logits, gen_verifier_logits)
from gpu_util import dev, rng_bf16

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    """A device tensor of `shape` and `dtype` between two guard bands."""

    def __init__(self, shape, dtype, init=None):
        esz = torch.empty((), dtype=dtype).element_size()
        self.n = int(np.prod(shape)) * esz
        self.buf = torch.full((self.n + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + self.n].view(dtype).view(shape)
        if init is not None:
            self.t.copy_(init)

    def check(self, name):
        torch.cuda.synchronize()
        b = self.buf.cpu().numpy()
        lo, hi = b[:GUARD], b[GUARD + self.n:]
        assert (lo == PATTERN).all(), f"{name}: {int((lo != PATTERN).sum())} bytes written below the buffer"
        assert (hi == PATTERN).all(), f"{name}: {int((hi != PATTERN).sum())} bytes written past the buffer"


def _ws(op, **shape):
    nbytes = dfl.workspace_size(op, **shape)
    return Guarded((max(nbytes, 16),), torch.uint8), nbytes


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dfl.build()
    dfl.load()
    torch.cuda.set_device(0)
    yield
    assert dfl.dfl_get_device_error() == 0


def test_mix_rmsnorm_writes_only_its_output():
    rows, d, L, D = 149, 256, 3, 2
    rng = np.random.default_rng(1)
    H = rng_bf16(rng, (L, rows, d))
    Xc = Guarded((D, rows, d), torch.bfloat16)
    dfl.dfl_layer_mix_rmsnorm(dev(H, "bf16"), rows * d, L, rows, d, dfl.DFL_BF16, D,
                              dev(rng.standard_normal((D, L)).astype(np.float32)), dev(np.ones((D, d), np.float32)),
                              1e-6, Xc.t, rows * d)
    Xc.check("Xc")


def test_dual_kv_proj_writes_only_its_outputs():
    N, C, B, d, Hq, Hkv, hd = 2, 200, 16, 520, 8, 2, 128
    rng = np.random.default_rng(2)
    kv, qd = Hkv * hd, Hq * hd
    W = {k: dev(rng_bf16(rng, (n, d), d ** -0.5), "bf16")
         for k, n in (("Wq", qd), ("Wkc", kv), ("Wvc", kv), ("Wkb", kv), ("Wvb", kv))}
    table = torch.empty((C + B, hd // 2, 2), dtype=torch.float32, device="cuda")
    dfl.dfl_rope_table(table, C + B, hd, 1e6)
    out = {k: Guarded(s, torch.bfloat16) for k, s in
           {"Q": (N * B, qd), "Kc": (N * C, kv), "Vc": (N * C, kv), "Kb": (N * B, kv), "Vb": (N * B, kv)}.items()}
    ws, wsb = _ws(dfl.DFL_OP_DUAL_KV_PROJ, N=N, B=B, d=d, dtype=dfl.DFL_BF16)
    dfl.dfl_dual_kv_proj(dev(rng_bf16(rng, (N * C, d)), "bf16"), dev(rng.standard_normal((N * B, d)).astype(np.float32)),
                         N, C, B, d, dfl.DFL_BF16, dev(np.ones(d, np.float32)), 1e-6, W["Wq"], W["Wkc"], W["Wvc"],
                         W["Wkb"], W["Wvb"], Hq, Hkv, hd, table, out["Q"].t, out["Kc"].t, out["Vc"].t, out["Kb"].t,
                         out["Vb"].t, ws.t, wsb)
    for k, g in out.items():
        g.check(k)
    ws.check("workspace")


@pytest.mark.parametrize("N,C,B,Hq,Hkv,hd,d", [(3, 150, 12, 4, 2, 128, 256), (2, 90, 16, 6, 2, 64, 192),
                                                (1, 1000, 33, 32, 8, 128, 512)])
def test_block_attn_writes_only_its_outputs(N, C, B, Hq, Hkv, hd, d):
    rng = np.random.default_rng(N * 7 + C)
    q = lambda *s: dev(rng_bf16(rng, s), "bf16")
    Xb = Guarded((N * B, d), torch.float32, torch.from_numpy(rng.standard_normal((N * B, d)).astype(np.float32)))
    ws, wsb = _ws(dfl.DFL_OP_BLOCK_ATTN, N=N, C=C, B=B, Hq=Hq, Hkv=Hkv, hd=hd, dtype=dfl.DFL_BF16)
    dfl.dfl_block_attn(q(N * B, Hq, hd), q(N * C, Hkv, hd), q(N * C, Hkv, hd), q(N * B, Hkv, hd), q(N * B, Hkv, hd),
                       N, C, B, Hq, Hkv, hd, dfl.DFL_BF16, dev(rng_bf16(rng, (d, Hq * hd), (Hq * hd) ** -0.5), "bf16"),
                       d, Xb.t, ws.t, wsb)
    Xb.check("Xb")
    ws.check("workspace")


@pytest.mark.parametrize("sample", [None, (4, 1.5, 7)])
def test_lm_head_writes_only_its_outputs(sample):
    N, B, row0, d, V = 2, 9, 1, 256, 5003
    rng = np.random.default_rng(3)
    nr = B - row0
    am = Guarded((N, nr), torch.int32)
    lg = Guarded((N * nr, V), torch.float32)
    sm = Guarded((N, sample[0], nr), torch.int32) if sample else None
    ws, wsb = _ws(dfl.DFL_OP_LM_HEAD, N=N, B=B, row0=row0, d=d, V=V, dtype=dfl.DFL_BF16)
    dfl.dfl_lm_head_argmax(dev(rng.standard_normal((N, B, d)).astype(np.float32)), N, B, row0, d, dfl.DFL_BF16,
                           dev(np.ones(d, np.float32)), 1e-6, dev(rng_bf16(rng, (V, d), d ** -0.5), "bf16"), V, am.t,
                           lg.t, sample, sm.t if sm else None, ws.t, wsb)
    am.check("argmax")
    lg.check("logits")
    if sm:
        sm.check("samples")
    ws.check("workspace")


def test_acceptance_epilogues_write_only_their_outputs():
    N, K, G, V = 3, 4, 8, 1000
    rng = np.random.default_rng(4)
    vlog = dev(rng_bf16(rng, (N, K, G + 1, V), 4.0), "bf16")
    drafts = dev(rng.integers(0, V, (N, K, G)).astype(np.int32))
    logits = dev(rng.standard_normal((N * G, V)).astype(np.float32))
    al, bo = Guarded((N,), torch.int32), Guarded((N,), torch.int32)
    dfl.dfl_greedy_accept(dev(rng.integers(0, 3, (N, G)).astype(np.int32)),
                          dev(rng.integers(0, 3, (N, G + 1)).astype(np.int32)), N, G, al.t, bo.t)
    al.check("greedy accept_len")
    bo.check("greedy bonus")
    sc, se = Guarded((N, K), torch.float32), Guarded((N,), torch.int32)
    ws, wsb = _ws(dfl.DFL_OP_SELF_SELECT, N=N, K=K, G=G)
    dfl.dfl_self_select(vlog, dfl.DFL_BF16, drafts, N, K, G, V, sc.t, se.t, al.t, bo.t, ws.t, wsb)
    for g, name in ((sc, "scores"), (se, "selected"), (al, "accept_len"), (bo, "bonus"), (ws, "workspace")):
        g.check("self-select " + name)
    alpha, tpd = Guarded((N, K, G), torch.float32), Guarded((N, K), torch.float32)
    ws, wsb = _ws(dfl.DFL_OP_TV_ACCEPTANCE, N=N, K=K, G=G)
    dfl.dfl_tv_acceptance(logits, 1.5, vlog, dfl.DFL_BF16, N, K, G, V, alpha.t, tpd.t, ws.t, wsb)
    for g, name in ((alpha, "alpha"), (tpd, "tokens per draft"), (ws, "workspace")):
        g.check("tv " + name)
    nt = Guarded((N,), torch.int32)
    ws, wsb = _ws(dfl.DFL_OP_SPEC_ACCEPT, N=N, G=G, V=V)
    dfl.dfl_spec_accept(logits, 1.5, vlog, dfl.DFL_BF16, drafts, se.t, N, K, G, V, 11, al.t, nt.t, ws.t, wsb)
    for g, name in ((al, "accept_len"), (nt, "next token"), (ws, "workspace")):
        g.check("stochastic acceptance " + name)


def test_block_ffn_writes_only_its_outputs():
    N, B, d, F = 3, 16, 256, 384
    rng = np.random.default_rng(5)
    Xb = Guarded((N * B, d), torch.float32, torch.from_numpy(rng.standard_normal((N * B, d)).astype(np.float32)))
    ws, wsb = _ws(dfl.DFL_OP_BLOCK_FFN, N=N, B=B, d=d, F=F, dtype=dfl.DFL_BF16)
    dfl.dfl_block_ffn(Xb.t, N, B, d, dfl.DFL_BF16, dev(np.ones(d, np.float32)), 1e-6,
                      dev(rng_bf16(rng, (F, d), d ** -0.5), "bf16"), dev(rng_bf16(rng, (F, d), d ** -0.5), "bf16"),
                      dev(rng_bf16(rng, (d, F), F ** -0.5), "bf16"), F, ws.t, wsb)
    Xb.check("Xb")
    ws.check("workspace")


def test_no_alloc_self_select_writes_only_its_outputs():
    N, K, G, V = 3, 4, 8, 1000
    rng = np.random.default_rng(6)
    vlog = dev(rng_bf16(rng, (N, K, G + 1, V), 4.0), "bf16")
    drafts = dev(rng.integers(0, V, (N, K, G)).astype(np.int32))
    sc, se = Guarded((N, K), torch.float32), Guarded((N,), torch.int32)
    al, bo = Guarded((N,), torch.int32), Guarded((N,), torch.int32)
    dfl.dfl_self_select_noalloc(vlog, dfl.DFL_BF16, drafts, N, K, G, V, sc.t, se.t, al.t, bo.t)
    for g, name in ((sc, "scores"), (se, "selected"), (al, "accept_len"), (bo, "bonus")):
        g.check("no-alloc self-select " + name)


def test_sampled_greedy_and_philox_write_only_their_outputs():
    N, K, G, V = 3, 4, 8, 1001
    rng = np.random.default_rng(7)
    vlog = dev(rng_bf16(rng, (N, K, G + 1, V), 4.0), "bf16")
    drafts = dev(rng.integers(0, V, (N, K, G)).astype(np.int32))
    al, nt = Guarded((N,), torch.int32), Guarded((N,), torch.int32)
    ws, wsb = _ws(dfl.DFL_OP_SAMPLED_GREEDY, N=N, G=G, V=V)
    dfl.dfl_sampled_greedy_accept(vlog, dfl.DFL_BF16, drafts, None, N, K, G, V, 5, al.t, nt.t, ws.t, wsb)
    for g, name in ((al, "accept_len"), (nt, "next token"), (ws, "workspace")):
        g.check("sampled greedy " + name)
    out = Guarded((5, 4), torch.int32)
    dfl.dfl_philox4x32_10(dev(rng.integers(0, 1 << 31, (5, 6)).astype(np.int32)), 5, out.t)
    out.check("philox")


def test_fc_fuse_writes_only_its_outputs():
    rows, d, L = 300, 256, 3
    rng = np.random.default_rng(8)
    Xc = Guarded((rows, d), torch.bfloat16)
    ws, wsb = _ws(dfl.DFL_OP_FC_FUSE, N=rows, C=1, d=d, dtype=dfl.DFL_BF16)
    dfl.dfl_fc_fuse(dev(rng_bf16(rng, (L, rows, d)), "bf16"), rows * d, L, rows, d, dfl.DFL_BF16,
                    dev(rng_bf16(rng, (d, L * d), (L * d) ** -0.5), "bf16"), dev(np.ones(d, np.float32)), 1e-6, Xc.t,
                    ws.t, wsb)
    Xc.check("Xc")
    ws.check("workspace")


def _small_model(w, **kw):
    shape = dfl.DraftShape(N=w.N, d=w.d, Hq=w.Hq, Hkv=w.Hkv, hd=w.hd, D=w.D, L=w.L, B=w.B, C=w.C, V=w.V,
                           dtype=w.dtype, K=w.K, T=w.T, seed=w.philox_seed, eps=w.eps, rope_theta=w.rope_theta,
                           fc=w.fc)
    g_mix, g_blk, g_fin = gen_gains(w)
    W_fc, g_fc = gen_fc_weights(w) if w.fc else (None, None)
    W_lm = torch.from_numpy(gen_lm_head(w, as_bits=True).view(np.int16)).view(torch.bfloat16)
    return dfl.DraftModel(shape, gen_mix_logits(w), g_mix, g_blk, g_fin, [gen_layer_weights(w, l) for l in range(w.D)],
                          W_lm, W_fc=W_fc, fc_gain=g_fc, **kw)


def _guard_outputs(model, names):
    """Replace the model's output buffers by guarded ones of the same shapes."""
    gs = {}
    for k in names:
        t = getattr(model, k)
        gs[k] = Guarded(tuple(t.shape), t.dtype)
        setattr(model, k, gs[k].t)
    return gs


@pytest.mark.parametrize("fc,host_input", [(0, False), (1, False), (0, True)])
def test_draft_step_writes_only_its_outputs(fc, host_input):
    w = Workload("gbstep", N=3, d=256, Hq=4, Hkv=2, hd=64, D=2, L=3, B=16, C=90, V=1200, dtype="bf16", seed=91,
                 fc=fc)
    model = _small_model(w)
    model.want_logits(True)
    gs = _guard_outputs(model, ("Xb", "draft", "logits", "accept_len", "bonus"))
    op = dfl._lib.DFL_OP_DRAFT_STEP_HOST if host_input else dfl.DFL_OP_DRAFT_STEP
    ws, wsb = _ws(op, N=w.N, C=w.C, B=w.B, d=w.d, Hq=w.Hq, Hkv=w.Hkv, hd=w.hd, D=w.D, L=w.L, V=w.V, K=0, G=w.B - 1,
                  row0=1, dtype=dfl.DFL_BF16, fc=fc)
    model.ws, model.ws_bytes = ws.t, wsb
    Hbits = torch.from_numpy(gen_hidden(w, as_bits=True).view(np.int16)).view(torch.bfloat16)
    X0 = torch.from_numpy(gen_block_init(w)).cuda()
    target = dev(np.random.default_rng(9).integers(0, w.V, (w.N, w.B)).astype(np.int32))
    if host_input:
        H_dev = Guarded(tuple(Hbits.shape), torch.bfloat16)
        model._step_host(Hbits.pin_memory(), H_dev.t, X0, target, None, 2, torch.cuda.current_stream())
        H_dev.check("H_dev")
    else:
        model.step(Hbits.cuda(), X0, target=target)
    for k, g in gs.items():
        g.check(k)
    ws.check("workspace")


@pytest.mark.parametrize("rule", [1, 2])
def test_self_selection_step_writes_only_its_outputs(rule):
    w = Workload("gbsel", N=3, d=256, Hq=4, Hkv=2, hd=64, D=2, L=3, B=9, C=80, V=1500, dtype="bf16", seed=93,
                 K=4, T=1.5, philox_seed=0x5EEDD1F5)
    model = _small_model(w, tv=True, accept_rule=rule, accept_seed=3)
    gs = _guard_outputs(model, ("Xb", "draft", "accept_len", "bonus", "samples", "scores", "selected", "tv_alpha",
                                "tv_tokens"))
    ws, wsb = _ws(dfl.DFL_OP_DRAFT_STEP, N=w.N, C=w.C, B=w.B, d=w.d, Hq=w.Hq, Hkv=w.Hkv, hd=w.hd, D=w.D, L=w.L,
                  V=w.V, K=w.K, G=w.B - 1, row0=1, dtype=dfl.DFL_BF16)
    model.ws, model.ws_bytes = ws.t, wsb
    vlog = torch.from_numpy(gen_verifier_logits(w, as_bits=True).view(np.int16)).cuda().view(torch.bfloat16)
    H = torch.from_numpy(gen_hidden(w, as_bits=True).view(np.int16)).view(torch.bfloat16).cuda()
    model.step(H, torch.from_numpy(gen_block_init(w)).cuda(), vlog=vlog)
    for k, g in gs.items():
        g.check(k)
    ws.check("workspace")
