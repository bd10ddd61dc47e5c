"""Whole draft steps through dfl_draft_step against the fp64 oracle (GPU).

Small shapes are checked completely; the full-size workloads run in the same
launch configuration the benchmark times and are checked on sampled
sequences (the oracle recomputes those one by one) plus bit-exact epilogue
checks on every sequence from the GPU's own logits / verifier buffers.
"""
import numpy as np
import pytest
import torch

import block_diffusion_speculative_dfl_gb300 as dfl
import oracle as orc
from dfl_synth import (WORKLOADS, Workload, gen_block_init, gen_fc_weights, gen_ffn_gains, gen_gains, gen_hidden,
                       gen_layer_weights, gen_lm_head, gen_mix_logits, gen_verifier_logits, geometric_prefix,
                       plant_targets)
from gpu_util import SAMPLE_BAND, assert_bf16_close, assert_f32_close, check_samples, host, near_tie_cap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dfl.build()
    dfl.load()
    torch.cuda.set_device(0)
    yield
    assert dfl.dfl_get_device_error() == 0


def _shape(w):
    return {"Hq": w.Hq, "Hkv": w.Hkv, "hd": w.hd}


def _model(w, random_gains=False):
    mix = gen_mix_logits(w)
    g_mix, g_blk, g_fin = gen_gains(w, random=random_gains)
    layers = [gen_layer_weights(w, l) for l in range(w.D)]
    W_lm = gen_lm_head(w, as_bits=(w.dtype == "bf16")) if w.V > 0 else None
    shape = dfl.DraftShape(N=w.N, d=w.d, Hq=w.Hq, Hkv=w.Hkv, hd=w.hd, D=w.D, L=w.L, B=w.B, C=w.C, V=w.V,
                           dtype=w.dtype, K=w.K, T=w.T, seed=w.philox_seed, eps=w.eps, rope_theta=w.rope_theta,
                           F=w.F, fc=w.fc)
    g_ffn = gen_ffn_gains(w, random=random_gains)
    W_lm_t = None
    if W_lm is not None:
        W_lm_t = torch.from_numpy(W_lm.view(np.int16)).view(torch.bfloat16) if w.dtype == "bf16" else \
            torch.from_numpy(W_lm)
    W_fc, g_fc = gen_fc_weights(w, random_gain=random_gains) if w.fc else (None, None)
    model = dfl.DraftModel(shape, None if w.fc else mix, None if w.fc else g_mix, g_blk, g_fin, layers, W_lm_t,
                           ffn_gain=g_ffn, W_fc=W_fc, fc_gain=g_fc)
    return model, dict(mix=mix, g_mix=g_mix, g_blk=g_blk, g_fin=g_fin, layers=layers, W_lm=W_lm, g_ffn=g_ffn,
                       W_fc=W_fc, g_fc=g_fc)


def _hidden_dev(w):
    if w.dtype == "bf16":
        return torch.from_numpy(gen_hidden(w, as_bits=True).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(gen_hidden(w)).cuda()


def _oracle_seq(w, p, n):
    """fp64 oracle draft forward + logits for sequence n."""
    Hn = gen_hidden(w, seqs=[n])
    Xb0 = gen_block_init(w)[n]
    layers = [dict(W, g_ffn=p["g_ffn"][l]) if w.F > 0 else W for l, W in enumerate(p["layers"])]
    fused = (p["W_fc"], p["g_fc"]) if w.fc else None
    out = orc.draft_forward(Xb0, Hn, p["mix"], p["g_mix"], p["g_blk"], layers, _shape(w), w.eps, w.rope_theta,
                            fused=fused)
    z = None
    if w.V > 0:
        from dfl_synth import bits_to_f32
        W_lm = bits_to_f32(p["W_lm"]) if w.dtype == "bf16" else p["W_lm"]
        z = orc.lm_head_logits(out["Xb"][1:], p["g_fin"], w.eps, W_lm)
    return out["Xb"], z


def _run_greedy_workload(w, seqs, random_gains=False):
    model, p = _model(w, random_gains)
    model.want_logits()
    H = _hidden_dev(w)
    X0 = torch.from_numpy(gen_block_init(w)).cuda()
    model.step(H, X0)
    torch.cuda.synchronize()
    drafts = host(model.draft)
    target = torch.from_numpy(plant_targets(w, drafts)).cuda()
    model.step(H, X0, target=target)
    torch.cuda.synchronize()
    # the step is deterministic: the second pass drafts the same tokens
    assert np.array_equal(host(model.draft), drafts)
    z = host(model.logits).reshape(w.N, w.B - 1, w.V)
    # argmax bit-exact on the GPU's own logits, every sequence
    assert np.array_equal(orc.argmax_lowest(z), drafts)
    # greedy acceptance bit-exact, every sequence; equals the planted prefix
    t = host(target)
    G = geometric_prefix(w)
    for n in range(w.N):
        a, b = orc.greedy_accept(drafts[n], t[n])
        assert (a, b) == (int(host(model.accept_len)[n]), int(host(model.bonus)[n]))
        assert a == G[n]
    Xb = host(model.Xb)
    for n in seqs:
        ref_xb, ref_z = _oracle_seq(w, p, n)
        if w.dtype == "f32":
            assert_f32_close(Xb[n], ref_xb, f"Xb[{n}]")
            assert_f32_close(z[n], ref_z, f"logits[{n}]")
        else:
            assert_bf16_close(Xb[n] - gen_block_init(w)[n], ref_xb - gen_block_init(w)[n], f"dXb[{n}]",
                              mean_bar=8e-3)
            assert_bf16_close(z[n], ref_z, f"logits[{n}]", mean_bar=8e-3)


def test_tiny_f32_workload_end_to_end():
    _run_greedy_workload(WORKLOADS["tiny_f32"], seqs=[0])


def test_tiny_f32_random_gains():
    _run_greedy_workload(WORKLOADS["tiny_f32"], seqs=[0], random_gains=True)


def test_small_bf16_drafter():
    w = Workload("small", N=3, d=512, Hq=8, Hkv=2, hd=128, D=3, L=5, B=16, C=200, V=3000, dtype="bf16", seed=41,
                 geom_p=0.3)
    _run_greedy_workload(w, seqs=[0, 2], random_gains=True)


def test_small_bf16_drafter_hd64():
    w = Workload("small64", N=2, d=320, Hq=8, Hkv=2, hd=64, D=2, L=7, B=8, C=130, V=1001, dtype="bf16", seed=43,
                 geom_p=0.2)
    _run_greedy_workload(w, seqs=[1])


def _run_select_workload(w, seqs, rows_checked):
    model, p = _model(w)
    model.want_logits()
    H = _hidden_dev(w)
    X0 = torch.from_numpy(gen_block_init(w)).cuda()
    vlog_bits = gen_verifier_logits(w, as_bits=True)
    vlog = torch.from_numpy(vlog_bits.view(np.int16)).cuda().view(torch.bfloat16)
    model.step(H, X0, vlog=vlog)
    torch.cuda.synchronize()
    G = w.gamma
    z = host(model.logits).reshape(w.N, G, w.V)
    samples = host(model.samples)
    assert np.array_equal(orc.argmax_lowest(z), host(model.draft))
    # samples: the oracle's inverse-CDF draw on the same logits
    check_samples(samples, lambda n, j: z[n, j], w.philox_seed, w.K, w.T, [(n, j) for n in seqs for j in rows_checked])
    # selection and acceptance from the GPU's samples and the verifier buffer
    from dfl_synth import bits_to_f32
    sel, al, bo, sc = host(model.selected), host(model.accept_len), host(model.bonus), host(model.scores)
    for n in seqs:
        vl = bits_to_f32(vlog_bits[n])
        scores, ks, a, b = orc.self_select(vl, samples[n])
        assert np.allclose(sc[n], scores, rtol=1e-4, atol=0)
        top = np.sort(scores)[::-1]
        if w.K > 1 and top[0] - top[1] <= 1e-5 * top[0]:
            assert scores[sel[n]] >= top[1]
        else:
            assert sel[n] == ks
        t = [int(np.argmax(vl[sel[n], j])) for j in range(G + 1)]
        assert (int(al[n]), int(bo[n])) == orc.greedy_accept(samples[n, sel[n]], t)
    Xb = host(model.Xb)
    for n in seqs[:1]:
        ref_xb, ref_z = _oracle_seq(w, p, n)
        X0n = gen_block_init(w)[n]
        assert_bf16_close(Xb[n] - X0n, ref_xb - X0n, f"dXb[{n}]", mean_bar=8e-3)
        assert_bf16_close(z[n], ref_z, f"logits[{n}]", mean_bar=8e-3)


def test_small_self_selection_step():
    w = Workload("smallsel", N=3, d=512, Hq=8, Hkv=2, hd=128, D=2, L=4, B=9, C=100, V=2000, dtype="bf16", seed=47,
                 K=8, T=1.5, philox_seed=0x5EEDD1F5)
    _run_select_workload(w, seqs=[0, 1, 2], rows_checked=range(w.gamma))


def test_step_from_host_matches_device_step():
    w = Workload("e2e", N=2, d=256, Hq=4, Hkv=2, hd=64, D=2, L=3, B=16, C=64, V=1000, dtype="bf16", seed=53,
                 geom_p=0.3)
    model, _ = _model(w)
    H_host = torch.from_numpy(gen_hidden(w, as_bits=True).view(np.int16)).view(torch.bfloat16).pin_memory()
    X_host = torch.from_numpy(gen_block_init(w)).pin_memory()
    model.step(H_host.cuda(), X_host.cuda())
    torch.cuda.synchronize()
    drafts = host(model.draft)
    t_host = torch.from_numpy(plant_targets(w, drafts)).pin_memory()
    out, _ = model.step_from_host(H_host, X_host, t_host)
    assert np.array_equal(out["draft"].numpy(), drafts)
    assert np.array_equal(out["accept_len"].numpy(), geometric_prefix(w))


@pytest.mark.parametrize("F,chunks,fc", [(0, 1, 0), (0, 2, 0), (0, 5, 0), (0, 16, 0), (384, 3, 0), (0, 3, 1)])
def test_host_input_step_is_bitwise_the_device_step(F, chunks, fc):
    # dfl_draft_step_host copies H in groups of sequences and mixes (or fuses)
    # and projects each group as it lands: every row's arithmetic is the
    # device step's, so the residual stream and the drafts must agree bit for bit.
    w = Workload("hoststep", N=5, d=256, Hq=4, Hkv=2, hd=128, D=3, L=4, B=16, C=96, V=1500, dtype="bf16", seed=59,
                 geom_p=0.3, F=F, fc=fc)
    model, _ = _model(w)
    H_host = torch.from_numpy(gen_hidden(w, as_bits=True).view(np.int16)).view(torch.bfloat16).pin_memory()
    X0 = torch.from_numpy(gen_block_init(w)).cuda()
    model.want_logits(True)
    model.step(H_host.cuda(), X0)
    torch.cuda.synchronize()
    Xb_ref, drafts, z_ref = host(model.Xb).copy(), host(model.draft).copy(), host(model.logits).copy()
    H_dev = torch.empty(H_host.shape, dtype=torch.bfloat16, device="cuda")
    model.Xb.zero_()
    model._step_host(H_host, H_dev, X0, None, None, chunks, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert np.array_equal(host(model.Xb).view(np.uint32), Xb_ref.view(np.uint32))
    assert np.array_equal(host(model.logits).view(np.uint32), z_ref.view(np.uint32))
    assert np.array_equal(host(model.draft), drafts)
    assert np.array_equal(host(H_dev.view(torch.int16)), H_host.view(torch.int16).numpy())


def test_step_replays_from_a_cuda_graph():
    # A call neither allocates nor synchronises and its pointers and launch
    # shapes are fixed for a shape, so a step captured once into a CUDA graph
    # replays the eager step bit for bit.
    w = Workload("graph", N=3, d=256, Hq=4, Hkv=2, hd=128, D=2, L=3, B=16, C=96, V=1500, dtype="bf16", seed=61,
                 geom_p=0.3)
    model, _ = _model(w)
    model.want_logits(True)
    H = _hidden_dev(w)
    X0 = torch.from_numpy(gen_block_init(w)).cuda()
    model.step(H, X0)
    torch.cuda.synchronize()
    target = torch.from_numpy(plant_targets(w, host(model.draft))).cuda()
    model.step(H, X0, target=target)   # eager, outside any capture
    torch.cuda.synchronize()
    ref = {k: host(getattr(model, k)).copy() for k in ("Xb", "logits", "draft", "accept_len", "bonus")}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        model.step(H, X0, target=target)
    for k in ref:
        getattr(model, k).zero_()
    torch.cuda.synchronize()
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for k, v in ref.items():
            got = host(getattr(model, k))
            assert np.array_equal(got.view(np.uint32), v.view(np.uint32)), k
    assert np.array_equal(ref["accept_len"], geometric_prefix(w))


# ---------------------------------------------------------- full sizes --

def test_qwen3_8b_single_layer_full_size():
    w = WORKLOADS["qwen3_8b_layer"]
    model, p = _model(w)
    H = _hidden_dev(w)
    X0 = torch.from_numpy(gen_block_init(w)).cuda()
    model.step(H, X0)
    torch.cuda.synchronize()
    ref_xb, _ = _oracle_seq(w, p, 0)
    X0n = gen_block_init(w)[0]
    assert_bf16_close(host(model.Xb)[0] - X0n, ref_xb - X0n, "dXb", mean_bar=8e-3)


def test_qwen3_8b_drafter_full_size():
    _run_greedy_workload(WORKLOADS["qwen3_8b_drafter"], seqs=[0, 31])


def test_gpt_oss_20b_drafter_full_size():
    _run_greedy_workload(WORKLOADS["gpt_oss_20b_drafter"], seqs=[5])


def test_specdiff2_selection_full_size():
    w = WORKLOADS["specdiff2_select"]
    _run_select_workload(w, seqs=[0, 15], rows_checked=[0, 1, 17, 31])


def test_self_selection_step_with_tv_and_stochastic_acceptance():
    w = Workload("selext", N=3, d=256, Hq=4, Hkv=2, hd=64, D=2, L=3, B=9, C=80, V=1500, dtype="bf16", seed=61,
                 K=4, T=1.5, philox_seed=0x5EEDD1F5)
    mix = gen_mix_logits(w)
    g_mix, g_blk, g_fin = gen_gains(w)
    layers = [gen_layer_weights(w, l) for l in range(w.D)]
    W_lm = gen_lm_head(w, as_bits=True)
    shape = dfl.DraftShape(N=w.N, d=w.d, Hq=w.Hq, Hkv=w.Hkv, hd=w.hd, D=w.D, L=w.L, B=w.B, C=w.C, V=w.V,
                           dtype=w.dtype, K=w.K, T=w.T, seed=w.philox_seed, eps=w.eps, rope_theta=w.rope_theta)
    seed = 0xABCDEF12345
    model = dfl.DraftModel(shape, mix, g_mix, g_blk, g_fin, layers,
                           torch.from_numpy(W_lm.view(np.int16)).view(torch.bfloat16), tv=True, accept_rule=1,
                           accept_seed=seed)
    model.want_logits()
    from dfl_synth import bits_to_f32
    vbits = gen_verifier_logits(w, as_bits=True)
    vlog = torch.from_numpy(vbits.view(np.int16)).cuda().view(torch.bfloat16)
    model.step(_hidden_dev(w), torch.from_numpy(gen_block_init(w)).cuda(), vlog=vlog)
    torch.cuda.synchronize()
    G = w.gamma
    z = host(model.logits).reshape(w.N, G, w.V)
    samples, sel = host(model.samples), host(model.selected)
    alpha = host(model.tv_alpha)
    near = 0
    for n in range(w.N):
        vl = bits_to_f32(vbits[n])
        ref = np.array([[orc.tv_alpha(z[n, j], w.T, vl[k, j]) for j in range(G)] for k in range(w.K)])
        assert np.max(np.abs(alpha[n] - ref)) <= 2e-5
        assert np.allclose(host(model.tv_tokens)[n], [orc.streak_score(r) for r in ref], rtol=1e-4, atol=1e-6)
        u_acc = [orc.draw_uniform_stream(seed, n, j, 0, 1) for j in range(G)]
        u_res = [orc.draw_uniform_stream(seed, n, j, 0, 2) for j in range(G + 1)]
        legit = orc.speculative_accept_outcomes(z[n], w.T, vl[sel[n]], samples[n, sel[n]], u_acc, u_res, 1e-5, 1e-5)
        assert (int(host(model.accept_len)[n]), int(host(model.bonus)[n])) in legit, (n, legit)
        near += len(legit) > 1
    assert near <= 1, near   # three sequences: a near tie at all is rare


def test_self_selection_step_with_sampled_greedy_acceptance():
    # accept_rule 2: the selected draft against the verifier's own samples
    w = Workload("selsg", N=4, d=256, Hq=4, Hkv=2, hd=64, D=2, L=3, B=9, C=80, V=1500, dtype="bf16", seed=63,
                 K=4, T=1.5, philox_seed=0x5EEDD1F5, verifier_scale=10.0)
    mix = gen_mix_logits(w)
    g_mix, g_blk, g_fin = gen_gains(w)
    layers = [gen_layer_weights(w, l) for l in range(w.D)]
    W_lm = gen_lm_head(w, as_bits=True)
    shape = dfl.DraftShape(N=w.N, d=w.d, Hq=w.Hq, Hkv=w.Hkv, hd=w.hd, D=w.D, L=w.L, B=w.B, C=w.C, V=w.V,
                           dtype=w.dtype, K=w.K, T=w.T, seed=w.philox_seed, eps=w.eps, rope_theta=w.rope_theta)
    seed = 0x1357924680
    model = dfl.DraftModel(shape, mix, g_mix, g_blk, g_fin, layers,
                           torch.from_numpy(W_lm.view(np.int16)).view(torch.bfloat16), accept_rule=2,
                           accept_seed=seed)
    from dfl_synth import bits_to_f32
    vbits = gen_verifier_logits(w, as_bits=True)
    vlog = torch.from_numpy(vbits.view(np.int16)).cuda().view(torch.bfloat16)
    model.step(_hidden_dev(w), torch.from_numpy(gen_block_init(w)).cuda(), vlog=vlog)
    torch.cuda.synchronize()
    G = w.gamma
    samples, sel = host(model.samples), host(model.selected)
    near, expected = 0, 0.0
    for n in range(w.N):
        vl = bits_to_f32(vbits[n])
        scores, ks, _, _ = orc.self_select(vl, samples[n])
        top = np.sort(scores)[::-1]
        assert sel[n] == ks or scores[sel[n]] >= top[1] >= top[0] * (1 - 1e-5)
        u = [orc.draw_uniform_stream(seed, n, j, 0, 3) for j in range(G + 1)]
        legit = orc.sampled_greedy_outcomes(vl[sel[n]], samples[n, sel[n]], u, SAMPLE_BAND)
        assert (int(host(model.accept_len)[n]), int(host(model.bonus)[n])) in legit, (n, legit)
        near += len(legit) > 1
        expected += sum(float(np.minimum(orc.softmax_t(vl[sel[n], j]), 2 * SAMPLE_BAND).sum()) for j in range(G + 1))
    assert near <= near_tie_cap(expected), (near, expected)


def test_small_bf16_drafter_with_dflash_fusion():
    w = Workload("smallfc", N=3, d=256, Hq=4, Hkv=2, hd=64, D=2, L=3, B=16, C=90, V=1200, dtype="bf16", seed=73,
                 geom_p=0.3, fc=1)
    _run_greedy_workload(w, seqs=[0, 2], random_gains=True)


def test_small_bf16_drafter_with_dflash_fusion_hd128():
    w = Workload("smallfc128", N=2, d=512, Hq=8, Hkv=2, hd=128, D=3, L=5, B=16, C=200, V=3000, dtype="bf16",
                 seed=79, geom_p=0.3, fc=1)
    _run_greedy_workload(w, seqs=[1])


def test_small_f32_drafter_with_dflash_fusion():
    w = Workload("smallfc32", N=1, d=128, Hq=2, Hkv=2, hd=64, D=2, L=3, B=8, C=40, V=500, dtype="f32", seed=83,
                 geom_p=0.3, hidden_scale=False, fc=1)
    _run_greedy_workload(w, seqs=[0], random_gains=True)


def test_qwen3_8b_drafter_dflash_full_size():
    _run_greedy_workload(WORKLOADS["qwen3_8b_drafter_dflash"], seqs=[3])



def test_small_bf16_drafter_with_ffn_layers():
    w = Workload("smallffn", N=3, d=256, Hq=4, Hkv=2, hd=64, D=2, L=3, B=16, C=90, V=1200, dtype="bf16", seed=67,
                 geom_p=0.3, F=384)
    _run_greedy_workload(w, seqs=[0, 2], random_gains=True)


def test_small_f32_drafter_with_ffn_layers():
    w = Workload("smallffn32", N=1, d=128, Hq=2, Hkv=2, hd=64, D=2, L=2, B=8, C=40, V=500, dtype="f32", seed=71,
                 geom_p=0.3, F=200, hidden_scale=False)
    _run_greedy_workload(w, seqs=[0], random_gains=True)


def test_qwen3_8b_drafter_ffn_full_size():
    _run_greedy_workload(WORKLOADS["qwen3_8b_drafter_ffn"], seqs=[7])
