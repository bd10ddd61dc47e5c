"""Draft steps over an incremental context K/V cache (dfl_draft_step_cached) vs the fp64 oracle (GPU).

The caches are filled by chains of cached steps (ragged appends with the
lengths advanced on the device), then a decoding step appends a few rows per
sequence and drafts a block.  Checked against the oracle: the cached keys and
values, the lengths, the block output and logits, argmax and greedy
acceptance (bit-exact on the GPU's own logits), and that cache rows past each
sequence's length are never written.
"""
import numpy as np
import pytest
import torch

import block_diffusion_speculative_dfl_gb300 as dfl
import oracle as orc
from dfl_synth import (WORKLOADS, Workload, bits_to_f32, gen_block_init, gen_cache_state, gen_gains,
                       gen_hidden_rows, gen_layer_weights, gen_lm_head, gen_mix_logits, geometric_prefix,
                       plant_targets)
from gpu_util import assert_bf16_close, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dfl.build()
    dfl.load()
    torch.cuda.set_device(0)
    yield
    assert dfl.dfl_get_device_error() == 0


def _cached_model(w, R_max, random_gains=False):
    mix = gen_mix_logits(w)
    g_mix, g_blk, g_fin = gen_gains(w, random=random_gains)
    layers = [gen_layer_weights(w, l) for l in range(w.D)]
    W_lm = gen_lm_head(w, as_bits=True)
    shape = dfl.DraftShape(N=w.N, d=w.d, Hq=w.Hq, Hkv=w.Hkv, hd=w.hd, D=w.D, L=w.L, B=w.B, C=w.C, V=w.V,
                           dtype="bf16", eps=w.eps, rope_theta=w.rope_theta)
    W_lm_t = torch.from_numpy(W_lm.view(np.int16)).view(torch.bfloat16)
    model = dfl.CachedDraftModel(shape, R_max, mix, g_mix, g_blk, g_fin, layers, W_lm_t)
    return model, dict(mix=mix, g_mix=g_mix, g_blk=g_blk, g_fin=g_fin, layers=layers, W_lm=W_lm)


def _h_new(w, R, starts, counts, seqs=None):
    """[L][N*R][d] bf16: rows starts[n] .. starts[n]+counts[n]-1 of each sequence, zero-padded to R rows.

    With ``seqs``, only those sequences carry hidden states (the rest zeros).
    """
    H = np.zeros((w.L, w.N * R, w.d), np.uint16)
    for n in range(w.N):
        if counts[n] > 0 and (seqs is None or n in seqs):
            H[:, n * R:n * R + counts[n]] = gen_hidden_rows(w, n, int(starts[n]), int(starts[n] + counts[n]),
                                                            as_bits=True)
    return torch.from_numpy(H.view(np.int16)).cuda().view(torch.bfloat16)


def _i32(x):
    return torch.from_numpy(np.asarray(x, np.int32)).cuda()


def _prefill(model, w, lengths, R, X0, seqs=None):
    """Fill each sequence's caches to lengths[n] by a chain of cached steps (ragged appends, advance on)."""
    cur = np.zeros(w.N, np.int64)
    lengths = np.asarray(lengths, np.int64)
    while (cur < lengths).any():
        m = np.minimum(lengths - cur, R)
        model.step(_h_new(w, R, cur, m, seqs), X0, _i32(m), R=R)
        cur += m
    torch.cuda.synchronize()
    assert np.array_equal(host(model.ctx_len), lengths)


def _oracle_kv(w, p, n, rows):
    """Oracle keys/values of the given positions of sequence n, every layer."""
    Hn = np.concatenate([gen_hidden_rows(w, n, int(r), int(r) + 1) for r in rows], axis=1)
    return [orc.context_kv_rows(Hn, p["mix"][l], p["g_mix"][l], p["layers"][l]["Wkc"], p["layers"][l]["Wvc"],
                                rows, {"Hq": w.Hq, "Hkv": w.Hkv, "hd": w.hd}, w.eps, w.rope_theta)
            for l in range(w.D)]


def _oracle_block(w, p, n, length):
    Hn = gen_hidden_rows(w, n, 0, length)
    Xb0 = gen_block_init(w)[n]
    out = orc.draft_forward(Xb0, Hn, p["mix"], p["g_mix"], p["g_blk"], p["layers"],
                            {"Hq": w.Hq, "Hkv": w.Hkv, "hd": w.hd}, w.eps, w.rope_theta)
    z = orc.lm_head_logits(out["Xb"][1:], p["g_fin"], w.eps, bits_to_f32(p["W_lm"]))
    return out["Xb"], z


def _decode_step(model, w, c0, m, R, X0, seqs=None):
    """The checked decoding step: drafts first (lengths held), then again with planted targets, advancing."""
    H = _h_new(w, R, c0, m, seqs)
    n_new = _i32(m)
    model.want_logits()
    model.step(H, X0, n_new, R=R, advance=False)
    torch.cuda.synchronize()
    drafts = host(model.draft)
    target = torch.from_numpy(plant_targets(w, drafts)).cuda()
    model.step(H, X0, n_new, target=target, R=R, advance=True)
    torch.cuda.synchronize()
    assert np.array_equal(host(model.draft), drafts)   # the same step twice drafts the same tokens
    z = host(model.logits).reshape(w.N, w.B - 1, w.V)
    assert np.array_equal(orc.argmax_lowest(z), drafts)
    t = host(target)
    G = geometric_prefix(w)
    for n in range(w.N):
        a, b = orc.greedy_accept(drafts[n], t[n])
        assert (a, b) == (int(host(model.accept_len)[n]), int(host(model.bonus)[n]))
        assert a == G[n]
    return z


def _check_cache_rows(model, w, p, n, length, rows):
    kv = _oracle_kv(w, p, n, rows)
    K = host(model.K_cache[:, n].float())
    V = host(model.V_cache[:, n].float())
    for l in range(w.D):
        assert_bf16_close(K[l, rows], kv[l][0], f"K[{l}][{n}]")
        assert_bf16_close(V[l, rows], kv[l][1], f"V[{l}][{n}]")
    # rows past the length were never written (the caches start zeroed)
    assert not K[:, length:].any() and not V[:, length:].any()


@pytest.mark.parametrize("hd,Hq,Hkv", [(128, 8, 2), (64, 8, 2)])
def test_small_cached_steps(hd, Hq, Hkv):
    w = Workload("small_cached", N=3, d=512, Hq=Hq, Hkv=Hkv, hd=hd, D=2, L=5, B=16, C=300, V=3000, dtype="bf16",
                 seed=47, geom_p=0.3, R=16)
    model, p = _cached_model(w, R_max=64, random_gains=True)
    X0 = torch.from_numpy(gen_block_init(w)).cuda()
    c0 = np.array([37, 0, 130])
    _prefill(model, w, c0, 64, X0)
    m = np.array([5, 16, 0])
    z = _decode_step(model, w, c0, m, 16, X0)
    length = c0 + m
    assert np.array_equal(host(model.ctx_len), length)
    Xb = host(model.Xb)
    for n in range(w.N):
        _check_cache_rows(model, w, p, n, int(length[n]), np.arange(length[n]))
        ref_xb, ref_z = _oracle_block(w, p, n, int(length[n]))
        X0n = gen_block_init(w)[n]
        assert_bf16_close(Xb[n] - X0n, ref_xb - X0n, f"dXb[{n}]", mean_bar=8e-3)
        assert_bf16_close(z[n], ref_z, f"logits[{n}]", mean_bar=8e-3)


def test_cached_step_rejects_out_of_range_lengths_on_the_device():
    # A sequence whose new rows exceed R is left as it was (nothing appended,
    # length unchanged) and the step records DFL_ERR_INVALID_ARG; the other
    # sequences proceed.
    w = Workload("small_cached_bad", N=3, d=256, Hq=4, Hkv=2, hd=64, D=1, L=3, B=8, C=64, V=500, dtype="bf16",
                 seed=49, R=8)
    model, p = _cached_model(w, R_max=8)
    X0 = torch.from_numpy(gen_block_init(w)).cuda()
    model.reset([10, 20, 30])
    m = np.array([3, 9, 60])   # 9 > R; 30 + 60 > C
    model.step(_h_new(w, 8, [10, 20, 30], np.minimum(m, 8)), X0, _i32(m))
    assert dfl.dfl_get_device_error() == dfl._lib.DFL_ERR_INVALID_ARG
    assert np.array_equal(host(model.ctx_len), [13, 20, 30])
    K = host(model.K_cache.float())
    assert K[:, 0, 10:13].any() and not K[:, 0, 13:].any()
    assert not K[:, 1:].any()
    assert dfl.dfl_get_device_error() == 0   # read and cleared


def test_full_size_cached_decoding_step():
    # Qwen3-8B drafter in steady-state decoding: caches of about 2048 positions
    # per sequence (ragged), up to 16 new rows per step, the benchmark's
    # launch configuration.  Sampled sequences carry hidden states and are
    # checked against the oracle; every sequence's argmax and acceptance is
    # checked on the GPU's own logits.
    w = WORKLOADS["qwen3_8b_drafter_cached"]
    seqs = [0, 17]
    model, p = _cached_model(w, R_max=512)
    X0 = torch.from_numpy(gen_block_init(w)).cuda()
    c0, m = gen_cache_state(w)
    _prefill(model, w, c0, 512, X0, seqs=seqs)
    z = _decode_step(model, w, c0, m, w.R, X0, seqs=seqs)
    length = c0 + m
    assert np.array_equal(host(model.ctx_len), length)
    Xb = host(model.Xb)
    for n in seqs:
        L = int(length[n])
        rows = np.r_[0:3, L // 2:L // 2 + 2, c0[n] - 2:L]   # early rows, middle rows, the rows of the last steps
        _check_cache_rows(model, w, p, n, L, rows)
        ref_xb, ref_z = _oracle_block(w, p, n, L)
        X0n = gen_block_init(w)[n]
        assert_bf16_close(Xb[n] - X0n, ref_xb - X0n, f"dXb[{n}]", mean_bar=8e-3)
        assert_bf16_close(z[n], ref_z, f"logits[{n}]", mean_bar=8e-3)
