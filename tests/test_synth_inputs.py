"""The seeded input generator: formats, determinism and subset regeneration."""
import numpy as np
import torch

from dfl_synth import (WORKLOADS, Workload, bf16_bits, bits_to_f32, gen_hidden,
                       gen_layer_weights, gen_verifier_logits, round_bf16)


def test_round_bf16_matches_torch_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.normal(size=100000).astype(np.float32) * 10.0 ** rng.integers(-20, 20, 100000),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, -0.0], np.float32)])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(round_bf16(x).view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(bits_to_f32(bf16_bits(round_bf16(x))), round_bf16(x))


def test_hidden_subset_regenerates_identically():
    w = Workload("t", N=3, d=16, Hq=2, Hkv=1, hd=8, D=2, L=3, B=4, C=5, V=10,
                 dtype="bf16", seed=5)
    full = gen_hidden(w)
    sub = gen_hidden(w, seqs=[2])
    assert np.array_equal(full[:, 2 * w.C:3 * w.C], sub[:, :w.C])
    assert np.array_equal(bits_to_f32(gen_hidden(w, as_bits=True)), full)
    assert np.array_equal(round_bf16(full), full)


def test_hidden_scale_range_and_workload_shapes():
    w = WORKLOADS["qwen3_8b_layer"]
    assert (w.d, w.Hq, w.Hkv, w.hd, w.L, w.B, w.C) == (4096, 32, 8, 128, 9, 16, 1024)
    c5 = WORKLOADS["specdiff2_select"]
    assert c5.gamma == 32 and c5.K == 8 and c5.T == 1.5
    small = Workload("t", N=2, d=8, Hq=1, Hkv=1, hd=8, D=1, L=4, B=2, C=3, V=0,
                     dtype="f32", seed=9)
    from dfl_synth import gen_hidden_scales
    s = gen_hidden_scales(small)
    assert s.shape == (2, 4) and np.all((s >= 0.5) & (s <= 2.0))


def test_weights_and_verifier_shapes():
    w = Workload("t", N=2, d=16, Hq=4, Hkv=2, hd=8, D=1, L=2, B=5, C=3, V=11,
                 dtype="bf16", seed=3, K=3)
    W = gen_layer_weights(w, 0)
    assert W["Wq"].shape == (32, 16) and W["Wkc"].shape == (16, 16) and W["Wo"].shape == (16, 32)
    v = gen_verifier_logits(w)
    assert v.shape == (2, 3, 5, 11)
    assert np.array_equal(gen_verifier_logits(w, seqs=[1]), v[1:2])
