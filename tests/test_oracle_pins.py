"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a
hand-worked case, a closed form, an invariant, brute-force enumeration, or an
independent scalar-loop restatement on tiny inputs.  CPU only.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle as orc
from dfl_synth import WORKLOADS, Workload, plant_targets

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- mixture --

def test_mix_coefficient_counts_match_pages():
    # DFlare post, "Per-draft-layer mixing": 7 draft layers x 9 target layers
    # = 63 coefficients; the GPT-OSS drafter is 8 layers x 7 target layers.
    assert WORKLOADS["qwen3_8b_drafter"].n_mix_coefficients == 63
    assert WORKLOADS["gpt_oss_20b_drafter"].n_mix_coefficients == 56
    a = orc.mix_weights(np.random.default_rng(0).normal(size=(7, 9)))
    assert a.shape == (7, 9)


@pytest.mark.parametrize("scale", [1.0, 30.0, 300.0])
def test_mix_weights_sum_to_one(scale):
    z = np.random.default_rng(1).normal(size=(7, 9)) * scale
    a = orc.mix_weights(z)
    assert np.all(a >= 0)
    assert np.max(np.abs(a.sum(axis=-1) - 1.0)) < 1e-12


def test_mix_worked_example():
    # logits (0, ln 3) -> ratios (1/4, 3/4); H_0 = (4, 0), H_1 = (0, 4)
    # -> x = (1, 3), mean(x^2) = 5 -> RMSNorm(x) = (1, 3)/sqrt(5)  (eps = 0).
    H = np.array([[[4.0, 0.0]], [[0.0, 4.0]]])
    out = orc.mix_rmsnorm(H, [0.0, math.log(3.0)], [1.0, 1.0], 0.0)
    assert np.allclose(out, [[1 / math.sqrt(5), 3 / math.sqrt(5)]], rtol=0, atol=1e-15)
    # gain multiplies after normalisation
    out = orc.mix_rmsnorm(H, [0.0, math.log(3.0)], [2.0, -1.0], 0.0)
    assert np.allclose(out, [[2 / math.sqrt(5), -3 / math.sqrt(5)]], atol=1e-15)


def test_rmsnorm_worked_example_with_eps():
    # x = (3, 4): mean(x^2) = 12.5; with eps = 0.5 the divisor is sqrt(13).
    out = orc.rmsnorm([3.0, 4.0], [1.0, 1.0], 0.5)
    assert np.allclose(out, [3 / math.sqrt(13), 4 / math.sqrt(13)], atol=1e-15)


def test_mix_one_hot_limit_is_rmsnorm_of_that_layer():
    rng = np.random.default_rng(2)
    H = rng.normal(size=(5, 7, 32))
    g = rng.uniform(0.5, 1.5, size=32)
    for i in range(5):
        z = np.zeros(5)
        z[i] = 50.0
        direct = H[i] / np.sqrt(np.mean(H[i] ** 2, axis=-1, keepdims=True) + 1e-6) * g
        assert np.allclose(orc.mix_rmsnorm(H, z, g, 1e-6), direct, rtol=1e-12, atol=1e-12)


def test_mix_of_equal_layers_ignores_logits():
    rng = np.random.default_rng(3)
    h = rng.normal(size=(4, 16))
    H = np.stack([h] * 3)
    ref = orc.rmsnorm(h, np.ones(16), 1e-6)
    for z in ([0, 0, 0], [5, -3, 1], [-40, 2, 9]):
        assert np.allclose(orc.mix_rmsnorm(H, z, np.ones(16), 1e-6), ref, atol=1e-12)


def test_rmsnorm_scale_invariance():
    rng = np.random.default_rng(4)
    x = rng.normal(size=(3, 64))
    a = orc.rmsnorm(x, np.ones(64), 1e-12)
    b = orc.rmsnorm(1e3 * x, np.ones(64), 1e-12)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)
    assert np.allclose(np.mean(a ** 2, axis=-1), 1.0, atol=1e-9)


def test_mix_is_linear_combination_then_norm_not_norm_then_mix():
    # Negative control for the order: normalising each layer first differs.
    rng = np.random.default_rng(5)
    H = rng.normal(size=(3, 2, 8)) * np.array([0.5, 1.0, 2.0])[:, None, None]
    z = np.array([0.3, -0.2, 0.9])
    a = orc.mix_weights(z)
    other = sum(a[i] * orc.rmsnorm(H[i], np.ones(8), 1e-6) for i in range(3))
    assert not np.allclose(orc.mix_rmsnorm(H, z, np.ones(8), 1e-6), other, atol=1e-3)


# ------------------------------------------------------------------- RoPE --

def test_rope_two_dim_closed_form():
    # hd = 2: one pair rotated by angle = position * theta^0 = position.
    cos, sin = orc.rope_cos_sin([0, 1, 2.5], 2, 1e6)
    x = np.array([[[1.0, 2.0]]] * 3)
    out = orc.apply_rope(x, cos, sin)
    for p_i, p in enumerate([0, 1, 2.5]):
        exp = [math.cos(p) - 2 * math.sin(p), 2 * math.cos(p) + math.sin(p)]
        assert np.allclose(out[p_i, 0], exp, atol=1e-15)


def test_rope_frequency_closed_form():
    hd, theta = 8, 10000.0
    cos, sin = orc.rope_cos_sin([3], hd, theta)
    for i in range(hd // 2):
        ang = 3 * theta ** (-2 * i / hd)
        assert abs(cos[0, i] - math.cos(ang)) < 1e-15
        assert abs(sin[0, i] - math.sin(ang)) < 1e-15


def test_rope_preserves_norm_and_is_relative():
    rng = np.random.default_rng(6)
    hd = 16
    q = rng.normal(size=(1, 1, hd))
    k = rng.normal(size=(1, 1, hd))

    def rot(x, p):
        c, s = orc.rope_cos_sin([p], hd, 1e4)
        return orc.apply_rope(x, c, s)[0, 0]

    assert np.allclose(rot(q, 0), q[0, 0], atol=1e-15)
    assert abs(np.linalg.norm(rot(q, 37)) - np.linalg.norm(q)) < 1e-12
    d1 = rot(q, 10) @ rot(k, 4)
    d2 = rot(q, 106) @ rot(k, 100)
    assert abs(d1 - d2) < 1e-10


# -------------------------------------------------------------- attention --

def _attention_scalar_loops(Q, K, V, visible):
    """Independent restatement: one query row and head at a time, scalars."""
    Bq, Hq, hd = Q.shape
    S, Hkv, _ = K.shape
    group = Hq // Hkv
    O = np.zeros_like(Q, dtype=float)
    for b in range(Bq):
        for h in range(Hq):
            g = h // group
            logits = []
            for s in range(S):
                if visible[b][s]:
                    logits.append((s, sum(Q[b, h, e] * K[s, g, e] for e in range(hd)) / math.sqrt(hd)))
            m = max(l for _, l in logits)
            ws = [(s, math.exp(l - m)) for s, l in logits]
            tot = sum(w for _, w in ws)
            for e in range(hd):
                O[b, h, e] = sum(w * V[s, g, e] for s, w in ws) / tot
    return O


@pytest.mark.parametrize("C,B,Hq,Hkv", [(3, 2, 2, 1), (0, 3, 4, 2), (5, 1, 2, 2)])
def test_attention_matches_scalar_loops(C, B, Hq, Hkv):
    rng = np.random.default_rng(7)
    hd = 4
    Q = rng.normal(size=(B, Hq, hd))
    K = rng.normal(size=(C + B, Hkv, hd))
    V = rng.normal(size=(C + B, Hkv, hd))
    vis = orc.block_visibility(C, B)
    assert vis.shape == (B, C + B) and vis.all()
    assert np.allclose(orc.attention(Q, K, V, vis), _attention_scalar_loops(Q, K, V, vis), atol=1e-12)
    causal = np.array([[s <= C + b for s in range(C + B)] for b in range(B)])
    assert np.allclose(orc.attention(Q, K, V, causal), _attention_scalar_loops(Q, K, V, causal), atol=1e-12)


def test_attention_single_key_returns_value():
    rng = np.random.default_rng(8)
    Q = rng.normal(size=(1, 2, 8))
    K = rng.normal(size=(1, 1, 8))
    V = rng.normal(size=(1, 1, 8))
    O = orc.attention(Q, K, V, orc.block_visibility(0, 1))
    assert np.allclose(O[0, 0], V[0, 0], atol=1e-15) and np.allclose(O[0, 1], V[0, 0], atol=1e-15)


def test_attention_identical_keys_average_values():
    rng = np.random.default_rng(9)
    Q = rng.normal(size=(3, 2, 8))
    K = np.repeat(rng.normal(size=(1, 1, 8)), 6, axis=0)
    V = rng.normal(size=(6, 1, 8))
    O = orc.attention(Q, K, V, orc.block_visibility(3, 3))
    assert np.allclose(O, V[:, 0].mean(axis=0)[None, None, :], atol=1e-12)


def test_attention_gqa_equals_repeated_kv_heads():
    rng = np.random.default_rng(10)
    Q = rng.normal(size=(4, 8, 16))
    K = rng.normal(size=(9, 2, 16))
    V = rng.normal(size=(9, 2, 16))
    vis = orc.block_visibility(5, 4)
    a = orc.attention(Q, K, V, vis)
    b = orc.attention(Q, np.repeat(K, 4, axis=1), np.repeat(V, 4, axis=1), vis)
    assert np.allclose(a, b, atol=1e-13)


def test_block_attention_is_bidirectional_and_order_free():
    # Every key is visible, so permuting keys with their values changes nothing,
    # while a causal mask (negative control) changes the early block rows.
    rng = np.random.default_rng(11)
    C, B = 6, 4
    Q = rng.normal(size=(B, 2, 8))
    K = rng.normal(size=(C + B, 1, 8))
    V = rng.normal(size=(C + B, 1, 8))
    vis = orc.block_visibility(C, B)
    perm = rng.permutation(C + B)
    a = orc.attention(Q, K, V, vis)
    assert np.allclose(a, orc.attention(Q, K[perm], V[perm], vis), atol=1e-13)
    causal = np.array([[s <= C + b for s in range(C + B)] for b in range(B)])
    c = orc.attention(Q, K, V, causal)
    assert not np.allclose(a[0], c[0], atol=1e-6)
    assert np.allclose(a[B - 1], c[B - 1], atol=1e-13)   # last row sees everything either way


# ------------------------------------------------------------ draft layer --

def _tiny_layer_inputs(seed=12, B=3, C=4, L=2, d=8, Hq=2, Hkv=1, hd=4):
    rng = np.random.default_rng(seed)
    W = {"Wq": rng.normal(size=(Hq * hd, d)), "Wkc": rng.normal(size=(Hkv * hd, d)),
         "Wvc": rng.normal(size=(Hkv * hd, d)), "Wkb": rng.normal(size=(Hkv * hd, d)),
         "Wvb": rng.normal(size=(Hkv * hd, d)), "Wo": rng.normal(size=(d, Hq * hd))}
    return dict(Xb=rng.normal(size=(B, d)), Hn=rng.normal(size=(L, C, d)),
                mix=rng.normal(size=L), g_mix=rng.uniform(0.5, 1.5, d),
                g_blk=rng.uniform(0.5, 1.5, d), W=W,
                shape={"Hq": Hq, "Hkv": Hkv, "hd": hd})


def _layer_scalar_loops(Xb, Hn, mix, g_mix, g_blk, W, shape, eps, theta):
    """Independent scalar restatement of one draft layer on tiny inputs."""
    B, d = Xb.shape
    L, C, _ = Hn.shape
    Hq, Hkv, hd = shape["Hq"], shape["Hkv"], shape["hd"]
    ez = [math.exp(z) for z in mix]
    a = [e / sum(ez) for e in ez]

    def norm(row, g):
        r = math.sqrt(sum(v * v for v in row) / len(row) + eps)
        return [row[i] / r * g[i] for i in range(len(row))]

    Xc = [norm([sum(a[i] * Hn[i, c, e] for i in range(L)) for e in range(d)], g_mix) for c in range(C)]
    Xn = [norm(list(Xb[b]), g_blk) for b in range(B)]

    def proj(rows, Wm):
        return [[sum(r[k] * Wm[o, k] for k in range(d)) for o in range(Wm.shape[0])] for r in rows]

    def rope(rows, heads, pos0):
        out = []
        for p, r in enumerate(rows):
            pos = pos0 + p
            nr = list(r)
            for h in range(heads):
                for i in range(hd // 2):
                    ang = pos * theta ** (-2.0 * i / hd)
                    x1, x2 = r[h * hd + i], r[h * hd + i + hd // 2]
                    nr[h * hd + i] = x1 * math.cos(ang) - x2 * math.sin(ang)
                    nr[h * hd + i + hd // 2] = x2 * math.cos(ang) + x1 * math.sin(ang)
            out.append(nr)
        return out

    Q = rope(proj(Xn, W["Wq"]), Hq, C)
    Kb = rope(proj(Xn, W["Wkb"]), Hkv, C)
    Kc = rope(proj(Xc, W["Wkc"]), Hkv, 0)
    Vb, Vc = proj(Xn, W["Wvb"]), proj(Xc, W["Wvc"])
    keys, vals = Kc + Kb, Vc + Vb
    O = [[0.0] * (Hq * hd) for _ in range(B)]
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            s = [sum(Q[b][h * hd + e] * k[g * hd + e] for e in range(hd)) / math.sqrt(hd) for k in keys]
            m = max(s)
            w = [math.exp(x - m) for x in s]
            for e in range(hd):
                O[b][h * hd + e] = sum(w[j] * vals[j][g * hd + e] for j in range(len(keys))) / sum(w)
    out = [[Xb[b, o] + sum(O[b][k] * W["Wo"][o, k] for k in range(Hq * hd)) for o in range(d)]
           for b in range(B)]
    return np.array(Xc), np.array(Q), np.array(out)


@pytest.mark.parametrize("Hq,Hkv", [(2, 1), (2, 2)])
def test_draft_layer_matches_scalar_restatement(Hq, Hkv):
    t = _tiny_layer_inputs(Hq=Hq, Hkv=Hkv)
    got = orc.draft_layer(t["Xb"], t["Hn"], t["mix"], t["g_mix"], t["g_blk"], t["W"], t["shape"], 1e-6, 100.0)
    Xc, Q, Xb = _layer_scalar_loops(t["Xb"], t["Hn"], t["mix"], t["g_mix"], t["g_blk"], t["W"], t["shape"], 1e-6, 100.0)
    assert np.allclose(got["Xc"], Xc, atol=1e-12)
    assert np.allclose(got["Q"].reshape(Q.shape), Q, atol=1e-12)
    assert np.allclose(got["Xb"], Xb, atol=1e-12)


def test_queries_come_from_draft_features_only():
    # DFlare post, "Separate KV projections by information source": queries
    # are built from the draft features, so the target hidden states reach Q
    # never and reach the output only through the context K/V.
    t = _tiny_layer_inputs()
    a = orc.draft_layer(t["Xb"], t["Hn"], t["mix"], t["g_mix"], t["g_blk"], t["W"], t["shape"], 1e-6, 100.0)
    b = orc.draft_layer(t["Xb"], 3.0 * t["Hn"][::-1], t["mix"], t["g_mix"], t["g_blk"], t["W"], t["shape"], 1e-6, 100.0)
    for k in ("Q", "Kb", "Vb"):
        assert np.allclose(a[k], b[k], atol=1e-14)
    assert not np.allclose(a["Kc"], b["Kc"]) and not np.allclose(a["Xb"], b["Xb"])


def test_context_and_block_kv_weights_are_separate():
    t = _tiny_layer_inputs()
    a = orc.draft_layer(t["Xb"], t["Hn"], t["mix"], t["g_mix"], t["g_blk"], t["W"], t["shape"], 1e-6, 100.0)
    W2 = dict(t["W"])
    W2["Wkc"], W2["Wkb"] = t["W"]["Wkb"], t["W"]["Wkc"]
    b = orc.draft_layer(t["Xb"], t["Hn"], t["mix"], t["g_mix"], t["g_blk"], W2, t["shape"], 1e-6, 100.0)
    assert not np.allclose(a["Xb"], b["Xb"], atol=1e-6)


def test_draft_forward_chains_layers():
    t = _tiny_layer_inputs()
    layers = [t["W"], {k: 0.5 * v for k, v in t["W"].items()}]
    mix = np.stack([t["mix"], -t["mix"]])
    g2 = np.stack([t["g_mix"]] * 2)
    gb = np.stack([t["g_blk"]] * 2)
    out = orc.draft_forward(t["Xb"], t["Hn"], mix, g2, gb, layers, t["shape"], 1e-6, 100.0)
    x1 = orc.draft_layer(t["Xb"], t["Hn"], mix[0], g2[0], gb[0], layers[0], t["shape"], 1e-6, 100.0)["Xb"]
    x2 = orc.draft_layer(x1, t["Hn"], mix[1], g2[1], gb[1], layers[1], t["shape"], 1e-6, 100.0)["Xb"]
    assert np.allclose(out["Xb"], x2, atol=1e-13)


# ---------------------------------------------------------------- LM head --

def test_lm_head_logits_scalar_and_chunking():
    rng = np.random.default_rng(13)
    X = rng.normal(size=(3, 6))
    W = rng.normal(size=(11, 6))
    g = rng.uniform(0.5, 1.5, 6)
    z = orc.lm_head_logits(X, g, 1e-6, W, chunk=4)
    for r in range(3):
        rms = math.sqrt(sum(v * v for v in X[r]) / 6 + 1e-6)
        for v in range(11):
            exp = sum(X[r, k] / rms * g[k] * W[v, k] for k in range(6))
            assert abs(z[r, v] - exp) < 1e-12
    assert np.array_equal(z, orc.lm_head_logits(X, g, 1e-6, W, chunk=1000))


def test_argmax_ties_take_lowest_index():
    z = np.array([[1.0, 3.0, 3.0, 2.0], [5.0, 5.0, 5.0, 5.0], [-1.0, -2.0, -1.0, -3.0]])
    assert orc.argmax_lowest(z).tolist() == [1, 0, 0]


# ----------------------------------------------------------------- greedy --

def _golden_greedy():
    rows = []
    with open(os.path.join(GOLDEN, "greedy_cases.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                d, t, a, b = [p.split() for p in line.split("|")]
                rows.append(([int(x) for x in d], [int(x) for x in t], int(a[0]), int(b[0])))
    return rows


@pytest.mark.parametrize("case", _golden_greedy())
def test_greedy_accept_golden(case):
    d, t, a, b = case
    assert orc.greedy_accept(d, t) == (a, b)


def test_greedy_planted_prefix_closed_form():
    # Targets planted to agree for exactly G_n leading positions give
    # accepted = G_n and bonus = t_{G_n+1}; the mean of G_n approaches
    # sum_{k=1}^{B-1} (1-p)^k (Geometric failures before the first success,
    # truncated at B-1).
    w = Workload("plant", N=20000, d=1, Hq=1, Hkv=1, hd=2, D=1, L=1, B=16,
                 C=1, V=1000, dtype="f32", seed=77, geom_p=0.15)
    rng = np.random.default_rng(14)
    drafts = rng.integers(0, w.V, size=(w.N, w.B - 1))
    t = plant_targets(w, drafts)
    from dfl_synth import geometric_prefix
    G = geometric_prefix(w)
    acc = [orc.greedy_accept(drafts[n], t[n]) for n in range(w.N)]
    assert all(a == G[n] and bonus == t[n, a] for n, (a, bonus) in enumerate(acc))
    expected = sum((1 - w.geom_p) ** k for k in range(1, w.B))
    assert abs(np.mean(G) - expected) < 0.08   # ~5 sigma at N = 20000
    assert abs(expected - 5.17) < 0.01          # B = 16, p = 0.15


# ----------------------------------------------------------------- Philox --

def _golden_philox():
    rows = []
    with open(os.path.join(GOLDEN, "philox_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                c, k, x = [[int(v, 16) for v in p.split()] for p in line.split("|")]
                rows.append((c, k, x))
    return rows


@pytest.mark.parametrize("case", _golden_philox())
def test_philox_known_answers(case):
    c, k, x = case
    assert list(orc.philox4x32_10(c, k)) == x


def test_philox_uniform_statistics():
    u = np.array([orc.draw_uniform(0x5EEDD1F5, n, j, k) for n in range(8) for j in range(64) for k in range(8)])
    assert np.all((u > 0) & (u < 1))
    counts, _ = np.histogram(u, bins=16, range=(0, 1))
    chi2 = np.sum((counts - len(u) / 16) ** 2 / (len(u) / 16))
    assert chi2 < 45.0   # 15 dof; p ~ 1e-4


def test_philox_avalanche():
    base = orc.philox4x32_10((1, 2, 3, 4), (5, 6))
    flips = []
    for bit in range(32):
        x = orc.philox4x32_10((1 ^ (1 << bit), 2, 3, 4), (5, 6))
        flips.append(sum(bin(a ^ b).count("1") for a, b in zip(base, x)))
    assert 48 < np.mean(flips) < 80   # ~64 of 128 output bits flip


# --------------------------------------------------------------- sampling --

def test_sampling_one_hot_is_deterministic():
    z = np.zeros(50)
    z[17] = 200.0
    for u in (1e-7, 0.3, 0.999999):
        assert orc.sample_inverse_cdf(z, 1.5, u)[0] == 17


def test_sampling_uniform_grid_reproduces_marginal():
    # Inversion of the CDF on the grid u_i = (i + 1/2)/M gives every token a
    # count within 1 of M * q_v, q = softmax(z / T).
    rng = np.random.default_rng(15)
    z, T, M = rng.normal(size=8) * 2, 1.5, 4000
    q = np.exp(z / T) / np.exp(z / T).sum()
    counts = np.zeros(8)
    for i in range(M):
        counts[orc.sample_inverse_cdf(z, T, (i + 0.5) / M)[0]] += 1
    assert np.all(np.abs(counts - M * q) <= 1.0 + 1e-9)


def test_sampling_low_temperature_is_argmax_and_margin():
    rng = np.random.default_rng(16)
    z = rng.normal(size=100)
    assert orc.sample_inverse_cdf(z, 1e-4, 0.5)[0] == int(np.argmax(z))
    v, margin = orc.sample_inverse_cdf(np.zeros(4), 1.0, 0.5)   # boundary exactly at 0.5
    assert margin == 0.0 and v == 2


# ------------------------------------------------------------ streak / TV --

def test_streak_worked_example():
    assert orc.streak_score([0.5, 0.5]) == 0.75
    assert orc.streak_score([1.0, 1.0, 1.0]) == 3.0
    assert orc.streak_score([0.0, 1.0]) == 0.0


@pytest.mark.parametrize("V,G", [(2, 1), (3, 3), (4, 4), (2, 4)])
def test_streak_equation_by_enumeration(V, G):
    # SpecDiff-2 notes, "Streak-Distillation": Tokens/Draft = E[sum_m prod_{j<=m} alpha_j].
    # Enumerate every verifier outcome y in V^G, y_j ~ P_j independently; a
    # draft token is accepted while y_j equals it; the expected number accepted
    # must equal the streak score of p_j = P_j(x_j).
    rng = np.random.default_rng(V * 10 + G)
    P = rng.dirichlet(np.ones(V), size=G)
    x = rng.integers(0, V, size=G)
    expect = 0.0
    for y in itertools.product(range(V), repeat=G):
        prob = np.prod([P[j, y[j]] for j in range(G)])
        acc = 0
        while acc < G and y[acc] == x[acc]:
            acc += 1
        expect += prob * acc
    assert abs(orc.streak_score([P[j, x[j]] for j in range(G)]) - expect) < 1e-12


def test_tv_acceptance_closed_form_and_theorem():
    rng = np.random.default_rng(17)
    for _ in range(20):
        P, Q = rng.dirichlet(np.ones(6)), rng.dirichlet(np.ones(6))
        a = orc.tv_acceptance(P, Q)
        assert abs(a - np.minimum(P, Q).sum()) < 1e-12      # 1 - TV = sum min
        assert a >= np.sum(P * Q) - 1e-15                    # alpha_SD >= alpha_greedy
    P = rng.dirichlet(np.ones(5))
    assert abs(orc.tv_acceptance(P, P) - 1.0) < 1e-15


def test_tv_acceptance_monte_carlo():
    # Speculative sampling accepts x ~ Q with probability min(1, P(x)/Q(x));
    # its acceptance rate is the TV proxy.
    rng = np.random.default_rng(18)
    P, Q = rng.dirichlet(np.ones(4)), rng.dirichlet(np.ones(4))
    n = 200000
    x = rng.choice(4, size=n, p=Q)
    acc = rng.random(n) < np.minimum(1.0, P[x] / Q[x])
    assert abs(acc.mean() - orc.tv_acceptance(P, Q)) < 5 * math.sqrt(0.25 / n)


# ---------------------------------------------------------- self-selection --

def test_self_select_scores_by_enumeration_and_greedy():
    rng = np.random.default_rng(19)
    K, G, V = 3, 3, 3
    vlog = rng.normal(size=(K, G + 1, V)) * 2
    drafts = rng.integers(0, V, size=(K, G))
    scores, ks, a, bonus = orc.self_select(vlog, drafts)
    for k in range(K):
        P = np.exp(vlog[k]) / np.exp(vlog[k]).sum(axis=-1, keepdims=True)
        expect = 0.0
        for y in itertools.product(range(V), repeat=G):
            prob = np.prod([P[j, y[j]] for j in range(G)])
            acc = 0
            while acc < G and y[acc] == drafts[k, acc]:
                acc += 1
            expect += prob * acc
        assert abs(scores[k] - expect) < 1e-12
    assert ks == int(np.argmax(scores))
    t = [int(np.argmax(vlog[ks, j])) for j in range(G + 1)]
    assert (a, bonus) == orc.greedy_accept(drafts[ks], t)


def test_self_select_ties_take_lowest_draft():
    vlog = np.zeros((3, 3, 4))
    drafts = np.array([[1, 2], [1, 2], [0, 0]])
    scores, ks, _, _ = orc.self_select(vlog, drafts)
    assert scores[0] == scores[1] == scores[2] and ks == 0


# ------------------------------------------------ stochastic acceptance --

def test_tv_alpha_matches_closed_form_and_limits():
    rng = np.random.default_rng(30)
    z, v = rng.normal(size=12), rng.normal(size=12) * 2
    P = np.exp(v) / np.exp(v).sum()
    Q = np.exp(z / 1.5) / np.exp(z / 1.5).sum()
    assert abs(orc.tv_alpha(z, 1.5, v) - np.minimum(P, Q).sum()) < 1e-14
    assert abs(orc.tv_alpha(v, 1.0, v) - 1.0) < 1e-14          # identical distributions
    zz = np.full(4, -1e3); zz[0] = 1e3
    vv = np.full(4, -1e3); vv[1] = 1e3
    assert abs(orc.tv_alpha(zz, 1.0, vv)) < 1e-12                # disjoint supports


def test_inverse_cdf_grid_and_margin():
    w = np.array([1.0, 0.0, 3.0])
    assert orc.inverse_cdf(w, 0.1)[0] == 0 and orc.inverse_cdf(w, 0.3)[0] == 2
    assert orc.inverse_cdf(w, 0.25)[1] == 0.0                    # exactly on a boundary
    v, margin = orc.inverse_cdf(w, 0.6)          # u*total = 2.4 in (1, 4]: 1.4 and 1.6 away, / 4
    assert v == 2 and abs(margin - 0.35) < 1e-15


def test_sampling_margin_worked_example():
    # weights (1, 1, 2), total 4, cumulative (1, 2, 4)
    for T in (1.0, 2.0):
        z = T * np.log([1.0, 1.0, 2.0])
        v, margin = orc.sample_inverse_cdf(z, T, 0.3)    # 1.2: 0.2 above 1, 0.8 below 2
        assert v == 1 and abs(margin - 0.05) < 1e-12
        v, margin = orc.sample_inverse_cdf(z, T, 0.45)   # 1.8: 0.8 above 1, 0.2 below 2
        assert v == 1 and abs(margin - 0.05) < 1e-12
        v, margin = orc.sample_inverse_cdf(z, T, 0.9)    # 3.6: 1.6 above 2, 0.4 below 4
        assert v == 2 and abs(margin - 0.1) < 1e-12


def test_speculative_accept_margin_worked_example():
    # Q = (1/2, 1/2), P_1 = (0.2, 0.8), P_2 = (0.25, 0.75); draft token 0 (q = 1/2, p = 0.2)
    z, v1, v2 = np.zeros(2), np.log([0.2, 0.8]), np.log([0.25, 0.75])
    run = lambda ua, ur: orc.speculative_accept([z], 1.0, [v1, v2], [0], [ua], ur)
    # rejected (0.3 >= 0.2, test 0.5 away); residual (0, 0.3) at 0.06: 0.2 of it away
    a, y, m = run(0.6, [0.2, 0.5])
    assert (a, y) == (0, 1) and abs(m - 0.2) < 1e-12
    # rejected closer to the boundary (0.225 vs 0.2: 0.125 of p)
    a, y, m = run(0.45, [0.2, 0.5])
    assert (a, y) == (0, 1) and abs(m - 0.125) < 1e-12
    # accepted (0.15 < 0.2, 0.25 away); bonus from P_2 at 0.4: 0.15 away
    a, y, m = run(0.3, [0.5, 0.4])
    assert (a, y) == (1, 1) and abs(m - 0.15) < 1e-12
    # accepted close to the boundary (0.19 vs 0.2): the accepted test sets the margin
    a, y, m = run(0.38, [0.5, 0.4])
    assert (a, y) == (1, 1) and abs(m - 0.05) < 1e-12


def _spec_output_distribution(z, T, v, n_grid=400):
    """Distribution of the first committed token, by exact enumeration over the
    draft token and midpoint grids of both uniforms (G = 1)."""
    V = len(z)
    Q = orc.softmax_t(z, T)
    out = np.zeros(V)
    grid = (np.arange(n_grid) + 0.5) / n_grid
    for x in range(V):
        for ua in grid:
            # token committed at position 1: x if accepted, else the residual draw
            acc, y, _ = orc.speculative_accept([z], T, [v, v], [x], [ua], [0.0, 0.0])
            if acc == 1:
                out[x] += Q[x] / n_grid
            else:
                for ur in grid:
                    _, y, _ = orc.speculative_accept([z], T, [v, v], [x], [ua], [ur, 0.0])
                    out[y] += Q[x] / n_grid / n_grid
    return out


def test_speculative_accept_keeps_the_verifier_distribution():
    # Lossless property: the first committed token is distributed as P_1,
    # whatever the drafter's Q (up to the discretisation of the uniforms).
    rng = np.random.default_rng(31)
    z, v = rng.normal(size=4) * 1.5, rng.normal(size=4)
    out = _spec_output_distribution(z, 1.3, v)
    assert np.allclose(out, orc.softmax_t(v), atol=6e-3)


def test_speculative_accept_rate_is_the_tv_proxy():
    # P(accept position 1) = sum_x Q(x) min(1, P(x)/Q(x)) = sum_x min(P, Q) = alpha.
    rng = np.random.default_rng(32)
    z, v = rng.normal(size=5), rng.normal(size=5)
    Q = orc.softmax_t(z, 1.0)
    grid = (np.arange(2000) + 0.5) / 2000
    rate = sum(Q[x] * np.mean([orc.speculative_accept([z], 1.0, [v, v], [x], [u], [0.5, 0.5])[0] == 1
                               for u in grid]) for x in range(5))
    assert abs(rate - orc.tv_alpha(z, 1.0, v)) < 2e-3


def test_speculative_accept_prefix_and_bonus():
    # Draft that the verifier is certain of: every position accepted, bonus
    # drawn from the last row; a draft the verifier gives no mass: rejected at 1
    # and the residual draw lands on the verifier's token.
    V = 6
    z = np.zeros(V)
    v_sure = np.full(V, -1e4); v_sure[2] = 0.0
    v_last = np.full(V, -1e4); v_last[5] = 0.0
    acc, y, _ = orc.speculative_accept([z, z], 1.0, [v_sure, v_sure, v_last], [2, 2], [0.99, 0.99], [0.3, 0.3, 0.3])
    assert (acc, y) == (2, 5)
    acc, y, _ = orc.speculative_accept([z, z], 1.0, [v_sure, v_sure, v_last], [4, 2], [0.01, 0.5], [0.7, 0.3, 0.3])
    assert (acc, y) == (0, 2)


def test_uniform_streams_are_distinct():
    a = orc.draw_uniform_stream(7, 1, 2, 0, 0)
    assert a == orc.draw_uniform(7, 1, 2, 0)
    assert len({orc.draw_uniform_stream(7, 1, 2, 0, s) for s in range(3)}) == 3


@pytest.mark.parametrize("case", _golden_philox())
def test_uniform_counter_words_follow_the_known_answers(case):
    # (sequence, window row, draft, stream) are counter words 0..3 and the seed's
    # low/high halves key words 0/1: the published vectors fix the mapping.
    c, k, x = case
    seed = k[0] | (k[1] << 32)
    want = ((x[0] >> 8) + 0.5) * 2.0 ** -24
    assert orc.draw_uniform_stream(seed, c[0], c[1], c[2], c[3]) == want
    if c[3] == 0:
        assert orc.draw_uniform(seed, c[0], c[1], c[2]) == want



# ----------------------------------------------------------- SwiGLU FFN --

def test_silu_closed_form():
    for x in (-3.0, -0.5, 0.0, 0.7, 4.0):
        assert abs(orc.silu(x) - x / (1 + math.exp(-x))) < 1e-15
    assert orc.silu(0.0) == 0.0


def test_swiglu_ffn_scalar_restatement_and_identity():
    rng = np.random.default_rng(40)
    B, d, F = 3, 6, 5
    Xb, g = rng.normal(size=(B, d)), rng.uniform(0.5, 1.5, d)
    W1, W3, W2 = rng.normal(size=(F, d)), rng.normal(size=(F, d)), rng.normal(size=(d, F))
    got = orc.swiglu_ffn(Xb, g, W1, W3, W2, 1e-6)
    for b in range(B):
        r = math.sqrt(sum(v * v for v in Xb[b]) / d + 1e-6)
        xn = [Xb[b, k] / r * g[k] for k in range(d)]
        h = []
        for f in range(F):
            a = sum(xn[k] * W1[f, k] for k in range(d))
            u = sum(xn[k] * W3[f, k] for k in range(d))
            h.append(a / (1 + math.exp(-a)) * u)
        for o in range(d):
            assert abs(got[b, o] - (Xb[b, o] + sum(h[f] * W2[o, f] for f in range(F)))) < 1e-12
    assert np.allclose(orc.swiglu_ffn(Xb, g, W1, W3, np.zeros((d, F)), 1e-6), Xb, atol=0)


def test_draft_layer_with_ffn_adds_the_ffn_after_attention():
    t = _tiny_layer_inputs()
    rng = np.random.default_rng(41)
    d, F = t["Xb"].shape[1], 7
    W = dict(t["W"], W1=rng.normal(size=(F, d)), W3=rng.normal(size=(F, d)), W2=rng.normal(size=(d, F)),
             g_ffn=rng.uniform(0.5, 1.5, d))
    a = orc.draft_layer(t["Xb"], t["Hn"], t["mix"], t["g_mix"], t["g_blk"], W, t["shape"], 1e-6, 100.0)
    b = orc.draft_layer(t["Xb"], t["Hn"], t["mix"], t["g_mix"], t["g_blk"], t["W"], t["shape"], 1e-6, 100.0)
    assert np.allclose(a["Xb_attn"], b["Xb"], atol=1e-13)
    assert np.allclose(a["Xb"], orc.swiglu_ffn(b["Xb"], W["g_ffn"], W["W1"], W["W3"], W["W2"], 1e-6), atol=1e-12)


# ------------------------------------------------ incremental context K/V --

def _two_layer_drafter(seed=51, B=3, C=11, L=2, d=8, Hq=4, Hkv=2, hd=4, F=0):
    rng = np.random.default_rng(seed)
    layers = []
    for _ in range(2):
        W = {"Wq": rng.normal(size=(Hq * hd, d)), "Wkc": rng.normal(size=(Hkv * hd, d)),
             "Wvc": rng.normal(size=(Hkv * hd, d)), "Wkb": rng.normal(size=(Hkv * hd, d)),
             "Wvb": rng.normal(size=(Hkv * hd, d)), "Wo": 0.3 * rng.normal(size=(d, Hq * hd))}
        if F:
            W.update(W1=rng.normal(size=(F, d)), W3=rng.normal(size=(F, d)), W2=0.3 * rng.normal(size=(d, F)),
                     g_ffn=rng.uniform(0.5, 1.5, d))
        layers.append(W)
    return dict(Xb=rng.normal(size=(B, d)), Hn=rng.normal(size=(L, C, d)), mix=rng.normal(size=(2, L)),
                g_mix=rng.uniform(0.5, 1.5, (2, d)), g_blk=rng.uniform(0.5, 1.5, (2, d)), layers=layers,
                shape={"Hq": Hq, "Hkv": Hkv, "hd": hd})


@pytest.mark.parametrize("F,chunks", [(0, (4, 0, 5, 2)), (5, (11,)), (0, (1,) * 11)])
def test_cached_steps_equal_the_one_shot_step(F, chunks):
    # Context K/V are a row-wise function of (hidden states, position), so a
    # context that arrives in pieces over several steps gives the caches and
    # the block output of one step over the whole context.
    t = _two_layer_drafter(F=F)
    D = 2
    Hkv, hd = t["shape"]["Hkv"], t["shape"]["hd"]
    cache = [(np.zeros((0, Hkv, hd)), np.zeros((0, Hkv, hd))) for _ in range(D)]
    c0 = 0
    for m in chunks:
        Xb, cache = orc.draft_step_cached(t["Xb"], t["Hn"][:, c0:c0 + m], cache, t["mix"], t["g_mix"], t["g_blk"],
                                          t["layers"], t["shape"], 1e-6, 100.0)
        c0 += m
        assert all(k.shape[0] == c0 and v.shape[0] == c0 for k, v in cache)
        # every intermediate step equals the one-shot step over the prefix seen so far
        ref = orc.draft_forward(t["Xb"], t["Hn"][:, :c0], t["mix"], t["g_mix"], t["g_blk"], t["layers"],
                                t["shape"], 1e-6, 100.0, keep_layers=True)
        assert np.allclose(Xb, ref["Xb"], atol=1e-12, rtol=0)
    for l in range(D):
        full = orc.draft_layer(t["Xb"], t["Hn"], t["mix"][l], t["g_mix"][l], t["g_blk"][l], t["layers"][l],
                               t["shape"], 1e-6, 100.0)
        assert np.allclose(cache[l][0], full["Kc"], atol=1e-12) and np.allclose(cache[l][1], full["Vc"], atol=1e-12)


def test_cached_step_block_positions_follow_the_context_length():
    # A step that appends nothing reproduces the output from the caches
    # alone, and a cached key carries the rotation of the position it was
    # appended at.
    t = _two_layer_drafter()
    C = t["Hn"].shape[1]
    empty = [(np.zeros((0, 2, 4)), np.zeros((0, 2, 4))) for _ in range(2)]
    Xa, cache = orc.draft_step_cached(t["Xb"], t["Hn"], empty, t["mix"], t["g_mix"], t["g_blk"], t["layers"],
                                      t["shape"], 1e-6, 100.0)
    # a step that appends nothing reproduces the same output from the caches alone
    Xb, cache2 = orc.draft_step_cached(t["Xb"], t["Hn"][:, :0], cache, t["mix"], t["g_mix"], t["g_blk"],
                                       t["layers"], t["shape"], 1e-6, 100.0)
    assert np.allclose(Xa, Xb, atol=1e-13)
    assert all(np.array_equal(a[0], b[0]) for a, b in zip(cache, cache2))
    # keys of one position, cached at another position, are a different rotation
    k_at_0, _ = orc.context_kv_rows(t["Hn"][:, :1], t["mix"][0], t["g_mix"][0], t["layers"][0]["Wkc"],
                                    t["layers"][0]["Wvc"], [0], t["shape"], 1e-6, 100.0)
    k_at_5, _ = orc.context_kv_rows(t["Hn"][:, :1], t["mix"][0], t["g_mix"][0], t["layers"][0]["Wkc"],
                                    t["layers"][0]["Wvc"], [5], t["shape"], 1e-6, 100.0)
    assert np.allclose(k_at_0, cache[0][0][:1], atol=1e-13)
    assert not np.allclose(k_at_0, k_at_5)
    # rotation keeps each rotated pair's norm
    assert np.allclose(np.linalg.norm(k_at_0), np.linalg.norm(k_at_5), atol=1e-12)


# --------------------------------------------- DFlash single-FC fusion --

def _fuse_inputs(seed=81, L=3, rows=5, d=6):
    rng = np.random.default_rng(seed)
    H = rng.normal(size=(L, rows, d)) * rng.uniform(0.5, 2.0, size=(L, 1, 1))
    g = rng.uniform(0.5, 1.5, size=d)
    return rng, H, g


def test_fc_fuse_with_scaled_identity_blocks_is_the_softmax_mix():
    # W_fc = [a_1 I | ... | a_L I] is the FC form of a mixture with ratios a:
    # it must give the (separately pinned) mix + RMSNorm of the same ratios.
    rng, H, g = _fuse_inputs()
    L, _, d = H.shape
    logits = rng.normal(size=L)
    a = orc.mix_weights(logits)
    W = np.concatenate([a[i] * np.eye(d) for i in range(L)], axis=1)
    assert np.allclose(orc.fc_fuse(H, W, g, 1e-6), orc.mix_rmsnorm(H, logits, g, 1e-6), atol=1e-13)


@pytest.mark.parametrize("i", [0, 2])
def test_fc_fuse_selecting_one_layer_is_its_rmsnorm(i):
    _, H, g = _fuse_inputs()
    L, _, d = H.shape
    W = np.zeros((d, L * d))
    W[:, i * d:(i + 1) * d] = np.eye(d)
    x = H[i]
    ref = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + 1e-6) * g
    assert np.allclose(orc.fc_fuse(H, W, g, 1e-6), ref, atol=1e-13)


def test_fc_fuse_output_features_and_layer_order():
    # Output feature o reads row o of W_fc; swapping two target layers
    # together with their column blocks of W_fc changes nothing, swapping
    # only the layers does; the norm makes a common scale of H irrelevant.
    rng, H, g = _fuse_inputs(seed=82)
    L, _, d = H.shape
    W = rng.normal(size=(d, L * d)) / np.sqrt(L * d)
    base = orc.fc_fuse(H, W, np.ones(d), 1e-12)
    perm = [2, 0, 1]
    Wp = np.concatenate([W[:, p * d:(p + 1) * d] for p in perm], axis=1)
    assert np.allclose(orc.fc_fuse(H[perm], Wp, np.ones(d), 1e-12), base, atol=1e-12)
    assert not np.allclose(orc.fc_fuse(H[perm], W, np.ones(d), 1e-12), base, atol=1e-3)
    assert np.allclose(orc.fc_fuse(7.0 * H, W, np.ones(d), 1e-12), base, atol=1e-12)
    # one output feature from a hand-computed dot product of the concatenation
    cat = np.concatenate([H[i] for i in range(L)], axis=1)
    pre = cat @ W.T
    r0 = pre[0] / np.sqrt(np.mean(pre[0] ** 2) + 1e-6)
    assert np.allclose(orc.fc_fuse(H, W, np.ones(d), 1e-6)[0], r0, atol=1e-13)


def test_fused_forward_shares_one_representation_across_layers():
    # With the scaled-identity FC, a one-layer fused forward equals the mixed
    # forward of the same ratios; with two layers every layer reads the same
    # context features (the mix logits, unused, may be anything).
    t = _two_layer_drafter()
    L, _, d = t["Hn"].shape
    a = orc.mix_weights(t["mix"][0])
    W = np.concatenate([a[i] * np.eye(d) for i in range(L)], axis=1)
    one = orc.draft_forward(t["Xb"], t["Hn"], t["mix"][:1], t["g_mix"][:1], t["g_blk"][:1], t["layers"][:1],
                            t["shape"], 1e-6, 100.0)
    fused1 = orc.draft_forward(t["Xb"], t["Hn"], None, None, t["g_blk"][:1], t["layers"][:1], t["shape"], 1e-6,
                               100.0, fused=(W, t["g_mix"][0]))
    assert np.allclose(one["Xb"], fused1["Xb"], atol=1e-12)
    fused2 = orc.draft_forward(t["Xb"], t["Hn"], None, None, t["g_blk"], t["layers"], t["shape"], 1e-6, 100.0,
                               keep_layers=True, fused=(W, t["g_mix"][0]))
    mixed = orc.draft_forward(t["Xb"], t["Hn"], [t["mix"][0]] * 2, [t["g_mix"][0]] * 2, t["g_blk"], t["layers"],
                              t["shape"], 1e-6, 100.0)
    assert np.allclose(fused2["layers"][0]["Xc"], fused2["layers"][1]["Xc"])
    assert np.allclose(fused2["Xb"], mixed["Xb"], atol=1e-12)


# ------------------------------- legitimate outcomes near a boundary --

def test_inverse_cdf_outcomes_worked_cases():
    w = np.array([1.0, 0.0, 3.0])                 # cumulative (1, 1, 4)
    assert orc.inverse_cdf_outcomes(w, 0.1, 1e-6) == {0}
    # exactly on the boundary 1: the empty interval of index 1 is skipped
    assert orc.inverse_cdf_outcomes(w, 0.25, 1e-6) == {0, 2}
    # 2.4 is 1.4 above 1 and 1.6 below 4 (0.35 and 0.4 of the total)
    assert orc.inverse_cdf_outcomes(w, 0.6, 0.3) == {2}
    assert orc.inverse_cdf_outcomes(w, 0.6, 0.36) == {0, 2}
    w = np.array([1.0, 1.0, 2.0])                 # cumulative (1, 2, 4)
    assert orc.inverse_cdf_outcomes(w, 0.4975, 0.01) == {1, 2}    # 1.99: 0.01 below 2
    assert orc.inverse_cdf_outcomes(w, 0.4975, 0.002) == {1}
    assert orc.inverse_cdf_outcomes(w, 0.2525, 0.01) == {0, 1}    # 1.01: 0.01 above 1
    # the top boundary has no interval above it
    assert orc.inverse_cdf_outcomes(w, 0.999999, 0.01) == {2}


def test_inverse_cdf_outcomes_hold_every_perturbed_draw():
    # Cumulative sums off by less than the band (relative to the total) can
    # only give draws inside the set, and the set's extra members are reached
    # by some such perturbation.
    rng = np.random.default_rng(83)
    band = 1e-3
    hits = 0
    for _ in range(400):
        V = int(rng.integers(2, 9))
        w = rng.uniform(0, 1, V) * (rng.uniform(0, 1, V) > 0.2)
        if w.sum() == 0:
            continue
        # targets often near a boundary
        cdf = np.cumsum(w) / w.sum()
        b = cdf[int(rng.integers(0, V))]
        u = float(np.clip(b + rng.uniform(-2 * band, 2 * band), 1e-9, 1 - 1e-9))
        legit = orc.inverse_cdf_outcomes(w, u, band)
        seen = set()
        for _ in range(60):
            noise = rng.uniform(-0.45 * band, 0.45 * band, V) * w.sum() / V
            wp = np.maximum(w + noise * (w > 0), 0.0)
            seen.add(orc.inverse_cdf(wp, u)[0])
        assert seen <= legit, (w, u, seen, legit)
        hits += len(legit) > 1
    assert hits > 50


def test_sample_outcomes_use_the_temperature():
    T = 2.0
    z = T * np.log([1.0, 1.0, 2.0])
    assert orc.sample_inverse_cdf_outcomes(z, T, 0.4975, 0.01) == {1, 2}
    assert orc.sample_inverse_cdf_outcomes(z, 1.0, 0.4975, 0.01) == {2}   # weights (1, 1, 4): 2.985 of 6


def test_speculative_outcomes_follow_both_branches_of_a_tied_test():
    # Q = (1/2, 1/2), P_1 = (0.2, 0.8), P_2 = (0.25, 0.75); draft token 0
    z, v1, v2 = np.zeros(2), np.log([0.2, 0.8]), np.log([0.25, 0.75])
    out = lambda ua, ur: orc.speculative_accept_outcomes([z], 1.0, [v1, v2], [0], [ua], ur, 1e-6, 1e-6)
    assert out(0.6, [0.2, 0.5]) == {(0, 1)}                  # clear rejection
    assert out(0.3, [0.5, 0.4]) == {(1, 1)}                  # clear acceptance, bonus 1
    assert out(0.3, [0.5, 0.1]) == {(1, 0)}                  # bonus 0 (0.1 < 0.25)
    # u q = 0.2 = p exactly: accepted or rejected are both legitimate
    assert out(0.4, [0.2, 0.1]) == {(0, 1), (1, 0)}
    # a bonus draw on its boundary (0.25) may give either token
    assert out(0.3, [0.5, 0.25]) == {(1, 0), (1, 1)}


def test_speculative_outcomes_hold_the_exact_result_and_perturbations():
    rng = np.random.default_rng(84)
    for _ in range(200):
        G, V, T = int(rng.integers(1, 4)), int(rng.integers(2, 6)), 1.3
        z = rng.normal(size=(G, V))
        v = np.vstack([z / T, rng.normal(size=(1, V))]) + rng.normal(size=(G + 1, V)) * 0.3
        x = rng.integers(0, V, G)
        ua, ur = rng.uniform(size=G), rng.uniform(size=G + 1)
        legit = orc.speculative_accept_outcomes(z, T, v, x, ua, ur, 1e-4, 1e-4)
        a, y, m = orc.speculative_accept(z, T, v, x, ua, ur)
        assert (a, y) in legit
        if m >= 1e-4:
            assert legit == {(a, y)}
        vp = v + rng.uniform(-1e-8, 1e-8, v.shape)
        assert orc.speculative_accept(z, T, vp, x, ua, ur)[:2] in legit


# ------------------------------------------ sampled-greedy acceptance --

def _midpoint_u(P_row, y):
    c = np.cumsum(P_row)
    lo = c[y - 1] if y > 0 else 0.0
    return (lo + c[y]) / 2 / c[-1]


@pytest.mark.parametrize("V,G", [(2, 1), (3, 2), (3, 3), (4, 2)])
def test_sampled_greedy_expected_acceptance_is_the_streak_score(V, G):
    # Enumerate every verifier sample y in V^(G+1) (each u_j at the middle of
    # y_j's CDF interval, weight prod P_j(y_j)).  The expected number
    # accepted is the streak equation of p_j = P_j(x_j), and the first
    # committed token is distributed as P_1 (the rule is lossless).
    rng = np.random.default_rng(V * 100 + G)
    v = rng.normal(size=(G + 1, V)) * 1.5
    P = np.exp(v) / np.exp(v).sum(axis=-1, keepdims=True)
    x = rng.integers(0, V, G)
    expect, first = 0.0, np.zeros(V)
    for y in itertools.product(range(V), repeat=G + 1):
        prob = np.prod([P[j, y[j]] for j in range(G + 1)])
        u = [_midpoint_u(P[j], y[j]) for j in range(G + 1)]
        a, tok, _ = orc.sampled_greedy_accept(v, x, u)
        expect += prob * a
        first[x[0] if a > 0 else tok] += prob
    assert abs(expect - orc.streak_score([P[j, x[j]] for j in range(G)])) < 1e-12
    assert np.allclose(first, P[0], atol=1e-12)


def test_sampled_greedy_with_certain_verifier_is_the_greedy_rule():
    # A verifier sure of its token (one-hot rows) samples its argmax, so the
    # rule reduces to the DFlare post's greedy rule against the argmax.
    rng = np.random.default_rng(85)
    for _ in range(50):
        G, V = 5, 7
        t = rng.integers(0, V, G + 1)
        v = np.full((G + 1, V), -1e4)
        v[np.arange(G + 1), t] = 0.0
        x = t[:G].copy()
        cut = int(rng.integers(0, G + 1))
        if cut < G:
            x[cut] = (x[cut] + 1) % V
        u = rng.uniform(size=G + 1)
        a, tok, _ = orc.sampled_greedy_accept(v, x, u)
        assert (a, tok) == orc.greedy_accept(x, t)


def test_sampled_greedy_worked_case_and_outcomes():
    # P_1 = P_2 = (0.5, 0.25, 0.25): CDF (0.5, 0.75, 1)
    v = np.log(np.array([[0.5, 0.25, 0.25]] * 3))
    x = [0, 2]
    assert orc.sampled_greedy_accept(v, x, [0.2, 0.9, 0.3])[:2] == (2, 0)    # y = (0, 2), bonus 0
    assert orc.sampled_greedy_accept(v, x, [0.2, 0.6, 0.3])[:2] == (1, 1)    # y_2 = 1 != 2
    assert orc.sampled_greedy_accept(v, x, [0.7, 0.9, 0.3])[:2] == (0, 1)    # y_1 = 1 != 0
    a, tok, m = orc.sampled_greedy_accept(v, x, [0.2, 0.6, 0.3])
    assert abs(m - 0.1) < 1e-12                      # 0.6 is 0.1 above the boundary 0.5 (0.2 is 0.2 from 0)
    assert orc.sampled_greedy_outcomes(v, x, [0.2, 0.6, 0.3], 1e-6) == {(1, 1)}
    # y_1 on the boundary 0.5: token 0 (accept, then y_2 = 2, bonus 0) or token 1 (reject)
    assert orc.sampled_greedy_outcomes(v, x, [0.5, 0.9, 0.3], 1e-6) == {(2, 0), (0, 1)}
