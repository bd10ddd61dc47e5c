"""Seeded synthetic inputs for the block-diffusion draft step.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds shapes, random draws and storage-format conversion
only: none of the drafting method's arithmetic (no mixing, normalisation,
projection, attention, argmax or acceptance rule) lives here.

Every tensor is drawn from its own NumPy PCG64 stream keyed by
``(workload seed, tensor id, indices...)``, so a subset (one sequence, one
layer) can be regenerated without drawing the rest.  bf16 workloads round each
tensor once, round-to-nearest-even, so that both sides see identical bits.

Distributions follow the workload descriptions of the pages' drafter shapes
(DFlare blog, "evaluation conditions and data scale": Qwen 7 draft layers /
block 16 / 9 target layers, GPT-OSS 8 / 8 / 7; SpecDiff-2 notes, "experimental
setup": window gamma = 32, one denoising step; "Self-Selection Acceptance":
K drafts, T = 1.5).  Datasets are not used; these draws stand in for them.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "round_bf16", "bf16_bits", "bits_to_f32",
    "gen_hidden", "gen_hidden_scales", "gen_mix_logits", "gen_gains",
    "gen_layer_weights", "gen_lm_head", "gen_block_init", "gen_verifier_logits",
    "plant_targets", "geometric_prefix", "WEIGHT_NAMES", "FFN_WEIGHT_NAMES", "gen_ffn_gains",
    "gen_hidden_rows", "gen_cache_state", "gen_fc_weights",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes and draw parameters of one synthetic drafting workload."""
    name: str
    N: int          # sequences in the batch
    d: int          # hidden size
    Hq: int         # query heads
    Hkv: int        # key/value heads
    hd: int         # head dim
    D: int          # draft layers
    L: int          # mixed target layers
    B: int          # block length (1 anchor + B-1 [MASK])
    C: int          # context positions per sequence
    V: int          # vocabulary (0: no LM head, layer output only)
    dtype: str      # "f32" or "bf16"
    seed: int
    geom_p: float = 0.0        # planted agreement prefix ~ Geometric(p)
    hidden_scale: bool = True  # per-(sequence, target layer) scale U(0.5, 2)
    K: int = 0                 # drafts per sequence (self-selection)
    T: float = 1.0             # sampling temperature
    philox_seed: int = 0
    verifier_scale: float = 4.0
    rope_theta: float = 1.0e6
    eps: float = 1.0e-6
    F: int = 0                 # feed-forward width of full draft layers (0: no FFN)
    R: int = 0                 # cached-context workloads: new context rows per step
                               # (C is then the cache capacity per sequence)
    fc: int = 0                # 1: context features from one FC over the L target layers
                               # (DFlash fusion) instead of per-layer mixtures

    @property
    def gamma(self) -> int:
        """Draft window: the B-1 mask positions."""
        return self.B - 1

    @property
    def n_mix_coefficients(self) -> int:
        return self.D * self.L


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", N=1, d=256, Hq=4, Hkv=4, hd=64, D=1, L=3,
                         B=16, C=64, V=1000, dtype="f32", seed=1001,
                         geom_p=0.2, hidden_scale=False),
    "qwen3_8b_layer": Workload("qwen3_8b_layer", N=1, d=4096, Hq=32, Hkv=8,
                               hd=128, D=1, L=9, B=16, C=1024, V=0,
                               dtype="bf16", seed=1002),
    "qwen3_8b_drafter": Workload("qwen3_8b_drafter", N=32, d=4096, Hq=32,
                                 Hkv=8, hd=128, D=7, L=9, B=16, C=2048,
                                 V=151936, dtype="bf16", seed=1003,
                                 geom_p=0.15),
    "gpt_oss_20b_drafter": Workload("gpt_oss_20b_drafter", N=32, d=2880,
                                    Hq=64, Hkv=8, hd=64, D=8, L=7, B=8,
                                    C=3072, V=201088, dtype="bf16",
                                    seed=1004, geom_p=0.2),
    "specdiff2_select": Workload("specdiff2_select", N=16, d=4096, Hq=32,
                                 Hkv=8, hd=128, D=7, L=9, B=33, C=1024,
                                 V=151936, dtype="bf16", seed=1005, K=8,
                                 T=1.5, philox_seed=0x5EEDD1F5),
    # A next-row workload (not one of the five): the Qwen3-8B drafter with full
    # decoder layers, i.e. a SwiGLU feed-forward block of Qwen3-8B's width.
    "qwen3_8b_drafter_ffn": Workload("qwen3_8b_drafter_ffn", N=32, d=4096, Hq=32,
                                     Hkv=8, hd=128, D=7, L=9, B=16, C=2048,
                                     V=151936, dtype="bf16", seed=1006,
                                     geom_p=0.15, F=12288),
    # A next-row workload: the Qwen3-8B drafter in steady-state decoding with
    # a per-layer context K/V cache.  Capacity 4096 positions per sequence,
    # cached lengths ragged around 2048, up to 16 new rows per step.
    "qwen3_8b_drafter_cached": Workload("qwen3_8b_drafter_cached", N=32, d=4096, Hq=32, Hkv=8, hd=128, D=7,
                                        L=9, B=16, C=4096, V=151936, dtype="bf16", seed=1007, geom_p=0.15,
                                        R=16),
    # A next-row workload: the Qwen3-8B drafter in DFlash's form, where one
    # fully connected layer fuses the 9 target layers into a representation
    # shared by all 7 draft layers (in place of DFlare's per-layer mixtures).
    "qwen3_8b_drafter_dflash": Workload("qwen3_8b_drafter_dflash", N=32, d=4096, Hq=32, Hkv=8, hd=128, D=7,
                                        L=9, B=16, C=2048, V=151936, dtype="bf16", seed=1008, geom_p=0.15,
                                        fc=1),
}

# Tensor ids keying the PCG64 streams.
_TID_H, _TID_HSCALE, _TID_MIX, _TID_W, _TID_LM = 1, 2, 3, 4, 5
_TID_ANCHOR, _TID_MASK, _TID_VLOG, _TID_PLANT, _TID_GAIN = 6, 7, 8, 9, 10
_TID_FFN_GAIN = 11
_TID_HROWS, _TID_CACHE = 12, 13
_TID_FC, _TID_FC_GAIN = 14, 15
_HCHUNK = 256   # positions per stream of gen_hidden_rows
WEIGHT_NAMES = ("Wq", "Wkc", "Wvc", "Wkb", "Wvb", "Wo")
FFN_WEIGHT_NAMES = ("W1", "W3", "W2")

_THREADS = max(1, min(16, len(os.sched_getaffinity(0))))


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> float32 holding the nearest bf16 value (ties to even)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = (b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))) \
        & np.uint32(0xFFFF0000)
    return b.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 (already bf16-exact) -> uint16 storage bits."""
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
            >> np.uint32(16)).astype(np.uint16)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 storage bits -> float32."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _finish(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_bf16(x) if dtype == "bf16" else x.astype(np.float32, copy=False)


def _normal(key, shape, std=1.0) -> np.ndarray:
    x = _rng(*key).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def _parallel(fn, items):
    if len(items) <= 1:
        return [fn(i) for i in items]
    with ThreadPoolExecutor(_THREADS) as ex:
        return list(ex.map(fn, items))


def gen_hidden_scales(w: Workload) -> np.ndarray:
    """Per-(sequence, target layer) scale s ~ U(0.5, 2); ones if disabled."""
    if not w.hidden_scale:
        return np.ones((w.N, w.L), np.float32)
    return _rng(w.seed, _TID_HSCALE).uniform(0.5, 2.0, (w.N, w.L)).astype(np.float32)


def gen_hidden(w: Workload, seqs=None, as_bits: bool = False) -> np.ndarray:
    """Target hidden-state stack H[L][len(seqs)*C][d], rows ordered (seq, pos).

    H_i[n] = s[n, i] * N(0, 1); values rounded to bf16 for bf16 workloads.
    With ``as_bits`` (bf16 only) returns uint16 storage bits instead.
    """
    seqs = list(range(w.N)) if seqs is None else list(seqs)
    scales = gen_hidden_scales(w)
    out_dtype = np.uint16 if as_bits else np.float32
    if as_bits and w.dtype != "bf16":
        raise ValueError("as_bits needs a bf16 workload")
    out = np.empty((w.L, len(seqs) * w.C, w.d), out_dtype)

    def one(job):
        i, j = job
        n = seqs[j]
        x = _normal((w.seed, _TID_H, i, n), (w.C, w.d))
        x *= scales[n, i]
        x = _finish(x, w.dtype)
        out[i, j * w.C:(j + 1) * w.C] = bf16_bits(x) if as_bits else x

    _parallel(one, [(i, j) for i in range(w.L) for j in range(len(seqs))])
    return out


def gen_hidden_rows(w: Workload, n: int, r0: int, r1: int, as_bits: bool = False) -> np.ndarray:
    """Target hidden states of positions r0..r1-1 of sequence n: [L][r1-r0][d].

    The cached-context workloads' hidden states: drawn in 256-position
    streams keyed (seed, tensor id, layer, sequence, chunk), so the rows that
    arrive with one step are regenerated without the positions before them.
    Same distribution as ``gen_hidden`` (per-(sequence, layer) scale times
    N(0, 1), bf16-rounded for bf16 workloads).
    """
    if as_bits and w.dtype != "bf16":
        raise ValueError("as_bits needs a bf16 workload")
    scales = gen_hidden_scales(w)
    out = np.empty((w.L, r1 - r0, w.d), np.uint16 if as_bits else np.float32)
    chunks = list(range(r0 // _HCHUNK, (r1 + _HCHUNK - 1) // _HCHUNK)) if r1 > r0 else []

    def one(job):
        i, c = job
        x = _normal((w.seed, _TID_HROWS, i, n, c), (_HCHUNK, w.d))
        a, b = max(r0, c * _HCHUNK), min(r1, (c + 1) * _HCHUNK)
        x = _finish(x[a - c * _HCHUNK:b - c * _HCHUNK] * scales[n, i], w.dtype)
        out[i, a - r0:b - r0] = bf16_bits(x) if as_bits else x

    _parallel(one, [(i, c) for i in range(w.L) for c in chunks])
    return out


def gen_cache_state(w: Workload):
    """Cached lengths c0[N] ~ U{C/4 .. 3C/4} and new rows n_new[N] = min(Geometric(p), R).

    n_new stands for the tokens a verifier accepted in the previous step plus
    its bonus token (at least 1, at most the R rows a step brings).
    """
    r = _rng(w.seed, _TID_CACHE)
    c0 = r.integers(w.C // 4, 3 * w.C // 4 + 1, size=w.N)
    m = np.minimum(r.geometric(w.geom_p, size=w.N), w.R)
    return c0.astype(np.int32), m.astype(np.int32)


def gen_mix_logits(w: Workload) -> np.ndarray:
    """Mixture logits [D][L] ~ N(0, 1), fp32."""
    return _normal((w.seed, _TID_MIX), (w.D, w.L))


def gen_gains(w: Workload, random: bool = False):
    """RMSNorm gains: mix [D][d], block-input [D][d], final [d] (fp32).

    The workloads use unit gains; ``random`` draws U(0.5, 1.5) for tests.
    """
    if not random:
        return (np.ones((w.D, w.d), np.float32), np.ones((w.D, w.d), np.float32),
                np.ones((w.d,), np.float32))
    r = _rng(w.seed, _TID_GAIN)
    return (r.uniform(0.5, 1.5, (w.D, w.d)).astype(np.float32),
            r.uniform(0.5, 1.5, (w.D, w.d)).astype(np.float32),
            r.uniform(0.5, 1.5, (w.d,)).astype(np.float32))


def weight_shapes(w: Workload) -> dict:
    """[out][in] shapes (nn.Linear layout) of one draft layer's weights."""
    shapes = {"Wq": (w.Hq * w.hd, w.d), "Wkc": (w.Hkv * w.hd, w.d),
              "Wvc": (w.Hkv * w.hd, w.d), "Wkb": (w.Hkv * w.hd, w.d),
              "Wvb": (w.Hkv * w.hd, w.d), "Wo": (w.d, w.Hq * w.hd)}
    if w.F > 0:
        shapes.update({"W1": (w.F, w.d), "W3": (w.F, w.d), "W2": (w.d, w.F)})
    return shapes


def gen_ffn_gains(w: Workload, random: bool = False) -> np.ndarray:
    """Feed-forward RMSNorm gains [D][d]: ones, or U(0.5, 1.5) for tests."""
    if not random:
        return np.ones((w.D, w.d), np.float32)
    return _rng(w.seed, _TID_FFN_GAIN).uniform(0.5, 1.5, (w.D, w.d)).astype(np.float32)


def gen_layer_weights(w: Workload, layer: int) -> dict:
    """One draft layer's weights, each N(0, std 1/sqrt(fan_in))."""
    shapes = weight_shapes(w)
    names = WEIGHT_NAMES + (FFN_WEIGHT_NAMES if w.F > 0 else ())

    def one(k):
        name = names[k]
        out_f, in_f = shapes[name]
        return _finish(_normal((w.seed, _TID_W, layer, k), (out_f, in_f),
                               1.0 / np.sqrt(in_f)), w.dtype)

    return dict(zip(names, _parallel(one, list(range(len(names))))))


def gen_fc_weights(w: Workload, random_gain: bool = False):
    """DFlash fusion: W_fc [d][L*d] ~ N(0, std 1/sqrt(L*d)) in the working
    dtype (drawn in row chunks), and its RMSNorm gain [d] (ones, or
    U(0.5, 1.5) for tests)."""
    chunk = 512
    out = np.empty((w.d, w.L * w.d), np.float32)

    def one(c):
        r0, r1 = c * chunk, min(w.d, (c + 1) * chunk)
        out[r0:r1] = _finish(_normal((w.seed, _TID_FC, c), (r1 - r0, w.L * w.d), 1.0 / np.sqrt(w.L * w.d)),
                             w.dtype)

    _parallel(one, list(range((w.d + chunk - 1) // chunk)))
    g = (_rng(w.seed, _TID_FC_GAIN).uniform(0.5, 1.5, w.d).astype(np.float32) if random_gain
         else np.ones((w.d,), np.float32))
    return out, g


def gen_lm_head(w: Workload, as_bits: bool = False) -> np.ndarray:
    """Shared LM head W_lm[V][d] ~ N(0, std 1/sqrt(d)), drawn in row chunks."""
    chunk = 8192
    out = np.empty((w.V, w.d), np.uint16 if as_bits else np.float32)

    def one(c):
        r0, r1 = c * chunk, min(w.V, (c + 1) * chunk)
        x = _finish(_normal((w.seed, _TID_LM, c), (r1 - r0, w.d),
                            1.0 / np.sqrt(w.d)), w.dtype)
        out[r0:r1] = bf16_bits(x) if as_bits else x

    _parallel(one, list(range((w.V + chunk - 1) // chunk)))
    return out


def gen_block_init(w: Workload) -> np.ndarray:
    """Initial block features Xb0[N][B][d] (fp32 storage).

    Row 0 of each sequence is its anchor token's embedding, rows 1..B-1 the
    shared [MASK] embedding; both N(0, 1), rounded to bf16 for bf16 workloads
    (an embedding table would be stored in the working dtype).
    """
    anchor = _finish(_normal((w.seed, _TID_ANCHOR), (w.N, w.d)), w.dtype)
    mask = _finish(_normal((w.seed, _TID_MASK), (w.d,)), w.dtype)
    x = np.empty((w.N, w.B, w.d), np.float32)
    x[:, 0] = anchor
    x[:, 1:] = mask
    return x


def gen_verifier_logits(w: Workload, seqs=None, as_bits: bool = False) -> np.ndarray:
    """Synthetic verifier logits vlog[n][K][gamma+1][V] = 4 * N(0, 1), bf16.

    Row j of draft k stands for the verifier's distribution at window
    position j+1 given the prefix s + x^k_{1..j}; row gamma serves the bonus.
    """
    seqs = list(range(w.N)) if seqs is None else list(seqs)
    G1 = w.gamma + 1
    out = np.empty((len(seqs), w.K, G1, w.V), np.uint16 if as_bits else np.float32)

    def one(job):
        j, k = job
        x = round_bf16(_normal((w.seed, _TID_VLOG, seqs[j], k), (G1, w.V),
                               w.verifier_scale))
        out[j, k] = bf16_bits(x) if as_bits else x

    _parallel(one, [(j, k) for j in range(len(seqs)) for k in range(w.K)])
    return out


def geometric_prefix(w: Workload) -> np.ndarray:
    """Planted agreement lengths G_n = min(G, B-1), G = failures before the
    first success of a Bernoulli(p) sequence, so P(G >= k) = (1-p)^k."""
    r = _rng(w.seed, _TID_PLANT, 0)
    g = r.geometric(w.geom_p, size=w.N) - 1
    return np.minimum(g, w.B - 1).astype(np.int64)


def plant_targets(w: Workload, drafts: np.ndarray) -> np.ndarray:
    """Target argmax tokens t[N][B] agreeing with ``drafts`` for a planted prefix.

    ``drafts`` is [N][B-1] (window positions 1..B-1).  For sequence n with
    planted length G_n: t_j = d_j for j <= G_n; if G_n < B-1 the token at
    j = G_n+1 is drawn uniformly among the V-1 tokens other than d_j; every
    later token (including the bonus slot t_B) is uniform over the vocabulary.
    Returned 0-based: column j-1 holds t_j.
    """
    drafts = np.asarray(drafts, dtype=np.int64)
    N, n = drafts.shape
    assert N == w.N and n == w.B - 1
    G = geometric_prefix(w)
    r = _rng(w.seed, _TID_PLANT, 1)
    t = r.integers(0, w.V, size=(N, w.B), dtype=np.int64)
    shift = r.integers(1, w.V, size=N, dtype=np.int64)   # 1..V-1
    for s in range(N):
        g = int(G[s])
        t[s, :g] = drafts[s, :g]
        if g < n:
            t[s, g] = (drafts[s, g] + shift[s]) % w.V
    return t.astype(np.int32)
