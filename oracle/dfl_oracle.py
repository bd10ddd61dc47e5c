"""CPU oracle for the block-diffusion draft step: plain, slow, fp64 NumPy.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
library or its Python binding; the one module both sides use is the seeded
input generator ``dfl_synth``.

Every function states the passage it restates.  Sources (page title, section):

* DFlare post -- "DFlare: Scaling Up Draft Capacity for Block Diffusion
  Speculative Decoding" (iplexlaw blog).  Sections used:
  "Generating candidates in parallel, the target decides acceptance" (one
  forward over the mask positions, bidirectional attention in the block,
  greedy rule: prefix up to the first mismatch plus one target token);
  "Per-draft-layer mixing of different information" (softmax-normalised
  mixing ratios over several target hidden states, then RMSNorm; 7 x 9 = 63
  coefficients); "Separate KV projections by information source" (separate
  key/value projections for target-context features and for the draft's
  anchor/mask features, queries from the draft features); "Stabilise the front,
  weight the back" (embedding and LM head frozen and shared).
* DFlash article -- "DFlash: Block Diffusion for Flash Speculative Decoding"
  (Qiita), section "Writing a whole block in one forward pass" (target
  features from several layers injected into the K/V of every draft layer).
* SpecDiff-2 notes -- "SpecDiff-2 -- Scaling Diffusion Drafter Alignment For
  Faster Speculative Decoding" (MLSys 2026 talk notes).  Sections used:
  "Parallel drafting with diffusion language models" (one denoising step gives
  per-position marginals q_1..q_gamma, a joint draft is sampled from them);
  "Streak-Distillation" (streak equation, TV acceptance proxy, Theorem C.3);
  "Self-Selection Acceptance" (K independent drafts, argmax of the streak
  score, greedy acceptance on the chosen draft reusing verifier posteriors).

Where the pages leave a step open the plainest reading is taken; each reading
is named in the docstring of the function that takes it.

Parity: every function here is pinned by a ``-m "not gpu"`` test against a
closed form, an invariant, brute-force enumeration, a hand-worked case or (for
``philox4x32_10``) the generator's published known-answer vectors.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# Per-draft-layer mixture and RMSNorm (DFlare post, "Per-draft-layer mixing")
# ---------------------------------------------------------------------------

def mix_weights(mix_logits) -> np.ndarray:
    """Softmax of one draft layer's mixing logits over the L target layers.

    DFlare post, "Per-draft-layer mixing": each draft layer learns mixing
    ratios over several target hidden states, normalised with softmax.
    Works on the last axis, so a [D][L] array gives D independent mixtures.
    """
    z = np.asarray(mix_logits, dtype=F64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def rmsnorm(x, gain, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x * g / sqrt(mean(x^2) + eps)."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gain, dtype=F64)


def mix_rmsnorm(H, mix_logits, gain, eps: float) -> np.ndarray:
    """Context features of one draft layer: RMSNorm(sum_i a_i H_i).

    DFlare post, "Per-draft-layer mixing": mix with the softmax ratios first,
    then apply RMSNorm (the order the section states).  H is [L][rows][d];
    the result is [rows][d].
    """
    a = mix_weights(mix_logits)
    H = np.asarray(H, dtype=F64)
    x = np.zeros(H.shape[1:], dtype=F64)
    for i in range(H.shape[0]):
        x += a[i] * H[i]
    return rmsnorm(x, gain, eps)


def fc_fuse(H, W_fc, gain, eps: float) -> np.ndarray:
    """DFlash's shared context representation: one FC over L target layers.

    DFlash article, "Writing a whole block in one forward pass": hidden
    features taken from several target layers are fused by a light
    projection and injected into the K/V of every draft layer; the DFlare
    post ("Per-draft-layer mixing") describes the same baseline as a fully
    connected layer that fuses the target features into one common
    representation, which DFlare replaces by per-layer softmax mixes.

    Reading: the L hidden states of a position are concatenated layer by
    layer into one vector of L*d values, W_fc [d][L*d] (no bias) maps it to d
    features, and an RMSNorm with gain ``gain`` follows (the normalisation
    DFlare keeps after its own mixture).  H is [L][rows][d]; the result is
    [rows][d], shared by every draft layer.
    """
    H = np.asarray(H, dtype=F64)
    L, rows, d = H.shape
    cat = np.empty((rows, L * d), dtype=F64)
    for i in range(L):
        cat[:, i * d:(i + 1) * d] = H[i]
    return rmsnorm(cat @ np.asarray(W_fc, dtype=F64).T, gain, eps)


# ---------------------------------------------------------------------------
# Rotary positions (reading: the pages give no position scheme)
# ---------------------------------------------------------------------------

def rope_cos_sin(positions, hd: int, theta: float):
    """cos/sin tables [P][hd/2] for rotate-half rotary embedding.

    Reading: the pages name no position encoding, yet without one every
    [MASK] row of the block is identical and could not predict different
    tokens, contradicting the position-wise drafting the DFlare post
    describes.  Rotary embedding with frequency theta^(-2i/hd) is taken.
    """
    i = np.arange(hd // 2, dtype=F64)
    inv_freq = float(theta) ** (-2.0 * i / hd)
    ang = np.asarray(positions, dtype=F64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def apply_rope(x, cos, sin) -> np.ndarray:
    """Rotate-half rotary embedding of x[P][heads][hd] by tables [P][hd/2].

    Pairs element i with element i + hd/2 of each head and rotates the pair
    by the position's angle.
    """
    x = np.asarray(x, dtype=F64)
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------------------
# Attention pattern (DFlare post, "Generating candidates in parallel";
# DFlash article, "Writing a whole block in one forward pass")
# ---------------------------------------------------------------------------

def block_visibility(C: int, B: int) -> np.ndarray:
    """Visibility of keys [context C ; block B] to the B block queries.

    Every block query sees every context key (target features enter the K/V
    of each draft layer) and attends bidirectionally inside the block, so
    nothing is hidden: an all-true [B][C+B] matrix.
    """
    return np.ones((B, C + B), dtype=bool)


def attention(Q, K, V, visible) -> np.ndarray:
    """Masked softmax attention with grouped K/V heads.

    Q [Bq][Hq][hd], K/V [S][Hkv][hd], visible [Bq][S] (True = may attend).
    Query head h reads K/V head h // (Hq/Hkv).  For each head an explicit
    score matrix QK^T/sqrt(hd) gets -inf where hidden, then a row softmax,
    then P V.
    """
    Q = np.asarray(Q, dtype=F64)
    K = np.asarray(K, dtype=F64)
    V = np.asarray(V, dtype=F64)
    Bq, Hq, hd = Q.shape
    S, Hkv, _ = K.shape
    group = Hq // Hkv
    bias = np.where(np.asarray(visible, dtype=bool), 0.0, -np.inf)
    O = np.empty((Bq, Hq, V.shape[-1]), dtype=F64)
    for h in range(Hq):
        g = h // group
        scores = Q[:, h, :] @ K[:, g, :].T / np.sqrt(hd) + bias
        m = scores.max(axis=1, keepdims=True)
        P = np.exp(scores - m)
        P /= P.sum(axis=1, keepdims=True)
        O[:, h, :] = P @ V[:, g, :]
    return O


# ---------------------------------------------------------------------------
# One draft layer and the whole draft forward
# ---------------------------------------------------------------------------

def draft_layer(Xb, Hn, mix_logits, g_mix, g_blk, W: dict, shape: dict,
                eps: float, theta: float, Xc=None) -> dict:
    """One block-diffusion draft layer for one sequence.

    Xb [B][d] is the block's residual stream (row 0 the anchor token, rows
    1..B-1 the [MASK] positions); Hn [L][C][d] the target hidden states of the
    sequence's C context positions.

    * context features: RMSNorm of the softmax mix of the L target layers
      (DFlare post, "Per-draft-layer mixing");
    * separate K/V weights for context features (Wkc, Wvc) and for the draft's
      own features (Wkb, Wvb); queries only from the draft features (Wq)
      (DFlare post, "Separate KV projections by information source");
    * attention where block queries see all context keys and attend
      bidirectionally in the block (DFlare post, "Generating candidates in
      parallel"; DFlash article, "Writing a whole block in one forward pass").

    Readings (the pages are silent on them): the block input is RMS-normalised
    before its projections (pre-norm, gain g_blk); the layer ends with an
    output projection Wo added to the residual stream; there is no FFN;
    rotary positions 0..C-1 for context and C..C+B-1 for the block.
    ``Xc`` [C][d], when given, replaces the layer's own mixture as the
    context features (the DFlash form, where one fused representation of the
    target features serves every draft layer; see ``fc_fuse``).
    Returns every intermediate for per-tensor comparison.
    """
    B, d = Xb.shape
    Hq, Hkv, hd = shape["Hq"], shape["Hkv"], shape["hd"]
    Xb = np.asarray(Xb, dtype=F64)
    if Xc is None:
        Xc = mix_rmsnorm(Hn, mix_logits, g_mix, eps)
    Xc = np.asarray(Xc, dtype=F64)
    C = Xc.shape[0]
    Xn = rmsnorm(Xb, g_blk, eps)
    f = {k: np.asarray(v, dtype=F64) for k, v in W.items()}
    Q = (Xn @ f["Wq"].T).reshape(B, Hq, hd)
    Kb = (Xn @ f["Wkb"].T).reshape(B, Hkv, hd)
    Vb = (Xn @ f["Wvb"].T).reshape(B, Hkv, hd)
    Kc = (Xc @ f["Wkc"].T).reshape(C, Hkv, hd)
    Vc = (Xc @ f["Wvc"].T).reshape(C, Hkv, hd)
    cos, sin = rope_cos_sin(np.arange(C + B), hd, theta)
    Q = apply_rope(Q, cos[C:], sin[C:])
    Kb = apply_rope(Kb, cos[C:], sin[C:])
    Kc = apply_rope(Kc, cos[:C], sin[:C])
    O = attention(Q, np.concatenate([Kc, Kb]), np.concatenate([Vc, Vb]),
                  block_visibility(C, B))
    Xb_out = Xb + O.reshape(B, Hq * hd) @ f["Wo"].T
    out = {"Xc": Xc, "Xn": Xn, "Q": Q, "Kc": Kc, "Vc": Vc, "Kb": Kb,
           "Vb": Vb, "O": O, "Xb_attn": Xb_out, "Xb": Xb_out}
    if "W1" in f:
        out["Xb"] = swiglu_ffn(Xb_out, W["g_ffn"], f["W1"], f["W3"], f["W2"], eps)
    return out


def silu(x) -> np.ndarray:
    """x * sigmoid(x)."""
    x = np.asarray(x, dtype=F64)
    return x / (1.0 + np.exp(-x))


def swiglu_ffn(Xb, g_ffn, W1, W3, W2, eps: float) -> np.ndarray:
    """Residual SwiGLU feed-forward block of a Qwen-style decoder layer.

    Reading (the pages give no width or form; the DFlash article's drafter
    layers are the target family's decoder layers): Xn = RMSNorm(Xb; g_ffn),
    Xb + (silu(Xn W1^T) * (Xn W3^T)) W2^T with W1, W3 [F][d] and W2 [d][F].
    """
    Xn = rmsnorm(Xb, g_ffn, eps)
    gate = Xn @ np.asarray(W1, dtype=F64).T
    up = Xn @ np.asarray(W3, dtype=F64).T
    return np.asarray(Xb, dtype=F64) + (silu(gate) * up) @ np.asarray(W2, dtype=F64).T


def lm_head_logits(X_rows, g_final, eps: float, W_lm, chunk: int = 8192) -> np.ndarray:
    """Logits of the shared frozen LM head: RMSNorm_final(x) W_lm^T.

    DFlare post, "Stabilise the front, weight the back": the embedding and the
    LM head are frozen and shared with the target.  Reading: a final RMSNorm
    (gain g_final) precedes the head, as in the Qwen-shaped targets.  The
    vocabulary is processed in slices of rows of W_lm only to bound memory;
    each logit is one dot product either way.
    """
    x = rmsnorm(X_rows, g_final, eps)
    V = W_lm.shape[0]
    z = np.empty((x.shape[0], V), dtype=F64)
    for v0 in range(0, V, chunk):
        v1 = min(V, v0 + chunk)
        z[:, v0:v1] = x @ np.asarray(W_lm[v0:v1], dtype=F64).T
    return z


def argmax_lowest(z) -> np.ndarray:
    """Row-wise argmax; equal maxima resolve to the lowest index."""
    z = np.asarray(z)
    return np.argmax(z, axis=-1)


def draft_forward(Xb0, Hn, mix, g_mix, g_blk, layers, shape: dict,
                  eps: float, theta: float, keep_layers: bool = False, fused=None) -> dict:
    """All D draft layers of one sequence (one single-pass block forward).

    DFlare post, "Generating candidates in parallel": one forward predicts
    every mask position.  ``layers`` is a list of D weight dicts.  With
    ``fused`` = (W_fc, g_fc) the context features of every layer are the one
    DFlash fusion ``fc_fuse(Hn, W_fc, g_fc)`` instead of per-layer mixtures
    (``mix`` and ``g_mix`` are then unused).
    """
    Xb = np.asarray(Xb0, dtype=F64)
    Xc = None if fused is None else fc_fuse(Hn, fused[0], fused[1], eps)
    per_layer = []
    for l, W in enumerate(layers):
        out = draft_layer(Xb, Hn, None if fused else mix[l], None if fused else g_mix[l], g_blk[l], W, shape,
                          eps, theta, Xc=Xc)
        Xb = out["Xb"]
        per_layer.append(out if keep_layers else {"Xb": Xb})
    return {"Xb": Xb, "layers": per_layer}


# ---------------------------------------------------------------------------
# Incremental context K/V (SpecDiff-2 notes, "Future work and limitations",
# hardware-optimisation item: KV-cache support for gamma-length drafts)
# ---------------------------------------------------------------------------

def context_kv_rows(H_rows, mix_logits, g_mix, Wkc, Wvc, positions, shape: dict,
                    eps: float, theta: float):
    """Context keys and values of some context positions of one draft layer.

    H_rows [L][m][d] holds the target hidden states of m context positions,
    ``positions`` [m] their absolute positions.  The context side of a draft
    layer works row by row: position t's key and value depend on the mixed,
    normalised hidden states of position t alone, and the key also on t
    through the rotary embedding.  So K/V computed for a context in pieces
    equal K/V computed for it at once, which is what lets a drafter keep them
    from one draft step to the next.
    """
    Hkv, hd = shape["Hkv"], shape["hd"]
    Xc = mix_rmsnorm(H_rows, mix_logits, g_mix, eps)
    m = Xc.shape[0]
    K = (Xc @ np.asarray(Wkc, dtype=F64).T).reshape(m, Hkv, hd)
    V = (Xc @ np.asarray(Wvc, dtype=F64).T).reshape(m, Hkv, hd)
    cos, sin = rope_cos_sin(np.asarray(positions), hd, theta)
    return apply_rope(K, cos, sin), V


def draft_step_cached(Xb0, H_new, cache, mix, g_mix, g_blk, layers, shape: dict,
                      eps: float, theta: float):
    """One draft step over cached context K/V, appending the new positions.

    ``cache`` is a list of D pairs (K [c0][Hkv][hd], V [c0][Hkv][hd]): the
    context keys/values of the c0 positions seen in earlier steps, one pair per
    draft layer.  H_new [L][m][d] holds the target hidden states of the m
    positions c0..c0+m-1 that arrive with this step (m = 0 allowed).  Each
    layer appends their K/V to its cache, then runs the block part over the
    C = c0 + m cached positions, with the block at positions C..C+B-1 (the
    same positions the one-shot step gives a context of length C).  Returns
    the block output and the extended caches.

    Reading (the pages name the missing cache, not its design): cached rows
    are never recomputed, so the result equals the one-shot step over the
    concatenated context.
    """
    Xb = np.asarray(Xb0, dtype=F64)
    B = Xb.shape[0]
    Hq, Hkv, hd = shape["Hq"], shape["Hkv"], shape["hd"]
    H_new = np.asarray(H_new, dtype=F64)
    m = H_new.shape[1]
    new_cache = []
    for l, W in enumerate(layers):
        Kold, Vold = cache[l]
        c0 = Kold.shape[0]
        if m > 0:
            Kn, Vn = context_kv_rows(H_new, mix[l], g_mix[l], W["Wkc"], W["Wvc"], np.arange(c0, c0 + m),
                                     shape, eps, theta)
            Kc, Vc = np.concatenate([Kold, Kn]), np.concatenate([Vold, Vn])
        else:
            Kc, Vc = np.asarray(Kold, dtype=F64), np.asarray(Vold, dtype=F64)
        new_cache.append((Kc, Vc))
        C = Kc.shape[0]
        f = {k: np.asarray(v, dtype=F64) for k, v in W.items()}
        Xn = rmsnorm(Xb, g_blk[l], eps)
        cos, sin = rope_cos_sin(np.arange(C, C + B), hd, theta)
        Q = apply_rope((Xn @ f["Wq"].T).reshape(B, Hq, hd), cos, sin)
        Kb = apply_rope((Xn @ f["Wkb"].T).reshape(B, Hkv, hd), cos, sin)
        Vb = (Xn @ f["Wvb"].T).reshape(B, Hkv, hd)
        O = attention(Q, np.concatenate([Kc, Kb]), np.concatenate([Vc, Vb]), block_visibility(C, B))
        Xb = Xb + O.reshape(B, Hq * hd) @ f["Wo"].T
        if "W1" in f:
            Xb = swiglu_ffn(Xb, W["g_ffn"], f["W1"], f["W3"], f["W2"], eps)
    return Xb, new_cache


# ---------------------------------------------------------------------------
# Greedy acceptance (DFlare post, "Generating candidates in parallel")
# ---------------------------------------------------------------------------

def greedy_accept(draft, target):
    """Accept the draft prefix up to the first mismatch, then one target token.

    draft [n] holds window positions 1..n, target [n+1] the target's argmax
    tokens t_1..t_{n+1} for the same positions.  Returns (a, bonus): a is the
    number of leading j with draft_j == t_j, bonus = t_{a+1}.  The tokens
    committed this step are a + 1.
    """
    draft = list(np.asarray(draft).tolist())
    target = list(np.asarray(target).tolist())
    assert len(target) == len(draft) + 1
    a = 0
    while a < len(draft) and draft[a] == target[a]:
        a += 1
    return a, target[a]


# ---------------------------------------------------------------------------
# Counter-based generator: Philox4x32-10 (Salmon, Moraes, Dror & Shaw,
# "Parallel random numbers: as easy as 1, 2, 3", SC'11)
# ---------------------------------------------------------------------------

_PHILOX_M = (0xD2511F53, 0xCD9E8D57)
_PHILOX_W = (0x9E3779B9, 0xBB67AE85)
_MASK32 = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox4x32 with 10 rounds, from the published definition.

    One round: two 32x32->64 products of the multipliers with counter words 0
    and 2; the new counter is (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0).  The
    key advances by the Weyl constants between rounds.  Python integers.
    """
    c = [int(v) & _MASK32 for v in ctr]
    k = [int(v) & _MASK32 for v in key]
    for _ in range(10):
        p0 = _PHILOX_M[0] * c[0]
        p1 = _PHILOX_M[1] * c[2]
        hi0, lo0 = p0 >> 32, p0 & _MASK32
        hi1, lo1 = p1 >> 32, p1 & _MASK32
        c = [hi1 ^ c[1] ^ k[0], lo1, hi0 ^ c[3] ^ k[1], lo0]
        k = [(k[0] + _PHILOX_W[0]) & _MASK32, (k[1] + _PHILOX_W[1]) & _MASK32]
    return tuple(c)


def draw_uniform(seed: int, n: int, j: int, k: int) -> float:
    """The uniform for sequence n, window row j, draft k.

    Counter (n, j, k, 0), key (low, high 32 bits of the seed); the top 24 bits
    of output word 0 give u = (x >> 8 + 1/2) 2^-24, strictly inside (0, 1).
    """
    x0 = philox4x32_10((n, j, k, 0), (seed & _MASK32, (seed >> 32) & _MASK32))[0]
    return ((x0 >> 8) + 0.5) * 2.0 ** -24


# ---------------------------------------------------------------------------
# K-draft sampling (SpecDiff-2 notes, "Parallel drafting with diffusion LMs",
# "Self-Selection Acceptance")
# ---------------------------------------------------------------------------

def sample_inverse_cdf(z, T: float, u: float):
    """One draw from softmax(z / T) by inversion of its CDF.

    One denoising step gives per-position marginals q_j; independent draws
    from them give the K joint drafts.  Returns (v, margin): v is the smallest
    index whose cumulative weight sum_{w<=v} exp((z_w - max z)/T) exceeds
    u * (total weight); margin is the distance from u * total to the nearest
    cumulative boundary, as a fraction of the total (how close the draw came
    to picking a neighbour).
    """
    z = np.asarray(z, dtype=F64)
    w = np.exp((z - z.max()) / T)
    cdf = np.cumsum(w)
    total = cdf[-1]
    t = u * total
    v = int(np.searchsorted(cdf, t, side="right"))
    v = min(v, len(z) - 1)
    lo = cdf[v - 1] if v > 0 else 0.0
    margin = min(abs(t - lo), abs(cdf[v] - t)) / total
    return v, margin


# ---------------------------------------------------------------------------
# Streak score, self-selection, TV acceptance (SpecDiff-2 notes,
# "Streak-Distillation", "Self-Selection Acceptance")
# ---------------------------------------------------------------------------

def streak_score(p) -> float:
    """Tokens/Draft = sum_{m=1}^{gamma} prod_{j<=m} p_j (streak equation).

    p [gamma] are the per-position acceptance probabilities of one draft.
    """
    total, prod = 0.0, 1.0
    for pj in np.asarray(p, dtype=F64):
        prod *= pj
        total += prod
    return total


def log_softmax_at(v_row, x: int) -> float:
    """log p(x) = v[x] - log sum exp(v) for one verifier row."""
    v = np.asarray(v_row, dtype=F64)
    m = v.max()
    return v[x] - (m + np.log(np.sum(np.exp(v - m))))


def self_select(vlog, drafts):
    """Pick the draft with the largest streak score and greedy-accept it.

    vlog [K][gamma+1][V] verifier logits (row j: distribution at window
    position j+1 given the draft's prefix; row gamma serves the bonus);
    drafts [K][gamma].  Score_k = sum_m prod_{j<=m} p_j(x_j^k) with the
    verifier's posteriors; k* = argmax (lowest k on ties); then greedy
    acceptance of x^{k*} against the argmax of its own verifier rows, reusing
    the cached verifier rows and ignoring draft probabilities.
    Returns (scores [K], k*, accepted a, bonus).
    """
    vlog = np.asarray(vlog)
    drafts = np.asarray(drafts)
    K, G = drafts.shape
    scores = np.empty(K, dtype=F64)
    for k in range(K):
        p = [np.exp(log_softmax_at(vlog[k, j], int(drafts[k, j]))) for j in range(G)]
        scores[k] = streak_score(p)
    ks = int(np.argmax(scores))
    targets = [int(np.argmax(np.asarray(vlog[ks, j], dtype=F64))) for j in range(G + 1)]
    a, bonus = greedy_accept(drafts[ks], targets)
    return scores, ks, a, bonus


def tv_acceptance(P, Q) -> float:
    """alpha = 1 - 1/2 sum_x |P(x) - Q(x)| (TV acceptance proxy)."""
    P = np.asarray(P, dtype=F64)
    Q = np.asarray(Q, dtype=F64)
    return 1.0 - 0.5 * np.sum(np.abs(P - Q))


# ---------------------------------------------------------------------------
# TV acceptance diagnostic and lossless stochastic acceptance (SpecDiff-2
# notes, "Streak-Distillation"; DFlare post, "Generating candidates in
# parallel, the target decides acceptance")
# ---------------------------------------------------------------------------

def softmax_t(z, T: float = 1.0) -> np.ndarray:
    """softmax(z / T) in fp64."""
    z = np.asarray(z, dtype=F64) / T
    e = np.exp(z - z.max())
    return e / e.sum()


def tv_alpha(z_row, T: float, v_row) -> float:
    """Per-position acceptance proxy alpha = 1 - TV(P, Q).

    Q = softmax(z / T) is the drafter's marginal at the position (the
    distribution the draft token is drawn from), P = softmax(v) the
    verifier's distribution there; alpha = 1 - 1/2 sum_x |P(x) - Q(x)|
    (SpecDiff-2 notes, "Streak-Distillation": the acceptance proxy).
    """
    return tv_acceptance(softmax_t(v_row), softmax_t(z_row, T))


def draw_uniform_stream(seed: int, n: int, j: int, k: int, stream: int) -> float:
    """u from Philox counter (n, j, k, stream): stream 0 draws the drafts,
    1 the acceptance tests, 2 the residual / bonus samples."""
    x0 = philox4x32_10((n, j, k, stream), (seed & _MASK32, (seed >> 32) & _MASK32))[0]
    return ((x0 >> 8) + 0.5) * 2.0 ** -24


def inverse_cdf(w, u: float):
    """Smallest index whose cumulative weight exceeds u * total (weights >= 0),
    and the distance of u * total to the nearest boundary / total."""
    w = np.asarray(w, dtype=F64)
    cdf = np.cumsum(w)
    total = cdf[-1]
    t = u * total
    v = min(int(np.searchsorted(cdf, t, side="right")), len(w) - 1)
    lo = cdf[v - 1] if v > 0 else 0.0
    return v, min(abs(t - lo), abs(cdf[v] - t)) / total


def speculative_accept(z_rows, T: float, v_rows, x, u_acc, u_res):
    """Lossless stochastic acceptance of one draft x_1..x_G.

    Position j (1-based) is accepted with probability min(1, P_j(x_j) /
    Q_j(x_j)), i.e. when u_acc[j] * Q_j(x_j) < P_j(x_j), with Q_j =
    softmax(z_j / T) the drafter's marginal and P_j = softmax(v_j) the
    verifier's.  At the first rejection the next token is drawn from the
    residual max(0, P_j - Q_j) (normalised) with u_res[j]; if all G are
    accepted the bonus token is drawn from P_{G+1} with u_res[G].  This keeps
    the verifier's distribution (the DFlare post's "proper acceptance
    procedure" for stochastic decoding).  Returns (accepted, token, margin):
    margin is the smallest relative distance to its boundary over every test
    made (accepted ones included: any of them could flip the result) and the
    final draw, i.e. how close floating point came to changing the result.
    """
    G = len(x)
    near = np.inf
    for j in range(G):
        Q = softmax_t(z_rows[j], T)
        P = softmax_t(v_rows[j])
        q, p = Q[x[j]], P[x[j]]
        near = min(near, abs(u_acc[j] * q - p) / max(p, 1e-300))
        if u_acc[j] * q < p:
            continue
        r = np.maximum(P - Q, 0.0)
        y, m = inverse_cdf(r, u_res[j])
        return j, y, min(near, m)
    y, m = inverse_cdf(softmax_t(v_rows[G]), u_res[G])
    return G, y, min(near, m)


# ---------------------------------------------------------------------------
# Sets of legitimate results where floating point may decide a draw or a test
# (used by the parity tests; the decisions themselves are the functions above)
# ---------------------------------------------------------------------------

def _nearest_nonempty(w, i: int, step: int):
    """First index from i in direction ``step`` whose weight is positive."""
    while 0 <= i < len(w):
        if w[i] > 0.0:
            return i
        i += step
    return None


def inverse_cdf_outcomes(w, u: float, band: float) -> set:
    """Every index an inverse-CDF draw of weights w at u may legitimately give.

    The draw is the smallest index whose cumulative weight exceeds u * total
    (``inverse_cdf``).  An implementation whose cumulative sums differ from
    the exact ones by less than ``band`` * total can only move a target that
    lies within that distance of a boundary into the interval on the other
    side of it: the set holds the exact index and, for each boundary closer
    than ``band`` * total, the nearest index with positive weight on the far
    side of that boundary.
    """
    w = np.asarray(w, dtype=F64)
    cdf = np.cumsum(w)
    total = cdf[-1]
    t = u * total
    v = min(int(np.searchsorted(cdf, t, side="right")), len(w) - 1)
    out = {v}
    lo = cdf[v - 1] if v > 0 else 0.0
    if v > 0 and t - lo < band * total:
        j = _nearest_nonempty(w, v - 1, -1)
        if j is not None:
            out.add(j)
    if cdf[v] - t < band * total:
        j = _nearest_nonempty(w, v + 1, +1)
        if j is not None:
            out.add(j)
    return out


def sample_inverse_cdf_outcomes(z, T: float, u: float, band: float) -> set:
    """``inverse_cdf_outcomes`` of the weights exp((z - max z) / T) that
    ``sample_inverse_cdf`` draws from."""
    z = np.asarray(z, dtype=F64)
    return inverse_cdf_outcomes(np.exp((z - z.max()) / T), u, band)


def speculative_accept_outcomes(z_rows, T: float, v_rows, x, u_acc, u_res,
                                band_test: float, band_draw: float) -> set:
    """Every (accepted, token) that ``speculative_accept`` may legitimately give.

    Follows the same rule position by position.  A test u * Q(x_j) < P(x_j)
    whose two sides differ by less than ``band_test`` * P(x_j) may go either
    way, so both branches are followed; each final draw contributes its
    ``inverse_cdf_outcomes`` with ``band_draw``.
    """
    G = len(x)
    out = set()

    def walk(j):
        if j == G:
            for y in inverse_cdf_outcomes(softmax_t(v_rows[G]), u_res[G], band_draw):
                out.add((G, y))
            return
        Q = softmax_t(z_rows[j], T)
        P = softmax_t(v_rows[j])
        q, p = Q[x[j]], P[x[j]]
        accept = u_acc[j] * q < p
        ambiguous = abs(u_acc[j] * q - p) < band_test * max(p, 1e-300)
        if accept or ambiguous:
            walk(j + 1)
        if not accept or ambiguous:
            r = np.maximum(P - Q, 0.0)
            if r.sum() > 0.0:
                for y in inverse_cdf_outcomes(r, u_res[j], band_draw):
                    out.add((j, y))

    walk(0)
    return out


# ---------------------------------------------------------------------------
# Sampled-greedy acceptance (SpecDiff-2 notes, "Streak-Distillation",
# "Self-Selection Acceptance")
# ---------------------------------------------------------------------------

def sampled_greedy_accept(v_rows, x, u):
    """Greedy acceptance against verifier samples instead of its argmax.

    Reading of the SpecDiff-2 notes' greedy-acceptance rule at temperature
    above zero: at window position j the verifier draws its own token y_j
    from P_j = softmax(v_j) (inverse CDF at u[j]), and the draft token x_j is
    accepted while it equals y_j.  At the first mismatch the verifier's own
    sample y_j is the committed token; when all G drafts are accepted the
    bonus is the sample y_G of row G.  Draft probabilities play no part (the
    section's point that the rule needs no drafter calibration), every
    committed token is a verifier sample (lossless), and the expected number
    accepted is sum_m prod_{j<=m} P_j(x_j), the streak equation of
    "Streak-Distillation".  v_rows [G+1][V], x [G], u [G+1].
    Returns (accepted, token, margin), margin being the smallest relative
    distance of any draw made to a CDF boundary.
    """
    G = len(x)
    near = np.inf
    for j in range(G + 1):
        y, m = inverse_cdf(softmax_t(v_rows[j]), u[j])
        near = min(near, m)
        if j == G or y != int(x[j]):
            return j, y, near
    raise AssertionError("unreachable")


def sampled_greedy_outcomes(v_rows, x, u, band: float) -> set:
    """Every (accepted, token) that ``sampled_greedy_accept`` may legitimately
    give when each draw may move across a boundary closer than ``band``."""
    G = len(x)
    out = set()

    def walk(j):
        ys = inverse_cdf_outcomes(softmax_t(v_rows[j]), u[j], band)
        for y in ys:
            if j < G and y == int(x[j]):
                walk(j + 1)
            else:
                out.add((j, y))

    walk(0)
    return out
