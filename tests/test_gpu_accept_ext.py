"""TV acceptance diagnostic and lossless stochastic acceptance vs the oracle (GPU)."""
import numpy as np
import pytest
import torch

import block_diffusion_speculative_dfl_gb300 as dfl
import oracle as orc
from gpu_util import SAMPLE_BAND, host, near_tie_cap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    dfl.build()
    dfl.load()
    torch.cuda.set_device(0)
    yield
    assert dfl.dfl_get_device_error() == 0


def _case(seed, N, K, G, V, T, closeness):
    """Drafter rows z and verifier rows near z/T (so acceptance is non-trivial)."""
    rng = np.random.default_rng(seed)
    z = (rng.standard_normal((N * G, V)) * 2.0).astype(np.float32)
    zz = z.reshape(N, G, V)
    v = np.empty((N, K, G + 1, V), np.float32)
    for k in range(K):
        v[:, k, :G] = zz / T + closeness * rng.standard_normal((N, G, V))
        v[:, k, G] = rng.standard_normal((N, V)) * 2.0
    from dfl_synth import round_bf16
    return z, round_bf16(v)


@pytest.mark.parametrize("N,K,G,V", [(3, 4, 6, 1000), (2, 9, 5, 2048), (1, 1, 1, 96)])
def test_tv_acceptance(N, K, G, V):
    T = 1.5
    z, v = _case(N * 100 + K, N, K, G, V, T, closeness=0.7)
    alpha = torch.empty((N, K, G), dtype=torch.float32, device="cuda")
    tpd = torch.empty((N, K), dtype=torch.float32, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_TV_ACCEPTANCE, N=N, K=K, G=G)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    zt = torch.from_numpy(z).cuda()
    vt = torch.from_numpy(v).cuda().to(torch.bfloat16)
    dfl.dfl_tv_acceptance(zt, T, vt, dfl.DFL_BF16, N, K, G, V, alpha, tpd, ws, wsb)
    a = host(alpha)
    zz = z.reshape(N, G, V)
    ref = np.array([[[orc.tv_alpha(zz[n, j], T, v[n, k, j]) for j in range(G)] for k in range(K)]
                    for n in range(N)])
    # fp32 sums of V terms of size <= 1 with expf errors of ~1e-7 relative
    assert np.max(np.abs(a - ref)) <= 2e-5, np.max(np.abs(a - ref))
    assert 0.05 < ref.mean() < 0.95     # a non-degenerate case
    tref = np.array([[orc.streak_score(ref[n, k]) for k in range(K)] for n in range(N)])
    assert np.allclose(host(tpd), tref, rtol=1e-4, atol=1e-5)


# Near-tie band of the stochastic rules: a test u*Q < P or a CDF draw whose
# two sides differ by less than this (relative) may legitimately go either way
# (fp32 probabilities on the GPU, fp64 in the oracle).
SPEC_BAND = 1e-5


def _spec_near_expectation(zz, v, T, x):
    """Upper bound on the chance that one sequence's acceptance meets a near
    tie: every test's band probability plus every possible draw's."""
    G = len(x)
    e = 0.0
    for j in range(G):
        Q, P = orc.softmax_t(zz[j], T), orc.softmax_t(v[j])
        e += min(1.0, 2 * SPEC_BAND * P[x[j]] / max(Q[x[j]], 1e-300))
        r = np.maximum(P - Q, 0.0)
        if r.sum() > 0:
            e += float(np.minimum(r / r.sum(), 2 * SPEC_BAND).sum())
    e += float(np.minimum(orc.softmax_t(v[G]), 2 * SPEC_BAND).sum())
    return e


@pytest.mark.parametrize("closeness", [0.05, 0.6, 3.0])
def test_spec_accept_matches_oracle(closeness):
    N, K, G, V, T, seed = 24, 3, 7, 1500, 1.3, 0x1234ABCD
    z, v = _case(int(closeness * 100), N, K, G, V, T, closeness)
    rng = np.random.default_rng(5)
    zz = z.reshape(N, G, V)
    # drafts drawn from the drafter's marginals, as the sampler would
    drafts = np.empty((N, K, G), np.int32)
    for n in range(N):
        for k in range(K):
            for j in range(G):
                drafts[n, k, j] = rng.choice(V, p=orc.softmax_t(zz[n, j], T))
    sel = rng.integers(0, K, N).astype(np.int32)
    al = torch.empty(N, dtype=torch.int32, device="cuda")
    nt = torch.empty(N, dtype=torch.int32, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_SPEC_ACCEPT, N=N, G=G, V=V)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    dfl.dfl_spec_accept(torch.from_numpy(z).cuda(), T, torch.from_numpy(v).cuda().to(torch.bfloat16), dfl.DFL_BF16,
                        torch.from_numpy(drafts).cuda(), torch.from_numpy(sel).cuda(), N, K, G, V, seed, al, nt, ws,
                        wsb)
    a_g, t_g = host(al), host(nt)
    near, expected = 0, 0.0
    for n in range(N):
        k = sel[n]
        u_acc = [orc.draw_uniform_stream(seed, n, j, 0, 1) for j in range(G)]
        u_res = [orc.draw_uniform_stream(seed, n, j, 0, 2) for j in range(G + 1)]
        legit = orc.speculative_accept_outcomes(zz[n], T, v[n, k], drafts[n, k], u_acc, u_res, SPEC_BAND, SPEC_BAND)
        assert (int(a_g[n]), int(t_g[n])) in legit, (n, a_g[n], t_g[n], legit)
        near += len(legit) > 1
        expected += _spec_near_expectation(zz[n], v[n, k], T, drafts[n, k])
    assert near <= near_tie_cap(expected), (near, expected)
    assert 0 <= a_g.min() and a_g.max() <= G


def _verifier_case(seed, N, K, G, V, dtype):
    """Verifier rows of mixed sharpness, drafts that copy the oracle's own
    verifier samples for a random prefix and then differ (so that accepted
    lengths spread over 0..G)."""
    rng = np.random.default_rng(seed)
    scale = rng.choice([1.0, 4.0, 12.0], size=(N, K, G + 1, 1))
    v = (rng.standard_normal((N, K, G + 1, V)) * scale).astype(np.float32)
    if dtype == dfl.DFL_BF16:
        from dfl_synth import round_bf16
        v = round_bf16(v)
    return rng, v


@pytest.mark.parametrize("N,K,G,V,dt", [(16, 3, 7, 1000, dfl.DFL_BF16), (4, 2, 32, 151936, dfl.DFL_BF16),
                                        (3, 1, 1, 96, dfl.DFL_BF16), (5, 4, 9, 1001, dfl.DFL_BF16),
                                        (6, 2, 5, 777, dfl.DFL_F32)])
def test_sampled_greedy_accept_matches_oracle(N, K, G, V, dt):
    seed = 0x5A5A1234 + N
    rng, v = _verifier_case(N * 1000 + G, N, K, G, V, dt)
    sel = rng.integers(0, K, N).astype(np.int32)
    drafts = rng.integers(0, V, (N, K, G)).astype(np.int32)
    for n in range(N):
        k = sel[n]
        cut = int(rng.integers(0, G + 1))
        for j in range(cut):   # copy the verifier's own draw at j (its exact inverse-CDF outcome)
            drafts[n, k, j] = orc.inverse_cdf(orc.softmax_t(v[n, k, j]), orc.draw_uniform_stream(seed, n, j, 0, 3))[0]
    al = torch.empty(N, dtype=torch.int32, device="cuda")
    nt = torch.empty(N, dtype=torch.int32, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_SAMPLED_GREEDY, N=N, G=G, V=V)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    vt = torch.from_numpy(v).cuda()
    if dt == dfl.DFL_BF16:
        vt = vt.to(torch.bfloat16)
    dfl.dfl_sampled_greedy_accept(vt, dt, torch.from_numpy(drafts).cuda(), torch.from_numpy(sel).cuda(), N, K, G, V,
                                  seed, al, nt, ws, wsb)
    a_g, t_g = host(al), host(nt)
    near, expected = 0, 0.0
    for n in range(N):
        k = sel[n]
        u = [orc.draw_uniform_stream(seed, n, j, 0, 3) for j in range(G + 1)]
        legit = orc.sampled_greedy_outcomes(v[n, k], drafts[n, k], u, SAMPLE_BAND)
        assert (int(a_g[n]), int(t_g[n])) in legit, (n, a_g[n], t_g[n], legit)
        near += len(legit) > 1
        expected += sum(float(np.minimum(orc.softmax_t(v[n, k, j]), 2 * SAMPLE_BAND).sum()) for j in range(G + 1))
    assert near <= near_tie_cap(expected), (near, expected)
    if G > 1:
        assert len(set(a_g.tolist())) > 1   # accepted lengths spread (the planted prefixes)


def test_sampled_greedy_without_selection_verifies_draft_zero():
    N, K, G, V, seed = 5, 3, 4, 512, 99
    rng, v = _verifier_case(7, N, K, G, V, dfl.DFL_BF16)
    drafts = rng.integers(0, V, (N, K, G)).astype(np.int32)
    al = torch.empty(N, dtype=torch.int32, device="cuda")
    nt = torch.empty(N, dtype=torch.int32, device="cuda")
    wsb = dfl.workspace_size(dfl.DFL_OP_SAMPLED_GREEDY, N=N, G=G, V=V)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    dfl.dfl_sampled_greedy_accept(torch.from_numpy(v).cuda().to(torch.bfloat16), dfl.DFL_BF16,
                                  torch.from_numpy(drafts).cuda(), None, N, K, G, V, seed, al, nt, ws, wsb)
    for n in range(N):
        u = [orc.draw_uniform_stream(seed, n, j, 0, 3) for j in range(G + 1)]
        legit = orc.sampled_greedy_outcomes(v[n, 0], drafts[n, 0], u, SAMPLE_BAND)
        assert (int(host(al)[n]), int(host(nt)[n])) in legit


def test_device_philox_matches_the_published_known_answers():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "philox_kat.txt")
    rows = []
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        c, k, x = (part.split() for part in line.split("|"))
        rows.append(([int(t, 16) for t in c + k], [int(t, 16) for t in x]))
    inp = torch.tensor(np.array([r[0] for r in rows], dtype=np.uint32).view(np.int32), device="cuda")
    out = torch.empty((len(rows), 4), dtype=torch.int32, device="cuda")
    dfl.dfl_philox4x32_10(inp, len(rows), out)
    got = host(out).view(np.uint32)
    assert np.array_equal(got, np.array([r[1] for r in rows], dtype=np.uint32))
    # and the uniforms of the sampling counters follow the oracle's generator
    seed = 0x0123456789ABCDEF
    ctr = [(n, j, k, s) for n in (0, 5) for j in (0, 31) for k in (0, 7) for s in range(4)]
    inp = torch.tensor(np.array([c + (seed & 0xFFFFFFFF, seed >> 32) for c in ctr], dtype=np.uint32).view(np.int32),
                       device="cuda")
    out = torch.empty((len(ctr), 4), dtype=torch.int32, device="cuda")
    dfl.dfl_philox4x32_10(inp, len(ctr), out)
    got = host(out).view(np.uint32)
    for i, c in enumerate(ctr):
        assert tuple(int(w) for w in got[i]) == orc.philox4x32_10(c, (seed & 0xFFFFFFFF, seed >> 32))
