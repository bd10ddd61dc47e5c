"""TV acceptance diagnostic and lossless stochastic acceptance vs the oracle (GPU)."""
import numpy as np
import pytest
import torch

import block_diffusion_speculative_dfl_gb300 as dfl
import oracle as orc
from gpu_util import host

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
    exact = near = 0
    for n in range(N):
        k = sel[n]
        u_acc = [orc.draw_uniform_stream(seed, n, j, 0, 1) for j in range(G)]
        u_res = [orc.draw_uniform_stream(seed, n, j, 0, 2) for j in range(G + 1)]
        a, y, margin = orc.speculative_accept(zz[n], T, v[n, k], drafts[n, k], u_acc, u_res)
        if margin >= 1e-5:
            assert (a_g[n], t_g[n]) == (a, y), (n, a_g[n], t_g[n], a, y, margin)
            exact += 1
        else:
            near += 1
    assert exact >= 0.8 * N
    assert 0 <= a_g.min() and a_g.max() <= G
