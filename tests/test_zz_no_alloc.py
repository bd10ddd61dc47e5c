"""dfl_self_select_noalloc: self-selection for callers that cannot allocate.

Some callers cannot give the library a device workspace (an engine that owns
every byte of device memory through its own pool, a serving loop that must
not call cudaMalloc).  dfl_self_select_noalloc keeps its scratch in a fixed
array inside the library instead.  These tests call it through the C ABI and
compare it with dfl_self_select (caller workspace) on two calls in a row, the
second with different inputs, so stale contents of the shared array cannot
leak into a result.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_diffusion_speculative_dfl_gb300 as dfl


def test_noalloc_rejects_sizes_beyond_its_array():
    lib = dfl.load()
    # 16 * 64 * 65 = 66560 verifier rows > 65536: refused on the host, nothing launched
    rc = lib.dfl_self_select_noalloc(16, 1, 16, 16, 64, 64, 1000, 16, 16, 16, 16, None)
    assert rc == 4   # DFL_ERR_WORKSPACE


def _case(seed, N, K, G, V):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((N, K, G + 1, V)) * 4).astype(np.float32)
    vlog = torch.from_numpy(x).cuda().to(torch.bfloat16)
    vl = vlog.float().cpu().numpy()
    drafts = rng.integers(0, V, (N, K, G)).astype(np.int32)
    for n in range(N):           # some drafts follow the verifier for a while
        for k in range(K):
            p = rng.integers(0, G + 1)
            drafts[n, k, :p] = np.argmax(vl[n, k, :p], axis=-1)
    return vlog, torch.from_numpy(drafts).cuda()


def _outputs(N, K):
    return (torch.empty((N, K), dtype=torch.float32, device="cuda"),
            *(torch.full((N,), -1, dtype=torch.int32, device="cuda") for _ in range(3)))


@pytest.mark.gpu
def test_noalloc_matches_workspace_version_twice():
    dfl.build()
    dfl.load()
    torch.cuda.set_device(0)
    for call, (N, K, G, V) in enumerate([(4, 8, 32, 3000), (3, 5, 20, 1000)]):
        vlog, drafts = _case(100 + call, N, K, G, V)
        ref = _outputs(N, K)
        wsb = dfl.workspace_size(dfl.DFL_OP_SELF_SELECT, N=N, K=K, G=G)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        dfl.dfl_self_select(vlog, dfl.DFL_BF16, drafts, N, K, G, V, *ref, ws, wsb)
        got = _outputs(N, K)
        dfl.dfl_self_select_noalloc(vlog, dfl.DFL_BF16, drafts, N, K, G, V, *got)
        torch.cuda.synchronize()
        assert np.allclose(got[0].cpu().numpy(), ref[0].cpu().numpy(), rtol=1e-4, atol=0)
        for a, b in zip(got[1:], ref[1:]):
            assert np.array_equal(a.cpu().numpy(), b.cpu().numpy())
    assert dfl.dfl_get_device_error() == 0
