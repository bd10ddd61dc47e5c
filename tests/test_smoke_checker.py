"""The smoke check's comparison with the oracle, exercised on the CPU.

smoke() runs on a GPU; here its checker is fed results made by the oracle
itself (which it must accept) and the same results with one planted mistake
(which it must refuse), so that a broken comparison cannot pass unnoticed.
"""
import numpy as np
import pytest

import __graft_entry__ as entry
import oracle as orc
from dfl_synth import WORKLOADS, Workload, bits_to_f32, plant_targets


def _oracle_results(w, inp):
    shp = {"Hq": w.Hq, "Hkv": w.Hkv, "hd": w.hd}
    W_lm = bits_to_f32(inp["W_lm_bits"]) if w.dtype == "bf16" else inp["W_lm"]
    Xb, z = [], []
    for n in range(w.N):
        ref = orc.draft_forward(inp["Xb0"][n], inp["H"][:, n * w.C:(n + 1) * w.C], inp["mix"], inp["g_mix"],
                                inp["g_blk"], inp["layers"], shp, w.eps, w.rope_theta)["Xb"]
        Xb.append(ref)
        z.append(orc.lm_head_logits(ref[1:], inp["g_fin"], w.eps, W_lm))
    logits = np.concatenate(z).astype(np.float32)
    draft = orc.argmax_lowest(logits.reshape(w.N, w.B - 1, w.V)).astype(np.int32)
    target = plant_targets(w, draft)
    acc = [orc.greedy_accept(draft[n], target[n]) for n in range(w.N)]
    return dict(Xb=np.stack(Xb).astype(np.float32), logits=logits, draft=draft, target=target,
                accept_len=np.array([a for a, _ in acc], np.int32), bonus=np.array([b for _, b in acc], np.int32))


@pytest.fixture(scope="module", params=["tiny_f32", "smoke_bf16"])
def case(request):
    w = WORKLOADS["tiny_f32"] if request.param == "tiny_f32" else Workload("smoke_bf16", **entry.SMOKE_BF16)
    inp = entry._smoke_inputs(w)
    return w, inp, _oracle_results(w, inp)


def test_checker_accepts_the_oracles_own_results(case):
    w, inp, res = case
    assert "worst Xb error" in entry._smoke_check(w, inp, res)


@pytest.mark.parametrize("mistake", ["Xb", "logits", "draft", "accept"])
def test_checker_refuses_a_planted_mistake(case, mistake):
    w, inp, res = case
    bad = {k: np.array(v, copy=True) for k, v in res.items()}
    if mistake == "Xb":
        bad["Xb"][0, 3] += 0.5 * np.sqrt(np.mean((res["Xb"][0] - inp["Xb0"][0]) ** 2)) + 1e-3
    elif mistake == "logits":
        bad["logits"][2] *= 1.2
    elif mistake == "draft":
        bad["draft"][0, 0] = (bad["draft"][0, 0] + 1) % w.V
    else:
        bad["accept_len"][0] += 1
    with pytest.raises(AssertionError):
        entry._smoke_check(w, inp, bad)
