"""bench.py's accounting on CPU: the algorithmic work a launch is credited
with, which bound and which measured peak a kernel's roofline fraction uses,
and when a recorded DRAM traffic figure is reported.

The work figures are checked against values fixed outside bench.py: the
grouped projection of the Qwen3-8B drafter shape (the context K/V
projection of 32 x 2048 rows and the block Q/K/V projection of 32 x 16 rows
from d = 4096) is 2 * 65,536 * 4,096 * 2,048 + 2 * 512 * 4,096 * 6,144
flops = 1.1253 TFLOP, and the mix + RMSNorm reads L = 9 target layers and
writes D = 7 mixed layers of 65,536 rows x 4,096 bf16 values.
"""
import hashlib
import os

import pytest

import bench


def _qwen():
    return bench.workload("qwen3_8b_drafter")


def test_grouped_projection_work_of_the_qwen_drafter():
    flops, nbytes = bench.kernel_work(_qwen())["gemm_kv_qkv"]
    assert flops == pytest.approx(1.1253e12, rel=2e-4)
    # A (65,536 x 4,096), Wk and Wv (2 x 1,024 x 4,096), the context K and V
    # out (65,536 x 2,048); the block rows in (512 x 4,096), Wq, Wkb, Wvb
    # (6,144 x 4,096) and Q/Kb/Vb out (512 x 6,144); all bf16
    ctx = 65536 * 4096 + 2048 * 4096 + 65536 * 2048
    blk = 512 * 4096 + 6144 * 4096 + 512 * 6144
    assert nbytes == 2 * (ctx + blk)


def test_mix_and_attention_bytes_of_the_qwen_drafter():
    work = bench.kernel_work(_qwen())
    assert work["mix_rmsnorm_bf16"][1] == 2 * (9 + 7) * 65536 * 4096
    # K and V of 2,048 context + 16 block keys per sequence and K/V head (8 x 128),
    # read once; Q in and O out (32 x 16 rows x 32 heads x 128)
    keys = 32 * (2048 + 16)
    assert work["attn_tc"][1] == 2 * (2 * keys * 8 * 128 + 2 * 512 * 4096)


def test_lm_head_work_counts_the_drafted_rows_only():
    w = _qwen()
    flops, nbytes = bench.kernel_work(w)["gemm_lm_head"]
    rows = 32 * 15   # the block's first row is the anchor, not a draft
    assert flops == 2 * rows * 151936 * 4096
    assert nbytes == 2 * (rows * 4096 + 151936 * 4096)   # greedy: no logits stored


@pytest.mark.parametrize("clk,key", [
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}, "bf16_tflops"),
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}, "bf16_tflops_sustained"),
    ({"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": []}, "bf16_tflops_sustained"),   # below 97% of max
    ({"sm_mhz": 2030.0, "sm_max_mhz": 2070.0, "reasons": []}, "bf16_tflops"),
    ({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}, "bf16_tflops"),
])
def test_tensor_peak_follows_the_sampled_clocks(clk, key):
    assert bench.tensor_peak_key(clk)[0] == key


def test_kernel_table_bound_achieved_and_fraction():
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0}
    # 2 TFLOP over 1 GB: tensor time 1 ms > memory time 0.167 ms -> tensor-bound
    # 1 GFLOP over 6 GB: memory time 1 ms > tensor time -> HBM-bound
    work = {"k_tensor": (2.0e12, 1.0e9), "k_hbm": (1.0e9, 6.0e9)}
    prof = {"k_tensor": (4, 8.0), "k_hbm": (2, 4.0), "k_other": (10, 1.0)}   # (launches, total ms)
    t = bench.kernel_table(prof, work, peaks, "bf16_tflops_sustained")
    assert list(t) == ["k_tensor", "k_hbm", "k_other"]                    # by total time
    assert t["k_tensor"]["bound"] == "tensor" and t["k_hbm"]["bound"] == "hbm"
    assert t["k_tensor"]["ms_per_launch"] == 2.0
    assert t["k_tensor"]["achieved"] == pytest.approx(1000.0)             # 2 TFLOP / 2 ms, TFLOP/s
    assert t["k_tensor"]["frac"] == pytest.approx(1000.0 / 1800.0, abs=1e-4)
    assert t["k_hbm"]["achieved"] == pytest.approx(3000.0)                # 6 GB / 2 ms, GB/s
    assert t["k_hbm"]["frac"] == pytest.approx(0.5)
    assert t["k_other"]["share"] == pytest.approx(1.0 / 13.0, abs=1e-4)
    assert "frac" not in t["k_other"]


def test_traffic_is_reported_only_for_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    csrc = tmp_path / "block_diffusion_speculative_dfl_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("kernel v1")
    (csrc / "common.cuh").write_text("helpers v1")
    digest = hashlib.sha256(b"kernel v1" + b"helpers v1").hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        "# header\nkern wl 123456 " + digest + "\nkern other_wl 7 " + digest + "\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"kern": ["k.cu", "common.cuh"]})
    assert bench.ncu_traffic("kern", "wl") == 123456.0
    assert bench.ncu_traffic("kern", "missing_wl") is None
    assert bench.ncu_traffic("unknown_kernel", "wl") is None
    (csrc / "common.cuh").write_text("helpers v2")   # a shared helper changed: the record is stale
    assert bench.ncu_traffic("kern", "wl") is None


def test_every_kernel_source_list_covers_the_shared_device_helpers():
    for kernel, files in bench.KERNEL_SOURCES.items():
        assert files[-1] == "common.cuh", kernel
        for f in files:
            assert os.path.exists(os.path.join(bench.ROOT, "block_diffusion_speculative_dfl_gb300", "csrc", f)), f
