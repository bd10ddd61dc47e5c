"""The C-ABI library builds, loads and exports every function include/dfl.h declares.

No compute call is made here: these run without a GPU.
"""
import ctypes
import os
import re

import pytest

import block_diffusion_speculative_dfl_gb300 as dfl

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "dfl.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dfl_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_six_path_calls():
    names = _declared()
    for n in ("dfl_layer_mix_rmsnorm", "dfl_dual_kv_proj", "dfl_block_attn", "dfl_lm_head_argmax",
              "dfl_greedy_accept", "dfl_self_select"):
        assert n in names


def test_library_exports_every_declared_symbol():
    dfl.build()
    lib = ctypes.CDLL(dfl.LIB)
    names = _declared()
    assert names, "no declarations parsed"
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(dfl.EXPORTED) == names


def test_host_only_calls_work_without_a_gpu():
    lib = dfl.load()
    assert dfl.version().startswith("dfl")
    assert dfl.status_string(0) == "ok"
    assert "workspace" in dfl.status_string(4)
    # workspace sizes are pure host arithmetic
    ws = dfl.workspace_size(dfl.DFL_OP_LM_HEAD, N=2, B=16, row0=1, d=256, V=1000, dtype=dfl.DFL_BF16)
    assert ws >= 2 * 15 * 256 * 2
    assert dfl.workspace_size(dfl.DFL_OP_LM_HEAD, N=2, B=16, row0=16, d=256, V=1000, dtype=1) == 0
    assert lib.dfl_set_wait_limit_ns(0) == 1   # invalid argument, checked on the host


def test_invalid_arguments_rejected_before_any_launch():
    # Host-side checks return a status without touching a device.
    lib = dfl.load()
    assert lib.dfl_greedy_accept(None, None, 1, 4, None, None, None) == 1
    assert lib.dfl_layer_mix_rmsnorm(None, 0, 9, 16, 64, 1, 7, None, None, 1e-6, None, 0, None) == 1
    sp = dfl._lib.SampleParams(0, 1.5, 1)
    assert lib.dfl_lm_head_argmax(16, 1, 16, 1, 64, 1, 16, 1e-6, 16, 100, 16, 16, ctypes.byref(sp), 16, 16,
                                  1 << 20, None) == 1   # K = 0 is invalid
    # misaligned pointer (not a multiple of 16) is refused on the host
    assert lib.dfl_self_select(8, 1, 16, 1, 2, 3, 100, 16, 16, 16, 16, 16, 1 << 20, None) == 3


@pytest.mark.parametrize("dt", [0, 1])
def test_step_workspace_grows_with_layers(dt):
    a = dfl.workspace_size(dfl.DFL_OP_DRAFT_STEP, N=1, C=64, B=16, d=256, Hq=4, Hkv=4, hd=64, D=1, L=3, V=1000,
                           K=0, G=15, row0=1, dtype=dt)
    b = dfl.workspace_size(dfl.DFL_OP_DRAFT_STEP, N=1, C=64, B=16, d=256, Hq=4, Hkv=4, hd=64, D=2, L=3, V=1000,
                           K=0, G=15, row0=1, dtype=dt)
    assert b - a >= 64 * 256 * (2 if dt else 4)


def _host_step_args(dtype=1):
    """A dfl_step_args whose device pointers are stand-in aligned addresses.

    Only the host-side checks read it; nothing is dereferenced on the device.
    """
    lib = dfl._lib
    fake = 1 << 20
    layers = (lib.LayerWeights * 2)()
    for w in layers:
        for n, _ in lib.LayerWeights._fields_[:6]:
            setattr(w, n, fake)
    a = lib.StepArgs()
    a.N, a.C, a.B, a.d, a.Hq, a.Hkv, a.hd, a.D, a.L, a.V, a.dtype = 2, 64, 16, 256, 4, 2, 64, 2, 3, 1000, dtype
    a.eps, a.h_layer_stride = 1e-6, 2 * 64 * 256
    for n in ("H", "mix_logits", "mix_gain", "blk_gain", "final_gain", "W_lm", "Xb0", "Xb", "draft"):
        setattr(a, n, fake)
    a.layers = layers
    return a, layers


def test_host_input_step_rejects_bad_arguments_on_the_host():
    lib = dfl.load()
    shape = dict(N=2, C=64, B=16, d=256, Hq=4, Hkv=2, hd=64, D=2, L=3, V=1000, K=0, G=15, row0=1, dtype=1)
    need = dfl.workspace_size(dfl.DFL_OP_DRAFT_STEP_HOST, **shape)
    assert need > dfl.workspace_size(dfl.DFL_OP_DRAFT_STEP, **shape)   # plus the context K/V of the later layers
    fake = 1 << 20
    a, keep = _host_step_args()
    call = lambda args, H_dev=fake, chunks=2, ws=fake, nbytes=need: lib.dfl_draft_step_host(
        ctypes.byref(args), H_dev, chunks, ws, nbytes, None)
    assert call(a, H_dev=None) == 1                  # no device copy of H
    assert call(a, chunks=0) == 1                    # at least one group
    assert call(a, ws=None) == 1
    assert call(a, H_dev=fake + 8) == 3              # H_dev off the 16-byte rule
    assert call(a, nbytes=need - 1) == 4             # workspace one byte short
    b, keep_b = _host_step_args(dtype=0)
    assert call(b) == 2                              # fp32 has no host-input path
    a.h_layer_stride = 2 * 64 * 256 - 8
    assert call(a) == 1                              # layer slabs overlap
    a.h_layer_stride, a.hd = 2 * 64 * 256, 96
    assert call(a) == 2                              # head size without a kernel
    a.hd, a.Xb = 64, None
    assert call(a) == 1


def test_header_is_plain_c_and_links(tmp_path):
    # A C99 program (tests/c_abi_host_calls.c) built with -pedantic -Werror
    # against include/dfl.h and libdfl.so, run on the host.
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    dfl.build()
    root = os.path.dirname(os.path.dirname(__file__))
    libdir = os.path.dirname(dfl.LIB)
    exe = str(tmp_path / "host_calls")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(root, "include"),
                    os.path.join(root, "tests", "c_abi_host_calls.c"), "-L", libdir, "-ldfl",
                    "-Wl,-rpath," + libdir, "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr


_OPS = ["DFL_OP_DUAL_KV_PROJ", "DFL_OP_BLOCK_ATTN", "DFL_OP_LM_HEAD", "DFL_OP_SELF_SELECT", "DFL_OP_DRAFT_STEP",
        "DFL_OP_TV_ACCEPTANCE", "DFL_OP_SPEC_ACCEPT", "DFL_OP_BLOCK_FFN", "DFL_OP_DRAFT_STEP_CACHED",
        "DFL_OP_DRAFT_STEP_HOST", "DFL_OP_FC_FUSE", "DFL_OP_SAMPLED_GREEDY"]
_SHAPE = dict(N=3, C=96, B=16, d=256, Hq=4, Hkv=2, hd=128, D=2, L=3, V=1500, K=4, G=15, row0=1, dtype=1, F=384, R=8,
              fc=0)


@pytest.mark.parametrize("op", _OPS)
def test_workspace_size_is_zero_for_invalid_shapes(op):
    code = getattr(dfl._lib, op)
    ok = dfl.workspace_size(code, **_SHAPE)
    assert 0 < ok < 1 << 32
    assert dfl.workspace_size(code, **dict(_SHAPE, dtype=7)) == 0
    for k in _SHAPE:
        if k != "dtype":
            assert dfl.workspace_size(code, **dict(_SHAPE, **{k: -1})) == 0, k


@pytest.mark.parametrize("op", ["DFL_OP_DRAFT_STEP", "DFL_OP_DRAFT_STEP_CACHED", "DFL_OP_DRAFT_STEP_HOST"])
def test_step_workspace_grows_with_the_batch(op):
    code = getattr(dfl._lib, op)
    sizes = [dfl.workspace_size(code, **dict(_SHAPE, N=n)) for n in (1, 2, 4, 8)]
    assert all(a < b for a, b in zip(sizes, sizes[1:])), sizes


_FAKE = 1 << 20   # stand-in device address (16-byte aligned); never dereferenced here


def _no_device(lib):
    # The sweep below passes stand-in addresses: it runs only where the library
    # finds no usable device, so that a call that passes its host checks stops
    # at NO_DEVICE instead of launching.
    code = ctypes.c_int32(0)
    return lib.dfl_get_device_error(None, ctypes.byref(code)) == 7


def _entry_points():
    """(function, valid arguments, indices of the pointers that may not be NULL,
    indices of those read or written with 16-byte or TMA accesses)."""
    sz = lambda op, **k: dfl.workspace_size(op, **k)
    F = _FAKE
    s = dict(N=2, C=64, B=16, d=256, Hq=4, Hkv=2, hd=128, dtype=1)
    ws_kv = sz(dfl.DFL_OP_DUAL_KV_PROJ, **s)
    ws_at = sz(dfl.DFL_OP_BLOCK_ATTN, **s)
    ws_lm = sz(dfl.DFL_OP_LM_HEAD, N=2, B=16, row0=1, d=256, V=1000, dtype=1)
    ws_sel = sz(dfl.DFL_OP_SELF_SELECT, N=2, K=4, G=8, V=1000, dtype=1)
    ws_tv = sz(dfl.DFL_OP_TV_ACCEPTANCE, N=2, K=4, G=8, V=1000, dtype=1)
    ws_sp = sz(dfl.DFL_OP_SPEC_ACCEPT, N=2, K=4, G=8, V=1000, dtype=1)
    ws_ffn = sz(dfl.DFL_OP_BLOCK_FFN, N=2, B=16, d=256, F=384, dtype=1)
    ws_fc = sz(dfl.DFL_OP_FC_FUSE, N=1, C=64, d=256, dtype=1)
    ws_sg = sz(dfl.DFL_OP_SAMPLED_GREEDY, N=2, G=8, V=1000, dtype=1)
    return [
        ("dfl_rope_table", [F, 80, 128, 1e6, None], [0], []),
        ("dfl_layer_mix_rmsnorm", [F, 64 * 256, 3, 64, 256, 1, 2, F, F, 1e-6, F, 64 * 256, None], [0, 7, 8, 10], [0, 8, 10]),
        ("dfl_dual_kv_proj", [F, F, 2, 64, 16, 256, 1, F, 1e-6, F, F, F, F, F, 4, 2, 128, None,
                              F, F, F, F, F, F, ws_kv, None], [0, 1, 7, 9, 10, 11, 12, 13, 18, 19, 20, 21, 22, 23],
         [0, 1, 7, 9, 10, 11, 12, 13, 18, 19, 20, 21, 22, 23]),
        ("dfl_block_attn", [F, F, F, F, F, 2, 64, 16, 4, 2, 128, 1, F, 256, F, F, ws_at, None],
         [0, 1, 2, 3, 4, 12, 14, 15], [0, 1, 2, 3, 4, 12, 14, 15]),
        ("dfl_lm_head_argmax", [F, 2, 16, 1, 256, 1, F, 1e-6, F, 1000, F, None, None, None, F, ws_lm, None],
         [0, 6, 8, 10, 14], [0, 6, 8, 14]),
        ("dfl_greedy_accept", [F, F, 2, 15, F, F, None], [0, 1, 4, 5], []),
        ("dfl_self_select", [F, 1, F, 2, 4, 8, 1000, F, F, F, F, F, ws_sel, None], [0, 2, 7, 8, 9, 10, 11], [0, 11]),
        ("dfl_self_select_noalloc", [F, 1, F, 2, 4, 8, 1000, F, F, F, F, None], [0, 2, 7, 8, 9, 10], [0]),
        ("dfl_tv_acceptance", [F, 1.5, F, 1, 2, 4, 8, 1000, F, None, F, ws_tv, None], [0, 2, 8, 10], [0, 2, 10]),
        ("dfl_spec_accept", [F, 1.5, F, 1, F, None, 2, 4, 8, 1000, 7, F, F, F, ws_sp, None], [0, 2, 4, 11, 12, 13], [0, 2, 13]),
        ("dfl_block_ffn", [F, 2, 16, 256, 1, F, 1e-6, F, F, F, 384, F, ws_ffn, None], [0, 5, 7, 8, 9, 11], [0, 5, 7, 8, 9, 11]),
    ]


@pytest.mark.parametrize("name,args,required,vec", _entry_points(), ids=lambda v: v if isinstance(v, str) else "")
def test_every_required_pointer_is_checked_on_the_host(name, args, required, vec):
    lib = dfl.load()
    if not _no_device(lib):
        pytest.skip("a usable device is present: the sweep's stand-in addresses must not reach a launch")
    fn = getattr(lib, name)
    assert fn(*args) == 7, "valid arguments should pass every host check and stop at NO_DEVICE"
    for i in required:
        bad = list(args)
        bad[i] = None
        assert fn(*bad) == 1, f"{name}: NULL argument {i} not rejected on the host"
    for i in vec:   # 8 bytes off: vector loads and TMA copies would fault, so the host refuses it
        bad = list(args)
        bad[i] = args[i] + 8
        assert fn(*bad) == 3, f"{name}: misaligned argument {i} not rejected on the host"


def test_step_refuses_a_misaligned_pointer_before_any_launch():
    lib = dfl.load()
    if not _no_device(lib):
        pytest.skip("a usable device is present: the stand-in addresses must not reach a launch")
    a, layers = _host_step_args()
    need = dfl.workspace_size(dfl.DFL_OP_DRAFT_STEP, N=2, C=64, B=16, d=256, Hq=4, Hkv=2, hd=64, D=2, L=3, V=1000,
                              K=0, G=15, row0=1, dtype=1)
    step = lambda: lib.dfl_draft_step(ctypes.byref(a), _FAKE, need, None)
    assert step() == 7
    for name in ("H", "Xb", "mix_gain", "blk_gain", "final_gain", "W_lm"):
        setattr(a, name, _FAKE + 8)
        assert step() == 3, name
        setattr(a, name, _FAKE)
    for name in ("Wq", "Wkc", "Wvc", "Wkb", "Wvb", "Wo"):
        setattr(layers[1], name, _FAKE + 8)
        assert step() == 3, name
        setattr(layers[1], name, _FAKE)
    assert lib.dfl_draft_step(ctypes.byref(a), _FAKE + 8, need, None) == 3   # workspace
    assert step() == 7


@pytest.mark.parametrize("field,value,status", [("L", 17, 1), ("Hq", 3, 1), ("hd", 60, 3), ("d", 260, 3),
                                                ("h_layer_stride", 2 * 64 * 256 - 8, 1),
                                                ("h_layer_stride", 2 * 64 * 256 + 4, 3)])
def test_step_refuses_a_bad_shape_before_any_launch(field, value, status):
    lib = dfl.load()
    if not _no_device(lib):
        pytest.skip("a usable device is present: the stand-in addresses must not reach a launch")
    a, layers = _host_step_args()
    need = dfl.workspace_size(dfl.DFL_OP_DRAFT_STEP, N=2, C=64, B=16, d=260, Hq=4, Hkv=2, hd=64, D=2, L=17,
                              V=1000, K=0, G=15, row0=1, dtype=1)
    setattr(a, field, value)
    if field == "d":
        a.h_layer_stride = 2 * 64 * 264   # large enough, so that only d itself is wrong
    assert lib.dfl_draft_step(ctypes.byref(a), _FAKE, need, None) == status


def test_row_counts_beyond_32_bits_are_refused():
    # TMA coordinates and GEMM extents are 32-bit: N*C or N*B of 2^31 rows and
    # more is an unsupported shape, refused on the host.
    lib = dfl.load()
    if not _no_device(lib):
        pytest.skip("a usable device is present: the stand-in addresses must not reach a launch")
    F = _FAKE
    big_n, big_c = 1 << 20, 1 << 11
    assert lib.dfl_block_attn(F, F, F, F, F, big_n, big_c, 16, 4, 2, 128, 1, F, 256, F, F, 1 << 40, None) == 2
    assert lib.dfl_dual_kv_proj(F, F, big_n, big_c, 16, 256, 1, F, 1e-6, F, F, F, F, F, 4, 2, 128, None,
                                F, F, F, F, F, F, 1 << 40, None) == 2
    assert lib.dfl_block_ffn(F, 1 << 27, 16, 256, 1, F, 1e-6, F, F, F, 384, F, 1 << 40, None) == 2
    a, layers = _host_step_args()
    a.N, a.C, a.h_layer_stride = big_n, big_c, big_n * big_c * 256
    assert lib.dfl_draft_step(ctypes.byref(a), F, 1 << 50, None) == 2
