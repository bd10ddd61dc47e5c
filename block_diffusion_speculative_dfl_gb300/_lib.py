"""ctypes binding of libdfl.so: same names as the C ABI, argument marshalling only.

Tensors are passed as device pointers (``torch.Tensor.data_ptr()`` or plain
ints); a non-zero ``dfl_status`` raises :class:`DflError`.  There is no
fallback: if the library cannot be loaded every call raises.
"""
from __future__ import annotations

import ctypes as C
import os

from ._build import LIB, LIB_CHECK

DFL_OK, DFL_ERR_INVALID_ARG, DFL_ERR_UNSUPPORTED_SHAPE, DFL_ERR_MISALIGNED = 0, 1, 2, 3
DFL_ERR_WORKSPACE, DFL_ERR_CUDA, DFL_ERR_TIMEOUT, DFL_ERR_NO_DEVICE, DFL_ERR_BOUNDS = 4, 5, 6, 7, 8
DFL_F32, DFL_BF16 = 0, 1
DFL_OP_DUAL_KV_PROJ, DFL_OP_BLOCK_ATTN, DFL_OP_LM_HEAD, DFL_OP_SELF_SELECT, DFL_OP_DRAFT_STEP = 1, 2, 3, 4, 5
DFL_OP_TV_ACCEPTANCE, DFL_OP_SPEC_ACCEPT, DFL_OP_BLOCK_FFN, DFL_OP_DRAFT_STEP_CACHED = 6, 7, 8, 9
DFL_OP_DRAFT_STEP_HOST, DFL_OP_FC_FUSE, DFL_OP_SAMPLED_GREEDY = 10, 11, 12

# Every function the header declares; tests check each is exported.
EXPORTED = ("dfl_version", "dfl_status_string", "dfl_workspace_size", "dfl_rope_table",
            "dfl_layer_mix_rmsnorm", "dfl_dual_kv_proj", "dfl_block_attn", "dfl_lm_head_argmax",
            "dfl_greedy_accept", "dfl_self_select", "dfl_draft_step", "dfl_get_device_error",
            "dfl_set_wait_limit_ns", "dfl_selftest_bounded_wait", "dfl_profile_enable", "dfl_profile_report",
            "dfl_self_select_noalloc", "dfl_tv_acceptance", "dfl_spec_accept", "dfl_block_ffn",
            "dfl_draft_step_cached", "dfl_draft_step_host", "dfl_fc_fuse", "dfl_sampled_greedy_accept",
            "dfl_philox4x32_10")


class DflError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed: {msg} (status {code})")
        self.code = code


class SampleParams(C.Structure):
    _fields_ = [("K", C.c_int32), ("T", C.c_float), ("seed", C.c_uint64)]


class Shape(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("N", "C", "B", "d", "Hq", "Hkv", "hd", "D", "L", "V", "K", "G", "row0",
                                         "dtype", "F", "R", "fc")]


class LayerWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("Wq", "Wkc", "Wvc", "Wkb", "Wvb", "Wo", "W1", "W3", "W2")]


class StepArgs(C.Structure):
    _fields_ = ([(n, C.c_int32) for n in ("N", "C", "B", "d", "Hq", "Hkv", "hd", "D", "L", "V", "dtype")] +
                [("eps", C.c_float), ("H", C.c_void_p), ("h_layer_stride", C.c_int64)] +
                [(n, C.c_void_p) for n in ("mix_logits", "mix_gain", "blk_gain", "final_gain", "rope")] +
                [("layers", C.POINTER(LayerWeights))] +
                [(n, C.c_void_p) for n in ("W_lm", "Xb0", "Xb", "draft", "logits", "target", "accept_len",
                                           "bonus")] +
                [("sample", C.POINTER(SampleParams))] +
                [(n, C.c_void_p) for n in ("samples", "vlog", "scores", "selected", "tv_alpha", "tv_tokens")] +
                [("accept_rule", C.c_int32), ("accept_seed", C.c_uint64), ("F", C.c_int32), ("ffn_gain", C.c_void_p)] +
                [("W_fc", C.c_void_p), ("fc_gain", C.c_void_p)])


class CtxCache(C.Structure):
    _fields_ = [("K", C.c_void_p), ("V", C.c_void_p), ("layer_stride", C.c_int64), ("R", C.c_int32),
                ("ctx_len", C.c_void_p), ("n_new", C.c_void_p), ("advance", C.c_int32)]


_P, _I32, _I64, _F, _D, _SZ = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_double, C.c_size_t
_SIGS = {
    "dfl_version": ([], C.c_char_p),
    "dfl_status_string": ([_I32], C.c_char_p),
    "dfl_workspace_size": ([_I32, C.POINTER(Shape)], _SZ),
    "dfl_rope_table": ([_P, _I32, _I32, _D, _P], _I32),
    "dfl_layer_mix_rmsnorm": ([_P, _I64, _I32, _I64, _I32, _I32, _I32, _P, _P, _F, _P, _I64, _P], _I32),
    "dfl_dual_kv_proj": ([_P, _P, _I32, _I32, _I32, _I32, _I32, _P, _F, _P, _P, _P, _P, _P, _I32, _I32, _I32, _P,
                          _P, _P, _P, _P, _P, _P, _SZ, _P], _I32),
    "dfl_block_attn": ([_P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _I32, _I32, _I32, _P, _I32, _P, _P, _SZ, _P],
                       _I32),
    "dfl_lm_head_argmax": ([_P, _I32, _I32, _I32, _I32, _I32, _P, _F, _P, _I32, _P, _P, C.POINTER(SampleParams),
                            _P, _P, _SZ, _P], _I32),
    "dfl_greedy_accept": ([_P, _P, _I32, _I32, _P, _P, _P], _I32),
    "dfl_self_select": ([_P, _I32, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _SZ, _P], _I32),
    "dfl_draft_step": ([C.POINTER(StepArgs), _P, _SZ, _P], _I32),
    "dfl_draft_step_cached": ([C.POINTER(StepArgs), C.POINTER(CtxCache), _P, _SZ, _P], _I32),
    "dfl_draft_step_host": ([C.POINTER(StepArgs), _P, _I32, _P, _SZ, _P], _I32),
    "dfl_get_device_error": ([_P, C.POINTER(_I32)], _I32),
    "dfl_set_wait_limit_ns": ([C.c_uint64], _I32),
    "dfl_selftest_bounded_wait": ([C.c_uint64, _P, _P], _I32),
    "dfl_profile_enable": ([_I32], _I32),
    "dfl_profile_report": ([C.c_char_p, _SZ, C.POINTER(_I32)], _I32),
    "dfl_self_select_noalloc": ([_P, _I32, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P], _I32),
    "dfl_tv_acceptance": ([_P, _F, _P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _SZ, _P], _I32),
    "dfl_spec_accept": ([_P, _F, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, C.c_uint64, _P, _P, _P, _SZ, _P], _I32),
    "dfl_block_ffn": ([_P, _I32, _I32, _I32, _I32, _P, _F, _P, _P, _P, _I32, _P, _SZ, _P], _I32),
    "dfl_fc_fuse": ([_P, _I64, _I32, _I64, _I32, _I32, _P, _P, _F, _P, _P, _SZ, _P], _I32),
    "dfl_sampled_greedy_accept": ([_P, _I32, _P, _P, _I32, _I32, _I32, _I32, C.c_uint64, _P, _P, _P, _SZ, _P],
                                  _I32),
    "dfl_philox4x32_10": ([_P, _I32, _P, _P], _I32),
}

_lib = None


def load(path: str | None = None) -> C.CDLL:
    """Load libdfl.so (building it first if absent) and declare signatures.

    With DFL_CHECKED_BUILD=1 in the environment the bounds-checked variant
    (libdfl_check.so) is loaded instead."""
    global _lib
    if _lib is not None:
        return _lib
    checked = os.environ.get("DFL_CHECKED_BUILD") == "1"
    path = path or (LIB_CHECK if checked else LIB)
    if not os.path.exists(path):
        from ._build import build
        build(checked=checked)
    lib = C.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def ptr(x) -> int | None:
    """Device pointer of a tensor (or int / None passthrough)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name: str, code: int) -> None:
    if code != DFL_OK:
        msg = load().dfl_status_string(code).decode()
        raise DflError(name, code, msg)


def status_string(code: int) -> str:
    return load().dfl_status_string(code).decode()


def version() -> str:
    return load().dfl_version().decode()


def workspace_size(op: int, **shape) -> int:
    s = Shape(**{k: int(v) for k, v in shape.items()})
    return int(load().dfl_workspace_size(op, C.byref(s)))


def dfl_rope_table(table, P, hd, theta, stream=None):
    _check("dfl_rope_table", load().dfl_rope_table(ptr(table), P, hd, theta, _stream(stream)))


def dfl_layer_mix_rmsnorm(H, layer_stride, L, rows, d, dt, D, mix_logits, gain, eps, Xc, xc_layer_stride,
                          stream=None):
    _check("dfl_layer_mix_rmsnorm",
           load().dfl_layer_mix_rmsnorm(ptr(H), layer_stride, L, rows, d, dt, D, ptr(mix_logits), ptr(gain), eps,
                                        ptr(Xc), xc_layer_stride, _stream(stream)))


def dfl_dual_kv_proj(Xc, Xb, N, C_, B, d, dt, blk_gain, eps, Wq, Wkc, Wvc, Wkb, Wvb, Hq, Hkv, hd, rope, Q, Kc, Vc,
                     Kb, Vb, ws, ws_bytes, stream=None):
    _check("dfl_dual_kv_proj",
           load().dfl_dual_kv_proj(ptr(Xc), ptr(Xb), N, C_, B, d, dt, ptr(blk_gain), eps, ptr(Wq), ptr(Wkc),
                                   ptr(Wvc), ptr(Wkb), ptr(Wvb), Hq, Hkv, hd, ptr(rope), ptr(Q), ptr(Kc), ptr(Vc),
                                   ptr(Kb), ptr(Vb), ptr(ws), ws_bytes, _stream(stream)))


def dfl_block_attn(Q, Kc, Vc, Kb, Vb, N, C_, B, Hq, Hkv, hd, dt, Wo, d, Xb, ws, ws_bytes, stream=None):
    _check("dfl_block_attn",
           load().dfl_block_attn(ptr(Q), ptr(Kc), ptr(Vc), ptr(Kb), ptr(Vb), N, C_, B, Hq, Hkv, hd, dt, ptr(Wo), d,
                                 ptr(Xb), ptr(ws), ws_bytes, _stream(stream)))


def dfl_lm_head_argmax(Xb, N, B, row0, d, dt, final_gain, eps, W_lm, V, argmax_out, logits_out=None, sample=None,
                       samples_out=None, ws=None, ws_bytes=0, stream=None):
    sp = C.byref(SampleParams(*sample)) if sample is not None else None
    _check("dfl_lm_head_argmax",
           load().dfl_lm_head_argmax(ptr(Xb), N, B, row0, d, dt, ptr(final_gain), eps, ptr(W_lm), V,
                                     ptr(argmax_out), ptr(logits_out), sp, ptr(samples_out), ptr(ws), ws_bytes,
                                     _stream(stream)))


def dfl_greedy_accept(draft, target, N, n, accept_len, bonus, stream=None):
    _check("dfl_greedy_accept",
           load().dfl_greedy_accept(ptr(draft), ptr(target), N, n, ptr(accept_len), ptr(bonus), _stream(stream)))


def dfl_self_select(vlog, dt, drafts, N, K, G, V, scores, selected, accept_len, bonus, ws, ws_bytes, stream=None):
    _check("dfl_self_select",
           load().dfl_self_select(ptr(vlog), dt, ptr(drafts), N, K, G, V, ptr(scores), ptr(selected),
                                  ptr(accept_len), ptr(bonus), ptr(ws), ws_bytes, _stream(stream)))


def dfl_draft_step(args: StepArgs, ws, ws_bytes, stream=None):
    _check("dfl_draft_step", load().dfl_draft_step(C.byref(args), ptr(ws), ws_bytes, _stream(stream)))


def dfl_draft_step_host(args: StepArgs, H_dev, chunks, ws, ws_bytes, stream=None):
    _check("dfl_draft_step_host",
           load().dfl_draft_step_host(C.byref(args), ptr(H_dev), int(chunks), ptr(ws), ws_bytes, _stream(stream)))


def dfl_draft_step_cached(args: StepArgs, cache: CtxCache, ws, ws_bytes, stream=None):
    _check("dfl_draft_step_cached",
           load().dfl_draft_step_cached(C.byref(args), C.byref(cache), ptr(ws), ws_bytes, _stream(stream)))


def dfl_get_device_error(stream=None) -> int:
    code = _I32(0)
    _check("dfl_get_device_error", load().dfl_get_device_error(_stream(stream), C.byref(code)))
    return int(code.value)


def dfl_set_wait_limit_ns(ns: int):
    _check("dfl_set_wait_limit_ns", load().dfl_set_wait_limit_ns(ns))


def dfl_selftest_bounded_wait(limit_ns, status_out, stream=None):
    _check("dfl_selftest_bounded_wait",
           load().dfl_selftest_bounded_wait(limit_ns, ptr(status_out), _stream(stream)))


def dfl_profile_enable(on: bool = True):
    _check("dfl_profile_enable", load().dfl_profile_enable(1 if on else 0))


def dfl_profile_report() -> tuple[dict, int]:
    """Per-kernel {name: (launches, total_ms)} since tracing was enabled, and the launch count."""
    import json
    buf = C.create_string_buffer(1 << 16)
    n = _I32(0)
    _check("dfl_profile_report", load().dfl_profile_report(buf, len(buf), C.byref(n)))
    return {k: (int(v[0]), float(v[1])) for k, v in json.loads(buf.value.decode()).items()}, int(n.value)


def dfl_self_select_noalloc(vlog, dt, drafts, N, K, G, V, scores, selected, accept_len, bonus, stream=None):
    """dfl_self_select with the scratch in the library's fixed device array (no workspace argument)."""
    _check("dfl_self_select_noalloc",
           load().dfl_self_select_noalloc(ptr(vlog), dt, ptr(drafts), N, K, G, V, ptr(scores), ptr(selected),
                                          ptr(accept_len), ptr(bonus), _stream(stream)))


def dfl_tv_acceptance(logits, T, vlog, dt, N, K, G, V, alpha, tokens_per_draft, ws, ws_bytes, stream=None):
    _check("dfl_tv_acceptance",
           load().dfl_tv_acceptance(ptr(logits), T, ptr(vlog), dt, N, K, G, V, ptr(alpha), ptr(tokens_per_draft),
                                    ptr(ws), ws_bytes, _stream(stream)))


def dfl_spec_accept(logits, T, vlog, dt, drafts, sel, N, K, G, V, seed, accept_len, next_token, ws, ws_bytes,
                    stream=None):
    _check("dfl_spec_accept",
           load().dfl_spec_accept(ptr(logits), T, ptr(vlog), dt, ptr(drafts), ptr(sel), N, K, G, V, seed,
                                  ptr(accept_len), ptr(next_token), ptr(ws), ws_bytes, _stream(stream)))


def dfl_block_ffn(Xb, N, B, d, dt, ffn_gain, eps, W1, W3, W2, F, ws, ws_bytes, stream=None):
    _check("dfl_block_ffn",
           load().dfl_block_ffn(ptr(Xb), N, B, d, dt, ptr(ffn_gain), eps, ptr(W1), ptr(W3), ptr(W2), F, ptr(ws),
                                ws_bytes, _stream(stream)))


def dfl_fc_fuse(H, layer_stride, L, rows, d, dt, W_fc, gain, eps, Xc, ws, ws_bytes, stream=None):
    _check("dfl_fc_fuse",
           load().dfl_fc_fuse(ptr(H), layer_stride, L, rows, d, dt, ptr(W_fc), ptr(gain), eps, ptr(Xc), ptr(ws),
                              ws_bytes, _stream(stream)))


def dfl_sampled_greedy_accept(vlog, dt, drafts, sel, N, K, G, V, seed, accept_len, next_token, ws, ws_bytes,
                              stream=None):
    _check("dfl_sampled_greedy_accept",
           load().dfl_sampled_greedy_accept(ptr(vlog), dt, ptr(drafts), ptr(sel), N, K, G, V, seed, ptr(accept_len),
                                            ptr(next_token), ptr(ws), ws_bytes, _stream(stream)))


def dfl_philox4x32_10(inp, n, out, stream=None):
    _check("dfl_philox4x32_10", load().dfl_philox4x32_10(ptr(inp), n, ptr(out), _stream(stream)))
