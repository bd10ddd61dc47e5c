"""Device-resident drafter and one-call draft step over the C ABI.

``DraftModel`` owns the drafter's parameters on the GPU (torch tensors used as
device memory only), the rotary table, the workspace and the output buffers
for a fixed shape; ``step()`` runs the whole single-pass draft step through
``dfl_draft_step`` on the current stream.  All pointers stay fixed between
calls, so a step can be captured into a CUDA graph.  ``step_from_host()``
is the end-to-end form: pinned host inputs are copied in and the per-sequence
results copied back on the same stream.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import DFL_BF16, DFL_F32, LayerWeights, SampleParams, StepArgs


@dataclass(frozen=True)
class DraftShape:
    N: int
    d: int
    Hq: int
    Hkv: int
    hd: int
    D: int
    L: int
    B: int
    C: int
    V: int
    dtype: str = "bf16"
    K: int = 0
    T: float = 1.0
    seed: int = 0
    eps: float = 1e-6
    rope_theta: float = 1e6
    F: int = 0
    fc: int = 0      # 1: DFlash fusion (one FC over the L target layers) instead of per-layer mixtures

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def dt(self) -> int:
        return DFL_BF16 if self.dtype == "bf16" else DFL_F32


class DraftModel:
    """Drafter parameters, workspace and outputs for one shape on one device."""

    def __init__(self, shape: DraftShape, mix_logits, mix_gain, blk_gain, final_gain, layers, W_lm=None,
                 device="cuda", tv=False, accept_rule=0, accept_seed=0, ffn_gain=None, W_fc=None, fc_gain=None):
        s = self.shape = shape
        dev = torch.device(device)
        wd = shape.torch_dtype

        def dev_t(x, dtype):
            return torch.as_tensor(x).to(device=dev, dtype=dtype).contiguous()

        self.mix_logits = dev_t(mix_logits, torch.float32) if mix_logits is not None else None
        self.mix_gain = dev_t(mix_gain, torch.float32) if mix_gain is not None else None
        if s.fc and (W_fc is None or fc_gain is None):
            raise ValueError("a fused drafter (shape.fc) needs W_fc and fc_gain")
        self.W_fc = dev_t(W_fc, wd) if s.fc else None
        self.fc_gain = dev_t(fc_gain, torch.float32) if s.fc else None
        self.blk_gain = dev_t(blk_gain, torch.float32)
        self.final_gain = dev_t(final_gain, torch.float32)
        self.layers = [{k: dev_t(v, wd) for k, v in w.items()} for w in layers]
        self.W_lm = dev_t(W_lm, wd) if (W_lm is not None and s.V > 0) else None
        self.rope = torch.empty((s.C + s.B, s.hd // 2, 2), dtype=torch.float32, device=dev)
        _lib.dfl_rope_table(self.rope, s.C + s.B, s.hd, s.rope_theta)
        names = ("Wq", "Wkc", "Wvc", "Wkb", "Wvb", "Wo") + (("W1", "W3", "W2") if s.F > 0 else ())
        self._lw = (LayerWeights * s.D)(*[LayerWeights(*[_lib.ptr(w[k]) for k in names]) for w in self.layers])
        self.ffn_gain = dev_t(ffn_gain, torch.float32) if s.F > 0 else None
        self._sp = SampleParams(s.K, s.T, s.seed) if s.K > 0 else None
        self.ws_bytes = self._workspace_bytes()
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.Xb = torch.empty((s.N, s.B, s.d), dtype=torch.float32, device=dev)
        n = s.B - 1
        self.draft = torch.empty((s.N, n), dtype=torch.int32, device=dev) if s.V > 0 else None
        self.accept_len = torch.empty((s.N,), dtype=torch.int32, device=dev)
        self.bonus = torch.empty((s.N,), dtype=torch.int32, device=dev)
        self.samples = torch.empty((s.N, s.K, n), dtype=torch.int32, device=dev) if s.K > 0 else None
        self.scores = torch.empty((s.N, s.K), dtype=torch.float32, device=dev) if s.K > 0 else None
        self.selected = torch.empty((s.N,), dtype=torch.int32, device=dev) if s.K > 0 else None
        self.logits = None
        # optional epilogues after self-selection: TV acceptance proxy, stochastic acceptance rule
        self.tv_alpha = torch.empty((s.N, s.K, n), dtype=torch.float32, device=dev) if (tv and s.K > 0) else None
        self.tv_tokens = torch.empty((s.N, s.K), dtype=torch.float32, device=dev) if (tv and s.K > 0) else None
        self.accept_rule, self.accept_seed = int(accept_rule), int(accept_seed)

    def _workspace_bytes(self) -> int:
        s = self.shape
        return _lib.workspace_size(_lib.DFL_OP_DRAFT_STEP, N=s.N, C=s.C, B=s.B, d=s.d, Hq=s.Hq, Hkv=s.Hkv, hd=s.hd,
                                   D=s.D, L=s.L, V=s.V, K=s.K, G=s.B - 1, row0=1, dtype=s.dt, F=s.F, fc=s.fc)

    def want_logits(self, on: bool = True):
        """Keep the fp32 logits [N*(B-1)][V] of each step (needed to check argmax bit-exactly)."""
        s = self.shape
        self.logits = (torch.empty((s.N * (s.B - 1), s.V), dtype=torch.float32, device=self.Xb.device)
                       if on and s.V > 0 else None)

    def _h_rows(self) -> int:
        return self.shape.C

    def _args(self, H, Xb0, target, vlog) -> StepArgs:
        s = self.shape
        a = StepArgs()
        a.N, a.C, a.B, a.d, a.Hq, a.Hkv, a.hd, a.D, a.L, a.V = s.N, s.C, s.B, s.d, s.Hq, s.Hkv, s.hd, s.D, s.L, s.V
        a.dtype, a.eps = s.dt, s.eps
        a.H, a.h_layer_stride = _lib.ptr(H), s.N * self._h_rows() * s.d
        a.mix_logits, a.mix_gain, a.blk_gain = _lib.ptr(self.mix_logits), _lib.ptr(self.mix_gain), _lib.ptr(self.blk_gain)
        a.final_gain, a.rope = _lib.ptr(self.final_gain), _lib.ptr(self.rope)
        a.layers = C.cast(self._lw, C.POINTER(LayerWeights))
        a.W_lm, a.Xb0, a.Xb = _lib.ptr(self.W_lm), _lib.ptr(Xb0), _lib.ptr(self.Xb)
        a.draft, a.logits = _lib.ptr(self.draft), _lib.ptr(self.logits)
        a.target = _lib.ptr(target)
        a.accept_len, a.bonus = _lib.ptr(self.accept_len), _lib.ptr(self.bonus)
        a.F, a.ffn_gain = s.F, _lib.ptr(self.ffn_gain)
        a.W_fc, a.fc_gain = _lib.ptr(self.W_fc), _lib.ptr(self.fc_gain)
        if self._sp is not None:
            a.sample = C.pointer(self._sp)
            a.samples = _lib.ptr(self.samples)
            if vlog is not None:
                a.vlog, a.scores, a.selected = _lib.ptr(vlog), _lib.ptr(self.scores), _lib.ptr(self.selected)
                a.tv_alpha, a.tv_tokens = _lib.ptr(self.tv_alpha), _lib.ptr(self.tv_tokens)
                a.accept_rule, a.accept_seed = self.accept_rule, self.accept_seed
        return a

    def step(self, H, Xb0, target=None, vlog=None, stream=None):
        """One draft step on device-resident inputs (H [L][N*C][d], Xb0 [N][B][d] fp32)."""
        self._last_args = self._args(H, Xb0, target, vlog)
        _lib.dfl_draft_step(self._last_args, self.ws, self.ws_bytes, stream)

    def _step_host(self, H_host, H_dev, Xb0, target, vlog, chunks, stream):
        """``dfl_draft_step_host``: H from (pinned) host memory through ``H_dev``."""
        s = self.shape
        need = _lib.workspace_size(_lib.DFL_OP_DRAFT_STEP_HOST, N=s.N, C=s.C, B=s.B, d=s.d, Hq=s.Hq, Hkv=s.Hkv,
                                   hd=s.hd, D=s.D, L=s.L, V=s.V, K=s.K, G=s.B - 1, row0=1, dtype=s.dt, F=s.F,
                                   fc=s.fc)
        if need > self.ws_bytes:   # the context K/V of every layer is kept: a larger workspace
            self.ws = torch.empty(need, dtype=torch.uint8, device=self.Xb.device)
            self.ws_bytes = need
        self._last_args = self._args(H_host, Xb0, target, vlog)
        _lib.dfl_draft_step_host(self._last_args, H_dev, chunks, self.ws, self.ws_bytes, stream)

    def step_from_host(self, H_host, Xb0_host, target_host=None, vlog_host=None, dev_in=None, stream=None,
                       chunks=8):
        """End-to-end step: copy pinned host inputs in, run, copy results out.

        ``dev_in`` is a dict of preallocated device buffers with the inputs'
        shapes (allocated on first use).  Returns host tensors of the
        per-sequence results.  For a bf16 model with pinned ``H_host`` the
        hidden states go through ``dfl_draft_step_host``: copied in ``chunks``
        groups of sequences while the groups already in are mixed and
        projected (``chunks=0``: one copy, then the device step).
        """
        st = stream or torch.cuda.current_stream()
        if dev_in is None:
            dev_in = {}
        overlap = chunks > 0 and self.shape.dt == DFL_BF16 and H_host.is_pinned()
        ins = {"H": H_host, "Xb0": Xb0_host, "target": target_host, "vlog": vlog_host}
        with torch.cuda.stream(st):
            for k, h in ins.items():
                if h is None:
                    continue
                if k not in dev_in:
                    dev_in[k] = torch.empty(h.shape, dtype=h.dtype, device=self.Xb.device)
                if not (overlap and k == "H"):
                    dev_in[k].copy_(h, non_blocking=True)
            if overlap:
                self._step_host(H_host, dev_in["H"], dev_in["Xb0"], dev_in.get("target"), dev_in.get("vlog"),
                                chunks, st)
            else:
                self.step(dev_in["H"], dev_in["Xb0"], dev_in.get("target"), dev_in.get("vlog"), stream=st)
            out = {"accept_len": self.accept_len.to("cpu", non_blocking=True),
                   "bonus": self.bonus.to("cpu", non_blocking=True)}
            if self.draft is not None:
                out["draft"] = self.draft.to("cpu", non_blocking=True)
            if self.selected is not None and vlog_host is not None:
                out["selected"] = self.selected.to("cpu", non_blocking=True)
        st.synchronize()
        return out, dev_in


class CachedDraftModel(DraftModel):
    """Drafter with per-layer context K/V caches (``dfl_draft_step_cached``).

    ``shape.C`` is the cache capacity per sequence; a step brings up to ``R``
    (at most ``R_max``) new context rows per sequence in H [L][N*R][d], whose
    keys/values are appended to the caches at positions ``ctx_len[n]..``; the
    block attends to every cached position of its sequence.  ``ctx_len``
    lives on the device and, with ``advance``, moves forward inside the step.
    """

    def __init__(self, shape: DraftShape, R_max: int, *args, **kw):
        if shape.dtype != "bf16":
            raise ValueError("the cached draft step runs in bf16")
        self.R_max = self.R = int(R_max)
        super().__init__(shape, *args, **kw)
        s = self.shape
        dev = self.Xb.device
        self.K_cache = torch.zeros((s.D, s.N, s.C, s.Hkv, s.hd), dtype=torch.bfloat16, device=dev)
        self.V_cache = torch.zeros_like(self.K_cache)
        self.ctx_len = torch.zeros((s.N,), dtype=torch.int32, device=dev)

    def _workspace_bytes(self) -> int:
        s = self.shape
        return _lib.workspace_size(_lib.DFL_OP_DRAFT_STEP_CACHED, N=s.N, C=s.C, B=s.B, d=s.d, Hq=s.Hq, Hkv=s.Hkv,
                                   hd=s.hd, D=s.D, L=s.L, V=s.V, K=s.K, G=s.B - 1, row0=1, dtype=s.dt, F=s.F,
                                   R=self.R_max, fc=s.fc)

    def _h_rows(self) -> int:
        return self.R

    def reset(self, ctx_len=None):
        """Set the cached lengths (default: empty caches)."""
        if ctx_len is None:
            self.ctx_len.zero_()
        else:
            self.ctx_len.copy_(torch.as_tensor(ctx_len, dtype=torch.int32))

    def step(self, H_new, Xb0, n_new, target=None, vlog=None, R=None, advance=True, stream=None):
        """One cached draft step.

        H_new [L][N*R][d]: the new context rows of each sequence (rows past
        n_new[n] are ignored); n_new [N] device int32.
        """
        s = self.shape
        self.R = self.R_max if R is None else int(R)
        if not 1 <= self.R <= self.R_max:
            raise ValueError(f"R={self.R} outside 1..{self.R_max}")
        cache = _lib.CtxCache()
        cache.K, cache.V = _lib.ptr(self.K_cache), _lib.ptr(self.V_cache)
        cache.layer_stride = s.N * s.C * s.Hkv * s.hd
        cache.R = self.R
        cache.ctx_len = _lib.ptr(self.ctx_len)
        cache.n_new = _lib.ptr(n_new)
        cache.advance = 1 if advance else 0
        self._last_args, self._last_cache = self._args(H_new, Xb0, target, vlog), cache
        _lib.dfl_draft_step_cached(self._last_args, cache, self.ws, self.ws_bytes, stream)

    def step_from_host(self, H_host, Xb0_host, n_new_host, target_host=None, vlog_host=None, dev_in=None, R=None,
                       advance=True, stream=None):
        """End-to-end cached step: pinned host inputs (the new rows, block init, n_new) in, results out.

        The caches and lengths stay on the device between calls.
        """
        st = stream or torch.cuda.current_stream()
        if dev_in is None:
            dev_in = {}
        ins = {"H": H_host, "Xb0": Xb0_host, "n_new": n_new_host, "target": target_host, "vlog": vlog_host}
        with torch.cuda.stream(st):
            for k, h in ins.items():
                if h is None:
                    continue
                if k not in dev_in:
                    dev_in[k] = torch.empty(h.shape, dtype=h.dtype, device=self.Xb.device)
                dev_in[k].copy_(h, non_blocking=True)
            self.step(dev_in["H"], dev_in["Xb0"], dev_in["n_new"], dev_in.get("target"), dev_in.get("vlog"), R=R,
                      advance=advance, stream=st)
            out = {"accept_len": self.accept_len.to("cpu", non_blocking=True),
                   "bonus": self.bonus.to("cpu", non_blocking=True)}
            if self.draft is not None:
                out["draft"] = self.draft.to("cpu", non_blocking=True)
        st.synchronize()
        return out, dev_in
