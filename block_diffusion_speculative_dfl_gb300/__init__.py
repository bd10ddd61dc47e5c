"""Block-diffusion speculative drafting on GB300 (sm_103a).

The compute path is libdfl.so (hand-written CUDA kernels behind a C ABI,
declared in include/dfl.h); this package only builds it, binds it with
ctypes and manages device buffers with torch.
"""
from ._build import build, LIB
from ._lib import (DflError, load, version, status_string, workspace_size, ptr, EXPORTED,
                   DFL_F32, DFL_BF16, DFL_OP_DUAL_KV_PROJ, DFL_OP_BLOCK_ATTN, DFL_OP_LM_HEAD,
                   DFL_OP_SELF_SELECT, DFL_OP_DRAFT_STEP,
                   dfl_rope_table, dfl_layer_mix_rmsnorm, dfl_dual_kv_proj, dfl_block_attn,
                   dfl_lm_head_argmax, dfl_greedy_accept, dfl_self_select, dfl_draft_step,
                   dfl_get_device_error, dfl_set_wait_limit_ns, dfl_selftest_bounded_wait,
                   dfl_profile_enable, dfl_profile_report, dfl_self_select_noalloc,
                   dfl_tv_acceptance, dfl_spec_accept, DFL_OP_TV_ACCEPTANCE, DFL_OP_SPEC_ACCEPT,
                   dfl_block_ffn, DFL_OP_BLOCK_FFN, dfl_draft_step_cached, DFL_OP_DRAFT_STEP_CACHED,
                   dfl_draft_step_host, DFL_OP_DRAFT_STEP_HOST, CtxCache, dfl_fc_fuse, DFL_OP_FC_FUSE,
                   dfl_sampled_greedy_accept, DFL_OP_SAMPLED_GREEDY, dfl_philox4x32_10)
from .step import DraftShape, DraftModel, CachedDraftModel

__all__ = [n for n in dir() if not n.startswith("_")]
