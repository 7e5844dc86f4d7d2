"""GB300-native (sm_103a) DDTree tree-verify MLA-absorb attention.

The compute path is libkdt.so (C ABI in include/kdt.h, CUDA kernels in csrc/);
this package holds the build script and a thin ctypes binding with the same names.
"""
from .kdt import (  # noqa: F401
    DEFAULT_SCALE, EXPORTS, IMPLS, KdtError, RopeArgs, VerifyArgs, build_visibility, host_buffer_size, kv_compact,
    lib, make_args, merge_attn_states, plan, rope_neox, status_str, tree_accept, tree_build, verify_attn,
    vc_up_proj, verify_attn_host, verify_attn_noalloc, workspace_size,
)

__version__ = "0.1.0"
