"""Row-wise normalization reduce for GB300 (sm_103a).

LayerNorm, RMSNorm, fused residual-add + RMSNorm, BatchNorm2d training
forward, inference forward, training backward and their synchronized
(multi-process) form, and row softmax, computed by the
hand-written CUDA kernels of libnrm.so (C ABI in include/nrm.h).  This
package is the thin Python binding over that library.
"""
from ._binding import (  # noqa: F401
    LIB_PATH, NRM_BF16, NRM_F16, NRM_F32, PLAN_AUTO, PLAN_CTA, PLAN_GENERIC, PLAN_NAMES,
    PLAN_CLUSTER, PLAN_PERSIST, PLAN_TMA, PLAN_WRAW, PLAN_WARP, NrmError, add_rms_fwd, bn_bwd,
    bn_bwd_workspace_size, bn_fwd_infer, bn_fwd_train, bn_fwd_train_noalloc,
    bn_fwd_train_workspace_size, device_fault, force_plan, last_plan, lib, ln_fwd, rms_fwd,
    set_bn_group_bytes, set_pointer_checks, set_wait_limit, softmax_fwd, status_string,
    bn_fwd_partial_stats, bn_fwd_apply_stats, bn_bwd_partial_sums, bn_bwd_apply_sums,
    add_rms_fwd_host, add_rms_fwd_host_workspace)
from .sync import exchange_parts, global_count, sync_bn_bwd, sync_bn_fwd_train  # noqa: F401


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libnrm.so in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force, verbose=verbose)
