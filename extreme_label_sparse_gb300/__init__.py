"""Group-shared fixed fan-in sparse output layer (HASTE) on GB300.

The compute lives in libsg.so (hand-written CUDA for sm_103a behind the C ABI
of include/sg.h); `sg` is its thin ctypes binding with the same entry-point
names.  `build()` compiles the library in-tree.
"""
from ._build import build, LIB as LIB_PATH  # noqa: F401
from .sg import (  # noqa: F401
    Layout, SGError, load,
    SG_OK, SG_ERR_INVALID, SG_ERR_UNSUPPORTED, SG_ERR_CUDA, SG_ERR_OOM,
    SG_ERR_TIMEOUT, SG_ERR_DATA, SG_ENGINE_AUTO, SG_ENGINE_SIMT, SG_ENGINE_TC, SG_ENGINE_FUSED,
    sg_device_status, sg_layout_build, sg_layout_export, sg_layout_set_engine, sg_layout_status,
    sg_pos_export, sg_fwd, sg_bce_grad, sg_fwd_bce, sg_bwd, sg_bwd_dW, sg_bwd_dh,
    sg_step, sg_step_sgd, sg_bce_grad_noalloc, sg_selftest_wait_timeout, sg_proj_fwd, sg_proj_bwd,
    sg_headtail_step, sg_step_plan, SG_PLAN_PER_PHASE, SG_PLAN_FUSED_FWDW, SG_PLAN_ONE_KERNEL,
    Grouping, sg_grouping_create, sg_grouping_status, sg_grouping_embed, sg_grouping_set_embeddings,
    sg_grouping_kmeans_init, sg_grouping_set_centroids, sg_grouping_kmeans_batch, sg_grouping_groups,
    sg_grouping_export, sg_rewire, sg_timing_start, sg_timing_stop, last_error, status_string, KIND_NAMES,
)
