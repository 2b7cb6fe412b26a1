"""libssa: Stratified Sparse Attention single-token decode on B300 (sm_103a).

The compute path is the CUDA library ``libssa.so`` (C ABI in include/ssa.h);
``ssa`` is its Python binding.  Functions keep the C names.
"""
from .ssa import (  # noqa: F401
    SsaError, ssa_shape, make_shape, shape_of, workspace, load_library, ssa_version,
    ssa_workspace_bytes, ssa_pack_summary, ssa_score, ssa_select, ssa_attend, ssa_decode,
    ssa_decode_host, ssa_get_device_status, ssa_query_plan, default_scale, EXPORTS, LIB_PATH,
    ssa_append, ssa_decode_append, ssa_select_capacity, ssa_select_strata, ssa_decode_strata,
    STRATA_SSA, STRATA_UNIFORM, STRATA_TOP_P, ssa_paged_kv, paged_shape, ssa_decode_paged,
    ssa_attend_early_stop, ssa_decode_early_stop,
)
