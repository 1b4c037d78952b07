"""GB300-native chunked forward of Kimi Delta Attention (KDA).

The compute path is ``libkda.so``: hand-written CUDA kernels for sm_103a
(tcgen05 MMAs with TMEM accumulators, TMA-fed shared memory) behind the C ABI
in ``include/kda.h``.  This package is its thin Python binding; importing it
does not load the library (that happens on the first call).
"""
from .binding import (  # noqa: F401
    EXPORTS,
    Dims,
    FwdOpts,
    KdaError,
    bwd_dh,
    chain_states,
    chunk_table,
    exact_path_tiles,
    fwd,
    fwd_host,
    fwd_intra,
    fwd_noalloc,
    host_arena_size,
    fwd_scan,
    library_path,
    load_library,
    make_dims,
    new_workspace,
    selftest_wait_timeout,
    state_map,
    status,
    status_string,
    workspace_layout,
    workspace_size,
)
