"""split_kv_mla_gb300: split-KV absorbed-MLA decode over a paged fp8 KV cache,
hand-written for GB300 (sm_103a).

The compute lives in ``libmla.so`` (CUDA kernels behind a C ABI, declared in
``include/mla_decode.h``); :mod:`split_kv_mla_gb300.mla` is the ctypes binding
with the same entry-point names, and :mod:`split_kv_mla_gb300.inputs` draws the
seeded synthetic workloads.  :mod:`split_kv_mla_gb300.dcp` holds the host
plumbing of decode context parallelism (rank page tables, the exchange step).
"""
from .mla import (  # noqa: F401
    MlaError,
    mla_dcp_lse_merge_ranks,
    mla_decode,
    mla_decode_dcp,
    mla_decode_dcp_splits,
    mla_decode_noalloc,
    mla_decode_splits,
    mla_decode_plan,
    mla_plan_force_splits,
    mla_plan_t,
    mla_read_device_error,
    mla_sparse_decode,
    mla_sparse_decode_extra,
    mla_sparse_decode_extra_splits,
    mla_sparse_decode_splits,
    mla_sparse_decode_plan,
    mla_splitk_reduce,
    mla_wave_fill_splits,
    mla_workspace_partials,
    mla_workspace_reset,
    workspace,
)
