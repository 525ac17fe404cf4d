"""Chunked gated delta rule forward for GB300 (sm_103a).

The compute lives in libgdr.so (CUDA, C ABI declared in include/gdr.h); this
package is its Python binding.  Importing it does not load the library; the
first call does, and raises if the library has not been built.
"""
from .api import (  # noqa: F401
    bwd_workspace_bytes,
    check_cu_seqlens,
    checkpoint_count_bound,
    chunk_count_bound,
    chunk_bwd,
    chunk_fwd,
    chunk_gated_delta_rule,
    chunk_fwd_alloc,
    chunk_fwd_checkpoints,
    chunk_index,
    chunk_out,
    chunk_prep,
    clear_device_status,
    device_status,
    split_pieces,
    split_plan,
    stage_workspace_bytes,
    state_scan,
    wait_selftest,
    workspace_bytes,
)
from ._native import GdrError  # noqa: F401

__version__ = "0.1.0"
