"""GB300-native context-parallel zigzag causal attention.

The ring of context-parallel ranks ("Sequence Parallelism IV: Megatron
Context Parallel and Load-Balanced Rings", sections 3-5) runs on one GPU with
every virtual rank's shard resident in HBM.  The compute lives in libcpattn
(C ABI, include/cpattn.h, CUDA kernels for sm_103a); this package is its thin
Python binding.  ``inputs`` holds the seeded synthetic workloads.
"""
from ._binding import (  # noqa: F401
    BF16, CONTIGUOUS, F32, GRAD_F32, ONEPASS, PATH_SIMT, PATH_TCGEN05, ZIGZAG, CpattnError,
    allgather_bwd, allgather_fwd, attention, attention_allgather_fwd_bwd, attention_docs,
    attention_docs_fwd_bwd, attention_fwd_bwd, device_status, doc_bounds, lib,
    hier_a2a, hier_fwd, hier_bwd, hier_workspace_bytes, attention_hier_fwd_bwd,
    lse_merge, padded_length, plan, ring_bwd, ring_bwd_docs, ring_bwd_noalloc,
    ring_bwd_workspace_bytes, ring_fwd, ring_fwd_census, ring_fwd_docs, ring_fwd_docs_census,
    ring_fwd_step, status_string, tile_counts, zigzag_permute, zigzag_permute_pad,
    zigzag_unpermute, zigzag_unpermute_pad, kv_allgather, ulysses_a2a, ulysses_fwd, ulysses_bwd,
    ulysses_workspace_bytes, attention_ulysses_fwd_bwd, attention_host,
    attention_host_workspace_bytes, attention_host_parts, attention_host_docs,
    attention_host_docs_workspace_bytes, wait_probe)
