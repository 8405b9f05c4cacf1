"""GB300 (sm_103a) sparse-attention decode/prefill chain: lightweight indexer -> Top-K ->
gather-driven sparse attention over a latent KV cache.

The compute lives in libdsa.so (C ABI in include/dsa.h); this package is its thin Python binding.
Importing it fails loudly when the library is not built.
"""
from .api import (DsaCall, dsa_decode, dsa_get_device_error, dsa_index_score, dsa_prefill,  # noqa: F401
                  dsa_sparse_attn, dsa_topk, dsa_workspace_size, ld_scores_for)
from ._native import DsaError, LIB_PATH, EXPORTS  # noqa: F401

INPUT_KEYS = ("q_idx", "q_idx_sf", "w", "k_idx", "k_idx_sf", "q", "kv", "kv_scale", "kv_v", "n_valid")


def call_from_tensors(tensors: dict, **kw) -> DsaCall:
    """DsaCall from a dict holding the input tensors under the names of dsa_args."""
    return DsaCall(**{k: tensors.get(k) for k in INPUT_KEYS}, **kw)
