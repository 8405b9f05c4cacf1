"""GB300 (sm_103a) sparse-attention decode/prefill chain: lightweight indexer -> Top-K ->
gather-driven sparse attention over a latent KV cache.

The compute lives in libdsa.so (C ABI in include/dsa.h); this package is its thin Python binding.
The library is loaded on first use of any entry point, and that use fails loudly when the library
is not built (`top_sparse_attention_gb300.build` builds it; importing that submodule does not
need the library).
"""
import importlib

_API = ("DsaCall", "dsa_decode", "dsa_get_device_error", "dsa_index_score", "dsa_launch_count", "dsa_prefill",
        "dsa_quantize_mxfp8", "dsa_quantize_fp8_rows", "dsa_quantize_fp8_tiles",
        "dsa_selftest_wait_timeout", "dsa_sparse_attn", "dsa_topk", "dsa_topk_noalloc", "dsa_workspace_size",
        "dsa_topk_pairs", "dsa_topk_merge", "dsa_sparse_attn_partial", "dsa_attn_combine",
        "dsa_set_attn_kernel", "ld_scores_for")
_NATIVE = ("DsaError", "LIB_PATH", "EXPORTS")

INPUT_KEYS = ("q_idx", "q_idx_sf", "w", "k_idx", "k_idx_sf", "q", "kv", "kv_scale", "kv_v", "n_valid")

__all__ = list(_API + _NATIVE) + ["call_from_tensors", "INPUT_KEYS"]


def __getattr__(name):
    if name in _API:
        return getattr(importlib.import_module(".api", __name__), name)
    if name in _NATIVE:
        return getattr(importlib.import_module("._native", __name__), name)
    raise AttributeError(name)


def call_from_tensors(tensors: dict, **kw):
    """DsaCall from a dict holding the input tensors under the names of dsa_args."""
    from .api import DsaCall

    return DsaCall(**{k: tensors.get(k) for k in INPUT_KEYS}, **kw)
