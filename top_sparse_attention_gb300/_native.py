"""ctypes binding of libdsa.so (include/dsa.h): argument marshalling only.

Every step of the chain runs in the CUDA kernels behind the C ABI.  PyTorch is used here only to
hold device memory and to name the current CUDA stream.  Importing this module fails loudly when
the library has not been built: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdsa.so")

DSA_OK = 0
DSA_BF16, DSA_FP8_E4M3, DSA_MXFP8_E4M3, DSA_FP8_E4M3_T128 = 0, 1, 2, 3
DSA_ATTN_AUTO, DSA_ATTN_TCGEN05 = 0, 1
DEVERR = {0: "none", 1: "index out of range", 2: "wait timeout", 3: "row-split Top-K counts disagree"}

EXPORTS = (
    "dsa_status_string", "dsa_abi_version", "dsa_get_device_error", "dsa_index_score",
    "dsa_topk", "dsa_topk_workspace_size", "dsa_sparse_attn", "dsa_sparse_attn_workspace_size",
    "dsa_quantize_mxfp8", "dsa_quantize_fp8_rows", "dsa_quantize_fp8_tiles",
    "dsa_workspace_size", "dsa_launch_count", "dsa_decode", "dsa_prefill", "dsa_topk_noalloc",
    "dsa_selftest_wait_timeout", "dsa_topk_pairs", "dsa_topk_merge", "dsa_sparse_attn_partial",
    "dsa_attn_combine", "dsa_set_attn_kernel",
)


class DsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class DsaArgs(ctypes.Structure):
    """Mirror of struct dsa_args."""
    _fields_ = [
        ("T", ctypes.c_int), ("q_per_seq", ctypes.c_int), ("q_pos0", ctypes.c_int),
        ("L", ctypes.c_int), ("K", ctypes.c_int),
        ("H_idx", ctypes.c_int), ("d_idx", ctypes.c_int),
        ("H", ctypes.c_int), ("D_qk", ctypes.c_int), ("D_v", ctypes.c_int),
        ("sm_scale", ctypes.c_float),
        ("idx_dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int),
        ("n_valid", ctypes.c_void_p),
        ("q_idx", ctypes.c_void_p), ("q_idx_sf", ctypes.c_void_p), ("w", ctypes.c_void_p),
        ("k_idx", ctypes.c_void_p), ("k_idx_sf", ctypes.c_void_p),
        ("k_seq_stride", ctypes.c_int64), ("k_sf_seq_stride", ctypes.c_int64),
        ("q", ctypes.c_void_p), ("kv", ctypes.c_void_p), ("kv_v", ctypes.c_void_p),
        ("kv_scale", ctypes.c_void_p),
        ("kv_row_stride", ctypes.c_int64), ("kv_seq_stride", ctypes.c_int64),
        ("v_row_stride", ctypes.c_int64), ("v_seq_stride", ctypes.c_int64),
        ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("idx_out", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("block_size", ctypes.c_int), ("max_blocks", ctypes.c_int), ("num_blocks", ctypes.c_int),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -m top_sparse_attention_gb300.build` "
                          "(or __graft_entry__.build()).  There is no fallback implementation.")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    sig = {
        "dsa_status_string": (ctypes.c_char_p, [I]),
        "dsa_abi_version": (I, []),
        "dsa_set_attn_kernel": (I, [I]),
        "dsa_get_device_error": (I, [ctypes.POINTER(I), P]),
        "dsa_selftest_wait_timeout": (I, [P]),
        "dsa_index_score": (I, [P, P, P, P, P, I64, I64, I, I, I, P, I, I, I, I, P, I64, P]),
        "dsa_topk": (I, [P, I64, I, I, I, P, I, I, P, P, SZ, P]),
        "dsa_topk_workspace_size": (SZ, [I, I, I]),
        "dsa_topk_noalloc": (I, [P, I64, I, I, I, P, I, I, P, P]),
        "dsa_sparse_attn": (I, [P, P, P, P, I64, I64, I64, I64, P, I, I, I, I, I, I, I, F, I, P, P,
                                P, SZ, P]),
        "dsa_sparse_attn_workspace_size": (SZ, [I, I, I, I]),
        "dsa_topk_pairs": (I, [P, I64, I, I, I, P, I, I, I, P, P, I64, P, SZ, P]),
        "dsa_topk_merge": (I, [P, P, I, I, I, I64, I64, I, P, P]),
        "dsa_sparse_attn_partial": (I, [P, P, P, P, I64, I64, I64, I64, P, I, I, I, I, I, I, I, F, I, I,
                                        P, P, P, SZ, P]),
        "dsa_attn_combine": (I, [P, P, I, I64, I64, I, I, I, P, P, P]),
        "dsa_quantize_mxfp8": (I, [P, I64, I, I, P, P, P, P]),
        "dsa_quantize_fp8_rows": (I, [P, I64, I, I, P, I64, P, P, P]),
        "dsa_quantize_fp8_tiles": (I, [P, I64, I, I, I, P, I64, P, P, P]),
        "dsa_workspace_size": (I, [ctypes.POINTER(DsaArgs), I, ctypes.POINTER(SZ)]),
        "dsa_launch_count": (I, [ctypes.POINTER(DsaArgs), I, ctypes.POINTER(ctypes.c_int)]),
        "dsa_decode": (I, [ctypes.POINTER(DsaArgs), P, SZ, P]),
        "dsa_prefill": (I, [ctypes.POINTER(DsaArgs), P, SZ, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.dsa_status_string(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != DSA_OK:
        raise DsaError(status, what)
