"""Python face of the C ABI: the same entry points as include/dsa.h, taking torch tensors.

Argument marshalling only (pointers, sizes, strides, dtype codes, the current stream); outputs and
workspaces that the caller does not pass are allocated with torch on the inputs' device.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

import torch

from . import _native as N

__all__ = ["dsa_index_score", "dsa_topk", "dsa_topk_noalloc", "dsa_topk_pairs", "dsa_topk_merge",
           "dsa_sparse_attn_partial", "dsa_attn_combine", "dsa_sparse_attn", "DsaCall", "dsa_decode", "dsa_prefill",
           "dsa_workspace_size", "dsa_launch_count", "dsa_get_device_error", "ld_scores_for",
           "dsa_quantize_mxfp8", "dsa_quantize_fp8_rows", "dsa_quantize_fp8_tiles"]


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _idx_dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return N.DSA_BF16
    if t.dtype == torch.uint8:
        return N.DSA_MXFP8_E4M3
    raise TypeError(f"indexer tensors must be bfloat16 or uint8 (E4M3 codes), got {t.dtype}")


def _kv_dtype(t: torch.Tensor, scale: Optional[torch.Tensor] = None) -> int:
    """bf16 rows; E4M3 rows with one scale per row (kv_scale without a last tile axis), or with
    one scale per 128-element tile (kv_scale [..., ceil(D_qk / 128)] beside the rows' axes)."""
    if t.dtype == torch.bfloat16:
        return N.DSA_BF16
    if t.dtype == torch.uint8:
        if scale is not None and scale.dim() == t.dim():
            return N.DSA_FP8_E4M3_T128
        return N.DSA_FP8_E4M3
    raise TypeError(f"kv must be bfloat16 or uint8 (E4M3 codes), got {t.dtype}")


def _seq_stride(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.stride(0) * t.element_size()


def ld_scores_for(L: int) -> int:
    return max(4, (L + 3) // 4 * 4)


def dsa_index_score(q_idx, w, k_idx, *, q_idx_sf=None, k_idx_sf=None, q_per_seq=1, q_pos0=-1,
                    n_valid=None, scores=None, stream=None) -> torch.Tensor:
    """Indexer scores [T, ld] fp32 (entries s >= n_t unspecified).  q_idx [T, H_idx, d],
    k_idx [n_seq, L, d] (rows packed), sf tensors for MXFP8."""
    T, H_idx, d = q_idx.shape
    L = k_idx.shape[1]
    if scores is None:
        scores = torch.empty(T, ld_scores_for(L), dtype=torch.float32, device=q_idx.device)
    st = N.lib.dsa_index_score(_p(q_idx), _p(q_idx_sf), _p(w), _p(k_idx), _p(k_idx_sf),
                               _seq_stride(k_idx), _seq_stride(k_idx_sf), T, q_per_seq, q_pos0,
                               _p(n_valid), L, H_idx, d, _idx_dtype(q_idx), _p(scores),
                               scores.stride(0), _stream(stream))
    N.check(st, "dsa_index_score")
    return scores


def dsa_topk(scores, K, *, L, q_per_seq=1, q_pos0=-1, n_valid=None, idx=None, ws=None, stream=None) -> torch.Tensor:
    """Top-K positions [T, K] int32 (ascending, -1 padded).  `ws`, if given, is a zero-filled
    uint8 tensor of at least dsa_topk_workspace_size bytes that later calls may reuse."""
    T = scores.shape[0]
    if idx is None:
        idx = torch.empty(T, K, dtype=torch.int32, device=scores.device)
    ws_bytes = N.lib.dsa_topk_workspace_size(T, L, K)
    if ws is None:
        ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=scores.device) if ws_bytes else None
    else:
        ws_bytes = ws.numel()
    st = N.lib.dsa_topk(_p(scores), scores.stride(0), T, q_per_seq, q_pos0, _p(n_valid), L, K, _p(idx),
                        _p(ws), ws_bytes, _stream(stream))
    N.check(st, "dsa_topk")
    return idx


def dsa_topk_noalloc(scores, K, *, L, q_per_seq=1, q_pos0=-1, n_valid=None, idx=None, stream=None) -> torch.Tensor:
    """dsa_topk without a workspace: the library's own fixed scratch serves as the exchange area
    (at most 16 queries per call; calls that overlap on the GPU race, see dsa.h)."""
    T = scores.shape[0]
    if idx is None:
        idx = torch.empty(T, K, dtype=torch.int32, device=scores.device)
    st = N.lib.dsa_topk_noalloc(_p(scores), scores.stride(0), T, q_per_seq, q_pos0, _p(n_valid), L, K,
                                _p(idx), _stream(stream))
    N.check(st, "dsa_topk_noalloc")
    return idx


def dsa_sparse_attn(q, kv, idx, *, sm_scale, kv_v=None, kv_scale=None, D_v=None, q_per_seq=1,
                    out=None, lse=None, ws=None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Attention over the rows named by idx.  q [T, H, D_qk] bf16; kv [n_seq, L, row] (bf16 or E4M3
    codes, row pitch from its stride); kv_v optional [n_seq, L, D_v] bf16; kv_scale [n_seq, L]."""
    T, H, D_qk = q.shape
    L = kv.shape[1]
    K = idx.shape[1]
    if D_v is None:
        D_v = kv_v.shape[-1] if kv_v is not None else (512 if D_qk == 576 else D_qk)
    if out is None:
        out = torch.empty(T, H, D_v, dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty(T, H, dtype=torch.float32, device=q.device)
    need = N.lib.dsa_sparse_attn_workspace_size(T, H, K, D_v)
    if ws is None and need:
        ws = torch.zeros(need, dtype=torch.uint8, device=q.device)
    st = N.lib.dsa_sparse_attn(_p(q), _p(kv), _p(kv_v), _p(kv_scale), kv.stride(1) * kv.element_size(),
                               _seq_stride(kv), 0 if kv_v is None else kv_v.stride(1) * 2, _seq_stride(kv_v),
                               _p(idx), T, q_per_seq, L, K, H, D_qk, D_v, float(sm_scale), _kv_dtype(kv, kv_scale),
                               _p(out), _p(lse), _p(ws), 0 if ws is None else ws.numel(), _stream(stream))
    N.check(st, "dsa_sparse_attn")
    return out, lse


def dsa_topk_pairs(scores, K, *, L, pos_offset, cand_pos, cand_scores, q_per_seq=1, q_pos0=-1, n_valid=None,
                   ws=None, stream=None):
    """One context slice's Top-K as (score, global position) pairs written into the [T, >= K]
    views cand_pos (int32) / cand_scores (fp32), which may be column slices of a wider buffer."""
    T = scores.shape[0]
    ws_bytes = N.lib.dsa_topk_workspace_size(T, L, K)
    if ws is None:
        ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device=scores.device)
    st = N.lib.dsa_topk_pairs(_p(scores), scores.stride(0), T, q_per_seq, q_pos0, _p(n_valid), L, K,
                              int(pos_offset), _p(cand_pos), _p(cand_scores), cand_pos.stride(0), _p(ws),
                              ws.numel(), _stream(stream))
    N.check(st, "dsa_topk_pairs")
    return cand_pos, cand_scores


def dsa_topk_merge(cand_scores, cand_pos, K, *, idx=None, stream=None) -> torch.Tensor:
    """The K best (score, position) pairs of each query's candidates (-1 positions are empty), in
    candidate order, -1 padded.  Candidates as [T, n] (one part per query row) or as [G, T, n]
    (G parts, e.g. gathered from G devices), contiguous in the last axis."""
    if cand_pos.dim() == 2:
        T, n = cand_pos.shape
        parts, ld, pst = 1, cand_pos.stride(0), 0
    else:
        parts, T, n = cand_pos.shape
        ld, pst = cand_pos.stride(1), cand_pos.stride(0)
    if idx is None:
        idx = torch.empty(T, K, dtype=torch.int32, device=cand_pos.device)
    st = N.lib.dsa_topk_merge(_p(cand_scores), _p(cand_pos), T, parts, n, ld, pst, K, _p(idx), _stream(stream))
    N.check(st, "dsa_topk_merge")
    return idx


def dsa_sparse_attn_partial(q, kv, idx, *, sm_scale, pos_lo, kv_v=None, kv_scale=None, D_v=None, q_per_seq=1,
                            o_part=None, lse_part=None, ws=None, stream=None):
    """Attention of one context slice (cache rows = positions pos_lo .. pos_lo + L - 1) over the
    entries of idx it holds: fp32 normalised output [T, H, D_v] and its log-sum-exp [T, H]."""
    T, H, D_qk = q.shape
    L = kv.shape[1]
    K = idx.shape[1]
    if D_v is None:
        D_v = kv_v.shape[-1] if kv_v is not None else (512 if D_qk == 576 else D_qk)
    if o_part is None:
        o_part = torch.empty(T, H, D_v, dtype=torch.float32, device=q.device)
    if lse_part is None:
        lse_part = torch.empty(T, H, dtype=torch.float32, device=q.device)
    need = N.lib.dsa_sparse_attn_workspace_size(T, H, K, D_v)
    if ws is None and need:
        ws = torch.zeros(need, dtype=torch.uint8, device=q.device)
    st = N.lib.dsa_sparse_attn_partial(
        _p(q), _p(kv), _p(kv_v), _p(kv_scale), kv.stride(1) * kv.element_size(), _seq_stride(kv),
        0 if kv_v is None else kv_v.stride(1) * 2, _seq_stride(kv_v), _p(idx), T, q_per_seq, L, K, H, D_qk, D_v,
        float(sm_scale), _kv_dtype(kv, kv_scale), int(pos_lo), _p(o_part), _p(lse_part), _p(ws),
        0 if ws is None else ws.numel(), _stream(stream))
    N.check(st, "dsa_sparse_attn_partial")
    return o_part, lse_part


def dsa_attn_combine(o_parts, lse_parts, *, out=None, lse=None, stream=None):
    """Merge of G partial outputs o_parts [G, T, H, D_v] fp32 / lse_parts [G, T, H] into the bf16
    output [T, H, D_v] and its log-sum-exp [T, H]."""
    G, T, H, D_v = o_parts.shape
    if out is None:
        out = torch.empty(T, H, D_v, dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty(T, H, dtype=torch.float32, device=o_parts.device)
    st = N.lib.dsa_attn_combine(_p(o_parts), _p(lse_parts), G, o_parts.stride(0), lse_parts.stride(0), T, H, D_v,
                                _p(out), _p(lse), _stream(stream))
    N.check(st, "dsa_attn_combine")
    return out, lse


class DsaCall:
    """One configured fused call (dsa_decode or dsa_prefill) with its outputs and workspace
    allocated once; calling it enqueues the chain on the current (or given) stream."""

    def __init__(self, *, q_idx, w, k_idx, q, kv, K, sm_scale, q_idx_sf=None, k_idx_sf=None,
                 kv_scale=None, kv_v=None, D_v=None, q_per_seq=1, q_pos0=-1, n_valid=None,
                 out=None, lse=None, idx_out=None, keep_idx=True, ws=None,
                 block_table=None, block_size=0, L=None):
        """Caches are [n_seq, L, ...] per sequence, or, with `block_table` (int32 [n_seq,
        max_blocks]) and `block_size`, pools of rows ([rows, ...]; kv_scale [rows]) shared by all
        sequences, with the positions per sequence `L` given explicitly."""
        T, H_idx, d_idx = q_idx.shape
        _, H, D_qk = q.shape
        paged = block_table is not None
        if paged:
            if L is None or block_size <= 0:
                raise ValueError("paged caches need L and block_size")
        else:
            L = k_idx.shape[1]
        if D_v is None:
            D_v = kv_v.shape[-1] if kv_v is not None else (512 if D_qk == 576 else D_qk)
        dev = q.device
        self.prefill = q_pos0 >= 0
        self.out = out if out is not None else torch.empty(T, H, D_v, dtype=torch.bfloat16, device=dev)
        self.lse = lse if lse is not None else torch.empty(T, H, dtype=torch.float32, device=dev)
        if idx_out is None and keep_idx:
            idx_out = torch.empty(T, K, dtype=torch.int32, device=dev)
        self.idx = idx_out
        a = N.DsaArgs()
        a.T, a.q_per_seq, a.q_pos0, a.L, a.K = T, q_per_seq, q_pos0, L, K
        a.H_idx, a.d_idx, a.H, a.D_qk, a.D_v = H_idx, d_idx, H, D_qk, D_v
        a.sm_scale = float(sm_scale)
        a.idx_dtype, a.kv_dtype = _idx_dtype(q_idx), _kv_dtype(kv, kv_scale)
        ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
        a.n_valid = ptr(n_valid)
        a.q_idx, a.q_idx_sf, a.w = ptr(q_idx), ptr(q_idx_sf), ptr(w)
        a.k_idx, a.k_idx_sf = ptr(k_idx), ptr(k_idx_sf)
        a.q, a.kv, a.kv_v, a.kv_scale = ptr(q), ptr(kv), ptr(kv_v), ptr(kv_scale)
        if paged:
            a.k_seq_stride = a.k_sf_seq_stride = a.kv_seq_stride = a.v_seq_stride = 0
            a.kv_row_stride = kv.stride(0) * kv.element_size()
            a.v_row_stride = 0 if kv_v is None else kv_v.stride(0) * kv_v.element_size()
            a.block_table = ptr(block_table)
            a.block_size = int(block_size)
            a.max_blocks = block_table.shape[1]
            a.num_blocks = k_idx.shape[0] // int(block_size)
        else:
            a.k_seq_stride, a.k_sf_seq_stride = _seq_stride(k_idx), _seq_stride(k_idx_sf)
            a.kv_row_stride = kv.stride(1) * kv.element_size()
            a.kv_seq_stride = _seq_stride(kv)
            a.v_row_stride = 0 if kv_v is None else kv_v.stride(1) * kv_v.element_size()
            a.v_seq_stride = _seq_stride(kv_v)
            a.block_table = None
        a.out, a.lse, a.idx_out = ptr(self.out), ptr(self.lse), ptr(self.idx)
        self.args = a
        # keep every tensor the struct points at alive as long as the call object
        self._keep = (q_idx, w, k_idx, q, kv, q_idx_sf, k_idx_sf, kv_scale, kv_v, n_valid, block_table)
        need = dsa_workspace_size(a, self.prefill)
        if ws is None:
            ws = torch.zeros(max(need, 16), dtype=torch.uint8, device=dev)
        elif ws.numel() < need:
            raise ValueError(f"workspace has {ws.numel()} bytes, needs {need}")
        self.ws = ws
        self._fn = N.lib.dsa_prefill if self.prefill else N.lib.dsa_decode
        self.launches = dsa_launch_count(a, self.prefill)  # kernels per call

    def __call__(self, stream=None):
        st = self._fn(ctypes.byref(self.args), _p(self.ws), self.ws.numel(), _stream(stream))
        N.check(st, "dsa_prefill" if self.prefill else "dsa_decode")
        return self.out, self.lse, self.idx


def dsa_workspace_size(args: N.DsaArgs, prefill: bool) -> int:
    n = ctypes.c_size_t(0)
    N.check(N.lib.dsa_workspace_size(ctypes.byref(args), int(bool(prefill)), ctypes.byref(n)),
            "dsa_workspace_size")
    return n.value


def dsa_quantize_mxfp8(x, *, codes=None, sf=None, dst_rows=None, stream=None):
    """bf16 rows x [rows, d] -> (E4M3 codes, E8M0 exponents per 32).  With `dst_rows` (int64
    [rows]) input row r is written to row dst_rows[r] of the given `codes` [*, d] / `sf`
    [*, d/32] (a cache append); without it new [rows, d] / [rows, d/32] tensors are returned."""
    rows, d = x.shape
    if codes is None:
        codes = torch.empty(rows, d, dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(rows, d // 32, dtype=torch.uint8, device=x.device)
    N.check(N.lib.dsa_quantize_mxfp8(_p(x), x.stride(0), rows, d, _p(codes), _p(sf), _p(dst_rows),
                                     _stream(stream)), "dsa_quantize_mxfp8")
    return codes, sf


def dsa_quantize_fp8_rows(x, *, codes=None, scales=None, dst_rows=None, stream=None):
    """bf16 rows x [rows, width] -> (E4M3 codes, one fp32 scale per row); `dst_rows` as in
    dsa_quantize_mxfp8 (codes [*, >= width] with any row pitch, scales [*])."""
    rows, width = x.shape
    if codes is None:
        codes = torch.empty(rows, width, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(rows, dtype=torch.float32, device=x.device)
    N.check(N.lib.dsa_quantize_fp8_rows(_p(x), x.stride(0), rows, width, _p(codes), codes.stride(0),
                                        _p(scales), _p(dst_rows), _stream(stream)),
            "dsa_quantize_fp8_rows")
    return codes, scales


def dsa_quantize_fp8_tiles(x, *, tile=128, codes=None, scales=None, dst_rows=None, stream=None):
    """bf16 rows x [rows, width] -> (E4M3 codes, fp32 scales [rows, ceil(width / tile)]): one
    scale per `tile` consecutive elements of a row; `dst_rows` as in dsa_quantize_mxfp8."""
    rows, width = x.shape
    nt = -(-width // tile)
    if codes is None:
        codes = torch.empty(rows, width, dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(rows, nt, dtype=torch.float32, device=x.device)
    N.check(N.lib.dsa_quantize_fp8_tiles(_p(x), x.stride(0), rows, width, tile, _p(codes), codes.stride(0),
                                         _p(scales), _p(dst_rows), _stream(stream)), "dsa_quantize_fp8_tiles")
    return codes, scales


def dsa_launch_count(args: N.DsaArgs, prefill: bool) -> int:
    """Kernels one dsa_decode / dsa_prefill call with `args` launches."""
    n = ctypes.c_int(0)
    N.check(N.lib.dsa_launch_count(ctypes.byref(args), int(bool(prefill)), ctypes.byref(n)),
            "dsa_launch_count")
    return n.value


def dsa_decode(**kw):
    """Fused indexer -> Top-K -> sparse attention for a decode batch; returns (out, lse, idx)."""
    return DsaCall(**kw)()


def dsa_prefill(**kw):
    """Fused chain for a causal chunk (q_pos0 >= 0); returns (out, lse, idx)."""
    if kw.get("q_pos0", -1) < 0:
        raise ValueError("dsa_prefill needs q_pos0 >= 0")
    return DsaCall(**kw)()


def dsa_set_attn_kernel(kernel: int) -> None:
    """Select the attention kernel for the 576/512 latent row (N.DSA_ATTN_AUTO or
    N.DSA_ATTN_TCGEN05; process-wide, for calls made afterwards)."""
    N.check(N.lib.dsa_set_attn_kernel(int(kernel)), "dsa_set_attn_kernel")


def dsa_get_device_error(stream=None) -> int:
    code = ctypes.c_int(0)
    N.check(N.lib.dsa_get_device_error(ctypes.byref(code), _stream(stream)), "dsa_get_device_error")
    return code.value


def dsa_selftest_wait_timeout(stream=None) -> None:
    """Enqueue the failure-path self-test: a kernel whose bounded wait runs out (about one second)
    and records the wait-timeout device error code; read it with dsa_get_device_error."""
    N.check(N.lib.dsa_selftest_wait_timeout(_stream(stream)), "dsa_selftest_wait_timeout")
