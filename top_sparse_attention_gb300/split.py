"""Decode with the context split over G slices (the KV cache distributed by token, "Day-0 Support
for Large Model Inference: From Operator Optimization to Production Serving"; each slice runs the
index and attention steps of "Day 0 Support for New LLM Architectures", Step 1, on the positions
it holds).

Slice g holds positions [lo_g, hi_g) of every sequence: its own indexer keys and latent KV rows.
Every position of the global Top-K is in the Top-K of its own slice, so one decode step is

  1. per slice: scores of its positions and its Top-K as (score, global position) pairs
     (dsa_index_score, dsa_topk_pairs);
  2. the G x K pairs of each query side by side -- an all-gather across devices -- and the global
     Top-K selected from them (dsa_topk_merge);
  3. per slice: attention over the selected positions it holds, as a normalised fp32 output and its
     log-sum-exp (dsa_sparse_attn_partial);
  4. the G partial outputs side by side -- a second all-gather -- merged (dsa_attn_combine).

Every step runs in the library's kernels; this module only plans the slices, holds the buffers
and moves the two small exchanges (for K = 2048: 16 KB of pairs and 16 x 512 fp32 outputs per
query and slice).  `SplitDecode` runs all slices on one device, writing the parts side by side
(the exchanges are then plain layout); `split_decode_rank` runs one slice per rank of a
torch.distributed group and exchanges the parts with all_gather.

A prefill chunk splits the other way, by query: `zigzag_prefill_rank` gives rank g the query
segments g and 2G - 1 - g of 2G equal segments, so every rank scores the same number of causal
positions, and gathers the rows back into query order.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import torch

from . import api

__all__ = ["SplitPlan", "SliceSteps", "SplitDecode", "slice_caches", "split_decode_rank", "zigzag_segments",
           "zigzag_work", "prefill_segment", "zigzag_prefill_rank"]

CACHE_KEYS = ("k_idx", "k_idx_sf", "kv", "kv_scale", "kv_v")


@dataclasses.dataclass(frozen=True)
class SplitPlan:
    """Slice boundaries: slice g holds positions [bounds[g], bounds[g + 1]) of every sequence."""

    L: int
    bounds: tuple

    @classmethod
    def even(cls, L: int, G: int, align: int = 128) -> "SplitPlan":
        """G slices of about L / G positions, inner boundaries on multiples of `align` (a whole
        number of 128-position index-score tiles per slice)."""
        if G < 1 or L < G:
            raise ValueError("need 1 <= G <= L")
        inner = [min(L, round(L * g / G / align) * align) for g in range(1, G)]
        b = [0] + inner + [L]
        if any(b[i] >= b[i + 1] for i in range(G)):
            raise ValueError(f"L = {L} is too short for {G} slices aligned to {align}")
        return cls(L, tuple(b))

    @property
    def G(self) -> int:
        return len(self.bounds) - 1

    def lo(self, g: int) -> int:
        return self.bounds[g]

    def length(self, g: int) -> int:
        return self.bounds[g + 1] - self.bounds[g]

    def visible(self, lengths: Optional[Sequence[int]], g: int) -> Optional[List[int]]:
        """Visible positions of each query inside slice g (None: every position of the slice)."""
        if lengths is None:
            return None
        return [max(0, min(int(n), self.bounds[g + 1]) - self.bounds[g]) for n in lengths]


def slice_caches(caches: Dict[str, Optional[torch.Tensor]], plan: SplitPlan, g: int) -> Dict[str, Optional[torch.Tensor]]:
    """Slice g's own caches, contiguous [n_seq, length, ...], copied out of whole-context caches
    [n_seq, L, ...] (set-up, as when each device is filled with its part of the cache)."""
    lo, hi = plan.bounds[g], plan.bounds[g + 1]
    return {k: (None if caches.get(k) is None else caches[k][:, lo:hi].contiguous()) for k in CACHE_KEYS}


class SliceSteps:
    """The per-slice steps of one split decode for T queries on the current device (C ABI calls).

    caches: slice g's k_idx [n_seq, len, d] (+ k_idx_sf), kv [n_seq, len, row] (+ kv_scale, kv_v).
    lengths: each query's visible length in the whole context (host ints) or None for L."""

    def __init__(self, plan: SplitPlan, g: int, caches, *, K: int, sm_scale: float, T: int,
                 lengths: Optional[Sequence[int]] = None, D_v: Optional[int] = None):
        self.plan, self.g, self.caches = plan, g, caches
        self.K, self.sm_scale, self.T, self.D_v = K, sm_scale, T, D_v
        self.L_g = plan.length(g)
        dev = caches["k_idx"].device
        vis = plan.visible(lengths, g)
        self.n_valid = None if vis is None else torch.tensor(vis, dtype=torch.int32, device=dev)
        self.scores = torch.empty(T, api.ld_scores_for(self.L_g), dtype=torch.float32, device=dev)
        from . import _native as N

        self.topk_ws = torch.zeros(max(16, N.lib.dsa_topk_workspace_size(T, self.L_g, K)), dtype=torch.uint8,
                                   device=dev)
        self.attn_ws = None

    def pairs(self, q_idx, q_idx_sf, w, cand_pos, cand_scores, stream=None):
        """Steps 1-2: this slice's Top-K as (score, global position) pairs into cand_pos /
        cand_scores ([T, K] views, int32 / fp32)."""
        c = self.caches
        api.dsa_index_score(q_idx, w, c["k_idx"], q_idx_sf=q_idx_sf, k_idx_sf=c["k_idx_sf"], n_valid=self.n_valid,
                            scores=self.scores, stream=stream)
        api.dsa_topk_pairs(self.scores, self.K, L=self.L_g, pos_offset=self.plan.lo(self.g), cand_pos=cand_pos,
                           cand_scores=cand_scores, n_valid=self.n_valid, ws=self.topk_ws, stream=stream)

    def partial(self, q, idx, o_part, lse_part, stream=None):
        """Step 4: attention over the selected positions this slice holds."""
        c = self.caches
        if self.attn_ws is None:
            from . import _native as N

            T, H, _ = q.shape
            D_v = o_part.shape[-1]
            need = N.lib.dsa_sparse_attn_workspace_size(T, H, idx.shape[1], D_v)
            self.attn_ws = torch.zeros(max(16, need), dtype=torch.uint8, device=q.device)
        api.dsa_sparse_attn_partial(q, c["kv"], idx, sm_scale=self.sm_scale, pos_lo=self.plan.lo(self.g),
                                    kv_v=c["kv_v"], kv_scale=c["kv_scale"], D_v=o_part.shape[-1], o_part=o_part,
                                    lse_part=lse_part, ws=self.attn_ws, stream=stream)


class SplitDecode:
    """All G slices of a split decode on one device: the parts are written side by side, so the two
    exchanges are plain layout.  Call it with the query-side inputs; returns (out, lse, idx)."""

    def __init__(self, plan: SplitPlan, slices: List[Dict[str, Optional[torch.Tensor]]], *, K: int,
                 sm_scale: float, T: int, H: int, D_v: int, lengths: Optional[Sequence[int]] = None):
        dev = slices[0]["k_idx"].device
        self.plan, self.K, self.T, self.H, self.D_v = plan, K, T, H, D_v
        self.steps = [SliceSteps(plan, g, slices[g], K=K, sm_scale=sm_scale, T=T, lengths=lengths, D_v=D_v)
                      for g in range(plan.G)]
        G = plan.G
        self.cand_pos = torch.empty(G, T, K, dtype=torch.int32, device=dev)
        self.cand_scores = torch.empty(G, T, K, dtype=torch.float32, device=dev)
        self.idx = torch.empty(T, K, dtype=torch.int32, device=dev)
        self.o_parts = torch.empty(G, T, H, D_v, dtype=torch.float32, device=dev)
        self.lse_parts = torch.empty(G, T, H, dtype=torch.float32, device=dev)
        self.out = torch.empty(T, H, D_v, dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty(T, H, dtype=torch.float32, device=dev)

    def __call__(self, q_idx, q_idx_sf, w, q, stream=None):
        for g, st in enumerate(self.steps):
            st.pairs(q_idx, q_idx_sf, w, self.cand_pos[g], self.cand_scores[g], stream=stream)
        api.dsa_topk_merge(self.cand_scores, self.cand_pos, self.K, idx=self.idx, stream=stream)
        for g, st in enumerate(self.steps):
            st.partial(q, self.idx, self.o_parts[g], self.lse_parts[g], stream=stream)
        api.dsa_attn_combine(self.o_parts, self.lse_parts, out=self.out, lse=self.lse, stream=stream)
        return self.out, self.lse, self.idx


def split_decode_rank(steps, q_idx, q_idx_sf, w, q, *, K: int, H: int, D_v: int, group=None, merge=None,
                      combine=None):
    """One rank's part of a split decode, slice = rank of `group` (torch.distributed).

    `steps` runs this rank's slice (SliceSteps, or any object with the same pairs / partial
    methods).  The candidate pairs [T, K] and the partial outputs [T, H, D_v] / [T, H] of every rank
    are exchanged with all_gather into [G, T, ...] buffers; every rank then merges and combines, so
    all ranks return the same (out, lse, idx).  `merge` / `combine` default to dsa_topk_merge /
    dsa_attn_combine on the parts layout."""
    import torch.distributed as dist

    merge = merge or (lambda cs, cp: api.dsa_topk_merge(cs, cp, K))
    combine = combine or (lambda o, l: api.dsa_attn_combine(o, l))
    G = dist.get_world_size(group)
    T = q.shape[0]
    dev = q.device
    cand_pos = torch.empty(T, K, dtype=torch.int32, device=dev)
    cand_scores = torch.empty(T, K, dtype=torch.float32, device=dev)
    steps.pairs(q_idx, q_idx_sf, w, cand_pos, cand_scores)
    all_pos = torch.empty(G, T, K, dtype=torch.int32, device=dev)
    all_scores = torch.empty(G, T, K, dtype=torch.float32, device=dev)
    dist.all_gather(list(all_pos.unbind(0)), cand_pos, group=group)
    dist.all_gather(list(all_scores.unbind(0)), cand_scores, group=group)
    idx = merge(all_scores, all_pos)
    o_part = torch.empty(T, H, D_v, dtype=torch.float32, device=dev)
    lse_part = torch.empty(T, H, dtype=torch.float32, device=dev)
    steps.partial(q, idx, o_part, lse_part)
    o_parts = torch.empty(G, T, H, D_v, dtype=torch.float32, device=dev)
    lse_parts = torch.empty(G, T, H, dtype=torch.float32, device=dev)
    dist.all_gather(list(o_parts.unbind(0)), o_part, group=group)
    dist.all_gather(list(lse_parts.unbind(0)), lse_part, group=group)
    out, lse = combine(o_parts, lse_parts)
    return out, lse, idx


# ------------------------------------------------------------------------------------------------
# Context-parallel prefill with zigzag segments ("Day 0 Support for New LLM Architectures", Key
# Optimization 3: the later a query sits in a causal chunk, the more history it scores, so rank g
# takes segments g and 2G - 1 - g of 2G equal segments; one gather then puts the rows back in
# order).  Each rank runs the fused prefill chain on its own queries against the whole context.


def zigzag_segments(T: int, G: int, rank: int):
    """Query ranges [a, b) of a T-query chunk that rank `rank` of G handles: segments rank and
    2G - 1 - rank of 2G equal segments (T a multiple of 2G)."""
    if T % (2 * G):
        raise ValueError("the chunk must split into 2G equal segments")
    seg = T // (2 * G)
    return [(rank * seg, (rank + 1) * seg), ((2 * G - 1 - rank) * seg, (2 * G - rank) * seg)]


def zigzag_work(T: int, G: int, rank: int, q_pos0: int) -> int:
    """Causal work of a rank: the positions its queries see, sum of (q_pos0 + t + 1)."""
    return sum(q_pos0 + t + 1 for a, b in zigzag_segments(T, G, rank) for t in range(a, b))


def prefill_segment(tensors: Dict[str, Optional[torch.Tensor]], a: int, b: int, *, K: int, sm_scale: float,
                    q_pos0: int, stream=None):
    """The fused prefill chain (dsa_prefill) on queries [a, b) of a chunk whose query 0 sits at
    position q_pos0: the query-side inputs are the rows a .. b - 1, the caches the whole context."""
    from . import call_from_tensors

    seg = dict(tensors)
    for k in ("q_idx", "q_idx_sf", "w", "q"):
        if seg.get(k) is not None:
            seg[k] = seg[k][a:b]
    call = call_from_tensors(seg, K=K, sm_scale=sm_scale, q_per_seq=b - a, q_pos0=q_pos0 + a)
    out, lse, idx = call(stream)
    return out, lse, idx


def zigzag_prefill_rank(run_segment, T: int, *, group=None):
    """One rank's part of a context-parallel prefill chunk of T queries: run_segment(a, b) computes
    (out [b-a, H, D_v], lse [b-a, H], idx [b-a, K]) for queries [a, b) on this rank; the rows of all
    ranks are exchanged with one all_gather each and returned in query order on every rank."""
    import torch.distributed as dist

    G = dist.get_world_size(group)
    rank = dist.get_rank(group)
    segs = zigzag_segments(T, G, rank)
    parts = [run_segment(a, b) for a, b in segs]
    mine = [torch.cat([p[i] for p in parts], dim=0).contiguous() for i in range(3)]  # [T/G, ...]
    result = []
    for x in mine:
        gathered = [torch.empty_like(x) for _ in range(G)]
        dist.all_gather(gathered, x, group=group)
        full = torch.empty((T,) + tuple(x.shape[1:]), dtype=x.dtype, device=x.device)
        for g, y in enumerate(gathered):
            off = 0
            for a, b in zigzag_segments(T, G, g):
                full[a:b] = y[off:off + (b - a)]
                off += b - a
        result.append(full)
    return tuple(result)
