"""Oracle for the indexer -> Top-K -> sparse-attention chain (TEST INFRASTRUCTURE).

A plain, slow, fp64 CPU statement of what the chain computes, written from the
source pages, used only by ``tests/``, the smoke check and the CPU-baseline leg
of ``bench.py``.  Nothing in the product path imports it, and it shares no code
with the CUDA kernels: it reads the same stored bytes (bf16 bits, E4M3 codes,
E8M0 exponents, fp32 scales) and decodes them with its own code.

Method, as the pages state it ("Day 0 Support for New LLM Architectures",
Step 1, the sparse attention modules; Key Optimization 1): a lightweight
indexer scores the relevance of every historical position, the Top-K positions
are selected, and a sparse-attention kernel reads only the selected entries of
the low-rank (latent) KV cache and computes exact attention over them.  The
score of position s for query t is

    I[t, s] = sum_h  w[t, h] * ReLU( q_idx[t, h, :] . k_idx[s, :] )

(per-head dot product, ReLU, head-weighted sum: the page's scoring, head-weighting
and Top-K chain).  Storage formats follow Key Optimization 2
of the same page: MXFP8 for the indexer (groups of 32 elements share one scale
factor) and FP8 for the sparse-attention KV cache.

Every function below is the plain definition; numpy's matmul and sort serve as
library primitives for the inner sums and the ordering.

Pinning: every function is pinned by ``tests/test_oracle_pins.py`` against
hand-worked fixtures (``tests/golden``), closed forms, library routines that
are independent of this file and brute force on tiny inputs.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence

import numpy as np

__all__ = [
    "bf16_bits_to_f64", "e4m3_to_f64", "e8m0_to_f64", "dequant_mxfp8", "dequant_fp8_rows",
    "e4m3_encode", "quantize_mxfp8", "quantize_fp8_rows", "dequant_fp8_tiles", "quantize_fp8_tiles",
    "index_scores", "topk_positions", "sparse_attention", "visible_length", "query_sequence",
    "Chain", "chain_query", "merge_candidates", "combine_partials",
]


# ----------------------------------------------------------------------------------------------
# Stored formats -> exact fp64 values
# (Day 0 Support for New LLM Architectures, Key Optimization 2: MXFP8 index path with groups of
#  32 sharing one scale factor; FP8 sparse-attention KV cache.)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> fp64.  A bf16 value is the top half of the fp32 with the
    same bits, so widening is exact."""
    b = np.asarray(bits).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32).astype(np.float64)


def e4m3_to_f64(codes) -> np.ndarray:
    """E4M3 ('fn' variant: no infinities, S.1111.111 is NaN) codes -> fp64.

    value = (-1)^s * 2^(e-7) * (1 + m/8)   for exponent field e in 1..15
          = (-1)^s * 2^(-6)  * (m/8)       for e = 0 (subnormal)
    NaN codes are rejected: they never appear in valid caches.
    """
    c = np.asarray(codes).astype(np.int64)
    if np.any((c & 0x7F) == 0x7F):
        raise ValueError("E4M3 NaN code in input")
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    return s * np.where(e == 0, sub, normal)


def e8m0_to_f64(codes) -> np.ndarray:
    """E8M0 exponent bytes -> 2^(code - 127).  Code 255 (NaN) is rejected."""
    c = np.asarray(codes).astype(np.int64)
    if np.any(c == 255):
        raise ValueError("E8M0 NaN code in input")
    return np.ldexp(1.0, c - 127)


def dequant_mxfp8(codes, sf, group: int = 32) -> np.ndarray:
    """MXFP8 tensor -> fp64: every element times 2^(shared exponent of its group of 32)."""
    v = e4m3_to_f64(codes)
    scale = e8m0_to_f64(sf)
    return v * np.repeat(scale, group, axis=-1)


def dequant_fp8_rows(codes, row_scale) -> np.ndarray:
    """FP8 E4M3 cache rows with one fp32 scale per row (token) -> fp64."""
    return e4m3_to_f64(codes) * np.asarray(row_scale, dtype=np.float64)[..., None]


def dequant_fp8_tiles(codes, tile_scale, tile: int = 128) -> np.ndarray:
    """FP8 E4M3 cache rows with one fp32 scale per `tile` consecutive elements of a row (the last
    tile may be shorter) -> fp64.  tile_scale has ceil(width / tile) entries per row.
    (Day 0 Support for New LLM Architectures, Key Optimization 2: FP8 KV cache with a scale per
    token and 128-element tile.)"""
    v = e4m3_to_f64(codes)
    width = v.shape[-1]
    sc = np.repeat(np.asarray(tile_scale, dtype=np.float64), tile, axis=-1)[..., :width]
    return v * sc


# ----------------------------------------------------------------------------------------------
# Values -> stored formats: the online quantisation that writes the caches
# (Day 0 Support for New LLM Architectures, Key Optimization 2: the indexer stores MXFP8 -- E4M3
#  elements, one shared power-of-two scale per group of 32 -- and the sparse-attention KV cache
#  stores FP8.  The group scale follows the OCP Microscaling Formats specification v1.0: the
#  shared exponent is floor(log2(amax)) minus the element format's largest exponent, 8 for E4M3.)

_E4M3_MAX = 448.0  # S.1111.110, the largest finite E4M3 value


def e4m3_encode(values) -> np.ndarray:
    """Values (fp64; exactly representable) -> E4M3 ('fn') codes, rounding to the nearest
    representable value with ties to the even code and saturating to +-448 (no NaN produced).

    Magnitudes below 2^-6 use the subnormal step 2^-9; a magnitude a >= 2^-6 with binary exponent
    E = floor(log2 a) uses the step 2^(E-3) (three mantissa bits).  The sign is kept, so values
    that round to zero from below give the negative zero code 0x80.
    """
    v = np.asarray(values, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    flat_v, flat_o = v.reshape(-1), out.reshape(-1)
    for i, x in enumerate(flat_v):
        if math.isnan(x):
            raise ValueError("NaN cannot be encoded")
        sign = 0x80 if math.copysign(1.0, x) < 0 else 0
        a = abs(x)
        if a >= _E4M3_MAX:
            code = 0x7E
        elif a < 2.0 ** -6:
            m = _round_half_even(a / 2.0 ** -9)  # 0..8; 8 is the smallest normal, code 0x08
            code = m
        else:
            e = math.floor(math.log2(a))
            # log2 of a value just below a power of two can round up: correct the exponent
            if 2.0 ** e > a:
                e -= 1
            elif 2.0 ** (e + 1) <= a:
                e += 1
            r = _round_half_even(a / 2.0 ** (e - 3))  # 8..16
            if r == 16:
                e, r = e + 1, 8
            code = ((e + 7) << 3) | (r - 8)
            code = min(code, 0x7E)
        flat_o[i] = sign | code
    return out


def _round_half_even(q: float) -> int:
    f = math.floor(q)
    d = q - f
    if d > 0.5 or (d == 0.5 and f % 2 == 1):
        return int(f) + 1
    return int(f)


def quantize_mxfp8(x, group: int = 32):
    """Rows of values (fp64, last axis a multiple of `group`) -> (E4M3 codes, E8M0 exponents).

    For each group of 32: amax = max |x|; shared exponent X = floor(log2 amax) - 8, clamped to
    E8M0's range [-127, 127] (0 for an all-zero group); the exponent byte is X + 127 and each
    element is e4m3_encode(x / 2^X).  Dividing by a power of two is exact.
    """
    x = np.asarray(x, dtype=np.float64)
    *lead, d = x.shape
    if d % group:
        raise ValueError("row length must be a multiple of the group size")
    g = x.reshape(*lead, d // group, group)
    amax = np.max(np.abs(g), axis=-1)
    exps = np.zeros(amax.shape, dtype=np.int64)
    nz = amax > 0
    exps[nz] = np.floor(np.log2(amax[nz])).astype(np.int64)
    # the same exact correction as in e4m3_encode
    too_big = nz & (np.ldexp(1.0, exps) > amax)
    exps[too_big] -= 1
    too_small = nz & (np.ldexp(1.0, exps + 1) <= amax)
    exps[too_small] += 1
    shared = np.where(nz, np.clip(exps - 8, -127, 127), 0)
    codes = e4m3_encode(g / np.ldexp(1.0, shared)[..., None]).reshape(*lead, d)
    return codes, (shared + 127).astype(np.uint8)


def quantize_fp8_rows(x):
    """Rows of values (exact in fp32) -> (E4M3 codes, fp32 scale per row), computed in fp32:
    s = amax / 448 rounded to fp32 (1 for an all-zero row) and codes = e4m3_encode of the fp32
    quotient x / s.  The quotient is not exact, so it is formed in the precision the cache
    writer uses (IEEE fp32 division, round to nearest)."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    s = np.where(amax > 0, amax / np.float32(_E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = (x32 / s[..., None]).astype(np.float32)
    return e4m3_encode(q.astype(np.float64)), s


def quantize_fp8_tiles(x, tile: int = 128):
    """Rows of values -> (E4M3 codes, fp32 scales [..., ceil(width / tile)]): every `tile`
    consecutive elements of a row (the last tile may be shorter) are one quantize_fp8_rows row."""
    x = np.asarray(x, dtype=np.float64)
    width = x.shape[-1]
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = []
    for t0 in range(0, width, tile):
        c, s = quantize_fp8_rows(x[..., t0:t0 + tile])
        codes[..., t0:t0 + tile] = c
        scales.append(s)
    return codes, np.stack(scales, axis=-1).astype(np.float32)


# ----------------------------------------------------------------------------------------------
# The three steps


def index_scores(q_idx: np.ndarray, w: np.ndarray, k_idx: np.ndarray) -> np.ndarray:
    """Indexer score of every visible position for one query.

    q_idx [H_idx, d_idx], w [H_idx], k_idx [n, d_idx] (all fp64) -> I [n]:
    I[s] = sum_h w[h] * max(0, q_idx[h] . k_idx[s]).
    (Day 0 Support for New LLM Architectures, Step 1 and Key Optimization 1: the indexer scores
    every historical position; relevance scoring, then head-weight application.)
    """
    logits = k_idx @ q_idx.T            # [n, H_idx]: per-head q.k
    return np.maximum(logits, 0.0) @ w  # ReLU, then the head-weighted sum


def topk_positions(scores: np.ndarray, K: int) -> np.ndarray:
    """Top-K selection by a full sort.

    Positions are ordered by score (descending), exact ties by position (ascending); the first
    min(K, n) are returned and the rest of the K slots hold -1.
    (Day 0 Support for New LLM Architectures, Step 1: select the Top-K positions.)
    """
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))
    out = np.full(K, -1, dtype=np.int64)
    m = min(K, n)
    out[:m] = order[:m]
    return out


def sparse_attention(q: np.ndarray, k_rows: np.ndarray, v_rows: np.ndarray, sm_scale: float):
    """Exact softmax attention of H heads over the selected rows only.

    q [H, D_qk], k_rows [m, D_qk], v_rows [m, D_v] -> out [H, D_v], lse [H] where
    logits = sm_scale * q . k, out = softmax(logits) @ v and lse = log(sum exp(logits)).
    With no selected rows (m = 0) the output is 0 and the lse is -inf.
    (Day 0 Support for New LLM Architectures, Step 1: the sparse-attention kernel reads only the
    selected KV entries and performs exact computation.)
    """
    H, D_v = q.shape[0], v_rows.shape[1]
    if k_rows.shape[0] == 0:
        return np.zeros((H, D_v)), np.full(H, -np.inf)
    logits = sm_scale * (q @ k_rows.T)           # [H, m]
    mx = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - mx)
    l = p.sum(axis=1, keepdims=True)
    out = (p @ v_rows) / l
    lse = (mx + np.log(l))[:, 0]
    return out, lse


# ----------------------------------------------------------------------------------------------
# A context split over slices (the KV cache distributed by token: "Day-0 Support for Large Model
# Inference: From Operator Optimization to Production Serving"; each slice runs the index and
# attention steps of "Day 0 Support for New LLM Architectures", Step 1, on its own positions)


def merge_candidates(scores: np.ndarray, positions: np.ndarray, K: int) -> np.ndarray:
    """Top-K of a list of (score, position) candidates; entries with a negative position are empty.

    The min(K, m) valid entries that come first in the order (score descending, position
    ascending) are kept and returned as positions in the order of the candidate list, followed by
    -1 in the remaining slots.
    """
    s = np.asarray(scores, dtype=np.float64)
    p = np.asarray(positions, dtype=np.int64)
    valid = np.flatnonzero(p >= 0)
    order = np.lexsort((p[valid], -s[valid]))
    kept = np.sort(valid[order[: min(K, valid.size)]])  # back into list order
    out = np.full(K, -1, dtype=np.int64)
    out[: kept.size] = p[kept]
    return out


def combine_partials(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Attention outputs of disjoint row sets merged into the output over their union.

    o_parts [G, H, D_v] (each normalised over its own rows), lse_parts [G, H] (natural log-sum-exp
    of its logits; -inf for an empty set) -> out [H, D_v], lse [H]:
    lse = log sum_g exp(lse_g) and out = sum_g exp(lse_g - lse) o_g.  All parts empty: 0 and -inf.
    """
    o = np.asarray(o_parts, dtype=np.float64)
    l = np.asarray(lse_parts, dtype=np.float64)
    M = np.max(l, axis=0)
    Mu = np.where(np.isfinite(M), M, 0.0)
    w = np.where(np.isfinite(l), np.exp(l - Mu[None, :]), 0.0)  # [G, H]
    tot = w.sum(axis=0)
    safe = np.where(tot > 0, tot, 1.0)
    out = np.einsum("gh,ghd->hd", w, np.where(np.isfinite(l)[..., None], o, 0.0)) / safe[:, None]
    lse = np.where(tot > 0, Mu + np.log(safe), -np.inf)
    return np.where(tot[:, None] > 0, out, 0.0), lse


# ----------------------------------------------------------------------------------------------
# Which positions a query sees


def query_sequence(t: int, q_per_seq: int) -> int:
    """Queries are grouped by cache: query t reads sequence t // q_per_seq."""
    return t // q_per_seq


def visible_length(t: int, L: int, q_per_seq: int, q_pos0: int, n_valid=None) -> int:
    """Number of positions query t may attend to.

    Decode (q_pos0 < 0): positions 0 .. n_valid[t]-1, or the whole cache of length L.
    Causal chunk (q_pos0 >= 0): query t sits at position q_pos0 + t % q_per_seq and sees that
    position and everything before it ("Achieving Day-0 Readiness...", section 2.3: prefill
    computes scores for all queries in a batch; "Day 0 Support for New LLM Architectures",
    Key Optimization 3: the later a position, the more history it sees).
    """
    if q_pos0 < 0:
        n = L if n_valid is None else int(n_valid[t])
    else:
        n = q_pos0 + (t % q_per_seq) + 1
    return max(0, min(n, L))


# ----------------------------------------------------------------------------------------------
# One query through the chain


class Chain:
    """Decoded view of one set of stored inputs (the dict ``synth.make_inputs`` returns, with
    tensors converted to numpy raw bits) plus the workload parameters.

    Decoding of the big caches is lazy and per sequence, so a query only pays for its own rows.
    """

    def __init__(self, arrays: Dict[str, Optional[np.ndarray]], *, L: int, K: int, q_per_seq: int,
                 q_pos0: int, idx_dtype: str, kv_dtype: str, sm_scale: float):
        self.a = arrays
        self.L, self.K, self.q_per_seq, self.q_pos0 = L, K, q_per_seq, q_pos0
        self.idx_dtype, self.kv_dtype, self.sm_scale = idx_dtype, kv_dtype, sm_scale
        self._kidx_cache: Dict[int, np.ndarray] = {}

    # stored -> fp64
    def q_idx(self, t: int) -> np.ndarray:
        if self.idx_dtype == "bf16":
            return bf16_bits_to_f64(self.a["q_idx"][t])
        return dequant_mxfp8(self.a["q_idx"][t], self.a["q_idx_sf"][t])

    def k_idx(self, seq: int, n: int) -> np.ndarray:
        if self.idx_dtype == "bf16":
            return bf16_bits_to_f64(self.a["k_idx"][seq, :n])
        return dequant_mxfp8(self.a["k_idx"][seq, :n], self.a["k_idx_sf"][seq, :n])

    def kv_rows(self, seq: int, rows: np.ndarray):
        kv = self.a["kv"][seq, rows]
        if self.kv_dtype == "bf16":
            k = bf16_bits_to_f64(kv)
        elif self.kv_dtype == "fp8_t128":
            k = dequant_fp8_tiles(kv, self.a["kv_scale"][seq, rows])
        else:
            k = dequant_fp8_rows(kv, self.a["kv_scale"][seq, rows])
        if self.a.get("kv_v") is not None:
            v = bf16_bits_to_f64(self.a["kv_v"][seq, rows])
        else:
            v = None
        return k, v

    def n_visible(self, t: int) -> int:
        return visible_length(t, self.L, self.q_per_seq, self.q_pos0, self.a.get("n_valid"))

    def scores(self, t: int) -> np.ndarray:
        seq = query_sequence(t, self.q_per_seq)
        n = self.n_visible(t)
        w = np.asarray(self.a["w"][t], dtype=np.float64)
        qi = self.q_idx(t)
        out = np.empty(n)
        step = 1 << 16  # bounded memory for million-row caches; each score is computed alone
        for r0 in range(0, n, step):
            r1 = min(n, r0 + step)
            if self.idx_dtype == "bf16":
                kk = bf16_bits_to_f64(self.a["k_idx"][seq, r0:r1])
            else:
                kk = dequant_mxfp8(self.a["k_idx"][seq, r0:r1], self.a["k_idx_sf"][seq, r0:r1])
            out[r0:r1] = index_scores(qi, w, kk)
        return out

    def attention(self, t: int, idx: np.ndarray, D_v: int):
        """Attention of query t over the positions in ``idx`` (entries < 0 are padding)."""
        seq = query_sequence(t, self.q_per_seq)
        rows = np.asarray(idx, dtype=np.int64)
        rows = rows[rows >= 0]
        q = bf16_bits_to_f64(self.a["q"][t])
        k, v = self.kv_rows(seq, rows)
        if v is None:  # latent cache: V is the first D_v columns of the same row
            v = k[:, :D_v]
        return sparse_attention(q, k, v, self.sm_scale)


def chain_query(chain: Chain, t: int, D_v: int):
    """Indexer scores -> Top-K -> sparse attention for query t.

    Returns a dict with the scores [n_t], idx [K] (-1 padded), out [H, D_v] and lse [H].
    """
    s = chain.scores(t)
    idx = topk_positions(s, chain.K)
    out, lse = chain.attention(t, idx, D_v)
    return {"scores": s, "idx": idx, "out": out, "lse": lse}
