"""Seeded synthetic inputs for the indexer -> Top-K -> sparse-attention chain.

This module is shared by the parity tests, ``bench.py`` and the smoke check.
It draws random numbers and stores them in the formats the chain reads:

* bf16 tensors (round-to-nearest-even from N(0,1) fp32 draws),
* MXFP8 indexer tensors: E4M3 codes plus one E8M0 exponent byte per group of
  32 elements along the feature axis,
* an FP8 E4M3 latent-KV cache with one fp32 scale per token (row).

The encoders here only *produce* those stored bytes, the way an upstream
quantiser would before the chain runs.  Nothing in this module scores,
selects, attends or decodes: the readers of these bytes (the oracle and the
CUDA kernels) each interpret them with their own code.

Workload shapes follow the five synthetic workloads of the sparse-attention
chain (a tiny decode, a batch-8 decode at 32K context in bf16 and in
MXFP8/FP8, a batch-1 decode at 1M context, and a 4096-token causal prefill
chunk at the end of a 128K context).  All draws are N(0,1) except the head
weights, which are U(0,1).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Sequence, Tuple

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "encode_mxfp8", "encode_fp8_rows", "encode_fp8_tiles",
           "to_bf16", "small_workload"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and storage formats of one synthetic workload.

    T          number of queries in one call
    q_per_seq  queries that share one cache: 1 for batched decode (query t reads
               sequence t), T for a prefill chunk (all queries read sequence 0)
    L          cache length (positions per sequence)
    H_idx/d_idx  indexer heads / indexer feature size
    K          top-k
    H, D_qk, D_v  attention heads, q.k feature size, value size
    separate_v True when V is stored apart from K (tiny case); otherwise V is
               the first D_v columns of each latent row
    q_pos0     -1 for decode (query t sees n_valid[t] or L positions);
               >= 0 for a causal chunk: query t sits at q_pos0 + t % q_per_seq
               and sees positions 0 .. q_pos0 + t % q_per_seq
    lengths    decode only: the visible length of each query (n_valid), or None
               for L everywhere
    """

    name: str
    T: int
    q_per_seq: int
    L: int
    H_idx: int
    d_idx: int
    idx_dtype: str  # "bf16" | "mxfp8"
    K: int
    H: int
    D_qk: int
    D_v: int
    kv_dtype: str  # "bf16" | "fp8" (one scale per row) | "fp8_t128" (one scale per 128 of a row)
    separate_v: bool
    q_pos0: int
    seed: int
    lengths: Optional[Tuple[int, ...]] = None

    @property
    def n_seq(self) -> int:
        return self.T // self.q_per_seq

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D_qk)

    @property
    def is_prefill(self) -> bool:
        return self.q_pos0 >= 0

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    # 1 query, L=2048, indexer 4 x 64 bf16, K=64, one head d=64 with separate K/V.
    "tiny_decode_l2k": Workload("tiny_decode_l2k", T=1, q_per_seq=1, L=2048, H_idx=4, d_idx=64,
                                idx_dtype="bf16", K=64, H=1, D_qk=64, D_v=64, kv_dtype="bf16",
                                separate_v=True, q_pos0=-1, seed=1000),
    # batch 8, L=32768, indexer 64 x 128 bf16, K=2048, 16 heads over a 576-wide latent row.
    "decode_b8_l32k_bf16": Workload("decode_b8_l32k_bf16", T=8, q_per_seq=1, L=32768, H_idx=64,
                                    d_idx=128, idx_dtype="bf16", K=2048, H=16, D_qk=576, D_v=512,
                                    kv_dtype="bf16", separate_v=False, q_pos0=-1, seed=1001),
    # the same with an MXFP8 indexer and an FP8 E4M3 latent cache (per-token fp32 scale).
    "decode_b8_l32k_mxfp8": Workload("decode_b8_l32k_mxfp8", T=8, q_per_seq=1, L=32768, H_idx=64,
                                     d_idx=128, idx_dtype="mxfp8", K=2048, H=16, D_qk=576, D_v=512,
                                     kv_dtype="fp8", separate_v=False, q_pos0=-1, seed=1002),
    # the MXFP8 decode batch with the page's FP8 KV variant: one fp32 scale per 128-element tile
    # of each latent row (576 = 4 x 128 + 64: five scales per row); the N1b row of the scope table.
    "decode_b8_l32k_mxfp8_kvt128": Workload("decode_b8_l32k_mxfp8_kvt128", T=8, q_per_seq=1, L=32768,
                                            H_idx=64, d_idx=128, idx_dtype="mxfp8", K=2048, H=16,
                                            D_qk=576, D_v=512, kv_dtype="fp8_t128", separate_v=False,
                                            q_pos0=-1, seed=1006),
    # batch 1 at L=1,048,576, MXFP8 indexer, FP8 latent cache.
    "decode_b1_l1m_mxfp8": Workload("decode_b1_l1m_mxfp8", T=1, q_per_seq=1, L=1 << 20, H_idx=64,
                                    d_idx=128, idx_dtype="mxfp8", K=2048, H=16, D_qk=576, D_v=512,
                                    kv_dtype="fp8", separate_v=False, q_pos0=-1, seed=1003),
    # a batch of 8 sequences of different lengths in caches of 65536 positions (the N3 row of the
    # scope table: variable-length batches, some shorter than K); otherwise as decode_b8_l32k_bf16.
    "decode_b8_varlen_bf16": Workload("decode_b8_varlen_bf16", T=8, q_per_seq=1, L=65536, H_idx=64,
                                      d_idx=128, idx_dtype="bf16", K=2048, H=16, D_qk=576, D_v=512,
                                      kv_dtype="bf16", separate_v=False, q_pos0=-1, seed=1005,
                                      lengths=(65536, 512, 33000, 2048, 16384, 100, 60000, 8000)),
    # causal prefill chunk: 4096 queries at positions 126976..131071 of L=131072, bf16.
    "prefill_t4096_l128k_bf16": Workload("prefill_t4096_l128k_bf16", T=4096, q_per_seq=4096,
                                         L=131072, H_idx=64, d_idx=128, idx_dtype="bf16", K=2048,
                                         H=16, D_qk=576, D_v=512, kv_dtype="bf16",
                                         separate_v=False, q_pos0=126976, seed=1004),
}


def small_workload(base: str, **kw) -> Workload:
    """A reduced copy of a named workload (same formats, smaller sizes)."""
    wl = WORKLOADS[base]
    name = kw.pop("name", base + "_small")
    return wl.replace(name=name, **kw)


# ----------------------------------------------------------------------------------------------
# draws


def _gen(seed: int, tensor_id: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 1009 + tensor_id * 7919 + 17)
    return g


def _randn(shape: Sequence[int], seed: int, tensor_id: int) -> torch.Tensor:
    return torch.randn(tuple(shape), generator=_gen(seed, tensor_id), dtype=torch.float32)


def to_bf16(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> bf16, round to nearest even (torch's conversion)."""
    return x.to(torch.bfloat16)


# ----------------------------------------------------------------------------------------------
# encoders (producers of the stored formats; the readers live elsewhere)

E4M3_MAX = 448.0
E4M3_EMAX = 8  # 448 = 1.75 * 2**8


def _to_e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """fp32 -> E4M3 (OCP 'fn' variant) codes, saturating to +-448, RNE (torch's cast)."""
    return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def encode_mxfp8(x: torch.Tensor, group: int = 32):
    """OCP MX v1.0 MXFP8 (E4M3) encoding along the last axis.

    Each group of ``group`` elements shares the exponent
    ``floor(log2(amax)) - 8`` stored as an E8M0 byte (bias 127, clamped to
    [0, 254]); an all-zero group stores exponent 0.  Elements are divided by
    2**exponent and cast to E4M3 with saturation.  Returns (codes u8, scale u8).
    """
    *lead, d = x.shape
    assert d % group == 0
    g = x.reshape(*lead, d // group, group).to(torch.float32)
    amax = g.abs().amax(dim=-1)
    _, e = torch.frexp(amax)  # amax = m * 2**e, m in [0.5, 1)
    shared = (e - 1 - E4M3_EMAX).to(torch.int32)
    shared = torch.where(amax > 0, shared, torch.zeros_like(shared))
    shared = shared.clamp(-127, 127)
    scaled = g * torch.pow(2.0, -shared.to(torch.float32)).unsqueeze(-1)
    codes = _to_e4m3_codes(scaled).reshape(*lead, d)
    sf = (shared + 127).to(torch.uint8)
    return codes.contiguous(), sf.contiguous()


def encode_fp8_rows(x: torch.Tensor):
    """E4M3 per-row encoding with one fp32 scale per row: scale = amax / 448
    (1 for an all-zero row); codes = E4M3(x / scale) with saturation."""
    x = x.to(torch.float32)
    amax = x.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    codes = _to_e4m3_codes(x / scale.unsqueeze(-1))
    return codes.contiguous(), scale.contiguous()


def encode_fp8_tiles(x: torch.Tensor, tile: int = 128):
    """E4M3 encoding with one fp32 scale per `tile` consecutive elements of a row (the last tile
    may be shorter): each tile is encoded as encode_fp8_rows encodes a row.  Returns (codes u8,
    scales [..., ceil(width / tile)] fp32)."""
    parts = [encode_fp8_rows(x[..., t0:t0 + tile]) for t0 in range(0, x.shape[-1], tile)]
    codes = torch.cat([c for c, _ in parts], dim=-1)
    scales = torch.stack([sc for _, sc in parts], dim=-1)
    return codes.contiguous(), scales.contiguous()


# ----------------------------------------------------------------------------------------------
# workload inputs

_CHUNK_ROWS = 1 << 16


def _cache_rows(n_seq: int, L: int, width: int, seed: int, tid: int, fmt: str, with_scale=False):
    """Draw an [n_seq, L, width] N(0,1) cache and store it in ``fmt``; drawn in row
    chunks so host memory stays bounded for million-row caches."""
    out_codes = None
    out_sf = None
    for s in range(n_seq):
        for r0 in range(0, L, _CHUNK_ROWS):
            r1 = min(L, r0 + _CHUNK_ROWS)
            x = _randn((r1 - r0, width), seed, tid * 100003 + s * 4099 + r0 // _CHUNK_ROWS)
            if fmt == "bf16":
                c = to_bf16(x)
                sf = None
            elif fmt == "mxfp8":
                c, sf = encode_mxfp8(x)
            elif fmt == "fp8":
                c, sf = encode_fp8_rows(x)
            elif fmt == "fp8_t128":
                c, sf = encode_fp8_tiles(x, 128)
            else:
                raise ValueError(fmt)
            if out_codes is None:
                out_codes = torch.empty((n_seq, L, width), dtype=c.dtype)
                if sf is not None:
                    out_sf = torch.empty((n_seq, L) + tuple(sf.shape[1:]), dtype=sf.dtype)
            out_codes[s, r0:r1] = c
            if sf is not None:
                out_sf[s, r0:r1] = sf
    return out_codes, out_sf


def make_inputs(wl: Workload, seed_offset: int = 0, n_valid: Optional[Sequence[int]] = None
                ) -> Dict[str, Optional[torch.Tensor]]:
    """CPU tensors for one call of the chain on workload ``wl``.

    Keys: q_idx, q_idx_sf, w, k_idx, k_idx_sf, q, kv, kv_scale, kv_v, n_valid.
    Absent formats map to None.  ``seed_offset`` draws an independent set of the
    same shapes (used to rotate inputs between timed steps).
    """
    seed = wl.seed + 7777 * seed_offset
    T, S = wl.T, wl.n_seq
    out: Dict[str, Optional[torch.Tensor]] = {}

    qi = _randn((T, wl.H_idx, wl.d_idx), seed, 1)
    if wl.idx_dtype == "bf16":
        out["q_idx"], out["q_idx_sf"] = to_bf16(qi), None
    elif wl.idx_dtype == "mxfp8":
        out["q_idx"], out["q_idx_sf"] = encode_mxfp8(qi)
    else:
        raise ValueError(wl.idx_dtype)
    out["w"] = torch.rand((T, wl.H_idx), generator=_gen(seed, 2), dtype=torch.float32)

    out["k_idx"], out["k_idx_sf"] = _cache_rows(S, wl.L, wl.d_idx, seed, 3, wl.idx_dtype)

    out["q"] = to_bf16(_randn((T, wl.H, wl.D_qk), seed, 4))
    kv_fmt = wl.kv_dtype
    out["kv"], out["kv_scale"] = _cache_rows(S, wl.L, wl.D_qk, seed, 5, kv_fmt)
    if wl.separate_v:
        assert wl.kv_dtype == "bf16"
        out["kv_v"], _ = _cache_rows(S, wl.L, wl.D_v, seed, 6, "bf16")
    else:
        out["kv_v"] = None
    if n_valid is None:
        n_valid = wl.lengths
    out["n_valid"] = None if n_valid is None else torch.tensor(list(n_valid), dtype=torch.int32)
    return out


def to_numpy_bits(inputs: Dict[str, Optional[torch.Tensor]]):
    """The same stored bytes as numpy arrays: bf16 as uint16 bit patterns, codes as uint8,
    fp32 as float32, int32 as int32.  A pure re-view, no arithmetic."""
    import numpy as np

    out = {}
    for k, v in inputs.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = v.contiguous().view(torch.int16).numpy().view(np.uint16)
        else:
            out[k] = v.contiguous().numpy()
    return out
