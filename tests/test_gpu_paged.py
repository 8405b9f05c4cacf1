"""Paged caches: the same caches stored as blocks of a shared pool in a random order, read through a
block table.  The chain over the pools must give exactly the outputs of the chain over the
contiguous caches (the same arithmetic on the same values; only the addresses differ), and the
contiguous chain is checked against the oracle."""
import numpy as np
import pytest
import torch

import synth
from gpu_helpers import check_chain, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_attention_gb300 import build

    build.build()
    import top_sparse_attention_gb300 as m

    torch.cuda.set_device(0)
    yield m
    torch.cuda.synchronize()
    assert m.dsa_get_device_error() == 0


def _to_pool(cache, table, block_size, n_blocks):
    """cache [n_seq, L, ...] -> pool [n_blocks * block_size, ...] with block j of sequence q at
    pool block table[q, j]; unused pool rows hold a constant that would spoil any result."""
    n_seq, L = cache.shape[:2]
    pool = torch.full((n_blocks * block_size,) + tuple(cache.shape[2:]), 0x5A if cache.dtype == torch.uint8 else 7.0,
                      dtype=cache.dtype)
    for q in range(n_seq):
        for j in range(table.shape[1]):
            lo = j * block_size
            if lo >= L:
                break
            hi = min(L, lo + block_size)
            b = int(table[q, j])
            pool[b * block_size: b * block_size + (hi - lo)] = cache[q, lo:hi]
    return pool


def _paged_call(dsa, wl, cpu, block_size, seed, extra_blocks=3):
    n_seq = wl.n_seq
    per_seq = -(-wl.L // block_size)
    n_blocks = n_seq * per_seq + extra_blocks
    rng = np.random.default_rng(seed)
    table = torch.from_numpy(rng.permutation(n_blocks)[: n_seq * per_seq].reshape(n_seq, per_seq).astype(np.int32))
    pools = {}
    for key in ("k_idx", "k_idx_sf", "kv", "kv_v"):
        if cpu[key] is not None:
            pools[key] = _to_pool(cpu[key], table, block_size, n_blocks)
    if cpu["kv_scale"] is not None:
        pools["kv_scale"] = _to_pool(cpu["kv_scale"], table, block_size, n_blocks)
    dev = to_device(dict(cpu, **pools))
    call = dsa.DsaCall(q_idx=dev["q_idx"], w=dev["w"], k_idx=dev["k_idx"], q=dev["q"], kv=dev["kv"], K=wl.K,
                       sm_scale=wl.sm_scale, q_idx_sf=dev["q_idx_sf"], k_idx_sf=dev["k_idx_sf"],
                       kv_scale=dev["kv_scale"], kv_v=dev["kv_v"], D_v=wl.D_v, q_per_seq=wl.q_per_seq,
                       q_pos0=wl.q_pos0, n_valid=dev["n_valid"], block_table=table.cuda(),
                       block_size=block_size, L=wl.L)
    return call()


def _contiguous_call(dsa, wl, cpu):
    dev = to_device(cpu)
    call = dsa.call_from_tensors(dev, K=wl.K, sm_scale=wl.sm_scale, q_per_seq=wl.q_per_seq, q_pos0=wl.q_pos0)
    return call()


CASES = [
    # name, base workload, overrides, n_valid, block size
    ("bf16_b64_ragged", "decode_b8_l32k_bf16", dict(T=3, L=3000, K=512), [3000, 130, 1999], 64),
    ("bf16_b192", "decode_b8_l32k_bf16", dict(T=2, L=2000, K=300), None, 192),
    ("mxfp8_fp8_b128", "decode_b8_l32k_mxfp8", dict(T=2, L=2500, K=400), [2500, 777], 128),
    ("mxfp8_fp8_b64", "decode_b8_l32k_mxfp8", dict(T=3, L=1300, K=256), None, 64),
    ("tiny_separate_v_b64", "tiny_decode_l2k", dict(), None, 64),
    ("prefill_grouped_b64", "prefill_t4096_l128k_bf16", dict(T=8, q_per_seq=8, L=700, K=128, q_pos0=400), None, 64),
    ("long_row_split_b256", "decode_b1_l1m_mxfp8", dict(L=300000), None, 256),
    ("fp8_tiles_b64", "decode_b8_l32k_mxfp8_kvt128", dict(T=2, L=1500, K=300), [1500, 640], 64),
]


@pytest.mark.parametrize("name,base,kw,n_valid,bs", CASES, ids=[c[0] for c in CASES])
def test_paged_chain_equals_contiguous_chain(dsa, name, base, kw, n_valid, bs):
    wl = synth.small_workload(base, name=name, **kw)
    cpu = synth.make_inputs(wl, n_valid=n_valid)
    out_c, lse_c, idx_c = [x.clone() for x in _contiguous_call(dsa, wl, cpu)]
    out_p, lse_p, idx_p = _paged_call(dsa, wl, cpu, bs, seed=sum(map(ord, name)))
    torch.cuda.synchronize()
    assert torch.equal(idx_p, idx_c)
    assert torch.equal(out_p, out_c)
    assert torch.equal(lse_p, lse_c)
    check_chain(dsa, wl, cpu)  # and that chain against the oracle


def test_paged_arguments_are_checked(dsa):
    wl = synth.small_workload("decode_b8_l32k_bf16", T=1, L=256, K=64)
    cpu = synth.make_inputs(wl)
    table = torch.zeros(1, 4, dtype=torch.int32)
    dev = to_device(cpu)
    for bs, L in ((48, 256), (64, 300)):  # not a multiple of 64; too few table entries
        with pytest.raises(Exception):
            dsa.DsaCall(q_idx=dev["q_idx"], w=dev["w"], k_idx=dev["k_idx"][0], q=dev["q"], kv=dev["kv"][0], K=64,
                        sm_scale=wl.sm_scale, block_table=table.cuda(), block_size=bs, L=L)()
