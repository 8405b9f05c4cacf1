"""Decode with the context split over G slices, on one GPU, through the C ABI.

* dsa_topk_merge against the oracle's merge of (score, position) candidates: bit-exact index lists
  (integer work on the same fp32 scores), with exact ties inside and across parts, empty entries,
  queries with fewer candidates than K, and both candidate layouts;
* dsa_sparse_attn_partial + dsa_attn_combine against the oracle's attention over the same indices;
* the whole split decode (SplitDecode) of the 1M-token MXFP8 / FP8 workload and of a bf16 batch of
  varying lengths: the same index sets as the unsplit fused chain (every score is computed by the
  same arithmetic, so the sets are identical), and attention against the oracle on those indices.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import ATTN_GUARD, ATTN_TOL, LSE_TOL, check_chain, oracle_chain, to_device

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


def _candidates(rng, G, T, K, n_pos, ties):
    """G parts x T queries x K candidates: ascending distinct positions per part (part g draws from
    its own position range), some empty (-1) entries at the end of a part, scores with or without
    heavy exact ties."""
    pos = np.full((G, T, K), -1, dtype=np.int32)
    sc = np.zeros((G, T, K), dtype=np.float32)
    width = n_pos // G
    for g in range(G):
        for t in range(T):
            m = K if (g + t) % 3 else int(rng.integers(0, K))  # some parts list fewer than K
            p = np.sort(rng.choice(width, size=m, replace=False)) + g * width
            pos[g, t, :m] = p
            s = rng.standard_normal(m)
            sc[g, t, :m] = (np.round(s * 2) if ties else s * 30 + 100).astype(np.float32)
    return pos, sc


@pytest.mark.parametrize("G,T,K,ties", [(4, 3, 300, False), (8, 2, 2048, True), (3, 4, 1000, True), (1, 2, 64, False)])
def test_topk_merge_is_bit_exact(dsa, G, T, K, ties):
    rng = np.random.default_rng(60 + G)
    pos, sc = _candidates(rng, G, T, K, 100000, ties)
    want = np.stack([oracle.merge_candidates(sc[:, t].reshape(-1), pos[:, t].reshape(-1), K) for t in range(T)])
    # parts layout [G, T, K] (as gathered from devices)
    got = dsa.dsa_topk_merge(torch.from_numpy(sc).cuda(), torch.from_numpy(pos).cuda(), K).cpu().numpy()
    np.testing.assert_array_equal(got, want)
    # one [T, G * K] row per query
    sc2 = np.ascontiguousarray(sc.transpose(1, 0, 2).reshape(T, G * K))
    pos2 = np.ascontiguousarray(pos.transpose(1, 0, 2).reshape(T, G * K))
    got2 = dsa.dsa_topk_merge(torch.from_numpy(sc2).cuda(), torch.from_numpy(pos2).cuda(), K).cpu().numpy()
    np.testing.assert_array_equal(got2, want)
    for t in range(T):  # parts in order, ascending within: ascending output
        v = got[t][got[t] >= 0]
        assert np.all(np.diff(v) > 0)


def test_topk_merge_fewer_candidates_than_k_and_empty(dsa):
    pos = torch.tensor([[[5, 9, -1, -1], [-1, -1, -1, -1]]], dtype=torch.int32).cuda()  # G=1, T=2
    sc = torch.tensor([[[1.0, 2.0, 0.0, 0.0], [0.0, 0.0, 0.0, 0.0]]], dtype=torch.float32).cuda()
    got = dsa.dsa_topk_merge(sc, pos, 3).cpu().numpy()
    np.testing.assert_array_equal(got, [[5, 9, -1], [-1, -1, -1]])


@pytest.fixture(params=["auto", "tcgen05"])
def attn_kernel(request, dsa):
    """The library's attention kernel, and again the tensor-memory kernel (dsa_set_attn_kernel)."""
    from top_sparse_attention_gb300 import _native as N

    dsa.dsa_set_attn_kernel(N.DSA_ATTN_TCGEN05 if request.param == "tcgen05" else N.DSA_ATTN_AUTO)
    yield request.param
    dsa.dsa_set_attn_kernel(N.DSA_ATTN_AUTO)


@pytest.mark.parametrize("kv", ["bf16", "fp8", "fp8_t128"])
def test_partial_attention_and_combine_match_the_oracle(dsa, attn_kernel, kv):
    base = {"bf16": "decode_b8_l32k_bf16", "fp8": "decode_b8_l32k_mxfp8", "fp8_t128": "decode_b8_l32k_mxfp8_kvt128"}[kv]
    wl = synth.small_workload(base, T=3, L=6000, K=2048)
    cpu = synth.make_inputs(wl)
    from top_sparse_attention_gb300 import split

    plan = split.SplitPlan(wl.L, (0, 1280, 3200, 6000))
    rng = np.random.default_rng(61)
    idx = np.stack([np.sort(rng.choice(wl.L, size=wl.K, replace=False)) for _ in range(wl.T)]).astype(np.int32)
    idx[1, -100:] = -1
    idx_d = torch.from_numpy(idx).cuda()
    q = cpu["q"].cuda()
    o_parts = torch.empty(plan.G, wl.T, wl.H, wl.D_v, dtype=torch.float32, device="cuda")
    lse_parts = torch.empty(plan.G, wl.T, wl.H, dtype=torch.float32, device="cuda")
    for g in range(plan.G):
        c = to_device(split.slice_caches(cpu, plan, g))
        dsa.dsa_sparse_attn_partial(q, c["kv"], idx_d, sm_scale=wl.sm_scale, pos_lo=plan.lo(g), kv_scale=c["kv_scale"],
                                    D_v=wl.D_v, o_part=o_parts[g], lse_part=lse_parts[g])
    out, lse = dsa.dsa_attn_combine(o_parts, lse_parts)
    out, lse = out.float().cpu().numpy(), lse.cpu().numpy()
    ch, a = oracle_chain(wl, cpu)
    for t in range(wl.T):
        ref, ref_lse = ch.attention(t, idx[t], wl.D_v)
        err = float(np.max(np.abs(out[t] - ref)))
        assert err <= ATTN_GUARD[kv], f"t={t}: max-abs {err}"
        assert np.all(np.abs(lse[t] - ref_lse) <= LSE_TOL)
        # each part alone: the oracle over the rows that part holds
        for g in range(plan.G):
            lo, n = plan.lo(g), plan.length(g)
            mine = np.where((idx[t] >= lo) & (idx[t] < lo + n), idx[t], -1)
            ref_g, ref_lg = ch.attention(t, mine, wl.D_v)
            assert np.max(np.abs(o_parts[g, t].cpu().numpy() - ref_g)) <= ATTN_GUARD[kv]
            assert np.all(np.abs(lse_parts[g, t].cpu().numpy() - ref_lg) <= LSE_TOL)


def test_partial_attention_of_a_slice_holding_no_selected_row(dsa):
    wl = synth.small_workload("decode_b8_l32k_bf16", T=1, L=512, K=64)
    cpu = synth.make_inputs(wl)
    dev = to_device(cpu)
    idx = torch.arange(64, dtype=torch.int32, device="cuda")[None] + 600  # all beyond this slice
    o, l = dsa.dsa_sparse_attn_partial(dev["q"], dev["kv"], idx, sm_scale=wl.sm_scale, pos_lo=0)
    assert torch.all(o == 0) and torch.all(torch.isneginf(l))
    out, lse = dsa.dsa_attn_combine(torch.stack([o, o]), torch.stack([l, l]))
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))


@pytest.mark.parametrize("name,G", [("decode_b1_l1m_mxfp8", 4), ("decode_b1_l1m_mxfp8", 8), ("decode_b8_varlen_bf16", 3)])
def test_split_decode_matches_the_fused_chain_and_the_oracle(dsa, name, G):
    from top_sparse_attention_gb300 import split

    wl = synth.WORKLOADS[name]
    cpu = synth.make_inputs(wl)
    dev = to_device(cpu)
    fused = dsa.call_from_tensors(dev, K=wl.K, sm_scale=wl.sm_scale)
    f_out, f_lse, f_idx = [x.clone() for x in fused()]
    plan = split.SplitPlan.even(wl.L, G)
    slices = [to_device(split.slice_caches(cpu, plan, g)) for g in range(G)]
    del dev, fused
    sd = split.SplitDecode(plan, slices, K=wl.K, sm_scale=wl.sm_scale, T=wl.T, H=wl.H, D_v=wl.D_v, lengths=wl.lengths)
    q = {k: (cpu[k].cuda() if cpu[k] is not None else None) for k in ("q_idx", "q_idx_sf", "w", "q")}
    out, lse, idx = sd(q["q_idx"], q["q_idx_sf"], q["w"], q["q"])
    torch.cuda.synchronize()
    assert torch.equal(idx, f_idx)  # identical fp32 scores and tie rule: identical ascending lists
    out, lse, idx = out.float().cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()
    assert np.max(np.abs(out - f_out.float().cpu().numpy())) <= ATTN_GUARD[wl.kv_dtype]
    ch, _ = oracle_chain(wl, cpu)
    for t in range(wl.T):
        oracle.parity.check_topk(idx[t], ch.scores(t), wl.K)
        ref, ref_lse = ch.attention(t, idx[t], wl.D_v)
        err = float(np.max(np.abs(out[t] - ref)))
        assert err <= ATTN_GUARD[wl.kv_dtype], f"t={t}: max-abs {err}"
        fin = np.isfinite(ref_lse)
        assert np.all(np.abs(lse[t][fin] - ref_lse[fin]) <= LSE_TOL)


# ------------------------------------------------------------------------------------------------
# context-parallel prefill: the zigzag segments of the 4096-query chunk, run one after another on
# this device as G ranks would run them, against the single fused prefill call


@pytest.mark.parametrize("G", [2, 4])
def test_zigzag_prefill_segments_match_the_whole_chunk(dsa, G):
    from top_sparse_attention_gb300 import split

    wl = synth.WORKLOADS["prefill_t4096_l128k_bf16"]
    cpu = synth.make_inputs(wl)
    dev = to_device(cpu)
    whole = dsa.call_from_tensors(dev, K=wl.K, sm_scale=wl.sm_scale, q_per_seq=wl.q_per_seq, q_pos0=wl.q_pos0)
    w_out, w_lse, w_idx = [x.clone() for x in whole()]
    del whole
    out = torch.empty_like(w_out)
    lse = torch.empty_like(w_lse)
    idx = torch.empty_like(w_idx)
    for g in range(G):
        for a, b in split.zigzag_segments(wl.T, G, g):
            o, l, i = split.prefill_segment(dev, a, b, K=wl.K, sm_scale=wl.sm_scale, q_pos0=wl.q_pos0)
            out[a:b], lse[a:b], idx[a:b] = o, l, i
    torch.cuda.synchronize()
    assert torch.equal(idx, w_idx)  # a query's scores do not depend on the other queries of its launch
    assert float((out.float() - w_out.float()).abs().max()) <= ATTN_GUARD["bf16"]
    assert float((lse - w_lse).abs().max()) <= LSE_TOL
    ch, _ = oracle_chain(wl, cpu)
    for t in (0, 1023, 1024, 2047, 3000, 4095):
        ref, _ = ch.attention(t, idx[t].cpu().numpy(), wl.D_v)
        assert np.max(np.abs(out[t].float().cpu().numpy() - ref)) <= ATTN_GUARD["bf16"]
