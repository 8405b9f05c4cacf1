"""Parity of the CUDA path (through the C ABI) with the oracle on the same seeded inputs.

Step-level checks isolate each kernel:
  * dsa_index_score vs the oracle's fp64 scores, within an fp32 accumulation bound,
  * dsa_topk on identical fp32 scores: the index set must be bit-exact (integer work),
  * dsa_sparse_attn on identical indices: max-abs 2e-2 (bf16) / 6e-2 (FP8) and a tighter guard.
The fused chain is checked on all five workloads: indices under the near-tie rule against the
oracle's fp64 scores, attention against the oracle evaluated on the GPU's own indices.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import ATTN_GUARD, ATTN_TOL, LSE_TOL, check_chain, oracle_chain, score_error_bound, to_device

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


# ------------------------------------------------------------------------------------------------
# step 1: index scores

SCORE_CASES = [
    # name, base workload, overrides, n_valid
    ("bf16_d128_h64_ragged", "decode_b8_l32k_bf16", dict(T=3, L=1000), None),
    ("bf16_d64_h4_tiny", "tiny_decode_l2k", dict(), None),
    ("bf16_d128_h1", "decode_b8_l32k_bf16", dict(T=2, L=300, H_idx=1), None),
    ("bf16_d128_h17", "decode_b8_l32k_bf16", dict(T=2, L=513, H_idx=17), None),
    ("bf16_d128_h33", "decode_b8_l32k_bf16", dict(T=2, L=257, H_idx=33), None),
    ("mxfp8_d128_h64", "decode_b8_l32k_mxfp8", dict(T=2, L=777), None),
    ("mxfp8_d128_h20", "decode_b8_l32k_mxfp8", dict(T=3, L=200, H_idx=20), None),
    ("mxfp8_d128_h8", "decode_b8_l32k_mxfp8", dict(T=3, L=300, H_idx=8), None),
    ("mxfp8_d128_h40_t1", "decode_b8_l32k_mxfp8", dict(T=1, L=1000, H_idx=40), None),
    ("mxfp8_wide_scales", "decode_b8_l32k_mxfp8", dict(T=3, L=900), None),
    ("mxfp8_varlen", "decode_b8_l32k_mxfp8", dict(T=4, L=1300), [1300, 5, 0, 777]),
    ("varlen", "decode_b8_l32k_bf16", dict(T=4, L=1000), [0, 1, 129, 1000]),
    ("prefill_grouped", "prefill_t4096_l128k_bf16", dict(T=8, q_per_seq=8, L=600, q_pos0=400), None),
    ("prefill_ungrouped_t6", "prefill_t4096_l128k_bf16", dict(T=6, q_per_seq=6, L=700, q_pos0=10), None),
    ("prefill_mx", "decode_b8_l32k_mxfp8", dict(T=5, q_per_seq=5, L=300, q_pos0=200), None),
]


@pytest.mark.parametrize("name,base,kw,n_valid", SCORE_CASES, ids=[c[0] for c in SCORE_CASES])
def test_index_score_parity(dsa, name, base, kw, n_valid):
    wl = synth.small_workload(base, name=name, **kw)
    cpu = synth.make_inputs(wl, n_valid=n_valid)
    if name == "bf16_d128_h17":
        cpu["w"] = cpu["w"] - 0.5  # negative head weights
    if name == "mxfp8_wide_scales":
        # every group, row and head its own exponent: a scale applied to the wrong group, row or
        # head changes the scores far beyond the bound
        g = torch.Generator().manual_seed(5)
        for key in ("q_idx_sf", "k_idx_sf"):
            cpu[key] = torch.randint(118, 137, tuple(cpu[key].shape), generator=g, dtype=torch.int32).to(torch.uint8)
    dev = to_device(cpu)
    scores = dsa.dsa_index_score(dev["q_idx"], dev["w"], dev["k_idx"], q_idx_sf=dev["q_idx_sf"],
                                 k_idx_sf=dev["k_idx_sf"], q_per_seq=wl.q_per_seq, q_pos0=wl.q_pos0,
                                 n_valid=dev["n_valid"]).cpu().numpy()
    ch, a = oracle_chain(wl, cpu)
    for t in range(wl.T):
        n = ch.n_visible(t)
        ref = ch.scores(t)
        seq = t // wl.q_per_seq
        bound = score_error_bound(ch.q_idx(t), a["w"][t].astype(np.float64), ch.k_idx(seq, n))
        err = np.abs(scores[t, :n].astype(np.float64) - ref)
        assert np.all(err <= bound), f"t={t}: worst error/bound {np.max(err / bound):.3g}"


# ------------------------------------------------------------------------------------------------
# step 2: Top-K on identical fp32 scores (bit-exact)


def _topk_case(dsa, scores_np, K, L, q_per_seq=1, q_pos0=-1, n_valid=None):
    T = scores_np.shape[0]
    ld = dsa.ld_scores_for(L)
    buf = np.full((T, ld), np.nan, dtype=np.float32)  # entries beyond n_t must not be read
    buf[:, :L] = scores_np
    dev = torch.from_numpy(buf).cuda()
    nv = None if n_valid is None else torch.tensor(n_valid, dtype=torch.int32).cuda()
    idx = dsa.dsa_topk(dev, K, L=L, q_per_seq=q_per_seq, q_pos0=q_pos0, n_valid=nv).cpu().numpy()
    for t in range(T):
        n = oracle.visible_length(t, L, q_per_seq, q_pos0, n_valid)
        buf[t, n:] = 0  # the oracle sees only the visible prefix
        want = oracle.topk_positions(scores_np[t, :n].astype(np.float64), K)
        m = min(K, n)
        got = idx[t]
        assert np.all(got[m:] == -1), f"t={t}: padding"
        assert np.all(np.diff(got[:m]) > 0), f"t={t}: positions must be ascending"
        assert np.array_equal(np.sort(want[:m]), got[:m]), f"t={t}: index set differs"


def test_topk_random_scores(dsa):
    rng = np.random.default_rng(11)
    _topk_case(dsa, rng.standard_normal((4, 32768)).astype(np.float32) * 30 + 140, 2048, 32768)


def test_topk_heavy_ties_and_negatives(dsa):
    rng = np.random.default_rng(12)
    s = (np.round(rng.standard_normal((3, 5000)) * 3) / 4).astype(np.float32)  # few distinct values
    s[1] = -np.abs(s[1])
    s[2, ::2] = -0.0
    s[2, 1::2] = 0.0
    _topk_case(dsa, s, 700, 5000)


def test_topk_all_equal_and_tiny_k(dsa):
    s = np.full((2, 3000), 1.5, dtype=np.float32)
    _topk_case(dsa, s, 1, 3000)
    _topk_case(dsa, s, 2048, 3000)


def test_topk_n_at_and_around_k(dsa):
    rng = np.random.default_rng(13)
    s = rng.standard_normal((5, 300)).astype(np.float32)
    _topk_case(dsa, s, 100, 300, n_valid=[0, 1, 99, 100, 101])
    _topk_case(dsa, s, 300, 300)
    _topk_case(dsa, s, 4096, 300)


def test_topk_long_rows_uncached_path(dsa):
    rng = np.random.default_rng(14)
    s = rng.standard_normal((2, 70001)).astype(np.float32)
    _topk_case(dsa, s, 4096, 70001)


# rows longer than 16 x 16384 positions take the row-split path (chunks on independent CTAs)


def test_topk_row_split_random_ragged(dsa):
    rng = np.random.default_rng(21)
    s = (rng.standard_normal((3, 300001)) * 30 + 140).astype(np.float32)
    _topk_case(dsa, s, 2048, 300001, n_valid=[300001, 262145, 150000])


def test_topk_row_split_heavy_ties(dsa):
    rng = np.random.default_rng(22)
    s = (np.round(rng.standard_normal((2, 400000)) * 2) / 2).astype(np.float32)  # ~20 distinct values
    s[1] = -np.abs(s[1])
    _topk_case(dsa, s, 4096, 400000)


def test_topk_row_split_all_equal(dsa):
    s = np.full((1, 270000), -2.25, dtype=np.float32)
    _topk_case(dsa, s, 2048, 270000)
    _topk_case(dsa, s, 1, 270000)


def test_topk_row_split_rows_at_and_below_k(dsa):
    rng = np.random.default_rng(23)
    s = rng.standard_normal((4, 280000)).astype(np.float32)
    _topk_case(dsa, s, 1000, 280000, n_valid=[0, 999, 1000, 1001])


def test_topk_row_split_workspace_reuse(dsa):
    # the histograms in the workspace must be zero again after each call
    rng = np.random.default_rng(24)
    T, L, K = 2, 300000, 2048
    from top_sparse_attention_gb300 import _native

    ws_bytes = _native.lib.dsa_topk_workspace_size(T, L, K)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    for rep in range(3):
        s = (rng.standard_normal((T, L)) * (1 + rep)).astype(np.float32)
        ld = dsa.ld_scores_for(L)
        buf = np.zeros((T, ld), dtype=np.float32)
        buf[:, :L] = s
        idx = dsa.dsa_topk(torch.from_numpy(buf).cuda(), K, L=L, ws=ws).cpu().numpy()
        for t in range(T):
            want = np.sort(oracle.topk_positions(s[t].astype(np.float64), K))
            assert np.array_equal(want, idx[t]), f"rep={rep} t={t}"


def test_topk_uncached_cluster_rows(dsa):
    # more rows than the row-split path takes (T > 32): 16-CTA clusters whose slices exceed the
    # shared-memory key cache re-read their keys from L2
    rng = np.random.default_rng(25)
    s = (rng.standard_normal((33, 270001)) * 30 + 140).astype(np.float32)
    s[5] = np.round(s[5] / 8) * 8  # heavy ties in one row
    _topk_case(dsa, s, 2048, 270001)


def test_topk_many_queries(dsa):
    # 64 or more queries in one launch take fewer, fuller CTAs per query: two CTAs of 35,001
    # positions each (slices past the shared-memory key cache), and one CTA for a short row
    rng = np.random.default_rng(26)
    s = (rng.standard_normal((64, 70001)) * 30 + 140).astype(np.float32)
    s[7] = np.round(s[7] / 8) * 8  # heavy ties in one row
    _topk_case(dsa, s, 2048, 70001, n_valid=[70001 - 37 * t for t in range(64)])
    s = (np.round(rng.standard_normal((80, 5000)) * 3) / 4).astype(np.float32)
    _topk_case(dsa, s, 700, 5000)


def test_topk_causal_rows(dsa):
    rng = np.random.default_rng(15)
    s = rng.standard_normal((6, 2600)).astype(np.float32)
    _topk_case(dsa, s, 512, 2600, q_per_seq=3, q_pos0=2000)


# ------------------------------------------------------------------------------------------------
# step 3: sparse attention on identical indices


@pytest.fixture(params=["auto", "tcgen05"])
def attn_kernel(request, dsa):
    """Runs a test on the library's attention kernel and again with the tensor-memory kernel
    selected (dsa_set_attn_kernel; it takes the 576 / 512 latent row, others keep the default)."""
    from top_sparse_attention_gb300 import _native as N

    dsa.dsa_set_attn_kernel(N.DSA_ATTN_TCGEN05 if request.param == "tcgen05" else N.DSA_ATTN_AUTO)
    yield request.param
    dsa.dsa_set_attn_kernel(N.DSA_ATTN_AUTO)


def _attn_case(dsa, wl, idx_np, kv_kind, guard=True):
    cpu = synth.make_inputs(wl)
    dev = to_device(cpu)
    idx = torch.from_numpy(idx_np.astype(np.int32)).cuda()
    out, lse = dsa.dsa_sparse_attn(dev["q"], dev["kv"], idx, sm_scale=wl.sm_scale, kv_v=dev["kv_v"],
                                   kv_scale=dev["kv_scale"], D_v=wl.D_v, q_per_seq=wl.q_per_seq)
    out = out.float().cpu().numpy()
    lse = lse.cpu().numpy()
    ch, _ = oracle_chain(wl, cpu)
    worst = 0.0
    for t in range(wl.T):
        ref, ref_lse = ch.attention(t, idx_np[t], wl.D_v)
        err = float(np.max(np.abs(out[t] - ref)))
        worst = max(worst, err)
        assert err <= ATTN_TOL[kv_kind], f"t={t}: max-abs {err}"
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse[t]))
        assert np.all(np.abs(lse[t][fin] - ref_lse[fin]) <= LSE_TOL)
    if guard:
        assert worst <= ATTN_GUARD[kv_kind], f"max-abs {worst} above the regression guard"
    return worst


def _random_idx(T, K, L, seed, pad=0):
    rng = np.random.default_rng(seed)
    idx = np.stack([np.sort(rng.choice(L, size=K, replace=False)) for _ in range(T)])
    if pad:
        idx[:, K - pad:] = -1
    return idx


@pytest.mark.parametrize("kv", ["bf16", "fp8", "fp8_t128"])
@pytest.mark.parametrize("K,pad", [(2048, 0), (2048, 37), (100, 0), (64, 64)])
def test_sparse_attn_mla(dsa, attn_kernel, kv, K, pad):
    base = {"bf16": "decode_b8_l32k_bf16", "fp8": "decode_b8_l32k_mxfp8", "fp8_t128": "decode_b8_l32k_mxfp8_kvt128"}[kv]
    wl = synth.small_workload(base, T=3, L=4000, K=K)
    _attn_case(dsa, wl, _random_idx(3, K, 4000, K + pad, pad), kv)


def test_sparse_attn_head_groups_and_ragged_heads(dsa):
    wl = synth.small_workload("decode_b8_l32k_bf16", T=2, L=3000, K=512, H=20)
    _attn_case(dsa, wl, _random_idx(2, 512, 3000, 5), "bf16")


def test_sparse_attn_small_head_separate_v(dsa):
    wl = synth.WORKLOADS["tiny_decode_l2k"]
    _attn_case(dsa, wl, _random_idx(1, 64, 2048, 6), "bf16")


def test_sparse_attn_repeated_rows(dsa):
    wl = synth.small_workload("decode_b8_l32k_bf16", T=2, L=500, K=256)
    idx = np.tile(np.arange(8), (2, 32))
    # each row's bf16-rounded probability repeats 32 times, so its rounding error does not average
    # out as it does over distinct rows: only the tolerance applies, not the tighter guard
    _attn_case(dsa, wl, idx, "bf16", guard=False)


@pytest.mark.parametrize("D,D_v,tiled", [(576, 512, False), (576, 512, True), (64, 64, False)])
def test_sparse_attn_fp8_rows_widen_exactly_for_every_code(dsa, attn_kernel, D, D_v, tiled):
    # One selected row: its softmax weight is exactly 1, so with power-of-two scales the output is
    # each value column's E4M3 value times its scale, exactly representable in bf16.  The rows
    # cycle through all 254 finite codes (subnormals and both zeros included) at shifted columns;
    # with 64-wide rows the eight rows together hold every code.
    L = 8
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    codes = np.stack([np.resize(np.roll(finite, -37 * r), D) for r in range(L)])
    assert len(set(codes[:, :D_v].ravel())) == 254
    rng = np.random.default_rng(3)
    shape = (1, L, (D + 127) // 128) if tiled else (1, L)
    sc = np.ldexp(1.0, rng.integers(-7, 6, shape)).astype(np.float32)
    rows = list(range(L))
    T = len(rows)
    q = torch.from_numpy(rng.standard_normal((T, 16, D))).to(torch.bfloat16)
    idx = torch.tensor([[r] for r in rows], dtype=torch.int32)
    out, lse = dsa.dsa_sparse_attn(q.cuda(), torch.from_numpy(codes).reshape(1, L, D).cuda(), idx.cuda(),
                                   sm_scale=0.1, kv_scale=torch.from_numpy(sc).cuda(), D_v=D_v, q_per_seq=T)
    out = out.float().cpu().numpy()
    for t, r in enumerate(rows):
        v = oracle.e4m3_to_f64(codes[r, :D_v])
        s = np.repeat(sc[0, r], 128)[:D_v] if tiled else sc[0, r]
        want = np.broadcast_to(v * s, (16, D_v))
        assert np.array_equal(out[t], want), f"t={t}: {np.flatnonzero(out[t][0] != want[0])[:8]}"
    assert torch.isfinite(lse).all()


def test_sparse_attn_small_fp8_rows(dsa):
    # E4M3 rows of 64 with V = the same row (each warp owns 16 value columns, half a 32-column
    # chunk of the row), against the oracle
    wl = synth.small_workload("decode_b8_l32k_mxfp8", T=3, L=1500, K=300, H=20, D_qk=64, D_v=64)
    _attn_case(dsa, wl, _random_idx(3, 300, 1500, 9, pad=7), "fp8")


def test_sparse_attn_out_of_range_index_is_skipped_and_recorded(dsa):
    wl = synth.small_workload("decode_b8_l32k_bf16", T=1, L=500, K=128)
    cpu = synth.make_inputs(wl)
    dev = to_device(cpu)
    good = _random_idx(1, 128, 500, 7)
    bad = good.copy()
    bad[0, 5] = 500          # one past the end: checked by the kernel, never read
    bad[0, 9] = -7
    dsa.dsa_get_device_error()  # clear
    out, _ = dsa.dsa_sparse_attn(dev["q"], dev["kv"], torch.from_numpy(bad.astype(np.int32)).cuda(),
                                 sm_scale=wl.sm_scale)
    assert dsa.dsa_get_device_error() == 1
    ch, _ = oracle_chain(wl, cpu)
    ref, _ = ch.attention(0, np.where((bad[0] >= 0) & (bad[0] < 500), bad[0], -1), wl.D_v)
    assert np.max(np.abs(out[0].float().cpu().numpy() - ref)) <= ATTN_TOL["bf16"]


# ------------------------------------------------------------------------------------------------
# fused chain


_check_chain = check_chain


@pytest.mark.parametrize("name", ["tiny_decode_l2k", "decode_b8_l32k_bf16", "decode_b8_l32k_mxfp8",
                                  "decode_b8_varlen_bf16", "decode_b8_l32k_mxfp8_kvt128"])
def test_chain_full_decode_workloads(dsa, name):
    wl = synth.WORKLOADS[name]
    _check_chain(dsa, wl, synth.make_inputs(wl))


def test_chain_long_context_decode(dsa):
    wl = synth.WORKLOADS["decode_b1_l1m_mxfp8"]
    _check_chain(dsa, wl, synth.make_inputs(wl))


def test_chain_prefill_chunk_sampled_rows(dsa):
    # 128 seeded rows of the 4096-query chunk, always with the first and last query (the
    # shortest and longest causal prefixes) and both ends of a four-query scoring group
    wl = synth.WORKLOADS["prefill_t4096_l128k_bf16"]
    rng = np.random.default_rng(16)
    rows = {0, 1, 2, 3, 2047, 2048, 4092, 4095}
    while len(rows) < 128:
        rows.add(int(rng.integers(0, 4096)))
    _check_chain(dsa, wl, synth.make_inputs(wl), queries=sorted(rows))


@pytest.mark.parametrize("case", ["short_context", "varlen", "small_causal", "ragged_fp8"])
def test_chain_edge_cases(dsa, case):
    if case == "short_context":   # L < K: every position then -1
        wl = synth.small_workload("decode_b8_l32k_bf16", T=2, L=100, K=256)
        cpu = synth.make_inputs(wl)
    elif case == "varlen":        # an empty query, one below K, one above
        wl = synth.small_workload("decode_b8_l32k_bf16", T=3, L=3000, K=512)
        cpu = synth.make_inputs(wl, n_valid=[0, 300, 2999])
    elif case == "small_causal":  # prefix shorter than K for the first queries
        wl = synth.small_workload("prefill_t4096_l128k_bf16", T=12, q_per_seq=12, L=700, K=256, q_pos0=250)
        cpu = synth.make_inputs(wl)
    else:
        wl = synth.small_workload("decode_b8_l32k_mxfp8", T=3, L=2345, K=333)
        cpu = synth.make_inputs(wl)
    _check_chain(dsa, wl, cpu)
    if case == "varlen":
        dev = to_device(cpu)
        call = dsa.call_from_tensors(dev, K=wl.K, sm_scale=wl.sm_scale)
        out, lse, idx = call()
        assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
        assert torch.all(idx[0] == -1)


def test_chain_empty_batch_is_a_no_op(dsa):
    wl = synth.small_workload("decode_b8_l32k_bf16", T=1, L=256, K=64)
    dev = to_device(synth.make_inputs(wl))
    dev = {k: (v[:0] if (v is not None and k in ("q_idx", "w", "q")) else v) for k, v in dev.items()}
    dev["k_idx"] = dev["k_idx"][:0]
    dev["kv"] = dev["kv"][:0]
    out, lse, idx = dsa.call_from_tensors(dev, K=64, sm_scale=wl.sm_scale)()
    assert out.shape[0] == 0 and idx.shape[0] == 0


@pytest.mark.parametrize("name", ["decode_b8_l32k_bf16", "decode_b8_l32k_mxfp8"])
def test_chain_repeat_calls_on_one_workspace_are_identical(dsa, name):
    # The workspace carries score histograms between kernels and every call must leave them at
    # zero: a call on a workspace that already served other inputs must give exactly what the same
    # call gives on a fresh zero-filled workspace, and the score-histogram region (after the
    # scores, dsa.h's fused-chain layout) must be all zero after each call.
    wl = synth.small_workload(name, T=3, L=5000, K=700)
    dev_a = to_device(synth.make_inputs(wl))
    dev_b = to_device(synth.make_inputs(wl, seed_offset=1))
    call_a = dsa.call_from_tensors(dev_a, K=wl.K, sm_scale=wl.sm_scale)
    ws = call_a.ws
    hist_lo = -(-(wl.T * dsa.ld_scores_for(wl.L) * 4) // 256) * 256
    hist = ws[hist_lo:hist_lo + wl.T * 4096 * 4]
    out1, lse1, idx1 = [x.clone() for x in call_a()]
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(hist)) == 0
    out2, lse2, idx2 = [x.clone() for x in call_a()]
    assert torch.equal(idx1, idx2) and torch.equal(out1, out2) and torch.equal(lse1, lse2)
    # other inputs on the used workspace vs. on a fresh one
    used = dsa.call_from_tensors(dev_b, K=wl.K, sm_scale=wl.sm_scale, ws=ws)
    fresh = dsa.call_from_tensors(dev_b, K=wl.K, sm_scale=wl.sm_scale)
    got = [x.clone() for x in used()]
    want = fresh()
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(hist)) == 0
    for g, w_ in zip(got, want):
        assert torch.equal(g, w_)
    assert not torch.equal(got[2], idx1)  # the second inputs select other positions


# ------------------------------------------------------------------------------------------------
# element-wise scores at the full decode sizes (the persistent unit walk over many tiles per CTA)


def test_index_score_full_size_bf16_every_position(dsa):
    wl = synth.WORKLOADS["decode_b8_l32k_bf16"]
    cpu = synth.make_inputs(wl)
    dev = to_device(cpu)
    scores = dsa.dsa_index_score(dev["q_idx"], dev["w"], dev["k_idx"]).cpu().numpy()
    ch, a = oracle_chain(wl, cpu)
    for t in range(wl.T):
        ref = ch.scores(t)
        bound = score_error_bound(ch.q_idx(t), a["w"][t].astype(np.float64), ch.k_idx(t, wl.L))
        err = np.abs(scores[t, :wl.L].astype(np.float64) - ref)
        assert np.all(err <= bound), f"t={t}: worst error/bound {np.max(err / bound):.3g}"


def test_index_score_full_size_mxfp8_1m_sampled_positions(dsa):
    # L = 1,048,576 MXFP8: 8192 seeded positions plus both ends and the edges of every 65,536-row
    # block, each checked against the oracle's score of that position alone
    wl = synth.WORKLOADS["decode_b1_l1m_mxfp8"]
    cpu = synth.make_inputs(wl)
    dev = {k: cpu[k].cuda() for k in ("q_idx", "q_idx_sf", "w", "k_idx", "k_idx_sf")}
    scores = dsa.dsa_index_score(dev["q_idx"], dev["w"], dev["k_idx"], q_idx_sf=dev["q_idx_sf"],
                                 k_idx_sf=dev["k_idx_sf"]).cpu().numpy()[0]
    a = synth.to_numpy_bits({k: cpu[k] for k in ("q_idx", "q_idx_sf", "w", "k_idx", "k_idx_sf")})
    rng = np.random.default_rng(41)
    edges = [e + d for e in range(0, wl.L + 1, 1 << 16) for d in (-1, 0) if 0 <= e + d < wl.L]
    pos = np.unique(np.concatenate([rng.integers(0, wl.L, 8192), [0, 127, 128, wl.L - 1], edges]))
    q = oracle.dequant_mxfp8(a["q_idx"][0], a["q_idx_sf"][0])
    w = a["w"][0].astype(np.float64)
    k = oracle.dequant_mxfp8(a["k_idx"][0, pos], a["k_idx_sf"][0, pos])
    ref = oracle.index_scores(q, w, k)
    bound = score_error_bound(q, w, k)
    err = np.abs(scores[pos].astype(np.float64) - ref)
    assert np.all(err <= bound), f"worst error/bound {np.max(err / bound):.3g}"
