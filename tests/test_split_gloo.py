"""The split-context decode protocol on CPU ranks (gloo): each rank holds one slice of the context and
runs `split_decode_rank`, which exchanges the (score, position) candidates and the partial attention
outputs with all_gather.  This test runs without a GPU, so the oracle stands in for the per-slice
kernel steps, the merge and the combine; what is under test is the plan, the buffers and the two
exchanges.  The ranks' common result must match the oracle's chain over the whole context."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class _OracleSlice:
    """The oracle in place of SliceSteps for slice g (same pairs / partial methods)."""

    def __init__(self, oracle, synth, split, plan, g, cpu, wl):
        self.oracle, self.plan, self.g, self.wl = oracle, plan, g, wl
        sl = dict(cpu)
        sl.update(split.slice_caches(cpu, plan, g))
        a = synth.to_numpy_bits(sl)
        a["n_valid"] = None if wl.lengths is None else np.array(plan.visible(wl.lengths, g))
        self.ch = oracle.Chain(a, L=plan.length(g), K=wl.K, q_per_seq=1, q_pos0=-1, idx_dtype=wl.idx_dtype,
                               kv_dtype=wl.kv_dtype, sm_scale=wl.sm_scale)

    def pairs(self, q_idx, q_idx_sf, w, cand_pos, cand_scores):
        lo = self.plan.lo(self.g)
        for t in range(self.wl.T):
            s = self.ch.scores(t)
            local = self.oracle.topk_positions(s, self.wl.K)
            sel = np.sort(local[local >= 0])  # ascending, as dsa_topk_pairs writes them
            cand_pos[t].fill_(-1)
            cand_scores[t].zero_()
            cand_pos[t, : sel.size] = torch.from_numpy(sel + lo)
            cand_scores[t, : sel.size] = torch.from_numpy(s[sel].astype(np.float32))

    def partial(self, q, idx, o_part, lse_part):
        lo, n = self.plan.lo(self.g), self.plan.length(self.g)
        for t in range(self.wl.T):
            row = idx[t].numpy().astype(np.int64)
            mine = np.where((row >= lo) & (row < lo + n), row - lo, -1)
            out, lse = self.ch.attention(t, mine, self.wl.D_v)
            o_part[t] = torch.from_numpy(out)
            lse_part[t] = torch.from_numpy(lse)


def _rank_main(rank, world, port, case, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import synth
    from top_sparse_attention_gb300 import split

    base, kw = case
    wl = synth.small_workload(base, **kw)
    cpu = synth.make_inputs(wl)
    plan = split.SplitPlan.even(wl.L, world)
    steps = _OracleSlice(oracle, synth, split, plan, rank, cpu, wl)

    def merge(cs, cp):
        G, T, K = cp.shape
        rows = [oracle.merge_candidates(cs[:, t].reshape(-1).numpy(), cp[:, t].reshape(-1).numpy(), wl.K)
                for t in range(T)]
        return torch.from_numpy(np.stack(rows).astype(np.int32))

    def combine(o, l):
        res = [oracle.combine_partials(o[:, t].numpy(), l[:, t].numpy()) for t in range(o.shape[1])]
        return torch.from_numpy(np.stack([r[0] for r in res])), torch.from_numpy(np.stack([r[1] for r in res]))

    res, lse, idx = split.split_decode_rank(steps, cpu["q_idx"], cpu["q_idx_sf"], cpu["w"], cpu["q"], K=wl.K, H=wl.H,
                                             D_v=wl.D_v, merge=merge, combine=combine)
    out[rank] = (res.numpy(), lse.numpy(), idx.numpy(), plan.bounds)
    dist.destroy_process_group()


CASES = [
    (2, ("decode_b8_l32k_bf16", dict(T=2, L=1000, K=100))),
    (3, ("decode_b8_l32k_mxfp8", dict(T=2, L=1100, K=64, lengths=(1100, 700)))),
]


@pytest.mark.parametrize("world,case", CASES)
def test_split_decode_ranks_exchange_candidates_and_partials(world, case):
    import oracle
    import synth
    from top_sparse_attention_gb300 import build

    build.build()  # the ranks import the package's binding, which loads the library

    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, case, out), nprocs=world, start_method="spawn", join=True)
    base, kw = case
    wl = synth.small_workload(base, **kw)
    cpu = synth.make_inputs(wl)
    a = synth.to_numpy_bits(cpu)
    ch = oracle.Chain(a, L=wl.L, K=wl.K, q_per_seq=1, q_pos0=-1, idx_dtype=wl.idx_dtype, kv_dtype=wl.kv_dtype,
                      sm_scale=wl.sm_scale)
    assert len(out[0][3]) == world + 1
    for r in range(1, world):  # every rank returns the same result
        for x, y in zip(out[0][:3], out[r][:3]):
            np.testing.assert_array_equal(x, y)
    res, lse, idx, _ = out[0]
    for t in range(wl.T):
        oracle.parity.check_topk(idx[t], ch.scores(t), wl.K)
        want = np.sort(oracle.topk_positions(ch.scores(t), wl.K))
        want = np.concatenate([want[want >= 0], want[want < 0]])
        np.testing.assert_array_equal(idx[t], want)  # slices in order: ascending positions
        ref, ref_lse = ch.attention(t, idx[t], wl.D_v)
        np.testing.assert_allclose(res[t], ref, rtol=0, atol=1e-6)   # fp32 partials exchanged
        np.testing.assert_allclose(lse[t], ref_lse, rtol=0, atol=1e-5)


# ------------------------------------------------------------------------------------------------
# context-parallel prefill with zigzag segments


def test_zigzag_segments_balance_the_causal_work():
    from top_sparse_attention_gb300 import split

    for G in (1, 2, 4, 8):
        segs = [split.zigzag_segments(4096, G, g) for g in range(G)]
        covered = sorted(x for s in segs for a, b in s for x in range(a, b))
        assert covered == list(range(4096))  # every query exactly once
        work = [split.zigzag_work(4096, G, g, 126976) for g in range(G)]
        assert max(work) == min(work)
    with pytest.raises(ValueError):
        split.zigzag_segments(100, 3, 0)


def _prefill_rank_main(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import synth
    from top_sparse_attention_gb300 import split

    wl = synth.small_workload("prefill_t4096_l128k_bf16", T=16, q_per_seq=16, L=700, K=128, q_pos0=600)
    cpu = synth.make_inputs(wl)
    ch = oracle.Chain(synth.to_numpy_bits(cpu), L=wl.L, K=wl.K, q_per_seq=wl.q_per_seq, q_pos0=wl.q_pos0,
                      idx_dtype=wl.idx_dtype, kv_dtype=wl.kv_dtype, sm_scale=wl.sm_scale)
    seen = []

    def run_segment(a, b):  # the oracle in place of this rank's dsa_prefill on queries [a, b)
        seen.append((a, b))
        rows = [oracle.chain_query(ch, t, wl.D_v) for t in range(a, b)]
        return (torch.from_numpy(np.stack([r["out"] for r in rows])), torch.from_numpy(np.stack([r["lse"] for r in rows])),
                torch.from_numpy(np.stack([r["idx"] for r in rows])))

    o, l, i = split.zigzag_prefill_rank(run_segment, wl.T)
    out[rank] = (o.numpy(), l.numpy(), i.numpy(), seen)
    dist.destroy_process_group()


def test_zigzag_prefill_ranks_gather_rows_back_in_query_order():
    import oracle
    import synth
    from top_sparse_attention_gb300 import build

    build.build()
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_prefill_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0][3] == [(0, 4), (12, 16)] and out[1][3] == [(4, 8), (8, 12)]
    wl = synth.small_workload("prefill_t4096_l128k_bf16", T=16, q_per_seq=16, L=700, K=128, q_pos0=600)
    ch = oracle.Chain(synth.to_numpy_bits(synth.make_inputs(wl)), L=wl.L, K=wl.K, q_per_seq=wl.q_per_seq,
                      q_pos0=wl.q_pos0, idx_dtype=wl.idx_dtype, kv_dtype=wl.kv_dtype, sm_scale=wl.sm_scale)
    for r in range(world):
        o, l, i, _ = out[r]
        for t in range(wl.T):
            want = oracle.chain_query(ch, t, wl.D_v)
            np.testing.assert_array_equal(i[t], want["idx"])
            np.testing.assert_array_equal(o[t], want["out"])
            np.testing.assert_array_equal(l[t], want["lse"])
