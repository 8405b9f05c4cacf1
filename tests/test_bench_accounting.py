"""Host logic of the measurement: the algorithmic bytes and FLOPs that the roofline fractions
divide by, and the rule that a committed ncu traffic figure is reported only for the kernel source
it was taken on.

The expected figures are the per-query sums of the compulsory reads and writes, written out term
by term below.  Each term is one array of the method: indexer keys (+ E8M0 bytes), query-side
indexer inputs, the K gathered latent rows (+ scales), and q plus the output.  None of them comes
from the code under test.
"""
import bench
import synth


def _wl(name):
    return synth.WORKLOADS[name]


def test_bytes_per_query_match_the_closed_forms():
    # tiny decode: L = 2048 keys of 64 bf16, 4 heads; K = 64 rows of separate K and V (64 bf16 each)
    tiny = 2048 * 64 * 2 + (4 * 64 * 2 + 4 * 4) + 64 * (64 + 64) * 2 + (64 * 2 + 64 * 2)
    assert tiny == 279_312
    # B = 8, L = 32K, bf16: keys 32768 x 128 x 2; q_idx 64 x 128 x 2 + w 64 x 4; 2048 rows of 1152 B;
    # q 16 x 576 x 2 + out 16 x 512 x 2
    bf16 = 32768 * 128 * 2 + (64 * 128 * 2 + 64 * 4) + 2048 * 1152 + (16 * 576 * 2 + 16 * 512 * 2)
    assert bf16 == 10_799_360
    # the same with MXFP8 keys (+ 4 E8M0 bytes per key and per query head) and E4M3 rows + fp32 scale
    mx = (32768 * 128 + 32768 * 4) + (64 * 128 + 64 * 4 + 64 * 4) + (2048 * 576 + 2048 * 4) + 34_816
    assert mx == 5_556_736
    # one query over L = 2^20 positions, MXFP8 + FP8
    l1m = (2**20 * 128 + 2**20 * 4) + (64 * 128 + 64 * 4 + 64 * 4) + (2048 * 576 + 2048 * 4) + 34_816
    assert l1m == 139_643_392
    # tiled KV scales: five fp32 per gathered row instead of one
    t128 = mx + 2048 * 4 * 4
    for name, want in (("tiny_decode_l2k", tiny), ("decode_b8_l32k_bf16", bf16), ("decode_b8_l32k_mxfp8", mx),
                       ("decode_b1_l1m_mxfp8", l1m), ("decode_b8_l32k_mxfp8_kvt128", t128)):
        assert bench.bytes_per_query(_wl(name)) == want, name


def test_step_bytes_count_each_query_own_visible_length():
    wl = _wl("decode_b8_varlen_bf16")
    want = 0
    for n in wl.lengths:
        rows = min(wl.K, n)
        want += n * 128 * 2 + (64 * 128 * 2 + 64 * 4) + rows * 1152 + 34_816
    assert bench.step_bytes(wl) == want
    wl = _wl("decode_b8_l32k_bf16")
    assert bench.step_bytes(wl) == 8 * 10_799_360


def test_index_score_bytes_and_flops():
    wl = _wl("decode_b8_l32k_bf16")
    # keys + q_idx + w read, fp32 scores written, per query
    assert bench.index_score_bytes(wl, 8) == 8 * (32768 * 256 + 64 * 256 + 64 * 4 + 32768 * 4)
    wl = _wl("decode_b8_l32k_mxfp8")
    assert bench.index_score_bytes(wl, 8) == 8 * (32768 * 132 + 64 * 132 + 64 * 4 + 32768 * 4)
    # causal prefill: query t at position 126976 + t sees 126977 + t positions
    wl = _wl("prefill_t4096_l128k_bf16")
    pairs = sum(126977 + t for t in range(4096))
    assert pairs == 528_484_352
    assert bench.index_score_flops(wl) == 2 * 64 * 128 * pairs


def test_traffic_is_reported_only_for_the_profiled_source(tmp_path, monkeypatch):
    src = tmp_path / "top_sparse_attention_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "index_score.cu").write_text("// kernel revision A\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    (tmp_path / "profiles" / "index_score_w.md").write_text(
        f"source_sha256_16: {h}\ndram_bytes_per_launch: 12345\n")
    assert bench.profiled_traffic("w") == 12345
    assert bench.profiled_traffic("other") is None  # no summary for this workload
    (src / "index_score.cu").write_text("// kernel revision B\n")
    assert bench.profiled_traffic("w") is None  # the kernel changed since the capture



def test_reference_arm_prints_the_gpu_arms_config(capsys, monkeypatch):
    """The oracle arm's line carries the same config, metric, unit and direction as the GPU arm's,
    with its own cpu_baseline and an e2e of no copies."""
    import argparse
    import json

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    wl = _wl("tiny_decode_l2k")
    args = argparse.Namespace(gpus=1, inflight=6, steps=3, warmup=3, impl="reference", workload=wl.name,
                              sets=0, no_graph=False, no_cpu_baseline=False, cpu_seconds=1.0, attn_kernel="auto")
    assert bench.run_reference(args, wl) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.run_config(args, wl)
    assert (line["metric"], line["unit"], line["higher_is_better"]) == (bench.METRIC, "queries/s", True)
    assert line["steps"] == 3 and line["warmup"] == 3 and line["value"] > 0
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"] == {"value": line["value"], "unit": "queries/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
