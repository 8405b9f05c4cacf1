"""Pins for the oracle: hand-worked fixtures, closed forms, library routines that are independent
of the oracle's code, invariants and brute force on tiny inputs.  CPU only."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from synth import inputs as synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------------------------------------
# stored formats


def test_e4m3_hand_values():
    g = _golden("hand_worked_quant.json")
    got = oracle.e4m3_to_f64(np.array(g["e4m3_codes"], dtype=np.uint8))
    np.testing.assert_array_equal(got, np.array(g["e4m3_values"]))
    assert math.copysign(1.0, got[-1]) == -1.0  # 0x80 is -0


def test_e4m3_all_codes_match_torch_cast():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.e4m3_to_f64(codes), ref)


def test_e4m3_rejects_nan():
    with pytest.raises(ValueError):
        oracle.e4m3_to_f64(np.array([0x7F], dtype=np.uint8))
    with pytest.raises(ValueError):
        oracle.e4m3_to_f64(np.array([0xFF], dtype=np.uint8))


def test_e8m0_hand_values_and_nan():
    g = _golden("hand_worked_quant.json")
    got = oracle.e8m0_to_f64(np.array(g["e8m0_codes"], dtype=np.uint8))
    np.testing.assert_array_equal(got, np.ldexp(1.0, np.array(g["e8m0_values_log2"])))
    with pytest.raises(ValueError):
        oracle.e8m0_to_f64(np.array([255], dtype=np.uint8))


def test_bf16_matches_torch():
    x = torch.randn(4096, generator=torch.Generator().manual_seed(3)) * 100
    b = x.to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(bits), b.to(torch.float64).numpy())


def test_mxfp8_dequant_unit_scale_is_plain_e4m3_and_scale_bump_doubles_group():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 0x7F, size=(3, 96)).astype(np.uint8)  # positive, no NaN
    sf = np.full((3, 3), 127, dtype=np.uint8)
    plain = oracle.e4m3_to_f64(codes)
    np.testing.assert_array_equal(oracle.dequant_mxfp8(codes, sf), plain)
    sf2 = sf.copy()
    sf2[1, 2] += 1
    d2 = oracle.dequant_mxfp8(codes, sf2)
    np.testing.assert_array_equal(d2[1, 64:96], 2 * plain[1, 64:96])
    np.testing.assert_array_equal(d2[1, :64], plain[1, :64])
    np.testing.assert_array_equal(d2[[0, 2]], plain[[0, 2]])


def test_mx_and_fp8_hand_scores():
    g = _golden("hand_worked_quant.json")
    q_codes = np.zeros((1, 32), dtype=np.uint8)
    q_codes[0, :2] = g["mx_q_codes_first2"]
    q = oracle.dequant_mxfp8(q_codes, np.array([[g["mx_q_sf"]]], dtype=np.uint8))
    k_codes = np.zeros((2, 32), dtype=np.uint8)
    k_codes[:, :2] = np.array(g["mx_k_rows_first2"], dtype=np.uint8)
    k = oracle.dequant_mxfp8(k_codes, np.array(g["mx_k_sf"], dtype=np.uint8)[:, None])
    s = oracle.index_scores(q, np.array([g["mx_w"]]), k)
    np.testing.assert_array_equal(s, np.array(g["expect_mx_scores"]))
    kv = oracle.dequant_fp8_rows(np.array(g["fp8_kv_codes"], dtype=np.uint8)[:, None],
                                 np.array(g["fp8_kv_scales"], dtype=np.float32))
    np.testing.assert_array_equal(kv[:, 0], np.array(g["expect_fp8_kv_values"]))


def test_synth_encoders_roundtrip_through_oracle_decoders():
    # inputs exactly representable as E4M3 * 2^e with a group max of 2^k round-trip exactly
    rng = np.random.default_rng(0)
    vals = oracle.e4m3_to_f64(rng.integers(0, 0x70, size=(4, 64)).astype(np.uint8))
    vals[:, 0] = 256.0
    vals[:, 32] = 256.0  # group amax 256 -> shared exponent 0
    codes, sf = synth.encode_mxfp8(torch.from_numpy(vals).float())
    back = oracle.dequant_mxfp8(codes.numpy(), sf.numpy())
    np.testing.assert_array_equal(back, vals)
    # random N(0,1): elementwise error within E4M3 rounding (2^-4 relative) plus saturation of the
    # few values scaled into (448, 512)
    x = torch.randn(64, 128, generator=torch.Generator().manual_seed(1))
    codes, sf = synth.encode_mxfp8(x)
    back = oracle.dequant_mxfp8(codes.numpy(), sf.numpy())
    xs = x.double().numpy()
    scale = np.repeat(oracle.e8m0_to_f64(sf.numpy()), 32, axis=-1)
    # E4M3 subnormals (scaled magnitude < 2^-6) have an absolute half-spacing of 2^-10 * scale
    bound = np.maximum(np.abs(xs) * 2.0 ** -4, np.maximum(np.abs(xs) - 448 * scale, 0)) + 2.0 ** -10 * scale
    assert np.all(np.abs(back - xs) <= bound + 1e-12)
    codes, rs = synth.encode_fp8_rows(x)
    back = oracle.dequant_fp8_rows(codes.numpy(), rs.numpy())
    assert np.all(np.abs(back - xs) <= np.abs(xs) * 2.0 ** -4 + 2.0 ** -10 * rs.numpy()[:, None] + 1e-12)


# ------------------------------------------------------------------------------------------------
# online quantisation (the cache writer): values -> stored formats


def test_e4m3_encode_round_trips_every_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_to_f64(codes)), codes)


def test_e4m3_encode_matches_torch_cast_on_random_values_and_ties():
    rng = np.random.default_rng(7)
    pos = np.sort(oracle.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = (pos[:-1] + pos[1:]) / 2  # exact midpoints between neighbouring codes: ties to even
    x = np.concatenate([rng.uniform(-440, 440, 4000), rng.standard_normal(4000),
                        rng.standard_normal(2000) * 2.0 ** -8, mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(x.astype(np.float64)), ref)


def test_e4m3_encode_saturates_and_keeps_the_sign_of_zero():
    got = oracle.e4m3_encode([448.0, 449.0, 464.0, 500.0, 1e9, -1e9, -0.0, -2.0 ** -11, 2.0 ** -11])
    np.testing.assert_array_equal(got, [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x80, 0x80, 0x00])


def test_online_quant_hand_worked():
    g = _golden("hand_worked_online_quant.json")
    codes, sf = oracle.quantize_mxfp8(np.array(g["mx_groups"]).reshape(1, -1))
    np.testing.assert_array_equal(sf[0], g["expect_mx_sf"])
    np.testing.assert_array_equal(codes.reshape(4, 32)[:, :4], g["expect_mx_codes_first4"])
    assert np.all(codes.reshape(4, 32)[:, 4:] == 0)
    codes, s = oracle.quantize_fp8_rows(np.array(g["fp8_rows"]))
    np.testing.assert_array_equal(s[:2], g["expect_fp8_scales_exact"])
    assert s[2] == np.float32(3.0) / np.float32(448.0)
    np.testing.assert_array_equal(codes, g["expect_fp8_codes"])


def _torch_mxfp8(x64):
    """The same OCP MX rule from torch primitives: frexp for the exponent, the float8 cast for
    the elements (after saturating to 448)."""
    x = torch.from_numpy(x64).reshape(x64.shape[0], -1, 32)
    amax = x.abs().amax(-1)
    _, e = torch.frexp(amax)  # amax = m * 2^e, m in [0.5, 1): floor(log2 amax) = e - 1
    shared = torch.where(amax > 0, (e - 1 - 8).clamp(-127, 127), torch.zeros_like(e))
    scaled = torch.ldexp(x, -shared[..., None].to(torch.float64)).clamp(-448, 448)
    codes = scaled.to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).reshape(x64.shape)
    return codes.numpy(), (shared + 127).to(torch.uint8).numpy()


def test_quantize_mxfp8_matches_torch_and_scales_by_powers_of_two():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((64, 128)) * np.ldexp(1.0, rng.integers(-30, 30, (64, 4))).repeat(32, 1)
    x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()  # bf16 inputs, as cached
    x[3, 32:64] = 0.0  # an all-zero group
    codes, sf = oracle.quantize_mxfp8(x)
    tc, tsf = _torch_mxfp8(x)
    np.testing.assert_array_equal(codes, tc)
    np.testing.assert_array_equal(sf, tsf)
    assert sf[3, 1] == 127 and np.all(codes[3, 32:64] == 0)
    # scaling a group by 2^k moves its exponent byte by k and leaves the element codes alone
    c2, s2 = oracle.quantize_mxfp8(x * 8.0)
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(s2.astype(int) - sf.astype(int), np.where(sf == 127, np.where(np.abs(x).reshape(64, 4, 32).max(-1) > 0, 3, 0), 3))
    # dequantised error: E4M3 rounding (half a step, <= amax / 32) or saturation (< amax / 8)
    back = oracle.dequant_mxfp8(codes, sf)
    amax = np.abs(x).reshape(64, 4, 32).max(-1).repeat(32, 1)
    assert np.all(np.abs(back - x) <= amax / 8 + 1e-300)


def test_quantize_fp8_rows_matches_torch_fp32():
    rng = np.random.default_rng(9)
    x = torch.from_numpy(rng.standard_normal((50, 576)) * np.ldexp(1.0, rng.integers(-10, 10, (50, 1))))
    x = x.to(torch.bfloat16).to(torch.float32)
    x[7] = 0.0
    codes, s = oracle.quantize_fp8_rows(x.double().numpy())
    amax = x.abs().amax(-1)
    ts = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    tq = (x / ts[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    np.testing.assert_array_equal(s, ts.numpy())
    np.testing.assert_array_equal(codes, tq.numpy())
    assert s[7] == 1.0 and np.all(codes[7] == 0)


def test_fp8_tiles_reduce_to_rows_and_match_torch():
    rng = np.random.default_rng(10)
    x = torch.from_numpy(rng.standard_normal((40, 576)) * np.ldexp(1.0, rng.integers(-8, 8, (40, 5))).repeat(128, 1)[:, :576])
    x = x.to(torch.bfloat16).to(torch.float32)
    x[3, 128:256] = 0.0  # an all-zero tile
    codes, s = oracle.quantize_fp8_tiles(x.double().numpy())
    assert s.shape == (40, 5) and s[3, 1] == 1.0 and np.all(codes[3, 128:256] == 0)
    # torch restatement, tile by tile (the last tile is 64 wide)
    for t0 in range(0, 576, 128):
        xt = x[:, t0:t0 + 128]
        amax = xt.abs().amax(-1)
        ts = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
        tq = (xt / ts[:, None]).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        np.testing.assert_array_equal(s[:, t0 // 128], ts.numpy())
        np.testing.assert_array_equal(codes[:, t0:t0 + 128], tq.numpy())
    # one scale repeated over all tiles of a row is the per-row format
    row_s = np.abs(rng.standard_normal(40)).astype(np.float32) + 0.5
    np.testing.assert_array_equal(oracle.dequant_fp8_tiles(codes, np.repeat(row_s[:, None], 5, 1)),
                                  oracle.dequant_fp8_rows(codes, row_s))
    # dequantised error within E4M3 rounding (1/16 of the tile's max) or saturation
    back = oracle.dequant_fp8_tiles(codes, s)
    tmax = np.repeat(np.maximum.reduceat(np.abs(x.double().numpy()), np.arange(0, 576, 128), axis=1), 128, 1)[:, :576]
    assert np.all(np.abs(back - x.double().numpy()) <= tmax / 16 + 1e-300)


# ------------------------------------------------------------------------------------------------
# indexer scores


def test_hand_worked_chain():
    g = _golden("hand_worked_chain.json")
    s = oracle.index_scores(np.array(g["q_idx"]), np.array(g["w"]), np.array(g["k_idx"]))
    np.testing.assert_array_equal(s, np.array(g["expect_scores"]))
    idx = oracle.topk_positions(s, g["K"])
    assert sorted(idx.tolist()) == g["expect_topk_set"]
    kk = np.array(g["kv_k"])[idx]
    vv = np.array(g["kv_v"])[idx]
    out, lse = oracle.sparse_attention(np.array(g["q"]), kk, vv, math.log(3.0))
    np.testing.assert_allclose(out, np.array(g["expect_out"]), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, [math.log(7.0)], rtol=0, atol=1e-12)


def test_scores_tiny_closed_form():
    # H_idx = 1, w = 1, d = 2: the score is max(0, q.k)
    q = np.array([[0.5, -2.0]])
    k = np.array([[2.0, 0.25], [1.0, 1.0], [-4.0, -1.0], [0.0, 0.0]])
    np.testing.assert_array_equal(oracle.index_scores(q, np.array([1.0]), k), [0.5, 0.0, 0.0, 0.0])


def test_scores_one_hot_weight_is_relu_of_one_head_gemv():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((6, 16))
    k = rng.standard_normal((50, 16))
    for h in range(6):
        w = np.zeros(6)
        w[h] = 1.0
        ref = torch.relu(torch.matmul(torch.from_numpy(k), torch.from_numpy(q[h]))).numpy()
        np.testing.assert_allclose(oracle.index_scores(q, w, k), ref, rtol=1e-13, atol=1e-13)


def test_scores_linear_in_weights_and_brute_force():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((3, 5))
    k = rng.standard_normal((7, 5))
    w1 = rng.uniform(-1, 1, 3)
    w2 = rng.uniform(-1, 1, 3)
    s = lambda w: oracle.index_scores(q, w, k)  # noqa: E731
    np.testing.assert_allclose(s(w1 + w2), s(w1) + s(w2), rtol=1e-12, atol=1e-12)
    brute = []
    for p in range(7):
        tot = 0.0
        for h in range(3):
            dot = 0.0
            for j in range(5):
                dot += q[h, j] * k[p, j]
            tot += w1[h] * (dot if dot > 0 else 0.0)
        brute.append(tot)
    np.testing.assert_allclose(s(w1), brute, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------------------
# Top-K


def _topk_by_partition(scores, K):
    """An independent selection: argpartition for the threshold, then the tie rule."""
    n = scores.shape[0]
    m = min(K, n)
    if m == 0:
        return set()
    tau = scores[np.argpartition(-scores, m - 1)[m - 1]]
    above = np.flatnonzero(scores > tau)
    ties = np.flatnonzero(scores == tau)
    return set(above.tolist()) | set(ties[: m - above.size].tolist())


@pytest.mark.parametrize("n,K", [(1, 1), (10, 3), (100, 100), (100, 150), (1000, 64), (5000, 2048)])
def test_topk_vs_partition_selection(n, K):
    rng = np.random.default_rng(n * 7 + K)
    s = np.round(rng.standard_normal(n) * 4) / 4  # many exact ties
    idx = oracle.topk_positions(s, K)
    m = min(K, n)
    assert np.all(idx[m:] == -1)
    assert set(idx[:m].tolist()) == _topk_by_partition(s, K)


def test_topk_brute_force_tiny():
    for n, K in itertools.product(range(0, 7), range(1, 8)):
        rng = np.random.default_rng(n * 31 + K)
        s = rng.integers(-2, 3, size=n).astype(np.float64)
        want = sorted(range(n), key=lambda p: (-s[p], p))[:K]
        got = oracle.topk_positions(s, K)
        assert got[: len(want)].tolist() == want
        assert np.all(got[len(want):] == -1)


def test_topk_invariants():
    rng = np.random.default_rng(4)
    s = rng.standard_normal(300)
    base = set(oracle.topk_positions(s, 40).tolist())
    assert set(oracle.topk_positions(np.exp(s), 40).tolist()) == base
    assert set(oracle.topk_positions(3.0 * s - 7.0, 40).tolist()) == base
    assert oracle.topk_positions(np.full(50, 2.5), 10).tolist() == list(range(10))
    assert oracle.topk_positions(np.zeros(0), 4).tolist() == [-1] * 4


# ------------------------------------------------------------------------------------------------
# sparse attention


def _sdpa(q, k, v, scale, mask=None):
    """torch's scaled_dot_product_attention in fp64 on CPU (a library routine)."""
    qt = torch.from_numpy(q)[None, :, None, :]          # [1, H, 1, D]
    kt = torch.from_numpy(k)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.from_numpy(v)[None, None].expand(1, q.shape[0], -1, -1)
    m = None if mask is None else torch.from_numpy(mask)[None, None, None, :]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    return out[0, :, 0, :].numpy()


def test_attention_all_positions_is_dense_attention():
    rng = np.random.default_rng(6)
    q, k, v = rng.standard_normal((4, 24)), rng.standard_normal((40, 24)), rng.standard_normal((40, 8))
    out, lse = oracle.sparse_attention(q, k, v, 0.3)
    np.testing.assert_allclose(out, _sdpa(q, k, v, 0.3), rtol=1e-12, atol=1e-12)
    from scipy.special import logsumexp
    np.testing.assert_allclose(lse, logsumexp(0.3 * q @ k.T, axis=1), rtol=1e-13, atol=1e-13)


def test_sparse_equals_dense_with_rowwise_mask():
    # "Achieving Day-0 Readiness...", section 2.3: sparse attention equals dense attention over
    # the full key tensor with a row-wise sparse mask.
    rng = np.random.default_rng(7)
    q, k, v = rng.standard_normal((3, 16)), rng.standard_normal((64, 16)), rng.standard_normal((64, 12))
    sel = rng.choice(64, size=9, replace=False)
    mask = np.zeros(64, dtype=bool)
    mask[sel] = True
    out, _ = oracle.sparse_attention(q, k[sel], v[sel], 0.25)
    np.testing.assert_allclose(out, _sdpa(q, k, v, 0.25, mask), rtol=1e-12, atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(8)
    k, v = rng.standard_normal((10, 6)), rng.standard_normal((10, 5))
    out, lse = oracle.sparse_attention(np.zeros((2, 6)), k, v, 1.0)
    np.testing.assert_allclose(out, np.tile(v.mean(axis=0), (2, 1)), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, [math.log(10)] * 2, rtol=1e-13)
    same_k = np.tile(k[3], (7, 1))
    same_v = np.tile(v[3], (7, 1))
    q = rng.standard_normal((2, 6))
    out, lse = oracle.sparse_attention(q, same_k, same_v, 0.5)
    np.testing.assert_allclose(out, np.tile(v[3], (2, 1)), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, 0.5 * q @ k[3] + math.log(7), rtol=1e-13)
    perm = rng.permutation(10)
    a, la = oracle.sparse_attention(q, k, v, 0.5)
    b, lb = oracle.sparse_attention(q, k[perm], v[perm], 0.5)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)
    out, lse = oracle.sparse_attention(q, k[:0], v[:0], 0.5)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_lse_combine_of_two_halves():
    # the split-K merge rule the kernels use is an identity of the definition
    rng = np.random.default_rng(9)
    q, k, v = rng.standard_normal((2, 8)), rng.standard_normal((30, 8)), rng.standard_normal((30, 4))
    full, lf = oracle.sparse_attention(q, k, v, 0.7)
    a, la = oracle.sparse_attention(q, k[:11], v[:11], 0.7)
    b, lb = oracle.sparse_attention(q, k[11:], v[11:], 0.7)
    lse = np.logaddexp(la, lb)
    comb = a * np.exp(la - lse)[:, None] + b * np.exp(lb - lse)[:, None]
    np.testing.assert_allclose(comb, full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lf, rtol=1e-13)


# ------------------------------------------------------------------------------------------------
# visibility and the chain


def test_visible_length():
    assert oracle.visible_length(3, 100, 1, -1) == 100
    assert oracle.visible_length(1, 100, 1, -1, n_valid=[5, 7]) == 7
    assert oracle.visible_length(0, 100, 8, 90) == 91
    assert oracle.visible_length(7, 100, 8, 90) == 98
    assert oracle.visible_length(9, 100, 8, 90) == 92  # second sequence restarts at q_pos0
    assert oracle.visible_length(0, 100, 1, -1, n_valid=[0]) == 0
    assert oracle.visible_length(0, 50, 4, 60) == 50


def _brute_chain(a, t, L, K, q_per_seq, q_pos0, sm_scale, H, D_v):
    """Whole chain with Python loops (bf16 inputs, separate V) for tiny shapes."""
    f = lambda x: float(oracle.bf16_bits_to_f64(np.array([x], dtype=np.uint16))[0])  # noqa: E731
    seq = t // q_per_seq
    n = L if q_pos0 < 0 else min(L, q_pos0 + t % q_per_seq + 1)
    qi, w, ki = a["q_idx"][t], a["w"][t], a["k_idx"][seq]
    scores = []
    for s in range(n):
        tot = 0.0
        for h in range(qi.shape[0]):
            dot = sum(f(qi[h, j]) * f(ki[s, j]) for j in range(qi.shape[1]))
            tot += float(w[h]) * max(0.0, dot)
        scores.append(tot)
    order = sorted(range(n), key=lambda s: (-scores[s], s))[:K]
    out, lse = [], []
    for h in range(H):
        logits = [sm_scale * sum(f(a["q"][t, h, j]) * f(a["kv"][seq, s, j])
                                 for j in range(a["q"].shape[2])) for s in order]
        mx = max(logits)
        p = [math.exp(x - mx) for x in logits]
        tot = sum(p)
        out.append([sum(p[i] * f(a["kv_v"][seq, order[i], c]) for i in range(len(order))) / tot
                    for c in range(D_v)])
        lse.append(mx + math.log(tot))
    return scores, order, np.array(out), np.array(lse)


@pytest.mark.parametrize("q_pos0,q_per_seq,T", [(-1, 1, 2), (5, 3, 3)])
def test_chain_query_matches_brute_force(q_pos0, q_per_seq, T):
    wl = synth.Workload("brute", T=T, q_per_seq=q_per_seq, L=12, H_idx=3, d_idx=4, idx_dtype="bf16",
                        K=4, H=2, D_qk=5, D_v=3, kv_dtype="bf16", separate_v=True,
                        q_pos0=q_pos0, seed=77)
    a = synth.to_numpy_bits(synth.make_inputs(wl))
    ch = oracle.Chain(a, L=wl.L, K=wl.K, q_per_seq=wl.q_per_seq, q_pos0=wl.q_pos0,
                      idx_dtype="bf16", kv_dtype="bf16", sm_scale=wl.sm_scale)
    for t in range(T):
        r = oracle.chain_query(ch, t, wl.D_v)
        s, order, out, lse = _brute_chain(a, t, wl.L, wl.K, q_per_seq, q_pos0, wl.sm_scale, wl.H, wl.D_v)
        np.testing.assert_allclose(r["scores"], s, rtol=1e-12, atol=1e-12)
        assert r["idx"][: len(order)].tolist() == order
        np.testing.assert_allclose(r["out"], out, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(r["lse"], lse, rtol=1e-12, atol=1e-12)


def test_chain_fp8_kv_latent_v_uses_row_scale_and_first_columns():
    wl = synth.Workload("q", T=1, q_per_seq=1, L=40, H_idx=2, d_idx=32, idx_dtype="mxfp8", K=8,
                        H=2, D_qk=48, D_v=32, kv_dtype="fp8", separate_v=False, q_pos0=-1, seed=5)
    a = synth.to_numpy_bits(synth.make_inputs(wl))
    ch = oracle.Chain(a, L=wl.L, K=wl.K, q_per_seq=1, q_pos0=-1, idx_dtype="mxfp8",
                      kv_dtype="fp8", sm_scale=wl.sm_scale)
    r = oracle.chain_query(ch, 0, wl.D_v)
    rows = r["idx"]
    kd = oracle.e4m3_to_f64(a["kv"][0, rows]) * a["kv_scale"][0, rows][:, None].astype(np.float64)
    q = oracle.bf16_bits_to_f64(a["q"][0])
    ref = _sdpa(q, kd, kd[:, :32].copy(), wl.sm_scale)
    np.testing.assert_allclose(r["out"], ref, rtol=1e-12, atol=1e-12)


def _torch_e4m3(codes):
    """E4M3 codes -> fp64 through torch's float8_e4m3fn cast (a library decoder independent of
    the oracle's bit-field code)."""
    return torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).to(torch.float64)


def _distinct_exponents(a, rng):
    """Every group, row and head its own E8M0 exponent (scales 2^-6 .. 2^6), so a scale applied
    to the wrong group, row, head or operand changes the scores."""
    for key in ("q_idx_sf", "k_idx_sf"):
        a[key] = rng.integers(121, 134, size=a[key].shape).astype(np.uint8)


def test_chain_mxfp8_scores_match_brute_force_with_distinct_exponents():
    # The oracle's MXFP8 scoring branch (Chain.scores) against Python loops over the raw codes:
    # I[s] = sum_h w[h] * max(0, sum_g 2^(eq[h,g]-127) 2^(ek[s,g]-127) sum_{j in g} q[h,j] k[s,j])
    # ("Day 0 Support for New LLM Architectures", Key Optimization 2: groups of 32 elements
    # share one scale factor).
    wl = synth.Workload("mxb", T=2, q_per_seq=1, L=9, H_idx=3, d_idx=64, idx_dtype="mxfp8", K=4,
                        H=1, D_qk=64, D_v=64, kv_dtype="fp8", separate_v=False, q_pos0=-1, seed=31)
    a = synth.to_numpy_bits(synth.make_inputs(wl))
    _distinct_exponents(a, np.random.default_rng(4))
    ch = oracle.Chain(a, L=wl.L, K=wl.K, q_per_seq=1, q_pos0=-1, idx_dtype="mxfp8", kv_dtype="fp8",
                      sm_scale=wl.sm_scale)
    for t in range(wl.T):
        qv = _torch_e4m3(a["q_idx"][t]).tolist()
        kv = _torch_e4m3(a["k_idx"][t]).tolist()
        want = []
        for s in range(wl.L):
            tot = 0.0
            for h in range(wl.H_idx):
                dot = 0.0
                for g in range(wl.d_idx // 32):
                    part = sum(qv[h][j] * kv[s][j] for j in range(32 * g, 32 * g + 32))
                    dot += part * 2.0 ** (int(a["q_idx_sf"][t, h, g]) - 127) * 2.0 ** (int(a["k_idx_sf"][t, s, g]) - 127)
                tot += float(a["w"][t, h]) * max(0.0, dot)
            want.append(tot)
        np.testing.assert_allclose(ch.scores(t), want, rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("idx_dtype", ["mxfp8", "bf16"])
def test_chain_scores_across_the_row_chunk_boundary(idx_dtype):
    # Chain.scores decodes the key cache in chunks of 65,536 rows; a cache longer than one chunk,
    # with every row's scale exponents its own, checks the chunk offsets on the codes and on the
    # scale array against one whole-cache product built from torch's decoders and matmul.
    L = (1 << 16) + 333
    wl = synth.Workload("chunks", T=1, q_per_seq=1, L=L, H_idx=2, d_idx=64, idx_dtype=idx_dtype, K=4,
                        H=1, D_qk=64, D_v=64, kv_dtype="bf16", separate_v=False, q_pos0=-1, seed=32)
    cpu = synth.make_inputs(wl)
    a = synth.to_numpy_bits(cpu)
    if idx_dtype == "mxfp8":
        _distinct_exponents(a, np.random.default_rng(5))
        scale_q = torch.pow(2.0, torch.from_numpy(a["q_idx_sf"][0].astype(np.float64) - 127))
        scale_k = torch.pow(2.0, torch.from_numpy(a["k_idx_sf"][0].astype(np.float64) - 127))
        q = _torch_e4m3(a["q_idx"][0]) * scale_q.repeat_interleave(32, dim=-1)
        k = _torch_e4m3(a["k_idx"][0]) * scale_k.repeat_interleave(32, dim=-1)
    else:
        q = cpu["q_idx"][0].to(torch.float64)
        k = cpu["k_idx"][0].to(torch.float64)
    w = torch.from_numpy(a["w"][0].astype(np.float64))
    want = (torch.relu(k @ q.T) @ w).numpy()
    ch = oracle.Chain(a, L=L, K=4, q_per_seq=1, q_pos0=-1, idx_dtype=idx_dtype, kv_dtype="bf16",
                      sm_scale=0.125)
    np.testing.assert_allclose(ch.scores(0), want, rtol=1e-12, atol=1e-300)


def test_chain_fp8_tiled_kv_applies_each_tiles_scale():
    # The oracle's tiled FP8 KV branch (Chain.kv_rows with fp8_t128): element j of a selected row
    # is E4M3(code) * scale[row][j // 128] (576 = 4 x 128 + 64: five scales per row; "Day 0
    # Support for New LLM Architectures", Key Optimization 2), V = its first 512 columns; checked
    # on selected rows of a second sequence against torch's float8 decode, an explicit per-element
    # tile lookup and torch's scaled_dot_product_attention.
    wl = synth.Workload("t128", T=2, q_per_seq=1, L=30, H_idx=2, d_idx=64, idx_dtype="bf16", K=7,
                        H=3, D_qk=576, D_v=512, kv_dtype="fp8_t128", separate_v=False, q_pos0=-1, seed=33)
    a = synth.to_numpy_bits(synth.make_inputs(wl))
    rng = np.random.default_rng(6)
    a["kv_scale"] = np.ldexp(1.0, rng.integers(-5, 6, size=a["kv_scale"].shape)).astype(np.float32)
    ch = oracle.Chain(a, L=wl.L, K=wl.K, q_per_seq=1, q_pos0=-1, idx_dtype="bf16", kv_dtype="fp8_t128",
                      sm_scale=wl.sm_scale)
    t, seq = 1, 1
    idx = np.array([29, 3, -1, 17, 0, 11, -1])
    rows = [r for r in idx.tolist() if r >= 0]
    vals = _torch_e4m3(a["kv"][seq, rows]).numpy()
    tile_of = np.array([j // 128 for j in range(wl.D_qk)])
    kd = vals * a["kv_scale"][seq, rows][:, tile_of].astype(np.float64)
    q = oracle.bf16_bits_to_f64(a["q"][t])
    out, _ = ch.attention(t, idx, wl.D_v)
    np.testing.assert_allclose(out, _sdpa(q, kd, kd[:, :wl.D_v].copy(), wl.sm_scale), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------------------------------------
# a context split over slices: candidate merge and partial-output combine


def test_merge_candidates_brute_force_tiny():
    # every candidate list of length 6 over scores {0, 1, 2} with empty entries, against Python's
    # sorted() on (-score, position) tuples
    rng = np.random.default_rng(50)
    for _ in range(300):
        n = 6
        s = rng.integers(0, 3, n).astype(np.float64)
        p = rng.permutation(40)[:n]
        p[rng.random(n) < 0.3] = -1
        K = int(rng.integers(1, 8))
        valid = [j for j in range(n) if p[j] >= 0]
        best = sorted(valid, key=lambda j: (-s[j], p[j]))[:K]
        want = [int(p[j]) for j in sorted(best)] + [-1] * (K - len(best))
        assert oracle.merge_candidates(s, p, K).tolist() == want


def test_merge_of_all_positions_is_topk_of_the_row():
    rng = np.random.default_rng(51)
    s = np.round(rng.standard_normal(3000) * 4)  # many exact ties
    pos = rng.permutation(3000)
    got = oracle.merge_candidates(s[pos], pos, 700)
    assert sorted(got.tolist()) == sorted(oracle.topk_positions(s, 700).tolist())


@pytest.mark.parametrize("G,tie", [(2, False), (5, False), (4, True)])
def test_merge_of_slice_topks_is_the_global_topk(G, tie):
    # the fact the split decode rests on: every global Top-K position is in its slice's Top-K, so
    # merging the slices' selections (slices in order, ascending positions) gives the global set in
    # ascending order; with ties across slices the lower positions still win
    rng = np.random.default_rng(52 + G)
    n, K = 5000, 300
    s = np.round(rng.standard_normal(n)) if tie else rng.standard_normal(n)
    bounds = np.linspace(0, n, G + 1).astype(int)
    cand_s, cand_p = [], []
    for g in range(G):
        lo, hi = bounds[g], bounds[g + 1]
        local = oracle.topk_positions(s[lo:hi], K)
        local = np.concatenate([np.sort(local[local >= 0]), local[local < 0]])  # ascending, as listed
        ok = local >= 0
        cand_p.append(np.where(ok, local + lo, -1))
        cand_s.append(np.where(ok, s[lo:hi][np.where(ok, local, 0)], 0.0))
    got = oracle.merge_candidates(np.concatenate(cand_s), np.concatenate(cand_p), K)
    want = np.sort(oracle.topk_positions(s, K))
    np.testing.assert_array_equal(got, want)


def test_combine_of_partials_over_a_partition_is_the_whole_attention():
    rng = np.random.default_rng(53)
    q, k, v = rng.standard_normal((3, 16)), rng.standard_normal((50, 16)) * 2, rng.standard_normal((50, 5))
    full, lf = oracle.sparse_attention(q, k, v, 0.4)
    cuts = [0, 7, 7, 31, 50]  # the second part is empty
    parts = [oracle.sparse_attention(q, k[a:b], v[a:b], 0.4) for a, b in zip(cuts[:-1], cuts[1:])]
    out, lse = oracle.combine_partials(np.stack([o for o, _ in parts]), np.stack([l for _, l in parts]))
    np.testing.assert_allclose(out, full, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, lf, rtol=1e-13)
    # against torch's scaled_dot_product_attention as well, and all-empty parts give 0 and -inf
    np.testing.assert_allclose(out, _sdpa(q, k, v, 0.4), rtol=1e-12, atol=1e-12)
    e_out, e_lse = oracle.combine_partials(np.zeros((2, 3, 5)), np.full((2, 3), -np.inf))
    assert np.all(e_out == 0) and np.all(np.isneginf(e_lse))


# ------------------------------------------------------------------------------------------------
# the parity rule itself (mistakes planted on the CPU)


def test_parity_rule_accepts_oracle_and_band_swaps_and_rejects_mistakes():
    rng = np.random.default_rng(10)
    s = rng.standard_normal(500) * 10 + 50
    s[123] = s[77] * (1 + 2e-4)  # a near tie
    K = 50
    idx = oracle.topk_positions(s, K)
    rep = parity.check_topk(idx, s, K)
    assert rep["swaps"] == 0
    order = np.lexsort((np.arange(500), -s))
    tau = s[order[K - 1]]
    # swap the K-th element for the next one when it lies inside the band
    s2 = s.copy()
    s2[order[K]] = tau * (1 - 5e-4)
    idx2 = oracle.topk_positions(s2, K).copy()
    idx2[idx2 == order[K - 1]] = order[K]
    assert parity.check_topk(idx2, s2, K)["swaps"] == 1
    bad = idx.copy()
    bad[0] = order[-1]  # lowest score
    with pytest.raises(AssertionError):
        parity.check_topk(bad, s, K)
    dup = idx.copy()
    dup[1] = dup[0]
    with pytest.raises(AssertionError):
        parity.check_topk(dup, s, K)
    short = idx.copy()
    short[-1] = -1
    with pytest.raises(AssertionError):
        parity.check_topk(short, s, K)
    with pytest.raises(AssertionError):
        parity.check_topk(np.where(idx == order[0], 600, idx), s, K)
