"""Parity of the online quantisation kernels (dsa_quantize_mxfp8, dsa_quantize_fp8_rows) with the
oracle's encoders: codes, exponent bytes and scales are integer / exactly-rounded results, so the
comparison is bit for bit.  The cache-append form (destination rows) must write exactly the rows
it names, and caches written this way must drive the fused chain to parity."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import check_chain

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


def _rows(seed, rows, width, group_spread=True):
    """bf16 rows: N(0,1) times a random power of two per group of 32, plus special rows."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, width))
    if group_spread:
        x *= np.ldexp(1.0, rng.integers(-60, 60, (rows, -(-width // 32)))).repeat(32, 1)[:, :width]
    t = torch.from_numpy(x).to(torch.bfloat16)
    t[0] = 0.0                                             # all-zero row
    t[1, : min(32, width)] = 0.0                           # an all-zero group
    t[2] = -0.0                                            # negative zeros
    t[3] = torch.from_numpy(rng.standard_normal(width) * 1e-39).to(torch.bfloat16)  # subnormals
    t[4] = torch.from_numpy(rng.standard_normal(width) * 1e36).to(torch.bfloat16)   # large
    t[5, 0] = 1.0e30                                       # one large value among small ones
    return t


def _f64(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("d,pitch", [(128, 128), (64, 64), (32, 32), (256, 256), (128, 132), (128, 129)])
def test_quantize_mxfp8_bit_exact(dsa, d, pitch):
    # 16-byte aligned rows take the wide form, 8-byte aligned rows with d a multiple of 128 the
    # four-element form, the others the generic one
    x = _rows(1 + d, 300, d)
    src = torch.zeros(300, pitch, dtype=torch.bfloat16)
    src[:, :d] = x
    codes, sf = dsa.dsa_quantize_mxfp8(src.cuda()[:, :d])
    want_codes, want_sf = oracle.quantize_mxfp8(_f64(x))
    np.testing.assert_array_equal(sf.cpu().numpy(), want_sf)
    np.testing.assert_array_equal(codes.cpu().numpy(), want_codes)


@pytest.mark.parametrize("width", [576, 64, 100, 102])
def test_quantize_fp8_rows_bit_exact(dsa, width):
    x = _rows(2 + width, 257, width)
    codes, s = dsa.dsa_quantize_fp8_rows(x.cuda())
    want_codes, want_s = oracle.quantize_fp8_rows(_f64(x))
    np.testing.assert_array_equal(s.cpu().numpy(), want_s)
    np.testing.assert_array_equal(codes.cpu().numpy(), want_codes)


@pytest.mark.parametrize("width,tile", [(576, 128), (100, 32), (576, 1024), (130, 64)])
def test_quantize_fp8_tiles_bit_exact(dsa, width, tile):
    x = _rows(3 + width + tile, 211, width)
    codes, s = dsa.dsa_quantize_fp8_tiles(x.cuda(), tile=tile)
    want_codes, want_s = oracle.quantize_fp8_tiles(_f64(x), tile)
    np.testing.assert_array_equal(s.cpu().numpy(), want_s)
    np.testing.assert_array_equal(codes.cpu().numpy(), want_codes)


def _all_bf16_up_to_448():
    b = np.arange(0, 1 << 16, dtype=np.uint32)
    v = (b << 16).view(np.float32)
    # magnitudes below 2^-100 are left out so that scaling by 2^-20 stays exact in bf16 (they are
    # far below E4M3's smallest midpoint, 2^-10)
    keep = np.isfinite(v) & (np.abs(v) <= 448) & ((np.abs(v) >= 2.0**-100) | (v == 0))
    return v[keep].astype(np.float64)


@pytest.mark.parametrize("k", [-20, 0, 13])
def test_quantize_fp8_rows_exact_ties_at_every_midpoint(dsa, k):
    # rows whose amax is 448 * 2^k have s = 2^k exactly, so x / s is the bf16 value itself: the rows
    # carry every bf16 value of magnitude <= 448, among them every midpoint of two E4M3 values
    # (an exact tie, resolved to even) and the values around it
    W = 576
    vals = _all_bf16_up_to_448()
    n = -(-vals.size // (W - 1))
    body = np.resize(vals, n * (W - 1)).reshape(n, W - 1)
    x = np.concatenate([np.full((n, 1), 448.0), body], axis=1) * 2.0**k
    t = torch.from_numpy(x).to(torch.bfloat16)
    assert np.array_equal(t.to(torch.float64).numpy(), x)  # every value is a bf16
    codes, s = dsa.dsa_quantize_fp8_rows(t.cuda())
    want_codes, want_s = oracle.quantize_fp8_rows(x)
    np.testing.assert_array_equal(s.cpu().numpy(), want_s)
    np.testing.assert_array_equal(codes.cpu().numpy(), want_codes)


def test_quantize_fp8_rows_large_random_batch(dsa):
    # 4096 latent rows with per-row magnitudes spread over 2^-40 .. 2^40
    rng = np.random.default_rng(77)
    x = rng.standard_normal((4096, 576)) * np.ldexp(1.0, rng.integers(-40, 40, (4096, 1)))
    t = torch.from_numpy(x).to(torch.bfloat16)
    codes, s = dsa.dsa_quantize_fp8_rows(t.cuda())
    want_codes, want_s = oracle.quantize_fp8_rows(_f64(t))
    np.testing.assert_array_equal(s.cpu().numpy(), want_s)
    np.testing.assert_array_equal(codes.cpu().numpy(), want_codes)


def test_cache_append_writes_only_its_rows(dsa):
    # new tokens of 3 sequences appended at their next positions of [3][L] caches
    L, d, W = 50, 128, 576
    x = _rows(5, 7, d)
    kvx = _rows(6, 7, W, group_spread=False)
    seq = np.array([0, 0, 1, 2, 2, 2, 1])
    pos = np.array([10, 11, 49, 0, 1, 2, 48])
    dst = torch.from_numpy(seq * L + pos).to(torch.int64)
    dst[3] = -1  # dropped row
    codes = torch.full((3 * L, d), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full((3 * L, d // 32), 0xCD, dtype=torch.uint8, device="cuda")
    kv = torch.full((3 * L, W + 16), 0xEF, dtype=torch.uint8, device="cuda")  # padded row pitch
    kvs = torch.full((3 * L,), -7.0, dtype=torch.float32, device="cuda")
    dsa.dsa_quantize_mxfp8(x.cuda(), codes=codes, sf=sf, dst_rows=dst.cuda())
    dsa.dsa_quantize_fp8_rows(kvx.cuda(), codes=kv[:, :W], scales=kvs, dst_rows=dst.cuda())
    codes, sf, kv, kvs = codes.cpu().numpy(), sf.cpu().numpy(), kv.cpu().numpy(), kvs.cpu().numpy()
    wc, wsf = oracle.quantize_mxfp8(_f64(x))
    wkv, wkvs = oracle.quantize_fp8_rows(_f64(kvx))
    written = set()
    for r, q in enumerate(dst.numpy()):
        if q < 0:
            continue
        written.add(int(q))
        np.testing.assert_array_equal(codes[q], wc[r])
        np.testing.assert_array_equal(sf[q], wsf[r])
        np.testing.assert_array_equal(kv[q, :W], wkv[r])
        assert kvs[q] == wkvs[r]
    untouched = [q for q in range(3 * L) if q not in written]
    assert np.all(codes[untouched] == 0xAB) and np.all(sf[untouched] == 0xCD)
    assert np.all(kv[untouched] == 0xEF) and np.all(kvs[untouched] == -7.0)
    assert np.all(kv[:, W:] == 0xEF)  # the row padding is never written


def test_quantised_caches_drive_the_chain(dsa):
    # bf16 indexer rows and latent rows quantised on the GPU are the oracle's caches byte for
    # byte, and the MXFP8 / FP8 chain over them meets the usual parity rule
    wl = synth.small_workload("decode_b8_l32k_mxfp8", T=2, L=1000, K=256)
    g = torch.Generator().manual_seed(11)
    q_idx = torch.randn(wl.T, wl.H_idx, wl.d_idx, generator=g).to(torch.bfloat16)
    k_idx = torch.randn(wl.T, wl.L, wl.d_idx, generator=g).to(torch.bfloat16)
    kvx = torch.randn(wl.T, wl.L, wl.D_qk, generator=g).to(torch.bfloat16)
    qc, qsf = dsa.dsa_quantize_mxfp8(q_idx.reshape(-1, wl.d_idx).cuda())
    kc, ksf = dsa.dsa_quantize_mxfp8(k_idx.reshape(-1, wl.d_idx).cuda())
    vc, vs = dsa.dsa_quantize_fp8_rows(kvx.reshape(-1, wl.D_qk).cuda())
    for (c, s), src, enc in (((qc, qsf), q_idx, oracle.quantize_mxfp8), ((kc, ksf), k_idx, oracle.quantize_mxfp8),
                             ((vc, vs), kvx, oracle.quantize_fp8_rows)):
        wc, ws = enc(_f64(src.reshape(-1, src.shape[-1])))
        np.testing.assert_array_equal(c.cpu().numpy(), wc)
        np.testing.assert_array_equal(s.cpu().numpy(), ws)
    cpu = synth.make_inputs(wl)  # q and w of the workload's recipe; caches replaced below
    cpu["q_idx"] = qc.cpu().reshape(wl.T, wl.H_idx, wl.d_idx)
    cpu["q_idx_sf"] = qsf.cpu().reshape(wl.T, wl.H_idx, wl.d_idx // 32)
    cpu["k_idx"] = kc.cpu().reshape(wl.T, wl.L, wl.d_idx)
    cpu["k_idx_sf"] = ksf.cpu().reshape(wl.T, wl.L, wl.d_idx // 32)
    cpu["kv"] = vc.cpu().reshape(wl.T, wl.L, wl.D_qk)
    cpu["kv_scale"] = vs.cpu().reshape(wl.T, wl.L)
    check_chain(dsa, wl, cpu)


def test_bad_arguments_are_rejected_before_launch(dsa):
    from top_sparse_attention_gb300 import _native as N

    x = torch.zeros(4, 128, dtype=torch.bfloat16, device="cuda")
    c = torch.zeros(4, 128, dtype=torch.uint8, device="cuda")
    assert N.lib.dsa_quantize_mxfp8(x.data_ptr(), 128, 4, 100, c.data_ptr(), c.data_ptr(), None, None) == 1
    assert N.lib.dsa_quantize_mxfp8(x.data_ptr(), 64, 4, 128, c.data_ptr(), c.data_ptr(), None, None) == 1
    assert N.lib.dsa_quantize_fp8_rows(x.data_ptr(), 128, 4, 128, c.data_ptr(), 64, c.data_ptr(), None, None) == 1
    assert N.lib.dsa_quantize_fp8_rows(None, 128, 4, 128, c.data_ptr(), 128, c.data_ptr(), None, None) == 1
