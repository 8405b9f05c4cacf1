"""dsa_topk_noalloc: Top-K for callers that cannot provide device memory.

Callers such as a host framework that owns every device allocation through its own pool, or a
decode loop that must not allocate while it runs, get the same selection as dsa_topk from an
entry point whose scratch lives in a fixed array inside the library.  This file checks, through
the C ABI, that two calls in a row give the same index sets as dsa_topk with a caller workspace
(bit-exact: both run the same selection on the same fp32 scores).  It is collected last so that a
run stopping at its first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def native():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_attention_gb300 import build

    build.build()
    from top_sparse_attention_gb300 import _native

    torch.cuda.set_device(0)
    return _native


def _scores(seed, T, L):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(T, L, generator=g) * 30 + 140
    s[:, ::97] = s[:, 5:6]  # some exact ties
    return s.cuda()


def _with_workspace(native, scores, K, L):
    T = scores.shape[0]
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    n = native.lib.dsa_topk_workspace_size(T, L, K)
    ws = torch.zeros(max(n, 16), dtype=torch.uint8, device="cuda")
    st = native.lib.dsa_topk(scores.data_ptr(), scores.stride(0), T, 1, -1, None, L, K, idx.data_ptr(),
                             ws.data_ptr(), n, None)
    assert st == 0, native.status_string(st)
    return idx


def _without_workspace(native, scores, K, L):
    T = scores.shape[0]
    idx = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    st = native.lib.dsa_topk_noalloc(scores.data_ptr(), scores.stride(0), T, 1, -1, None, L, K,
                                     idx.data_ptr(), None)
    assert st == 0, native.status_string(st)
    return idx


@pytest.mark.parametrize("T,L,K", [
    (8, 32768, 2048),     # 4-CTA clusters, keys kept in shared memory
    (16, 200000, 2048),   # the whole scratch array: 16 queries on 16-CTA clusters
    (4, 300000, 2048),    # rows past 16 x 16384 keys: dsa_topk splits them over independent CTAs,
                          # this entry keeps one 16-CTA cluster per row (keys re-read from L2)
])
def test_noalloc_topk_matches_the_workspace_entry_on_two_calls(native, T, L, K):
    a, b = _scores(1, T, L), _scores(2, T, L)
    ref_a = _with_workspace(native, a, K, L)
    ref_b = _with_workspace(native, b, K, L)
    got_a = _without_workspace(native, a, K, L)  # first call on this device sets up the scratch
    got_b = _without_workspace(native, b, K, L)  # second call reuses the array left by the first
    torch.cuda.synchronize()
    for got, ref in ((got_a, ref_a), (got_b, ref_b)):
        g, r = got.cpu().numpy(), ref.cpu().numpy()
        for t in range(T):
            assert np.array_equal(np.sort(g[t]), np.sort(r[t])), f"query {t}"
    code = ctypes.c_int(0)
    assert native.lib.dsa_get_device_error(ctypes.byref(code), None) == 0 and code.value == 0


def test_noalloc_topk_rejects_more_queries_than_its_scratch_holds(native):
    T, L, K = 17, 4096, 64
    s = torch.zeros(T, L, device="cuda")
    idx = torch.empty(T, K, dtype=torch.int32, device="cuda")
    st = native.lib.dsa_topk_noalloc(s.data_ptr(), L, T, 1, -1, None, L, K, idx.data_ptr(), None)
    assert st == 2  # DSA_ERR_UNSUPPORTED, before any launch
