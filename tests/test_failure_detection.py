"""Failure detection without a GPU fault: a bounded wait that runs out reports an error status.

Every wait in the chain's kernels (on an mbarrier that TMA or the tensor core completes) has a
limit of about one second; when it runs out the kernel records DSA_DEVERR_WAIT_TIMEOUT in the
device error word and returns.  The self-test entry makes such a wait run out on purpose (a barrier
that nothing arrives on); this test checks that the host reads the status and that the context
still runs the chain correctly afterwards.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

DSA_DEVERR_WAIT_TIMEOUT = 2


@pytest.fixture(scope="module")
def dsa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_sparse_attention_gb300 import build

    build.build()
    import top_sparse_attention_gb300 as dsa

    torch.cuda.set_device(0)
    return dsa


def test_wait_timeout_is_reported_and_the_context_stays_usable(dsa):
    import synth
    from gpu_helpers import check_chain

    wl = synth.small_workload("decode_b8_l32k_bf16", T=3, L=3000, K=512)
    cpu = synth.make_inputs(wl)

    assert dsa.dsa_get_device_error() == 0  # nothing pending before the test
    dsa.dsa_selftest_wait_timeout()
    assert dsa.dsa_get_device_error() == DSA_DEVERR_WAIT_TIMEOUT
    assert dsa.dsa_get_device_error() == 0  # reading clears the word
    check_chain(dsa, wl, cpu)               # the same context still computes the chain
    assert dsa.dsa_get_device_error() == 0
