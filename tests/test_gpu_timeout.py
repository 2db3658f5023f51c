"""The bounded-wait failure path, exercised without hanging or faulting the GPU:
a kernel waits on an mbarrier that nothing completes, gives up after a short
limit, and the host reads KB_ERR_TIMEOUT; the context stays usable."""
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


def test_wait_that_runs_out_is_reported_and_cleared():
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    kbattn.kb_selftest_timeout(2_000_000)  # 2 ms
    assert kbattn.kb_check_device_error() == kbattn.Status.TIMEOUT
    assert kbattn.kb_check_device_error() == kbattn.Status.OK  # read clears it


def test_context_still_usable_after_timeout(oracle):
    kbattn.kb_selftest_timeout(1_000_000)
    assert kbattn.kb_check_device_error() == kbattn.Status.TIMEOUT
    w = inputs.Workload("after", 1, 1, 128, 64, True, "bf16", 21, "normal")
    q, k, v = inputs.make_qkv(w)
    o = kbattn.kb_attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    want = oracle.attn(q, k, v, True, w.scale)
    assert float((o.float().cpu() - torch.from_numpy(want)).abs().max()) <= 2e-2
