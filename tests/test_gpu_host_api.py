"""kb_attn_fwd_host, the host-to-host call: its result in the host buffer is
the device-resident call's result bit for bit, for the tensor-core, fp32 flash
and Q15 paths, with pinned and with pageable host buffers."""
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import Variant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


CASES = [(inputs.Workload("h_bf16", 2, 3, 300, 128, True, "bf16", 51, "normal"), Variant.TC),
         (inputs.Workload("h_f16", 1, 2, 513, 64, False, "f16", 52, "normal"), Variant.TC),
         (inputs.Workload("h_f32", 1, 2, 200, 64, True, "f32", 53, "uniform"), Variant.FLASH),
         (inputs.Workload("h_q15", 1, 2, 77, 32, True, "q15", 54, "uniform"), Variant.FIXEDPOINT)]


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("w,variant", CASES, ids=lambda x: getattr(x, "name", None))
def test_host_call_equals_device_call(w, variant, pinned):
    qh, kh, vh = inputs.make_qkv(w)
    if pinned:
        qh, kh, vh = (t.pin_memory() for t in (qh, kh, vh))
    want = kbattn.kb_attn_fwd(qh.cuda(), kh.cuda(), vh.cuda(), causal=w.causal, scale=w.scale, variant=variant)
    stage = [torch.full(qh.shape, 0, dtype=qh.dtype, device="cuda") for _ in range(4)]
    oh = torch.empty(qh.shape, dtype=qh.dtype, pin_memory=pinned)
    stream = torch.cuda.Stream()
    kbattn.kb_attn_fwd_host(qh, kh, vh, oh, *stage, causal=w.causal, scale=w.scale, variant=variant, stream=stream)
    stream.synchronize()
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    assert torch.equal(oh, want.cpu())
    assert torch.equal(stage[0].cpu(), qh)  # the staging buffers hold the copied inputs
