"""GPU Triad a = b + s*c: bit-exact against the oracle (one rounding), every
block size, ragged lengths, and the STREAM constant check."""
import numpy as np
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from tests.gpu_util import Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


@pytest.mark.parametrize("block", [128, 256, 512, 1024])
@pytest.mark.parametrize("n", [1, 3, 4, 5, 1023, 4099, (1 << 20) + 7, 3 * (1 << 22) + 2])
def test_triad_bit_exact(oracle, n, block):
    b, c = inputs.make_triad_inputs(n, seed=n)
    s = -0.3711
    g = Guarded((n,), torch.float32)
    kbattn.kb_triad(g.out, b.cuda(), c.cuda(), s, block=block)
    got = g.check().cpu().numpy()
    want = oracle.triad(b.numpy(), c.numpy(), s)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_triad_stream_constants():
    n = 64 << 20
    b = torch.ones(n, device="cuda")
    c = torch.full((n,), 2.0, device="cuda")
    a = torch.empty(n, device="cuda")
    kbattn.kb_triad(a, b, c, 3.0)
    assert bool((a == 7.0).all())


def test_triad_bench_reports_every_iteration():
    n = 16 << 20
    a, b, c = (torch.zeros(n, device="cuda") for _ in range(3))
    ms = kbattn.kb_triad_bench(a, b, c, 1.5, block=256, warmup=2, iters=5)
    assert len(ms) == 5 and all(t > 0 for t in ms)


def test_device_info_is_gb300_class():
    info = kbattn.kb_device_info(torch.cuda.current_device())
    assert (info["cc_major"], info["cc_minor"]) == (10, 3)
    assert info["sm_count"] > 100 and info["mem_bus_width_bits"] > 0 and info["mem_clock_khz"] > 0


@pytest.mark.parametrize("block", [128, 256, 512, 1024])
@pytest.mark.parametrize("n", [1, 3, 4, 1023, 4099, (1 << 20) + 7])
def test_copy_write_read_match_oracle(oracle, n, block):
    b, _ = inputs.make_triad_inputs(n, seed=n + 1)
    g = Guarded((n,), torch.float32)
    kbattn.kb_hbm_copy(g.out, b.cuda(), block=block)
    assert np.array_equal(g.check().cpu().numpy().view(np.uint32), oracle.copy(b.numpy()).view(np.uint32))
    g = Guarded((n,), torch.float32)
    kbattn.kb_hbm_write(g.out, -1.75, block=block)
    assert np.array_equal(g.check().cpu().numpy(), oracle.fill(n, -1.75))
    # small integers: every fp32 partial sum is exact, so the read kernel's sum is exact
    ints = ((torch.arange(n) % 7) - 3).to(torch.float32)
    out = torch.full((1,), 123.0, device="cuda")
    kbattn.kb_hbm_read(ints.cuda(), out, block=block)
    assert float(out.item()) == oracle.sum(ints.numpy())


def test_hbm_bench_runs_every_kernel():
    n = 8 << 20
    a, b, c = (torch.ones(n, device="cuda") for _ in range(3))
    out = torch.zeros(1, device="cuda")
    for op in kbattn.HbmOp:
        ms = kbattn.kb_hbm_bench(op, a, b, c, 2.0, out, block=256, warmup=1, iters=3)
        assert len(ms) == 3 and all(t > 0 for t in ms)
    assert float(out.item()) == n  # the last READ summed n ones
