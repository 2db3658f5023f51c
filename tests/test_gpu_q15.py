"""GPU parity of the Q15 fixed-point path (integer arithmetic only) against the
oracle's Q15 model: bit-exact, element by element, on small shapes with ragged
tails, on the full fixed-point workloads, and on inputs that drive the rescale,
the table's zero region and the int16 saturation."""
import numpy as np
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import Variant
from tests.gpu_util import run_twice

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


def run_q15(q, k, v, causal, scale):
    q, k, v = q.cuda(), k.cuda(), v.cuda()

    def launch(out):
        kbattn.kb_attn_fwd(q, k, v, out, causal=causal, scale=scale, variant=Variant.FIXEDPOINT)
        assert kbattn.kb_check_device_error() == kbattn.Status.OK

    return run_twice(q.shape, torch.int16, launch).cpu().numpy()


def assert_bit_exact(got, want):
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[0].tolist()}: {got[tuple(bad[0])]} vs {want[tuple(bad[0])]}"


SMALL = [  # (B, H, S, d, causal)
    (1, 1, 1, 32, False), (1, 1, 1, 128, True), (1, 2, 31, 64, True), (1, 1, 32, 32, False),
    (2, 1, 33, 128, True), (1, 3, 95, 64, False), (1, 2, 200, 32, True), (1, 1, 257, 128, False),
    (2, 2, 64, 64, True),
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}h{}s{}d{}{}".format(*s[:4], "c" if s[4] else ""))
def test_small_shapes_bit_exact(oracle, shape):
    B, H, S, d, causal = shape
    w = inputs.Workload("t", B, H, S, d, causal, "q15", 300 + S + d, "uniform")
    q, k, v = inputs.make_qkv(w)
    assert_bit_exact(run_q15(q, k, v, causal, w.scale), oracle.attn_q15(q, k, v, causal, w.scale))


@pytest.mark.parametrize("w", [inputs.Q15_SINGLE_HEAD, inputs.Q15_S1024, inputs.Q15_S1024_CAUSAL],
                         ids=lambda w: w.name)
def test_fixed_point_workloads_bit_exact(oracle, w):
    q, k, v = inputs.make_qkv(w)
    assert_bit_exact(run_q15(q, k, v, w.causal, w.scale), oracle.attn_q15(q, k, v, w.causal, w.scale))


@pytest.mark.parametrize("scale", [0.05, 1.0, 20.0, 700.0])
def test_sharp_scores_and_rescales_bit_exact(oracle, scale):
    """Large scales make the running maximum jump between tiles (rescales by
    tiny or zero factors) and push most weights into the table's zero region."""
    w = inputs.Workload("t", 1, 2, 300, 64, False, "q15", 77, "uniform")
    q, k, v = inputs.make_qkv(w)
    for causal in (False, True):
        assert_bit_exact(run_q15(q, k, v, causal, scale), oracle.attn_q15(q, k, v, causal, scale))


def test_extreme_codes_bit_exact(oracle):
    """Every input at -32768 or 32767: the largest products, the largest dot
    products and outputs at the int16 limits."""
    g = torch.Generator().manual_seed(5)
    shape = (1, 2, 130, 128)
    q, k, v = (torch.where(torch.rand(shape, generator=g) < 0.5, -32768, 32767).to(torch.int16) for _ in range(3))
    for causal in (False, True):
        for scale in (128 ** -0.5, 0.001):
            assert_bit_exact(run_q15(q, k, v, causal, scale), oracle.attn_q15(q, k, v, causal, scale))


def test_table_matches_the_oracle_table(oracle):
    assert kbattn.kb_q15_exp_table() == oracle.q15_exp_table().tolist()


def test_graph_replay_of_the_fixed_point_path(oracle):
    w = inputs.Q15_SINGLE_HEAD
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    ms = []

    def launch(out):
        ms.extend(kbattn.kb_attn_bench_graph(q, k, v, out, causal=False, scale=w.scale,
                                             variant=Variant.FIXEDPOINT, launches=50, warmup=1, iters=2))

    got = run_twice(q.shape, torch.int16, launch).cpu().numpy()
    assert len(ms) == 4 and all(x > 0 for x in ms)
    assert_bit_exact(got, oracle.attn_q15(*inputs.make_qkv(w), False, w.scale))
