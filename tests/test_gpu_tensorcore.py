"""GPU parity of the tcgen05 tensor-core kernel (bf16 / f16) against the
oracle run on the same 16-bit-rounded inputs: max-abs <= 2e-2 and mean-abs
<= 2e-3 (the 16-bit tolerances). Small shapes are compared element by
element; the full-size workloads, in the launch configuration the benchmark
times, on a fixed seeded sample of rows (rows are independent, so each sampled
row is exactly the row the full evaluation gives)."""
import numpy as np
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import Variant
from tests.gpu_util import Guarded, errors

pytestmark = pytest.mark.gpu

MAX_TOL = 2e-2
MEAN_TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


def run_tc(q, k, v, causal, scale):
    g = Guarded(q.shape, q.dtype)
    kbattn.kb_attn_fwd(q.cuda(), k.cuda(), v.cuda(), g.out, causal=causal, scale=scale, variant=Variant.TC)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    return g.check()


SMALL = [  # (B, H, S, d, causal): one tile, several tiles, ragged tails, S = 1
    (1, 1, 128, 128, False), (1, 1, 128, 128, True), (1, 1, 128, 64, False), (1, 2, 256, 128, True),
    (1, 2, 256, 64, True), (2, 1, 300, 128, False), (1, 1, 1, 128, True), (1, 1, 1, 64, False),
    (1, 2, 77, 64, False), (1, 1, 513, 64, True), (1, 3, 640, 128, True), (2, 2, 383, 128, False),
    # d = 32: the d = 64 kernel on tiles zero-filled past feature 32
    (1, 1, 1, 32, True), (1, 1, 64, 32, False), (1, 2, 300, 32, True), (2, 1, 129, 32, False),
    # d = 256: one query tile per CTA, 64-key tiles, two score buffers
    (1, 1, 1, 256, True), (1, 1, 64, 256, False), (1, 2, 65, 256, True), (1, 1, 128, 256, True),
    (2, 1, 200, 256, False), (1, 2, 300, 256, True), (1, 1, 513, 256, True), (1, 1, 1024, 256, False),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}h{}s{}d{}{}".format(*s[:4], "c" if s[4] else ""))
def test_small_shapes_match_oracle(oracle, shape, dtype):
    B, H, S, d, causal = shape
    w = inputs.Workload("t", B, H, S, d, causal, dtype, 200 + S + d, "normal")
    q, k, v = inputs.make_qkv(w)
    got = run_tc(q, k, v, causal, w.scale).float().cpu().numpy()
    want = oracle.attn(q, k, v, causal, w.scale)
    mx, mean, _ = errors(got, want)
    assert mx <= MAX_TOL and mean <= MEAN_TOL, (mx, mean)


@pytest.mark.parametrize("d", [128, 256])
def test_sharp_softmax_rescale_path(oracle, d):
    """Scores spread over tens of units force repeated O rescaling in TMEM."""
    w = inputs.Workload("sharp", 1, 2, 1024, d, True, "bf16", 9, "normal", sigma_qk=3.0)
    q, k, v = inputs.make_qkv(w)
    got = run_tc(q, k, v, True, w.scale).float().cpu().numpy()
    want = oracle.attn(q, k, v, True, w.scale)
    mx, mean, _ = errors(got, want)
    assert mx <= MAX_TOL and mean <= MEAN_TOL, (mx, mean)


@pytest.mark.parametrize("d", [64, 256])
def test_increasing_scores_rescale_every_tile(oracle, d):
    """Keys whose scores grow with position make the row max rise in every tile."""
    S = 1024
    q = torch.zeros(1, 1, S, d)
    q[..., 0] = 1.0
    k = torch.zeros(1, 1, S, d)
    k[..., 0] = torch.arange(S, dtype=torch.float32) * 1.1  # the max grows ~25 (base 2) per tile
    v = torch.randn(1, 1, S, d, generator=torch.Generator().manual_seed(3))
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    for causal in (False, True):
        got = run_tc(q, k, v, causal, d ** -0.5).float().cpu().numpy()
        want = oracle.attn(q, k, v, causal, d ** -0.5)
        mx, mean, _ = errors(got, want)
        assert mx <= MAX_TOL and mean <= MEAN_TOL, (causal, mx, mean)


def test_constant_values_give_constant_output():
    w = inputs.Workload("const", 1, 2, 384, 128, True, "bf16", 11, "normal")
    q, k, _ = inputs.make_qkv(w)
    v = torch.full(q.shape, 0.75, dtype=torch.bfloat16)
    got = run_tc(q, k, v, True, w.scale).float()
    assert torch.equal(got, torch.full_like(got, 0.75))


@pytest.mark.parametrize("w", [inputs.BF16_CAUSAL_S4096, inputs.BF16_S2048_D64, inputs.BF16_CAUSAL_S16384,
                               inputs.BF16_CAUSAL_D256], ids=lambda w: w.name)
def test_full_size_workloads_on_sampled_rows(oracle, w):
    q, k, v = inputs.make_qkv(w)
    got = run_tc(q, k, v, w.causal, w.scale)
    heads, rows = inputs.sample_rows(w, per_head=8 if w.S > 8192 else 16)
    flat = got.view(w.N, w.S, w.d)
    got_rows = flat[heads.cuda(), rows.cuda()].float().cpu().numpy()
    want = oracle.attn_rows(q, k, v, w.causal, w.scale, heads.numpy(), rows.numpy())
    mx, mean, _ = errors(got_rows, want)
    assert mx <= MAX_TOL and mean <= MEAN_TOL, (mx, mean)
    # rows the oracle did not evaluate still hold finite values of bounded size
    assert torch.isfinite(got).all()
    assert float(got.abs().max()) <= float(v.abs().max()) + 1e-2


@pytest.mark.parametrize("d", [128, 256])
def test_repeat_calls_are_deterministic(d):
    w = inputs.Workload("det", 2, 2, 512, d, True, "bf16", 13, "normal")
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    a = kbattn.kb_attn_fwd(q, k, v, causal=True, variant=Variant.TC)
    b = kbattn.kb_attn_fwd(q, k, v, causal=True, variant=Variant.TC)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("d,dtype", [(32, "bf16"), (64, "f16"), (128, "bf16"), (256, "bf16")])
def test_output_base_aligned_to_16_bytes_only(oracle, d, dtype):
    """The epilogue writes 32 bytes per store when the output base is 32-byte
    aligned and two 16-byte stores when it is only 16-byte aligned (what the
    boundary accepts): the second path gives the same bits, in place."""
    w = inputs.Workload("t", 1, 2, 300, d, True, dtype, 41 + d, "normal")
    q, k, v = inputs.make_qkv(w)
    wide = run_tc(q, k, v, w.causal, w.scale)
    assert wide.data_ptr() % 32 == 0
    g = Guarded(q.shape, q.dtype, lead=8)  # 8 elements of 2 bytes
    assert g.out.data_ptr() % 32 == 16
    kbattn.kb_attn_fwd(q.cuda(), k.cuda(), v.cuda(), g.out, causal=w.causal, scale=w.scale, variant=Variant.TC)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    narrow = g.check()
    assert torch.equal(narrow, wide)
    mx, mean, _ = errors(narrow.float().cpu().numpy(), oracle.attn(q, k, v, w.causal, w.scale))
    assert mx <= MAX_TOL and mean <= MEAN_TOL, (mx, mean)


def test_tc_rejects_unsupported_head_dim():
    st = kbattn.kb_attn_fwd_ptr(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1, 1, 128, 96, False, 0.17,
                                kbattn.DType.BF16, Variant.TC, 0)
    assert st == kbattn.Status.UNSUPPORTED


@pytest.mark.parametrize("d,dtype", [(64, "bf16"), (128, "f16"), (256, "bf16")])
def test_work_list_schedule_direct_and_graph(oracle, d, dtype):
    """More query units than CTAs, so the host-built per-CTA work lists (a
    grid-constant kernel parameter) drive the kernel: every unit is computed
    exactly once (sampled rows of every head against the oracle, the canaries
    intact), and replaying 20 captured launches in a CUDA graph leaves the same
    bits as one direct launch."""
    S = 2048 if d < 256 else 1024
    w = inputs.Workload("t", 2, 12 if d < 256 else 24, S, d, True, dtype, 31 + d, "normal")
    q, k, v = inputs.make_qkv(w)
    direct = run_tc(q, k, v, w.causal, w.scale)
    g = Guarded(q.shape, q.dtype)
    ms = kbattn.kb_attn_bench_graph(q.cuda(), k.cuda(), v.cuda(), g.out, causal=w.causal, scale=w.scale,
                                    variant=Variant.TC, launches=20, warmup=1, iters=2)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    assert len(ms) == 2 and all(x > 0 for x in ms)
    assert torch.equal(g.check(), direct)
    N = w.B * w.H
    heads = torch.arange(N).repeat_interleave(3)
    rows = torch.tensor([0, S // 2 + 77, S - 1] * N)
    got = direct.reshape(N, S, d)[heads.cuda(), rows.cuda()].float().cpu().numpy()
    want = oracle.attn_rows(q, k, v, w.causal, w.scale, heads.numpy(), rows.numpy())
    mx, mean, _ = errors(got, want)
    assert mx <= MAX_TOL and mean <= MEAN_TOL, (mx, mean)
