"""GPU parity of the three fp32 CUDA-core variants (naive, fused-row, flash)
against the oracle, element by element, max-abs <= 1e-4 (the fp32 tolerance)."""
import numpy as np
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import Variant
from tests.gpu_util import Guarded, errors

pytestmark = pytest.mark.gpu

F32_TOL = 1e-4
VARIANTS = [Variant.NAIVE, Variant.FUSED, Variant.FLASH]


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


def run(w, variant, use_ws=False):
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    g = Guarded(q.shape, torch.float32)
    if use_ws:
        nbytes = kbattn.kb_attn_workspace_bytes(w.B, w.H, w.S, w.d, kbattn.DType.F32, variant)
        ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
        kbattn.kb_attn_fwd_ws(q, k, v, g.out, ws, causal=w.causal, scale=w.scale, variant=variant)
    else:
        kbattn.kb_attn_fwd(q, k, v, g.out, causal=w.causal, scale=w.scale, variant=variant)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    return g.check().cpu().numpy()


SMALL = [  # (B, H, S, d, causal): single tiles, several tiles, ragged tails, S = 1
    (1, 1, 1, 32, False), (1, 2, 1, 64, True), (1, 1, 7, 64, True), (2, 1, 64, 32, False),
    (1, 2, 65, 128, True), (1, 1, 129, 64, False), (2, 3, 200, 32, True), (1, 2, 255, 128, False),
    (1, 1, 256, 64, True), (1, 1, 300, 128, True),
]


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: v.name)
@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "b{}h{}s{}d{}{}".format(*s[:4], "c" if s[4] else ""))
def test_small_shapes_match_oracle(oracle, variant, shape):
    B, H, S, d, causal = shape
    w = inputs.Workload("t", B, H, S, d, causal, "f32", 100 + S + d, "uniform")
    got = run(w, variant)
    want = oracle.attn(*inputs.make_qkv(w), causal, w.scale)
    mx, mean, _ = errors(got, want)
    assert mx <= F32_TOL, (mx, mean)


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: v.name)
@pytest.mark.parametrize("w", [inputs.SINGLE_HEAD_F32, inputs.F32_S1024, inputs.F32_S1024_CAUSAL],
                         ids=lambda w: w.name)
def test_f32_workloads_match_oracle(oracle, variant, w):
    got = run(w, variant)
    want = oracle.attn(*inputs.make_qkv(w), w.causal, w.scale)
    mx, mean, rel = errors(got, want)
    assert mx <= F32_TOL, (mx, mean, rel)


@pytest.fixture(scope="module")
def sweep_oracle(oracle):
    cache = {}

    def get(w):
        if w.name not in cache:
            cache[w.name] = oracle.attn_threads(*inputs.make_qkv(w), w.causal, w.scale)
        return cache[w.name]
    return get


@pytest.mark.parametrize("variant", VARIANTS, ids=lambda v: v.name)
@pytest.mark.parametrize("w", inputs.KBENCH_SWEEP, ids=lambda w: w.name)
def test_kbench_sequence_sweep_matches_oracle(sweep_oracle, variant, w):
    """The kbench page's own sweep (16 heads, d = 64, S = 128 ... 2048), every
    element of every variant against the oracle."""
    got = run(w, variant)
    mx, mean, rel = errors(got, sweep_oracle(w))
    assert mx <= F32_TOL, (mx, mean, rel)


def test_naive_with_caller_workspace_matches_cached(oracle):
    w = inputs.F32_S1024_CAUSAL.with_(H=2, S=320)
    a = run(w, Variant.NAIVE, use_ws=False)
    b = run(w, Variant.NAIVE, use_ws=True)
    assert np.array_equal(a, b)


def test_variants_agree_on_scale_and_large_scores(oracle):
    """A large scale makes the softmax sharp: every variant must still match."""
    w = inputs.Workload("sharp", 1, 2, 192, 64, True, "f32", 7, "uniform")
    q, k, v = inputs.make_qkv(w)
    q = (q * 6).contiguous()
    want = oracle.attn(q, k, v, True, 2.0)
    for variant in VARIANTS:
        g = Guarded(q.shape, torch.float32)
        kbattn.kb_attn_fwd(q.cuda(), k.cuda(), v.cuda(), g.out, causal=True, scale=2.0, variant=variant)
        mx, _, _ = errors(g.check().cpu().numpy(), want)
        assert mx <= F32_TOL, (variant, mx)


def test_fused_rejects_rows_longer_than_shared_memory():
    info = kbattn.kb_device_info(torch.cuda.current_device())
    S = info["smem_per_block_optin"] // 4 + 1024
    st = kbattn.kb_attn_fwd_ptr(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1, 1, S, 64, False, 0.125,
                                kbattn.DType.F32, Variant.FUSED, 0)
    assert st == kbattn.Status.UNSUPPORTED


@pytest.mark.parametrize("variant", VARIANTS + [Variant.TC], ids=lambda v: v.name)
def test_graph_replay_matches_oracle(oracle, variant):
    """The CUDA-graph timing path (200 captured launches of the smallest
    workload) leaves the same output as one plain call."""
    w = inputs.SINGLE_HEAD_F32
    if variant == Variant.TC:
        w = inputs.Workload("t", 1, 1, 64, 64, False, "bf16", 0, "uniform")
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    g = Guarded(q.shape, q.dtype)
    ms = kbattn.kb_attn_bench_graph(q, k, v, g.out, causal=w.causal, scale=w.scale, variant=variant,
                                    launches=200, warmup=2, iters=3)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    assert len(ms) == 3 and all(x > 0 for x in ms)
    got = g.check().float().cpu().numpy()
    want = oracle.attn(*inputs.make_qkv(w), w.causal, w.scale)
    mx, _, _ = errors(got, want)
    assert mx <= (F32_TOL if variant != Variant.TC else 2e-2), mx


@pytest.mark.parametrize("shape", [(1, 8, 1023, 64, False), (1, 8, 1021, 64, True), (2, 4, 777, 32, True),
                                   (1, 4, 513, 128, False), (1, 3, 1030, 128, True), (1, 4, 2047, 64, True),
                                   (1, 2, 2046, 32, False)],
                         ids=lambda s: "b{}h{}s{}d{}{}".format(*s[:4], "c" if s[4] else ""))
def test_fused_multi_row_blocks_with_ragged_tails(oracle, shape):
    """Grids large enough that the fused-row kernel takes several query rows
    per block: eight where two such blocks fit in one SM's shared memory (the
    S ~ 1000 shapes at d <= 64 and S = 2046 at d = 32), else four (S = 2047 at
    d = 64, and d = 128). S is not a
    multiple of the rows per block (the last block of each head is partial) nor
    of the 64-key tile or the 4-key quad, and causal rows' key ranges differ
    within a block."""
    B, H, S, d, causal = shape
    w = inputs.Workload("t", B, H, S, d, causal, "f32", 500 + S, "uniform")
    got = run(w, Variant.FUSED)
    want = oracle.attn(*inputs.make_qkv(w), causal, w.scale)
    mx, mean, _ = errors(got, want)
    assert mx <= F32_TOL, (mx, mean)


@pytest.mark.parametrize("shape", [(1, 8, 1024, 64), (1, 3, 700, 128), (2, 2, 333, 32)],
                         ids=lambda s: "b{}h{}s{}d{}".format(*s))
def test_flash_causal_split_paths(oracle, shape):
    """Causal fp32 flash on a small grid runs the heavier half of its query tiles
    as two blocks over two key ranges (partial states in a workspace, combined by
    a merge kernel). The library's cached workspace and a caller's full workspace
    give the same bits; a caller's too-small workspace runs every tile whole; all
    three are within the fp32 tolerance of the oracle."""
    B, H, S, d = shape
    w = inputs.Workload("split", B, H, S, d, True, "f32", 500 + S, "uniform")
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    want = oracle.attn(*inputs.make_qkv(w), True, w.scale)
    nbytes = kbattn.kb_attn_workspace_bytes(B, H, S, d, kbattn.DType.F32, Variant.FLASH)
    assert nbytes > 0
    outs = []
    for ws in (None, torch.empty(nbytes, dtype=torch.uint8, device="cuda"),
               torch.empty(16, dtype=torch.uint8, device="cuda")):
        g = Guarded(q.shape, torch.float32)
        if ws is None:
            kbattn.kb_attn_fwd(q, k, v, g.out, causal=True, scale=w.scale, variant=Variant.FLASH)
        else:
            kbattn.kb_attn_fwd_ws(q, k, v, g.out, ws, causal=True, scale=w.scale, variant=Variant.FLASH)
        assert kbattn.kb_check_device_error() == kbattn.Status.OK
        got = g.check()
        mx, _, _ = errors(got.cpu().numpy(), want)
        assert mx <= F32_TOL, mx
        outs.append(got)
    assert torch.equal(outs[0], outs[1])
