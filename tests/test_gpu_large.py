"""Tensors of more than 2^31 elements. The last heads of such a problem sit at
element offsets past 2^31, where an index computed in 32 bits would wrap, so
each kernel family runs one (inputs drawn on the device, sequence length 1024
to keep the work small) and is compared with the oracle on sampled rows of the
first, a middle and the last head (the Q15 path bit-exact on those whole
heads). The poisoned guards around every output check that each element was
written and nothing outside it. About 45 GB of device memory at most."""
import numpy as np
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import Variant
from tests.gpu_util import Guarded, errors, run_twice

pytestmark = pytest.mark.gpu

BIG = 1 << 31
S = 1024


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


def heads_of(N):
    return [0, N // 2, N - 1]


def big_workload(name, d, causal, dtype, seed, dist, extra):
    """H heads of S x d, the smallest multiple past 2^31 elements plus ``extra`` heads."""
    w = inputs.Workload(name, 1, BIG // (S * d) + extra, S, d, causal, dtype, seed, dist)
    assert w.N * S * d > BIG
    return w


def sampled_rows(oracle, q, k, v, out, causal, scale):
    """(got, want) for rows 0, S/2 + 77 and S - 1 of the first, a middle and the last head."""
    N, d = q.shape[0] * q.shape[1], q.shape[3]
    heads = heads_of(N)
    rows = [0, S // 2 + 77, S - 1]
    sel = lambda t: t.reshape(N, S, d)[heads].cpu()
    want = oracle.attn_rows(sel(q), sel(k), sel(v), causal, scale,
                            np.repeat(np.arange(len(heads)), len(rows)), np.tile(rows, len(heads)))
    hh = torch.tensor(heads).repeat_interleave(len(rows)).cuda()
    rr = torch.tensor(rows * len(heads)).cuda()
    got = out.reshape(N, S, d)[hh, rr].float().cpu().numpy()
    return got, want


def test_fp32_flash_and_fused_past_2_31_elements(oracle):
    w = big_workload("big_f32", 64, True, "f32", 71, "uniform", 64)
    q, k, v = inputs.make_qkv_device(w)
    for variant in (Variant.FLASH, Variant.FUSED):
        g = Guarded(q.shape, q.dtype)
        kbattn.kb_attn_fwd(q, k, v, g.out, causal=w.causal, scale=w.scale, variant=variant)
        assert kbattn.kb_check_device_error() == kbattn.Status.OK
        got, want = sampled_rows(oracle, q, k, v, g.check(), w.causal, w.scale)
        mx, _, _ = errors(got, want)
        assert mx <= 1e-4, (variant, mx)
        del g
        torch.cuda.empty_cache()


@pytest.mark.parametrize("d", [128, 256])
def test_tensor_core_past_2_31_elements(oracle, d):
    w = big_workload(f"big_tc{d}", d, True, "bf16", 72 + d, "normal", 16)
    q, k, v = inputs.make_qkv_device(w)
    g = Guarded(q.shape, q.dtype)
    kbattn.kb_attn_fwd(q, k, v, g.out, causal=w.causal, scale=w.scale, variant=Variant.TC)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    got, want = sampled_rows(oracle, q, k, v, g.check(), w.causal, w.scale)
    mx, mean, _ = errors(got, want)
    assert mx <= 2e-2 and mean <= 2e-3, (mx, mean)


def test_q15_past_2_31_elements(oracle):
    w = big_workload("big_q15", 64, False, "q15", 74, "uniform", 64)
    q, k, v = inputs.make_qkv_device(w)

    def launch(out):
        kbattn.kb_attn_fwd(q, k, v, out, causal=w.causal, scale=w.scale, variant=Variant.FIXEDPOINT)
        assert kbattn.kb_check_device_error() == kbattn.Status.OK

    out = run_twice(q.shape, torch.int16, launch)
    N = w.N
    heads = heads_of(N)
    sel = lambda t: t.reshape(N, S, w.d)[heads].cpu()
    want = oracle.attn_q15(sel(q), sel(k), sel(v), w.causal, w.scale)
    got = out.reshape(N, S, w.d)[heads].cpu().numpy()
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[0].tolist()}"
