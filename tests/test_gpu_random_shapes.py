"""Seeded random shapes for every GPU path, against the oracle: batch and head
counts, sequence lengths that are rarely multiples of the tile sizes, every
supported head dimension, both masks and both 16-bit types. The shapes are
drawn once from a fixed seed, so a failure names a reproducible case."""
import random

import numpy as np
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import Variant
from tests.gpu_util import Guarded, errors, run_twice

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


def _shapes(seed, count, s_max, dims):
    rnd = random.Random(seed)
    out = []
    for _ in range(count):
        out.append((rnd.randint(1, 3), rnd.randint(1, 3), rnd.randint(1, s_max), rnd.choice(dims),
                    rnd.random() < 0.5))
    return out


def _id(s):
    return "b{}h{}s{}d{}{}".format(*s[:4], "c" if s[4] else "")


TC_SHAPES = _shapes(2024, 14, 700, [32, 64, 128, 256])
F32_SHAPES = _shapes(2025, 12, 400, [32, 64, 128])
Q15_SHAPES = _shapes(2026, 10, 300, [32, 64, 128])


@pytest.mark.parametrize("shape", TC_SHAPES, ids=_id)
def test_tensor_core_random_shapes(oracle, shape):
    B, H, S, d, causal = shape
    dtype = "bf16" if (S + d) % 2 else "f16"
    w = inputs.Workload("r", B, H, S, d, causal, dtype, 7000 + S, "normal", sigma_qk=1.5)
    q, k, v = inputs.make_qkv(w)
    g = Guarded(q.shape, q.dtype)
    kbattn.kb_attn_fwd(q.cuda(), k.cuda(), v.cuda(), g.out, causal=causal, scale=w.scale, variant=Variant.TC)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    got = g.check().float().cpu().numpy()
    mx, mean, _ = errors(got, oracle.attn(q, k, v, causal, w.scale))
    assert mx <= 2e-2 and mean <= 2e-3, (mx, mean)


@pytest.mark.parametrize("variant", [Variant.NAIVE, Variant.FUSED, Variant.FLASH], ids=lambda v: v.name)
@pytest.mark.parametrize("shape", F32_SHAPES, ids=_id)
def test_fp32_random_shapes(oracle, shape, variant):
    B, H, S, d, causal = shape
    w = inputs.Workload("r", B, H, S, d, causal, "f32", 8000 + S, "uniform")
    q, k, v = inputs.make_qkv(w)
    g = Guarded(q.shape, torch.float32)
    kbattn.kb_attn_fwd(q.cuda(), k.cuda(), v.cuda(), g.out, causal=causal, scale=w.scale, variant=variant)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    got = g.check().cpu().numpy()
    mx, _, _ = errors(got, oracle.attn(q, k, v, causal, w.scale))
    assert mx <= 1e-4, mx


@pytest.mark.parametrize("shape", Q15_SHAPES, ids=_id)
def test_fixed_point_random_shapes(oracle, shape):
    B, H, S, d, causal = shape
    w = inputs.Workload("r", B, H, S, d, causal, "q15", 9000 + S, "uniform")
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))

    def launch(out):
        kbattn.kb_attn_fwd(q, k, v, out, causal=causal, scale=w.scale, variant=Variant.FIXEDPOINT)
        assert kbattn.kb_check_device_error() == kbattn.Status.OK

    got = run_twice(q.shape, torch.int16, launch).cpu().numpy()
    want = oracle.attn_q15(*inputs.make_qkv(w), causal, w.scale)
    assert np.array_equal(got, want), int((got != want).sum())
