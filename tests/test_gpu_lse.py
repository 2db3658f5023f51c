"""GPU parity of the log-sum-exp output (kb_attn_fwd_lse) against the oracle:
tensor-core kernel (bf16 / f16 inputs, fp32 scores) and fp32 flash kernel.
The row LSE only involves fp32 scores and sums (P's 16-bit rounding does not
enter it), so the tolerance is 1e-3 absolute for the tensor-core kernel and
1e-4 for fp32; O must be bit-identical to kb_attn_fwd's."""
import numpy as np
import pytest
import torch

from roofline_benchmarking_gb300 import inputs
from roofline_benchmarking_gb300 import kbattn
from roofline_benchmarking_gb300.kbattn import Status, Variant
from tests.gpu_util import Guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


CASES = [  # (B, H, S, d, causal, dtype, variant, tol)
    (1, 2, 128, 128, False, "bf16", Variant.TC, 1e-3), (1, 2, 300, 128, True, "bf16", Variant.TC, 1e-3),
    (2, 1, 513, 64, True, "f16", Variant.TC, 1e-3), (1, 3, 1024, 64, False, "bf16", Variant.TC, 1e-3),
    (1, 2, 130, 64, True, "f32", Variant.FLASH, 1e-4), (2, 2, 64, 32, False, "f32", Variant.FLASH, 1e-4),
    # causal fp32 flash on a small grid: the split query tiles' LSE comes from the merge kernel
    (1, 3, 700, 64, True, "f32", Variant.FLASH, 1e-4), (2, 2, 1000, 128, True, "f32", Variant.FLASH, 1e-4),
    (1, 1, 1, 128, True, "bf16", Variant.TC, 1e-3),
    (1, 2, 200, 256, True, "bf16", Variant.TC, 1e-3), (1, 1, 130, 256, False, "f16", Variant.TC, 1e-3),
    (1, 2, 257, 32, True, "bf16", Variant.TC, 1e-3),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}s{}d{}{}-{}".format(*c[:4], "c" if c[4] else "", c[5]))
def test_lse_matches_oracle(oracle, case):
    B, H, S, d, causal, dtype, variant, tol = case
    w = inputs.Workload("lse", B, H, S, d, causal, dtype, 400 + S, "normal" if dtype != "f32" else "uniform",
                        sigma_qk=2.0)
    q, k, v = inputs.make_qkv(w)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    lse = Guarded((B, H, S), torch.float32)
    o, _ = kbattn.kb_attn_fwd_lse(qc, kc, vc, lse=lse.out, causal=causal, scale=w.scale, variant=variant)
    assert kbattn.kb_check_device_error() == Status.OK
    got = lse.check().cpu().numpy()
    want = oracle.lse(q, k, causal, w.scale)
    assert np.max(np.abs(got - want)) <= tol
    o2 = kbattn.kb_attn_fwd(qc, kc, vc, causal=causal, scale=w.scale, variant=variant)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)


def test_lse_full_size_sampled_rows(oracle):
    w = inputs.BF16_CAUSAL_S4096
    q, k, v = inputs.make_qkv(w)
    o, lse = kbattn.kb_attn_fwd_lse(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    heads = [0, 17, 63]
    for n in heads:
        b, h = divmod(n, w.H)
        want = oracle.lse(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], True, w.scale)[0, 0]
        assert np.max(np.abs(lse[b, h].cpu().numpy() - want)) <= 1e-3


def test_lse_unsupported_variants():
    fake = 1 << 20
    L = kbattn.load()
    for variant in (Variant.NAIVE, Variant.FUSED):
        st = L.kb_attn_fwd_lse(fake, fake, fake, fake, fake, 1, 1, 64, 64, 0, 0.125, kbattn.DType.F32, variant, None)
        assert st == Status.UNSUPPORTED
