"""GPU parity of the tensor-core sequence sweep: 16 heads, bf16 inputs with fp32
accumulation, d = 64 and 128, non-causal, S = 128 ... 16384, launched through
kb_attn_fwd exactly as the harness times it. Up to S = 2048 every output
element is compared with the oracle (run over the heads on the host's threads);
at longer S every element is checked written and finite, and seeded rows of
every head, the first and the last included, are compared with the oracle
(rows are independent problems, so a sampled row is exact). Tolerance:
max-abs <= 2e-2 and mean-abs <= 2e-3 against the oracle on the bf16-rounded
inputs."""
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
WHOLE_UP_TO = 2048


@pytest.fixture(scope="module", autouse=True)
def lib():
    from roofline_benchmarking_gb300 import build
    build.build()
    return kbattn.load()


@pytest.mark.parametrize("w", inputs.TC_SWEEP, ids=lambda w: w.name)
def test_tc_sweep_matches_oracle(oracle, w):
    q, k, v = inputs.make_qkv(w)
    g = Guarded(q.shape, q.dtype)
    kbattn.kb_attn_fwd(q.cuda(), k.cuda(), v.cuda(), g.out, causal=w.causal, scale=w.scale, variant=Variant.TC)
    assert kbattn.kb_check_device_error() == kbattn.Status.OK
    got = g.check()
    assert torch.isfinite(got).all()
    flat = got.view(w.N, w.S, w.d)
    if w.S <= WHOLE_UP_TO:
        want = oracle.attn_threads(q, k, v, w.causal, w.scale).reshape(w.N, w.S, w.d)
        mx, mean, _ = errors(flat.float().cpu().numpy(), want)
    else:
        heads, rows = inputs.sample_rows(w, per_head=24)
        got_rows = flat[heads.cuda(), rows.cuda()].float().cpu().numpy()
        want = oracle.attn_rows(q, k, v, w.causal, w.scale, heads.numpy(), rows.numpy())
        mx, mean, _ = errors(got_rows, want)
    assert mx <= MAX_TOL and mean <= MEAN_TOL, (w.name, mx, mean)
