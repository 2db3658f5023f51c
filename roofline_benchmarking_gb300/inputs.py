"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no attention arithmetic: it only draws random numbers and
rounds them to the storage dtype. Both the CUDA path and the oracle consume the
exact bytes it produces.

Draw recipe (one reading, fixed here): a CPU ``torch.Generator`` seeded with
the workload's seed draws Q, then K, then V, each as a full fp32 [B, H, S, d]
tensor. "uniform" is ``rand * 2 - 1`` (U[-1, 1]); "normal(0, sigma)" is
``randn * sigma`` (sigma is the standard deviation). bf16 workloads then round
each fp32 draw to bf16 with round-to-nearest-even (``Tensor.to(torch.bfloat16)``).
Q15 workloads (int16, value = x / 2^15) round each fp32 draw times 2^15 to the
nearest integer (ties to even) and saturate it to [-32768, 32767].
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    d: int
    causal: bool
    dtype: str          # "f32", "bf16", "f16" or "q15"
    seed: int
    dist: str           # "uniform" or "normal"
    sigma_qk: float = 1.0
    sigma_v: float = 1.0

    @property
    def N(self) -> int:
        return self.B * self.H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """4*B*H*S^2*d, halved when causal (the benchmark's FLOP convention)."""
        f = 4.0 * self.B * self.H * self.S * self.S * self.d
        return f / 2 if self.causal else f

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def io_bytes(self) -> int:
        """Q, K, V read once and O written once."""
        return 4 * self.B * self.H * self.S * self.d * self.elem_bytes

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The pages' workloads, restated. Names say what each one is.
SINGLE_HEAD_F32 = Workload("f32_b1h1s64d32", 1, 1, 64, 32, False, "f32", 0, "uniform")
F32_S1024 = Workload("f32_b1h8s1024d64", 1, 8, 1024, 64, False, "f32", 1, "uniform")
F32_S1024_CAUSAL = F32_S1024.with_(name="f32_b1h8s1024d64_causal", causal=True)
BF16_CAUSAL_S4096 = Workload("bf16_causal_b4h16s4096d128", 4, 16, 4096, 128, True, "bf16", 2, "normal")
BF16_S2048_D64 = Workload("bf16_b16h12s2048d64", 16, 12, 2048, 64, False, "bf16", 3, "normal")
BF16_CAUSAL_S16384 = Workload("bf16_causal_b1h32s16384d128_sharp", 1, 32, 16384, 128, True, "bf16", 4,
                              "normal", sigma_qk=3.0, sigma_v=1.0)
# Head dimension 256 (not among the pages' workloads): the tensor-core path's
# one-query-tile-per-CTA layout, at the bench workload's sequence length.
BF16_CAUSAL_D256 = Workload("bf16_causal_b2h16s4096d256", 2, 16, 4096, 256, True, "bf16", 6, "normal")

# fp16 operands on the tensor-core path: the bench workload's and the d = 64
# workload's shapes and draws, rounded to fp16 instead of bf16.
F16_CAUSAL_S4096 = BF16_CAUSAL_S4096.with_(name="f16_causal_b4h16s4096d128", dtype="f16")
F16_S2048_D64 = BF16_S2048_D64.with_(name="f16_b16h12s2048d64", dtype="f16")

# The Q15 fixed-point model runs on the fp32 workloads' shapes and draws.
Q15_SINGLE_HEAD = SINGLE_HEAD_F32.with_(name="q15_b1h1s64d32", dtype="q15")
Q15_S1024 = F32_S1024.with_(name="q15_b1h8s1024d64", dtype="q15")
Q15_S1024_CAUSAL = F32_S1024_CAUSAL.with_(name="q15_b1h8s1024d64_causal", dtype="q15")

# The kbench page's own sequence sweep (section "Running": --seq 128,256,512,1024,2048
# --heads 16 --dim 64, fp32, every kernel), whose "Expected results" give the
# three variants' relative latency at S = 2048. The page names no batch, seed or
# distribution: one batch, non-causal, U[-1, 1] as in the other fp32 workloads,
# seed 5.
KBENCH_SWEEP_S = (128, 256, 512, 1024, 2048)
KBENCH_SWEEP = tuple(Workload(f"f32_b1h16s{S}d64", 1, 16, S, 64, False, "f32", 5, "uniform")
                     for S in KBENCH_SWEEP_S)

# The same sweep on the tensor-core path: 16 heads, bf16 with fp32 accumulation,
# d = 64 and 128, non-causal, S from 128 to 16384 (from a handful of CTAs to a
# full persistent grid), N(0, 1) draws rounded to bf16, seed 5.
TC_SWEEP_S = (128, 256, 512, 1024, 2048, 4096, 8192, 16384)
TC_SWEEP = tuple(Workload(f"bf16_b1h16s{S}d{d}", 1, 16, S, d, False, "bf16", 5, "normal")
                 for d in (64, 128) for S in TC_SWEEP_S)

WORKLOADS = {w.name: w for w in (SINGLE_HEAD_F32, F32_S1024, F32_S1024_CAUSAL,
                                 BF16_CAUSAL_S4096, BF16_S2048_D64, BF16_CAUSAL_S16384, BF16_CAUSAL_D256,
                                 F16_CAUSAL_S4096, F16_S2048_D64,
                                 Q15_SINGLE_HEAD, Q15_S1024, Q15_S1024_CAUSAL, *KBENCH_SWEEP, *TC_SWEEP)}

# STREAM Triad working set: three fp32 arrays of 2 GiB each.
TRIAD_ARRAY_BYTES = 2 << 30
TRIAD_N = TRIAD_ARRAY_BYTES // 4

_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "q15": torch.int16}


def torch_dtype(dtype: str) -> torch.dtype:
    return _TORCH_DTYPE[dtype]


def make_qkv(w: Workload):
    """Q, K, V for workload ``w`` as CPU tensors of its storage dtype, [B, H, S, d]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    shape = (w.B, w.H, w.S, w.d)
    out = []
    for which in ("q", "k", "v"):
        if w.dist == "uniform":
            x = torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0
        elif w.dist == "normal":
            sigma = w.sigma_v if which == "v" else w.sigma_qk
            x = torch.randn(shape, generator=g, dtype=torch.float32) * sigma
        else:
            raise ValueError(f"unknown distribution {w.dist!r}")
        if w.dtype == "q15":
            out.append(to_q15(x))
        else:
            out.append(x.to(torch_dtype(w.dtype)).contiguous())
    return tuple(out)


def make_qkv_device(w: Workload, device: str = "cuda"):
    """Q, K, V for workload ``w`` drawn directly on ``device`` with that device's
    generator seeded by ``w.seed``: the same distributions and storage rounding
    as ``make_qkv`` (other values: another generator), for problems whose fp32
    draws would not fit comfortably in host memory."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed)
    shape = (w.B, w.H, w.S, w.d)
    out = []
    for which in ("q", "k", "v"):
        if w.dist == "uniform":
            x = torch.rand(shape, generator=g, device=device, dtype=torch.float32).mul_(2.0).sub_(1.0)
        elif w.dist == "normal":
            sigma = w.sigma_v if which == "v" else w.sigma_qk
            x = torch.randn(shape, generator=g, device=device, dtype=torch.float32).mul_(sigma)
        else:
            raise ValueError(f"unknown distribution {w.dist!r}")
        out.append(to_q15(x) if w.dtype == "q15" else x.to(torch_dtype(w.dtype)).contiguous())
        del x
    return tuple(out)


def to_q15(x: torch.Tensor) -> torch.Tensor:
    """Storage rounding to Q15: round(x * 2^15) (ties to even), saturated to int16."""
    return torch.round(x.float() * 32768.0).clamp(-32768, 32767).to(torch.int16).contiguous()


def from_q15(x) -> torch.Tensor:
    """The exact value an int16 Q15 tensor stands for, as float64."""
    return torch.as_tensor(x).double() / 32768.0


def sample_rows(w: Workload, per_head: int = 64, seed: int = 12345):
    """A fixed seeded subset of (head, row) pairs: per head, rows 0 and S-1 plus
    ``per_head - 2`` distinct others. Returns two int64 tensors (heads, rows)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    heads, rows = [], []
    k = min(per_head, w.S)
    for n in range(w.N):
        chosen = {0, w.S - 1}
        if k > len(chosen):
            perm = torch.randperm(w.S, generator=g).tolist()
            for r in perm:
                if len(chosen) >= k:
                    break
                chosen.add(r)
        for r in sorted(chosen):
            heads.append(n)
            rows.append(r)
    return torch.tensor(heads, dtype=torch.int64), torch.tensor(rows, dtype=torch.int64)


def make_triad_inputs(n: int, seed: int = 5):
    """b and c for the Triad as fp32 CPU tensors: U[-1, 1] draws from ``seed``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    b = torch.rand(n, generator=g, dtype=torch.float32) * 2.0 - 1.0
    c = torch.rand(n, generator=g, dtype=torch.float32) * 2.0 - 1.0
    return b, c
