"""Pins of the oracle's Q15 fixed-point model (kbench page, "CPU reference +
cache profiling": Q15 inputs, Q15.16 score accumulation, a 64-entry exp table;
"ARM Cortex-M4 firmware": one row at a time, online-rescaled softmax).

Each pin checks the model against something other than itself: the table
against 50-digit arithmetic, exact results that follow from the model's stated
readings in special cases (computed here with Python fractions), bounds that
follow from the table's resolution, a structural property of the causal mask,
and the page's own accuracy figures (under 5 % relative L2, about 1e-2)
against the double-precision oracle. Planted mistakes must each fail a pin."""
from fractions import Fraction
import math
import shutil

import mpmath
import numpy as np
import pytest
import torch

import oracle as oracle_mod
from roofline_benchmarking_gb300 import inputs


def _round_half_away(x: Fraction) -> int:
    return int(math.floor(x + Fraction(1, 2))) if x >= 0 else -int(math.floor(-x + Fraction(1, 2)))


def pin_exp_table(o):
    """T[f] = round(2^15 * 2^(-f/64)), f = 0..63, from 50-digit arithmetic."""
    mpmath.mp.dps = 50
    want = [int(mpmath.nint(mpmath.mpf(32768) * mpmath.power(2, mpmath.mpf(-f) / 64))) for f in range(64)]
    got = o.q15_exp_table().tolist()
    assert got == want, (got[:4], want[:4])
    assert got[0] == 32768 and all(a > b for a, b in zip(got, got[1:]))


def pin_single_key_is_exact(o):
    """One visible key: its weight is 2^15, so O = V bit for bit (S = 1, and
    causal row 0 for any S)."""
    w = inputs.Q15_SINGLE_HEAD.with_(S=1)
    q, k, v = inputs.make_qkv(w)
    assert np.array_equal(o.attn_q15(q, k, v, False, w.scale), v.numpy())
    w = inputs.Q15_SINGLE_HEAD.with_(S=40, seed=5)
    q, k, v = inputs.make_qkv(w)
    out = o.attn_q15(q, k, v, True, w.scale)
    assert np.array_equal(out[..., 0, :], v.numpy()[..., 0, :])


def pin_zero_query_is_rounded_mean(o):
    """Q = 0: every score is 0, no rescale ever happens and every weight is
    2^15, so o_c = round(sum_j v_jc / count) (halves away from zero) exactly,
    with count = S (or i + 1 under the causal mask)."""
    w = inputs.Q15_SINGLE_HEAD.with_(S=75, d=8, seed=9)
    _, k, v = inputs.make_qkv(w)
    q = torch.zeros_like(k)
    vv = v.numpy()[0, 0].astype(np.int64)
    for causal in (False, True):
        out = o.attn_q15(q, k, v, causal, w.scale)[0, 0]
        for i in (0, 1, 31, 32, 33, 74):
            cnt = i + 1 if causal else w.S
            want = [_round_half_away(Fraction(int(vv[:cnt, c].sum()), cnt)) for c in range(w.d)]
            assert out[i].tolist() == want, (causal, i)


def _hard_case(S=100, d=4, top=70):
    q = torch.zeros(1, 1, S, d, dtype=torch.int16)
    q[..., 0] = 32767
    k = torch.zeros_like(q)
    k[0, 0, top, 0] = 32767
    g = torch.Generator().manual_seed(2)
    v = inputs.to_q15(torch.rand(1, 1, S, d, generator=g) * 2 - 1)
    return q, k, v


def pin_hard_attention_after_rescale(o):
    """One key whose score is 20*log2(e) > 16 base-2 units above the rest, in
    the third tile: the rescale by 2^(-28) sends everything earlier to 0 and the
    later keys' weights are 0, so every row that sees that key returns its value
    row exactly; causal rows before it see only equal scores (rounded mean)."""
    q, k, v = _hard_case()
    out = o.attn_q15(q, k, v, False, 20.0)[0, 0]
    assert np.array_equal(out, np.broadcast_to(v.numpy()[0, 0, 70], out.shape))
    out = o.attn_q15(q, k, v, True, 20.0)[0, 0]
    assert np.array_equal(out[70:], np.broadcast_to(v.numpy()[0, 0, 70], out[70:].shape))
    vv = v.numpy()[0, 0].astype(np.int64)
    for i in (0, 5, 69):
        want = [_round_half_away(Fraction(int(vv[:i + 1, c].sum()), i + 1)) for c in range(4)]
        assert out[i].tolist() == want, i


def pin_two_keys_within_table_resolution(o):
    """Two keys with scores x0 > x1 (natural units): the true weight of key 1 is
    w = 1 / (1 + e^(x0 - x1)). The model's base-2 gap t is floored to the table's
    1/64 step and the entry is rounded to 2^-15, and the product C is floored, so
    its weight lies in [w(t), w(t - 1/64)] up to 2 units in the last place; the
    output is the convex combination with that weight."""
    d = 1
    for q0, k1, scale in ((20000, 9000, 3.0), (30000, -20000, 1.0), (16384, 8192, 7.5), (32767, 1, 0.8)):
        q = torch.tensor([[[[q0], [q0]]]], dtype=torch.int16)
        k = torch.tensor([[[[32767], [k1]]]], dtype=torch.int16)
        v = torch.tensor([[[[-30000], [30000]]]], dtype=torch.int16)
        out = int(o.attn_q15(q, k, v, False, scale)[0, 0, 0, 0])
        x0 = q0 * 32767 / 2 ** 30 * scale
        x1 = q0 * k1 / 2 ** 30 * scale
        t = (x0 - x1) * math.log2(math.e)
        lo_w = 1 / (1 + 2 ** t)
        hi_w = 1 / (1 + 2 ** max(t - 1 / 64 - 2 ** -14, 0.0))
        lo = -30000 + 60000 * lo_w - 2
        hi = -30000 + 60000 * hi_w + 2
        assert lo <= out <= hi, (q0, k1, scale, lo, out, hi)


def pin_causal_row_is_prefix_problem(o):
    """Under the causal mask row i is the last row of the non-causal problem on
    keys 0..i, bit for bit (the mask is exactly a truncation)."""
    w = inputs.Q15_SINGLE_HEAD.with_(S=97, d=16, seed=13)
    q, k, v = inputs.make_qkv(w)
    full = o.attn_q15(q, k, v, True, w.scale)[0, 0]
    for i in (0, 31, 32, 63, 64, 96):
        sub = o.attn_q15(q[..., :i + 1, :], k[..., :i + 1, :], v[..., :i + 1, :], False, w.scale)[0, 0]
        assert np.array_equal(full[i], sub[i]), i


def pin_accuracy_against_double_oracle(o):
    """The page's figures for the fixed-point path: under 5 % relative L2
    against the floating-point reference, error about 1e-2. Checked on the
    fp32 workloads' shapes and draws (with Q15 inputs), against the double
    oracle run on the exact values the Q15 inputs stand for."""
    for w in (inputs.Q15_SINGLE_HEAD, inputs.Q15_S1024.with_(H=2), inputs.Q15_S1024_CAUSAL.with_(H=2)):
        q, k, v = inputs.make_qkv(w)
        got = o.attn_q15(q, k, v, w.causal, w.scale).astype(np.float64) / 32768
        ref = o.attn(inputs.from_q15(q), inputs.from_q15(k), inputs.from_q15(v), w.causal, w.scale)
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel < 2e-2, (w.name, rel)
        assert np.abs(got - ref).max() < 1e-2, w.name


PINS = [pin_exp_table, pin_single_key_is_exact, pin_zero_query_is_rounded_mean, pin_hard_attention_after_rescale,
        pin_two_keys_within_table_resolution, pin_causal_row_is_prefix_problem, pin_accuracy_against_double_oracle]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_q15_pin(oracle, pin):
    pin(oracle)


def test_q15_rejects_out_of_range_arguments(oracle):
    z = torch.zeros(1, 1, 4, 4, dtype=torch.int16)
    for scale in (0.0, -1.0, float("inf"), float("nan"), 1e5):
        with pytest.raises(ValueError):
            oracle.attn_q15(z, z, z, False, scale)


MUTANTS = {
    "q15_score_shift": ("const int64_t s16 = q15_floor_shift(dot, 14);",
                        "const int64_t s16 = q15_floor_shift(dot, 13);"),
    "q15_dropped_scale": ("z[j - t0] = q15_floor_shift(s16 * C, 16);", "z[j - t0] = s16;"),
    "q15_table_step": ("(uint16_t)llround(32768.0 * exp2(-(double)f / 64.0));",
                       "(uint16_t)llround(32768.0 * exp2(-(double)f / 32.0));"),
    "q15_fraction_bits": ("const int64_t f = (t % 65536) / 1024;", "const int64_t f = (t % 65536) / 2048;"),
    "q15_no_rescale": ("    } else if (mt > m) {", "    } else if (0) {"),
    "q15_rescale_l_only": ("for (int64_t c = 0; c < d; ++c) acc[c] = q15_floor_shift(acc[c] * a, 15);", ""),
    "q15_truncating_division": ("return a >= 0 ? (a + b / 2) / b : -((-a + b / 2) / b);", "return a / b;"),
    "q15_first_key_as_tile_max": ("if (j == t0 || z[j - t0] > mt) mt = z[j - t0];",
                                  "if (j == t0) mt = z[j - t0];"),
    "q15_mask_off_by_one": ("const int64_t last_key = causal ? i : S - 1;",
                            "const int64_t last_key = causal ? (i > 0 ? i - 1 : 0) : S - 1;"),
    "q15_clipped_tile_drops_last_key": ("t0 + KB_Q15_TILE - 1 : last_key;",
                                        "t0 + KB_Q15_TILE - 1 : last_key - (last_key > t0);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_each_planted_q15_mistake_fails_a_pin(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTANTS[name]
    src = open(oracle_mod.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    mutated = tmp_path / "attn_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    mutant = oracle_mod.Oracle(oracle_mod.build(str(mutated), str(tmp_path / "libmutant.so"), force=True))
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, ValueError, OverflowError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passed every pin"
