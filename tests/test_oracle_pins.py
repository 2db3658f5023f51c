"""Pins for the CPU oracle: it is checked against things other than itself.

The attention pages print no attention output values, so the oracle is pinned
by (1) a brute-force evaluation in high-precision arithmetic on tiny inputs,
written independently (full score matrix, no max subtraction, exact-ish exp),
and (2) closed forms and invariants that the definition
O = softmax(Q K^T * scale [+ causal mask]) V fixes (kbench page, section
"Implementation details / The three GPU kernels"). The Triad a = b + s*c
(TileOPs "Hardware Microbenchmarks" README, section "HBM Bandwidth") is pinned
by exact rational arithmetic and by the STREAM constant check.

``test_each_planted_mistake_fails_a_pin`` recompiles the oracle with one
plausible mistake at a time (dropped term, wrong sign, wrong index, transposed
operand) and checks that at least one pin catches it.
"""
import math
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle as oracle_mod

TOL = 1e-12


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(rng, shape, lo=-1.0, hi=1.0):
    return rng.uniform(lo, hi, size=shape)


# --------------------------------------------------------------------------
# independent brute force
# --------------------------------------------------------------------------
def _brute_force(q, k, v, causal, scale):
    """Full S x S probability matrix in 40-digit arithmetic (mpmath), no max
    subtraction; falls back to math.fsum in double when mpmath is absent."""
    try:
        import mpmath
        mp = mpmath.mp
        mp.dps = 40
        mpf, mexp, msum = mpmath.mpf, mpmath.exp, mpmath.fsum
    except ImportError:  # pragma: no cover - the GPU host has no mpmath
        mpf, mexp, msum = float, math.exp, math.fsum
    B, H, S, d = q.shape
    out = np.zeros(q.shape)
    for b in range(B):
        for h in range(H):
            Q = [[mpf(float(x)) for x in row] for row in q[b, h]]
            K = [[mpf(float(x)) for x in row] for row in k[b, h]]
            V = [[mpf(float(x)) for x in row] for row in v[b, h]]
            # score matrix, entry by entry
            E = [[None] * S for _ in range(S)]
            for i in range(S):
                for j in range(S):
                    if causal and j > i:
                        E[i][j] = mpf(0)
                    else:
                        E[i][j] = mexp(mpf(float(scale)) * msum(Q[i][c] * K[j][c] for c in range(d)))
            for i in range(S):
                Z = msum(E[i])
                for c in range(d):
                    out[b, h, i, c] = float(msum(E[i][j] * V[j][c] for j in range(S)) / Z)
    return out


# --------------------------------------------------------------------------
# pins: each takes an Oracle and raises AssertionError on a violation
# --------------------------------------------------------------------------
def pin_brute_force(orc):
    rng = _rng(11)
    for (B, H, S, d) in [(1, 1, 1, 1), (1, 1, 2, 3), (1, 2, 3, 2), (2, 1, 5, 4), (1, 1, 6, 4), (2, 2, 4, 1)]:
        for causal in (False, True):
            q, k, v = (_rand(rng, (B, H, S, d), -2, 2) for _ in range(3))
            scale = float(rng.uniform(0.2, 1.5))
            got = orc.attn(q, k, v, causal, scale)
            want = _brute_force(q, k, v, causal, scale)
            err = np.max(np.abs(got - want))
            assert err < 1e-13, f"brute force {B,H,S,d} causal={causal}: {err}"


def pin_rows_are_probabilities(orc):
    """With V = I (d = S), O is the probability matrix: rows are >= 0, sum to 1,
    and are zero above the diagonal under the causal mask."""
    rng = _rng(12)
    S = 7
    q, k = _rand(rng, (1, 2, S, S)), _rand(rng, (1, 2, S, S))
    v = np.broadcast_to(np.eye(S), (1, 2, S, S)).copy()
    for causal in (False, True):
        P = orc.attn(q, k, v, causal, 0.9)
        assert np.all(P >= 0)
        assert np.max(np.abs(P.sum(-1) - 1.0)) < TOL
        if causal:
            assert np.all(P[..., np.triu_indices(S, 1)[0], np.triu_indices(S, 1)[1]] == 0.0)
            assert np.all(P[..., np.tril_indices(S)[0], np.tril_indices(S)[1]] > 0.0)
        else:
            assert np.all(P > 0.0)


def pin_constant_v(orc):
    rng = _rng(13)
    q, k = _rand(rng, (2, 2, 9, 4)), _rand(rng, (2, 2, 9, 4))
    const = np.array([0.5, -1.25, 3.0, 7.5])
    v = np.broadcast_to(const, (2, 2, 9, 4)).copy()
    for causal in (False, True):
        o = orc.attn(q, k, v, causal, 0.7)
        assert np.max(np.abs(o - const)) < TOL


def pin_zero_query_is_mean(orc):
    """Q = 0 (or scale = 0): uniform weights, so O is the mean of V over the
    visible keys: all keys, or the running prefix mean under the causal mask."""
    rng = _rng(14)
    S, d = 10, 3
    k, v = _rand(rng, (1, 3, S, d)), _rand(rng, (1, 3, S, d))
    q0 = np.zeros((1, 3, S, d))
    mean = v.mean(axis=2, keepdims=True)
    prefix = np.cumsum(v, axis=2) / np.arange(1, S + 1)[None, None, :, None]
    assert np.max(np.abs(orc.attn(q0, k, v, False, 0.8) - mean)) < TOL
    assert np.max(np.abs(orc.attn(q0, k, v, True, 0.8) - prefix)) < TOL
    q = _rand(rng, (1, 3, S, d))
    assert np.max(np.abs(orc.attn(q, k, v, True, 0.0) - prefix)) < TOL


def pin_causal_first_row_and_single_key(orc):
    rng = _rng(15)
    q, k, v = (_rand(rng, (2, 2, 6, 5)) for _ in range(3))
    o = orc.attn(q, k, v, True, 1.3)
    assert np.array_equal(o[:, :, 0, :], v[:, :, 0, :])
    q1, k1, v1 = (_rand(rng, (2, 3, 1, 4)) for _ in range(3))
    for causal in (False, True):
        assert np.array_equal(orc.attn(q1, k1, v1, causal, 0.5), v1)


def pin_causal_is_prefix_attention(orc):
    """Causal row i equals non-causal attention over keys 0..i only."""
    rng = _rng(16)
    S, d = 8, 3
    q, k, v = (_rand(rng, (1, 1, S, d)) for _ in range(3))
    oc = orc.attn(q, k, v, True, 1.1)
    for i in range(S):
        sub = orc.attn(q[:, :, :i + 1], k[:, :, :i + 1], v[:, :, :i + 1], False, 1.1)
        assert np.max(np.abs(oc[:, :, i] - sub[:, :, i])) < TOL, i


def pin_key_permutation(orc):
    rng = _rng(17)
    q, k, v = (_rand(rng, (1, 2, 9, 4)) for _ in range(3))
    perm = rng.permutation(9)
    a = orc.attn(q, k, v, False, 0.6)
    b = orc.attn(q, k[:, :, perm], v[:, :, perm], False, 0.6)
    assert np.max(np.abs(a - b)) < TOL


def pin_key_shift(orc):
    """Adding one vector u to every key adds q.u to each score of a row: O unchanged."""
    rng = _rng(18)
    q, k, v = (_rand(rng, (1, 2, 7, 4)) for _ in range(3))
    u = _rand(rng, (4,), -3, 3)
    for causal in (False, True):
        a = orc.attn(q, k, v, causal, 0.9)
        b = orc.attn(q, k + u, v, causal, 0.9)
        assert np.max(np.abs(a - b)) < 1e-11


def pin_affine_in_v(orc):
    rng = _rng(19)
    q, k, v = (_rand(rng, (1, 1, 6, 3)) for _ in range(3))
    alpha, beta = -2.5, 0.75
    for causal in (False, True):
        a = orc.attn(q, k, alpha * v + beta, causal, 0.9)
        b = alpha * orc.attn(q, k, v, causal, 0.9) + beta
        assert np.max(np.abs(a - b)) < TOL


def pin_hard_attention_limit(orc):
    """A huge scale with a unique best key turns softmax into argmax; scores of
    order 1e5 also check that exp never overflows."""
    rng = _rng(20)
    S, d = 6, 4
    q, k, v = (_rand(rng, (1, 1, S, d)) for _ in range(3))
    scale = 1e5
    o = orc.attn(q, k, v, False, scale)
    s = q[0, 0] @ k[0, 0].T
    for i in range(S):
        assert np.allclose(o[0, 0, i], v[0, 0, int(np.argmax(s[i]))], atol=1e-12), i
    oc = orc.attn(q, k, v, True, scale)
    for i in range(S):
        assert np.allclose(oc[0, 0, i], v[0, 0, int(np.argmax(s[i, :i + 1]))], atol=1e-12), i


def pin_two_key_closed_form(orc):
    """S = 2, d = 1, q = 1, keys 0 and ln(2)/scale: weights 1/3 and 2/3."""
    scale = 0.5
    q = np.array([1.0, 1.0]).reshape(1, 1, 2, 1)
    k = np.array([0.0, math.log(2.0) / scale]).reshape(1, 1, 2, 1)
    v = np.array([3.0, -6.0]).reshape(1, 1, 2, 1)
    o = orc.attn(q, k, v, False, scale)
    want = (1 * 3.0 + 2 * -6.0) / 3.0
    assert abs(o[0, 0, 0, 0] - want) < 1e-14 and abs(o[0, 0, 1, 0] - want) < 1e-14
    oc = orc.attn(q, k, v, True, scale)
    assert oc[0, 0, 0, 0] == 3.0 and abs(oc[0, 0, 1, 0] - want) < 1e-14


def pin_heads_are_independent(orc):
    """The [B, H, S, d] layout: head (b, h) equals a one-head evaluation of its slice."""
    rng = _rng(21)
    q, k, v = (_rand(rng, (2, 3, 5, 4)) for _ in range(3))
    o = orc.attn(q, k, v, True, 0.7)
    for b in range(2):
        for h in range(3):
            one = orc.attn(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], True, 0.7)
            assert np.array_equal(o[b, h], one[0, 0])


def pin_rows_api_matches_full(orc):
    rng = _rng(22)
    q, k, v = (_rand(rng, (2, 2, 11, 3)) for _ in range(3))
    full = orc.attn(q, k, v, True, 0.8)
    heads = np.array([0, 3, 1, 2, 3])
    rows = np.array([0, 10, 5, 7, 0])
    got = orc.attn_rows(q, k, v, True, 0.8, heads, rows)
    flat = full.reshape(4, 11, 3)
    assert np.array_equal(got, flat[heads, rows])


def pin_threaded_heads_match_full(orc):
    """attn_threads deals heads to host threads: the same bits as one call."""
    rng = _rng(24)
    q, k, v = (_rand(rng, (2, 5, 9, 3)) for _ in range(3))
    for causal in (False, True):
        full = orc.attn(q, k, v, causal, 0.6)
        for threads in (1, 3, 4, 16):
            assert np.array_equal(orc.attn_threads(q, k, v, causal, 0.6, threads=threads), full)


def pin_triad_exact(orc):
    """a = b + s*c rounded once to fp32: compare with exact rational arithmetic."""
    rng = _rng(23)
    n = 4000
    b = rng.uniform(-1, 1, n).astype(np.float32)
    c = rng.uniform(-1, 1, n).astype(np.float32)
    # values whose exact sum sits near a rounding boundary
    b[:1000] = (np.float32(1.0) + rng.integers(0, 1 << 10, 1000).astype(np.float32) * np.float32(2 ** -23))
    c[:1000] = rng.integers(1, 1 << 12, 1000).astype(np.float32) * np.float32(2 ** -30)
    for s in (np.float32(3.0), np.float32(-0.3711), np.float32(1.0e-3)):
        a = orc.triad(b, c, float(s))
        for i in range(0, n, 7):
            exact = Fraction(float(b[i])) + Fraction(float(s)) * Fraction(float(c[i]))
            want = np.float32(_round_to_f32(exact))
            assert a[i] == want, (i, a[i], want)


def _round_to_f32(x: Fraction) -> float:
    """Round an exact rational to the nearest fp32 value, ties to even."""
    f = float(x)  # nearest double; refine to fp32 by exact comparison
    lo = np.float32(f)
    cands = {float(lo), float(np.nextafter(lo, np.float32(np.inf))), float(np.nextafter(lo, np.float32(-np.inf)))}
    best = min(cands, key=lambda y: (abs(Fraction(y) - x), int(np.float32(y).view(np.uint32)) & 1))
    return best


def pin_triad_stream_constants(orc):
    """STREAM's own check: b = 1, c = 2, s = 3 gives a = 7 exactly."""
    b = np.ones(1025, np.float32)
    c = np.full(1025, 2.0, np.float32)
    a = orc.triad(b, c, 3.0)
    assert np.all(a == 7.0)


def pin_lse(orc):
    """log-sum-exp of the score rows: 40-digit brute force, and closed forms."""
    rng = _rng(24)
    try:
        import mpmath
        mpmath.mp.dps = 40
        mexp, mlog, mpf = mpmath.exp, mpmath.log, mpmath.mpf
    except ImportError:  # pragma: no cover
        mexp, mlog, mpf = math.exp, math.log, float
    for (B, H, S, d) in [(1, 1, 1, 2), (1, 2, 5, 3), (2, 1, 6, 4)]:
        for causal in (False, True):
            q, k = _rand(rng, (B, H, S, d), -2, 2), _rand(rng, (B, H, S, d), -2, 2)
            scale = 0.7
            got = orc.lse(q, k, causal, scale)
            for b in range(B):
                for h in range(H):
                    for i in range(S):
                        last = i if causal else S - 1
                        z = sum(mexp(mpf(scale) * sum(mpf(float(q[b, h, i, c])) * mpf(float(k[b, h, j, c]))
                                                      for c in range(d))) for j in range(last + 1))
                        assert abs(got[b, h, i] - float(mlog(z))) < 1e-13
    # Q = 0: every visible score is 0, so lse = log(#visible keys)
    S = 9
    z = orc.lse(np.zeros((1, 2, S, 3)), _rand(rng, (1, 2, S, 3)), True, 0.5)
    assert np.max(np.abs(z - np.log(np.arange(1, S + 1))[None, None, :])) < TOL
    z = orc.lse(np.zeros((1, 2, S, 3)), _rand(rng, (1, 2, S, 3)), False, 0.5)
    assert np.max(np.abs(z - math.log(S))) < TOL
    # S = 1: lse is the single score; huge scores do not overflow (the max is subtracted)
    q, k = _rand(rng, (1, 1, 1, 4)), _rand(rng, (1, 1, 1, 4))
    assert abs(orc.lse(q, k, False, 1e5)[0, 0, 0] - 1e5 * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-6
    # shifting every key by u shifts row i by scale * q_i . u
    q, k = _rand(rng, (1, 1, 7, 3)), _rand(rng, (1, 1, 7, 3))
    u = _rand(rng, (3,), -2, 2)
    d0, d1 = orc.lse(q, k, True, 0.9), orc.lse(q, k + u, True, 0.9)
    assert np.max(np.abs(d1 - d0 - 0.9 * (q[0, 0] @ u))) < 1e-12


def pin_hbm_reference_kernels(orc):
    """copy, fill and sum on values whose exact results are known."""
    b = (np.arange(1, 5001) % 97).astype(np.float32)
    assert np.array_equal(orc.copy(b), b)
    assert np.all(orc.fill(3001, -2.5) == np.float32(-2.5)) and orc.fill(3001, 1.0).size == 3001
    assert orc.sum(b) == float(sum(int(x) for x in b))          # small integers: exact
    assert orc.sum(np.full(1 << 12, 0.25, np.float32)) == 1024.0
    assert orc.sum(np.zeros(0, np.float32)) == 0.0


PINS = [pin_brute_force, pin_rows_are_probabilities, pin_constant_v, pin_zero_query_is_mean,
        pin_causal_first_row_and_single_key, pin_causal_is_prefix_attention, pin_key_permutation,
        pin_key_shift, pin_affine_in_v, pin_hard_attention_limit, pin_two_key_closed_form,
        pin_heads_are_independent, pin_rows_api_matches_full, pin_threaded_heads_match_full, pin_triad_exact,
        pin_triad_stream_constants, pin_hbm_reference_kernels, pin_lse]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin, oracle):
    pin(oracle)


def test_oracle_rejects_bad_arguments(oracle):
    q = np.zeros((1, 1, 0, 4))
    with pytest.raises(ValueError):
        oracle.attn(q, q, q, False, 1.0)
    q = np.zeros((1, 1, 2, 4))
    with pytest.raises(ValueError):
        oracle.attn(q, q, q, False, float("nan"))
    with pytest.raises(ValueError):
        oracle.attn_rows(q, q, q, False, 1.0, [0], [2])


# --------------------------------------------------------------------------
# planted mistakes: every one must fail at least one pin
# --------------------------------------------------------------------------
MUTANTS = {
    "transposed_key_operand": ("dot += qi[c] * kh[j * d + c];", "dot += qi[c] * kh[c * S + j];"),
    "dropped_scale": ("p[j] = scale * dot;", "p[j] = dot;"),
    "mask_off_by_one": ("int64_t last = causal ? i : S - 1;",
                        "int64_t last = causal ? (i > 0 ? i - 1 : 0) : S - 1;"),
    "no_causal_mask": ("int64_t last = causal ? i : S - 1;", "int64_t last = S - 1;"),
    "exp_sign": ("p[j] = exp(p[j] - m);", "p[j] = exp(m - p[j]);"),
    "min_instead_of_max": ("if (p[j] > m) m = p[j];", "if (p[j] < m) m = p[j];"),
    "dropped_normalisation": ("o_row[c] = acc / l;", "o_row[c] = acc;"),
    "wrong_head_index_k": ("const double* kh = k + n * S * d;", "const double* kh = k;"),
    "wrong_query_index": ("const double* qi = q + (n * S + i) * d;", "const double* qi = q + (n * S) * d;"),
    "wrong_value_column": ("acc += p[j] * vh[j * d + c];", "acc += p[j] * vh[j * d];"),
    "dropped_first_key": ("for (int64_t j = 0; j <= last; ++j) {\n    p[j] = exp",
                          "p[0] = 0.0;\n  for (int64_t j = 1; j <= last; ++j) {\n    p[j] = exp"),
    "triad_two_roundings": ("a[i] = fmaf(s, c[i], b[i]);", "a[i] = b[i] + s * c[i];"),
    "triad_swapped_operands": ("a[i] = fmaf(s, c[i], b[i]);", "a[i] = fmaf(s, b[i], c[i]);"),
    "copy_off_by_one": ("for (int64_t i = 0; i < n; ++i) a[i] = b[i];",
                        "for (int64_t i = 1; i < n; ++i) a[i] = b[i - 1];"),
    "lse_drops_max": ("      lse[n * S + i] = m + log(l);", "      lse[n * S + i] = log(l);"),
    "sum_drops_last": ("for (int64_t i = 0; i < n; ++i) acc += (double)b[i];",
                       "for (int64_t i = 0; i + 1 < n; ++i) acc += (double)b[i];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_each_planted_mistake_fails_a_pin(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new = MUTANTS[name]
    src = open(oracle_mod.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique in the oracle source"
    mutated = tmp_path / "attn_oracle_mutant.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle_mod.build(str(mutated), str(tmp_path / "libmutant.so"), force=True)
    mutant = oracle_mod.Oracle(lib)
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mutant)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name!r} passed every pin"
