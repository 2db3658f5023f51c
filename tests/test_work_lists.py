"""The tensor-core path's per-CTA work lists (host logic, no GPU): every query
unit is scheduled exactly once, the lists have the properties of list
scheduling in a head-grouped heaviest-first order, and the kernel's fallback
cases are reported. The lists decide which CTA computes which rows, so a unit
missing here would be a block of output rows never written."""
import collections

import pytest

from roofline_benchmarking_gb300 import build as kb_build
from roofline_benchmarking_gb300 import kbattn

GROUP_KV_BYTES = 32 * 1024 * 1024  # the L2 share of one head group (include/kbattn.h)

# (N heads, S, d, causal, grid): the bench workload, the long sharp one, d = 64
# non-causal, d = 256, a ragged sequence length and a grid that is not the SM count
SHAPES = [(64, 4096, 128, True, 152), (32, 16384, 128, True, 152), (192, 2048, 64, False, 152),
          (32, 4096, 256, True, 152), (24, 3000, 128, True, 152), (40, 2048, 32, True, 100)]


@pytest.fixture(scope="module", autouse=True)
def lib():
    kb_build.build()
    return kbattn.load()


def geometry(S, d):
    """Rows per unit and keys per key tile of the kernel that runs d."""
    return (128, 64) if d == 256 else (256, 128)


def unit_cost(t, S, d, causal):
    rows, keys = geometry(S, d)
    nkv = -(-S // keys)
    tiles = min((rows // keys) * (t + 1), nkv) if causal else nkv
    return tiles + 1.0


def head_group(n, N, S, d):
    groups = max(1, min(N, -(-(N * 2 * S * d * 2) // GROUP_KV_BYTES)))
    for g in range(groups):
        if N * g // groups <= n < N * (g + 1) // groups:
            return g
    raise AssertionError(n)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "n{}s{}d{}{}g{}".format(*s[:3], "c" if s[3] else "", s[4]))
def test_every_unit_once_and_list_scheduling_invariants(shape):
    N, S, d, causal, grid = shape
    rows, _ = geometry(S, d)
    units = -(-S // rows)
    lists = kbattn.kb_attn_work_lists(N, S, d, causal, grid)
    assert lists is not None and len(lists) == grid
    seen = collections.Counter(u for lst in lists for u in lst)
    assert set(seen) == {(n, t) for n in range(N) for t in range(units)}
    assert max(seen.values()) == 1
    cost = lambda u: unit_cost(u[1], S, d, causal)
    loads = [sum(cost(u) for u in lst) for lst in lists]
    # each unit went to a least-loaded CTA, and loads only grow: a CTA's load
    # before its last unit is at most every CTA's final load
    for lst, load in zip(lists, loads):
        if lst:
            assert load - cost(lst[-1]) <= min(loads) + 1e-9
    # the heads are visited group by group, each group heaviest unit first
    for lst in lists:
        keys = [(head_group(n, N, S, d), -cost((n, t))) for n, t in lst]
        assert keys == sorted(keys)


@pytest.mark.parametrize("shape,floor", [((64, 4096, 128, True, 152), 0.985), ((32, 16384, 128, True, 152), 0.985),
                                         ((32, 4096, 256, True, 152), 0.98)],
                         ids=["bench", "s16384", "d256"])
def test_modelled_balance_of_the_benchmarked_shapes(shape, floor):
    N, S, d, causal, grid = shape
    loads = [sum(unit_cost(t, S, d, causal) for _, t in lst) for lst in kbattn.kb_attn_work_lists(*shape)]
    assert sum(loads) / len(loads) / max(loads) >= floor


def test_first_round_stays_in_the_first_head_group():
    # bench workload: 64 heads x 2 MiB of K and V -> 4 groups of 16 heads; all
    # 152 CTAs start on group 0, so the concurrently streamed K/V fits in L2
    lists = kbattn.kb_attn_work_lists(64, 4096, 128, True, 152)
    assert {lst[0][0] for lst in lists} <= set(range(16))


def test_lists_are_deterministic():
    a = kbattn.kb_attn_work_lists(32, 16384, 128, True, 152)
    b = kbattn.kb_attn_work_lists(32, 16384, 128, True, 152)
    assert a == b


@pytest.mark.parametrize("args", [(1, 512, 128, True, 2),      # no more units than CTAs
                                  (4096, 4096, 128, True, 152),  # more than 4096 units
                                  (64, 4096, 128, True, 300)],   # more CTAs than the table holds
                         ids=["units<=grid", "units>4096", "grid>256"])
def test_fallback_cases_report_no_lists(args):
    assert kbattn.kb_attn_work_lists(*args) is None


@pytest.mark.parametrize("args", [(0, 4096, 128, True, 152), (8, 0, 128, True, 152), (8, 4096, 96, True, 152),
                                  (8, 4096, 128, True, 0)], ids=["N0", "S0", "d96", "grid0"])
def test_invalid_arguments_are_rejected(args):
    with pytest.raises(RuntimeError):
        kbattn.kb_attn_work_lists(*args)
