"""Pins for the oracle's route alignment and the block-membership checks.

What fixes the alignment independently of the oracle:
  * the worked example of "Route-Block Membership Selects Packed-AWQ
    Arithmetic" (M=21, k=8, 128 experts, b=8: 168 valid routes, 400 aligned
    rows, 50 active blocks), reproduced by the closed-form fixture;
  * brute force over every routing of tiny shapes against two independent
    formulations (a comparison sort and a counting sort);
  * the page's invariants: sentinels excluded, a swap inside a block keeps
    the identity, a move across a block boundary changes it;
  * the page's split-K schedule numbers (600 / 492 / 41 / 33).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from top_moe_expert_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _canon_sort(ids, E, b):
    """Comparison-sort formulation: sorted((expert, r)) over valid routes."""
    flat = ids.reshape(-1)
    mk = flat.size
    routes = sorted((int(e), r) for r, e in enumerate(flat) if 0 <= e < E)
    rows, blocks = [], []
    i = 0
    while i < len(routes):
        e = routes[i][0]
        run = [r for (ee, r) in routes if ee == e]
        i += len(run)
        pad = (-len(run)) % b
        rows += run + [mk] * pad
        blocks += [e] * ((len(run) + pad) // b)
    return rows, blocks


def _counting_sort(ids, E, b):
    """Counting-sort formulation: histogram, padded exclusive prefix, scatter."""
    flat = ids.reshape(-1)
    mk = flat.size
    valid = (flat >= 0) & (flat < E)
    cnt = np.bincount(flat[valid], minlength=E)
    padded = -(-cnt // b) * b
    start = np.concatenate([[0], np.cumsum(padded)[:-1]])
    total = int(padded.sum())
    rows = np.full(total, mk, dtype=np.int64)
    fill = np.zeros(E, dtype=np.int64)
    for r in range(mk):
        e = flat[r]
        if 0 <= e < E:
            rows[start[e] + fill[e]] = r
            fill[e] += 1
    blocks = np.repeat(np.arange(E), padded // b)
    return rows.tolist(), blocks.tolist()


def test_fixture_a_reproduces_the_pages_counts():
    g = json.load(open(os.path.join(GOLDEN, "alignment_worked_example.json")))
    ids = inputs.fixture_a_ids(g["M"], g["k"], g["E"])
    sorted_ids, expert_ids, npp, ninv = oracle.align(ids, g["E"], g["b"])
    mk = g["M"] * g["k"]
    valid = int(np.sum(sorted_ids[:npp] != mk))
    blocks = int(np.sum(expert_ids >= 0))
    assert ninv == 0
    assert valid == g["valid_routes"]
    assert npp == g["aligned_rows"]
    assert blocks == g["active_blocks"]
    assert len(np.unique(ids)) == g["active_blocks"]


@pytest.mark.parametrize("M,k,E,b", [(1, 1, 3, 1), (2, 1, 3, 2), (2, 2, 3, 2), (1, 2, 4, 4),
                                     (3, 1, 4, 2), (2, 2, 2, 4)])
def test_alignment_brute_force_all_routings(M, k, E, b):
    # every routing of the tiny shape, including one invalid id value (E)
    for combo in itertools.product(range(E + 1), repeat=M * k):
        ids = np.array(combo, dtype=np.int32).reshape(M, k)
        s, ex, npp, ninv = oracle.align(ids, E, b)
        rows1, blocks1 = _canon_sort(ids, E, b)
        rows2, blocks2 = _counting_sort(ids, E, b)
        assert rows1 == rows2 and blocks1 == blocks2
        assert npp == len(rows1)
        assert s[:npp].tolist() == rows1
        assert ex[:len(blocks1)].tolist() == blocks1
        assert np.all(s[npp:] == M * k) and np.all(ex[len(blocks1):] == -1)
        assert ninv == int(np.sum(ids == E))


def test_alignment_random_against_counting_sort():
    g = np.random.Generator(np.random.PCG64(5))
    for M, k, E, b in [(21, 8, 128, 8), (64, 8, 128, 16), (7, 4, 16, 1), (33, 6, 40, 32)]:
        ids = g.integers(-2, E + 2, size=(M, k)).astype(np.int32)
        s, ex, npp, ninv = oracle.align(ids, E, b)
        rows, blocks = _counting_sort(ids, E, b)
        assert s[:npp].tolist() == rows and ex[:len(blocks)].tolist() == blocks
        assert ninv == int(np.sum((ids < 0) | (ids >= E)))


def test_alignment_capacity_and_history_independence():
    ids = inputs.fixture_a_ids()
    cap_rows, cap_blocks = oracle.align_capacity(21, 8, 128, 8)
    assert cap_rows >= 400
    with pytest.raises(ValueError):
        oracle.align(ids, 128, 8, cap_rows=399, cap_blocks=50)
    # stable construction depends only on the id array: two calls, and a call
    # after an unrelated alignment, agree exactly
    a = oracle.align(ids, 128, 8)
    oracle.align(np.zeros((5, 8), dtype=np.int32), 128, 8)
    b = oracle.align(ids, 128, 8)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def _multi_block_fixture():
    # expert 3 gets 11 routes (two blocks at b=8), expert 9 gets 2
    ids = np.full((13, 1), 3, dtype=np.int32)
    ids[4, 0] = 9
    ids[10, 0] = 9
    return ids


def test_identity_swap_inside_block_preserved_and_across_boundary_changed():
    ids = _multi_block_fixture()
    b, mk = 8, 13
    s, ex, npp, _ = oracle.align(ids, 16, b)
    base = oracle.block_identity(s, ex, npp, b, mk)
    assert [blk[0] for blk in base] == [3, 3, 9]
    # sentinels are excluded: the last block of expert 3 holds 3 routes
    assert len(base[1][2]) == 3 and all(r != mk for blk in base for r in blk[2])
    # swap two routes inside block 0: identity unchanged
    s2 = s.copy()
    s2[1], s2[5] = s2[5], s2[1]
    assert oracle.block_identity(s2, ex, npp, b, mk) == base
    # move a route across the 8-row boundary (swap rows 2 and 9): changed
    s3 = s.copy()
    s3[2], s3[9] = s3[9], s3[2]
    assert oracle.block_identity(s3, ex, npp, b, mk) != base


def test_split_k_schedule_reproduces_the_pages_derivation():
    g = json.load(open(os.path.join(GOLDEN, "split_k_schedule.json")))
    for case in g["cases"]:
        got = oracle.split_k_schedule(g["moe_blocks"], g["N"], g["K"], g["thread_n"],
                                      g["thread_k"], case["grid"])
        assert got["n_tiles"] == g["n_tiles"] and got["k_tiles"] == g["k_tiles"]
        assert got["total_tiles"] == g["total_tiles"]
        assert got["direct_tiles"] == case["direct_tiles"]
        assert got["remainder_start_block"] == case["remainder_start_block"]
        assert got["slices"] == case["slices"]
        assert got["k_tiles_per_slice"] == case["k_tiles_per_slice"]


def test_fixed_capacity_layout_by_hand_and_against_alignment():
    """The fixed-capacity layout [SQ App. D.1] on a hand-checked case, and on
    random routings: each expert's rows carry the same routes in the same
    order as its run in the stable-construction alignment, which the worked
    example and brute force above pin."""
    # M=3, k=2: routes 0..5 with experts 2,0 | 2,1 | 0,2; E=3, b=2, C=4
    ids = np.array([[2, 0], [2, 1], [0, 2]], dtype=np.int32)
    s, e, br, npp, bad = oracle.align_fixed_capacity(ids, 3, 2, 4)
    S = 6
    assert s.tolist() == [1, 4, S, S, 3, S, S, S, 0, 2, 5, S]
    assert e.tolist() == [0, 1, 2, 2, -1, -1] and br.tolist() == [0, 4, 8, 10, 0, 0]
    assert npp == 8 and bad == 0
    # capacity 2: expert 2's third route (5) is dropped and counted
    s, e, br, npp, bad = oracle.align_fixed_capacity(ids, 3, 2, 2)
    assert s.tolist() == [1, 4, 3, S, 0, 2] and e.tolist() == [0, 1, 2] and br.tolist() == [0, 2, 4]
    assert npp == 6 and bad == 1
    rng = np.random.default_rng(5)
    for _ in range(20):
        M, k, E, b = int(rng.integers(1, 12)), int(rng.integers(1, 5)), int(rng.integers(1, 9)), 4
        ids = rng.integers(-1, E + 1, (M, k)).astype(np.int32)
        counts = [int(np.sum(ids == x)) for x in range(E)]
        C = (max(counts + [1]) + b - 1) // b * b
        s, e, br, npp, bad = oracle.align_fixed_capacity(ids, E, b, C)
        sa, ea, nppa, ninv = oracle.align(ids, E, b)
        assert bad == ninv and npp == nppa               # no drops at C >= max count: the same blocks
        assert e[:npp // b].tolist() == ea[:nppa // b].tolist()
        for x in range(E):
            run = [int(r) for r, ex in zip(sa[:nppa], np.repeat(ea[:nppa // b], b)) if ex == x and r < M * k]
            assert s[x * C:x * C + counts[x]].tolist() == run
