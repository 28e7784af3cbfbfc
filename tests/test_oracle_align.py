"""Pins of the oracle's routing alignment (no GPU).

The step is moe_align_block_size(local_ids, block_size_m, num_experts) of
"013-moe-middle-tiles.py" (kernel_fn), which returns (sorted_ids, block_experts,
n_padded); the invalid-block marker -1 follows the expert-id scan of "Marlin MoE
kernel occupancy ..." (sglang PR #31552), marlin_template.h excerpt.  The pages
do not print its output, so the pins are a hand-worked example and a brute-force
check of every defining property on all small id tensors.
"""
import itertools
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "align_hand_example.txt")


def read_golden():
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    M, k, E, B, base = map(int, rows[0])
    ids = np.array([list(map(int, r)) for r in rows[1:1 + M]], dtype=np.int32)
    sorted_ids = np.array(list(map(int, rows[1 + M])), dtype=np.int32)
    expert_ids = np.array(list(map(int, rows[2 + M])), dtype=np.int32)
    n_padded = int(rows[3 + M][0])
    return M, k, E, B, base, ids, sorted_ids, expert_ids, n_padded


def test_hand_example(orc):
    M, k, E, B, base, ids, s_ref, e_ref, n_ref = read_golden()
    s, e, n = orc.align(ids, E, B, base)
    assert n == n_ref
    np.testing.assert_array_equal(s, s_ref)
    np.testing.assert_array_equal(e, e_ref)
    assert orc.align_capacity(M, k, E, B) == len(s_ref)


def check_properties(ids, E, B, base, s, eids, n):
    """Every property that, together, fixes the alignment output uniquely."""
    M, k = ids.shape
    P = M * k
    flat = ids.reshape(-1).astype(np.int64) - base
    local = [(p, int(flat[p])) for p in range(P) if 0 <= flat[p] < E]
    counts = np.bincount([e for _, e in local], minlength=E) if local else np.zeros(E, np.int64)
    padded = (counts + B - 1) // B * B
    assert n == int(padded.sum())
    cap = len(s)
    assert cap % B == 0 and cap >= n and len(eids) == cap // B
    assert np.all(s[n:] == P) and np.all(eids[n // B:] == -1)
    pos = 0
    for e in range(E):  # experts in ascending order, empty experts take no block
        run = s[pos:pos + padded[e]]
        want = [p for p, ee in local if ee == e]  # ascending pair id
        assert list(run[:counts[e]]) == want
        assert np.all(run[counts[e]:] == P)
        assert np.all(eids[pos // B:(pos + padded[e]) // B] == e)
        pos += padded[e]
    assert pos == n


@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_bruteforce_small(orc, B):
    # every id tensor with M <= 2, k <= 2 over 5 routed ids, local range [1, 4)
    for M, k in [(1, 1), (1, 2), (2, 1), (2, 2), (3, 1)]:
        for flat in itertools.product(range(5), repeat=M * k):
            ids = np.array(flat, dtype=np.int32).reshape(M, k)
            s, e, n = orc.align(ids, 3, B, 1)
            check_properties(ids, 3, B, 1, s, e, n)


@pytest.mark.parametrize("M,k,E,B,base,nid", [(0, 2, 4, 4, 0, 4), (1, 8, 32, 16, 0, 256),
                                              (123, 2, 8, 16, 0, 8), (517, 8, 128, 64, 0, 128),
                                              (64, 8, 32, 8, 96, 256)])
def test_random_properties(orc, M, k, E, B, base, nid):
    rng = np.random.default_rng(M + k + E)
    ids = np.array([rng.permutation(nid)[:k] for _ in range(M)], dtype=np.int32).reshape(M, k)
    s, e, n = orc.align(ids, E, B, base)
    check_properties(ids, E, B, base, s, e, n)


def test_capacity_bound(orc):
    # the capacity covers the worst case: every pair on its own expert
    for M, k, E, B in [(1, 8, 32, 16), (4, 2, 8, 64), (100, 8, 128, 16)]:
        ids = np.arange(M * k, dtype=np.int32).reshape(M, k) % E
        s, _, n = orc.align(ids, E, B)
        assert n <= orc.align_capacity(M, k, E, B) == len(s)
