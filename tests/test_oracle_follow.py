"""Pins of the oracle's follow mode (CPU).

The GPU parity tests let the oracle continue past a selection that the CUDA path
made differently only when the two differ on a near-tie: a score gap that is not
zero and below the tolerance. These tests pin that rule, so that a follow mode
that adopted too much (which would make every parity test vacuous) or too little
fails here, on the CPU:
  * a near-tie is adopted and flagged; later depths use the adopted ranks;
  * a gap at or above the tolerance, an exact tie (decided by the stated tie
    order: lower flat index p*K + c inside a depth; shallower depth, then lower
    rank in the deferred prune), a repeated or unknown entry, a wrong length and
    a prune set that is not prefix-closed are mismatches, and the oracle keeps
    its own choice.
"""
import numpy as np
import pytest

import oracle
from oracle.dartree import _adopt
from dartree_inputs import make_config, make_tie_inputs
from _tiny import tiny_inputs


def _run(own, other, scores, tol=1e-3, valid=None):
    flags, mism = [], []
    got = _adopt(own, other, lambda x: scores[x], valid or (lambda x: x in scores), tol, "w", flags, mism)
    return got, flags, mism


# --------------------------------------------------------------------------- the rule itself

def test_identical_selection_is_neither_flag_nor_mismatch():
    got, flags, mism = _run([1, 2, 3], [1, 2, 3], {1: 0.0, 2: -1.0, 3: -2.0})
    assert got == [1, 2, 3] and flags == [] and mism == []
    got, flags, mism = _run([1, 2], None, {1: 0.0, 2: -1.0})
    assert got == [1, 2] and flags == [] and mism == []


def test_near_tie_is_adopted_and_flagged():
    s = {1: 0.0, 2: -1.0, 3: -1.0004, 4: -3.0}
    got, flags, mism = _run([1, 2, 3], [1, 3, 2], s)
    assert got == [1, 3, 2] and mism == []
    assert len(flags) == 1 and flags[0][0] == "w" and flags[0][1] == pytest.approx(4e-4)
    # a different member at the boundary, also within the tolerance
    s[5] = -1.0009
    got, flags, mism = _run([1, 2, 3], [1, 2, 5], s)
    assert got == [1, 2, 5] and len(flags) == 1 and mism == []


def test_gap_at_or_above_tolerance_is_a_mismatch():
    s = {1: 0.0, 2: -1.0, 3: -1.002, 4: -1.001}
    got, flags, mism = _run([1, 2, 3], [1, 3, 2], s)
    assert got == [1, 2, 3] and flags == [] and mism == ["w"]
    got, flags, mism = _run([1, 2], [1, 4], {1: 0.0, 2: -1.0, 4: -1.0011})
    assert got == [1, 2] and flags == [] and mism == ["w"]


def test_exact_tie_is_decided_by_the_tie_order_not_adopted():
    s = {1: 0.0, 2: -1.0, 3: -1.0}
    got, flags, mism = _run([1, 2, 3], [1, 3, 2], s)
    assert got == [1, 2, 3] and flags == [] and mism == ["w"]
    # one exact tie among near-ties is enough to refuse the whole alternative
    s = {1: 0.0, 2: -1.0, 3: -1.0005, 4: -2.0, 5: -2.0}
    got, flags, mism = _run([1, 2, 3, 4], [1, 3, 2, 5], s)
    assert got == [1, 2, 3, 4] and flags == [] and mism == ["w"]


def test_repeated_unknown_or_short_selections_are_mismatches():
    s = {1: 0.0, 2: -1.0, 3: -1.0001}
    for other in ([1, 1, 2], [1, 2, 9], [1, 2], [1, 2, 3, 3]):
        got, flags, mism = _run([1, 2, 3], other, s)
        assert got == [1, 2, 3] and flags == [] and mism == ["w"], other
    # an index the oracle could score (Python negative indexing) but that is no entry
    lst = [0.0, -1.0, -1.0001]
    flags, mism = [], []
    got = _adopt([0], [-1], lambda f: lst[f], lambda f: 0 <= f < len(lst), 1e-3, "w", flags, mism)
    assert got == [0] and mism == ["w"]


# --------------------------------------------------------------------------- follow mode inside build()

def _replay(o, K):
    """Follow callables that replay the oracle's own selections."""
    def depth(i, d):
        n = int(o["st_n"][i, d - 1])
        rank = {int(t): c for c, t in enumerate(o["cand_tok"][i, d - 1])}
        return [int(o["st_par"][i, d - 1, k]) * K + rank[int(o["st_tok"][i, d - 1, k])] for k in range(n)]

    def prune(i):
        return [(int(o["depth"][i, j]), int(o["rank"][i, j])) for j in range(1, int(o["n_nodes"][i]))]
    return dict(depth=depth, prune=prune)


def _same_tree(a, b):
    for k in ("st_tok", "st_par", "st_s", "st_n", "tok", "par", "depth", "score", "n_nodes", "mask", "pos"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


@pytest.mark.parametrize("seed", range(4))
def test_replaying_the_oracle_changes_nothing(seed):
    inp = tiny_inputs(seed, C=2)
    o = oracle.build(inp)
    f = oracle.build(inp, follow=_replay(o, inp["cfg"].K))
    assert f["flags"] == [] and f["mismatches"] == []
    _same_tree(o, f)


def _closest_pair(o, i, d, K):
    """Ranks (a, b) of two kept children of depth d with the smallest score gap."""
    s = o["st_s"][i, d - 1, :int(o["st_n"][i, d - 1])]
    k = int(np.argmin(np.diff(-s)))
    return k, k + 1, float(s[k] - s[k + 1])


def test_adopted_near_tie_changes_the_ranks_that_later_depths_use():
    inp = tiny_inputs(3, C=1, L=4, K=3, W=3, B=8)
    K = inp["cfg"].K
    o = oracle.build(inp)
    a, b, gap = _closest_pair(o, 0, 1, K)
    assert gap > 0
    rep = _replay(o, K)
    swapped = rep["depth"](0, 1)
    swapped[a], swapped[b] = swapped[b], swapped[a]
    follow = dict(depth=lambda i, d: swapped if d == 1 else None, prune=lambda i: None)
    f = oracle.build(inp, follow=follow, tie_tol=2 * gap)
    assert f["mismatches"] == [] and [x[0] for x in f["flags"]] == [("depth", 0, 1)]
    # the swap is visible at depth 1 and in the parent ranks of depth 2
    assert f["st_tok"][0, 0, a] == o["st_tok"][0, 0, b] and f["st_tok"][0, 0, b] == o["st_tok"][0, 0, a]
    par_o, par_f = o["st_par"][0, 1], f["st_par"][0, 1]
    remap = {a: b, b: a}
    n2 = int(o["st_n"][0, 1])
    assert sorted(zip(o["st_tok"][0, 1, :n2], [remap.get(int(p), int(p)) for p in par_o[:n2]])) == \
        sorted(zip(f["st_tok"][0, 1, :n2], par_f[:n2].tolist()))
    # the same swap against the default tolerance is a mismatch when the gap is not small
    if gap >= oracle.TIE_TOL:
        g = oracle.build(inp, follow=follow)
        assert g["mismatches"] == [("depth", 0, 1)] and g["flags"] == []
        _same_tree(o, g)


def test_exact_tie_swap_inside_a_depth_is_a_mismatch():
    cfg = make_config("cfg0_tiny").replace(C=1, L=3, V=24, H=8, K=4, W=4, B=8, beta=0.0, seed=5)
    inp = make_tie_inputs(cfg)
    o = oracle.build(inp)
    rep = _replay(o, cfg.K)
    # find two kept children of one depth with exactly equal scores
    for d in range(1, cfg.L + 1):
        s = o["st_s"][0, d - 1, :int(o["st_n"][0, d - 1])]
        eq = [(k, k + 1) for k in range(len(s) - 1) if s[k] == s[k + 1]]
        if eq:
            break
    assert eq, "the tie recipe must produce an exact tie"
    a, b = eq[0]
    sel = rep["depth"](0, d)
    sel[a], sel[b] = sel[b], sel[a]
    f = oracle.build(inp, follow=dict(depth=lambda i, dd: sel if dd == d else None, prune=lambda i: None))
    assert f["mismatches"] == [("depth", 0, d)] and f["flags"] == []
    _same_tree(o, f)


def test_exact_tie_in_the_prune_is_a_mismatch():
    """beta = 0 and q = 1 make children tie with their parents across depths; the
    shallower node comes first, so choosing the deeper one instead is a mismatch."""
    cfg = make_config("cfg0_tiny").replace(C=1, L=4, V=24, H=8, K=4, W=4, B=6, beta=0.0, seed=7)
    inp = make_tie_inputs(cfg)
    o = oracle.build(inp)
    chosen = [(int(o["depth"][0, j]), int(o["rank"][0, j])) for j in range(1, int(o["n_nodes"][0]))]
    nodes = {(d, k): float(o["st_s"][0, d - 1, k]) for d in range(1, cfg.L + 1)
             for k in range(int(o["st_n"][0, d - 1]))}
    left = [dk for dk in nodes if dk not in chosen]
    # a left-out node whose score equals that of a chosen node
    swap = [(c, x) for c in chosen for x in left if nodes[c] == nodes[x]]
    assert swap, "the tie recipe must leave a tied node out of the budget"
    c, x = swap[0]
    alt = [x if y == c else y for y in chosen]
    f = oracle.build(inp, follow=dict(depth=lambda i, d: None, prune=lambda i: alt))
    assert f["mismatches"] == [("prune", 0)] and f["flags"] == []
    _same_tree(o, f)


def test_prune_near_tie_is_adopted_and_non_prefix_closed_sets_are_refused():
    inp = tiny_inputs(11, C=1, L=4, K=3, W=3, B=5)
    o = oracle.build(inp)
    cfg = inp["cfg"]
    chosen = [(int(o["depth"][0, j]), int(o["rank"][0, j])) for j in range(1, int(o["n_nodes"][0]))]
    nodes = {(d, k): (float(o["st_s"][0, d - 1, k]), int(o["st_par"][0, d - 1, k]))
             for d in range(1, cfg.L + 1) for k in range(int(o["st_n"][0, d - 1]))}
    left = [dk for dk in nodes if dk not in chosen]
    ch = set(chosen)
    # the weakest chosen node with no chosen child, swapped for the best left-out
    # node whose parent is chosen: a prefix-closed alternative
    leaves = [dk for dk in chosen if not any(nodes[x][1] == dk[1] and x[0] == dk[0] + 1 for x in chosen)]
    worst = min(leaves, key=lambda dk: nodes[dk][0])
    ok_left = [dk for dk in left if dk[0] == 1 or (dk[0] - 1, nodes[dk][1]) in ch - {worst}]
    best = max(ok_left, key=lambda dk: nodes[dk][0])
    gap = abs(nodes[worst][0] - nodes[best][0])
    alt = [best if y == worst else y for y in chosen]
    f = oracle.build(inp, follow=dict(depth=lambda i, d: None, prune=lambda i: alt), tie_tol=max(2 * gap, 1e-9))
    if gap > 0:
        assert f["mismatches"] == [] and [x[0] for x in f["flags"]] == [("prune", 0)]
        got = [(int(f["depth"][0, j]), int(f["rank"][0, j])) for j in range(1, int(f["n_nodes"][0]))]
        assert sorted(got) == sorted(alt)
    # a set with a node whose parent is left out is refused at any tolerance
    orphan = [dk for dk in left if dk[0] > 1 and (dk[0] - 1, nodes[dk][1]) not in ch]
    if orphan:
        bad = [orphan[0] if y == worst else y for y in chosen]
        g = oracle.build(inp, follow=dict(depth=lambda i, d: None, prune=lambda i: bad), tie_tol=1e9)
        assert g["mismatches"] == [("prune", 0)] and g["flags"] == []
        _same_tree(o, g)


def test_a_follow_that_disagrees_everywhere_is_caught():
    """A selection far from the oracle's at every depth is a mismatch at every depth:
    follow mode cannot be used to make a wrong GPU tree pass."""
    inp = tiny_inputs(2, C=1, L=4, K=3, W=2, B=6)
    cfg = inp["cfg"]
    o = oracle.build(inp)
    rep = _replay(o, cfg.K)

    def worst(i, d):
        n = int(o["st_n"][i, d - 1])
        sc = o["children"][i][d - 1].reshape(-1)
        return [int(f) for f in np.argsort(sc, kind="stable")[:n]]
    f = oracle.build(inp, follow=dict(depth=worst, prune=lambda i: None))
    bad = [d for d in range(1, cfg.L + 1) if worst(0, d) != rep["depth"](0, d)]
    assert bad and f["mismatches"] == [("depth", 0, d) for d in bad] and f["flags"] == []
    _same_tree(o, f)


@pytest.mark.parametrize("seed,beta", [(0, 0.0), (1, 0.0), (2, -0.25), (3, 0.0)])
def test_tie_recipe_trees_follow_lemma_1(seed, beta):
    """On the tie recipe (exact ties everywhere) the deferred top-B still holds the
    same nodes as best-first popping on the materialised supertree, and the chosen
    set is prefix-closed."""
    cfg = make_config("cfg0_tiny").replace(C=2, L=5, V=30, H=8, K=4, W=5, B=9, beta=beta, seed=seed)
    inp = make_tie_inputs(cfg)
    o = oracle.build(inp)
    for i in range(cfg.C):
        popped = oracle.heap_best_first(o, i, cfg.B)
        got = [(int(o["depth"][i, j]), int(o["rank"][i, j])) for j in range(1, int(o["n_nodes"][i]))]
        assert sorted(got) == sorted(popped)
        for j in range(1, int(o["n_nodes"][i])):
            p = int(o["par"][i, j])
            assert 0 <= p < j and o["depth"][i, p] == o["depth"][i, j] - 1
    # exact ties are present: equal scores inside a depth, and (beta = 0) a child
    # with its parent's score
    s = o["st_s"][:, :, :]
    assert any(np.any(s[i, d, 1:int(o["st_n"][i, d])] == s[i, d, :int(o["st_n"][i, d]) - 1])
               for i in range(cfg.C) for d in range(cfg.L))
    if beta == 0.0:
        assert any(o["score"][i, j] == o["score"][i, int(o["par"][i, j])]
                   for i in range(cfg.C) for j in range(2, int(o["n_nodes"][i])))
