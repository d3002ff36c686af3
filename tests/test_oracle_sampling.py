"""Pins of the oracle's temperature-T verification and adaptive budget against facts
that do not come from the oracle itself: the generator's published known answers,
the exactness of the Gumbel-max draw (chi-square against the softmax), the greedy
limit, the closed-form acceptance law of a hand-made tree, and the budget values the
DARTree blog post gives (section 4.4)."""
import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from oracle import sampling as osm
from dartree_inputs import make_target_per_node
from _tiny import load_golden, tiny_inputs


def test_philox_known_answers():
    kat = load_golden("philox4x32_10_kat.json")
    for vec in kat["vectors"]:
        ctr = [int(w, 16) for w in vec["counter"]]
        key = [int(w, 16) for w in vec["key"]]
        out = [int(w) for w in osm.philox4x32(ctr, key)]
        assert out == [int(w, 16) for w in vec["output"]]


def test_uniforms_are_odd_multiples_inside_the_unit_interval():
    u = osm.uniforms(seed=0x1234_5678_9ABC, request=3, row=5, V=100_003)
    assert u.dtype == np.float32 and u.shape == (100_003,)
    k = u.astype(np.float64) * 2.0 ** 24
    assert np.all(k == np.round(k)) and np.all(np.round(k) % 2 == 1)   # (2m + 1) 2^-24
    assert u.min() >= 2.0 ** -24 and u.max() <= 1 - 2.0 ** -24
    # uniform: mean 1/2, variance 1/12, and a flat histogram
    assert abs(u.mean() - 0.5) < 0.005 and abs(u.var() - 1 / 12) < 0.002
    h, _ = np.histogram(u, bins=20, range=(0, 1))
    assert scipy.stats.chisquare(h).pvalue > 1e-4
    # every coordinate of the counter and both halves of the seed change the stream
    base = osm.uniforms(7, 1, 2, 64)
    for other in (osm.uniforms(7 + (1 << 32), 1, 2, 64), osm.uniforms(8, 1, 2, 64),
                  osm.uniforms(7, 2, 2, 64), osm.uniforms(7, 1, 3, 64)):
        assert np.mean(base == other) < 0.1


def test_uniform_extremes_of_the_word_map():
    # w = 0 -> 2^-24, w = 2^32 - 1 -> 1 - 2^-24 (through the same arithmetic)
    for w, want in ((0, 2.0 ** -24), (0xFFFFFFFF, 1 - 2.0 ** -24), (1 << 31, 0.5 + 2.0 ** -24)):
        num = (np.uint64(w) >> np.uint64(9)) * np.uint64(2) + np.uint64(1)
        assert float(np.float32(num) * np.float32(2.0 ** -24)) == want


@pytest.mark.parametrize("T", [1.0, 0.6, 2.5])
def test_gumbel_max_draws_follow_the_softmax(T):
    x = np.array([1.0, 0.25, -0.5, 2.0, 0.0, 1.5], np.float32)
    n = 12_000
    counts = np.zeros(x.size, np.int64)
    for r in range(n):
        t, _ = osm.sample_token(x, T, seed=99, request=r, row=0)
        counts[t] += 1
    p = scipy.special.softmax(x.astype(np.float64) / T)
    assert scipy.stats.chisquare(counts, n * p).pvalue > 1e-4
    # a wrong sign of the noise, or the noise unscaled by 1/T, fails this
    assert np.abs(counts / n - p).max() < 0.02


def test_equal_perturbed_values_go_to_the_lower_token():
    x = np.zeros(8, np.float32)
    U = np.full(8, 0.5, np.float32)      # all eight perturbed values equal
    y = osm.perturbed(x, 1.0, U)
    assert np.all(y == y[0]) and int(np.argmax(y)) == 0


def _tree(n, tok, par, depth):
    S = len(tok)
    return dict(tok=np.tile(np.asarray(tok, np.int64), (n, 1)), par=np.tile(np.asarray(par, np.int64), (n, 1)),
                depth=np.tile(np.asarray(depth, np.int64), (n, 1)), n_nodes=np.full(n, S, np.int64))


def test_acceptance_law_of_a_hand_made_tree():
    """Root children carry tokens 0 and 2; the child with token 0 has one child, token 1.
    Per-position rows: P(len >= 1) = p0(0) + p0(2), P(len = 2) = p0(0) p1(1)."""
    n, T = 6000, 1.0
    tree = _tree(n, tok=[7, 0, 2, 1], par=[-1, 0, 0, 1], depth=[0, 1, 1, 2])
    rows = np.array([[1.0, 0.2, 0.5, -0.3], [0.1, 0.9, -0.5, 0.0]], np.float32)
    target = np.tile(rows, (n, 1, 1))
    out = osm.verify_sample(tree, target, "f32", "position", 2, T, seed=2024)
    p0, p1 = (scipy.special.softmax(rows[k].astype(np.float64) / T) for k in (0, 1))
    law = np.array([1 - p0[0] - p0[2], p0[2] + p0[0] * (1 - p1[1]), p0[0] * p1[1]])
    counts = np.bincount(out["accepted_len"], minlength=3)
    assert scipy.stats.chisquare(counts, n * law).pvalue > 1e-4
    # the bonus is the rejected draw: never a token the current node's children carry
    b0 = out["bonus"][out["accepted_len"] == 0]
    assert set(np.unique(b0)) <= {1, 3}
    # after a full block (depth L) there is no row, hence no bonus
    assert np.all(out["bonus"][out["accepted_len"] == 2] == -1)
    acc1 = out["accepted_len"] >= 1
    assert set(np.unique(out["path"][acc1, 0])) <= {1, 2}


def test_per_node_rows_use_the_slot_index():
    """Per-node rows: slot j draws with counter row j. Two root children with the same
    token never both match; a slot's draw does not depend on the slot's depth."""
    n = 4000
    tree = _tree(n, tok=[5, 0, 1, 1], par=[-1, 0, 0, 2], depth=[0, 1, 1, 2])
    rows = np.array([[0.3, 0.3, -1.0, -1.0], [0.0, 0.0, 0.0, 0.0], [0.0, 2.0, 0.0, 0.0], [0.0, 0.0, 0.0, 0.0]],
                    np.float32)
    target = np.tile(rows, (n, 1, 1))
    out = osm.verify_sample(tree, target, "f32", "node", 2, 1.0, seed=11)
    p0, p2 = (scipy.special.softmax(rows[k].astype(np.float64)) for k in (0, 2))
    law = np.array([1 - p0[0] - p0[1], p0[0] + p0[1] * (1 - p2[1]), p0[1] * p2[1]])
    counts = np.bincount(out["accepted_len"], minlength=3)
    assert scipy.stats.chisquare(counts, n * law).pvalue > 1e-4
    # a fully accepted per-node walk still has a row (slot 3): a bonus is drawn there
    assert np.all(out["bonus"][out["accepted_len"] == 2] >= 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows", ["position", "node"])
def test_small_temperature_is_the_greedy_rule(dtype, rows):
    inp = tiny_inputs(3, dtype=dtype, rows=rows, C=4)
    out = oracle.build(inp)
    cfg = inp["cfg"]
    L = cfg.L
    tgt = inp["target"] if rows == "position" else make_target_per_node(cfg, inp, out["depth"])
    g = oracle.verify(out, tgt, dtype, rows, L)
    # T small enough that the noise (|G| < 17 T) is far below every row's top-2 gap
    s = osm.verify_sample(out, tgt, dtype, rows, L, 1e-7, seed=5)
    for k in ("accepted_len", "path", "bonus"):
        np.testing.assert_array_equal(s[k], g[k], err_msg=k)


def test_temperature_must_be_positive():
    tree = _tree(1, tok=[0], par=[-1], depth=[0])
    for T in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(ValueError):
            osm.verify_sample(tree, np.zeros((1, 1, 4), np.float32), "f32", "position", 1, T, 0)


def test_adaptive_budget_values():
    assert [osm.adaptive_budget(C) for C in (1, 2, 3)] == [(64, 12)] * 3
    assert [osm.adaptive_budget(C) for C in (4, 5, 16, 64)] == [(32, 3)] * 4
    with pytest.raises(ValueError):
        osm.adaptive_budget(0)


def test_request_ids_key_the_draws():
    """Checking request i of a batch on its own (requests=[i]) draws what the batch
    call draws for entry i."""
    n = 5
    tree = _tree(n, tok=[7, 0, 2, 1], par=[-1, 0, 0, 1], depth=[0, 1, 1, 2])
    rng = np.random.default_rng(0)
    target = rng.standard_normal((n, 2, 4)).astype(np.float32)
    full = osm.verify_sample(tree, target, "f32", "position", 2, 1.0, seed=3)
    for i in range(n):
        sub = {k: v[i:i + 1] for k, v in tree.items()}
        one = osm.verify_sample(sub, target[i:i + 1], "f32", "position", 2, 1.0, seed=3, requests=[i])
        for k in ("accepted_len", "path", "bonus"):
            np.testing.assert_array_equal(one[k][0], full[k][i])
