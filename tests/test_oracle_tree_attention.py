"""Pins of the oracle's tree attention against facts that do not come from the oracle:
rotary embedding in closed form and through complex rotation, its relative-position
property, single-key and uniform-weight closed forms, mask semantics, the causal
special case (a chain tree is plain causal attention over prefix + chain), and the
query-to-key/value head grouping."""
import math

import numpy as np
import pytest
import scipy.special

from oracle import mask_pos
from oracle import tree_attention as ota


def test_rope_closed_form():
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    got = ota.rope(x, np.array([1]), theta=100.0)[0]
    # D = 4: inverse frequencies 100^0 = 1 and 100^(-1/2) = 0.1
    want = [1 * math.cos(1) - 3 * math.sin(1), 2 * math.cos(0.1) - 4 * math.sin(0.1),
            3 * math.cos(1) + 1 * math.sin(1), 4 * math.cos(0.1) + 2 * math.sin(0.1)]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


def test_rope_is_a_complex_rotation_and_relative():
    rng = np.random.default_rng(0)
    D, n = 16, 6
    x = rng.standard_normal((n, D))
    p = rng.integers(0, 5000, n)
    got = ota.rope(x, p)
    w = ota.ROPE_THETA ** (-np.arange(D // 2) * 2.0 / D)
    z = (x[:, :D // 2] + 1j * x[:, D // 2:]) * np.exp(1j * p[:, None] * w[None, :])
    np.testing.assert_allclose(got, np.concatenate([z.real, z.imag], axis=1), rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(got, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    np.testing.assert_array_equal(ota.rope(x, np.zeros(n, int)), x)
    # <R(p) q, R(p') k> depends on p - p' only
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    a = ota.rope(q[None], np.array([100]))[0] @ ota.rope(k[None], np.array([37]))[0]
    b = ota.rope(q[None], np.array([1063]))[0] @ ota.rope(k[None], np.array([1000]))[0]
    assert abs(a - b) < 1e-10


def _case(C=1, S=5, Hq=4, Hkv=2, D=8, N=6, seed=0, par=None):
    rng = np.random.default_rng(seed)
    f = lambda *s: rng.standard_normal(s).astype(np.float32)  # noqa: E731
    if par is None:
        par = [-1, 0, 0, 1, 2][:S]
    par = np.tile(np.asarray(par), (C, 1))
    depth = np.zeros_like(par)
    for j in range(1, S):
        depth[:, j] = depth[:, par[0, j]] + 1
    n_nodes = np.full(C, S)
    mask, pos = mask_pos(par, depth, n_nodes)
    return dict(q=f(C, S, Hq, D), k_tree=f(C, S, Hkv, D), v_tree=f(C, S, Hkv, D), k_cache=f(C, Hkv, N, D),
                v_cache=f(C, Hkv, N, D), n_ctx=np.full(C, N), mask=mask, pos=pos, n_nodes=n_nodes)


def _run(c):
    return ota.tree_attention(c["q"], c["k_tree"], c["v_tree"], c["k_cache"], c["v_cache"], c["n_ctx"],
                              c["mask"], c["pos"], c["n_nodes"], "f32")


def test_a_lone_root_sees_only_itself():
    c = _case(S=1, N=6, par=[-1])
    c["n_ctx"][:] = 0
    out = _run(c)
    for h in range(4):
        np.testing.assert_allclose(out[0, 0, h], c["v_tree"][0, 0, h // 2], rtol=1e-12, atol=1e-12)


def test_zero_queries_average_the_visible_values():
    c = _case()
    c["q"][:] = 0
    out = _run(c)
    anc = {0: [0], 1: [0, 1], 2: [0, 2], 3: [0, 1, 3], 4: [0, 2, 4]}
    for j, a in anc.items():
        for h in range(4):
            g = h // 2
            vals = np.concatenate([c["v_cache"][0, g], c["v_tree"][0, a, g]]).astype(np.float64)
            np.testing.assert_allclose(out[0, j, h], vals.mean(axis=0), rtol=1e-12, atol=1e-12)


def test_only_visible_slots_matter():
    c = _case(seed=3)
    base = _run(c)
    c2 = {k: v.copy() for k, v in c.items()}
    c2["k_tree"][0, 2] += 5.0    # slot 2 is visible to slots 2 and 4 only
    c2["v_tree"][0, 2] -= 3.0
    out = _run(c2)
    for j in (0, 1, 3):
        np.testing.assert_array_equal(out[0, j], base[0, j])
    for j in (2, 4):
        assert np.abs(out[0, j] - base[0, j]).max() > 1e-3


def test_a_chain_is_causal_attention():
    """Slots 0..S-1 in one chain: slot j sits at position N + j and sees the prefix
    and slots 0..j, i.e. causal attention over the sequence prefix + chain."""
    S, Hq, Hkv, D, N = 6, 4, 2, 8, 7
    c = _case(S=S, Hq=Hq, Hkv=Hkv, D=D, N=N, seed=5, par=[-1, 0, 1, 2, 3, 4])
    out = _run(c)
    w = ota.ROPE_THETA ** (-np.arange(D // 2) * 2.0 / D)

    def rot(x, p):  # complex-number form of the rotation
        z = (x[..., :D // 2] + 1j * x[..., D // 2:]) * np.exp(1j * p * w)
        return np.concatenate([z.real, z.imag], axis=-1)

    for h in range(Hq):
        g = h // (Hq // Hkv)
        K = np.concatenate([c["k_cache"][0, g], np.stack([rot(c["k_tree"][0, j, g], N + j) for j in range(S)])])
        Vv = np.concatenate([c["v_cache"][0, g], c["v_tree"][0, :, g]])
        Q = np.stack([rot(c["q"][0, j, h], N + j) for j in range(S)])
        sc = Q @ K.T / math.sqrt(D)
        sc[np.triu(np.ones((S, N + S), bool), k=N + 1)] = -np.inf   # row j sees columns < N + j + 1
        np.testing.assert_allclose(out[0, :, h], scipy.special.softmax(sc, axis=1) @ Vv, rtol=1e-10, atol=1e-12)


def test_query_heads_share_their_group_key_value_head():
    c = _case(Hq=4, Hkv=2, seed=9)
    out = _run(c)
    for g in range(2):     # the same result as a one-key-head layer on group g's heads
        cg = dict(c, q=c["q"][:, :, 2 * g:2 * g + 2], k_tree=c["k_tree"][:, :, g:g + 1],
                  v_tree=c["v_tree"][:, :, g:g + 1], k_cache=c["k_cache"][:, g:g + 1],
                  v_cache=c["v_cache"][:, g:g + 1])
        np.testing.assert_allclose(_run(cg), out[:, :, 2 * g:2 * g + 2], rtol=1e-13, atol=1e-13)


def test_unused_slots_and_short_prefixes():
    c = _case(C=2, seed=11)
    c["n_nodes"][1] = 3
    c["n_ctx"][1] = 2
    c["pos"][1, 3:] = -1
    out = _run(c)
    assert np.all(out[1, 3:] == 0)
    c2 = {k: v.copy() for k, v in c.items()}
    c2["k_cache"][1, :, 2:] = 100.0      # past request 1's prefix: never read
    np.testing.assert_array_equal(_run(c2)[1], out[1])
