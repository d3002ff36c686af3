"""Pins of the oracle's LM head + S1 against facts that do not come from the oracle:
exact rational dot products on tiny inputs, a head whose rows are scaled basis
vectors (logits known in closed form), and the tie rule on duplicated rows."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import lm_head as olm
from dartree_inputs import bf16_bits_to_f32, make_config, make_lm_head, round_to_bf16_bits


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_logits_are_the_exact_dot_products(dtype):
    rng = np.random.default_rng(5)
    R, V, H = 3, 11, 7
    h = rng.standard_normal((R, H)).astype(np.float32)
    W = rng.standard_normal((V, H)).astype(np.float32)
    if dtype == "bf16":
        h, W = round_to_bf16_bits(h), round_to_bf16_bits(W)
        hv, Wv = bf16_bits_to_f32(h), bf16_bits_to_f32(W)
    else:
        hv, Wv = h, W
    got = olm.lm_head_logits(h, W, dtype)
    for r in range(R):
        for v in range(V):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(hv[r], Wv[v]))
            assert abs(got[r, v] - float(exact)) <= 1e-12 * max(1.0, abs(float(exact)))


def test_basis_rows_give_closed_form_logits_and_candidates():
    """W_lm[v] = a_v e_(v mod H): L[r, v] = a_v h[r, v mod H]."""
    R, V, H, K = 2, 40, 8, 5
    a = np.linspace(0.5, 2.0, V).astype(np.float32)
    W = np.zeros((V, H), np.float32)
    W[np.arange(V), np.arange(V) % H] = a
    h = np.array([[1, -2, 3, 0.5, -1, 2, 0, 1.5], [0, 0, 0, 0, 0, 0, 0, 0]], np.float32)
    tok, val, logits = olm.lm_head_topk(h, W, K, "f32")
    want = a[None, :].astype(np.float64) * h.astype(np.float64)[:, np.arange(V) % H]
    np.testing.assert_array_equal(logits, want)
    # row 0: the largest a_v h[v mod 8] come from component 2 (h=3) at the largest a_v
    best = sorted(range(V), key=lambda v: (-want[0, v], v))[:K]
    assert list(tok[0]) == best and best[0] == 34   # v = 34: 34 mod 8 = 2, a_34 largest of that class
    # row 1 is all zero: every logit ties, the K lowest ids win in order
    assert list(tok[1]) == list(range(K)) and np.all(val[1] == 0)


def test_duplicate_rows_tie_to_the_lower_token():
    rng = np.random.default_rng(1)
    W = rng.standard_normal((30, 6)).astype(np.float32)
    W[17] = W[4] * 10      # the two largest logits of a positive row, equal
    W[23] = W[4] * 10
    h = W[4:5].copy()
    tok, val, _ = olm.lm_head_topk(h, W, 3, "f32")
    assert list(tok[0][:2]) == [17, 23] and val[0][0] == val[0][1]


def test_stand_in_weights_have_the_configured_spread():
    cfg = make_config("cfg1_qwen3_4b_c1").replace(V=4096)
    W = bf16_bits_to_f32(make_lm_head(cfg))
    assert W.shape == (4096, cfg.H)
    assert abs(W.std() * np.sqrt(cfg.H) - cfg.sigma) < 0.02
    np.testing.assert_array_equal(make_lm_head(cfg), make_lm_head(cfg))   # seeded


def test_closed_form_across_vocabulary_chunks():
    """More vocabulary rows than one float64 chunk: every chunk boundary keeps its rows."""
    V, H = 2 * olm.CHUNK_ROWS + 7, 8
    a = (1.0 + np.arange(V) / V).astype(np.float32)
    W = np.zeros((V, H), np.float32)
    W[np.arange(V), np.arange(V) % H] = a
    h = np.arange(1, H + 1, dtype=np.float32)[None, :]
    logits = olm.lm_head_logits(h, W, "f32")
    np.testing.assert_array_equal(logits[0], a.astype(np.float64) * (np.arange(V) % H + 1))
    tok, _, _ = olm.lm_head_topk(h, W, 3, "f32")
    top = max(v for v in range(V) if v % H == H - 1)   # component H (h = 8) at the largest a_v
    assert list(tok[0]) == [top, top - H, top - 2 * H]
