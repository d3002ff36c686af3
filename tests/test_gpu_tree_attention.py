"""Parity of the verification pass's tree attention (dartree_tree_attention) with the
oracle's float64 layer, through the C ABI.

The kernel takes bf16 operands, accumulates scores and sums in fp32, rounds the
probabilities to bf16 for the P V product (relative error <= 2^-9 per weight, so at
most 2^-9 * max|v| ~ 0.01 on an output of N(0, 1) values) and writes bf16 (half an
ulp, <= 2^-9 relative): outputs are compared at atol 1.5e-2, rtol 1e-2. Unused slots
must be exactly zero.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from oracle import tree_attention as ota  # noqa: E402
from dartree_inputs import bf16_bits_to_f32, make_attention_inputs  # noqa: E402

pytestmark = pytest.mark.gpu

ATOL, RTOL = 1.5e-2, 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_drafter_draft_gb300 as dd
    from diffusion_drafter_draft_gb300 import _build
    _build.build()
    dd.lib()


from _gpu import t  # noqa: E402


def _tree(C, S, seed, n_nodes=None, width=12):
    """Seeded trees with DARTree's slot layout: `width` slots per depth after the root,
    each slot's parent one depth up; S9's mask and positions from the oracle."""
    rng = np.random.default_rng(seed)
    depth = np.zeros(S, np.int64)
    depth[1:] = 1 + np.arange(S - 1) // width
    par = np.full((C, S), -1, np.int64)
    for c in range(C):
        for j in range(1, S):
            par[c, j] = rng.choice(np.flatnonzero(depth[:j] == depth[j] - 1))
    nn = np.full(C, S, np.int64) if n_nodes is None else np.asarray(n_nodes, np.int64)
    dep = np.tile(depth, (C, 1))
    for c in range(C):
        par[c, nn[c]:] = -1
        dep[c, nn[c]:] = -1
    mask, pos = oracle.mask_pos(par, dep, nn)
    return mask, pos, nn


def _run(C, S, Hq, Hkv, N, seed, n_ctx=None, n_nodes=None, check=None):
    import diffusion_drafter_draft_gb300 as dd
    D = 128
    x = make_attention_inputs(C, S, Hq, Hkv, D, N, seed, n_ctx=n_ctx)
    mask, pos, nn = _tree(C, S, seed, n_nodes)
    tree = dict(mask=torch.from_numpy(mask).cuda(), pos=torch.from_numpy(pos.astype(np.int32)).cuda(),
                n_nodes=torch.from_numpy(nn.astype(np.int32)).cuda())
    vt = np.ascontiguousarray(x["v_cache"].transpose(0, 1, 3, 2))
    out = dd.tree_attention(t(x["q"], "bf16"), t(x["k_tree"], "bf16"), t(x["v_tree"], "bf16"),
                            t(x["k_cache"], "bf16"), t(vt, "bf16"), torch.from_numpy(x["n_ctx"]).cuda(), tree)
    torch.cuda.synchronize()
    g = bf16_bits_to_f32(out.view(torch.int16).cpu().numpy().view(np.uint16))
    reqs = range(C) if check is None else check
    for c in reqs:
        sl = slice(c, c + 1)
        o = ota.tree_attention(x["q"][sl], x["k_tree"][sl], x["v_tree"][sl], x["k_cache"][sl], x["v_cache"][sl],
                               x["n_ctx"][sl], mask[sl], pos[sl], nn[sl], "bf16")
        np.testing.assert_allclose(g[c], o[0], atol=ATOL, rtol=RTOL, err_msg=f"request {c}")
        assert np.all(g[c, int(nn[c]):] == 0)
    return g


@pytest.mark.parametrize("C,S,Hq,Hkv,N,n_ctx", [
    (2, 7, 4, 2, 200, [200, 77]),             # tiny tree, ragged prefixes (last block partly used)
    (1, 65, 32, 8, 2048, None),               # one request: 16 prefix blocks + the tree, chunked
    (4, 65, 32, 8, 1024, [1024, 1000, 5, 0]), # short and empty prefixes
    (3, 48, 16, 2, 512, None),                # 8 query heads per group: 384 rows = 3 full tiles
    (2, 128, 4, 2, 128, [128, 64]),           # the largest tree: 128 slots, 2 query heads per group
    (2, 9, 4, 2, 0, None),                    # no cache at all (N = 0): the tree block alone
    (2, 33, 8, 8, 384, [300, 384]),           # one query head per key/value head (grp = 1)
    (3, 1, 8, 2, 256, [256, 3, 0]),           # root-only trees (S = 1)
])
def test_tree_attention_matches_oracle(C, S, Hq, Hkv, N, n_ctx):
    _run(C, S, Hq, Hkv, N, seed=C * 100 + S, n_ctx=n_ctx)


def test_unused_slots_are_zero_and_ignored():
    g = _run(3, 65, 8, 2, 256, seed=5, n_nodes=[65, 20, 1])
    assert np.all(g[1, 20:] == 0) and np.all(g[2, 1:] == 0)


def test_tree_attention_at_the_64_request_size():
    """64 requests (one chunk per row tile: the output is written by the attention
    launch itself), the oracle checks both ends of the batch and two inside."""
    _run(64, 65, 32, 8, 512, seed=64, check=(0, 21, 42, 63))
