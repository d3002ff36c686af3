"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Node sets, parents, depths, masks, position ids, accepted lengths, paths and bonus
tokens must be bit-exact; scores agree within 2e-3 absolute. A per-depth or
global selection that differs from the oracle's only on a score gap that is not
zero and below 1e-3 is adopted by the oracle (follow mode) and counted (printed
at the end of the run), not failed; exact ties must follow the stated order, and
the tie-recipe cases allow no adopted selection at all.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from dartree_inputs import (breadth_first_slot_depth, make_config, make_inputs,  # noqa: E402
                            make_target_per_node, make_tie_inputs, round_to_bf16_bits, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_drafter_draft_gb300 as dd
    from diffusion_drafter_draft_gb300 import _build
    _build.build()
    dd.lib()


from _gpu import compare_build, compare_verify, host, run_gpu_build, t, upload  # noqa: E402


# --------------------------------------------------------------------------- S1 top-K

def _topk_case(rows, V, K, dtype, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "gauss":
        x = rng.standard_normal((rows, V)).astype(np.float32) * 2.5
    elif kind == "ties":
        x = rng.integers(-3, 4, size=(rows, V)).astype(np.float32)
    elif kind == "const":
        x = np.zeros((rows, V), np.float32)
        x[:, ::3] = -0.0
    else:  # planted peaks over heavy ties
        x = np.round(rng.standard_normal((rows, V)).astype(np.float32) * 4) / 4
        x[np.arange(rows), rng.integers(0, V, rows)] = 30.0
    return round_to_bf16_bits(x) if dtype == "bf16" else x


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,V,K", [(3, 1000, 8), (5, 151936, 64), (2, 151936, 512), (4, 4099, 1024),
                                      (7, 37, 37), (1, 9, 1), (16, 65543, 100)])
@pytest.mark.parametrize("kind", ["gauss", "ties", "const", "peaks"])
def test_topk_matches_oracle(dtype, rows, V, K, kind):
    import diffusion_drafter_draft_gb300 as dd
    x = _topk_case(rows, V, K, dtype, kind, seed=rows * 7 + V)
    tok, val = dd.topk(t(x, dtype), K)
    tok, val = host(tok), host(val)
    xf = to_f64(x, dtype)
    for r in range(rows):
        et, ev = oracle.topk_candidates(xf[r], K)
        np.testing.assert_array_equal(tok[r], et)
        np.testing.assert_array_equal(val[r], ev.astype(np.float32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,V,K,kind", [(320, 151936, 512, "gauss"), (320, 151936, 512, "const"),
                                           (304, 151936, 64, "ties"), (400, 4104, 100, "gauss"),
                                           (400, 4104, 100, "peaks"), (400, 4104, 1024, "ties")])
def test_topk_many_rows(dtype, rows, V, K, kind):
    """At least two rows per SM: one CTA per row streams its row twice (heavy
    ties take the exact radix fallback). Rows are independent, so a sample of
    rows is checked against the oracle."""
    import diffusion_drafter_draft_gb300 as dd
    x = _topk_case(rows, V, K, dtype, kind, seed=rows + V + K)
    tok, val = dd.topk(t(x, dtype), K)
    tok, val = host(tok), host(val)
    xf = to_f64(x, dtype)
    for r in sorted(set(range(0, rows, max(1, rows // 24))) | {rows - 1}):
        et, ev = oracle.topk_candidates(xf[r], K)
        np.testing.assert_array_equal(tok[r], et)
        np.testing.assert_array_equal(val[r], ev.astype(np.float32))


# --------------------------------------------------------------------------- S8 / S9 / S10 on oracle intermediates

@pytest.mark.parametrize("name", ["cfg0_tiny", "cfg3_c4_adaptive"])
def test_prune_mask_verify_on_oracle_supertree(name):
    import diffusion_drafter_draft_gb300 as dd
    cfg = make_config(name)
    inp = make_inputs(cfg)
    o = oracle.build(inp)
    st = dict(tok=torch.from_numpy(o["st_tok"].astype(np.int32)).cuda(),
              par=torch.from_numpy(o["st_par"].astype(np.int32)).cuda(),
              score=torch.from_numpy(o["st_s"].astype(np.float32)).cuda(),
              n=torch.from_numpy(o["st_n"].astype(np.int32)).cuda())
    anchor = torch.from_numpy(inp["anchor"]).cuda()
    tr = dd.prune(st, anchor, cfg.B)
    dd.tree_mask(tr, cfg.L)
    g = host(tr)
    for k in ("tok", "par", "depth", "n_nodes", "mask", "pos"):
        np.testing.assert_array_equal(g[k], o[k], err_msg=k)
    np.testing.assert_array_equal(g["score"], o["score"].astype(np.float32))
    target = t(inp["target"], cfg.dtype)
    gv = host(dd.verify(tr, target, dd.ROWS_PER_POSITION, cfg.L))
    compare_verify(o, gv, inp["target"], cfg, "position")


# --------------------------------------------------------------------------- S2-S7 on the oracle's candidates

@pytest.mark.parametrize("C,L,V,H,K,W,B,dtype", [(2, 5, 3001, 512, 64, 12, 30, "bf16"),
                                                 (3, 4, 1500, 256, 128, 6, 12, "bf16"),
                                                 (2, 4, 999, 64, 8, 3, 7, "f32")])
def test_expand_from_oracle_candidates(C, L, V, H, K, W, B, dtype):
    """dartree_expand fed the oracle's candidate table (kernel-level parity of
    S2-S7; the supertree is then pruned and masked by dartree_prune and
    dartree_tree_mask). The first shape takes the candidate-side path with its own
    gather of the candidates' rows (no top-K launch copies them here), the second
    the per-depth path, the third the fp32 path."""
    import diffusion_drafter_draft_gb300 as dd
    cfg = make_config("cfg1_qwen3_4b_c1").replace(C=C, L=L, V=V, H=H, K=K, W=W, B=B, dtype=dtype,
                                                   seed=7 * C + K)
    inp = make_inputs(cfg)
    o0 = oracle.build(inp)
    x = upload(inp)
    ct = torch.from_numpy(o0["cand_tok"].astype(np.int32)).cuda()
    cv = torch.from_numpy(o0["cand_logit"].astype(np.float32)).cuda()
    st = dd.expand(x["E"], x["Wq"], x["hidden"], x["anchor"], ct, cv, cfg.W, cfg.beta)
    tr = dd.prune(st, x["anchor"], cfg.B)
    dd.tree_mask(tr, cfg.L)
    g = host(dict(tr, st=st, cand_tok=ct, cand_val=cv))
    compare_build(inp, g)


# --------------------------------------------------------------------------- end to end

@pytest.mark.parametrize("name", ["cfg0_tiny", "cfg1_qwen3_4b_c1", "cfg2_qwen3_8b_fixed", "cfg3_c4_adaptive",
                                  "cfg3_c2"])
def test_build_and_verify_match_oracle(name):
    import diffusion_drafter_draft_gb300 as dd
    cfg = make_config(name)
    inp = make_inputs(cfg)
    g, x = run_gpu_build(inp)
    o = compare_build(inp, g)
    tr = {k: torch.from_numpy(v).cuda() for k, v in g.items() if k in ("tok", "par", "depth", "n_nodes")}
    gv = host(dd.verify(tr, x["target"], dd.ROWS_PER_POSITION, cfg.L))
    compare_verify(o, gv, inp["target"], cfg, "position")


def test_tiny_shapes_with_ragged_tails():
    """Several small shapes whose sizes are not multiples of any tile."""
    import diffusion_drafter_draft_gb300 as dd
    for seed, (L, V, H, K, W, B) in enumerate([(3, 211, 24, 5, 7, 9), (5, 1031, 40, 17, 3, 11),
                                                (2, 99, 8, 33, 40, 50), (6, 517, 72, 1, 4, 5),
                                                (4, 3001, 256, 16, 6, 12), (7, 2003, 520, 37, 5, 20)]):
        for dtype in ("f32", "bf16"):
            cfg = make_config("cfg0_tiny").replace(C=3, L=L, V=V, H=H, K=K, W=W, B=B, dtype=dtype, seed=seed,
                                                   beta=-0.05 * seed)
            inp = make_inputs(cfg)
            g, x = run_gpu_build(inp)
            o = compare_build(inp, g)
            tr = {k: torch.from_numpy(v).cuda() for k, v in g.items() if k in ("tok", "par", "depth", "n_nodes")}
            gv = host(dd.verify(tr, x["target"], dd.ROWS_PER_POSITION, cfg.L))
            compare_verify(o, gv, inp["target"], cfg, "position")


@pytest.mark.parametrize("C,L,V,H,K,W,B,dtype", [(5, 5, 3001, 256, 200, 12, 30, "bf16"),
                                                 (9, 4, 1500, 128, 33, 16, 40, "bf16"),
                                                 (7, 6, 2048, 384, 128, 8, 25, "bf16"),
                                                 (6, 4, 1500, 128, 40, 12, 30, "f32"),
                                                 (32, 3, 1000, 64, 16, 4, 8, "f32")])
def test_large_batch_path_shapes(C, L, V, H, K, W, B, dtype):
    """Batches with C*W > 48 take the per-depth path (tcgen05 projection and
    tensor-core contraction when H is a multiple of 128 and the head is bf16; the
    plain projection and contraction kernels for fp32 heads). From C = 32 the batch
    expands as two halves on two streams (the last case: fp32 halves)."""
    import diffusion_drafter_draft_gb300 as dd
    cfg = make_config("cfg1_qwen3_4b_c1").replace(C=C, L=L, V=V, H=H, K=K, W=W, B=B, dtype=dtype,
                                                  seed=C * 100 + K)
    inp = make_inputs(cfg)
    g, x = run_gpu_build(inp)
    o = compare_build(inp, g)
    tr = {k: torch.from_numpy(v).cuda() for k, v in g.items() if k in ("tok", "par", "depth", "n_nodes")}
    gv = host(dd.verify(tr, x["target"], dd.ROWS_PER_POSITION, cfg.L))
    compare_verify(o, gv, inp["target"], cfg, "position")


@pytest.mark.parametrize("C,L,V,H,K,W,B", [(2, 5, 3001, 512, 64, 16, 40), (3, 3, 2000, 768, 24, 5, 10),
                                           (1, 16, 4096, 1024, 8, 1, 16), (4, 7, 1500, 256, 64, 12, 30),
                                           (1, 4, 151936, 512, 8, 4, 8), (2, 3, 50000, 256, 24, 6, 12)])
def test_candidate_side_projection_shapes(C, L, V, H, K, W, B):
    """Small bf16 batches with K <= 64 and W <= 16 take the candidate-side
    projection path (G = E[cand] W_q once per round, one cluster per request);
    H = 768 and H = 256 run it with 8-CTA clusters, the others with 16. The top-K
    launch copies the candidates' rows of E itself: with one CTA per row (small V),
    with 4-CTA clusters (V = 50000, 6 ranks per CTA) and with 16-CTA clusters where
    only half of the CTAs have a rank to copy (V = 151936, K = 8)."""
    import diffusion_drafter_draft_gb300 as dd
    cfg = make_config("cfg1_qwen3_4b_c1").replace(C=C, L=L, V=V, H=H, K=K, W=W, B=B, seed=C * 1000 + K)
    inp = make_inputs(cfg)
    g, x = run_gpu_build(inp)
    o = compare_build(inp, g)
    tr = {k: torch.from_numpy(v).cuda() for k, v in g.items() if k in ("tok", "par", "depth", "n_nodes")}
    gv = host(dd.verify(tr, x["target"], dd.ROWS_PER_POSITION, cfg.L))
    compare_verify(o, gv, inp["target"], cfg, "position")


def test_stress_batch_sampled_requests():
    """Full C=64, K=512 batch on the GPU; the oracle checks a sample of requests
    (each request is drawn from its own stream, so a sample is bit-identical).
    The sample holds the first and last request of both halves that the batch is
    split into (0, 31 | 32, 63) and four more."""
    import diffusion_drafter_draft_gb300 as dd
    cfg = make_config("cfg4_c64_stress")
    full = make_inputs(cfg)
    g, x = run_gpu_build(full)
    sample = [0, 9, 23, 31, 32, 37, 50, 63]
    small = make_inputs(cfg, requests=sample)
    o = compare_build(small, g, rows=sample)
    # per-node target rows: sampled requests use their true slot depths, the rest a fixed layout
    depths = np.broadcast_to(breadth_first_slot_depth(cfg), (cfg.C, cfg.B + 1)).copy()
    for i, r in enumerate(sample):
        depths[r] = o["depth"][i]
    tgt = make_target_per_node(cfg, full, depths)
    tr = {k: torch.from_numpy(v).cuda() for k, v in g.items() if k in ("tok", "par", "depth", "n_nodes")}
    gv = host(dd.verify(tr, t(tgt, cfg.dtype), dd.ROWS_PER_NODE, cfg.L))
    gvs = {k: v[sample] for k, v in gv.items()}
    compare_verify(o, gvs, tgt[sample], cfg, "node")


@pytest.mark.parametrize("name,C,rows", [("cfg1_qwen3_4b_c1", None, "position"), ("cfg3_c4_adaptive", None, "position"),
                                         ("cfg0_tiny", 3, "position"), ("cfg2_qwen3_8b_fixed", 2, "node"),
                                         ("cfg4_c64_stress", 4, "node"), ("cfg4_c64_stress", 3, "position")])
def test_round_entry_point(name, C, rows):
    """dartree_round (row maxima on a side stream, fused finish kernel) gives the
    same tree and verification as dartree_build_tree + dartree_verify, and that
    tree matches the oracle."""
    import diffusion_drafter_draft_gb300 as dd
    cfg = make_config(name)
    if C:
        cfg = cfg.replace(C=C)
    cfg = cfg.replace(rows=rows)
    inp = make_inputs(cfg)
    x = upload(inp)
    if rows == "node":
        depths = np.broadcast_to(breadth_first_slot_depth(cfg), (cfg.C, cfg.B + 1)).copy()
        x["target"] = t(make_target_per_node(cfg, inp, depths), cfg.dtype)
    mode = dd.ROWS_PER_POSITION if rows == "position" else dd.ROWS_PER_NODE
    rnd = dd.Round(x["E"], x["Wq"], cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, mode)
    a = {k: v.clone() for k, v in rnd.run(x["base"], x["hidden"], x["anchor"], x["target"]).items()}
    ta = {k: v.clone() for k, v in rnd.tree.items()}
    b = {k: v.clone() for k, v in rnd.run_two_calls(x["base"], x["hidden"], x["anchor"], x["target"]).items()}
    tb = {k: v.clone() for k, v in rnd.tree.items()}
    torch.cuda.synchronize()
    assert dd.read_status(rnd.ws) == 0
    for k in a:
        assert torch.equal(a[k], b[k]), k
    for k in ta:
        assert torch.equal(ta[k], tb[k]), k
    g, _ = run_gpu_build(inp, dev_inputs=x)
    compare_build(inp, g)
    for k in ("tok", "par", "depth", "n_nodes", "mask", "pos"):
        np.testing.assert_array_equal(host(ta[k]), g[k], err_msg=k)


# --------------------------------------------------------------------------- exact ties

@pytest.mark.parametrize("name,C,L,V,H,K,W,B,beta,dtype", [
    ("f32 simple path", 2, 5, 30, 8, 4, 5, 9, 0.0, "f32"),
    ("f32 ragged", 3, 4, 211, 24, 5, 7, 9, 0.0, "f32"),
    ("bf16 candidate side", 2, 6, 3001, 256, 16, 6, 12, 0.0, "bf16"),
    ("bf16 candidate side, beta<0", 3, 5, 2000, 512, 64, 12, 30, -0.25, "bf16"),
    ("bf16 per-depth path", 5, 5, 3001, 256, 200, 12, 30, 0.0, "bf16"),
    ("qwen3-4b shape", 1, 16, 151936, 2560, 64, 12, 64, 0.0, "bf16"),
    ("qwen3-4b shape, beta<0", 1, 16, 151936, 2560, 64, 12, 64, -0.25, "bf16"),
])
def test_exact_ties_follow_the_stated_order(name, C, L, V, H, K, W, B, beta, dtype):
    """Tie-recipe inputs (E = 0, integer base logits with q = 1 for the top
    candidate): every selection is decided by exact ties, which the GPU must break
    as stated (top-K: lower token id; a depth's top-W: lower flat index p*K + c;
    the deferred prune: shallower depth, then lower rank). No near-tie adoption
    is allowed: the tree must equal the oracle's outright."""
    import diffusion_drafter_draft_gb300 as dd
    cfg = make_config("cfg1_qwen3_4b_c1").replace(C=C, L=L, V=V, H=H, K=K, W=W, B=B, beta=beta, dtype=dtype,
                                                   seed=100 + C * L + K)
    inp = make_tie_inputs(cfg)
    g, x = run_gpu_build(inp)
    o = compare_build(inp, g, max_flags=0)
    # scores are exact here: integers plus beta * depth
    np.testing.assert_array_equal(g["score"], o["score"].astype(np.float32))
    tr = {k: torch.from_numpy(v).cuda() for k, v in g.items() if k in ("tok", "par", "depth", "n_nodes")}
    gv = host(dd.verify(tr, x["target"], dd.ROWS_PER_POSITION, cfg.L))
    compare_verify(o, gv, inp["target"], cfg, "position")
    # the one-call round gives the same tree
    rnd = dd.Round(x["E"], x["Wq"], cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, dd.ROWS_PER_POSITION)
    out = {k: v.clone() for k, v in rnd.run(x["base"], x["hidden"], x["anchor"], x["target"]).items()}
    torch.cuda.synchronize()
    assert dd.read_status(rnd.ws) == 0
    for k in ("tok", "par", "depth", "n_nodes", "mask", "pos"):
        np.testing.assert_array_equal(host(rnd.tree[k]), o[k], err_msg=k)
    for k in ("accepted_len", "path", "bonus"):
        np.testing.assert_array_equal(host(out[k]), gv[k], err_msg=k)
