"""Two callers on two streams at the C=64 stress shape.

Each dartree_round call of a 64-request batch forks the second half of its
expansion onto a library side stream that belongs to the caller's stream; two
callers on two streams therefore run concurrently without sharing a side stream.
Both rounds, enqueued back to back on their own streams several times, must give
exactly the trees and verification results of dartree_build_tree followed by
dartree_verify on the default stream (which the other parity tests check against
the oracle).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from dartree_inputs import make_config, make_inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dd():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from diffusion_drafter_draft_gb300 import _build
    _build.build()
    import diffusion_drafter_draft_gb300 as m
    m.lib()
    return m


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def test_two_streams_run_c64_rounds_concurrently(dd):
    cfg = make_config("cfg4_c64_stress").replace(rows="position")
    inp = make_inputs(cfg)
    E, Wq = _dev(inp["E"]), _dev(inp["Wq"])
    a = dict(base=_dev(inp["base"]), hidden=_dev(inp["hidden"]), anchor=torch.from_numpy(inp["anchor"]).cuda(),
             target=_dev(inp["target"]))
    # the second caller's batch: the same requests in reverse order
    b = {k: v.flip(0).contiguous() for k, v in a.items()}
    mode = dd.ROWS_PER_POSITION

    def reference(x):
        t = dd.build_tree(E, Wq, x["base"], x["hidden"], x["anchor"], cfg.K, cfg.W, cfg.B, cfg.beta)
        v = dd.verify(t, x["target"], mode, cfg.L)
        torch.cuda.synchronize()
        return {k: t[k].cpu().numpy() for k in ("tok", "par", "depth", "score", "n_nodes", "mask", "pos")}, \
            {k: w.cpu().numpy() for k, w in v.items()}

    ref_a, vref_a = reference(a)
    ref_b, vref_b = reference(b)
    # the reversed batch gives the reversed results
    for k in ref_a:
        np.testing.assert_array_equal(ref_b[k], ref_a[k][::-1], err_msg=k)

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    ra = dd.Round(E, Wq, cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, mode)
    rb = dd.Round(E, Wq, cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, mode)
    torch.cuda.synchronize()
    for _ in range(3):
        with torch.cuda.stream(s1):
            out_a = ra.run(a["base"], a["hidden"], a["anchor"], a["target"])
        with torch.cuda.stream(s2):
            out_b = rb.run(b["base"], b["hidden"], b["anchor"], b["target"])
    torch.cuda.synchronize()
    assert dd.read_status(ra.ws) == 0 and dd.read_status(rb.ws) == 0
    for r, out, ref, vref in ((ra, out_a, ref_a, vref_a), (rb, out_b, ref_b, vref_b)):
        for k in ref:
            np.testing.assert_array_equal(r.tree[k].cpu().numpy(), ref[k], err_msg=k)
        for k in vref:
            np.testing.assert_array_equal(out[k].cpu().numpy(), vref[k], err_msg=k)


def test_host_rounds_match_device_rounds(dd):
    """dd.HostRounds (inputs copied from pinned host memory on a copy stream while the
    previous round runs, results copied back) gives, round after round, the results of
    Round.run on device inputs. Three different input sets alternate, so a round that
    read a stale input set would show."""
    cfg = make_config("cfg1_qwen3_4b_c1").replace(C=2)
    sets = []
    for seed in (11, 12, 13):
        inp = make_inputs(cfg.replace(seed=seed))
        sets.append(inp)
    E, Wq = _dev(sets[0]["E"]), _dev(sets[0]["Wq"])   # the head of seed 11 for every round
    rnd = dd.Round(E, Wq, cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, dd.ROWS_PER_POSITION)

    def host_set(inp):
        return dict(base=_dev(inp["base"]).cpu().pin_memory(), hidden=_dev(inp["hidden"]).cpu().pin_memory(),
                    anchor=torch.from_numpy(inp["anchor"]).pin_memory(),
                    target=_dev(inp["target"]).cpu().pin_memory())

    hs = [host_set(inp) for inp in sets]
    want = []
    for h in hs:
        o = rnd.run(*(h[k].cuda() for k in dd.HostRounds.KEYS))
        torch.cuda.synchronize()
        want.append({k: v.cpu().clone() for k, v in o.items()})
    hr = dd.HostRounds(rnd, hs[0])
    n = 7
    outs = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in rnd.out.items()} for _ in range(n)]
    hr.copy_in(0, hs[0])
    for i in range(n):
        if i + 1 < n:
            hr.copy_in(i + 1, hs[(i + 1) % 3])
        hr.run(i, outs[i])
    torch.cuda.synchronize()
    for i in range(n):
        for k in want[i % 3]:
            assert torch.equal(outs[i][k], want[i % 3][k]), (i, k)


@pytest.mark.gpu
def test_host_session_order_is_checked(dd):
    """dartree_host_round with no staged inputs, and a third stage while two staged
    sets wait for their rounds, are rejected (DARTREE_EINVAL) without enqueueing work;
    the session carries on afterwards."""
    cfg = make_config("cfg1_qwen3_4b_c1").replace(C=1)
    inp = make_inputs(cfg)
    E, Wq = _dev(inp["E"]), _dev(inp["Wq"])
    rnd = dd.Round(E, Wq, cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, dd.ROWS_PER_POSITION)
    h = dict(base=_dev(inp["base"]).cpu().pin_memory(), hidden=_dev(inp["hidden"]).cpu().pin_memory(),
             anchor=torch.from_numpy(inp["anchor"]).pin_memory(), target=_dev(inp["target"]).cpu().pin_memory())
    out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in rnd.out.items()}
    hr = dd.HostRounds(rnd)
    with pytest.raises(dd.DartreeError) as e:
        hr.run(0, out)
    assert e.value.code == dd.EINVAL
    hr.copy_in(0, h)
    hr.copy_in(1, h)
    with pytest.raises(dd.DartreeError) as e:
        hr.copy_in(2, h)
    assert e.value.code == dd.EINVAL
    for i in range(2):
        hr.run(i, out)
    torch.cuda.synchronize()
    want = rnd.run(*(h[k].cuda() for k in dd.HostRounds.KEYS))
    torch.cuda.synchronize()
    for k, v in want.items():
        assert torch.equal(out[k], v.cpu()), k


def test_host_session_per_node_rows_f32(dd):
    """The host session with an fp32 head and per-node target rows ([C, B+1, V]):
    round after round equal to Round.run on device copies of the same inputs, with
    two input sets alternating."""
    from dartree_inputs import breadth_first_slot_depth, make_target_per_node
    cfg = make_config("cfg0_tiny").replace(C=3, rows="node")
    sets = []
    for seed in (5, 6):
        inp = make_inputs(cfg.replace(seed=seed))
        inp["target"] = make_target_per_node(cfg, inp, breadth_first_slot_depth(cfg))
        sets.append(inp)
    E = torch.from_numpy(sets[0]["E"]).cuda()
    Wq = torch.from_numpy(sets[0]["Wq"]).cuda()
    rnd = dd.Round(E, Wq, cfg.C, cfg.L, cfg.K, cfg.W, cfg.B, cfg.beta, dd.ROWS_PER_NODE)
    hs = [{k: torch.from_numpy(np.ascontiguousarray(s[k])).pin_memory() for k in dd.HostRounds.KEYS} for s in sets]
    want = []
    for h in hs:
        o = rnd.run(*(h[k].cuda() for k in dd.HostRounds.KEYS))
        torch.cuda.synchronize()
        want.append({k: v.cpu().clone() for k, v in o.items()})
    hr = dd.HostRounds(rnd)
    n = 5
    outs = [{k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in rnd.out.items()} for _ in range(n)]
    hr.copy_in(0, hs[0])
    for i in range(n):
        if i + 1 < n:
            hr.copy_in(i + 1, hs[(i + 1) % 2])
        hr.run(i, outs[i])
    torch.cuda.synchronize()
    for i in range(n):
        for k in want[i % 2]:
            assert torch.equal(outs[i][k], want[i % 2][k]), (i, k)
