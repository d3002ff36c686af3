"""Seeded synthetic inputs for the DARTree draft-tree build and verify step.

This module is shared by the CPU oracle, the tests and the benchmark. It holds
none of the method's arithmetic: it only draws random tensors, plants peaks and
stores them in the storage type of a configuration (fp32, or bf16 kept as raw
uint16 bit patterns).

What stands in for what (DARTree, "3.1 Basic flow"): the block drafter's base
logits L_d^base, its shared hidden states H_d, the anchor token, the stand-in
correction head (embedding E and projection W_q) and the target model's logits
are all drawn here, because the drafter, the head and the target are trained
models that do not exist in this repository.

Recipe (all draws float32 from numpy PCG64):
  head weights   SeedSequence([seed, 2**31-1]): E[V,H] ~ N(0, 1/H), then W_q[H,H] ~ N(0, 1/H)
  request r      SeedSequence([seed, r]), in this order:
    anchor ~ U{0..V-1}
    base[L,V] ~ N(0, sigma^2); per position j a peak:
        'single8': one token U{0..V-1} raised by +8
        'zipf10' : m ~ U{1..4} distinct tokens, the i-th (i = 1..m) raised by 10 * i**-1.1
    hidden[L,H] ~ N(0, 1)
    per-position target[L,V] ~ N(0, sigma^2); per position j:
        'plant' : with probability agree_p the rank-1 planted token of base row j,
                  else a uniformly chosen other token, is raised by the rank-1 boost
        'argmax': after rounding, with probability agree_p the drafter's argmax of
                  base row j (lowest id among ties), else a uniformly chosen other
                  token, is set to rowmax + 1 (then rounded again)
  per-node target row j of request r: SeedSequence([seed, r, j]); noise ~ N(0, sigma^2),
    and the 'plant' rule with the planted token of position slot_depth[j]
    (no peak agreement when slot_depth[j] is -1 or >= L).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

__all__ = [
    "Config", "CONFIGS", "make_config", "make_inputs", "make_head",
    "make_target_per_node", "breadth_first_slot_depth", "make_tie_inputs", "round_to_bf16_bits",
    "bf16_bits_to_f32", "to_f32", "to_f64", "make_lm_head", "make_attention_inputs",
]

HEAD_STREAM = 2**31 - 1
TIE_STREAM = 2**31 - 2
LM_HEAD_STREAM = 2**31 - 3
ATTN_STREAM = 2**31 - 4


@dataclass(frozen=True)
class Config:
    name: str
    C: int        # concurrent requests
    L: int        # block length = maximum tree depth
    V: int        # vocabulary
    H: int        # hidden width of the stand-in head
    K: int        # candidates kept per block position
    W: int        # nodes kept per depth
    B: int        # node budget of the verification tree (root excluded)
    beta: float   # depth term, <= 0
    dtype: str    # 'f32' or 'bf16' (storage type of every float input)
    seed: int
    rows: str     # target logits 'position' [C,L,V] or 'node' [C,B+1,V]
    sigma: float
    plant: str    # 'single8' or 'zipf10'
    target: str   # 'plant' or 'argmax'
    agree_p: float

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


_CFG1 = Config("cfg1_qwen3_4b_c1", C=1, L=16, V=151936, H=2560, K=64, W=12, B=64,
               beta=-0.1, dtype="bf16", seed=1, rows="position", sigma=2.5,
               plant="zipf10", target="plant", agree_p=0.7)

CONFIGS: dict[str, Config] = {
    # tiny fp32 case the oracle finishes in well under a second
    "cfg0_tiny": Config("cfg0_tiny", C=1, L=8, V=1024, H=64, K=8, W=2, B=16, beta=-0.1,
                        dtype="f32", seed=0, rows="position", sigma=3.0,
                        plant="single8", target="plant", agree_p=0.7),
    # Qwen3-4B-shaped default, one request
    "cfg1_qwen3_4b_c1": _CFG1,
    # Qwen3-8B-shaped fixed-width variant (B = L*W: the prune keeps everything)
    "cfg2_qwen3_8b_fixed": _CFG1.replace(name="cfg2_qwen3_8b_fixed", H=4096, W=4, B=64,
                                         beta=-0.2, seed=2, target="argmax", agree_p=0.6),
    # concurrent serving batch with the adaptive budget, and the C=2 run
    "cfg3_c4_adaptive": _CFG1.replace(name="cfg3_c4_adaptive", C=4, W=3, B=32, seed=3),
    "cfg3_c2": _CFG1.replace(name="cfg3_c2", C=2, W=12, B=64, seed=3),
    # stress batch with per-node target rows
    "cfg4_c64_stress": _CFG1.replace(name="cfg4_c64_stress", C=64, H=4096, K=512, W=12,
                                     B=64, seed=4, rows="node"),
}


def make_config(name: str, **overrides) -> Config:
    return CONFIGS[name].replace(**overrides) if overrides else CONFIGS[name]


# --------------------------------------------------------------------------- storage

def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even on the uint32 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return round_to_bf16_bits(x)
    return np.ascontiguousarray(x, dtype=np.float32)


def to_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored array -> exact float32 values."""
    return bf16_bits_to_f32(a) if dtype == "bf16" else np.asarray(a, dtype=np.float32)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Stored array -> exact float64 values."""
    return to_f32(a, dtype).astype(np.float64)


# --------------------------------------------------------------------------- generators

def _rng(*words: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(words))))


def make_head(cfg: Config) -> tuple[np.ndarray, np.ndarray]:
    """Shared stand-in head weights (E[V,H], W_q[H,H]) in storage form."""
    rng = _rng(cfg.seed, HEAD_STREAM)
    scale = np.float32(1.0 / np.sqrt(cfg.H))
    E = np.empty((cfg.V, cfg.H), dtype=np.uint16 if cfg.dtype == "bf16" else np.float32)
    step = max(1, (1 << 24) // cfg.H)
    for r0 in range(0, cfg.V, step):
        r1 = min(cfg.V, r0 + step)
        E[r0:r1] = _store(rng.standard_normal((r1 - r0, cfg.H), dtype=np.float32) * scale, cfg.dtype)
    Wq = _store(rng.standard_normal((cfg.H, cfg.H), dtype=np.float32) * scale, cfg.dtype)
    return E, Wq


def make_lm_head(cfg: Config) -> np.ndarray:
    """Stand-in LM-head weights W_lm [V, H] of the block drafter in storage form,
    N(0, sigma^2 / H), so that the logits of the N(0, 1) block hidden states have the
    spread (sigma) of the configuration's base-logit noise."""
    rng = _rng(cfg.seed, LM_HEAD_STREAM)
    scale = np.float32(cfg.sigma / np.sqrt(cfg.H))
    W = np.empty((cfg.V, cfg.H), dtype=np.uint16 if cfg.dtype == "bf16" else np.float32)
    step = max(1, (1 << 24) // cfg.H)
    for r0 in range(0, cfg.V, step):
        r1 = min(cfg.V, r0 + step)
        W[r0:r1] = _store(rng.standard_normal((r1 - r0, cfg.H), dtype=np.float32) * scale, cfg.dtype)
    return W


def make_attention_inputs(C: int, S: int, Hq: int, Hkv: int, D: int, N: int, seed: int, n_ctx=None,
                          dtype: str = "bf16") -> dict:
    """One target attention layer's operands for the tree of each request, N(0, 1):
    tree queries q [C, S, Hq, D], tree keys/values k_tree, v_tree [C, S, Hkv, D]
    (queries and keys unrotated), and the cached prefix k_cache, v_cache
    [C, Hkv, N, D] (keys stored rotated); n_ctx [C] cached lengths (default N). Each
    request draws from its own stream, so a sample of a batch is bit-identical."""
    sdt = np.uint16 if dtype == "bf16" else np.float32
    out = dict(q=np.empty((C, S, Hq, D), sdt), k_tree=np.empty((C, S, Hkv, D), sdt),
               v_tree=np.empty((C, S, Hkv, D), sdt), k_cache=np.empty((C, Hkv, N, D), sdt),
               v_cache=np.empty((C, Hkv, N, D), sdt),
               n_ctx=np.full(C, N, np.int32) if n_ctx is None else np.asarray(n_ctx, np.int32))
    for r in range(C):
        rng = _rng(seed, ATTN_STREAM, r)
        for k, shape in (("q", (S, Hq, D)), ("k_tree", (S, Hkv, D)), ("v_tree", (S, Hkv, D)),
                         ("k_cache", (Hkv, N, D)), ("v_cache", (Hkv, N, D))):
            out[k][r] = _store(rng.standard_normal(shape, dtype=np.float32), dtype)
    return out


def _other_token(rng: np.random.Generator, V: int, avoid: int) -> int:
    return int((avoid + 1 + rng.integers(0, V - 1)) % V)


def _boosts(cfg: Config, rng: np.random.Generator) -> tuple[np.ndarray, np.ndarray]:
    if cfg.plant == "single8":
        return np.array([rng.integers(0, cfg.V)], dtype=np.int64), np.array([8.0], np.float32)
    m = int(rng.integers(1, 5))
    toks = rng.choice(cfg.V, size=m, replace=False).astype(np.int64)
    return toks, (10.0 * np.arange(1, m + 1, dtype=np.float64) ** -1.1).astype(np.float32)


def _argmax_low(row: np.ndarray) -> int:
    return int(np.argmax(row))  # first occurrence = lowest id among equal maxima


def make_inputs(cfg: Config, requests=None, with_head: bool = True) -> dict:
    """All per-request inputs (and, by default, the shared head) in storage form.

    requests: optional iterable of request ids (default range(C)); the result then
    holds only those requests, each drawn from its own stream exactly as in the full
    batch, so a sample of a large batch is bit-identical to the batch's rows.
    """
    reqs = list(range(cfg.C)) if requests is None else [int(r) for r in requests]
    n = len(reqs)
    sdt = np.uint16 if cfg.dtype == "bf16" else np.float32
    base = np.empty((n, cfg.L, cfg.V), sdt)
    hidden = np.empty((n, cfg.L, cfg.H), sdt)
    anchor = np.empty((n,), np.int32)
    planted = np.empty((n, cfg.L), np.int32)
    boost1 = np.empty((n, cfg.L), np.float32)
    target = np.empty((n, cfg.L, cfg.V), sdt) if cfg.rows == "position" else None
    for i, r in enumerate(reqs):
        rng = _rng(cfg.seed, r)
        anchor[i] = rng.integers(0, cfg.V)
        b = rng.standard_normal((cfg.L, cfg.V), dtype=np.float32) * np.float32(cfg.sigma)
        for j in range(cfg.L):
            toks, amt = _boosts(cfg, rng)
            b[j, toks] += amt
            planted[i, j] = toks[0]
            boost1[i, j] = amt[0]
        base[i] = _store(b, cfg.dtype)
        hidden[i] = _store(rng.standard_normal((cfg.L, cfg.H), dtype=np.float32), cfg.dtype)
        if target is None:
            continue
        t = rng.standard_normal((cfg.L, cfg.V), dtype=np.float32) * np.float32(cfg.sigma)
        if cfg.target == "plant":
            for j in range(cfg.L):
                agree = rng.random() < cfg.agree_p
                tok = int(planted[i, j]) if agree else _other_token(rng, cfg.V, int(planted[i, j]))
                t[j, tok] += boost1[i, j]
            target[i] = _store(t, cfg.dtype)
        else:  # 'argmax'
            ts = to_f32(_store(t, cfg.dtype), cfg.dtype).copy()
            bs = to_f32(base[i], cfg.dtype)
            for j in range(cfg.L):
                a = _argmax_low(bs[j])
                agree = rng.random() < cfg.agree_p
                tok = a if agree else _other_token(rng, cfg.V, a)
                ts[j, tok] = ts[j].max() + np.float32(1.0)
            target[i] = _store(ts, cfg.dtype)
    out = dict(cfg=cfg, requests=np.array(reqs, np.int64), base=base, hidden=hidden,
               anchor=anchor, planted=planted, boost1=boost1)
    if target is not None:
        out["target"] = target
    if with_head:
        out["E"], out["Wq"] = make_head(cfg)
    return out


def breadth_first_slot_depth(cfg: Config) -> np.ndarray:
    """A slot-depth layout that needs no tree: W slots per depth after the root.

    Used where per-node target rows are wanted without building a tree first.
    """
    d = np.zeros(cfg.B + 1, np.int64)
    d[1:] = 1 + (np.arange(cfg.B) // cfg.W)
    return np.minimum(d, cfg.L)


def make_target_per_node(cfg: Config, inputs: dict, slot_depth: np.ndarray) -> np.ndarray:
    """Per-node target rows [n, B+1, V] in storage form.

    slot_depth[i, j] is the depth of slot j of the i-th request of `inputs` (or a
    1-D layout shared by all requests); -1 marks an unused slot.
    """
    reqs = inputs["requests"]
    sd = np.asarray(slot_depth)
    if sd.ndim == 1:
        sd = np.broadcast_to(sd, (len(reqs), sd.shape[0]))
    nslot = cfg.B + 1
    sdt = np.uint16 if cfg.dtype == "bf16" else np.float32
    out = np.empty((len(reqs), nslot, cfg.V), sdt)
    for i, r in enumerate(reqs):
        for j in range(nslot):
            rng = _rng(cfg.seed, int(r), j)
            t = rng.standard_normal(cfg.V, dtype=np.float32) * np.float32(cfg.sigma)
            dj = int(sd[i, j]) if j < sd.shape[1] else -1
            if 0 <= dj < cfg.L:
                agree = rng.random() < cfg.agree_p
                p = int(inputs["planted"][i, dj])
                tok = p if agree else _other_token(rng, cfg.V, p)
                t[tok] += inputs["boost1"][i, dj]
            out[i, j] = _store(t, cfg.dtype)
    return out


def make_tie_inputs(cfg: Config, requests=None) -> dict:
    """Inputs on which the tree is decided by exact ties (tie-order checks).

    Starts from make_inputs(cfg, requests) and replaces two things:
      E = 0, so every parent sees the same corrected logits (the base logits);
      base row j of request r (stream SeedSequence([seed, r, 2**31-2])): one token
        U{0..V-1} at 8, n ~ U{0..K} other distinct tokens at 8 - (64 + j mod 16),
        every other token at 8 - (96 + j mod 16).
    Every value is an integer, and the gaps below the top token are large enough
    that the other tokens' exponentials vanish next to it, so the log-softmax of
    the top candidate is exactly 0 and the others sit at exactly -(64 + j mod 16)
    or -(96 + j mod 16). Scores are sums of integers and beta*d: with beta = 0 or
    a short binary fraction they are exact in float32 and float64 alike, and
    children that tie do so exactly (inside a depth, and, with beta = 0, with
    their parents across depths). Heavy ties at the K-th candidate exercise the
    top-K order too. Target rows (per-position layout) are the make_inputs rows
    with, per position and with probability 0.7, the top base token set to the
    row maximum + 1, so that verification accepts part of the block.
    """
    out = make_inputs(cfg, requests)
    reqs = out["requests"]
    out["E"] = np.zeros_like(out["E"])
    base = np.empty((len(reqs), cfg.L, cfg.V), np.float32)
    tops = np.empty((len(reqs), cfg.L), np.int64)
    for i, r in enumerate(reqs):
        rng = _rng(cfg.seed, int(r), TIE_STREAM)
        for j in range(cfg.L):
            row = np.full(cfg.V, np.float32(8 - (96 + j % 16)), np.float32)
            top = int(rng.integers(0, cfg.V))
            n2 = int(rng.integers(0, min(cfg.K, cfg.V - 1) + 1))
            others = rng.choice(cfg.V - 1, size=n2, replace=False)
            others = others + (others >= top)          # distinct from the top token
            row[others] = np.float32(8 - (64 + j % 16))
            row[top] = np.float32(8.0)
            base[i, j] = row
            tops[i, j] = top
        if "target" in out:
            t = to_f32(out["target"][i], cfg.dtype).copy()
            for j in range(cfg.L):
                if rng.random() < 0.7:
                    t[j, tops[i, j]] = t[j].max() + np.float32(1.0)
            out["target"][i] = _store(t, cfg.dtype)
    out["base"] = _store(base, cfg.dtype)
    out["planted"] = tops.astype(np.int32)
    return out
