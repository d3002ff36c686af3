"""Python binding of libdartree.so, the sm_103a DARTree draft-tree build and verify step.

Argument marshalling only: every step runs in the library's CUDA kernels. Tensors
are torch CUDA tensors (PyTorch supplies device memory and the current stream);
they are passed to the C ABI as raw device pointers. There is no CPU fallback:
if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "DartreeError", "lib", "library_path", "F32", "BF16", "ROWS_PER_POSITION", "ROWS_PER_NODE",
    "workspace_bytes", "new_workspace", "topk", "expand", "prune", "tree_mask", "build_tree",
    "verify", "read_status", "clear_status", "Round", "EXPORTS", "heap_build", "HeapRound",
    "verify_sample", "adaptive_budget", "lm_head_topk", "tree_attention", "AttnParams", "HostRounds",
    "HostInputs", "HostOutputs",
]

F32, BF16 = 0, 1
ROWS_PER_POSITION, ROWS_PER_NODE = 0, 1
OK, EINVAL, EDTYPE, EWORKSPACE, ECUDA, ETIMEOUT, EINTERNAL, EUNSUPPORTED = 0, -1, -2, -3, -4, -5, -6, -7

EXPORTS = ("dartree_head_init", "dartree_workspace_bytes", "dartree_topk", "dartree_expand", "dartree_prune",
           "dartree_tree_mask", "dartree_build_tree", "dartree_verify", "dartree_read_status",
           "dartree_clear_status", "dartree_status_string", "dartree_verify_static", "dartree_gemm_bf16",
           "dartree_head_prepare", "dartree_round", "dartree_selftest_wait", "dartree_timing",
           "dartree_timing_read", "dartree_kernel_name", "dartree_heap_workspace_bytes", "dartree_heap_build",
           "dartree_verify_sample", "dartree_adaptive_budget", "dartree_lm_head_workspace_bytes",
           "dartree_lm_head_topk", "dartree_tree_attention_workspace_bytes", "dartree_tree_attention", "dartree_host_session_create",
           "dartree_host_session_destroy", "dartree_host_stage", "dartree_host_round", "dartree_host_input_bytes")


class DartreeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {code} ({status_string(code)})")


class Head(ctypes.Structure):
    _fields_ = [("E", ctypes.c_void_p), ("Wq", ctypes.c_void_p), ("V", ctypes.c_int), ("H", ctypes.c_int),
                ("dtype", ctypes.c_int), ("WqT", ctypes.c_void_p)]


class Params(ctypes.Structure):
    _fields_ = [("C", ctypes.c_int), ("L", ctypes.c_int), ("K", ctypes.c_int), ("W", ctypes.c_int),
                ("B", ctypes.c_int), ("beta", ctypes.c_float)]


class Candidates(ctypes.Structure):
    _fields_ = [("tok", ctypes.c_void_p), ("logit", ctypes.c_void_p)]


class Supertree(ctypes.Structure):
    _fields_ = [("tok", ctypes.c_void_p), ("par", ctypes.c_void_p), ("score", ctypes.c_void_p),
                ("n", ctypes.c_void_p)]


class AttnParams(ctypes.Structure):
    _fields_ = [("C", ctypes.c_int), ("S", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
                ("D", ctypes.c_int), ("N", ctypes.c_int), ("theta", ctypes.c_float)]


class Tree(ctypes.Structure):
    _fields_ = [("tok", ctypes.c_void_p), ("par", ctypes.c_void_p), ("depth", ctypes.c_void_p),
                ("score", ctypes.c_void_p), ("n_nodes", ctypes.c_void_p), ("mask", ctypes.c_void_p),
                ("pos", ctypes.c_void_p)]


_LIB = None


def library_path() -> str:
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), "libdartree.so")


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with diffusion_drafter_draft_gb300._build.build()")
    L = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "dartree_head_init": (i, [P(Head), vp, vp, i, i, i]),
        "dartree_round": (i, [P(Head), P(Params), vp, vp, vp, vp, i, P(Tree), vp, vp, vp, vp, sz, vp]),
        "dartree_selftest_wait": (i, [vp, sz, i, ctypes.c_uint, vp]),
        "dartree_timing": (i, [i]),
        "dartree_timing_read": (i, [i, P(ctypes.c_int), P(ctypes.c_double)]),
        "dartree_kernel_name": (ctypes.c_char_p, [i]),
        "dartree_head_prepare": (i, [P(Head), vp, vp]),
        "dartree_heap_workspace_bytes": (sz, [P(Params), i, i, i]),
        "dartree_heap_build": (i, [P(Head), P(Params), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "dartree_workspace_bytes": (sz, [P(Params), i, i, i]),
        "dartree_topk": (i, [vp, i, i, i, i, vp, vp, vp, sz, vp]),
        "dartree_expand": (i, [P(Head), P(Params), vp, vp, P(Candidates), P(Supertree), vp, sz, vp]),
        "dartree_prune": (i, [P(Params), P(Supertree), vp, P(Tree), vp]),
        "dartree_tree_mask": (i, [P(Params), P(Tree), vp]),
        "dartree_build_tree": (i, [P(Head), P(Params), vp, vp, vp, P(Tree), P(Supertree), P(Candidates), vp, sz,
                                   vp]),
        "dartree_verify": (i, [P(Params), P(Tree), vp, i, i, i, vp, vp, vp, vp, sz, vp]),
        "dartree_verify_static": (i, [P(Params), P(Tree), vp, i, i, i, vp, vp, vp, vp]),
        "dartree_verify_sample": (i, [P(Params), P(Tree), vp, i, i, i, ctypes.c_float, ctypes.c_uint64, vp, vp, vp,
                                      vp, sz, vp]),
        "dartree_adaptive_budget": (i, [i, P(ctypes.c_int), P(ctypes.c_int)]),
        "dartree_lm_head_workspace_bytes": (sz, [i, i, i, i]),
        "dartree_tree_attention_workspace_bytes": (sz, [P(AttnParams)]),
        "dartree_tree_attention": (i, [P(AttnParams), vp, vp, vp, vp, vp, vp, P(Tree), vp, vp, sz, vp]),
        "dartree_lm_head_topk": (i, [vp, vp, i, i, i, i, i, vp, vp, vp, sz, vp]),
        "dartree_gemm_bf16": (i, [vp, vp, vp, i, i, i, vp, vp]),
        "dartree_read_status": (i, [vp, P(ctypes.c_int32), vp]),
        "dartree_clear_status": (i, [vp, vp]),
        "dartree_status_string": (ctypes.c_char_p, [i]),
        "dartree_host_session_create": (i, [P(Head), P(Params), i, P(vp)]),
        "dartree_host_session_destroy": (None, [vp]),
        "dartree_host_stage": (i, [vp, P(HostInputs)]),
        "dartree_host_round": (i, [vp, P(HostOutputs), vp]),
        "dartree_host_input_bytes": (sz, [vp, i]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype, f.argtypes = res, args
    _LIB = L
    return L


def status_string(code: int) -> str:
    try:
        return lib().dartree_status_string(code).decode()
    except Exception:  # library missing while formatting an error
        return "?"


def _call(name: str, *args) -> None:
    rc = getattr(lib(), name)(*args)
    if rc != OK:
        raise DartreeError(rc, name)


# --------------------------------------------------------------------------- tensors

_DT = {torch.float32: F32, torch.bfloat16: BF16}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DT:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DT[t.dtype]


def _need(t: torch.Tensor, name: str, dtype=None, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream=None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _keep(stream, *tensors) -> None:
    """Tensors allocated here and used by work enqueued on a side stream are not
    reused by the caching allocator before that work is done."""
    if stream is None or stream == torch.cuda.current_stream():
        return
    for t in tensors:
        if t is not None:
            t.record_stream(stream)


def _params(C, L, K, W, B, beta) -> Params:
    return Params(int(C), int(L), int(K), int(W), int(B), float(beta))


def workspace_bytes(C, L, K, W, B, beta, V, H, dtype_code) -> int:
    n = lib().dartree_workspace_bytes(ctypes.byref(_params(C, L, K, W, B, beta)), int(V), int(H), int(dtype_code))
    if n == 0:
        raise DartreeError(EINVAL, "dartree_workspace_bytes")
    return int(n)


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    ws = torch.zeros(int(nbytes), dtype=torch.uint8, device=device or "cuda")
    if ws.data_ptr() % 256:
        raise RuntimeError("workspace is not 256-byte aligned")
    return ws


def read_status(ws: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32(0)
    _call("dartree_read_status", ctypes.c_void_p(ws.data_ptr()), ctypes.byref(v), _stream(stream))
    return int(v.value)


def selftest_wait(ws: torch.Tensor, which: int, limit_us: int, stream=None) -> None:
    """Enqueues a bounded wait on something never signalled (0: mbarrier, 1: grid
    barrier); it must end after limit_us with DARTREE_ETIMEOUT in ws's status word."""
    _call("dartree_selftest_wait", ctypes.c_void_p(ws.data_ptr()), ws.numel(), int(which), int(limit_us),
          _stream(stream))


def num_kernel_ids() -> int:
    """Kernel families the library times (ids 0 .. n-1; the last one is "other")."""
    n = 0
    while lib().dartree_kernel_name(n).decode() != "unknown":
        n += 1
    return n


def timing(enable: bool) -> None:
    """Starts (clearing earlier records) or stops per-kernel launch timing."""
    _call("dartree_timing", int(bool(enable)))


def kernel_times() -> dict:
    """{kernel family: (launches, total device ms)} recorded since timing(True)."""
    out = {}
    for k in range(num_kernel_ids()):
        n, ms = ctypes.c_int(0), ctypes.c_double(0.0)
        _call("dartree_timing_read", k, ctypes.byref(n), ctypes.byref(ms))
        if n.value:
            out[lib().dartree_kernel_name(k).decode()] = (int(n.value), float(ms.value))
    return out


def clear_status(ws: torch.Tensor, stream=None) -> None:
    _call("dartree_clear_status", ctypes.c_void_p(ws.data_ptr()), _stream(stream))


def _head(E: torch.Tensor, Wq: torch.Tensor, prepare: bool = False, stream=None):
    """(head description, W_q^T tensor or None). With prepare, bf16 heads get W_q^T
    for the small-batch path; the caller keeps the returned tensor alive while the
    head is used."""
    V, H = E.shape
    _need(E, "E")
    _need(Wq, "Wq", E.dtype, (H, H))
    h = Head()
    _call("dartree_head_init", ctypes.byref(h), ctypes.c_void_p(E.data_ptr()), ctypes.c_void_p(Wq.data_ptr()),
          int(V), int(H), _dtype_code(E))
    wqt = None
    if prepare and E.dtype == torch.bfloat16:
        wqt = torch.empty((H, H), dtype=E.dtype, device=E.device)
        _call("dartree_head_prepare", ctypes.byref(h), ctypes.c_void_p(wqt.data_ptr()), _stream(stream))
    return h, wqt


# --------------------------------------------------------------------------- steps

def topk(logits: torch.Tensor, K: int, ws: torch.Tensor | None = None, stream=None):
    """S1: top-K of every row of logits [rows, V] -> (tok int32 [rows, K], val float32 [rows, K])."""
    rows, V = logits.shape
    _need(logits, "logits")
    dev = logits.device
    tok = torch.empty((rows, K), dtype=torch.int32, device=dev)
    val = torch.empty((rows, K), dtype=torch.float32, device=dev)
    ws = ws if ws is not None else new_workspace(256, dev)
    _call("dartree_topk", ctypes.c_void_p(logits.data_ptr()), int(rows), int(V), int(K), _dtype_code(logits),
          ctypes.c_void_p(tok.data_ptr()), ctypes.c_void_p(val.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
          ws.numel(), _stream(stream))
    return tok, val


def _alloc_supertree(C, L, W, dev):
    return dict(tok=torch.empty((C, L, W), dtype=torch.int32, device=dev),
                par=torch.empty((C, L, W), dtype=torch.int32, device=dev),
                score=torch.empty((C, L, W), dtype=torch.float32, device=dev),
                n=torch.empty((C, L), dtype=torch.int32, device=dev))


def _st_struct(st) -> Supertree:
    return Supertree(st["tok"].data_ptr(), st["par"].data_ptr(), st["score"].data_ptr(), st["n"].data_ptr())


def _alloc_tree(C, B, dev, with_mask=True):
    S = B + 1
    t = dict(tok=torch.empty((C, S), dtype=torch.int32, device=dev),
             par=torch.empty((C, S), dtype=torch.int32, device=dev),
             depth=torch.empty((C, S), dtype=torch.int32, device=dev),
             score=torch.empty((C, S), dtype=torch.float32, device=dev),
             n_nodes=torch.empty((C,), dtype=torch.int32, device=dev))
    if with_mask:
        t["mask"] = torch.empty((C, S, S), dtype=torch.uint8, device=dev)
        t["pos"] = torch.empty((C, S), dtype=torch.int32, device=dev)
    return t


def _tree_struct(t) -> Tree:
    g = lambda k: t[k].data_ptr() if k in t and t[k] is not None else None  # noqa: E731
    return Tree(g("tok"), g("par"), g("depth"), g("score"), g("n_nodes"), g("mask"), g("pos"))


def expand(E, Wq, hidden, anchor, cand_tok, cand_val, W, beta, ws=None, stream=None):
    """S2-S7 from a candidate table -> supertree dict (tok, par, score, n)."""
    C, L, H = hidden.shape
    K = cand_tok.shape[-1]
    head, wqt = _head(E, Wq, prepare=True, stream=stream)
    _need(hidden, "hidden", E.dtype, (C, L, H))
    _need(anchor, "anchor", torch.int32, (C,))
    _need(cand_tok, "cand_tok", torch.int32, (C, L, K))
    _need(cand_val, "cand_val", torch.float32, (C, L, K))
    p = _params(C, L, K, W, 1, beta)
    ws = ws if ws is not None else new_workspace(workspace_bytes(C, L, K, W, 1, beta, E.shape[0], H, head.dtype),
                                                 hidden.device)
    st = _alloc_supertree(C, L, W, hidden.device)
    cand = Candidates(cand_tok.data_ptr(), cand_val.data_ptr())
    sts = _st_struct(st)
    _call("dartree_expand", ctypes.byref(head), ctypes.byref(p), ctypes.c_void_p(hidden.data_ptr()),
          ctypes.c_void_p(anchor.data_ptr()), ctypes.byref(cand), ctypes.byref(sts), ctypes.c_void_p(ws.data_ptr()),
          ws.numel(), _stream(stream))
    _keep(stream, ws, wqt)
    return st


def prune(st, anchor, B, stream=None):
    """S8: deferred pruning of a supertree -> tree dict (tok, par, depth, score, n_nodes)."""
    C, L, W = st["tok"].shape
    for k in ("tok", "par", "n"):
        _need(st[k], k, torch.int32)
    _need(st["score"], "score", torch.float32)
    _need(anchor, "anchor", torch.int32, (C,))
    t = _alloc_tree(C, B, anchor.device, with_mask=False)
    p = _params(C, L, 1, W, B, 0.0)
    ts, sts = _tree_struct(t), _st_struct(st)
    _call("dartree_prune", ctypes.byref(p), ctypes.byref(sts), ctypes.c_void_p(anchor.data_ptr()), ctypes.byref(ts),
          _stream(stream))
    return t


def tree_mask(tree, L, stream=None):
    """S9: adds mask and pos to a tree dict (in place) and returns it."""
    C, S = tree["par"].shape
    for k in ("par", "depth", "n_nodes"):
        _need(tree[k], k, torch.int32)
    tree["mask"] = torch.empty((C, S, S), dtype=torch.uint8, device=tree["par"].device)
    tree["pos"] = torch.empty((C, S), dtype=torch.int32, device=tree["par"].device)
    p = _params(C, L, 1, 1, S - 1, 0.0)
    ts = _tree_struct(tree)
    _call("dartree_tree_mask", ctypes.byref(p), ctypes.byref(ts), _stream(stream))
    return tree


def verify(tree, target, rows: int, L: int, ws=None, stream=None):
    """S10: greedy longest accepted prefix -> dict(accepted_len, path, bonus)."""
    C, S = tree["tok"].shape
    V = target.shape[-1]
    _need(target, "target", None, (C, L, V) if rows == ROWS_PER_POSITION else (C, S, V))
    dev = target.device
    out = dict(accepted_len=torch.empty((C,), dtype=torch.int32, device=dev),
               path=torch.empty((C, L), dtype=torch.int32, device=dev),
               bonus=torch.empty((C,), dtype=torch.int32, device=dev))
    if ws is None:
        ws = new_workspace(256 + 8 * C * max(L, S), dev)
    p = _params(C, L, 1, 1, S - 1, 0.0)
    ts = _tree_struct(tree)
    _call("dartree_verify", ctypes.byref(p), ctypes.byref(ts), ctypes.c_void_p(target.data_ptr()), int(rows), int(V),
          _dtype_code(target), ctypes.c_void_p(out["accepted_len"].data_ptr()), ctypes.c_void_p(out["path"].data_ptr()),
          ctypes.c_void_p(out["bonus"].data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    return out


def verify_sample(tree, target, rows: int, L: int, temperature: float, seed: int, ws=None, stream=None):
    """S10 at temperature T > 0 (Gumbel-max draws, Philox4x32-10 noise keyed by seed)
    -> dict(accepted_len, path, bonus)."""
    C, S = tree["tok"].shape
    V = target.shape[-1]
    _need(target, "target", None, (C, L, V) if rows == ROWS_PER_POSITION else (C, S, V))
    dev = target.device
    out = dict(accepted_len=torch.empty((C,), dtype=torch.int32, device=dev),
               path=torch.empty((C, L), dtype=torch.int32, device=dev),
               bonus=torch.empty((C,), dtype=torch.int32, device=dev))
    if ws is None:
        ws = new_workspace(256 + 8 * C * max(L, S), dev)
    p = _params(C, L, 1, 1, S - 1, 0.0)
    ts = _tree_struct(tree)
    _call("dartree_verify_sample", ctypes.byref(p), ctypes.byref(ts), ctypes.c_void_p(target.data_ptr()), int(rows),
          int(V), _dtype_code(target), float(temperature), int(seed) & 0xFFFFFFFFFFFFFFFF,
          ctypes.c_void_p(out["accepted_len"].data_ptr()), ctypes.c_void_p(out["path"].data_ptr()),
          ctypes.c_void_p(out["bonus"].data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    return out


def adaptive_budget(C: int) -> tuple[int, int]:
    """(B, W) for C concurrent requests (dartree_adaptive_budget)."""
    B, W = ctypes.c_int(), ctypes.c_int()
    _call("dartree_adaptive_budget", int(C), ctypes.byref(B), ctypes.byref(W))
    return B.value, W.value


def lm_head_topk(hidden, W_lm, K: int, ws=None, stream=None):
    """The drafter's LM head fused with S1: hidden [R, H] x W_lm[V, H]^T -> per-row
    top-K (tok [R, K] int32, val [R, K] fp32), logits never written."""
    R, H = hidden.shape
    V = W_lm.shape[0]
    _need(hidden, "hidden", torch.bfloat16, (R, H))
    _need(W_lm, "W_lm", torch.bfloat16, (V, H))
    dev = hidden.device
    tok = torch.empty((R, K), dtype=torch.int32, device=dev)
    val = torch.empty((R, K), dtype=torch.float32, device=dev)
    need = lib().dartree_lm_head_workspace_bytes(R, V, H, K)
    if need == 0:
        raise DartreeError(EUNSUPPORTED, "dartree_lm_head_workspace_bytes")
    if ws is None:
        ws = new_workspace(need, dev)
    _call("dartree_lm_head_topk", ctypes.c_void_p(hidden.data_ptr()), ctypes.c_void_p(W_lm.data_ptr()), R, V, H,
          int(K), BF16, ctypes.c_void_p(tok.data_ptr()), ctypes.c_void_p(val.data_ptr()),
          ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    return tok, val


def tree_attention(q, k_tree, v_tree, k_cache, vt_cache, n_ctx, tree, theta: float = 1.0e6, ws=None,
                   stream=None):
    """One attention layer of the verification pass over the tree (dartree_tree_attention):
    q [C, S, Hq, D], k_tree/v_tree [C, S, Hkv, D], k_cache [C, Hkv, N, D], vt_cache
    [C, Hkv, D, N] (bf16), n_ctx [C] int32, tree with mask/pos/n_nodes -> out [C, S, Hq, D]."""
    C, S, Hq, D = q.shape
    Hkv = k_tree.shape[2]
    N = k_cache.shape[2]
    for name, x, shp in (("q", q, (C, S, Hq, D)), ("k_tree", k_tree, (C, S, Hkv, D)),
                         ("v_tree", v_tree, (C, S, Hkv, D)), ("k_cache", k_cache, (C, Hkv, N, D)),
                         ("vt_cache", vt_cache, (C, Hkv, D, N))):
        _need(x, name, torch.bfloat16, shp)
    _need(n_ctx, "n_ctx", torch.int32, (C,))
    _need(tree["mask"], "mask", torch.uint8, (C, S, S))
    _need(tree["pos"], "pos", torch.int32, (C, S))
    _need(tree["n_nodes"], "n_nodes", torch.int32, (C,))
    p = AttnParams(C, S, Hq, Hkv, D, N, float(theta))
    need = lib().dartree_tree_attention_workspace_bytes(ctypes.byref(p))
    if need == 0:
        raise DartreeError(EUNSUPPORTED, "dartree_tree_attention_workspace_bytes")
    if ws is None:
        ws = new_workspace(need, q.device)
    out = torch.empty((C, S, Hq, D), dtype=torch.bfloat16, device=q.device)
    ts = _tree_struct({k: tree[k] for k in ("mask", "pos", "n_nodes")})
    _call("dartree_tree_attention", ctypes.byref(p), *(ctypes.c_void_p(x.data_ptr()) for x in
                                                       (q, k_tree, v_tree, k_cache, vt_cache, n_ctx)),
          ctypes.byref(ts), ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(),
          _stream(stream))
    return out


def verify_static(tree, target, rows: int, L: int, stream=None):
    """S10 through dartree_verify_static (no workspace; scratch in a fixed device array)."""
    C, S = tree["tok"].shape
    V = target.shape[-1]
    _need(target, "target", None, (C, L, V) if rows == ROWS_PER_POSITION else (C, S, V))
    dev = target.device
    out = dict(accepted_len=torch.empty((C,), dtype=torch.int32, device=dev),
               path=torch.empty((C, L), dtype=torch.int32, device=dev),
               bonus=torch.empty((C,), dtype=torch.int32, device=dev))
    p = _params(C, L, 1, 1, S - 1, 0.0)
    ts = _tree_struct(tree)
    _call("dartree_verify_static", ctypes.byref(p), ctypes.byref(ts), ctypes.c_void_p(target.data_ptr()), int(rows),
          int(V), _dtype_code(target), ctypes.c_void_p(out["accepted_len"].data_ptr()),
          ctypes.c_void_p(out["path"].data_ptr()), ctypes.c_void_p(out["bonus"].data_ptr()), _stream(stream))
    return out


def gemm_bf16(A, B, status=None, stream=None):
    """Building block: D = A . B^T (bf16 in, fp32 out) through the tcgen05 GEMM."""
    M, K = A.shape
    N = B.shape[0]
    _need(A, "A", torch.bfloat16)
    _need(B, "B", torch.bfloat16, (N, K))
    D = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _call("dartree_gemm_bf16", ctypes.c_void_p(A.data_ptr()), ctypes.c_void_p(B.data_ptr()),
          ctypes.c_void_p(D.data_ptr()), int(M), int(N), int(K),
          ctypes.c_void_p(status.data_ptr()) if status is not None else None, _stream(stream))
    return D


def build_tree(E, Wq, base, hidden, anchor, K, W, B, beta, ws=None, keep_intermediates=False, stream=None):
    """S1-S9: one tree build -> tree dict (+ 'cand_tok', 'cand_val', 'st' when keep_intermediates)."""
    C, L, V = base.shape
    H = E.shape[1]
    head, wqt = _head(E, Wq, prepare=True, stream=stream)
    _need(base, "base", E.dtype, (C, L, V))
    _need(hidden, "hidden", E.dtype, (C, L, H))
    _need(anchor, "anchor", torch.int32, (C,))
    dev = base.device
    p = _params(C, L, K, W, B, beta)
    ws = ws if ws is not None else new_workspace(workspace_bytes(C, L, K, W, B, beta, V, H, head.dtype), dev)
    t = _alloc_tree(C, B, dev)
    ts = _tree_struct(t)
    st_p = cand_p = None
    if keep_intermediates:
        st = _alloc_supertree(C, L, W, dev)
        t["st"] = st
        t["cand_tok"] = torch.empty((C, L, K), dtype=torch.int32, device=dev)
        t["cand_val"] = torch.empty((C, L, K), dtype=torch.float32, device=dev)
        st_p = ctypes.byref(_st_struct(st))
        cand_p = ctypes.byref(Candidates(t["cand_tok"].data_ptr(), t["cand_val"].data_ptr()))
    _call("dartree_build_tree", ctypes.byref(head), ctypes.byref(p), ctypes.c_void_p(base.data_ptr()),
          ctypes.c_void_p(hidden.data_ptr()), ctypes.c_void_p(anchor.data_ptr()), ctypes.byref(ts), st_p, cand_p,
          ctypes.c_void_p(ws.data_ptr()), ws.numel(), _stream(stream))
    _keep(stream, ws, wqt)
    return t


class Round:
    """One draft round (build + verify) with every buffer allocated once.

    run() enqueues dartree_build_tree and dartree_verify on the current stream and
    allocates nothing, so it can be timed, repeated or captured in a CUDA graph.
    """

    def __init__(self, E, Wq, C, L, K, W, B, beta, rows, device=None):
        self.E, self.Wq = E, Wq
        self.V, self.H = E.shape
        self.C, self.L, self.K, self.W, self.B, self.beta, self.rows = C, L, K, W, B, beta, rows
        dev = device or E.device
        self.head, self.wqt = _head(E, Wq, prepare=True)
        self.p = _params(C, L, K, W, B, beta)
        self.ws = new_workspace(workspace_bytes(C, L, K, W, B, beta, self.V, self.H, self.head.dtype), dev)
        self.tree = _alloc_tree(C, B, dev)
        self._ts = _tree_struct(self.tree)
        self.out = dict(accepted_len=torch.empty((C,), dtype=torch.int32, device=dev),
                        path=torch.empty((C, L), dtype=torch.int32, device=dev),
                        bonus=torch.empty((C,), dtype=torch.int32, device=dev))
        self.dtype_code = self.head.dtype

    def run(self, base, hidden, anchor, target, stream=None):
        """dartree_round: build + verify in one call."""
        _call("dartree_round", ctypes.byref(self.head), ctypes.byref(self.p), ctypes.c_void_p(base.data_ptr()),
              ctypes.c_void_p(hidden.data_ptr()), ctypes.c_void_p(anchor.data_ptr()),
              ctypes.c_void_p(target.data_ptr()), int(self.rows), ctypes.byref(self._ts),
              ctypes.c_void_p(self.out["accepted_len"].data_ptr()), ctypes.c_void_p(self.out["path"].data_ptr()),
              ctypes.c_void_p(self.out["bonus"].data_ptr()), ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(),
              _stream(stream))
        return self.out

    def run_two_calls(self, base, hidden, anchor, target, stream=None):
        """The same round as dartree_build_tree followed by dartree_verify."""
        s = _stream(stream)
        _call("dartree_build_tree", ctypes.byref(self.head), ctypes.byref(self.p), ctypes.c_void_p(base.data_ptr()),
              ctypes.c_void_p(hidden.data_ptr()), ctypes.c_void_p(anchor.data_ptr()), ctypes.byref(self._ts), None,
              None, ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(), s)
        _call("dartree_verify", ctypes.byref(self.p), ctypes.byref(self._ts), ctypes.c_void_p(target.data_ptr()),
              int(self.rows), int(self.V), int(self.dtype_code), ctypes.c_void_p(self.out["accepted_len"].data_ptr()),
              ctypes.c_void_p(self.out["path"].data_ptr()), ctypes.c_void_p(self.out["bonus"].data_ptr()),
              ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(), s)
        return self.out


class HostInputs(ctypes.Structure):
    _fields_ = [("base_logits", ctypes.c_void_p), ("block_hidden", ctypes.c_void_p), ("anchor", ctypes.c_void_p),
                ("target", ctypes.c_void_p)]


class HostOutputs(ctypes.Structure):
    _fields_ = [("accepted_len", ctypes.c_void_p), ("path", ctypes.c_void_p), ("bonus", ctypes.c_void_p)]


class HostRounds:
    """Rounds fed from host buffers through the library's host session
    (dartree_host_session_create / dartree_host_stage / dartree_host_round): the
    session holds two device sets of the inputs, and round i runs from set i % 2
    while round i + 1's inputs are copied into the other set on the session's copy
    stream. Each round's results are copied into the caller's host buffers on the
    current stream right after the round, complete once that stream is synchronised.
    Host tensors should be pinned for the copies to overlap the rounds.
    """

    KEYS = ("base", "hidden", "anchor", "target")

    def __init__(self, rnd: "Round", like: dict = None):
        self.rnd = rnd
        h = ctypes.c_void_p()
        _call("dartree_host_session_create", ctypes.byref(rnd.head), ctypes.byref(rnd.p), int(rnd.rows),
              ctypes.byref(h))
        self._s = h
        self._keep = []  # host tensors of the rounds in flight

    def __del__(self):
        s = getattr(self, "_s", None)
        if s is not None and s.value and _LIB is not None:
            _LIB.dartree_host_session_destroy(s)
            self._s = None

    def h2d_bytes(self) -> int:
        return sum(int(lib().dartree_host_input_bytes(self._s, k)) for k in range(4))

    @staticmethod
    def _host(t: torch.Tensor, name: str) -> int:
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host tensor")
        return t.data_ptr()

    def copy_in(self, i: int, host: dict):
        """Stage round i's inputs (host tensors, pinned for overlap): dartree_host_stage."""
        x = HostInputs(*(self._host(host[k], k) for k in self.KEYS))
        _call("dartree_host_stage", self._s, ctypes.byref(x))
        self._keep = (self._keep + [host])[-2:]

    def run(self, i: int, host_out: dict, stream=None):
        """Round i on the current stream from its staged inputs, results into host_out
        (host int32 tensors shaped like Round.out): dartree_host_round."""
        o = HostOutputs(*(self._host(host_out[k], k) for k in ("accepted_len", "path", "bonus")))
        _call("dartree_host_round", self._s, ctypes.byref(o), _stream(stream))
        return host_out


class HeapRound:
    """Node-by-node best-first drafting (one head evaluation per popped node), the
    baseline the deferred search replaces; every buffer allocated once, run()
    allocates nothing (it can be timed or captured in a CUDA graph)."""

    def __init__(self, E, Wq, C, L, K, B, beta, device=None):
        self.V, self.H = E.shape
        self.C, self.L, self.K, self.B, self.beta = C, L, K, B, beta
        dev = device or E.device
        self.head, self.wqt = _head(E, Wq, prepare=True)
        self.p = _params(C, L, K, 1, B, beta)
        n = lib().dartree_heap_workspace_bytes(ctypes.byref(self.p), int(self.V), int(self.H), int(self.head.dtype))
        if n == 0:
            raise DartreeError(EUNSUPPORTED, "dartree_heap_workspace_bytes")
        self.ws = new_workspace(n, dev)
        self.out = dict(tok=torch.empty((C, B), dtype=torch.int32, device=dev),
                        parent=torch.empty((C, B), dtype=torch.int32, device=dev),
                        depth=torch.empty((C, B), dtype=torch.int32, device=dev),
                        score=torch.empty((C, B), dtype=torch.float32, device=dev))

    def run(self, base, hidden, anchor, stream=None):
        o = self.out
        _call("dartree_heap_build", ctypes.byref(self.head), ctypes.byref(self.p), ctypes.c_void_p(base.data_ptr()),
              ctypes.c_void_p(hidden.data_ptr()), ctypes.c_void_p(anchor.data_ptr()),
              ctypes.c_void_p(o["tok"].data_ptr()), ctypes.c_void_p(o["parent"].data_ptr()),
              ctypes.c_void_p(o["depth"].data_ptr()), ctypes.c_void_p(o["score"].data_ptr()),
              ctypes.c_void_p(self.ws.data_ptr()), self.ws.numel(), _stream(stream))
        return o


def heap_build(E, Wq, base, hidden, anchor, K, B, beta, stream=None):
    """dartree_heap_build on fresh buffers -> dict(tok, parent, depth, score) [C, B] in pop order."""
    C, L, _ = base.shape
    h = HeapRound(E, Wq, C, L, K, B, beta, device=base.device)
    out = h.run(base, hidden, anchor, stream)
    _keep(stream, h.ws, h.wqt)
    out["_keep"] = (h.ws, h.wqt)
    return out
