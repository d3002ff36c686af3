"""Small hand-made and random inputs for the oracle pins (no method arithmetic)."""
import json
import os

import numpy as np

from dartree_inputs import Config, make_config, make_inputs, round_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def golden_inputs(g, dtype):
    c = g["config"]
    cfg = Config("golden", C=c["C"], L=c["L"], V=c["V"], H=c["H"], K=c["K"], W=c["W"],
                 B=c["B"], beta=c["beta"], dtype=dtype, seed=0, rows=c["rows"], sigma=0.0,
                 plant="single8", target="plant", agree_p=0.0)

    def st(a):
        a = np.asarray(a, dtype=np.float32)
        return round_to_bf16_bits(a) if dtype == "bf16" else a

    gi = g["inputs"]
    return dict(cfg=cfg, requests=np.arange(c["C"]), anchor=np.asarray(gi["anchor"], np.int32),
                base=st(gi["base"]), hidden=st(gi["hidden"]), E=st(gi["E"]), Wq=st(gi["Wq"]),
                target=st(gi["target"]))


def tiny_config(seed, L=4, V=16, H=8, K=3, W=3, B=6, beta=-0.1, dtype="f32", C=1, rows="position"):
    return make_config("cfg0_tiny").replace(name="tiny", C=C, L=L, V=V, H=H, K=K, W=W, B=B,
                                            beta=beta, dtype=dtype, seed=seed, rows=rows)


def tiny_inputs(seed, ties=False, **kw):
    cfg = tiny_config(seed, **kw)
    inp = make_inputs(cfg)
    if ties:
        # coarse base logits and a zero head make many exact score ties
        b = np.round(np.asarray(inp["base"], np.float32) / 4.0)
        inp["base"] = b.astype(np.float32) if cfg.dtype == "f32" else round_to_bf16_bits(b)
        inp["E"] = np.zeros_like(inp["E"])
    return inp
