"""Writes tests/golden/tiny_kda.json from the fp64 oracle (nothing else is called).

The pages print no worked numeric example for the KDA layer, so this file is a regression anchor for
the oracle and the input generator, not an external pin: the tiny configuration (one sequence, H=2,
dk=dv=16, conv width 4, 64-token prefill from a zero state with checkpoints every 32 tokens, then 8
decode steps).  Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import kda_inputs as ki  # noqa: E402
import oracle  # noqa: E402

SEED, H, D, W, T, STEPS, INTERVAL = 1, 2, 16, 4, 64, 8, 32


def compute():
    cfg = oracle.Cfg(H=H, dk=D, dv=D, W=W)
    wts = ki.layer_weights(SEED, H, D, D, W)
    tok = ki.token_inputs(SEED, T + STEPS, H, D, D)
    f = {k: (ki.bf16_bits_to_f64(v) if v is not None else None) for k, v in tok.items()}
    pre = oracle.forward(cfg, [0, T], [0], f["q"][:T], f["k"][:T], f["v"][:T], f["a"][:T], f["b"][:T],
                         f["z"][:T], wts["conv_w"], wts["norm_w"], np.zeros((1, H, D, D)),
                         np.zeros((1, H, W - 1, 3 * D)), interval=INTERVAL)
    S, C = pre["S"], pre["conv"]
    ys = []
    for s in range(STEPS):
        t = T + s
        r = oracle.forward(cfg, [0, 1], [t], f["q"][t:t + 1], f["k"][t:t + 1], f["v"][t:t + 1], f["a"][t:t + 1],
                           f["b"][t:t + 1], f["z"][t:t + 1], wts["conv_w"], wts["norm_w"], S, C)
        S, C = r["S"], r["conv"]
        ys.append(r["y"][0])
    return dict(prefill_y_last4=pre["y"][-4:], ckpt_pos=pre["ckpt_pos"], ckpt_S=pre["ckpt_S"],
                decode_y=np.array(ys), final_S=S)


if __name__ == "__main__":
    out = {k: np.asarray(v).tolist() for k, v in compute().items()}
    out["_about"] = __doc__.strip().splitlines()[0]
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_kda.json"), "w") as fh:
        json.dump(out, fh, separators=(",", ":"))
