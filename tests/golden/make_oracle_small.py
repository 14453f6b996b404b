"""Writes oracle_small.json: the oracle's outputs on small seeded cases, kept
as a regression fixture (a change to the oracle's arithmetic shows up as a
diff here, and its commit names the passage that justifies it).  Calls only
oracle/ and the input generator.  Floats are stored as exact hex strings.

    python tests/golden/make_oracle_small.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
import oracle  # noqa: E402
import synth  # noqa: E402


def fhex(a):
    return [float(v).hex() for v in np.asarray(a, dtype=np.float64).ravel()]


def cases():
    orc = oracle.get()
    out = {}
    x = synth.gen_x(3, 512, 41, outlier_frac=0.01)
    qs, d, bs = orc.quantize_q8k(x)
    out["quantize_q8k"] = {"x_seed": 41, "M": 3, "K": 512, "qs": qs.ravel().tolist(), "d": fhex(d),
                           "bsums": bs.ravel().tolist()}
    for wtype, N, K, seed in ((4, 5, 512, 42), (6, 4, 512, 43), (1, 3, 256, 44)):
        gen = {4: synth.gen_q4k, 6: synth.gen_q6k, 1: synth.gen_ptq1}[wtype]
        w = gen(N, K, seed)
        xq = orc.quantize_q8k(synth.gen_x(2, K, seed + 100))
        y, absc = orc.gemm(wtype, w, K, *xq)
        out[f"gemm_w{wtype}"] = {"N": N, "K": K, "w_seed": seed, "x_seed": seed + 100, "M": 2, "y": fhex(y),
                                 "absc": fhex(absc)}
    E, N, K, M, top_k = 3, 4, 256, 4, 2
    w = synth.gen_q4k(E * N, K, 45)
    xq = orc.quantize_q8k(synth.gen_x(M, K, 46))
    ids = synth.gen_ids(M, top_k, E, 47)
    y, _ = orc.gemm_id(4, w, E, K, *xq, ids)
    out["gemm_id_w4"] = {"E": E, "N": N, "K": K, "M": M, "top_k": top_k, "seeds": [45, 46, 47], "y": fhex(y)}
    v = np.array([[-3.0, -0.5, 0.0, 0.25, 1.0, 2.5]])
    out["epilogue"] = {"v": fhex(v), "relu": fhex(orc.epilogue(v, act=1)), "silu": fhex(orc.epilogue(v, act=2)),
                       "gelu": fhex(orc.epilogue(v, act=3))}
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(cases(), f, indent=0, sort_keys=True)
        f.write("\n")
    print("wrote", os.path.join(HERE, "oracle_small.json"))
