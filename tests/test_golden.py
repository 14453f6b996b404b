"""Golden fixtures under tests/golden/.

- page_values.txt: block facts the source pages print, checked against the
  oracle's byte layouts (the Q8_K interop block and the PTQ1_0 block).
- oracle_small.json: the oracle's outputs on small seeded cases, written by
  tests/golden/make_oracle_small.py, which calls only oracle/ and synth.  A
  change to the oracle's arithmetic shows up here.  Q8_K and the GEMM sums are
  compared bit for bit: integer work, and fp64 compiled without contraction.
  The activations go through libm's exp/erf and are compared to 1e-15 relative,
  since another platform's libm may round differently."""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def page_values():
    vals = {}
    with open(os.path.join(GOLDEN, "page_values.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, value = line.split("|")[0].split()
                vals[name] = int(value)
    return vals


def test_q8k_block_is_the_pages_size():
    v = page_values()
    orc = oracle.get()
    K = 2 * v["q8k_block_elements"]
    qs, d, bs = orc.quantize_q8k(synth.gen_x(2, K, 3))
    aos = orc.q8k_to_aos(qs, d, bs)
    assert aos.shape[1] == 2 * v["q8k_block_bytes"]
    # one block: fp32 d, the 256 codes, the 16 int16 sums -- 4 + 256 + 32 bytes
    blk = aos[1, v["q8k_block_bytes"]:]
    assert blk[:4].tobytes() == d[1, 1].tobytes()
    assert np.array_equal(blk[4:260].view(np.int8), qs[1, 256:])
    assert np.array_equal(blk[260:292].view(np.int16), bs[1, 16:])
    back = orc.q8k_from_aos(aos, 2, K)
    assert all(np.array_equal(a, b) for a, b in zip(back, (qs, d, bs)))


def test_ptq1_block_is_the_pages_size():
    v = page_values()
    orc = oracle.get()
    t = np.random.default_rng(5).integers(0, 3, v["ptq1_block_weights"]).astype(np.int32)
    blk = orc.ptq1_pack(0x3C00, t)                       # d = 1.0
    assert blk.size == v["ptq1_block_bytes"]
    d, back = orc.ptq1_fields(blk)
    assert d == 1.0 and np.array_equal(back, t)
    # five ternary digits per qs byte: every byte value of the 24 qs bytes is below 3^5
    assert v["ptq1_trits_per_byte"] == 5 and blk[:24].max() < 3 ** 5
    assert 24 * v["ptq1_trits_per_byte"] + 2 * 4 == v["ptq1_block_weights"]   # + 4 digits in each qh byte


def unhex(a):
    return np.array([float.fromhex(s) for s in a])


@pytest.fixture(scope="module")
def golden():
    with open(os.path.join(GOLDEN, "oracle_small.json")) as f:
        return json.load(f)


def test_oracle_quantize_matches_golden(golden):
    g = golden["quantize_q8k"]
    qs, d, bs = oracle.get().quantize_q8k(synth.gen_x(g["M"], g["K"], g["x_seed"], outlier_frac=0.01))
    assert qs.ravel().tolist() == g["qs"] and bs.ravel().tolist() == g["bsums"]
    assert np.array_equal(d.astype(np.float64).ravel(), unhex(g["d"]))


@pytest.mark.parametrize("wtype", [4, 6, 1])
def test_oracle_gemm_matches_golden(golden, wtype):
    g = golden[f"gemm_w{wtype}"]
    orc = oracle.get()
    gen = {4: synth.gen_q4k, 6: synth.gen_q6k, 1: synth.gen_ptq1}[wtype]
    w = gen(g["N"], g["K"], g["w_seed"])
    y, absc = orc.gemm(wtype, w, g["K"], *orc.quantize_q8k(synth.gen_x(g["M"], g["K"], g["x_seed"])))
    assert np.array_equal(y.ravel(), unhex(g["y"])) and np.array_equal(absc.ravel(), unhex(g["absc"]))


def test_oracle_gemm_id_matches_golden(golden):
    g = golden["gemm_id_w4"]
    orc = oracle.get()
    sw, sx, si = g["seeds"]
    w = synth.gen_q4k(g["E"] * g["N"], g["K"], sw)
    xq = orc.quantize_q8k(synth.gen_x(g["M"], g["K"], sx))
    y, _ = orc.gemm_id(4, w, g["E"], g["K"], *xq, synth.gen_ids(g["M"], g["top_k"], g["E"], si))
    assert np.array_equal(y.ravel(), unhex(g["y"]))


def test_oracle_epilogue_matches_golden(golden):
    g = golden["epilogue"]
    orc = oracle.get()
    v = unhex(g["v"]).reshape(1, -1)
    for act, key in ((1, "relu"), (2, "silu"), (3, "gelu")):
        got = orc.epilogue(v, act=act).ravel()
        assert np.allclose(got, unhex(g[key]), rtol=1e-15, atol=0.0), key
