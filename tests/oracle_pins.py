"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each check takes an ``oracle.Oracle`` and raises AssertionError on a mismatch.
The same checks run against the real oracle (test_oracle_pins.py) and against
deliberately broken builds of it (test_oracle_mutations.py), which shows that
each planted mistake is caught by at least one pin.

What pins what:
  * fp16 decode            -> numpy's float16 conversion, all 65536 patterns
  * Q4_K / Q6_K unpack     -> hand-derived byte/bit cases from the format
                              statement; pack/unpack round trips
  * dequantize             -> the format formulas on hand-built blocks with
                              fp16-exact d, dmin
  * Q8_K quantizer         -> |x - d*q| <= d/2 bound, amax -> +-127, the tie
                              cases of round-half-away, amax = 0, bsums = sums,
                              d equal to numpy's correctly rounded fp32 amax/127
  * GEMM (block-integer)   -> fp64 brute force on tiny shapes; hand-built
                              single-superblock cases that reduce to a plain
                              integer dot product (numpy) or to the dmin term
"""
from __future__ import annotations

import numpy as np

import synth

F16_ONE = 0x3C00     # 1.0
F16_HALF = 0x3800    # 0.5
F16_ZERO = 0x0000


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ fp16 --
def check_half_decode(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    # sample every pattern through the C decoder (cheap: 65536 ctypes calls)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "NaN patterns differ"
    assert np.array_equal(got[~nan], ref[~nan]), "fp16 decode differs from numpy"


# ------------------------------------------------------------------ Q4_K --
def check_q4k_scale_bytes_hand(orc):
    """Hand-derived from the 12-byte scale packing: j<4 low 6 bits; j>=4 low
    nibble/high nibble of bytes 8..11 plus the top 2 bits of bytes 0..7."""
    blk = np.zeros(144, np.uint8)
    blk[4:16] = [1, 2, 3, 4, 5, 6, 7, 8, 0x21, 0x43, 0x65, 0x87]
    _, _, sc, mn, _ = orc.q4k_fields(blk)
    assert list(sc) == [1, 2, 3, 4, 1, 3, 5, 7], sc
    assert list(mn) == [5, 6, 7, 8, 2, 4, 6, 8], mn
    # top bits: byte 0 = 0xC1 -> sc_0 = 1 and bits 4..5 of sc_4 = 3;
    # byte 5 = 0x80|6 -> m_1 = 6 and bits 4..5 of m_5 = 2
    blk[4] = 0xC1
    blk[9] = 0x86
    _, _, sc, mn, _ = orc.q4k_fields(blk)
    assert sc[0] == 1 and sc[4] == 1 + 48, sc
    assert mn[1] == 6 and mn[5] == 4 + 32, mn


def check_q4k_header_bytes_hand(orc):
    """The block header, written byte by byte (no pack function): fp16 d in
    bytes 0-1 and fp16 dmin in bytes 2-3, little-endian."""
    blk = np.zeros(144, np.uint8)
    blk[0:4] = [0x00, 0x3C, 0x00, 0x40]          # d = 1.0 (0x3C00), dmin = 2.0 (0x4000)
    d, dmin, _, _, _ = orc.q4k_fields(blk)
    assert (d, dmin) == (1.0, 2.0), (d, dmin)
    blk[0:4] = [0x00, 0x38, 0x00, 0x3C]          # d = 0.5, dmin = 1.0
    blk[4] = 3                                   # sc_0 = 3
    blk[8] = 5                                   # m_0 = 5
    blk[16] = 0x07                               # q_0 = 7, q_32 = 0
    d, dmin, _, _, _ = orc.q4k_fields(blk)
    assert (d, dmin) == (0.5, 1.0), (d, dmin)
    w = orc.dequant(4, blk)
    assert w[0] == 0.5 * 3 * 7 - 1.0 * 5, w[0]   # d * sc_0 * q_0 - dmin * m_0
    assert w[1] == -5.0, w[1]                    # q_1 = 0
    # the packer writes the same bytes
    sc = np.zeros(8, int); mn = np.zeros(8, int); q = np.zeros(256, int)
    sc[0], mn[0], q[0] = 3, 5, 7
    assert np.array_equal(orc.q4k_pack(0x3800, 0x3C00, sc, mn, q), blk)


def check_q4k_nibble_bytes_hand(orc):
    """qs byte 32c+l: low nibble = weight 64c+l, high nibble = weight 64c+32+l."""
    blk = np.zeros(144, np.uint8)
    for c in range(4):
        for l in range(32):
            lo = (c * 5 + l) % 16
            hi = (c * 3 + 2 * l + 1) % 16
            blk[16 + 32 * c + l] = lo | (hi << 4)
    _, _, _, _, q = orc.q4k_fields(blk)
    for c in range(4):
        for l in range(32):
            assert q[64 * c + l] == (c * 5 + l) % 16
            assert q[64 * c + 32 + l] == (c * 3 + 2 * l + 1) % 16


def check_q4k_roundtrip(orc):
    r = _rng(11)
    for t in range(300):
        sc = r.integers(0, 64, 8); mn = r.integers(0, 64, 8); q = r.integers(0, 16, 256)
        blk = orc.q4k_pack(F16_ONE, F16_HALF, sc, mn, q)
        d, dmin, sc2, mn2, q2 = orc.q4k_fields(blk)
        assert d == 1.0 and dmin == 0.5
        assert np.array_equal(sc, sc2) and np.array_equal(mn, mn2) and np.array_equal(q, q2)
    # every 6-bit value in every position
    for v in range(64):
        for j in range(8):
            sc = np.zeros(8, int); mn = np.full(8, 63 - v)
            sc[j] = v
            blk = orc.q4k_pack(F16_ONE, F16_ONE, sc, mn, np.zeros(256, int))
            _, _, sc2, mn2, _ = orc.q4k_fields(blk)
            assert np.array_equal(sc2, sc) and np.array_equal(mn2, mn)
    # random bytes decode to in-range fields and re-pack to the same bytes
    for t in range(200):
        blk = r.integers(0, 256, 144).astype(np.uint8)
        d, dmin, sc, mn, q = orc.q4k_fields(blk)
        assert sc.min() >= 0 and sc.max() < 64 and mn.max() < 64 and q.max() < 16
        again = orc.q4k_pack(int(blk[0]) | int(blk[1]) << 8, int(blk[2]) | int(blk[3]) << 8, sc, mn, q)
        assert np.array_equal(again, blk)


def check_q4k_dequant_hand(orc):
    """w = d*sc_j*q - dmin*m_j with d = 1.0, dmin = 0.5 (fp16 exact)."""
    sc = np.arange(8) * 7 + 1          # 1, 8, ..., 50
    mn = 63 - np.arange(8) * 5         # 63, 58, ...
    q = (np.arange(256) * 7) % 16
    blk = orc.q4k_pack(F16_ONE, F16_HALF, sc, mn, q)
    w = orc.dequant(4, blk)
    j = np.arange(256) // 32
    assert np.array_equal(w, 1.0 * sc[j] * q - 0.5 * mn[j])


# ------------------------------------------------------------------ Q6_K --
def check_q6k_bytes_hand(orc):
    """Single-bit probes of the ql/qh split (format statement, both halves)."""
    for h in range(2):
        for l in (0, 5, 31):
            for part in range(4):
                blk = np.zeros(210, np.uint8)
                L = 64 * h + l + (32 if part in (1, 3) else 0)
                nib_hi = part in (2, 3)
                blk[L] = (9 << 4) if nib_hi else 9            # low 4 bits = 9
                blk[128 + 32 * h + l] = 2 << (2 * part)        # high 2 bits = 2
                _, _, q = orc.q6k_fields(blk)
                i = 128 * h + l + 32 * part
                expect = np.zeros(256, int)
                expect[i] = 9 | (2 << 4)
                assert np.array_equal(q, expect), (h, l, part)
    blk = np.zeros(210, np.uint8)
    blk[192:208] = np.arange(-8, 8).astype(np.int8).view(np.uint8)
    blk[208:210] = [0x00, 0x3C]
    d, sc, _ = orc.q6k_fields(blk)
    assert d == 1.0 and list(sc) == list(range(-8, 8))


def check_q6k_roundtrip(orc):
    r = _rng(12)
    for t in range(300):
        sc = r.integers(-128, 128, 16); q = r.integers(0, 64, 256)
        blk = orc.q6k_pack(F16_HALF, sc, q)
        d, sc2, q2 = orc.q6k_fields(blk)
        assert d == 0.5 and np.array_equal(sc, sc2) and np.array_equal(q, q2)
    for t in range(200):
        blk = r.integers(0, 256, 210).astype(np.uint8)
        d, sc, q = orc.q6k_fields(blk)
        assert q.min() >= 0 and q.max() < 64
        again = orc.q6k_pack(int(blk[208]) | int(blk[209]) << 8, sc, q)
        assert np.array_equal(again, blk)


def check_q6k_dequant_hand(orc):
    sc = np.arange(16) - 8
    q = (np.arange(256) * 5) % 64
    blk = orc.q6k_pack(F16_HALF, sc, q)
    w = orc.dequant(6, blk)
    assert np.array_equal(w, 0.5 * sc[np.arange(256) // 16] * (q - 32))


# ------------------------------------------------------------------ Q8_K --
def _adversarial_rows(K=512):
    r = _rng(13)
    rows = [r.standard_normal(K).astype(np.float32),
            (r.standard_normal(K) * 1e-30).astype(np.float32),
            (r.standard_normal(K) * 1e-41).astype(np.float32),           # subnormal x
            (r.standard_normal(K) * 3e4).astype(np.float32),
            np.zeros(K, np.float32),
            np.concatenate([np.zeros(256, np.float32), r.standard_normal(K - 256).astype(np.float32)]),
            r.integers(-127, 128, K).astype(np.float32),
            (r.integers(-254, 255, K) * 0.5).astype(np.float32)]
    spiky = r.standard_normal(K).astype(np.float32)
    spiky[::37] *= 200.0
    rows.append(spiky)
    # amax/127 underflows to zero in fp32 (smallest subnormals): quantizes to zero
    tiny = np.zeros(K, np.float32)
    tiny[:4] = [1e-45, -1e-45, 1e-45, 0.0]
    tiny[256:258] = [-2.8e-45, 1.4e-45]
    rows.append(tiny)
    return np.stack(rows)


def check_q8k_bound_and_extremes(orc):
    x = _adversarial_rows()
    qs, d, bs = orc.quantize_q8k(x)
    M, K = x.shape
    for m in range(M):
        for b in range(K // 256):
            xb = x[m, 256 * b:256 * b + 256].astype(np.float64)
            qb = qs[m, 256 * b:256 * b + 256].astype(np.int64)
            amax = np.float32(np.abs(x[m, 256 * b:256 * b + 256]).max())
            db = d[m, b]
            assert db == np.float32(amax) / np.float32(127.0), "d is not fp32 amax/127"
            if db == 0:
                assert not qb.any() and not bs[m, 16 * b:16 * b + 16].any()
                continue
            # |x - d q| <= d/2, allowing the fp32 rounding of x/d (relative 2^-23 of |x/d| <= 127)
            err = np.abs(xb - float(db) * qb)
            assert np.all(err <= float(db) * (0.5 + 127 * 2.0 ** -23)), err.max() / db
            imax = np.argmax(np.abs(xb))
            assert abs(qb[imax]) == 127 and np.sign(qb[imax]) == np.sign(xb[imax])
            assert np.abs(qb).max() <= 127


def check_q8k_ties(orc):
    """amax = 127 makes d = 1 exactly; x = +-2.5 -> +-3, +-0.5 -> +-1, +-1.5 -> +-2."""
    x = np.zeros((1, 256), np.float32)
    x[0, :8] = [127.0, 2.5, -2.5, 0.5, -0.5, 1.5, -1.5, -127.0]
    x[0, 8:12] = [3.5, -3.5, 0.49999997, -0.49999997]
    qs, d, bs = orc.quantize_q8k(x)
    assert d[0, 0] == 1.0
    assert list(qs[0, :12]) == [127, 3, -3, 1, -1, 2, -2, -127, 4, -4, 0, 0]


def check_q8k_bsums(orc):
    x = synth.gen_x(5, 1024, 77)
    qs, d, bs = orc.quantize_q8k(x)
    ref = qs.astype(np.int64).reshape(5, 64, 16).sum(axis=2)
    assert np.array_equal(bs.astype(np.int64), ref)


def check_q8k_matches_numpy_rounding(orc):
    """q equals round-half-away(fp32(x)/fp32(d)), the division done by numpy."""
    x = np.concatenate([_adversarial_rows(), synth.gen_x(4, 512, 5, outlier_frac=0.01)])
    qs, d, bs = orc.quantize_q8k(x)
    M, K = x.shape
    for m in range(M):
        for b in range(K // 256):
            db = d[m, b]
            if db == 0:
                continue
            v = (x[m, 256 * b:256 * b + 256] / np.float32(db)).astype(np.float64)
            ref = np.clip(np.sign(v) * np.floor(np.abs(v) + 0.5), -127, 127)
            assert np.array_equal(qs[m, 256 * b:256 * b + 256].astype(np.float64), ref)


def check_q8k_aos_roundtrip(orc):
    x = synth.gen_x(3, 768, 9)
    qs, d, bs = orc.quantize_q8k(x)
    aos = orc.q8k_to_aos(qs, d, bs)
    assert aos.shape == (3, 3 * 292)
    # field placement: d at 0, qs at 4, bsums at 260 of each 292-byte block
    assert aos[1, 292:296].view(np.float32)[0] == d[1, 1]
    assert np.array_equal(aos[2, 4:260].view(np.int8), qs[2, :256])
    assert np.array_equal(aos[0, 2 * 292 + 260:2 * 292 + 292].view(np.int16), bs[0, 32:48])
    qs2, d2, bs2 = orc.q8k_from_aos(aos, 3, 768)
    assert np.array_equal(qs, qs2) and np.array_equal(d, d2) and np.array_equal(bs, bs2)


# ------------------------------------------------------------------ GEMM --
def _q8k_direct(r, M, K, dvals=None):
    """A Q8_K operand built directly (not through the quantizer)."""
    qs = r.integers(-127, 128, (M, K)).astype(np.int8)
    d = (np.ones((M, K // 256), np.float32) if dvals is None else dvals.astype(np.float32))
    bs = qs.astype(np.int64).reshape(M, K // 16, 16).sum(axis=2).astype(np.int16)
    return qs, d, bs


def check_gemm_vs_brute(orc):
    r = _rng(14)
    for wtype in (4, 6):
        for (M, N, K) in ((1, 1, 256), (2, 3, 256), (3, 5, 512), (5, 2, 512), (5, 5, 256)):
            w = (synth.gen_q4k if wtype == 4 else synth.gen_q6k)(N, K, int(r.integers(1 << 30)))
            x = synth.gen_x(M, K, int(r.integers(1 << 30)), outlier_frac=0.01)
            qs, d, bs = orc.quantize_q8k(x)
            y, absc = orc.gemm(wtype, w, K, qs, d, bs)
            yb = orc.brute(wtype, w, K, qs, d)
            assert np.all(np.abs(y - yb) <= 1e-12 * absc + 1e-300), (wtype, M, N, K)


def check_gemm_unit_scales_q4k(orc):
    """sc_j = 1, dmin = 0, d = 1, dx = 1: Y = plain integer dot sum_i q_i * qx_i."""
    r = _rng(15)
    N, K, M = 3, 512, 4
    blocks = []
    for n in range(N):
        row = []
        for b in range(K // 256):
            q = r.integers(0, 16, 256)
            row.append((q, orc.q4k_pack(F16_ONE, F16_ZERO, np.ones(8, int), r.integers(0, 64, 8), q)))
        blocks.append(row)
    w = np.stack([np.concatenate([blk for _, blk in row]) for row in blocks])
    qfull = np.stack([np.concatenate([q for q, _ in row]) for row in blocks])
    qs, d, bs = _q8k_direct(r, M, K)
    y, _ = orc.gemm(4, w, K, qs, d, bs)
    ref = qs.astype(np.int64) @ qfull.T.astype(np.int64)
    assert np.array_equal(y, ref.astype(np.float64))


def check_gemm_zero_quants_q4k(orc):
    """All q = 0: c_b = -dx * dmin * sum_j m_j * (bsums[2j] + bsums[2j+1])."""
    r = _rng(16)
    K, M = 256, 3
    mn = r.integers(0, 64, 8)
    w = orc.q4k_pack(F16_ONE, F16_HALF, r.integers(0, 64, 8), mn, np.zeros(256, int))[None, :]
    dx = np.array([[0.25], [1.0], [2.0]], np.float32)
    qs, d, bs = _q8k_direct(r, M, K, dx)
    y, _ = orc.gemm(4, w, K, qs, d, bs)
    bs32 = qs.astype(np.int64).reshape(M, 8, 32).sum(axis=2)      # per sub-block sums
    ref = -dx[:, 0].astype(np.float64) * 0.5 * (bs32 @ mn)
    assert np.array_equal(y[:, 0], ref)


def check_gemm_subblock_scales_q4k(orc):
    """q = 1 everywhere, dmin = 0: Y = sum_j sc_j * (sum of qx over sub-block j)."""
    r = _rng(17)
    K, M = 256, 2
    sc = np.array([1, 2, 4, 8, 16, 32, 63, 5])
    w = orc.q4k_pack(F16_ONE, F16_ZERO, sc, r.integers(0, 64, 8), np.ones(256, int))[None, :]
    qs, d, bs = _q8k_direct(r, M, K)
    y, _ = orc.gemm(4, w, K, qs, d, bs)
    ref = qs.astype(np.int64).reshape(M, 8, 32).sum(axis=2) @ sc
    assert np.array_equal(y[:, 0], ref.astype(np.float64))


def check_gemm_q6k_offset(orc):
    """All q = 32 -> Y = 0; sc = 1, d = 1 -> Y = sum_i (q_i - 32) * qx_i."""
    r = _rng(18)
    K, M = 512, 3
    qs, d, bs = _q8k_direct(r, M, K)
    blk = orc.q6k_pack(F16_ONE, r.integers(-32, 32, 16), np.full(256, 32))
    w = np.concatenate([blk, blk])[None, :]
    y, _ = orc.gemm(6, w, K, qs, d, bs)
    assert np.all(y == 0.0)
    q = r.integers(0, 64, (2, 256))
    w = np.concatenate([orc.q6k_pack(F16_ONE, np.ones(16, int), q[0]),
                        orc.q6k_pack(F16_ONE, np.ones(16, int), q[1])])[None, :]
    y, _ = orc.gemm(6, w, K, qs, d, bs)
    ref = qs.astype(np.int64) @ (q.reshape(-1) - 32)
    assert np.array_equal(y[:, 0], ref.astype(np.float64))


def check_gemm_q6k_subblock_scales(orc):
    """q = 33 (q-32 = 1), d = 1: Y = sum_j sc_j * (sum of qx over sub-block j of 16)."""
    r = _rng(19)
    K, M = 256, 2
    sc = np.arange(16) * 3 - 20
    w = orc.q6k_pack(F16_ONE, sc, np.full(256, 33))[None, :]
    qs, d, bs = _q8k_direct(r, M, K)
    y, _ = orc.gemm(6, w, K, qs, d, bs)
    ref = qs.astype(np.int64).reshape(M, 16, 16).sum(axis=2) @ sc
    assert np.array_equal(y[:, 0], ref.astype(np.float64))


def check_gemm_rows_subset(orc):
    """Evaluating a subset of token rows gives the same values as the full run."""
    r = _rng(20)
    w = synth.gen_q4k(7, 512, 21)
    qs, d, bs = orc.quantize_q8k(synth.gen_x(9, 512, 22))
    y, a = orc.gemm(4, w, 512, qs, d, bs)
    rows = np.array([8, 0, 3])
    y2, a2 = orc.gemm(4, w, 512, qs, d, bs, rows=rows)
    assert np.array_equal(y[rows], y2) and np.array_equal(a[rows], a2)


def check_gemm_id_vs_brute(orc):
    """Routed GEMM: row (m, s) equals expert ids[m, s]'s brute-force row m
    (dequantized fp64 weights of that expert's N rows, then a plain dot)."""
    r = _rng(23)
    for wtype in (4, 6):
        E, N, K, M, topk = 3, 4, 512, 5, 2
        gen = synth.gen_q4k if wtype == 4 else synth.gen_q6k
        w = gen(E * N, K, int(r.integers(1 << 30)))
        qs, d, bs = orc.quantize_q8k(synth.gen_x(M, K, int(r.integers(1 << 30))))
        ids = r.integers(0, E, (M, topk)).astype(np.int32)
        ids[0] = [2, 2]                       # one token, the same expert twice
        y, a = orc.gemm_id(wtype, w, E, K, qs, d, bs, ids)
        for m in range(M):
            for s in range(topk):
                e = int(ids[m, s])
                yb = orc.brute(wtype, w[e * N:(e + 1) * N], K, qs, d)[m]
                row = m * topk + s
                assert np.all(np.abs(y[row] - yb) <= 1e-12 * a[row] + 1e-300), (wtype, m, s)


def check_gemm_id_bad_ids_and_slots(orc):
    """Ids outside [0, E) leave their rows untouched; swapping a token's slots swaps its rows."""
    E, N, K, M = 2, 3, 256, 3
    w = synth.gen_q4k(E * N, K, 24)
    qs, d, bs = orc.quantize_q8k(synth.gen_x(M, K, 25))
    ids = np.array([[0, 1], [-1, 1], [1, E]], np.int32)
    y, _ = orc.gemm_id(4, w, E, K, qs, d, bs, ids)
    assert np.isnan(y[2]).all() and np.isnan(y[5]).all()
    assert np.isfinite(y[[0, 1, 3, 4]]).all()
    y2, _ = orc.gemm_id(4, w, E, K, qs, d, bs, ids[:, ::-1].copy())
    assert np.array_equal(y[0], y2[1]) and np.array_equal(y[1], y2[0])
    assert not np.array_equal(y[0], y[1])   # the two experts differ


def check_epilogue_values(orc):
    """Printed constants: sigmoid(1) = 0.7310585786300049 (SiLU(1)), the standard
    normal CDF Phi(1) = 0.8413447460685429 (GELU(1)) and 1 - Phi(1) (-GELU(-1));
    ReLU by sign; large arguments pass through or vanish."""
    y = np.array([[1.0, -1.0, 0.0, 20.0, -20.0, 3.0, -2.0]])
    relu = orc.epilogue(y, act=1)[0]
    assert np.array_equal(relu, [1.0, 0.0, 0.0, 20.0, 0.0, 3.0, 0.0])
    silu = orc.epilogue(y, act=2)[0]
    assert abs(silu[0] - 0.7310585786300049) < 1e-15 and silu[2] == 0.0
    assert abs(silu[3] - 20.0) < 1e-6 and abs(silu[4]) < 1e-7
    gelu = orc.epilogue(y, act=3)[0]
    assert abs(gelu[0] - 0.8413447460685429) < 1e-15 and abs(gelu[1] + 0.15865525393145707) < 1e-15
    assert gelu[2] == 0.0 and gelu[3] == 20.0 and abs(gelu[4]) < 1e-80
    assert np.array_equal(orc.epilogue(y, act=0), y)


def check_epilogue_odd_part_and_bias(orc):
    """For all three activations act(v) - act(-v) = v; a bias is added per column before the activation."""
    r = _rng(26)
    v = r.normal(0, 3, (5, 9))
    for act in (1, 2, 3):
        d = orc.epilogue(v, act=act) - orc.epilogue(-v, act=act)
        assert np.all(np.abs(d - v) <= 1e-12 * (1 + np.abs(v))), act
    b = r.normal(0, 1, 9).astype(np.float32)
    assert np.array_equal(orc.epilogue(v, bias=b), v + b.astype(np.float64)[None, :])
    relu_b = orc.epilogue(v, bias=b, act=1)
    assert np.array_equal(relu_b, np.maximum(v + b.astype(np.float64)[None, :], 0.0))


def check_ptq1_bytes_hand(orc):
    """Hand-derived PTQ1_0 bytes: a lone trit 1 at weight k = 24 i + j sets qs
    byte j to 3^i; weight 120 + r sets qh byte r % 2 to 3^(r // 2); all 2s give
    242 (qs) and 80 (qh); d sits little-endian at byte 26."""
    t = np.zeros(128, np.int32)
    t[49] = 1                       # i = 2, j = 1
    t[123] = 1                      # r = 3: qh byte 1, digit 1
    blk = orc.ptq1_pack(0x3800, t)
    exp = np.zeros(28, np.uint8)
    exp[1] = 9
    exp[25] = 3
    exp[26], exp[27] = 0x00, 0x38
    assert np.array_equal(blk, exp), blk
    blk2 = orc.ptq1_pack(0x3C00, np.full(128, 2, np.int32))
    assert (blk2[:24] == 242).all() and (blk2[24:26] == 80).all()
    # decode of a hand-built byte: 5 = 2 + 1*3 -> weight 5 is +d, weight 29 is 0, all others -d
    raw = np.zeros(28, np.uint8)
    raw[5] = 5
    raw[26], raw[27] = 0x00, 0x38   # d = 0.5
    w = orc.dequant(1, raw)
    want = np.full(128, -0.5)
    want[5], want[29] = 0.5, 0.0
    assert np.array_equal(w, want)


def check_ptq1_roundtrip(orc):
    """Every valid byte value decodes to its 5 (qs) or 4 (qh) base-3 digits and packs back."""
    r = _rng(27)
    for _ in range(20):
        t = r.integers(0, 3, 128).astype(np.int32)
        d_bits = int(r.integers(0x1000, 0x5000))
        d, t2 = orc.ptq1_fields(orc.ptq1_pack(d_bits, t))
        assert np.array_equal(t, t2) and d == orc.half_to_double(d_bits)
    blk = np.zeros(28, np.uint8)
    for v in range(243):
        blk[7] = v
        _, t = orc.ptq1_fields(blk)
        digits = [t[24 * i + 7] for i in range(5)]
        assert sum(dg * 3 ** i for i, dg in enumerate(digits)) == v
    blk[7] = 0
    for v in range(81):
        blk[24] = v
        _, t = orc.ptq1_fields(blk)
        assert sum(t[120 + 2 * i] * 3 ** i for i in range(4)) == v


def check_gemm_ptq1(orc):
    """PTQ1_0 GEMM vs the brute force (dequantized weights, plain dot); all +1
    weights with d = 1 and activation scale 1 give numpy's integer row sums."""
    r = _rng(28)
    for (M, N, K) in ((1, 1, 256), (3, 4, 512), (5, 2, 768)):
        w = synth.gen_ptq1(N, K, int(r.integers(1 << 30)))
        qs, d, bs = orc.quantize_q8k(synth.gen_x(M, K, int(r.integers(1 << 30))))
        y, absc = orc.gemm(1, w, K, qs, d, bs)
        yb = orc.brute(1, w, K, qs, d)
        assert np.all(np.abs(y - yb) <= 1e-12 * absc + 1e-300), (M, N, K)
    K, M = 512, 3
    blk = orc.ptq1_pack(0x3C00, np.full(128, 2, np.int32))
    w = np.tile(blk, (2, K // 128))
    qs, d, bs = _q8k_direct(r, M, K)
    y, _ = orc.gemm(1, w, K, qs, d, bs)
    tot = qs.astype(np.int64).sum(axis=1).astype(np.float64)
    assert np.array_equal(y, np.stack([tot, tot], axis=1))


ALL_CHECKS = [
    check_half_decode,
    check_q4k_header_bytes_hand, check_q4k_scale_bytes_hand, check_q4k_nibble_bytes_hand, check_q4k_roundtrip,
    check_q4k_dequant_hand,
    check_q6k_bytes_hand, check_q6k_roundtrip, check_q6k_dequant_hand,
    check_q8k_bound_and_extremes, check_q8k_ties, check_q8k_bsums,
    check_q8k_matches_numpy_rounding, check_q8k_aos_roundtrip,
    check_gemm_vs_brute, check_gemm_unit_scales_q4k, check_gemm_zero_quants_q4k,
    check_gemm_subblock_scales_q4k, check_gemm_q6k_offset, check_gemm_q6k_subblock_scales,
    check_gemm_rows_subset, check_gemm_id_vs_brute, check_gemm_id_bad_ids_and_slots,
    check_epilogue_values, check_epilogue_odd_part_and_bias,
    check_ptq1_bytes_hand, check_ptq1_roundtrip, check_gemm_ptq1,
]
