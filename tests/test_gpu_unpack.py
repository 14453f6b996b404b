"""The tile GEMM's weight expansion, on its own, against the CPU oracle's
decoding of the same bytes: qgemm_debug_expand runs the GEMM's expanders
(the device functions its unpack warps call) over 10^4+ blocks per weight
type, and every operand value, side value and flag is compared with what the
oracle's field decoding (oracle_q4k_fields / oracle_q6k_fields /
oracle_ptq1_fields) says it must be.  Among the blocks: every 6-bit value in
every Q4_K scale and min position, the int8 sub-scale extremes in every Q6_K
position, every PTQ1_0 byte value.  (The review of llama.cpp PR #214
checks its tile loader by emulating it on 10,000 packed blocks; this is that
check on the device.)"""
import numpy as np
import pytest
import torch

import oracle
import block_quantized_matmul_quantize_gb300 as qg
from gpu_common import ensure_built, to_dev

pytestmark = pytest.mark.gpu

NBLK = 12000


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()


def _k_order():
    """TMEM column j of chunk c, fp16 half h -> the weight index it holds."""
    c = np.arange(4)[:, None, None]
    j = np.arange(32)[None, :, None]
    h = np.arange(2)[None, None, :]
    return (64 * c + 4 * (j // 2) + (j % 2) + 2 * h).reshape(-1)


KIDX = _k_order()
assert np.array_equal(np.sort(KIDX), np.arange(256))


def _operand(words):
    """int32 [n, 128] words -> float64 [n, 256] in weight order."""
    u = words.astype(np.int64) & 0xffffffff
    halves = np.stack([(u & 0xffff), (u >> 16)], axis=-1).astype(np.uint16).view(np.float16)
    out = np.empty((words.shape[0], 256))
    out[:, KIDX] = halves.reshape(words.shape[0], -1).astype(np.float64)
    return out


def _expand(wtype, blocks_np, n):
    rec = qg.qgemm_debug_expand(wtype, to_dev(blocks_np), n)
    torch.cuda.synchronize()
    return rec.cpu().numpy()


def _f16(bits):
    return np.array([bits], np.uint16).view(np.float16).astype(np.float64)[0]


def _floor_log2(x):
    m, e = np.frexp(abs(x))
    return e - 1


# ------------------------------------------------------------------ Q4_K --
def _q4k_blocks(orc, r):
    blks = []
    # every 6-bit value in every scale and min position
    for v in range(64):
        for j in range(8):
            sc = r.integers(0, 64, 8)
            mn = r.integers(0, 64, 8)
            sc[j] = v
            mn[(j + 3) % 8] = 63 - v
            blks.append(orc.q4k_pack(int(r.integers(0x1000, 0x2000)), int(r.integers(0x1000, 0x2000)), sc, mn,
                                     r.integers(0, 16, 256)))
    # header cases: d = 0, dmin = 0, tiny d (large dmin/d), subnormal d, the declined range
    hdrs = [(0x0000, 0x2000), (0x2000, 0x0000), (0x0000, 0x0000), (0x0001, 0x3C00), (0x0003, 0x3800),
            (0x0200, 0x3C00), (0x0400, 0x4000), (0x0001, 0x4400), (0x0001, 0x4000), (0x3C00, 0x3C00)]
    for db, mb in hdrs:
        for _ in range(40):
            blks.append(orc.q4k_pack(db, mb, r.integers(0, 64, 8), r.integers(0, 64, 8), r.integers(0, 16, 256)))
    # random bytes after a random normal header
    while len(blks) < NBLK:
        b = r.integers(0, 256, 144).astype(np.uint8)
        b[0:2] = np.array([int(r.integers(0x0400, 0x3C00))], np.uint16).view(np.uint8)
        b[2:4] = np.array([int(r.integers(0x0400, 0x3C00))], np.uint16).view(np.uint8)
        blks.append(b)
    return np.stack(blks)


def test_q4k_expansion_matches_oracle_fields():
    orc = oracle.get()
    r = np.random.default_rng(1)
    blocks = _q4k_blocks(orc, r)
    n = len(blocks)
    rec = _expand(4, blocks, n)
    main = _operand(rec[:, :128])
    a1 = (rec[:, 256:264].astype(np.int64) & 0xffff).astype(np.uint16).view(np.float16).astype(np.float64)
    a2 = (rec[:, 264:272].astype(np.int64) & 0xffff).astype(np.uint16).view(np.float16).astype(np.float64)
    e = rec[:, 272].view(np.float32).astype(np.float64)
    ok = (rec[:, 273] & 1).astype(bool)
    shift = (rec[:, 273] >> 8) & 0xff
    assert np.all(rec[:, 128:256] == 0)
    bad = 0
    for i in range(n):
        d, dmin, sc, mn, q = orc.q4k_fields(blocks[i])
        # the documented shift: s = clamp(E(dmin) - E(d) - 8, 0, 14), 0 for d = 0
        s = 0 if d == 0 else int(np.clip((_floor_log2(dmin) if dmin != 0 else -200) - _floor_log2(d) - 8, 0, 14))
        assert shift[i] == s, (i, shift[i], s)
        want = np.zeros(256) if d == 0 else np.repeat(sc, 32) * q * 2.0 ** -s
        if not np.array_equal(main[i], want):
            bad += 1
            continue
        ratio32 = np.float32(-1.0) if d == 0 else (np.float32(-dmin) / np.float32(d)) * np.float32(2.0 ** -s)
        # declined only at the largest shift, when 63 * |r * 2^-14| would pass fp16's 65504
        in_range = s != 14 or abs(float(ratio32)) <= 1039.0
        assert ok[i] == in_range, (i, d, dmin)
        if not in_range:
            assert np.isnan(e[i])
            continue
        assert e[i] == (dmin if d == 0 else d * 2.0 ** s), (i, e[i], d, s)
        exact = mn * ((-1.0) if d == 0 else (-dmin / d) * 2.0 ** -s)
        err = np.abs(a1[i] + a2[i] - exact)
        # 22 bits in the fp16 hi + lo pair (the lo part may be subnormal: 2^-24 absolute)
        assert np.all(err <= 2.0 ** -21 * np.abs(exact) + 2.0 ** -24), (i, err, exact)
    assert bad == 0, f"{bad} of {n} Q4_K blocks expand to the wrong operand"
    assert (~ok).sum() >= 40        # the (6e-8, 4.0) header rows are declined


# ------------------------------------------------------------------ Q6_K --
EXTREMES = [-128, -127, -65, -64, -1, 0, 1, 63, 64, 65, 127]


def _q6k_blocks(orc, r):
    blks = []
    for v in EXTREMES:
        for j in range(16):
            sc = r.integers(-128, 128, 16)
            sc[j] = v
            blks.append(orc.q6k_pack(int(r.integers(0x0800, 0x2000)), sc, r.integers(0, 64, 256)))
    for v in range(64):                          # every 6-bit code in every position of a sub-block
        q = (np.arange(256) + v) % 64
        blks.append(orc.q6k_pack(0x3C00, r.integers(-128, 128, 16), q))
    while len(blks) < NBLK:
        b = r.integers(0, 256, 210).astype(np.uint8)
        b[208:210] = np.array([int(r.integers(0x0400, 0x3C00))], np.uint16).view(np.uint8)
        blks.append(b)
    return np.stack(blks)


def test_q6k_expansion_matches_oracle_fields():
    orc = oracle.get()
    r = np.random.default_rng(2)
    blocks = _q6k_blocks(orc, r)
    n = len(blocks)
    packed = qg.qgemm_q6k_prepack(to_dev(blocks), n, 256)
    rec = qg.qgemm_debug_expand(6, packed, n)
    torch.cuda.synchronize()
    rec = rec.cpu().numpy()
    hi = _operand(rec[:, :128])
    lo = _operand(rec[:, 128:256])
    e = rec[:, 272].view(np.float32).astype(np.float64)
    assert np.all(rec[:, 273] == 1) and np.all(rec[:, 256:272] == 0)
    for i in range(n):
        d, sc, q = orc.q6k_fields(blocks[i])
        v = q - 32.0
        scw = np.repeat(sc, 16).astype(np.float64)
        assert np.array_equal(hi[i] + lo[i], scw * v), i          # the two parts add to sc*(q - 32) exactly
        split = (np.abs(scw) > 64) & (np.abs(scw) % 2 == 1)       # lo = 1 exactly for odd |sc| > 64
        assert np.array_equal(lo[i], np.where(split, v, 0.0)), i
        assert np.all(np.abs(hi[i]) <= 4096)
        assert e[i] == d, i


# ---------------------------------------------------------------- PTQ1_0 --
def test_ptq1_expansion_matches_oracle_fields():
    orc = oracle.get()
    r = np.random.default_rng(3)
    nb = NBLK                                   # 128-weight blocks, two per superblock row
    blks = []
    for i in range(nb):
        b = np.zeros(28, np.uint8)
        b[:24] = (np.arange(24) + i) % 243 if i < 243 else r.integers(0, 243, 24)   # every byte value
        b[24:26] = r.integers(0, 81, 2)
        b[26:28] = np.array([int(r.integers(0x0400, 0x3C00))], np.uint16).view(np.uint8)
        blks.append(b)
    raw = np.stack(blks).reshape(nb // 2, 56)
    packed = qg.qgemm_ptq1_prepack(to_dev(raw), nb // 2, 256)
    rec = qg.qgemm_debug_expand(1, packed, nb // 2)
    torch.cuda.synchronize()
    rec = rec.cpu().numpy()
    op = _operand(rec[:, :128])
    assert np.all(rec[:, 128:272] == 0) and np.all(rec[:, 272].view(np.float32) == 1.0)
    for s in range(nb // 2):
        for j in range(2):
            d, t = orc.ptq1_fields(raw[s, 28 * j:28 * j + 28])
            want = d * (t - 1.0)                     # exact in fp16: +-d or 0
            assert np.array_equal(op[s, 128 * j:128 * j + 128], want), (s, j)
