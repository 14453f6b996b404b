"""Plant mistakes in a copy of the oracle (on the CPU) and check that the pins
catch every one of them: a pin suite that passes a broken oracle proves
nothing.  Each mutant is built from oracle.c with one textual change (or,
where one mistake must be made in two places to survive the round trips, a
list of changes)."""
import os
import shutil

import pytest

import oracle
from oracle_pins import ALL_CHECKS

MUTATIONS = {
    "half_exponent_bias": ("ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)"),
    "q4k_low_nibble_from_high": ("q[64 * c + l] = qs[32 * c + l] & 15;", "q[64 * c + l] = qs[32 * c + l] >> 4;"),
    "q4k_scale_index": ("sc[j] = s[j] & 63;", "sc[j] = s[j + 4] & 63;"),
    "q4k_high_scale_bits": ("sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);", "sc[j] = (s[j + 4] & 15) | ((s[j] >> 6) << 4);"),
    "q6k_qh_shift": ("o[l + 32] = (L[l + 32] & 15) | (((H[l] >> 2) & 3) << 4);", "o[l + 32] = (L[l + 32] & 15) | (((H[l] >> 4) & 3) << 4);"),
    "q6k_pack_halves": ("uint8_t *L = ql + 64 * h;\n        uint8_t *H", "uint8_t *L = ql + 32 * h;\n        uint8_t *H"),
    "q8k_round_half_even": ("float r = roundf(xb[i] / db);", "float r = rintf(xb[i] / db);"),
    "q8k_scale_128": ("float db = amax / 127.0f;", "float db = amax / 128.0f;"),
    "q8k_bsum_offbyone": ("sb[g] = (int16_t)s;", "sb[g] = (int16_t)(s + (g == 3));"),
    "q8k_amax_signed": ("float a = fabsf(xb[i]);", "float a = xb[i];"),
    "gemm_q4k_drop_dmin": ("(d * (double)dot - dmin * (double)corr)", "(d * (double)dot - 0.0 * (double)corr)"),
    "gemm_q4k_bsum_pair": ("corr += (int64_t)mn[j] * (bs[2 * j] + bs[2 * j + 1]);", "corr += (int64_t)mn[j] * (bs[j] + bs[j + 8]);"),
    "gemm_q4k_subblock_width": ("for (int i = 32 * j; i < 32 * j + 32; ++i)", "for (int i = 32 * j; i < 32 * j + 31; ++i)"),
    "gemm_q6k_offset_31": ("dot += (int64_t)sc[j] * (I - 32 * (int64_t)bs[j]);", "dot += (int64_t)sc[j] * (I - 31 * (int64_t)bs[j]);"),
    "gemm_q6k_transposed_x": ("const int8_t *xq = qs + m * K + b * 256;\n                const int16_t *bs = bsums + m * (K / 16) + b * 16;\n                int64_t dot = 0;\n", "const int8_t *xq = qs + m * K + b * 256 + (b > 0 ? -256 : 0);\n                const int16_t *bs = bsums + m * (K / 16) + b * 16;\n                int64_t dot = 0;\n"),
    "gemm_absc_signed": ("absc[r * N + n] += fabs(cb);\n            }\n        }\n    }\n    free(own);\n}\n\nvoid oracle_gemm_q6k", "absc[r * N + n] += cb;\n            }\n        }\n    }\n    free(own);\n}\n\nvoid oracle_gemm_q6k"),
    "gemm_id_expert_offset": ("const uint8_t *we = w + e * N * ldw;", "const uint8_t *we = w + e * ldw;"),
    "gemm_id_pair_row": ("const int64_t pair = m * top_k + s;", "const int64_t pair = m + s * M;"),
    "epilogue_silu_sign": ("v = v / (1.0 + exp(-v));", "v = v / (1.0 + exp(v));"),
    "epilogue_gelu_scale": ("v = 0.5 * v * (1.0 + erf(v / sqrt(2.0)));", "v = 0.5 * v * (1.0 + erf(v / 2.0));"),
    "epilogue_bias_row": ("(bias ? (double)bias[n] : 0.0)", "(bias ? (double)bias[r % N] : 0.0)"),
    "ptq1_digit_order": ("t[k] = ptq1_digit(blk[k % 24], k / 24);", "t[k] = ptq1_digit(blk[k % 24], 4 - k / 24);"),
    "ptq1_qh_byte": ("t[120 + r] = ptq1_digit(blk[24 + r % 2], r / 2);", "t[120 + r] = ptq1_digit(blk[24 + r / 4], r % 4);"),
    "ptq1_gemm_offset": ("I[h] += (int64_t)(t[h][k] - 1) * xq[128 * h + k];", "I[h] += (int64_t)t[h][k] * xq[128 * h + k];"),
    # d and dmin swapped in both the decoder and the packer (their round trip still agrees)
    "q4k_d_dmin_swapped": [("*d = oracle_half_to_double(rd16(blk));\n    *dmin = oracle_half_to_double(rd16(blk + 2));",
                            "*d = oracle_half_to_double(rd16(blk + 2));\n    *dmin = oracle_half_to_double(rd16(blk));"),
                           ("wr16(blk, d_bits);\n    wr16(blk + 2, dmin_bits);",
                            "wr16(blk + 2, d_bits);\n    wr16(blk, dmin_bits);")],
    "brute_dmin_sign": ("w[i] = d * sc[i / 32] * q[i] - dmin * mn[i / 32];", "w[i] = d * sc[i / 32] * q[i] + dmin * mn[i / 32];"),
}


def _fails(orc):
    failed = []
    for check in ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            failed.append(check.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutant_is_caught(name, tmp_path):
    src = open(oracle.SRC).read()
    changes = MUTATIONS[name]
    for old, new in ([changes] if isinstance(changes, tuple) else changes):
        assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
        src = src.replace(old, new)
    mdir = tmp_path / "mut"
    mdir.mkdir()
    shutil.copy(os.path.join(oracle.HERE, "oracle.h"), mdir / "oracle.h")
    (mdir / "oracle.c").write_text(src)
    lib = oracle.build(str(mdir / "oracle.c"), str(mdir / "liboracle_mut.so"), force=True)
    failed = _fails(oracle.Oracle(lib))
    assert failed, f"no pin catches mutation {name}"
