/*
 * oracle.h -- plain, single-threaded CPU definition of the k-quant prefill
 * matmul (Q4_K / Q6_K weights x Q8_K activations -> fp32 output).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path (the CUDA library
 * and its Python binding) may include, link, load or call this code; only the
 * tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no header, helper, table or constant with the CUDA path.
 *
 * What it computes, and where that is written down:
 *   - The operation is the quantized prefill GEMM the pages study:
 *     "perf(KERNEL-QUANT-CIQ-GEMM-ROCM): cooperative-tile WMMA kernels --
 *     Shared rejected, BigTile accepted" (vllm.cpp PR #3036), commit 1
 *     (Q4_K/Q6_K prefill shapes) and commit 4 (BlockQ8_K, 292 B / 256
 *     elements), and "cuda: branch-free PTQ1_0 MMQ tile loader" (llama.cpp
 *     PR #214), Summary (mul_mat_q prefill path).
 *   - Field semantics of the three block types, as this library defines them:
 *       Q4_K: 256 weights = 8 sub-blocks of 32; 4-bit q; 6-bit sub-scale sc_j
 *             and sub-min m_j; fp16 d and dmin;  w = d*sc_j*q - dmin*m_j.
 *       Q6_K: 256 weights = 16 sub-blocks of 16; 6-bit q split into a low
 *             nibble (ql) and 2 high bits (qh); int8 sub-scale; fp16 d;
 *             w = d*sc_j*(q - 32).
 *       Q8_K: 256 int8 q; fp32 d = amax/127; q = round-half-away(x/d)
 *             clamped to +-127; 16 int16 bsums (sum of each 16 q).
 *   - Byte packing is not printed on any page; the reading used here is the
 *     common GGUF packing (see the layout comments in oracle.c).
 *
 * Pins (what this code is checked against, in tests/test_oracle_*.py):
 *   fp16 decode vs numpy on all 65536 patterns; pack/unpack round trips and
 *   hand-derived field cases; the quantizer's d/2 bound, tie, amax and
 *   all-zero cases; brute-force fp64 dequantize-then-matmul on tiny shapes;
 *   the block-integer form vs the dequantized dot product; the hand-built
 *   single-superblock cases (zero quants -> -dx*dmin*sum m_j*bsum_j, unit
 *   scales -> plain integer dot, Q6_K q = 32 -> 0).  Outputs at the large
 *   benchmark shapes have no closed form and rest on those pins.
 */
#ifndef QGEMM_ORACLE_H
#define QGEMM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_QK 256          /* weights per superblock            */
#define ORACLE_Q4K_BYTES 144   /* 2+2+12+128                        */
#define ORACLE_Q6K_BYTES 210   /* 128+64+16+2                       */
#define ORACLE_PTQ1_BYTES 28   /* 24+2+2, 128 ternary weights        */
#define ORACLE_Q8K_BYTES 292   /* 4+256+32 (interop AoS form)       */

/* IEEE binary16 bit pattern -> double (exact). */
double oracle_half_to_double(uint16_t h);

/* Unpack one Q4_K block into its fields.  q[256] in 0..15, sc[8], mn[8] in
 * 0..63.  d and dmin are returned exactly (fp16 -> double). */
void oracle_q4k_fields(const uint8_t *blk, double *d, double *dmin,
                       int sc[8], int mn[8], int q[256]);
/* Pack fields into one Q4_K block (inverse of oracle_q4k_fields). */
void oracle_q4k_pack(uint16_t d_bits, uint16_t dmin_bits, const int sc[8],
                     const int mn[8], const int q[256], uint8_t *blk);

/* Unpack one Q6_K block.  q[256] in 0..63 (unsigned, before the -32 offset),
 * sc[16] in -128..127. */
void oracle_q6k_fields(const uint8_t *blk, double *d, int sc[16], int q[256]);
void oracle_q6k_pack(uint16_t d_bits, const int sc[16], const int q[256],
                     uint8_t *blk);

/* Dequantize one block to 256 doubles (the spec formulas, in fp64). */
void oracle_dequant_q4k(const uint8_t *blk, double w[256]);
void oracle_dequant_q6k(const uint8_t *blk, double w[256]);

/* PTQ1_0 ("cuda: branch-free PTQ1_0 MMQ tile loader ...", llama.cpp PR #214,
 * commit "load_tiles_ptq1_0"): 128 ternary weights in 28 bytes -- qs words
 * 0-5 (24 bytes, 5 trits each), word 6 = qh[0] | qh[1] << 8 | d << 16 (two
 * bytes of 4 trits each, then the fp16 scale).  The pages leave the trit
 * order open; the reading here: a byte holds its digits base 3, least
 * significant first (digit i = (byte / 3^i) mod 3), a digit t stands for the
 * value t - 1, and the weights are digit-major -- weight k < 120 is digit
 * k / 24 of qs byte k % 24, weight 120 + r is digit r / 2 of qh byte r % 2.
 *   w_k = d * (t_k - 1). */
void oracle_ptq1_fields(const uint8_t *blk, double *d, int t[128]);
void oracle_ptq1_pack(uint16_t d_bits, const int t[128], uint8_t *blk);
void oracle_dequant_ptq1(const uint8_t *blk, double w[128]);
/* Y = X_q8k * W_ptq1^T as for Q4_K/Q6_K, K a multiple of 256 (two blocks per
 * Q8_K superblock b): c_b = dx[m][b] * (d_0 * I_0 + d_1 * I_1), I the exact
 * integer dot of the block's t - 1 with the activations. */
void oracle_gemm_ptq1(const uint8_t *w, int64_t N, int64_t K, int64_t ldw,
                      const int8_t *qs, const float *dx, int64_t M, const int64_t *rows, int64_t nrows,
                      double *y, double *absc);

/* Q8_K quantizer, rows of x[M][ldx] fp32 with K % 256 == 0.
 * Outputs (SoA): qs[M][K] int8, d[M][K/256] fp32, bsums[M][K/16] int16. */
void oracle_quantize_q8k(const float *x, int64_t M, int64_t K, int64_t ldx,
                         int8_t *qs, float *d, int16_t *bsums);

/* Q8_K SoA <-> 292-byte AoS blocks {float d; int8 qs[256]; int16 bsums[16]}. */
void oracle_q8k_to_aos(const int8_t *qs, const float *d, const int16_t *bsums,
                       int64_t M, int64_t K, uint8_t *aos);
void oracle_q8k_from_aos(const uint8_t *aos, int64_t M, int64_t K, int8_t *qs,
                         float *d, int16_t *bsums);

/* The GEMM in block-integer form, fp64.
 *   w: N rows, each nb = K/256 consecutive blocks, row stride ldw bytes.
 *   X: Q8_K SoA (qs[M][K], d[M][nb], bsums[M][K/16]).
 *   rows: the token indices m to evaluate (nrows of them); NULL = all M.
 *   y[r][n]    = sum over superblocks b (ascending) of c_b
 *   absc[r][n] = sum over b of |c_b|   (for the tolerance), may be NULL. */
void oracle_gemm_q4k(const uint8_t *w, int64_t N, int64_t K, int64_t ldw,
                     const int8_t *qs, const float *dx, const int16_t *bsums,
                     int64_t M, const int64_t *rows, int64_t nrows,
                     double *y, double *absc);
void oracle_gemm_q6k(const uint8_t *w, int64_t N, int64_t K, int64_t ldw,
                     const int8_t *qs, const float *dx, const int16_t *bsums,
                     int64_t M, const int64_t *rows, int64_t nrows,
                     double *y, double *absc);

/* Expert-routed GEMM (MUL_MAT_ID, tested beside MUL_MAT on the page
 * "cuda: branch-free PTQ1_0 MMQ tile loader ..." (llama.cpp PR #214)):
 * w holds E experts of N rows each, back to back (expert e = rows e*N ..
 * e*N+N-1); for token m and slot s the expert e = ids[m*top_k + s] and
 *   y[m*top_k + s][n] = the row-n, token-m output of expert e's GEMM above.
 * Pairs whose id is outside [0, E) are left as they are in y (and absc).
 * type 4 = Q4_K (ldw row stride), 6 = Q6_K (210-B blocks). */
void oracle_gemm_id(int type, const uint8_t *w, int64_t E, int64_t N, int64_t K, int64_t ldw,
                    const int8_t *qs, const float *dx, const int16_t *bsums, int64_t M,
                    const int32_t *ids, int64_t top_k, double *y, double *absc);

/* Output epilogue, in place on y[R][N] in fp64:
 *   y[r][n] = act(y[r][n] + bias[n])   (bias may be NULL)
 * act: 0 none, 1 ReLU max(v, 0), 2 SiLU v / (1 + exp(-v)),
 *      3 GELU 0.5 v (1 + erf(v / sqrt 2)).
 * (Rounding to an fp16 / bf16 output type is left to the caller.) */
void oracle_epilogue(double *y, int64_t R, int64_t N, const float *bias, int act);

/* Brute force: dequantize W and X to fp64, then a plain triple loop.
 * type 4 = Q4_K, 6 = Q6_K, 1 = PTQ1_0.  y[M][N]. */
void oracle_brute(int type, const uint8_t *w, int64_t N, int64_t K, int64_t ldw,
                  const int8_t *qs, const float *dx, int64_t M, double *y);

#ifdef __cplusplus
}
#endif
#endif
