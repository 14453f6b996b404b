/*
 * qgemm.h -- C ABI of the k-quant prefill matmul library for GB300 (sm_103a).
 *
 * The operation is the quantized prefill GEMM of llama.cpp-style models:
 * weights stored as Q4_K or Q6_K blocks multiply activations quantized on the
 * fly to Q8_K, giving an fp32 output.  The pages this library follows study
 * it as "KQuantGemmKWmmaQ4K/Q6K" ("perf(KERNEL-QUANT-CIQ-GEMM-ROCM):
 * cooperative-tile WMMA kernels -- Shared rejected, BigTile accepted",
 * vllm.cpp PR #3036) and as llama.cpp's mul_mat_q ("cuda: branch-free PTQ1_0
 * MMQ tile loader and full Ampere tile table", llama.cpp PR #214).
 *
 * Block formats (field meaning; the byte packing is the GGUF one):
 *   Q4_K, 144 B / 256 weights: fp16 d, fp16 dmin, 12 bytes holding eight
 *         6-bit sub-scales sc_j and eight 6-bit sub-mins m_j, 128 bytes of
 *         4-bit quants; sub-block j = weights 32j..32j+31;
 *         w = d*sc_j*q - dmin*m_j.
 *   Q6_K, 210 B / 256 weights: ql[128] (low 4 bits), qh[64] (high 2 bits),
 *         int8 scales[16] (sub-block j = weights 16j..16j+15), fp16 d;
 *         w = d*sc_j*(q - 32).
 *   Q8_K, 256 activations: fp32 d = amax/127, int8 q = round-half-away(x/d)
 *         clamped to +-127, int16 bsums[16] = sums of each 16 q (PR #3036,
 *         commit 4, gives the block as 292 bytes per 256 elements).  Here kept
 *         as three planes: qs [M][K] int8, d [M][K/256] fp32, bsums [M][K/16]
 *         int16, each contiguous with row stride K, K/256, K/16 elements.
 *
 * Conventions (all calls):
 *   - Device pointers are caller-owned; the library never allocates or frees
 *     device memory.  Scratch ("workspace") is passed in, sized by a query
 *     function -- the caller-owned-scratch convention of the pages
 *     (hip_linear_attention_prefill_scratch_bytes, hip-ep PR #627).
 *   - Three arrays may instead live in page-locked host memory that the
 *     device can address (cudaHostAlloc, or cudaHostRegister with
 *     cudaHostRegisterMapped, under unified addressing): the fp32 X of the
 *     quantizers, the expert ids of the routed calls, and every GEMM's Y.
 *     The kernels then move those bytes across the host link themselves,
 *     with no staging copy: X and ids are read once per call, and Y is
 *     written once and never read back.  Every other array (weights, Q8_K
 *     planes, workspace) must be device memory; this is not checked.
 *   - Calls enqueue work on `stream` and return; they do not synchronize.
 *   - Argument errors are reported synchronously and nothing is launched
 *     (a nonzero status, so the caller can fall back to another path, the
 *     convention of hip-ep PR #627).  Unsupported
 *     shapes are declined, never computed wrongly.  qgemm_last_error()
 *     gives a one-line reason (thread-local).
 *   - Y is fully overwritten (beta = 0).
 *   - The library keeps process-global launch counters and options (not
 *     synchronized between threads that change options concurrently).
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QGEMM_API __attribute__((visibility("default")))
#else
#define QGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qgemm_stream_t; /* = cudaStream_t; NULL = legacy default stream */
typedef struct CUevent_st *qgemm_event_t;   /* = cudaEvent_t */

typedef enum {
    QGEMM_OK = 0,
    QGEMM_EINVAL = 1,       /* bad size, null pointer, too-small workspace   */
    QGEMM_EALIGN = 2,       /* pointer or stride not aligned as required     */
    QGEMM_EUNSUPPORTED = 3, /* shape outside what the kernels handle         */
    QGEMM_ECUDA = 4,        /* a CUDA launch or runtime call failed          */
    QGEMM_ETIMEOUT = 5,     /* a kernel's bounded wait gave up (device status) */
    QGEMM_EDEVICE = 6       /* a device-side value check failed (status)     */
} qgemm_status;

/* Library version, major*10000 + minor*100 + patch. */
QGEMM_API int qgemm_version(void);

/* One-line description of the last failure in this thread ("" if none). */
QGEMM_API const char *qgemm_last_error(void);

/* ------------------------------------------------------------- Q8_K ----
 * qgemm_quantize_q8k: fp32 activations -> Q8_K planes (the activation
 * quantization that precedes the GEMM; PR #3036 commit 5, EnsureQuantScratch).
 *   x      device or pinned host (Conventions), fp32 [M][ldx] row-major,
 *          16-B aligned, ldx % 4 == 0,
 *          ldx >= K; values must be finite.
 *   M      rows (tokens), M >= 0 (M == 0: nothing to do, QGEMM_OK).
 *   K      columns, K >= 256 and K % 256 == 0.
 *   qs     device, int8 [M][K], 16-B aligned.
 *   d      device, fp32 [M][K/256], 16-B aligned.
 *   bsums  device, int16 [M][K/16], 16-B aligned.
 * Bit-exact with the IEEE definition: d = amax/127 (fp32), q = roundf(x/d)
 * clamped to +-127; d == 0 (amax == 0, or amax/127 underflowing to zero)
 * -> q = 0, bsums = 0.
 * Errors: EINVAL (sizes, null), EALIGN, ECUDA (launch). */
QGEMM_API int qgemm_quantize_q8k(const float *x, int64_t M, int64_t K, int64_t ldx, int8_t *qs, float *d,
                       int16_t *bsums, qgemm_stream_t stream);

/* Caller-owned Q8_K storage (the pages' caller-owned-scratch convention,
 * hip_linear_attention_prefill_scratch_bytes, hip-ep PR #627):
 * qgemm_q8k_bytes(M, K) is the size of one buffer that holds the three planes
 * of M rows of depth K (0 for M <= 0 or K not a positive multiple of 256);
 * qgemm_q8k_planes splits such a buffer (256-B aligned) into the plane
 * pointers the other calls take: qs at offset 0, then d, then bsums, each
 * plane starting on a 256-B boundary.  Host-only arithmetic, no device access.
 * Errors: EINVAL (sizes, null), EALIGN (base). */
QGEMM_API size_t qgemm_q8k_bytes(int64_t M, int64_t K);
QGEMM_API int qgemm_q8k_planes(void *base, int64_t M, int64_t K, int8_t **qs, float **d, int16_t **bsums);

/* The pages' 292-byte Q8_K block ("BlockQ8_K (292B/256 elements)", PR #3036,
 * commit 4), for exchange with code that keeps Q8_K as an array of blocks.
 * Field order within a block (this library's reading; the page gives only
 * the size): fp32 d at byte 0, int8 qs[256] at byte 4, int16 bsums[16] at
 * byte 260, little-endian.  Block (m, b) -- row m, superblock b -- is block
 * number m*(K/256) + b of the array.
 *   qgemm_q8k_aos_bytes(M, K) = M*(K/256)*292 (0 for bad sizes).
 *   qgemm_pack_q8k_aos:   planes (device, as qgemm_quantize_q8k writes them,
 *                         16-B aligned) -> aos (device, 4-B aligned).
 *   qgemm_unpack_q8k_aos: aos -> planes.
 * One device kernel each, enqueued on `stream`; the bytes are copied, not
 * recomputed, so both directions are exact.  M == 0: nothing to do.
 * Errors: EINVAL (sizes, null), EALIGN, ECUDA (launch). */
QGEMM_API size_t qgemm_q8k_aos_bytes(int64_t M, int64_t K);
QGEMM_API int qgemm_pack_q8k_aos(const int8_t *qs, const float *d, const int16_t *bsums, int64_t M, int64_t K,
                                 void *aos, qgemm_stream_t stream);
QGEMM_API int qgemm_unpack_q8k_aos(const void *aos, int64_t M, int64_t K, int8_t *qs, float *d, int16_t *bsums,
                                   qgemm_stream_t stream);

/* ------------------------------------------------------------- GEMM ----
 * Workspace bytes the GEMM calls need for M tokens, N weight rows and depth K
 * on the current device: the fp16 tensor-core operand copy of the Q8_K
 * activations (about 2.1 B per element of M*K), the cut-tile counters
 * (32 KiB), the Q4_K side words (68 B per weight block: the dmin-correction
 * operands and scales that the Q4_K tile GEMM calls make from the weights
 * before the GEMM; counted for every weight type), and the
 * partial tiles of the cut tiles (128 x BM fp32 per K part; tiles are cut
 * when there are fewer of them than SMs, or when a last round would leave at
 * least half of the SMs idle).  With N = 0: the activation part alone (what
 * qgemm_quantize_q8k_prep writes).  0 for M = 0 or an invalid K.  The
 * workspace must be 256-B aligned. */
QGEMM_API size_t qgemm_workspace_bytes(int64_t M, int64_t N, int64_t K);

/* qgemm_q4k: Y[M][N] = X_q8k[M][K] * W_q4k[N][K]^T.
 *   w      device, N rows of K/256 Q4_K blocks (144 B each), row stride ldw
 *          bytes; 16-B aligned; ldw % 16 == 0; ldw >= (K/256)*144.
 *   N      weight rows, N >= 1.     K: K >= 256, K % 256 == 0.
 *   xqs, xd, xbsums   the Q8_K planes of M tokens (as qgemm_quantize_q8k
 *          writes them).   M >= 0 (0: nothing to do).
 *   y      device or pinned host (Conventions), fp32 [M][ldy], ldy >= N,
 *          4-B aligned.  Overwritten.
 *   workspace, workspace_bytes   device scratch >= qgemm_workspace_bytes.
 * Accuracy: |Y - Y_exact| <= 2e-5 * sum_b |c_b| + 1e-6 per element, c_b the
 * contribution of superblock b (fp32 accumulation of exact integer partials).
 * Y is deterministic for a given shape and device: a cut tile's K parts are
 * summed in ascending part order, whichever part finishes last.
 * Value range: every Q4_K block is computed except one with |dmin/d| >
 * 1039 * 2^14 (about 1.7e7, e.g. d = 6e-8 with dmin >= 2), whose dmin
 * correction leaves fp16's range even on the largest power-of-two shifted
 * scale: such a block row is declined -- its output elements become NaN --
 * and device status QGEMM_DEV_Q4K_RANGE is set.  (The small-M path
 * computes every block in fp32.)
 * Errors: EINVAL, EALIGN, EUNSUPPORTED (M, N >= 2^31), ECUDA. */
QGEMM_API int qgemm_q4k(const void *w, int64_t N, int64_t K, int64_t ldw, const int8_t *xqs, const float *xd,
              const int16_t *xbsums, int64_t M, float *y, int64_t ldy, void *workspace,
              size_t workspace_bytes, qgemm_stream_t stream);

/* Q6_K weights are used in a repacked form: each 210-B block padded to 224 B
 * (16-B aligned blocks and rows for TMA).  Repack once, e.g. at model load;
 * the repack is not part of the GEMM.
 *   w_aos  device, N rows of K/256 Q6_K blocks (210 B), row stride ldw >=
 *          (K/256)*210 bytes, no alignment requirement.
 *   w_packed device, qgemm_q6k_packed_bytes(N, K) bytes, 16-B aligned. */
QGEMM_API size_t qgemm_q6k_packed_bytes(int64_t N, int64_t K);
QGEMM_API int qgemm_q6k_prepack(const void *w_aos, int64_t N, int64_t K, int64_t ldw, void *w_packed,
                      qgemm_stream_t stream);

/* qgemm_q6k: as qgemm_q4k, with Q6_K weights repacked by qgemm_q6k_prepack.
 * Every int8 sub-scale (-128..127) is computed exactly: on the tile path
 * a sub-scale beyond +-64 is split into two parts whose fp16 operands are
 * both exact, multiplied into the same accumulator. */
QGEMM_API int qgemm_q6k(const void *w_packed, int64_t N, int64_t K, const int8_t *xqs, const float *xd,
              const int16_t *xbsums, int64_t M, float *y, int64_t ldy, void *workspace,
              size_t workspace_bytes, qgemm_stream_t stream);

/* ------------------------------------------------ prepared workspace ----
 * A step that quantizes and then multiplies can skip one launch: the
 * quantizer writes the tile GEMM's fp16 operand planes into the GEMM's
 * workspace in the same pass (a step toward fusing the quantizer into the
 * GEMM's producer; the pages have no such call).
 *
 * qgemm_quantize_q8k_prep: exactly qgemm_quantize_q8k (same Q8_K planes,
 * bit-exact), and in the same launch it fills `workspace` (>=
 * qgemm_workspace_bytes(M, N, K) bytes for any N, 256-B aligned) with the
 * operand planes derived from those Q8_K values.
 *
 * qgemm_q4k_prepared / qgemm_q6k_prepared: exactly qgemm_q4k / qgemm_q6k,
 * except that the workspace must be one that qgemm_quantize_q8k_prep filled
 * from these same Q8_K planes (same M, K; neither changed since), and it is
 * only read.  For M <= QGEMM_OPT_SMALL_M_MAX the workspace is not used at
 * all (the small-M path reads the planes).  Passing any other workspace
 * gives undefined Y (the library cannot tell).
 * Errors: as the calls they mirror. */
QGEMM_API int qgemm_quantize_q8k_prep(const float *x, int64_t M, int64_t K, int64_t ldx, int8_t *qs, float *d,
                                      int16_t *bsums, void *workspace, size_t workspace_bytes,
                                      qgemm_stream_t stream);
QGEMM_API int qgemm_q4k_prepared(const void *w, int64_t N, int64_t K, int64_t ldw, const int8_t *xqs,
                                 const float *xd, const int16_t *xbsums, int64_t M, float *y, int64_t ldy,
                                 const void *workspace, size_t workspace_bytes, qgemm_stream_t stream);
QGEMM_API int qgemm_q6k_prepared(const void *w_packed, int64_t N, int64_t K, const int8_t *xqs, const float *xd,
                                 const int16_t *xbsums, int64_t M, float *y, int64_t ldy, const void *workspace,
                                 size_t workspace_bytes, qgemm_stream_t stream);

/* ------------------------------------------ fp32 activations in ----
 * The whole path behind one call: X (fp32) is quantized to Q8_K and
 * multiplied, Y[M][N] = Q8_K(X) . W^T, as qgemm_quantize_q8k followed by
 * qgemm_q4k / qgemm_q6k (the same Y and Q8_K values, bit for bit; the pages
 * quantize the activations as the step before the GEMM, vllm.cpp PR #3036,
 * commit 5, and suggest doing it inside the GEMM's load stage).
 *   x, ldx          fp32 [M][ldx], device or pinned host memory; 16-B aligned,
 *                   ldx >= K, ldx % 4 == 0 (as qgemm_quantize_q8k).
 *   qs, d, bsums    the Q8_K planes of X, written in every case.
 *   workspace       >= qgemm_workspace_bytes(M, N, K), 256-B aligned; used
 *                   only above the small-M path (may be NULL at or below it).
 *   w, ldw, N, K, y, ldy   as qgemm_q4k (Q6_K: the repacked blocks).
 * For M <= 2 within the small-M path (QGEMM_OPT_SMALL_M_MAX, K <= 15360) it
 * is one launch: the weight-streaming kernel quantizes the activations
 * itself, each lane the values it multiplies, while the first weights are
 * in flight (counted in small_fused).  Otherwise the quantizer runs first
 * (for the tile GEMM it also fills the workspace's operand planes) and the
 * GEMM starts under it.  Errors: as qgemm_quantize_q8k and qgemm_q4k. */
QGEMM_API int qgemm_q4k_f32(const void *w, int64_t N, int64_t K, int64_t ldw, const float *x, int64_t ldx,
                            int64_t M, int8_t *qs, float *d, int16_t *bsums, float *y, int64_t ldy, void *workspace,
                            size_t workspace_bytes, qgemm_stream_t stream);
QGEMM_API int qgemm_q6k_f32(const void *w_packed, int64_t N, int64_t K, const float *x, int64_t ldx, int64_t M,
                            int8_t *qs, float *d, int16_t *bsums, float *y, int64_t ldy, void *workspace,
                            size_t workspace_bytes, qgemm_stream_t stream);

/* ------------------------------------ expert-routed GEMM (MUL_MAT_ID) ----
 * The routed form of the GEMM that the pages test beside MUL_MAT (llama.cpp
 * PR #214 "cuda: branch-free PTQ1_0 MMQ tile loader ...", test-backend-ops
 * MUL_MAT_ID): E experts of N weight rows each, stored back to back (expert
 * e's rows are rows e*N .. e*N+N-1 of one weight matrix), and for every token
 * i and slot s < top_k an expert id; the output row of pair (i, s) is
 *     Y[i*top_k + s][n] = sum_k W[ids[i*top_k + s]*N + n][k] * X_q8k[i][k]
 * with the same accuracy bound as qgemm_q4k (per output element, c_b the
 * contributions of expert ids[i][s]'s row n).
 *   w, ldw      as qgemm_q4k, E*N rows (Q6_K: the 224-B repacked blocks of all
 *               E*N rows, qgemm_q6k_prepack with N = E*N).
 *   experts     E, 1..1024.   N, K, xqs, xd, xbsums, M: as qgemm_q4k.
 *   ids         device or pinned host, int32 [M][top_k], 4-B aligned; ids outside [0, E) set
 *               device status QGEMM_DEV_BAD_EXPERT and their output rows are
 *               left untouched.
 *   top_k       slots per token, >= 1;  M * top_k and E * N below 2^31.
 *   y           device or pinned host, fp32 [M * top_k][ldy], ldy >= N, 4-B aligned.
 *   workspace   >= qgemm_id_workspace_bytes(M, top_k, E, K), 256-B aligned:
 *               the routing (pairs grouped by expert) and the operand planes of
 *               the M * top_k routed rows.
 * Three launches: routing, operand gather, and one tile GEMM over all
 * experts (a token tile never mixes experts; the epilogue writes each row to
 * its pair).  Y does not depend on the order of the pairs within an expert.
 * Errors: as qgemm_q4k. */
QGEMM_API size_t qgemm_id_workspace_bytes(int64_t M, int64_t top_k, int64_t experts, int64_t K);
QGEMM_API int qgemm_q4k_id(const void *w, int64_t experts, int64_t N, int64_t K, int64_t ldw, const int8_t *xqs,
                           const float *xd, const int16_t *xbsums, int64_t M, const int32_t *ids, int64_t top_k,
                           float *y, int64_t ldy, void *workspace, size_t workspace_bytes, qgemm_stream_t stream);
QGEMM_API int qgemm_q6k_id(const void *w_packed, int64_t experts, int64_t N, int64_t K, const int8_t *xqs,
                           const float *xd, const int16_t *xbsums, int64_t M, const int32_t *ids, int64_t top_k,
                           float *y, int64_t ldy, void *workspace, size_t workspace_bytes, qgemm_stream_t stream);

/* ---------------------------------------------------------- PTQ1_0 ----
 * Ternary weights ("cuda: branch-free PTQ1_0 MMQ tile loader ...", llama.cpp
 * PR #214): 28-byte blocks of 128 weights -- 24 qs bytes of 5 base-3 digits
 * each, 2 qh bytes of 4, fp16 d at byte 26.  A byte holds its digits least
 * significant first (digit i = (byte / 3^i) mod 3); digit t means t - 1;
 * weight 24 i + j is digit i of qs byte j (j < 24), weight 120 + r digit r / 2
 * of qh byte r % 2.  w = d * (t - 1).  (The pages give the word layout; the
 * digit order within it is this library's reading, and its oracle is its own
 * codec.)
 * qgemm_ptq1_prepack: N rows of K/128 blocks (row stride ldw bytes, ldw >=
 *   (K/128)*28) -> 32-byte blocks (the same 28 bytes, 4 zero), rows of K/4
 *   bytes, w_packed 16-B aligned, qgemm_ptq1_packed_bytes(N, K) bytes.
 * qgemm_ptq1: Y[M][N] = X_q8k[M][K] * W^T from the repacked weights, K a
 *   multiple of 256; arguments, workspace and errors as qgemm_q4k.  The tile
 *   GEMM runs for every M (d is folded into the fp16 operand exactly).
 *   Accuracy: |Y - Y_exact| <= 2e-5 * sum_b |c_b| + 1e-6. */
QGEMM_API size_t qgemm_ptq1_packed_bytes(int64_t N, int64_t K);
QGEMM_API int qgemm_ptq1_prepack(const void *w, int64_t N, int64_t K, int64_t ldw, void *w_packed,
                                 qgemm_stream_t stream);
QGEMM_API int qgemm_ptq1(const void *w_packed, int64_t N, int64_t K, const int8_t *xqs, const float *xd,
                         const int16_t *xbsums, int64_t M, float *y, int64_t ldy, void *workspace,
                         size_t workspace_bytes, qgemm_stream_t stream);
/* qgemm_ptq1_f32: fp32 X in, Y out, as qgemm_q4k_f32 (the quantizer with the
 * operand planes, then the tile GEMM started under it; every M runs on the tile
 * GEMM, and the workspace is always needed). */
QGEMM_API int qgemm_ptq1_f32(const void *w_packed, int64_t N, int64_t K, const float *x, int64_t ldx, int64_t M,
                             int8_t *qs, float *d, int16_t *bsums, float *y, int64_t ldy, void *workspace,
                             size_t workspace_bytes, qgemm_stream_t stream);
/* qgemm_ptq1_prepared: as qgemm_ptq1 from a workspace that
 * qgemm_quantize_q8k_prep filled for the same X (see the prepared calls). */
QGEMM_API int qgemm_ptq1_prepared(const void *w_packed, int64_t N, int64_t K, const int8_t *xqs, const float *xd,
                                  const int16_t *xbsums, int64_t M, float *y, int64_t ldy, const void *workspace,
                                  size_t workspace_bytes, qgemm_stream_t stream);

/* ------------------------------------------------ output epilogue ----
 * The GEMM with its output epilogue fused into the final store: the output
 * type (the pages' OutT template parameter of the BigTile kernels, vllm.cpp
 * PR #3036 commit 4) and an optional bias and activation:
 *     y[m][n] = out_type( act( acc[m][n] + bias[n] ) )
 * acc the fp32 GEMM result of qgemm_q4k / qgemm_q6k (same accuracy bound);
 * act evaluated in fp32 (ReLU max(v, 0); SiLU v / (1 + exp(-v)); GELU in
 * its erf form 0.5 v (1 + erf(v / sqrt 2))); fp16 / bf16 outputs rounded to
 * nearest even.  epilogue == NULL: fp32 output, no bias, no activation.
 *   out_type     QGEMM_OUT_F32 / _F16 / _BF16: the element type of y.
 *   bias         device fp32 [N], 4-B aligned, or NULL.
 *   y, ldy       y aligned to its element size (4 or 2 bytes); ldy in elements.
 * Other arguments and errors as qgemm_q4k / qgemm_q6k (EINVAL for an unknown
 * out_type or activation, EALIGN for a misaligned bias). */
#define QGEMM_OUT_F32 0
#define QGEMM_OUT_F16 1
#define QGEMM_OUT_BF16 2
#define QGEMM_ACT_NONE 0
#define QGEMM_ACT_RELU 1
#define QGEMM_ACT_SILU 2
#define QGEMM_ACT_GELU 3
typedef struct {
    int out_type;
    int activation;
    const float *bias;
} qgemm_epilogue;
QGEMM_API int qgemm_q4k_ex(const void *w, int64_t N, int64_t K, int64_t ldw, const int8_t *xqs, const float *xd,
                           const int16_t *xbsums, int64_t M, void *y, int64_t ldy, const qgemm_epilogue *epilogue,
                           void *workspace, size_t workspace_bytes, qgemm_stream_t stream);
QGEMM_API int qgemm_q6k_ex(const void *w_packed, int64_t N, int64_t K, const int8_t *xqs, const float *xd,
                           const int16_t *xbsums, int64_t M, void *y, int64_t ldy, const qgemm_epilogue *epilogue,
                           void *workspace, size_t workspace_bytes, qgemm_stream_t stream);

/* -------------------------------------------- allocation-free Q4_K GEMM ----
 * The pages have no counterpart to this call; it serves callers that cannot
 * allocate device memory where they call the GEMM (for example a plugin
 * inside a host framework that owns all device memory and gives the plugin
 * no allocator, or code where cudaMalloc is not allowed, such as a host
 * callback, or not acceptable on a latency-critical path).
 *
 * qgemm_q4k_noalloc computes exactly what qgemm_q4k computes (same
 * arguments minus the workspace) but takes its scratch from a fixed array of
 * QGEMM_NOALLOC_SCRATCH_BYTES bytes that the library keeps in device memory
 * (one per GPU that loads the library, held until the process exits).  It
 * allocates nothing.
 *   - Size limit: qgemm_workspace_bytes(M, N, K) must not exceed
 *     QGEMM_NOALLOC_SCRATCH_BYTES (16 MiB).  The operand copy alone allows
 *     M*K up to about 7.8 million (e.g. M = 512 at K = 11008); grids with
 *     cut tiles add their partial tiles on top (e.g. M = 512, K = 2048,
 *     N = 11008 needs 9.7 MiB on a 152-SM GB300, 2.1 MiB of it the copy).  Larger calls return
 *     QGEMM_EUNSUPPORTED with a message and launch nothing.
 *   - The first call on each device looks up the scratch array's device
 *     address (cudaGetSymbolAddress) with that device current.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents; every byte the GEMM reads is rewritten by the same call, so
 *     nothing needs clearing.  Calls that overlap on the GPU (e.g. on two
 *     streams at once) race on the array: serialize them. */
#define QGEMM_NOALLOC_SCRATCH_BYTES (16u << 20)
QGEMM_API int qgemm_q4k_noalloc(const void *w, int64_t N, int64_t K, int64_t ldw, const int8_t *xqs,
                                const float *xd, const int16_t *xbsums, int64_t M, float *y, int64_t ldy,
                                qgemm_stream_t stream);

/* ------------------------------------------------- expansion check ----
 * Diagnostic for tests: the tile GEMM's weight expansion on its own.  For
 * each of `nblocks` superblock rows it runs the same device functions the
 * GEMM's unpack warps run and writes one QGEMM_DEBUG_EXPAND_BYTES record of
 * 32-bit words to `out` (device, 16-B aligned):
 *   [0, 128)   the fp16 operand pairs of the four K64 chunks (chunk c in words
 *              32c..32c+31; word j holds weights k and k + 2, k = 64c +
 *              4*(j/2) + j%2, low half first) -- Q4_K: sc_j*q*2^-s; Q6_K: the
 *              hi part of sc_j*(q - 32); PTQ1_0: d*(t - 1);
 *   [128, 256) Q6_K: the lo part (hi + lo = sc_j*(q - 32), both exact);
 *   [256, 272) Q4_K: the dmin-correction operands m_j*(-dmin/d)*2^-s as fp16
 *              hi (words 256..263) and lo (264..271) parts, in both halves;
 *              s = clamp(E(dmin) - E(d) - 8, 0, 14), E = floor(log2 |x|);
 *   [272]      the epilogue factor e (fp32): Q4_K d*2^s (dmin when d = 0,
 *              NaN when declined), Q6_K d, PTQ1_0 1;
 *   [273]      bit 0: in range (not declined); bits 8..15: the Q4_K shift s.
 * blocks (device, 16-B aligned): wtype 4 = 144-byte Q4_K blocks; 6 = the
 * 224-byte blocks of qgemm_q6k_prepack; 1 = superblocks of two 32-byte
 * blocks from qgemm_ptq1_prepack.  The pages have no such call (llama.cpp
 * PR #214's review checks its loader by emulating it on 10^4 blocks; this is
 * that check's device side).  Errors: EINVAL, EALIGN, ECUDA. */
#define QGEMM_DEBUG_EXPAND_BYTES 1152
QGEMM_API int qgemm_debug_expand(int wtype, const void *blocks, int64_t nblocks, void *out, qgemm_stream_t stream);

/* ------------------------------------------------------ diagnostics ----
 * Launch counters per path (proof of which kernel ran: the per-variant
 * dispatch counters of PR #3036, commit 4). */
typedef struct {
    uint64_t quantize;     /* qgemm_quantize_q8k launches           */
    uint64_t xprep;        /* operand-preparation launches         */
    uint64_t q4k_tc;       /* Q4_K tensor-core tile GEMM launches   */
    uint64_t q6k_tc;       /* Q6_K tensor-core tile GEMM launches   */
    uint64_t q4k_small;    /* Q4_K small-M streaming launches       */
    uint64_t q6k_small;    /* Q6_K small-M streaming launches       */
    uint64_t q6k_prepack;  /* Q6_K repack launches                  */
    uint64_t split_k;      /* GEMM launches with cut tiles (K parts) */
    uint64_t routed;       /* expert-routed GEMM launches (_id)     */
    uint64_t ptq1_tc;      /* PTQ1_0 tile GEMM launches             */
    uint64_t ptq1_prepack; /* PTQ1_0 repack launches                */
    uint64_t small_fused;  /* small-M launches that quantized X themselves (also counted in q4k/q6k_small) */
    uint64_t q4k_side;     /* Q4_K side-data launches (before the tile GEMM, QGEMM_OPT_Q4K_SIDE_MIN_TILES) */
} qgemm_counters;
QGEMM_API int qgemm_get_counters(qgemm_counters *out);
QGEMM_API int qgemm_reset_counters(void);

/* Device status word of the current device.  Bits: */
#define QGEMM_DEV_TIMEOUT 0x1u   /* a pipeline wait gave up (bounded waits) */
#define QGEMM_DEV_Q4K_RANGE 0x2u /* a Q4_K block row was declined (NaN output): |dmin/d| > 1039*2^14 */
/* (0x4u is not used: Q6_K sub-scales of the whole int8 range are computed) */
#define QGEMM_DEV_BAD_EXPERT 0x8u /* a routed GEMM id was outside [0, E)    */
/* Synchronizes the device, returns the status bits in *bits and the site of
 * the first timed-out wait (0 = none) in *site (may be NULL), then clears
 * both.  Return value: QGEMM_OK when no bit was set; QGEMM_ETIMEOUT when a
 * bounded wait gave up (the kernel stopped early and did not write the
 * affected output tiles: Y is incomplete); QGEMM_EDEVICE when only value
 * checks fired; QGEMM_ECUDA if the device is unusable. */
QGEMM_API int qgemm_get_device_status(uint32_t *bits, uint32_t *site);

/* ----------------------------------------------------------- options ----
 * Process-global knobs, mainly for tests and tuning. */
typedef enum {
    QGEMM_OPT_SMALL_M_MAX = 0,  /* M <= this uses the small-M path: 0 = off, at most 8 (default 8) */
    QGEMM_OPT_FORCE_BM = 1,     /* tokens per CTA for the tile path: 0 = auto, 16/32/64/128 */
    QGEMM_OPT_FORCE_SPLITS = 2, /* split-K factor: 0 = auto, else 1..K/256       */
    /* The limit of every pipeline wait in the kernels, in microseconds (0 =
     * the default of 2 s; at most 10 s).  A wait that runs out records
     * QGEMM_DEV_TIMEOUT and its site, its CTA stops without writing its
     * outputs, and qgemm_get_device_status returns QGEMM_ETIMEOUT.  Read
     * by each call when it launches its kernels (a kernel parameter): it
     * applies to the calls made after it is set, on every device. */
    QGEMM_OPT_WAIT_LIMIT_US = 3,
    /* Test only: make the waits run out without any fault.  1: the tile
     * GEMM's first CTA leaves out its first weight load; 2: the small-M
     * kernel's first CTA issues no weight stage.  The waits behind the left-
     * out copy run out after the wait limit, the CTA's other roles give up
     * at once, and that CTA's output tiles are left unwritten; the other
     * CTAs finish normally.  0 (default): off.  Taken at launch, as above.
     * After a timeout, a workspace filled by qgemm_quantize_q8k_prep must be
     * filled again before another _prepared call (its cut-tile counters may
     * be left nonzero); the other calls prepare their workspace themselves. */
    QGEMM_OPT_TEST_SKIP_ARRIVAL = 4,
    /* Q4_K tile GEMM (not the routed one): the side words of the
     * weight blocks (the dmin-correction operands and scales, which depend
     * on the weights alone) are made by a kernel of their own and loaded by
     * the GEMM when a weight tile meets at least this many token tiles;
     * below that, the GEMM makes them itself.  Y is the same either way.
     * 0 = always the separate kernel; default 4. */
    QGEMM_OPT_Q4K_SIDE_MIN_TILES = 5
} qgemm_option;
QGEMM_API int qgemm_set_option(int option, int64_t value);
QGEMM_API int64_t qgemm_get_option(int option);

/* Profiling hook: if set (non-NULL), every GEMM call records `before` on its
 * stream just before the main GEMM kernel and `after` just after it, so a
 * caller can time that kernel alone.  Pass NULLs to disable. */
QGEMM_API int qgemm_set_profile_events(qgemm_event_t before, qgemm_event_t after);

#ifdef __cplusplus
}
#endif
#endif /* QGEMM_H */
