// internal.h -- declarations shared by the CUDA translation units of the
// library (not installed, not part of the C ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace qg {

// Device status bits (the word lives in qgemm_api.cu; kernels get its address).
enum : uint32_t {
    ST_TIMEOUT = 1u << 0,       // an mbarrier wait gave up (pipeline broken)
    ST_Q4K_RANGE = 1u << 1,     // Q4_K block row declined: |dmin/d| beyond the shifted fp16 range (NaN output)
    // (1u << 2 is not used: Q6_K sub-scales of the whole int8 range are computed exactly)
    ST_BAD_EXPERT = 1u << 3,    // routed GEMM: an expert id outside [0, E) (that row is skipped)
};
// The status array (one per device, 8 words, 8-byte aligned):
//   [0]     OR of the bits above;
//   [1]     1 + the site id of the first wait that timed out (0 = none);
//   [2..7]  not used.
constexpr int ST_WORDS = 8;

// Wait control, handed by value to every kernel with bounded waits (a kernel
// parameter: reading it costs no memory access on the way to the first load):
// the wait limit in microseconds (0 = QG_WAIT_NS), and a test-only switch that
// makes one producer leave out one arrival (ST_SKIP_*; 0 = none) so that the
// bounded waits behind it run out.
struct WaitCfg {
    int limit_us;
    int test_skip;
};
enum : int { ST_SKIP_TILE_WEIGHTS = 1, ST_SKIP_SMALLM_STAGE = 2 };

constexpr uint64_t QG_WAIT_NS = 2000000000ull;  // 2 s of wall time per wait (default)
constexpr uint32_t QG_WAIT_ITERS = 1u << 28;    // and at most this many polls

// Output epilogue (the pages' OutT output type, plus an optional fused bias
// and activation), applied where a kernel stores a finished output element:
//   y = out_type(act(acc + bias[n])).
enum : int { OUT_F32 = 0, OUT_F16 = 1, OUT_BF16 = 2 };
enum : int { ACT_NONE = 0, ACT_RELU = 1, ACT_SILU = 2, ACT_GELU = 3 };
struct Epi {
    int out;             // OUT_*
    int act;             // ACT_*
    const float* bias;   // [N] or nullptr
};

constexpr int Q4K_BLOCK = 144;
constexpr int Q6K_BLOCK = 210;
constexpr int Q6K_PACKED = 224;                 // 210 B + 14 B of zero padding (16-B aligned)
constexpr int PTQ1_BLOCK = 28;                  // 128 ternary weights: 24 B qs, 2 B qh, fp16 d
constexpr int PTQ1_PACKED = 32;                 // 28 B + 4 B of zero padding (16-B aligned)

// ---- kernels' host launchers (each returns cudaError_t of the launch) ----
// With xh != nullptr the same launch also writes the tile GEMM's operand
// planes (as launch_xprep would from its output) and zeroes the split-tile
// counters (TC_COUNTERS ints).  `dependent`: launched as a programmatic
// dependent of the preceding kernel (the Q4_K side-data kernel), which it
// joins before it ends.
cudaError_t launch_quantize_q8k(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs, float* d,
                                int16_t* bsums, cudaStream_t s, __half* xh = nullptr, __half* xbs = nullptr,
                                float* dxT = nullptr, int64_t Mp = 0, int* counters = nullptr, bool dependent = false);

// Q8_K planes -> tensor-core operand planes in the workspace:
//   xh  [M][K] fp16 (the int8 values), xbs [M][K/16] fp16 (bsums),
//   dxT [nb][Mp] fp32 (d transposed, Mp = M rounded up to 4, tail zeroed).
cudaError_t launch_xprep(const int8_t* qs, const float* d, const int16_t* bsums, int64_t M, int64_t K,
                         __half* xh, __half* xbs, float* dxT, int64_t Mp, int* counters, cudaStream_t s,
                         bool dependent = false);

// Expert routing (route.cu) for the routed GEMM (MUL_MAT_ID): the P = M *
// top_k (token, slot) pairs are grouped by expert id.  Each expert's rows
// start on a multiple of 4 (the GEMM loads the transposed scales with TMA,
// whose innermost coordinate must be 16-byte aligned), so there are at most
// P + 3E routed rows, the gaps being padding.  One CTA writes
//   row_off [E + 1]  first routed row of each expert; row_off[E] = total rows;
//   row_end [E]      one past the expert's last row (row_off[e] + its pairs);
//   tile_off[E + 1]  prefix of bm-row token tiles per expert;
//   perm    [rows]   the pair index (token * top_k + slot) of each routed row,
//                    -1 for padding rows,
// and ORs ST_BAD_EXPERT into status for ids outside [0, E) (those pairs get
// no routed row).  The order of the pairs within an expert is not fixed; no
// output value depends on it.
constexpr int ROUTE_MAX_EXPERTS = 1024;
inline int64_t routed_rows_max(int64_t P, int64_t E) { return P + 3 * E; }
cudaError_t launch_route(const int32_t* ids, int64_t P, int E, int bm, int* row_off, int* row_end, int* tile_off,
                         int* perm, uint32_t* status, cudaStream_t s);
// The operand planes of the routed rows: row p of xh / xbs / dxT holds token
// perm[p] / top_k's Q8_K values (as launch_xprep writes them); padding rows
// and rows p >= row_off[E] up to Pp are zero.
cudaError_t launch_xgather(const int8_t* qs, const float* d, const int16_t* bsums, int64_t K, int top_k,
                           const int* perm, const int* rows_valid, int64_t P, __half* xh, __half* xbs, float* dxT,
                           int64_t Pp, cudaStream_t s);

// Work items of the tile GEMM: the first `full_items` tiles (token tiles
// varying fastest) whole, then each remaining tile cut into `parts` K ranges.
// A cut tile's parts write fp32 partial tiles to `partials` (slot = (tile -
// full_items) * parts + part, 128 x bm floats each).  Each of the eight
// epilogue warps owns a fixed slice of the tile and finishes it on its own: it
// bumps `counters[(tile - full_items) * TC_EPI_WARPS + warp]`, and the warp
// that finds the other parts' warps done adds the slice's parts in ascending
// part order, stores Y and resets its counter.  No atomics on Y, and the
// result does not depend on which part finishes last.
struct TcWork {
    int n_tiles, m_tiles;
    // Work order: token tiles in groups of m_group; tile t lies in group
    // t / (m_group * n_tiles), and within a group the token tiles vary
    // fastest.  m_group = m_tiles: one group (token tiles fastest overall).
    int m_group;
    // The work decode's divisions, by m_group * n_tiles, by m_group and by the
    // last group's token-tile count, as a multiply and a shift: q = (n * mul)
    // >> shr with mul = ceil(2^shr / d), shr = 32 + ceil(log2 d), exact for
    // 0 <= n < 2^32 (division by invariant integers, Granlund and Montgomery,
    // PLDI 1994).
    uint64_t dv_gsz_mul, dv_mg_mul, dv_ml_mul;
    int dv_gsz_shr, dv_mg_shr, dv_ml_shr;
    int full_items;       // whole tiles
    int parts;            // K parts of each remaining tile (1: none)
    int items;            // full_items + (tiles - full_items) * parts
    float* partials;
    int* counters;        // TC_MAX_CUT_TILES * TC_EPI_WARPS, zero between calls
    WaitCfg wait;
    // Expert-routed GEMM (experts > 0): the token rows are the routed rows,
    // grouped by expert; the work list is read from device memory (written by
    // the routing kernel that precedes the GEMM).  No cut tiles in this mode.
    int experts;          // E (0: the plain GEMM)
    const int* tile_off;  // [E + 1] prefix of token tiles per expert
    const int* row_off;   // [E + 1] first routed row of each expert (a multiple of 4)
    const int* row_end;   // [E] one past the expert's last routed row
    const int* perm;      // [rows] output row of each routed row
};
constexpr int TC_MAX_CUT_TILES = 1024;   // cut tiles a workspace has counters for
constexpr int TC_EPI_WARPS = 8;          // epilogue warps of the tile GEMM (a counter each per cut tile)
constexpr int TC_COUNTERS = TC_MAX_CUT_TILES * TC_EPI_WARPS;

struct TcLaunch {
    int wtype;            // 4 or 6
    int bm;               // tokens per CTA: 16, 32, 64, 128
    int64_t M, N, K;
    TcWork work;
    int sm_count;         // persistent grid: min(work items, SMs)
    void* y;              // element type per epi.out
    int64_t ldy;          // in elements
    Epi epi;
    uint32_t* status;
    const CUtensorMap* tm_w;    // raw weight blocks, 2D uint8
    const CUtensorMap* tm_xh;   // fp16 [M][K], box {64, bm}, 128B swizzle
    const CUtensorMap* tm_xbs;  // fp16 [M][K/16], box {16, bm}, 32B swizzle (Q4_K only)
    const CUtensorMap* tm_dx;   // fp32 [nb][Mp], box {bm, 1}
    // Q4_K, plain and epilogue variants: the side words of every (row,
    // superblock), made by launch_q4k_side before the GEMM (q4k_side's values:
    // the dmin-correction operands and the scale e), loaded beside the raw
    // blocks; null where the GEMM makes them itself
    const CUtensorMap* tm_side; // uint32 [2 nb][N][8] (superblock b: slabs 2b, 2b+1), box {8, 128, 2}, 32B swizzle
    const CUtensorMap* tm_e;    // fp32 [nb][Np], box {128, 1}
};
// The side words: a1 (slab 2b) and a2 (slab 2b+1) of row n at [slab][n][0..7],
// e at e[b][n] (row stride Np = N rounded up to 4).
cudaError_t launch_q4k_side(const void* w, int64_t N, int64_t nb, int64_t ldw, uint32_t* side, float* e,
                            int64_t Np, cudaStream_t s);
size_t tc_smem_bytes(int wtype, int bm);
cudaError_t tc_prepare(int wtype, int bm);   // sets the dynamic smem attribute (per device)
cudaError_t launch_gemm_tc(const TcLaunch& a, cudaStream_t s);
// (the epilogue instantiations, gemm_tc_epi.cu; launch_gemm_tc dispatches to them)
cudaError_t tc_prepare_epi(int wtype, int bm);
cudaError_t launch_gemm_tc_epi(const TcLaunch& a, cudaStream_t s);
// (Q4_K with the side words made in the kernel, gemm_tc_self.cu and
// gemm_tc_epi_self.cu: a launch without tm_side)
cudaError_t tc_prepare_self(int bm);
cudaError_t launch_gemm_tc_self(const TcLaunch& a, cudaStream_t s);
cudaError_t tc_prepare_epi_self(int bm);
cudaError_t launch_gemm_tc_epi_self(const TcLaunch& a, cudaStream_t s);
// (the routed instantiations, gemm_tc_routed.cu: work.experts > 0)
cudaError_t tc_prepare_routed(int wtype, int bm);
cudaError_t launch_gemm_tc_routed(const TcLaunch& a, cudaStream_t s);

// Small-M streaming path (smallm.cu): M <= SMALL_M_LIMIT tokens, reads the
// Q8_K planes directly (no workspace).
constexpr int SMALL_M_LIMIT = 8;
// The small-M kernel's activations: the Q8_K planes, or (fused: x non-null)
// fp32 X, which the kernel quantizes itself and also stores as Q8_K planes
// (oqs, od, obs).
struct SmallAct {
    const int8_t* xqs;
    const float* xd;
    const int16_t* xbs;
    const float* x;       // fp32 [M][ldx], 16-byte aligned rows (fused)
    int64_t ldx;
    int8_t* oqs;
    float* od;
    int16_t* obs;
};
constexpr int SMALL_FUSED_M_MAX = 2;   // tokens the small-M kernel quantizes itself, at most
struct SmallLaunch {
    int wtype;            // 4 or 6 (Q6_K: the 224-B repacked blocks)
    int64_t M, N, K;
    const void* w;
    int64_t ldw;          // bytes between weight rows (multiple of 16)
    SmallAct act;
    void* y;              // element type per epi.out
    int64_t ldy;          // in elements
    Epi epi;
    int sm_count;
    uint32_t* status;
    WaitCfg wait;
};
bool small_supported(int wtype, int64_t M, int64_t K);
cudaError_t launch_small(const SmallLaunch& a, cudaStream_t s);

// Record a one-line message for qgemm_last_error() and return `code`.
int set_last_error(int code, const char* msg);

// Q8_K planes <-> 292-byte blocks {fp32 d; int8 qs[256]; int16 bsums[16]}
// (4-byte aligned aos), M*K/256 blocks in row-major block order.
constexpr int Q8K_AOS_BLOCK = 292;
cudaError_t launch_q8k_aos(int8_t* qs, float* d, int16_t* bsums, int64_t M, int64_t K, void* aos, bool to_aos,
                           cudaStream_t s);

cudaError_t launch_ptq1_prepack(const uint8_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* out,
                                cudaStream_t s);
cudaError_t launch_q6k_prepack(const uint8_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* out,
                               cudaStream_t s);

}  // namespace qg
