// gemm_tc_kernel.cuh -- Q4_K / Q6_K weights x Q8_K activations on the sm_103a tensor
// cores (tcgen05, TMEM accumulators, TMA-staged operands).
//
// The operation (the pages' prefill quantized matmul, "perf(KERNEL-QUANT-CIQ-
// GEMM-ROCM): cooperative-tile WMMA kernels", vllm.cpp PR #3036, and llama.cpp's
// mul_mat_q as read there, commit 2): Y[m][n] = sum over superblocks b of
//   Q4_K: dx[m,b] * ( d[n,b] * sum_j sc_j * I_j - dmin[n,b] * sum_j m_j * B_j )
//   Q6_K: dx[m,b] * d[n,b] * sum_j sc_j * (I_j - 32 * B_j)
// with I_j the integer dot of sub-block j and B_j the activation sums.
//
// How this kernel computes it on sm_103a (no kind::i8 there):
//   * One CTA owns 128 weight rows (the MMA's M) x BM tokens (the MMA's N)
//     and, with split-K, a range of superblocks.  The lesson the pages arrive
//     at (commit 2 and 4 of PR #3036; the Ampere mmq_x table of llama.cpp
//     PR #214) is that a tile must be loaded once per CTA and shared by all
//     its warps, and that the weight unpack must be amortised over many
//     token rows: here TMA stages each tile once into shared memory and the
//     single MMA-issuing thread feeds the whole tile to the tensor core.
//   * Operands are fp16 holding exact integers: weights as sc_j*q (Q4_K,
//     0..945) or sc_j*(q-32) (Q6_K), tokens as the int8 q (|q| <= 127).
//     Q6_K's int8 sub-scales are split sc = hi + lo with lo in {0, 1} and hi
//     even whenever |sc| > 63, so that both hi*(q-32) (|.| <= 4096, even) and
//     lo*(q-32) are exact fp16 operands; the lo part is a second operand fed
//     into the same accumulator, its MMAs issued only for stages where some
//     row has one.  Products and their fp32 sums are exact while partial sums
//     stay below 2^24, so the tensor core computes the per-superblock integer
//     form sum_j sc_j * I_j.
//   * The Q4_K dmin term rides along as two extra K=16 MMAs per superblock:
//     A = the sub-mins times r = -dmin/d split into two fp16 parts (a1 + a2,
//     about 22 significant bits), B = the 16 bsums in fp16.  The TMEM
//     accumulator then holds  sum_j sc_j I_j - (dmin/d) sum_j m_j B_j  and the
//     epilogue multiplies by d * dx.  (d = 0: the main part is zeroed and the
//     multiplier is dmin with r = -1, exact.  A block with a very large
//     dmin/d runs on a power-of-two shifted scale: unpack.cuh.)
//   * Per superblock the accumulator is read once (tcgen05.ld) and folded
//     into fp32 registers: Y += (S * d) * dx.  Two TMEM accumulators let the
//     MMA of superblock b+1 run while the epilogue drains superblock b.
//
//   * The unpacked weight operand never touches shared memory: each unpack
//     thread builds its row's 64 fp16 values of a K64 chunk in registers and
//     writes them to tensor memory with tcgen05.st; the MMA reads A from TMEM
//     and B (the activations) from TMA-filled shared memory.  Shared-memory
//     stores from the SM's load/store unit compete with TMA writes for the
//     same shared-memory bandwidth (measured on GB300: four warps storing
//     ~60 B/clk halve TMA delivery), so keeping them off the hot path keeps
//     the activation stream fed.
//
// TMEM columns: [0, 2*BM) two fp32 accumulators (superblock t uses t & 1);
// [256, 512) four 64-column stages of the weight operand (K128, or for Q6_K
// K64 hi + K64 lo).  A finished
// tile goes out through the slot of its last superblock's accumulator, which
// is released to the MMA only after that store.
//
// MMA issue is the critical path.  On GB300 a tcgen05.mma (M128 N128 K16)
// holds its issuing thread for ~55 of the ~64 cycles it runs, and the pipe
// keeps only about one more queued, so the barrier waits, commits and loop
// bookkeeping of a single issuing thread leave the tensor pipe idle between
// MMAs (measured: ~35% busy with 4 MMAs per handshake).  Two issuing threads
// in different warps, each owning one of the two accumulators (even / odd
// superblocks), hide each other's bookkeeping; per thread the handshakes are
// K128 (8 MMAs) with a non-blocking look-ahead probe of the next step's
// barriers between the MMAs of the current one.
//
// Warp roles (16 warps for Q4_K, 20 for Q6_K and PTQ1_0, whose heavier
// expansion has a second unpack group; persistent CTAs looping over (n-tile,
// m-tile, split) work items, token tiles varying fastest within a group of
// token tiles that the host sizes so that its activations stay in L2):
//   warp 0      TMA producer of the activation stages (K128 or K256 per stage,
//               one barrier each)
//   warps 1, 3  MMA issuers (one thread each): even / odd superblocks; warp 1
//               also owns the TMEM allocation
//   warp 2      TMA producer: raw weight blocks (+ L2 prefetch ahead) and the
//               per-superblock side data (bsums, dx)
//   warps 4-7   unpack: thread = weight row; branch-free expand of each K64
//               chunk into registers, tcgen05.st into TMEM (Q6_K, PTQ1_0:
//               warps 4-11; PTQ1_0 group g expands K128 step g of each
//               superblock, Q6_K group g the whole superblocks t % 2 == g)
//   last 8      epilogue: warp w reads TMEM lanes 32*(w%4).. and half of the
//               token columns, accumulates Y in registers, stores per tile
//               through TMEM in a rolled loop; for Q4_K the second half also
//               writes each superblock's dmin-correction operands and scale e
// Every wait is bounded (see ptx.cuh); a timeout sets the status word and the
// CTA runs to completion without touching Y.
#pragma once
#include <cuda_fp16.h>

#include "internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"
#include "unpack.cuh"

namespace qg {
namespace {

constexpr int BN = 128;        // weight rows per CTA = MMA M
// Warps: 4 control, 4 or 8 unpack (one or two groups of four), 8 epilogue.
// Q6_K's heavier expansion gets the second unpack group; for Q4_K it did not
// pay for the registers it costs the epilogue (measured on GB300).
template <int WT>
struct Warps {
    static constexpr int UNPACK_GROUPS = WT == 4 ? 1 : 2;
    static constexpr int EPI0 = 4 + 4 * UNPACK_GROUPS;
    static constexpr int N = EPI0 + 8;
    static constexpr int THREADS = 32 * N;
};
constexpr int A_STAGES = 4;    // weight-operand K128 stages in TMEM (64 columns each)
constexpr int A_TMEM_COL = 256;
constexpr int KCH = 64;        // K elements per stage
constexpr int SB_SLOTS = 3;    // per-superblock side-data slots
constexpr int W_PREFETCH = 3;  // raw-weight L2 prefetch distance, in superblocks (3: measured best of 3/6/10)
constexpr int SMEM_LIMIT = 232448;

// warp roles
constexpr int W_PROD_X = 0;
constexpr int W_MMA = 1;
constexpr int W_PROD_W = 2;
constexpr int W_MMA2 = 3;
constexpr int W_UNPACK0 = 4;


__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }
__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }

template <int WT>
struct WTraits;
// RAW_BLOCK: bytes of one weight row's superblock as staged; CORR: the Q4_K
// dmin correction rides along as two extra MMAs; SPLIT: the weight operand
// has a second (lo) part (Q6_K's full int8 sub-scale range), so its stages
// are K64 (hi and lo side by side) instead of K128.
template <>
struct WTraits<4> {
    static constexpr int RAW_BLOCK = Q4K_BLOCK;
    static constexpr bool CORR = true;
    static constexpr bool SPLIT = false;
};
template <>
struct WTraits<6> {
    static constexpr int RAW_BLOCK = Q6K_PACKED;
    static constexpr bool CORR = false;
    static constexpr bool SPLIT = true;
};
// PTQ1_0: a superblock's two 128-weight blocks, each repacked to 32 bytes
template <>
struct WTraits<1> {
    static constexpr int RAW_BLOCK = 2 * PTQ1_PACKED;
    static constexpr bool CORR = false;
    static constexpr bool SPLIT = false;
};

template <int WT, int BM>
struct Layout {
    static constexpr int RAW_SLOTS = 3;
    static constexpr bool CORR = WTraits<WT>::CORR;
    // An activation stage carries SCH K64 boxes that complete on one barrier:
    // a whole superblock for BM <= 64, half of one for BM = 128.  (Measured on
    // GB300: a TMA ring handing over 16 KB per barrier phase delivers about a
    // third of what the same ring moves in 32 KB or 64 KB phases.)
    static constexpr int SCH = BM >= 128 ? 2 : 4;
    static constexpr int SPS = 4 / SCH;                  // stages per superblock
    static constexpr int BOX = BM * 128;                 // one K64 box: BM rows x 128 B
    static constexpr int B_STAGE = SCH * BOX;
    static constexpr int RAW = BN * WTraits<WT>::RAW_BLOCK;
    // per-superblock side slot
    static constexpr int SB_ACORR = 0;                                       // 2 slabs x 128 rows x 32 B
    static constexpr int SB_BCORR = CORR ? 2 * BN * 32 : 0;                 // BM rows x 32 B
    static constexpr int SB_E = SB_BCORR + (CORR ? align_up(BM * 32, 1024) : 0);
    static constexpr int SB_DX = SB_E + BN * 4;
    static constexpr int SB = align_up(SB_DX + BM * 4, 1024);
    // CTA layout: raw ring, side slots, then as many activation stages as fit (even count)
    static constexpr int OFF_RAW = 0;
    static constexpr int OFF_SB = OFF_RAW + align_up(RAW_SLOTS * RAW, 1024);
    static constexpr int OFF_B = OFF_SB + SB_SLOTS * SB;
    static constexpr int RESERVE = 1024 /* base alignment */ + 512 /* barriers, misc */;
    static constexpr int B_STAGES = cmin(12, (SMEM_LIMIT - RESERVE - OFF_B) / B_STAGE) & ~1;
    static constexpr int OFF_BAR = OFF_B + B_STAGES * B_STAGE;
    static constexpr int NBAR = 2 * RAW_SLOTS + 2 * A_STAGES + 2 * B_STAGES + 2 * SB_SLOTS + 4 + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;   // TMEM address, wait control
    static constexpr int OFF_LOFLAG = OFF_MISC + 16;        // per weight-operand stage: a lo part was written
    static constexpr int TOTAL = OFF_LOFLAG + 4 * A_STAGES + 1024;
    static constexpr int CPT = BM / 2;                   // token columns per epilogue thread
    static_assert(2 * BM <= A_TMEM_COL, "accumulators overlap the weight-operand stages");
    static_assert(B_STAGES >= 4, "activation ring too shallow");
    static_assert(NBAR * 8 + 16 + 4 * A_STAGES <= 512, "barrier area");
    static_assert(TOTAL <= SMEM_LIMIT, "shared memory budget");
};


// a[0..3] += (S[0..3] * e) * dx[0..3], two columns per packed fp32 instruction
__device__ __forceinline__ void fold4(float* a, const uint32_t* S, float2 ee, float4 dx) {
    const float2 lo = __ffma2_rn(__fmul2_rn(make_float2(__uint_as_float(S[0]), __uint_as_float(S[1])), ee),
                                 make_float2(dx.x, dx.y), make_float2(a[0], a[1]));
    const float2 hi = __ffma2_rn(__fmul2_rn(make_float2(__uint_as_float(S[2]), __uint_as_float(S[3])), ee),
                                 make_float2(dx.z, dx.w), make_float2(a[2], a[3]));
    a[0] = lo.x;
    a[1] = lo.y;
    a[2] = hi.x;
    a[3] = hi.y;
}


// Kernel variants, each compiled only with the code it needs (measured on
// GB300: routing and epilogue code in one kernel doubled the register
// spills and slowed the plain GEMM by 5-8%):
//   VAR_PLAIN     fp32 output, the work list from the host plan;
//   VAR_EPI       plus the output epilogue (bias, activation, fp16/bf16 output);
//   VAR_ROUTED    the routed GEMM (work list and output rows from the routing);
//   VAR_SELF      VAR_PLAIN for Q4_K with the side words computed in the
//                 kernel rather than loaded (for few token tiles per weight
//                 tile, where each tile's side words are made few times);
//   VAR_EPI_SELF  VAR_EPI for Q4_K with the side words computed in the kernel.
// Q4_K's plain and epilogue variants load the side words (PRE).
enum : int { VAR_PLAIN = 0, VAR_EPI = 1, VAR_ROUTED = 2, VAR_SELF = 3, VAR_EPI_SELF = 4 };
template <int WT, int BM, int VAR>
__global__ void __launch_bounds__(Warps<WT>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_xh,
                   const __grid_constant__ CUtensorMap tm_xbs, const __grid_constant__ CUtensorMap tm_dx,
                   const __grid_constant__ CUtensorMap tm_side, const __grid_constant__ CUtensorMap tm_e,
                   void* __restrict__ y, int64_t ldy, const Epi epi, int M, int N, int nb, const TcWork wk,
                   uint32_t* __restrict__ status) {
    using L = Layout<WT, BM>;
    constexpr int UG = Warps<WT>::UNPACK_GROUPS;
    constexpr int W_EPI0 = Warps<WT>::EPI0;
    constexpr int R = L::RAW_SLOTS;
    constexpr int BS = L::B_STAGES;
    constexpr int SBN = SB_SLOTS;
    // Weight-operand stages: K128 (8 MMAs) per stage.  SPLIT (Q6_K): a K128
    // step's hi part in one stage use and, where some row of the superblock
    // has one, its lo part in the next use, against the same activations.
    constexpr bool SPLIT = WTraits<WT>::SPLIT;
    constexpr int KSTEP = 128;
    constexpr int STEPS = 256 / KSTEP;   // K128 steps per superblock
    // With two-box stages and as many activation stages as weight-operand
    // stages, every K128 step consumes exactly one stage of each ring, so one
    // commit (on a_empty) releases both and the activation producers wait on it.
    constexpr bool MERGED_RELEASE = !SPLIT && (L::SCH == 2) && (BS == A_STAGES);
    // Q4_K, plain and epilogue variants: the side data (dmin-correction
    // operands and the scale e of each row and superblock) depend on the
    // weights alone, so they are made once per call (launch_q4k_side) and
    // loaded by TMA beside the raw block, instead of being recomputed for every
    // token tile (measured on GB300: recomputing them in four epilogue warps
    // cost 2-3% of the plain GEMM at M=8192 K=N=5120, on the sub-partitions the
    // expansion warps need, and 6% of the epilogue GEMM at M=2048 K=4096
    // N=14336).  The self-side and routed variants keep the side-data warps.
    constexpr bool PRE = L::CORR && (VAR == VAR_PLAIN || VAR == VAR_EPI);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + R;
    uint64_t* a_full = raw_empty + R;
    uint64_t* a_empty = a_full + A_STAGES;
    uint64_t* b_full = a_empty + A_STAGES;
    uint64_t* b_empty = b_full + BS;
    uint64_t* sb_full = b_empty + BS;
    uint64_t* sb_empty = sb_full + SBN;
    uint64_t* acc_full = sb_empty + SBN;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain_bar = acc_empty + 2;   // [2]: each MMA thread's last commit, before the CTA ends
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
    // wait control (ptx.cuh): [0] abort flag, [1] wait limit
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
    // SPLIT: word s is nonzero when the stage's current (hi) use is followed by
    // a lo use of the same step (written by the expansion group before its
    // a_full arrivals; read by the issuer after its wait)
    volatile uint32_t* lo_flag = reinterpret_cast<volatile uint32_t*>(smem + L::OFF_LOFLAG);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // routed mode: the work list comes from the preceding (routing) grid
    constexpr bool EPI = VAR == VAR_EPI || VAR == VAR_EPI_SELF;
    constexpr bool ROUTED = VAR == VAR_ROUTED;
    if constexpr (ROUTED) griddep_wait();
    int num_work = wk.items;
    if constexpr (ROUTED) num_work = wk.n_tiles * wk.tile_off[wk.experts];

    auto b_stage = [&](int s) { return smem + L::OFF_B + s * L::B_STAGE; };
    auto raw_slot = [&](int r) { return smem + L::OFF_RAW + r * L::RAW; };
    auto sb_slot = [&](int p) { return smem + L::OFF_SB + p * L::SB; };
    // work item -> (n0, m0, kb0, kb1); token tiles vary fastest (within a group
    // of token tiles, TcWork::m_group), so the CTAs running at the same time
    // share weight tiles (one DRAM read, L2 hits after)
    // (cut tiles: cut = index among the cut tiles, part = its K part; -1 for whole tiles)
    auto work_cut = [&](int wi, int& n0, int& m0, int& kb0, int& kb1, int& cut, int& part) {
        int tile;
        if constexpr (ROUTED) {
            // routed: item = (weight tile, global token tile); token tiles vary
            // fastest; the expert is the one whose tile range holds the token tile
            const int tt = wk.tile_off[wk.experts];
            const int nt = wi / tt, gm = wi - nt * tt;
            int lo = 0, hi = wk.experts - 1;   // largest e with tile_off[e] <= gm
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (wk.tile_off[mid] <= gm) lo = mid; else hi = mid - 1;
            }
            n0 = lo * N + nt * BN;   // weight rows of expert lo, stacked
            m0 = wk.row_off[lo] + (gm - wk.tile_off[lo]) * BM;
            kb0 = 0;
            kb1 = nb;
            cut = -1;
            part = 0;
            return;
        }
        if (wi < wk.full_items) {
            tile = wi;
            cut = -1;
            part = 0;
            kb0 = 0;
            kb1 = nb;
        } else {
            const int j = wi - wk.full_items;
            cut = j / wk.parts;
            part = j - cut * wk.parts;
            tile = wk.full_items + cut;
            // (32-bit: nb * parts < 2^31.  Measured on GB300: the 64-bit forms of
            // these two divisions, decoded in every role's loop, cost 4.7% on
            // Q6_K M=512 K=11008 N=2048 and 9% on Q4_K M=64 K=N=2048.)
            kb0 = nb * part / wk.parts;
            kb1 = nb * (part + 1) / wk.parts;
        }
        // groups of m_group token tiles; within a group, token tiles vary fastest
        // (the CTAs running at once share the group's activations in L2)
        // (the divisions by multiply and shift, TcWork::dv_*)
        const int gsz = wk.m_group * wk.n_tiles;
        const int grp = static_cast<int>((static_cast<uint64_t>(tile) * wk.dv_gsz_mul) >> wk.dv_gsz_shr);
        const int r = tile - grp * gsz;
        const bool full_group = (grp + 1) * wk.m_group <= wk.m_tiles;
        const int gm = full_group ? wk.m_group : wk.m_tiles - grp * wk.m_group;   // token tiles in this group
        const int rq = static_cast<int>((static_cast<uint64_t>(r) * (full_group ? wk.dv_mg_mul : wk.dv_ml_mul)) >>
                                        (full_group ? wk.dv_mg_shr : wk.dv_ml_shr));
        n0 = rq * BN;
        m0 = (grp * wk.m_group + (r - rq * gm)) * BM;
    };
    auto work_of = [&](int wi, int& n0, int& m0, int& kb0, int& kb1) {
        int cut, part;
        work_cut(wi, n0, m0, kb0, kb1, cut, part);
    };
    // The i-th superblock a work item visits: its K range rotated by the weight-
    // tile index, so that the CTAs sharing a token tile at the same time read
    // different activation lines instead of queueing on the same ones.  (The
    // fp32 sum over superblocks is order-independent up to rounding.)
    auto sb_at = [&](int i, int k0, int k1, int n0) {
        const int len = k1 - k0;
        return k0 + (i - k0 + n0 / BN) % len;
    };

    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], 4 * UG + (L::CORR && !PRE ? 4 : 0));   // unpack warps (+ side-data warps)
        }
        for (int s = 0; s < A_STAGES; ++s) {
            mbar_init(&a_full[s], 4);
            mbar_init(&a_empty[s], 1);
        }
        for (int s = 0; s < BS; ++s) {
            mbar_init(&b_full[s], 1);
            mbar_init(&b_empty[s], 1);
        }
        for (int p = 0; p < SBN; ++p) {
            mbar_init(&sb_full[p], PRE ? 1 : 1 + 4);   // producer's bytes (+ the four warps writing the slot)
            mbar_init(&sb_empty[p], 8);   // the epilogue warps, after acc_full covered the MMAs reading it
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(&acc_full[p], 1);
            mbar_init(&acc_empty[p], 8);
        }
        mbar_init(&drain_bar[0], 1);
        mbar_init(&drain_bar[1], 1);
        wait_ctl_init(abort_flag, wk.wait);
        fence_mbar_init();
    }
    if (warp == W_PROD_X && lane == 0) tma_prefetch_desc(&tm_xh);
    if (warp == W_PROD_W && lane == 0) {
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_dx);
        if (L::CORR) tma_prefetch_desc(&tm_xbs);
        if (PRE) {
            tma_prefetch_desc(&tm_side);
            tma_prefetch_desc(&tm_e);
        }
    }
    if (warp == W_MMA) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;


    if (warp == W_PROD_X) {
        // ------------------------------------------------ activation producer
        if (lane == 0) {
            griddep_wait();   // the activation planes come from the preceding grid
            int g = 0;   // running stage counter
            bool ok = true;
            for (int wi = blockIdx.x; wi < num_work && ok; wi += gridDim.x) {
                int n0, m0, kb0, kb1;
                work_of(wi, n0, m0, kb0, kb1);
                for (int i = kb0; i < kb1 && ok; ++i) {
                    const int b = sb_at(i, kb0, kb1, n0);
                    for (int h = 0; h < L::SPS; ++h, ++g) {
                        const int s = g % BS;
                        ok = mbar_wait(MERGED_RELEASE ? &a_empty[s] : &b_empty[s], ((g / BS) & 1) ^ 1, abort_flag,
                                       status, 2);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&b_full[s], L::B_STAGE);
#pragma unroll
                        for (int q = 0; q < L::SCH; ++q)
                            tma_load_2d(&tm_xh, &b_full[s], b_stage(s) + q * L::BOX, b * 256 + KCH * (h * L::SCH + q),
                                        m0);
                    }
                }
            }
        }
    } else if (warp == W_PROD_W) {
        // ------------------------------------------------ weight + side-data producer
        if (lane == 0) {
            int t = 0;
            bool ok = true;
            // Test only (WaitCfg): CTA 0 leaves out its first weight load, so
            // that the waits for it run out and the kernel's timeout path is
            // exercised without any fault.
            const bool skip_first = blockIdx.x == 0 && wk.wait.test_skip == ST_SKIP_TILE_WEIGHTS;
            // L2 prefetch cursor, W_PREFETCH superblocks ahead of the loads.  It
            // starts after the first load, which nothing else then delays (on a
            // short launch that load is on the critical path).
            int pwi = blockIdx.x, pb = 0, pb1 = 0, pn0 = 0, pm0 = 0, pk0 = 0;
            auto prefetch_next = [&](bool issue) {
                if (pwi >= num_work) return;
                if (issue) tma_prefetch_l2_2d(&tm_w, sb_at(pb, pk0, pb1, pn0) * WTraits<WT>::RAW_BLOCK, pn0);
                if (++pb >= pb1) {
                    pwi += gridDim.x;
                    if (pwi < num_work) work_of(pwi, pn0, pm0, pk0, pb1), pb = pk0;
                }
            };
            for (int wi = blockIdx.x; wi < num_work && ok; wi += gridDim.x) {
                int n0, m0, kb0, kb1;
                work_of(wi, n0, m0, kb0, kb1);
                for (int i = kb0; i < kb1; ++i, ++t) {
                    const int b = sb_at(i, kb0, kb1, n0);
                    if (t > 0) prefetch_next(true);
                    const int r = t % R;
                    ok = mbar_wait(&raw_empty[r], ((t / R) & 1) ^ 1, abort_flag, status, 3);
                    if (!ok) break;
                    if (!(skip_first && t == 0)) {
                        mbar_arrive_expect_tx(&raw_full[r], L::RAW);
                        tma_load_2d(&tm_w, &raw_full[r], raw_slot(r), b * WTraits<WT>::RAW_BLOCK, n0);
                    }
                    if (t == 0) {   // the cursor: past superblock 0 (loading), then W_PREFETCH ahead
                        work_of(pwi, pn0, pm0, pk0, pb1);
                        pb = pk0;
                        prefetch_next(false);
                        for (int k = 0; k < W_PREFETCH; ++k) prefetch_next(true);
                    }
                    const int p = t % SBN;
                    ok = mbar_wait(&sb_empty[p], ((t / SBN) & 1) ^ 1, abort_flag, status, 1);
                    if (!ok) break;
                    if (t == 0) griddep_wait();   // bsums and scales come from the preceding grid
                    uint8_t* sb = sb_slot(p);
                    mbar_arrive_expect_tx(&sb_full[p], (L::CORR ? BM * 32 : 0) + BM * 4 + (PRE ? 2 * BN * 32 + BN * 4 : 0));
                    if (L::CORR) tma_load_2d(&tm_xbs, &sb_full[p], sb + L::SB_BCORR, b * 16, m0);
                    tma_load_2d(&tm_dx, &sb_full[p], sb + L::SB_DX, m0, b);
                    if constexpr (PRE) {   // both correction slabs, then the scales e
                        tma_load_3d(&tm_side, &sb_full[p], sb + L::SB_ACORR, 0, n0, 2 * b);
                        tma_load_2d(&tm_e, &sb_full[p], sb + L::SB_E, n0, b);
                    }
                }
            }
        }
    } else if (warp == W_MMA || warp == W_MMA2) {
        // ------------------------------------------------ MMA issuers
        // Thread `par` takes the superblocks t with t % 2 == par, i.e. always
        // accumulator `par`, weight-operand stages 2*par and 2*par+1 and (two-
        // box activation stages) the same two activation stages: every stage
        // barrier is waited on by one thread, phase after phase.  Per
        // superblock: two K128 steps of 8 MMAs (for SPLIT each followed by a lo
        // use of 8 more where the expansion group flagged one), +2 correction
        // MMAs for Q4_K, and the commits; readiness of the next step, the side
        // slot and the next accumulator is probed without blocking between the
        // MMAs of the current step.
        if (lane == 0) {
            const int par = (warp == W_MMA) ? 0 : 1;
            constexpr uint32_t IDESC = idesc_f16_f32(BN, BM);
            // descriptor of activation stage 0; stage s, box q, K-step kk adds (s*B_STAGE + q*BOX + 32*kk) >> 4
            const uint64_t bdesc0 = smem_desc(smem_u32(b_stage(0)), 16, 1024, SWZ_128B);
            // correction operands of side slot 0; slot p adds (p * SB) >> 4
            const uint32_t sb0 = smem_u32(sb_slot(0));
            const uint64_t acorr0 = smem_desc(sb0 + L::SB_ACORR, 16, 256, SWZ_32B);
            const uint64_t bcorr0 = smem_desc(sb0 + L::SB_BCORR, 16, 256, SWZ_32B);
            const uint32_t d_tmem = tmem_base + par * BM;
            // weight-operand stage and phase parity of step h of superblock t:
            // g = 2t + h over the four stages (superblocks of parity par use
            // stages 2par, 2par+1)
            auto a_at = [&](int t, int h, int& s, uint32_t& ph) {
                const int g = 2 * t + h;
                s = g % A_STAGES;
                ph = static_cast<uint32_t>(g / A_STAGES) & 1u;
            };
            // activation stage of step h of superblock t, and the step's first box in it
            auto b_at = [&](int t, int h, int& s, uint32_t& ph, int& q0) {
                const int kk = h * (KSTEP / 64);
                const int g = t * L::SPS + kk / L::SCH;
                s = g % BS;
                ph = static_cast<uint32_t>(g / BS) & 1u;
                q0 = kk % L::SCH;
            };
            int t = 0;
            bool step_ok = false;   // next step's A (and B) stage seen complete
            bool acc_ok = false;    // next superblock's accumulator seen free
            bool ok = true;
            if constexpr (SPLIT) {
                // Q6_K: this thread's superblocks use stages 2par and 2par+1 in
                // turn, one use after another: use u is stage 2par + (u & 1) with
                // phase parity (u >> 1) & 1, and expansion group par counts its
                // uses the same way.  A step's hi use says (lo_flag) whether a lo
                // use follows.
                int u = 0;
                for (int wi = blockIdx.x; wi < num_work && ok; wi += gridDim.x) {
                    int n0, m0, kb0, kb1;
                    work_of(wi, n0, m0, kb0, kb1);
                    for (int b = kb0; b < kb1 && ok; ++b, ++t) {
                        if ((t & 1) != par) continue;
                        ok = mbar_wait(&acc_empty[par], ((t >> 1) & 1) ^ 1, abort_flag, status, 4);
                        if (!ok) break;
                        for (int h = 0; h < STEPS && ok; ++h) {
                            int sx, q0;
                            uint32_t px;
                            b_at(t, h, sx, px, q0);
                            if (q0 == 0) {
                                ok = mbar_wait(&b_full[sx], px, abort_flag, status, 5);
                                if (!ok) break;
                            }
                            const uint64_t bd = bdesc0 + static_cast<uint64_t>((sx * L::B_STAGE + q0 * L::BOX) >> 4);
                            const uint64_t bd1 = bd + (L::BOX >> 4);
                            bool more = true;   // the hi use, then the lo use if flagged
                            for (int part = 0; more; ++part) {
                                const int sa = 2 * par + (u & 1);
                                ok = mbar_wait(&a_full[sa], static_cast<uint32_t>(u >> 1) & 1u, abort_flag, status, 12);
                                if (!ok) break;
                                tc_fence_after();
                                more = part == 0 && lo_flag[sa] != 0u;
                                const uint32_t a0 = tmem_base + A_TMEM_COL + 64 * sa;
                                mma_f16_ta(d_tmem, a0, bd, IDESC, (h | part) != 0);
                                mma_f16_ta(d_tmem, a0 + 8, bd + 2, IDESC, 1u);
                                mma_f16_ta(d_tmem, a0 + 16, bd + 4, IDESC, 1u);
                                mma_f16_ta(d_tmem, a0 + 24, bd + 6, IDESC, 1u);
                                mma_f16_ta(d_tmem, a0 + 32, bd1, IDESC, 1u);
                                mma_f16_ta(d_tmem, a0 + 40, bd1 + 2, IDESC, 1u);
                                mma_f16_ta(d_tmem, a0 + 48, bd1 + 4, IDESC, 1u);
                                mma_f16_ta(d_tmem, a0 + 56, bd1 + 6, IDESC, 1u);
                                mma_commit(&a_empty[sa]);
                                ++u;
                            }
                            if (!ok) break;
                            if (q0 + KSTEP / 64 == L::SCH) mma_commit(&b_empty[sx]);   // the step ends its B stage
                        }
                        if (!ok) break;
                        mma_commit(&acc_full[par]);   // the epilogue then also frees the side slot
                    }
                }
            } else
            for (int wi = blockIdx.x; wi < num_work && ok; wi += gridDim.x) {
                int n0, m0, kb0, kb1;
                work_of(wi, n0, m0, kb0, kb1);
                for (int b = kb0; b < kb1 && ok; ++b, ++t) {
                    if ((t & 1) != par) continue;
                    const int p = t % SBN;
                    if (!acc_ok) {
                        ok = mbar_wait(&acc_empty[par], ((t >> 1) & 1) ^ 1, abort_flag, status, 4);
                        if (!ok) break;
                    }
                    bool sb_ok = !L::CORR;
#pragma unroll
                    for (int h = 0; h < STEPS; ++h) {
                        int sa, sx, q0;
                        uint32_t pa, px;
                        a_at(t, h, sa, pa);
                        b_at(t, h, sx, px, q0);
                        if (!step_ok) {
                            ok = mbar_wait(&a_full[sa], pa, abort_flag, status, 12);
                            if (ok && q0 == 0) ok = mbar_wait(&b_full[sx], px, abort_flag, status, 5);
                            if (!ok) break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = tmem_base + A_TMEM_COL + 64 * sa;
                        const uint64_t bd = bdesc0 + static_cast<uint64_t>((sx * L::B_STAGE + q0 * L::BOX) >> 4);
                        mma_f16_ta(d_tmem, a0, bd, IDESC, h != 0);
                        mma_f16_ta(d_tmem, a0 + 8, bd + 2, IDESC, 1u);
                        mma_f16_ta(d_tmem, a0 + 16, bd + 4, IDESC, 1u);
                        mma_f16_ta(d_tmem, a0 + 24, bd + 6, IDESC, 1u);
                        // probes, while these run: this thread's next step is step h + 1
                        // of superblock t, or step 0 of superblock t + 2
                        const bool last_b = (q0 + KSTEP / 64 == L::SCH);   // this step ends its B stage
                        {
                            const int nt = h + 1 < STEPS ? t : t + 2, nh = (h + 1) % STEPS;
                            int na, nx, nq;
                            uint32_t npa, npx;
                            a_at(nt, nh, na, npa);
                            b_at(nt, nh, nx, npx, nq);
                            const bool ta = mbar_test_wait(&a_full[na], npa);
                            const bool tb = (nq != 0) || mbar_test_wait(&b_full[nx], npx);
                            if (h == 0 && L::CORR) sb_ok = mbar_test_wait(&sb_full[p], (t / SBN) & 1);
                            if (h == STEPS - 1) acc_ok = mbar_test_wait(&acc_empty[par], (((t + 2) >> 1) & 1) ^ 1);
                            step_ok = ta && tb;
                        }
                        {
                            const uint64_t bd1 = bd + (L::BOX >> 4);
                            mma_f16_ta(d_tmem, a0 + 32, bd1, IDESC, 1u);
                            mma_f16_ta(d_tmem, a0 + 40, bd1 + 2, IDESC, 1u);
                            mma_f16_ta(d_tmem, a0 + 48, bd1 + 4, IDESC, 1u);
                            mma_f16_ta(d_tmem, a0 + 56, bd1 + 6, IDESC, 1u);
                        }
                        // frees the A stage (and, with MERGED_RELEASE, the B stage of this step)
                        mma_commit(&a_empty[sa]);
                        if (last_b && !MERGED_RELEASE) mma_commit(&b_empty[sx]);
                    }
                    if (!ok) break;
                    if (L::CORR) {
                        if (!sb_ok) {
                            ok = mbar_wait(&sb_full[p], (t / SBN) & 1, abort_flag, status, 6);
                            if (!ok) break;
                        }
                        tc_fence_after();
                        const uint64_t po = static_cast<uint64_t>((p * L::SB) >> 4);
                        mma_f16(d_tmem, acorr0 + po, bcorr0 + po, IDESC, 1u);
                        mma_f16(d_tmem, acorr0 + po + ((BN * 32) >> 4), bcorr0 + po, IDESC, 1u);
                    }
                    // completion of everything so far: the epilogue then also frees side slot p
                    mma_commit(&acc_full[par]);
                }
            }
            // every MMA this thread issued has completed before the CTA frees TMEM
            mma_commit(&drain_bar[par]);
            mbar_wait_drain(&drain_bar[par], 0, abort_flag);
        }
    } else if (warp >= W_UNPACK0 && warp < W_EPI0) {
        // ------------------------------------------------ unpack (thread = weight row)
        // One or two groups of four warps (TMEM lanes 32*(warp%4).., as any
        // warp must).  Q4_K: one group.  PTQ1_0: group g expands K128 step g
        // of every superblock; group 0 also writes the superblock's side data.
        // Q6_K (SPLIT): group g owns the superblocks t with t % 2 == g -- the
        // same ones as MMA thread g -- and expands both K128 steps of each, hi
        // parts and (where needed) lo parts, into stages 2g and 2g+1 in turn,
        // writing its side data too.
        const int grp = (warp - W_UNPACK0) >> 2;
        const int j0 = UG == 2 ? grp : 0, j1 = UG == 2 ? grp + 1 : 2;   // this warp's K128 steps
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const uint32_t lane_base = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + A_TMEM_COL;
        // A K128 step's a_full is signalled only after the next chunk has been
        // expanded, so the wait for its tcgen05.st to land overlaps that work;
        // it is signalled at once before any wait that might block.
        int pend = -1;   // A stage whose a_full is still to be signalled
        auto signal = [&]() {
            if (pend >= 0) {
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[pend]);
                pend = -1;
            }
        };
        int u = 0;   // (SPLIT) this group's stage uses, as MMA thread grp counts them
        int t = 0;
        bool ok = true;
        for (int wi = blockIdx.x; wi < num_work && ok; wi += gridDim.x) {
            int n0, m0, kb0, kb1;
            work_of(wi, n0, m0, kb0, kb1);
            for (int b = kb0; b < kb1; ++b, ++t) {
                const int r = t % R;
                if (!mbar_test_wait(&raw_full[r], (t / R) & 1)) signal();
                ok = mbar_wait(&raw_full[r], (t / R) & 1, abort_flag, status, 7);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                const uint8_t* blk = raw_slot(r) + row * WTraits<WT>::RAW_BLOCK;
                const int p = t % SBN;

                if constexpr (WT == 4) {
                    const Q4kScales qs4 = q4k_scales(*reinterpret_cast<const uint4*>(blk));
                    if (qs4.declined) atomicOr(status, ST_Q4K_RANGE);   // (its outputs become NaN)
                    // (the dmin correction operands and the scale e of this superblock
                    // are written by the epilogue's side-data warps)
                    // this warp's K128 steps: the second chunk is expanded while the
                    // first one's tcgen05.st is in flight, one wait::st and one a_full
#pragma unroll 1
                    for (int j = j0; j < j1; ++j) {
                        const int g = 2 * t + j;
                        const int s = g % A_STAGES;
                        // sub-block scales of chunks 2j (bytes 0, 1) and 2j+1 (bytes 2, 3)
                        const uint32_t scw = j == 0 ? qs4.sc03 : qs4.sc47;
                        uint32_t v0[32], v1[32];
                        q4k_expand<0>(blk, 2 * j, scw, qs4, v0);
                        signal();
                        ok = mbar_wait(&a_empty[s], ((g / A_STAGES) & 1) ^ 1, abort_flag, status, 9);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                        tc_fence_after();
                        tmem_st_32x32b_x32(lane_base + 64 * s, v0);
                        q4k_expand<1>(blk, 2 * j + 1, scw, qs4, v1);
                        tmem_st_32x32b_x32(lane_base + 64 * s + 32, v1);
                        pend = s;
                    }
                    if (!ok) break;
                } else if constexpr (WT == 1) {
                    // PTQ1_0: the scale d is folded into the operand (an exact fp16
                    // product), so the superblock's epilogue factor e is 1
                    if (grp == 0) {
                        if (!mbar_test_wait(&sb_empty[p], ((t / SBN) & 1) ^ 1)) signal();
                        ok = mbar_wait(&sb_empty[p], ((t / SBN) & 1) ^ 1, abort_flag, status, 8);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                        reinterpret_cast<float*>(sb_slot(p) + L::SB_E)[row] = 1.0f;
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sb_full[p]);
                    }
                    // this warp's K128 steps: step j is block j of the superblock
#pragma unroll 1
                    for (int j = j0; j < j1; ++j) {
                        const int g = 2 * t + j;
                        const int s = g % A_STAGES;
                        Ptq1State pst;
                        uint32_t v0[32], v1[32];
                        unpack_ptq1_lo(blk + PTQ1_PACKED * j, pst, v0);
                        signal();
                        ok = mbar_wait(&a_empty[s], ((g / A_STAGES) & 1) ^ 1, abort_flag, status, 9);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                        tc_fence_after();
                        tmem_st_32x32b_x32(lane_base + 64 * s, v0);
                        unpack_ptq1_hi(pst, v1);
                        tmem_st_32x32b_x32(lane_base + 64 * s + 32, v1);
                        pend = s;
                    }
                    if (!ok) break;
                } else {
                    // Q6_K.  The other group's superblock: only its raw slot's phase.
                    if ((t & 1) != grp) {
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&raw_empty[r]);
                        continue;
                    }
                    // sub-block scales split into exact hi and lo parts (q6k_split)
                    const uint4 scv = *reinterpret_cast<const uint4*>(blk + 192);
                    // Does step j need a lo use?  Yes if any of the CTA's 128 rows has a
                    // lo part among the step's eight sub-block scales (every warp of the
                    // group reads them all and decides alike).
                    bool lo_step[2];
                    {
                        uint32_t need0 = 0u, need1 = 0u;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint4 sv = *reinterpret_cast<const uint4*>(raw_slot(r) + (lane + 32 * k) *
                                                                             WTraits<WT>::RAW_BLOCK + 192);
                            uint32_t h0, l0, l1, l2, l3;
                            q6k_split(sv.x, h0, l0);
                            q6k_split(sv.y, h0, l1);
                            q6k_split(sv.z, h0, l2);
                            q6k_split(sv.w, h0, l3);
                            need0 |= l0 | l1;
                            need1 |= l2 | l3;
                        }
                        lo_step[0] = __any_sync(0xffffffffu, need0 != 0u);
                        lo_step[1] = __any_sync(0xffffffffu, need1 != 0u);
                    }
                    {
                        const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
                        if (!mbar_test_wait(&sb_empty[p], ((t / SBN) & 1) ^ 1)) signal();
                        ok = mbar_wait(&sb_empty[p], ((t / SBN) & 1) ^ 1, abort_flag, status, 8);
                        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                        reinterpret_cast<float*>(sb_slot(p) + L::SB_E)[row] = d;
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sb_full[p]);
                    }
                    // step j: chunks 2j and 2j+1, the hi parts in one stage use, then the
                    // lo parts (zero for rows without one) in the next if lo_step[j]
#pragma unroll 1
                    for (int j = 0; j < 2 && ok; ++j) {
                        const uint32_t sw0 = j == 0 ? scv.x : scv.z, sw1 = j == 0 ? scv.y : scv.w;
                        uint32_t slo0, slo1, v[32];
                        const int nuse = lo_step[j] ? 2 : 1;
                        for (int use = 0; use < nuse; ++use) {
                            if (use == 0)
                                q6k_expand_hi(blk, 2 * j, sw0, slo0, v);
                            else
                                q6k_expand_lo(blk, 2 * j, slo0, v);
                            signal();
                            const int s = 2 * grp + (u & 1);
                            ok = mbar_wait(&a_empty[s], ((u >> 1) & 1) ^ 1, abort_flag, status, 9);
                            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                            tc_fence_after();
                            tmem_st_32x32b_x32(lane_base + 64 * s, v);
                            if (use == 0)
                                q6k_expand_hi(blk, 2 * j + 1, sw1, slo1, v);
                            else
                                q6k_expand_lo(blk, 2 * j + 1, slo1, v);
                            tmem_st_32x32b_x32(lane_base + 64 * s + 32, v);
                            if (quad == 0 && lane == 0) lo_flag[s] = (use == 0 && nuse == 2) ? 1u : 0u;
                            pend = s;
                            ++u;
                        }
                    }
                    if (!ok) break;
                    signal();   // the superblock's last stage now: the other group's superblock comes next
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&raw_empty[r]);
            }
        }
        signal();
    } else if (warp >= W_EPI0) {
        // ------------------------------------------------ epilogue
        constexpr int CPT = L::CPT;
        // The tile's store goes through TMEM (see below).  Not for the routed
        // variant: there it raised the spills of the per-superblock loop from
        // 8 to 204 B and slowed the 8-expert M=512 K=4096 N=14336 call from
        // 231 to 308 us (measured on GB300).
        constexpr bool STAGED = CPT >= 32 && !ROUTED;
        const int quad = warp & 3;
        const int half = (warp - W_EPI0) >> 2;
        const int row = 32 * quad + lane;
        const int col0 = half * CPT;
        int t = 0;
        bool ok = true;
        // Q4_K: the second half's four warps also write the side data of each
        // superblock (the dmin correction operands and the scale e, from the
        // block header in the raw ring), SBN - 1 superblocks ahead of the
        // accumulator they wait for, while the unpack warps only expand.
        const bool side_writer = L::CORR && !PRE && half == 1;
        int ts = 0;         // next superblock whose side data is due
        int total_sb = 0;   // this CTA's superblocks
        if (side_writer) {
            for (int wi = blockIdx.x; wi < num_work; wi += gridDim.x) {
                int n0, m0, kb0, kb1, cut, part;
                work_cut(wi, n0, m0, kb0, kb1, cut, part);
                total_sb += kb1 - kb0;
            }
        }
        auto side_upto = [&](int lim) -> bool {
            for (; ts <= lim && ts < total_sb; ++ts) {
                const int r = ts % R, ps = ts % SBN;
                bool fine = mbar_wait(&raw_full[r], (ts / R) & 1, abort_flag, status, 15);
                if (!__all_sync(0xffffffffu, fine)) return false;
                const uint4 hdr = *reinterpret_cast<const uint4*>(raw_slot(r) + row * WTraits<WT>::RAW_BLOCK);
                __syncwarp();
                if (lane == 0) mbar_arrive(&raw_empty[r]);
                fine = mbar_wait(&sb_empty[ps], ((ts / SBN) & 1) ^ 1, abort_flag, status, 16);
                if (!__all_sync(0xffffffffu, fine)) return false;
                uint8_t* sbw = sb_slot(ps);
                // e and the correction operands, on the scale 2^-s the unpack uses
                // (q4k_side), each word stored as it is made (few live registers
                // beside the accumulators); a row out of even the shifted range gets
                // e = NaN: its outputs are declined, visibly, rather than computed
                // wrongly (the unpack records the status bit).  Correction slabs,
                // 32-byte swizzle: word j of a row at
                // row * 32 + ((j / 4) ^ ((row >> 2) & 1)) * 16 + (j % 4) * 4.
                uint32_t* s1 = reinterpret_cast<uint32_t*>(sbw + L::SB_ACORR + row * 32);
                uint32_t* s2 = s1 + BN * 8;
                const int x = (row >> 2) & 1;
                float e;
                q4k_side(hdr, e, [&](int j, uint32_t w1, uint32_t w2) {
                    const int o = (((j >> 2) ^ x) << 2) + (j & 3);
                    s1[o] = w1;
                    s2[o] = w2;
                });
                reinterpret_cast<float*>(sbw + L::SB_E)[row] = e;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sb_full[ps]);
            }
            return true;
        };
        for (int wi = blockIdx.x; wi < num_work && ok; wi += gridDim.x) {
            int n0, m0, kb0, kb1, cut, part;
            work_cut(wi, n0, m0, kb0, kb1, cut, part);
            float acc[CPT];
#pragma unroll
            for (int j = 0; j < CPT; ++j) acc[j] = 0.0f;
            float bias_n = 0.0f;   // (epilogue variant) loaded now, used at the tile's store
            if constexpr (EPI) {
                if (epi.bias && n0 + row < N) bias_n = epi.bias[n0 + row];
            }
            for (int b = kb0; b < kb1; ++b, ++t) {
                const int buf = t & 1;
                const int p = t % SBN;
                if (side_writer && !side_upto(t + SBN - 1)) { ok = false; break; }
                ok = mbar_wait(&acc_full[buf], (t >> 1) & 1, abort_flag, status, 10);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                ok = mbar_wait(&sb_full[p], (t / SBN) & 1, abort_flag, status, 11);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                const uint8_t* sb = sb_slot(p);
                const float e = reinterpret_cast<const float*>(sb + L::SB_E)[row];
                const float2 ee = make_float2(e, e);
                const float4* dx4 = reinterpret_cast<const float4*>(sb + L::SB_DX) + col0 / 4;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + buf * BM + col0;
                if constexpr (CPT >= 16 && UG == 1 && (PRE || !L::CORR) && !ROUTED) {
                    // one 16-column load per wait (measured on GB300: two in flight per
                    // wait cost 32 more live registers and 3.6% on M=2048 K=4096 N=14336)
                    constexpr int PAIR = 1;
#pragma unroll
                    for (int ch = 0; ch < CPT / 16; ch += PAIR) {
                        uint32_t v[PAIR][16];
#pragma unroll
                        for (int u = 0; u < PAIR; ++u) tmem_ld_32x32b_x16(taddr + 16 * (ch + u), v[u]);
                        tmem_ld_wait();
#pragma unroll
                        for (int u = 0; u < PAIR; ++u) {
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4)
                                fold4(acc + 16 * (ch + u) + 4 * q4, v[u] + 4 * q4, ee, dx4[4 * (ch + u) + q4]);
                        }
                    }
                } else {
                    // 8-column loads where registers are short: the kernels with two
                    // expansion groups run at 96 registers, and the Q4_K variants with
                    // the side-data writer or the routed decode hold more beside the 64
                    // accumulators; 16 columns in flight spilled there (measured on
                    // GB300, Y bit-identical: Q6_K M=512 K=11008 N=2048 136 B of spill
                    // stores -> 40 B, 50.8 -> 47.0 us; PTQ1_0 M=2048 K=N=5120 149.3 ->
                    // 140.0 us; routed Q4_K 36 B -> 0, MoE 8 experts 225.7 -> 220.1 us)
#pragma unroll
                    for (int ch = 0; ch < CPT / 8; ++ch) {
                        uint32_t v[8];
                        tmem_ld_32x32b_x8(taddr + 8 * ch, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int q4 = 0; q4 < 2; ++q4)
                            fold4(acc + 8 * ch + 4 * q4, v + 4 * q4, ee, dx4[2 * ch + q4]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                // (STAGED: the item's last accumulator is released after the tile's store)
                const bool hold = STAGED && b == kb1 - 1;
                if (lane == 0) {
                    if (!hold) mbar_arrive(&acc_empty[buf]);
                    mbar_arrive(&sb_empty[p]);
                }
            }
            if (!ok) break;
            const int hbuf = (t - 1) & 1;   // the accumulator of the item's last superblock
            auto release_held = [&]() {
                if constexpr (STAGED) {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&acc_empty[hbuf]);
                }
            };
            if (cut >= 0) {
                griddep_wait();   // the counters are zeroed by the preceding grid
                // A part of a cut tile.  Each epilogue warp finishes its own slice
                // of the tile (TMEM lanes 32*quad.., token columns col0..) with no
                // other warp: it publishes its partial slice, bumps the slice's
                // counter, and the warp that completes the slice adds all parts in
                // ascending part order.  (A part's element (row, col) sits at
                // col*128 + row: each warp-wide store or load is one 128-B line.)
                int* ctr = wk.counters + cut * TC_EPI_WARPS + (warp - W_EPI0);
                float* mine = wk.partials + (static_cast<int64_t>(cut) * wk.parts + part) * (BN * BM) +
                              col0 * BN + row;
#pragma unroll
                for (int j = 0; j < CPT; ++j) __stcg(mine + j * BN, acc[j]);
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = atomicAdd(ctr, 1) == wk.parts - 1;
                if (!__shfl_sync(0xffffffffu, last, 0)) {
                    release_held();
                    continue;
                }
                __threadfence();
                const float* base = wk.partials + static_cast<int64_t>(cut) * wk.parts * (BN * BM) + col0 * BN + row;
                if constexpr (CPT <= 32) {
                    // this part's own values from registers, the others from memory
                    float sum[CPT];
#pragma unroll
                    for (int j = 0; j < CPT; ++j) sum[j] = part == 0 ? acc[j] : __ldcg(base + j * BN);
                    for (int p2 = 1; p2 < wk.parts; ++p2) {
                        if (p2 == part) {
#pragma unroll
                            for (int j = 0; j < CPT; ++j) sum[j] += acc[j];
                        } else {
#pragma unroll
                            for (int j = 0; j < CPT; ++j) sum[j] += __ldcg(base + p2 * (BN * BM) + j * BN);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < CPT; ++j) acc[j] = sum[j];
                } else {
                    // all parts, this one included, from memory
#pragma unroll
                    for (int j = 0; j < CPT; ++j) acc[j] = __ldcg(base + j * BN);
                    for (int p2 = 1; p2 < wk.parts; ++p2) {
#pragma unroll
                        for (int j = 0; j < CPT; ++j) acc[j] += __ldcg(base + p2 * (BN * BM) + j * BN);
                    }
                }
                __syncwarp();
                if (lane == 0) *ctr = 0;   // ready for the next call
            }
            if constexpr (STAGED) {
                // The finished tile goes out through the TMEM slot of the item's
                // last accumulator: two stores, then a rolled loop over column
                // chunks.  (Measured on GB300: the 64-way unrolled store is
                // several KB of code run once per tile; cold in the instruction
                // cache it held every role behind the epilogue ~3 us per tile.)
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + hbuf * BM + col0;
#pragma unroll
                for (int h = 0; h < CPT / 32; ++h) {
                    uint32_t r[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(acc[32 * h + j]);
                    tmem_st_32x32b_x32(taddr + 32 * h, r);
                }
                tmem_st_wait();
                const int n = n0 + row;
                const bool live = !*abort_flag && n < N;
                float bn = 0.0f;
                if constexpr (EPI) bn = bias_n;
                // Without an activation (the plain variant, and the epilogue
                // variant's bias and output-type forms) in chunks of 32 columns,
                // each element at most one add and one converting store; with an
                // activation in chunks of 8, the activation unrolled over the
                // chunk.  This code runs once per tile, cold in the instruction
                // cache, so its size is much of its cost: measured on GB300 (M=2048
                // K=4096 N=14336, bias and bf16 output), every form on the 8-column
                // path took 292.9 us, the no-activation forms on this one 256.0 us
                // (plain fp32: 241.7 us); 32-column chunks also took 2% off the
                // plain GEMM against 8.
                constexpr int CH = CPT < 32 ? CPT : 32;
                const bool add_bias = EPI && epi.bias != nullptr;
                if (!EPI || epi.act == ACT_NONE) {
#pragma unroll 1
                    for (int c = 0; c < CPT; c += CH) {
                        uint32_t v[CH];
                        __syncwarp();   // (the TMEM load is warp-collective: every lane, converged)
                        if constexpr (CH == 32)
                            tmem_ld_32x32b_x32(taddr + c, v);
                        else
                            tmem_ld_32x32b_x8(taddr + c, v);
                        tmem_ld_wait();
                        const int mc = m0 + col0 + c;
                        if (live) {
                            if (!EPI || epi.out == OUT_F32) {
                                float* yp = static_cast<float*>(y) + static_cast<int64_t>(mc) * ldy + n;
#pragma unroll
                                for (int u = 0; u < CH; ++u) {
                                    const float a = __uint_as_float(v[u]);
                                    if (mc + u < M) *yp = add_bias ? a + bn : a;
                                    yp += ldy;
                                }
                            } else {
                                // fp16 or bf16, stored as their 16-bit patterns
                                const bool f16 = epi.out == OUT_F16;
                                unsigned short* yp =
                                    static_cast<unsigned short*>(y) + static_cast<int64_t>(mc) * ldy + n;
#pragma unroll
                                for (int u = 0; u < CH; ++u) {
                                    const float a = add_bias ? __uint_as_float(v[u]) + bn : __uint_as_float(v[u]);
                                    const unsigned short h = f16 ? __half_as_ushort(__float2half_rn(a))
                                                                 : __bfloat16_as_ushort(__float2bfloat16_rn(a));
                                    if (mc + u < M) *yp = h;
                                    yp += ldy;
                                }
                            }
                        }
                    }
                } else if constexpr (EPI) {
                    constexpr int CA = 8;
#pragma unroll 1
                    for (int c = 0; c < CPT; c += CA) {
                        uint32_t v[CA];
                        __syncwarp();
                        tmem_ld_32x32b_x8(taddr + c, v);
                        tmem_ld_wait();
                        const int mc = m0 + col0 + c;
                        if (live) {
                            float vv[CA];
#pragma unroll
                            for (int u = 0; u < CA; ++u) vv[u] = __uint_as_float(v[u]);
                            epi_tile<CA>(vv, epi, bn, y, ldy, n, mc, M);
                        }
                    }
                }
                release_held();
                continue;
            }
            if constexpr (ROUTED) {
                // routed: column n of the expert, token rows up to the expert's end,
                // each written to its output row
                const int e = n0 / N;
                const int n = n0 - e * N + row;
                const int m_end = wk.row_end[e];
                if (!*abort_flag && n < N) {
                    if constexpr (!EPI) {
                        float* yf = static_cast<float*>(y);
#pragma unroll
                        for (int j = 0; j < CPT; ++j) {
                            const int m = m0 + col0 + j;
                            if (m < m_end) yf[static_cast<int64_t>(wk.perm[m]) * ldy + n] = acc[j];
                        }
                    } else {
                        const float bn = epi.bias ? epi.bias[n] : 0.0f;
#pragma unroll
                        for (int j = 0; j < CPT; ++j) {
                            const int m = m0 + col0 + j;
                            if (m < m_end)
                                epi_store(y, static_cast<int64_t>(wk.perm[m]) * ldy + n,
                                          epi_value(acc[j], bn, epi.act), epi.out);
                        }
                    }
                }
                continue;
            }
            const int n = n0 + row;
            if (!*abort_flag && n < N) {
                if constexpr (!EPI) {
                    float* yf = static_cast<float*>(y);
#pragma unroll
                    for (int j = 0; j < CPT; ++j) {
                        const int m = m0 + col0 + j;
                        if (m < M) yf[static_cast<int64_t>(m) * ldy + n] = acc[j];
                    }
                } else {
                    epi_tile<CPT>(acc, epi, bias_n, y, ldy, n, m0 + col0, M);
                }
            }
        }
    }

    settle_after_abort(abort_flag);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_MMA) {
        __syncwarp();
        tmem_dealloc(tmem_base, 512);
    }
}

template <int WT, int BM, int VAR>
cudaError_t launch_t(const TcLaunch& a, cudaStream_t s) {
    using L = Layout<WT, BM>;
    const int grid = a.work.items < a.sm_count ? a.work.items : a.sm_count;
    // A programmatic dependent of the preceding kernel: the CTAs may start
    // (barrier set-up, weight loads and expansion) while that kernel finishes;
    // every read of its output waits for it (griddep_wait).
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(Warps<WT>::THREADS);
    cfg.dynamicSmemBytes = L::TOTAL;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const CUtensorMap tm_xbs = a.tm_xbs ? *a.tm_xbs : *a.tm_xh;
    const CUtensorMap tm_side = a.tm_side ? *a.tm_side : *a.tm_xh;   // (read only where the side words are loaded)
    const CUtensorMap tm_e = a.tm_e ? *a.tm_e : *a.tm_xh;
    if (L::CORR && (VAR == VAR_PLAIN || VAR == VAR_EPI) && (!a.tm_side || !a.tm_e)) return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<WT, BM, VAR>, *a.tm_w, *a.tm_xh, tm_xbs, *a.tm_dx, tm_side, tm_e,
                              a.y, a.ldy, a.epi,
                              static_cast<int>(a.M), static_cast<int>(a.N), static_cast<int>(a.K / 256), a.work,
                              a.status);
}

template <int WT, int BM, int VAR>
cudaError_t prepare_t() {
    return cudaFuncSetAttribute(gemm_tc_kernel<WT, BM, VAR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Layout<WT, BM>::TOTAL);
}

}  // namespace
}  // namespace qg
