// gemm_tc.cu -- Q4_K / Q6_K weights x Q8_K activations on the sm_103a tensor
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
//     0..945) or sc_j*(q-32) (Q6_K, |.| <= 2048 for |sc_j| <= 64), tokens as
//     the int8 q (|q| <= 127).  Products and their fp32 sums are exact while
//     partial sums stay below 2^24, so the tensor core computes the per-
//     superblock integer form sum_j sc_j * I_j.
//   * The Q4_K dmin term rides along as two extra K=16 MMAs per superblock:
//     A = the sub-mins times r = -dmin/d split into two fp16 parts (a1 + a2,
//     about 22 significant bits), B = the 16 bsums in fp16.  The TMEM
//     accumulator then holds  sum_j sc_j I_j - (dmin/d) sum_j m_j B_j  and the
//     epilogue multiplies by d * dx.  (d = 0: the main part is zeroed and the
//     multiplier is dmin with r = -1, exact.)
//   * Per superblock the accumulator is read once (tcgen05.ld) and folded
//     into fp32 registers: Y += (S * d) * dx.  Two TMEM accumulators let the
//     MMA of superblock b+1 run while the epilogue drains superblock b.
//
// Warp roles (512 threads):
//   warp 0      TMA producer: activation K-chunks and per-superblock side data
//   warp 1      TMEM owner + MMA issuer (one thread)
//   warp 2      TMA producer: raw weight blocks
//   warp 3      idle
//   warps 4-7   unpack: thread t expands weight row t of the tile into the
//               128B-swizzled K-major fp16 operand, branch-free
//   warps 8-15  epilogue: warp w reads TMEM lanes 32*(w%4).. and half of the
//               token columns, accumulates Y in registers, stores at the end
// Every wait is bounded (see ptx.cuh); a timeout sets the status word and the
// CTA runs to completion without touching Y.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace qg {
namespace {

constexpr int BN = 128;        // weight rows per CTA = MMA M
constexpr int NTHREADS = 512;
constexpr int STAGES = 4;      // K64 operand stages
constexpr int KCH = 64;        // K elements per stage (one 128-byte swizzle row of fp16)

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int WT>
struct WTraits;
template <>
struct WTraits<4> {
    static constexpr int RAW_BLOCK = Q4K_BLOCK;
    static constexpr int RAW_SLOTS = 3;
    static constexpr bool CORR = true;
};
template <>
struct WTraits<6> {
    static constexpr int RAW_BLOCK = Q6K_PACKED;
    static constexpr int RAW_SLOTS = 2;
    static constexpr bool CORR = false;
};

template <int WT, int BM>
struct Layout {
    static constexpr int RAW_SLOTS = WTraits<WT>::RAW_SLOTS;
    static constexpr bool CORR = WTraits<WT>::CORR;
    static constexpr int A_STAGE = BN * 128;
    static constexpr int B_STAGE = BM * 128;
    static constexpr int RAW = BN * WTraits<WT>::RAW_BLOCK;
    // per-superblock side slot
    static constexpr int SB_ACORR = 0;                                       // 2 slabs x 128 rows x 32 B
    static constexpr int SB_BCORR = CORR ? 2 * BN * 32 : 0;                 // BM rows x 32 B
    static constexpr int SB_E = SB_BCORR + (CORR ? align_up(BM * 32, 1024) : 0);
    static constexpr int SB_DX = SB_E + BN * 4;
    static constexpr int SB = align_up(SB_DX + BM * 4, 1024);
    // CTA layout
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_STAGE;
    static constexpr int OFF_RAW = OFF_B + STAGES * B_STAGE;
    static constexpr int OFF_SB = OFF_RAW + align_up(RAW_SLOTS * RAW, 1024);
    static constexpr int OFF_BAR = OFF_SB + 2 * SB;
    static constexpr int NBAR = 2 * RAW_SLOTS + 2 * STAGES + 8;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int TOTAL = OFF_MISC + 16 + 1024;  // + slack for aligning the base
    static constexpr int TMEM_COLS = (2 * BM < 32) ? 32 : 2 * BM;
    static constexpr int CPT = BM / 2;                   // token columns per epilogue thread
    static_assert(TOTAL <= 232448, "shared memory budget");
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) { return __byte_perm(a, 0u, sel); }

__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ uint32_t hsub2u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
__device__ __forceinline__ uint32_t h2dup(__half h) {
    const uint32_t u = __half_as_ushort(h);
    return u | (u << 16);
}

// ---------------------------------------------------------------- unpack
// Q4_K: expand K64 chunk c of one 144-byte block into 64 fp16 values sc_j*q
// (sub-block 2c from the low nibbles, 2c+1 from the high nibbles) and store
// them as one 128-byte swizzled row of the operand.
__device__ __forceinline__ void unpack_q4k_chunk(const uint8_t* blk, int c, uint32_t scL, uint32_t cL,
                                                 uint32_t scH, uint32_t cH, uint8_t* arow, int row) {
    const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c + 16);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    constexpr uint32_t MAGIC = 0x64006400u;  // fp16 1024 in both halves
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        // bytes of words 2jj, 2jj+1 hold weights 8jj..8jj+7 (low nibbles) and +32 (high)
        const uint32_t a01 = prmt(w[2 * jj], 0x4140), a23 = prmt(w[2 * jj], 0x4342);
        const uint32_t b01 = prmt(w[2 * jj + 1], 0x4140), b23 = prmt(w[2 * jj + 1], 0x4342);
        uint4 lo, hi;
        lo.x = hfma2u((a01 & 0x000F000Fu) | MAGIC, scL, cL);
        lo.y = hfma2u((a23 & 0x000F000Fu) | MAGIC, scL, cL);
        lo.z = hfma2u((b01 & 0x000F000Fu) | MAGIC, scL, cL);
        lo.w = hfma2u((b23 & 0x000F000Fu) | MAGIC, scL, cL);
        hi.x = hfma2u((a01 & 0x00F000F0u) | MAGIC, scH, cH);
        hi.y = hfma2u((a23 & 0x00F000F0u) | MAGIC, scH, cH);
        hi.z = hfma2u((b01 & 0x00F000F0u) | MAGIC, scH, cH);
        hi.w = hfma2u((b23 & 0x00F000F0u) | MAGIC, scH, cH);
        *reinterpret_cast<uint4*>(arow + ((jj ^ (row & 7)) << 4)) = lo;
        *reinterpret_cast<uint4*>(arow + (((4 + jj) ^ (row & 7)) << 4)) = hi;
    }
}

// Q6_K: K64 chunk c = weights 64c..64c+63 of a 224-byte packed block.
// Half h = c/2, parts 2*(c&1) + {0,1}; low nibbles for c even, high for odd.
template <int C>
__device__ __forceinline__ void unpack_q6k_chunk(const uint8_t* blk, const uint32_t (&sc2)[16], uint8_t* arow,
                                                 int row) {
    constexpr int H = C >> 1, HN = C & 1;
    const uint4* Lp = reinterpret_cast<const uint4*>(blk + 64 * H);
    const uint4* Hp = reinterpret_cast<const uint4*>(blk + 128 + 32 * H);
    const uint4 l0 = Lp[0], l1 = Lp[1], l2 = Lp[2], l3 = Lp[3];
    const uint4 h0 = Hp[0], h1 = Hp[1];
    const uint32_t Lw[16] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w,
                             l2.x, l2.y, l2.z, l2.w, l3.x, l3.y, l3.z, l3.w};
    const uint32_t Hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    constexpr uint32_t MAGIC = 0x64006400u;
    constexpr uint32_t OFF = 0x64206420u;  // fp16 1056 = 1024 + 32 in both halves
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int pp = j >> 2, jj = j & 3;
        const int part = 2 * HN + pp;
        const int sh = 2 * part;                       // qh bit offset of this part
        const uint32_t s2 = sc2[4 * C + 2 * pp + (jj >> 1)];
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t lw = Lw[(32 * pp + 8 * jj) / 4 + k];
            const uint32_t hw = Hw[2 * jj + k];
#pragma unroll
            for (int hpair = 0; hpair < 2; ++hpair) {
                const uint32_t sel = hpair ? 0x4342u : 0x4140u;
                const uint32_t pl = prmt(lw, sel), ph = prmt(hw, sel);
                const uint32_t nib = HN ? ((pl >> 4) & 0x000F000Fu) : (pl & 0x000F000Fu);
                const uint32_t hb = (sh <= 4 ? (ph << (4 - sh)) : (ph >> (sh - 4))) & 0x00300030u;
                const uint32_t v = nib | hb | MAGIC;      // fp16 1024 + q
                o[2 * k + hpair] = hmul2u(hsub2u(v, OFF), s2);  // (q - 32) * sc, exact
            }
        }
        *reinterpret_cast<uint4*>(arow + ((j ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

template <int WT, int BM>
__global__ void __launch_bounds__(NTHREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_xh,
                   const __grid_constant__ CUtensorMap tm_xbs, const __grid_constant__ CUtensorMap tm_dx,
                   float* __restrict__ y, int64_t ldy, int M, int N, int nb, int splits,
                   uint32_t* __restrict__ status) {
    using L = Layout<WT, BM>;
    constexpr int R = L::RAW_SLOTS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
    uint64_t* raw_full = bars;
    uint64_t* raw_empty = raw_full + R;
    uint64_t* st_full = raw_empty + R;
    uint64_t* st_empty = st_full + STAGES;
    uint64_t* sb_full = st_empty + STAGES;
    uint64_t* sb_empty = sb_full + 2;
    uint64_t* acc_full = sb_empty + 2;
    uint64_t* acc_empty = acc_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    const int m0 = blockIdx.y * BM;
    const int split = blockIdx.z;
    const int kb0 = static_cast<int>(static_cast<int64_t>(nb) * split / splits);
    const int kb1 = static_cast<int>(static_cast<int64_t>(nb) * (split + 1) / splits);
    const int nsb = kb1 - kb0;

    auto a_stage = [&](int s) { return smem + L::OFF_A + s * L::A_STAGE; };
    auto b_stage = [&](int s) { return smem + L::OFF_B + s * L::B_STAGE; };
    auto raw_slot = [&](int r) { return smem + L::OFF_RAW + r * L::RAW; };
    auto sb_slot = [&](int p) { return smem + L::OFF_SB + p * L::SB; };

    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], 4);
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&st_full[s], 1 + 4);
            mbar_init(&st_empty[s], 1);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(&sb_full[p], 1 + 4);
            mbar_init(&sb_empty[p], (L::CORR ? 1 : 0) + 8);
            mbar_init(&acc_full[p], 1);
            mbar_init(&acc_empty[p], 8);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_xh);
        tma_prefetch_desc(&tm_dx);
        if (L::CORR) tma_prefetch_desc(&tm_xbs);
    }
    if (warp == 1) tmem_alloc(tmem_slot, L::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ activation producer
        if (lane == 0) {
            bool ok = true;
            for (int t = 0; t < nsb && ok; ++t) {
                const int b = kb0 + t;
                const int p = t & 1;
                ok = mbar_wait(&sb_empty[p], ((t >> 1) & 1) ^ 1, abort_flag, status, 1);
                if (!ok) break;
                uint8_t* sb = sb_slot(p);
                mbar_arrive_expect_tx(&sb_full[p], (L::CORR ? BM * 32 : 0) + BM * 4);
                if (L::CORR) tma_load_2d(&tm_xbs, &sb_full[p], sb + L::SB_BCORR, b * 16, m0);
                tma_load_2d(&tm_dx, &sb_full[p], sb + L::SB_DX, m0, b);
                for (int c = 0; c < 4; ++c) {
                    const int g = 4 * t + c;
                    const int s = g % STAGES;
                    ok = mbar_wait(&st_empty[s], ((g / STAGES) & 1) ^ 1, abort_flag, status, 2);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&st_full[s], BM * 128);
                    tma_load_2d(&tm_xh, &st_full[s], b_stage(s), b * 256 + KCH * c, m0);
                }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------ weight producer
        if (lane == 0) {
            for (int t = 0; t < nsb; ++t) {
                const int r = t % R;
                if (!mbar_wait(&raw_empty[r], ((t / R) & 1) ^ 1, abort_flag, status, 3)) break;
                mbar_arrive_expect_tx(&raw_full[r], L::RAW);
                tma_load_2d(&tm_w, &raw_full[r], raw_slot(r), (kb0 + t) * WTraits<WT>::RAW_BLOCK, n0);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_f16_f32(BN, BM);
            bool ok = true;
            for (int t = 0; t < nsb && ok; ++t) {
                const int buf = t & 1;
                ok = mbar_wait(&acc_empty[buf], ((t >> 1) & 1) ^ 1, abort_flag, status, 4);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BM;
                for (int c = 0; c < 4 && ok; ++c) {
                    const int g = 4 * t + c;
                    const int s = g % STAGES;
                    ok = mbar_wait(&st_full[s], (g / STAGES) & 1, abort_flag, status, 5);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(a_stage(s));
                    const uint32_t b0 = smem_u32(b_stage(s));
#pragma unroll
                    for (int kk = 0; kk < KCH / 16; ++kk) {
                        mma_f16(d_tmem, smem_desc(a0 + 32 * kk, 16, 1024, SWZ_128B),
                                smem_desc(b0 + 32 * kk, 16, 1024, SWZ_128B), IDESC, (c | kk) != 0);
                    }
                    mma_commit(&st_empty[s]);
                }
                if (!ok) break;
                if (L::CORR) {
                    const int p = t & 1;
                    ok = mbar_wait(&sb_full[p], (t >> 1) & 1, abort_flag, status, 6);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t sb = smem_u32(sb_slot(p));
                    const uint64_t bdesc = smem_desc(sb + L::SB_BCORR, 16, 256, SWZ_32B);
                    mma_f16(d_tmem, smem_desc(sb + L::SB_ACORR, 16, 256, SWZ_32B), bdesc, IDESC, 1u);
                    mma_f16(d_tmem, smem_desc(sb + L::SB_ACORR + BN * 32, 16, 256, SWZ_32B), bdesc, IDESC, 1u);
                    mma_commit(&sb_empty[p]);
                }
                mma_commit(&acc_full[buf]);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ unpack (thread = weight row)
        const int row = threadIdx.x - 128;
        for (int t = 0; t < nsb; ++t) {
            const int r = t % R;
            bool ok = mbar_wait(&raw_full[r], (t / R) & 1, abort_flag, status, 7);
            if (!__all_sync(0xffffffffu, ok)) break;
            const uint8_t* blk = raw_slot(r) + row * WTraits<WT>::RAW_BLOCK;
            const int p = t & 1;
            ok = mbar_wait(&sb_empty[p], ((t >> 1) & 1) ^ 1, abort_flag, status, 8);
            if (!__all_sync(0xffffffffu, ok)) break;
            uint8_t* sb = sb_slot(p);

            if constexpr (WT == 4) {
                const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
                const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xffffu)));
                const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
                const uint32_t sc03 = hdr.y & 0x3f3f3f3fu;
                const uint32_t mn03 = hdr.z & 0x3f3f3f3fu;
                const uint32_t sc47 = (hdr.w & 0x0f0f0f0fu) | ((hdr.y >> 2) & 0x30303030u);
                const uint32_t mn47 = ((hdr.w >> 4) & 0x0f0f0f0fu) | ((hdr.z >> 2) & 0x30303030u);
                int sc[8], mn[8];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    sc[j] = (sc03 >> (8 * j)) & 0xff;
                    sc[4 + j] = (sc47 >> (8 * j)) & 0xff;
                    mn[j] = (mn03 >> (8 * j)) & 0xff;
                    mn[4 + j] = (mn47 >> (8 * j)) & 0xff;
                }
                const bool main_on = (d != 0.0f);
                const float e = main_on ? d : dmin;
                const float ratio = main_on ? -dmin / d : -1.0f;
                if (!(fabsf(ratio) <= 1000.0f)) atomicOr(status, ST_Q4K_RANGE);
                uint32_t a1[8], a2[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float v = static_cast<float>(mn[j]) * ratio;
                    const __half h1 = __float2half_rn(v);
                    const __half h2 = __float2half_rn(v - __half2float(h1));
                    a1[j] = h2dup(h1);
                    a2[j] = h2dup(h2);
                }
                // correction slabs, 32-byte swizzle: row * 32 + (chunk ^ ((row >> 2) & 1)) * 16
                uint8_t* s1 = sb + L::SB_ACORR + row * 32;
                uint8_t* s2 = s1 + BN * 32;
                const int x = (row >> 2) & 1;
                *reinterpret_cast<uint4*>(s1 + ((0 ^ x) << 4)) = make_uint4(a1[0], a1[1], a1[2], a1[3]);
                *reinterpret_cast<uint4*>(s1 + ((1 ^ x) << 4)) = make_uint4(a1[4], a1[5], a1[6], a1[7]);
                *reinterpret_cast<uint4*>(s2 + ((0 ^ x) << 4)) = make_uint4(a2[0], a2[1], a2[2], a2[3]);
                *reinterpret_cast<uint4*>(s2 + ((1 ^ x) << 4)) = make_uint4(a2[4], a2[5], a2[6], a2[7]);
                reinterpret_cast<float*>(sb + L::SB_E)[row] = e;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sb_full[p]);

                for (int c = 0; c < 4; ++c) {
                    const int g = 4 * t + c;
                    const int s = g % STAGES;
                    ok = mbar_wait(&st_empty[s], ((g / STAGES) & 1) ^ 1, abort_flag, status, 9);
                    if (!__all_sync(0xffffffffu, ok)) break;
                    const int sl = main_on ? sc[2 * c] : 0, sh = main_on ? sc[2 * c + 1] : 0;
                    const uint32_t scL = h2dup(__int2half_rn(sl));
                    const uint32_t cL = h2dup(__int2half_rn(-1024 * sl));
                    const uint32_t scH = h2dup(__float2half_rn(static_cast<float>(sh) * 0.0625f));
                    const uint32_t cH = h2dup(__int2half_rn(-64 * sh));
                    unpack_q4k_chunk(blk, c, scL, cL, scH, cH, a_stage(s) + row * 128, row);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&st_full[s]);
                }
                if (!__all_sync(0xffffffffu, ok)) break;
            } else {
                const uint4 scv = *reinterpret_cast<const uint4*>(blk + 192);
                const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
                const uint32_t sw[4] = {scv.x, scv.y, scv.z, scv.w};
                uint32_t sc2[16];
                bool bad = false;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int v = static_cast<int8_t>((sw[j >> 2] >> (8 * (j & 3))) & 0xff);
                    bad |= (v > 64) || (v < -64);
                    sc2[j] = h2dup(__int2half_rn(v));
                }
                if (bad) atomicOr(status, ST_Q6K_SCALE);
                reinterpret_cast<float*>(sb + L::SB_E)[row] = d;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sb_full[p]);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int g = 4 * t + c;
                    const int s = g % STAGES;
                    ok = mbar_wait(&st_empty[s], ((g / STAGES) & 1) ^ 1, abort_flag, status, 9);
                    if (!__all_sync(0xffffffffu, ok)) break;
                    uint8_t* arow = a_stage(s) + row * 128;
                    if (c == 0) unpack_q6k_chunk<0>(blk, sc2, arow, row);
                    if (c == 1) unpack_q6k_chunk<1>(blk, sc2, arow, row);
                    if (c == 2) unpack_q6k_chunk<2>(blk, sc2, arow, row);
                    if (c == 3) unpack_q6k_chunk<3>(blk, sc2, arow, row);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&st_full[s]);
                }
                if (!__all_sync(0xffffffffu, ok)) break;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&raw_empty[r]);
        }
    } else if (warp >= 8) {
        // ------------------------------------------------ epilogue
        constexpr int CPT = L::CPT;
        const int quad = warp & 3;
        const int half = (warp - 8) >> 2;
        const int row = 32 * quad + lane;
        const int col0 = half * CPT;
        float acc[CPT];
#pragma unroll
        for (int j = 0; j < CPT; ++j) acc[j] = 0.0f;
        bool ok = true;
        for (int t = 0; t < nsb; ++t) {
            const int buf = t & 1;
            const int p = t & 1;
            ok = mbar_wait(&acc_full[buf], (t >> 1) & 1, abort_flag, status, 10);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            ok = mbar_wait(&sb_full[p], (t >> 1) & 1, abort_flag, status, 11);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const uint8_t* sb = sb_slot(p);
            const float e = reinterpret_cast<const float*>(sb + L::SB_E)[row];
            const float* dx = reinterpret_cast<const float*>(sb + L::SB_DX) + col0;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + buf * BM + col0;
            if constexpr (CPT >= 32) {
#pragma unroll
                for (int ch = 0; ch < CPT / 32; ++ch) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + 32 * ch, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        acc[32 * ch + j] = fmaf(__uint_as_float(v[j]) * e, dx[32 * ch + j], acc[32 * ch + j]);
                }
            } else if constexpr (CPT == 16) {
                uint32_t v[16];
                tmem_ld_32x32b_x16(taddr, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[j] = fmaf(__uint_as_float(v[j]) * e, dx[j], acc[j]);
            } else {
                uint32_t v[8];
                tmem_ld_32x32b_x8(taddr, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[j] = fmaf(__uint_as_float(v[j]) * e, dx[j], acc[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[buf]);
                mbar_arrive(&sb_empty[p]);
            }
        }
        const int n = n0 + row;
        if (ok && !*abort_flag && n < N) {
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                const int m = m0 + col0 + j;
                if (m < M) {
                    float* dst = y + static_cast<int64_t>(m) * ldy + n;
                    if (splits > 1)
                        atomicAdd(dst, acc[j]);
                    else
                        *dst = acc[j];
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, L::TMEM_COLS);
}

template <int WT, int BM>
cudaError_t launch_t(const TcLaunch& a, cudaStream_t s) {
    using L = Layout<WT, BM>;
    const dim3 grid(static_cast<unsigned>((a.N + BN - 1) / BN), static_cast<unsigned>((a.M + BM - 1) / BM),
                    static_cast<unsigned>(a.splits));
    gemm_tc_kernel<WT, BM><<<grid, NTHREADS, L::TOTAL, s>>>(
        *a.tm_w, *a.tm_xh, a.tm_xbs ? *a.tm_xbs : *a.tm_xh, *a.tm_dx, a.y, a.ldy, static_cast<int>(a.M),
        static_cast<int>(a.N), static_cast<int>(a.K / 256), a.splits, a.status);
    return cudaGetLastError();
}

template <int WT, int BM>
cudaError_t prepare_t() {
    return cudaFuncSetAttribute(gemm_tc_kernel<WT, BM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Layout<WT, BM>::TOTAL);
}

}  // namespace

size_t tc_smem_bytes(int wtype, int bm) {
#define QG_CASE(W, B) \
    if (wtype == W && bm == B) return Layout<W, B>::TOTAL;
    QG_CASE(4, 16) QG_CASE(4, 32) QG_CASE(4, 64) QG_CASE(4, 128)
    QG_CASE(6, 16) QG_CASE(6, 32) QG_CASE(6, 64) QG_CASE(6, 128)
#undef QG_CASE
    return 0;
}

cudaError_t tc_prepare(int wtype, int bm) {
#define QG_CASE(W, B) \
    if (wtype == W && bm == B) return prepare_t<W, B>();
    QG_CASE(4, 16) QG_CASE(4, 32) QG_CASE(4, 64) QG_CASE(4, 128)
    QG_CASE(6, 16) QG_CASE(6, 32) QG_CASE(6, 64) QG_CASE(6, 128)
#undef QG_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc(const TcLaunch& a, cudaStream_t s) {
#define QG_CASE(W, B) \
    if (a.wtype == W && a.bm == B) return launch_t<W, B>(a, s);
    QG_CASE(4, 16) QG_CASE(4, 32) QG_CASE(4, 64) QG_CASE(4, 128)
    QG_CASE(6, 16) QG_CASE(6, 32) QG_CASE(6, 64) QG_CASE(6, 128)
#undef QG_CASE
    return cudaErrorInvalidValue;
}

}  // namespace qg
