// smallm.cu -- the small-M streaming path: Y[M][N] = X_q8k[M][K] * W[N][K]^T
// for a handful of tokens (M <= 8), where the weight bytes are all that
// matter (Q4_K K = N = 5120: 14.7 MB of weights against 0.04 MB per token).
//
// The pages' mat-vec lesson (llama.cpp's MMVQ path and its column-count
// crossover, "perf(KERNEL-QUANT-CIQ-GEMM-ROCM)", vllm.cpp PR #3036): below a
// few columns a kernel that streams each weight row once and does the
// integer dot products on the CUDA cores beats the tile GEMM.
//
// Design on sm_103a:
//   * One CTA per SM.  One producer thread streams the CTA's contiguous range
//     of weight rows into a shared-memory ring with 1D bulk copies (TMA), a
//     stage of whole rows per copy, up to 16 stages and ~200 KB per ring.
//     (Measured on GB300: a read-only stream needs ~64 KB in flight per SM to
//     reach ~6.4 TB/s; per-thread cp.async stopped near 3.8 TB/s however deep
//     its ring, while bulk copies of 16-48 KB reach 6.3-6.4 TB/s.  A grid of
//     ~600 small CTAs also cost ~1.3 us more to launch than one of 152.)
//   * The stage's rows are dealt round-robin to RL "row lanes", each a group
//     of WPR = ceil(K/1024) consumer warps that together cover one row's K:
//     warp wk of a row lane owns blocks 4wk .. 4wk+3, lane = a fixed
//     32-weight slice (8 lanes per block).
//   * The slice's Q8_K activations of all M tokens (int8 values, the two
//     bsums it needs, the block scale dx) stay in registers for the whole
//     kernel.  They are read with plain loads after the wait for the
//     preceding grid, beside the weight stream rather than behind it.
//   * Integer part with dp4a, exact: per block and token the slice adds
//       Q4_K: dx * (d * (sc_lo*I_lo + sc_hi*I_hi) - dmin * (m_lo*B_lo + m_hi*B_hi))
//       Q6_K: dx * d * (sc_a*(I_a - 32*B_a) + sc_b*(I_b - 32*B_b))
//     with I the int dot of unsigned weight codes and int8 activations and B
//     the activation sums over the slice's 16-value groups (the bsums).
//     Every integer partial stays below 2^24, so its fp32 conversion is exact.
//   * Per stage, each warp reduces its rows x M tokens over its lanes (about
//     one shuffle per output), writes the partials to shared memory, and the
//     row lane's warps meet at one named barrier; warp 0 of the row lane adds
//     the WPR partials in a fixed order and stores.  Y is deterministic.
// Every mbarrier wait is bounded (a timeout records a status bit and the
// warp carries on without data, so it still meets its row lane at every
// named barrier); the producer waits for its copies in flight before it ends.
#include <cuda_fp16.h>

#include <mutex>
#include <unordered_set>

#include "internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"
#include "q8k.cuh"

namespace qg {
namespace {

constexpr int SM_MAX_WPR = 15;                 // warps per row: K <= 15360
constexpr int SM_MAX_ROW_LANES = 15;           // named barriers 1..15
constexpr int SM_MAX_SLOTS = 16;               // ring stages
constexpr int SM_RING_BYTES = 200 * 1024;      // weight ring per CTA
constexpr int SM_SLOT_TARGET = 48 * 1024;      // bytes per stage, at most (unless one row lane's rows exceed it)

template <int WT>
struct SmallTraits;
template <>
struct SmallTraits<4> {
    static constexpr int BLOCK = Q4K_BLOCK;
};
template <>
struct SmallTraits<6> {
    static constexpr int BLOCK = Q6K_PACKED;
};

__host__ __device__ constexpr int pow2_at_least(int m) { return m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : 8; }

// Consumer warps per CTA at most, by token count: the activations of MT
// tokens live in registers (8*MT words + 2*MT bsums + MT scales per lane).
__host__ __device__ constexpr int small_max_warps(int mt) { return mt <= 2 ? 20 : mt <= 4 ? 16 : 15; }
// shared memory of the fused path's quantized activations: int8 [M][K], then fp32 d [M][K/256]
__host__ __device__ constexpr int small_act_bytes(int mt, int nb) { return mt * nb * 256 + mt * nb * 4; }
// Rows per row lane and stage, at most: the stage's R x pow2(MT) outputs of
// a warp are reduced in one pass (at most 16 values per lane).
__host__ __device__ constexpr int small_stage_rows(int wt, int mt) {
    return wt == 6 ? 2 : pow2_at_least(mt) >= 8 ? 2 : 4;
}

// Sum v[0..P) over the 32 lanes; afterwards lane l holds the total of value
// l / (32 / P) (lanes l % (32/P) == 0 are the representatives).
template <int P>
__device__ __forceinline__ float reduce_scatter(float (&v)[P], int lane) {
#pragma unroll
    for (int n = P, bit = 16; n > 1; n >>= 1, bit >>= 1) {
        const bool up = (lane & bit) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[n / 2 + i];
            const float keep = up ? v[n / 2 + i] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, bit);
        }
    }
    float r = v[0];
#pragma unroll
    for (int bit = 16 / P; bit >= 1; bit >>= 1) r += __shfl_xor_sync(0xffffffffu, r, bit);
    return r;
}

// Barrier of the `threads` threads of one row lane (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void row_lane_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// FUSED: the kernel quantizes its activations itself, from fp32 X (below).
template <int WT, int MT, bool FUSED>
__global__ void __launch_bounds__(32 * (small_max_warps(MT) + 1), 1)
    smallm_kernel(const uint8_t* __restrict__ w, int64_t ldw, int N, int nb, const SmallAct act,
                  void* __restrict__ y, int64_t ldy, const Epi epi, int wpr, int rl, int rps, int nsb,
                  uint32_t* status, const WaitCfg wcfg) {
    constexpr int BLK = SmallTraits<WT>::BLOCK;
    constexpr int P = pow2_at_least(MT);          // token slots per row
    constexpr int R = small_stage_rows(WT, MT);   // rows per row lane and stage, at most
    constexpr int VALS = R * P;                   // outputs per stage and warp
    static_assert(VALS <= 16, "stage shape");
    __shared__ float red[2][small_max_warps(MT)][VALS];
    __shared__ uint64_t full[SM_MAX_SLOTS], empty[SM_MAX_SLOTS];
    __shared__ int wait_ctl[2];   // abort flag, wait limit (ptx.cuh)
    extern __shared__ __align__(128) uint8_t ring[];   // [nsb][srw rows of row_bytes]

    const int K = nb * 256;
    const int row_bytes = nb * BLK;
    const int srw = rl * rps;                     // rows per stage
    const int slot_bytes = srw * row_bytes;
    const int ncons = rl * wpr;                   // consumer warps; warp ncons is the producer
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = static_cast<int>(static_cast<int64_t>(N) * blockIdx.x / gridDim.x);
    const int r1 = static_cast<int>(static_cast<int64_t>(N) * (blockIdx.x + 1) / gridDim.x);
    const int nst = (r1 - r0 + srw - 1) / srw;    // stages of this CTA

    if (threadIdx.x == 0) {
        for (int i = 0; i < nsb; ++i) {
            mbar_init(&full[i], 1);          // the producer's expect_tx; completes on the bytes
            mbar_init(&empty[i], ncons);     // one arrival per consumer warp
        }
        wait_ctl_init(wait_ctl, wcfg);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == ncons) {
        // ---- producer: whole-row stages by 1D bulk copies.  The weights do
        // not depend on the preceding grid: no wait for it here, so with a
        // programmatic dependent launch they stream while it finishes.
        if (lane == 0) {
            // Test only (WaitCfg): CTA 0 issues no stage, so that its
            // consumers' waits run out (and nothing is in flight).
            const bool skip_all = blockIdx.x == 0 && wcfg.test_skip == ST_SKIP_SMALLM_STAGE;
            int issued = 0;
            for (int g = 0; g < nst && !skip_all; ++g) {
                const int sl = g % nsb;
                if (g >= nsb && !mbar_wait(&empty[sl], ((g / nsb) - 1) & 1, wait_ctl, status, 20)) break;
                const int ra = r0 + g * srw;
                const int nr = min(srw, r1 - ra);
                uint8_t* dst = ring + static_cast<size_t>(sl) * slot_bytes;
                mbar_arrive_expect_tx(&full[sl], static_cast<uint32_t>(nr * row_bytes));
                if (ldw == row_bytes) {
                    bulk_load(dst, w + static_cast<int64_t>(ra) * ldw, static_cast<uint32_t>(nr * row_bytes), &full[sl]);
                } else {
                    for (int q = 0; q < nr; ++q)
                        bulk_load(dst + q * row_bytes, w + static_cast<int64_t>(ra + q) * ldw,
                                  static_cast<uint32_t>(row_bytes), &full[sl]);
                }
                ++issued;
            }
            // the copies still in flight land before the CTA may end (not cut
            // short by the abort flag)
            for (int g = issued > nsb ? issued - nsb : 0; g < issued; ++g)
                mbar_wait_drain(&full[g % nsb], (g / nsb) & 1, wait_ctl);
        }
        return;
    }

    // ---- consumers: row lane lj takes rows lj, lj + rl, ... of every stage
    const int lj = warp / wpr, wk = warp - lj * wpr;
    const int b = 4 * wk + (lane >> 3);   // this lane's block
    const int sub = lane & 7;             // and its 32-weight slice in it
    const bool active = b < nb;
    // K offsets (within the block) of the slice's two 16-value groups, and
    // the byte offsets of its weights in a block
    int ka, kb, wq0, wq1;
    if constexpr (WT == 4) {
        const int c = sub >> 1, h = sub & 1;   // chunk (64 weights), half
        ka = 64 * c + 16 * h;                  // low nibbles: sub-block 2c
        kb = ka + 32;                          // high nibbles: sub-block 2c+1
        wq0 = 16 + 32 * c + 16 * h;            // the 16 code bytes
        wq1 = 0;
    } else {
        const int hh = sub >> 2, pp = (sub >> 1) & 1, s = sub & 1;
        ka = 128 * hh + 32 * pp + 16 * s;      // chunk 2hh: low nibbles, qh bits 2pp
        kb = ka + 64;                          // chunk 2hh+1: high nibbles, qh bits 4+2pp
        wq0 = 64 * hh + 32 * pp + 16 * s;      // ql bytes
        wq1 = 128 + 32 * hh + 16 * s;          // qh bytes
    }

    griddep_wait();   // the activations come from the preceding grid

    // the slice's activations, all tokens, in registers
    uint32_t xa[MT][4], xb[MT][4];
    int bsa[MT], bsb[MT];
    float dx[MT];
    if constexpr (FUSED) {
        // Quantized here, from fp32 X, once per CTA: the consumer warps take
        // the M * nb chunks of 256 values in turn (a lane 8 values, as in the
        // quantizer kernel, with its arithmetic: q8k.cuh, so the values are
        // those qgemm_quantize_q8k writes) into shared memory after the ring;
        // CTA 0 also stores them as the Q8_K planes.  Then every lane reads
        // its slices, and its two group sums are dp4a against ones.
        int8_t* sq = reinterpret_cast<int8_t*>(ring + static_cast<size_t>(nsb) * slot_bytes);
        float* sd = reinterpret_cast<float*>(sq + MT * K);
        const int nchunk = MT * nb;
        for (int c = warp; c < nchunk; c += ncons) {
            const int m = c / nb, cb = c - m * nb;
            const float4* src = reinterpret_cast<const float4*>(act.x + static_cast<int64_t>(m) * act.ldx + 256 * cb) + 2 * lane;
            const float4 v0 = src[0], v1 = src[1];
            const float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            float amax = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(v[k]));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            int q[8];
            const float d = q8k_quantize<8>(v, amax, q);
            uint2 packed;
            packed.x = static_cast<uint32_t>(q[0] & 0xff) | (static_cast<uint32_t>(q[1] & 0xff) << 8) |
                       (static_cast<uint32_t>(q[2] & 0xff) << 16) | (static_cast<uint32_t>(q[3] & 0xff) << 24);
            packed.y = static_cast<uint32_t>(q[4] & 0xff) | (static_cast<uint32_t>(q[5] & 0xff) << 8) |
                       (static_cast<uint32_t>(q[6] & 0xff) << 16) | (static_cast<uint32_t>(q[7] & 0xff) << 24);
            *reinterpret_cast<uint2*>(sq + m * K + 256 * cb + 8 * lane) = packed;
            if (lane == 0) sd[m * nb + cb] = d;
            if (blockIdx.x == 0) {
                *reinterpret_cast<uint2*>(act.oqs + static_cast<int64_t>(m) * K + 256 * cb + 8 * lane) = packed;
                int sum = q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7];
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);   // lanes 2g, 2g+1: group g
                if ((lane & 1) == 0)
                    act.obs[static_cast<int64_t>(m) * (K / 16) + 16 * cb + (lane >> 1)] = static_cast<int16_t>(sum);
                if (lane == 0) act.od[static_cast<int64_t>(m) * nb + cb] = d;
            }
        }
        asm volatile("bar.sync 0, %0;" ::"r"(32 * ncons) : "memory");   // the consumer warps only
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (active) {
                const uint4 va = *reinterpret_cast<const uint4*>(sq + m * K + 256 * b + ka);
                const uint4 vb = *reinterpret_cast<const uint4*>(sq + m * K + 256 * b + kb);
                xa[m][0] = va.x, xa[m][1] = va.y, xa[m][2] = va.z, xa[m][3] = va.w;
                xb[m][0] = vb.x, xb[m][1] = vb.y, xb[m][2] = vb.z, xb[m][3] = vb.w;
                int sa = 0, sb = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    sa = __dp4a(static_cast<int>(xa[m][k]), 0x01010101, sa);
                    sb = __dp4a(static_cast<int>(xb[m][k]), 0x01010101, sb);
                }
                bsa[m] = sa;
                bsb[m] = sb;
                dx[m] = sd[m * nb + b];
            } else {
#pragma unroll
                for (int k = 0; k < 4; ++k) xa[m][k] = xb[m][k] = 0u;
                bsa[m] = bsb[m] = 0;
                dx[m] = 0.0f;
            }
        }
    } else {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (active) {
            const int8_t* xr = act.xqs + static_cast<int64_t>(m) * K + 256 * b;
            const uint4 va = *reinterpret_cast<const uint4*>(xr + ka);
            const uint4 vb = *reinterpret_cast<const uint4*>(xr + kb);
            xa[m][0] = va.x, xa[m][1] = va.y, xa[m][2] = va.z, xa[m][3] = va.w;
            xb[m][0] = vb.x, xb[m][1] = vb.y, xb[m][2] = vb.z, xb[m][3] = vb.w;
            const int16_t* br = act.xbs + static_cast<int64_t>(m) * (K / 16) + 16 * b;
            bsa[m] = br[ka / 16];
            bsb[m] = br[kb / 16];
            dx[m] = act.xd[static_cast<int64_t>(m) * nb + b];
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) xa[m][k] = xb[m][k] = 0u;
            bsa[m] = bsb[m] = 0;
            dx[m] = 0.0f;
        }
    }
    }

    // A failed wait (timeout, status recorded) does not end the loop: the
    // warp still meets its row lane at every barrier, only without data.
    bool ok = true;
    for (int g = 0; g < nst; ++g) {
        const int sl = g % nsb;
        const int ra = r0 + g * srw;
        const int nr = min(srw, r1 - ra);
        if (ok) ok = mbar_wait(&full[sl], (g / nsb) & 1, wait_ctl, status, 22);
        float v[VALS];
#pragma unroll
        for (int t = 0; t < VALS; ++t) v[t] = 0.0f;
        const uint8_t* slot = ring + static_cast<size_t>(sl) * slot_bytes + b * BLK;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const int q = lj + rl * rr;
            if (rr >= rps || q >= nr || !ok || !active) break;
            const uint8_t* blk = slot + q * row_bytes;
            if constexpr (WT == 4) {
                const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
                const uint4 qv = *reinterpret_cast<const uint4*>(blk + wq0);
                const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xffffu)));
                const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
                // 6-bit sub-block scales and mins (bytes 4..15 of the block)
                const uint32_t sc03 = hdr.y & 0x3f3f3f3fu;
                const uint32_t sc47 = (hdr.w & 0x0f0f0f0fu) | ((hdr.y >> 2) & 0x30303030u);
                const uint32_t mn03 = hdr.z & 0x3f3f3f3fu;
                const uint32_t mn47 = ((hdr.w >> 4) & 0x0f0f0f0fu) | ((hdr.z >> 2) & 0x30303030u);
                const int c = sub >> 1;
                const int sh = 16 * (c & 1);
                const uint32_t scw = c < 2 ? sc03 : sc47, mnw = c < 2 ? mn03 : mn47;
                const int sc_lo = (scw >> sh) & 0xff, sc_hi = (scw >> (sh + 8)) & 0xff;
                const int mn_lo = (mnw >> sh) & 0xff, mn_hi = (mnw >> (sh + 8)) & 0xff;
                const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
                uint32_t lo[4], hi[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    lo[k] = qw[k] & 0x0f0f0f0fu;
                    hi[k] = (qw[k] >> 4) & 0x0f0f0f0fu;
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    int il = 0, ih = 0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        il = __dp4a(static_cast<int>(lo[k]), static_cast<int>(xa[m][k]), il);
                        ih = __dp4a(static_cast<int>(hi[k]), static_cast<int>(xb[m][k]), ih);
                    }
                    const int s1 = sc_lo * il + sc_hi * ih;
                    const int s2 = mn_lo * bsa[m] + mn_hi * bsb[m];
                    v[rr * P + m] = dx[m] * fmaf(d, static_cast<float>(s1), -dmin * static_cast<float>(s2));
                }
            } else {
                const uint4 ql = *reinterpret_cast<const uint4*>(blk + wq0);
                const uint4 qh = *reinterpret_cast<const uint4*>(blk + wq1);
                const uint2 scv = *reinterpret_cast<const uint2*>(blk + 192 + 8 * (sub >> 2));
                const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
                const int pp = (sub >> 1) & 1, ga = sub & 3;   // ga = 2*pp + s: group in its chunk
                const int sc_a = static_cast<int8_t>((scv.x >> (8 * ga)) & 0xffu);
                const int sc_b = static_cast<int8_t>((scv.y >> (8 * ga)) & 0xffu);
                const uint32_t lw[4] = {ql.x, ql.y, ql.z, ql.w};
                const uint32_t hw[4] = {qh.x, qh.y, qh.z, qh.w};
                uint32_t qa[4], qb[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    qa[k] = (lw[k] & 0x0f0f0f0fu) | (((hw[k] >> (2 * pp)) & 0x03030303u) << 4);
                    qb[k] = ((lw[k] >> 4) & 0x0f0f0f0fu) | (((hw[k] >> (4 + 2 * pp)) & 0x03030303u) << 4);
                }
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    int ia = 0, ib = 0;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        ia = __dp4a(static_cast<int>(qa[k]), static_cast<int>(xa[m][k]), ia);
                        ib = __dp4a(static_cast<int>(qb[k]), static_cast<int>(xb[m][k]), ib);
                    }
                    const int sv = sc_a * (ia - 32 * bsa[m]) + sc_b * (ib - 32 * bsb[m]);
                    v[rr * P + m] = (dx[m] * d) * static_cast<float>(sv);
                }
            }
        }
        __syncwarp();   // every lane of the warp is done with the slot
        if (lane == 0) mbar_arrive(&empty[sl]);

        // lane l now holds the warp total of value t = l / (32 / VALS), i.e.
        // row lj + rl * (t / P), token t % P of the stage
        const float tot = reduce_scatter<VALS>(v, lane);
        if ((lane & (32 / VALS - 1)) == 0) red[g & 1][warp][lane / (32 / VALS)] = tot;
        // the row lane's partials are out; warp 0 of the row lane adds them.
        // (red[g & 1] is written again at stage g + 2, after the barrier of
        // stage g + 1, which warp 0 reaches only once this sum is done.)
        row_lane_sync(1 + lj, 32 * wpr);
        if (wk == 0 && lane < VALS && ok) {
            const int rr = lane / P, m = lane % P, q = lj + rl * rr;
            if (m < MT && rr < rps && q < nr) {
                float sum = 0.0f;
                for (int u = 0; u < wpr; ++u) sum += red[g & 1][lj * wpr + u][lane];
                const int n = ra + q;
                epi_store(y, static_cast<int64_t>(m) * ldy + n,
                          epi_value(sum, epi.bias ? epi.bias[n] : 0.0f, epi.act), epi.out);
            }
        }
    }
}

// The ring is above the default 48 KB of dynamic shared memory: raise each
// instantiation's limit once per device.
cudaError_t ensure_smem_limit(const void* kernel, size_t bytes) {
    static std::mutex mtx;
    static std::unordered_set<uint64_t> done;   // (device, kernel)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t key = (static_cast<uint64_t>(dev) << 56) ^ reinterpret_cast<uint64_t>(kernel);
    std::lock_guard<std::mutex> lk(mtx);
    if (done.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess) done.insert(key);
    return e;
}

// A programmatic dependent launch of the small-M kernel: its CTAs may start
// (and fetch weights) while the preceding kernel in the stream finishes; the
// kernel waits for that grid before it reads the activations.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), int grid, int threads, size_t smem, cudaStream_t st,
                             Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);   // (arguments converted to the parameter types)
}

template <int WT, bool FUSED>
cudaError_t launch_small_wt(const uint8_t* w, int64_t ldw, int N, int nb, const SmallAct& act, int M, void* y,
                            int64_t ldy, const Epi& epi, int sm_count, uint32_t* status, const WaitCfg& wcfg,
                            cudaStream_t st) {
    const int wpr = (nb + 3) / 4;   // warps per row lane
    if (wpr < 1 || wpr > SM_MAX_WPR || sm_count < 1) return cudaErrorInvalidValue;
    const int grid = sm_count < N ? sm_count : N;   // one CTA per SM
    const int row_bytes = nb * SmallTraits<WT>::BLOCK;
#define QG_SMALL_CASE(MT)                                                                               \
    case MT: {                                                                                          \
        auto k = smallm_kernel<WT, MT, FUSED>;                                                          \
        int rl = small_max_warps(MT) / wpr;                                                             \
        if (rl > SM_MAX_ROW_LANES) rl = SM_MAX_ROW_LANES;                                               \
        /* rows per row lane and stage: a stage of at most SM_SLOT_TARGET bytes, one row each at least */ \
        int rps = SM_SLOT_TARGET / (rl * row_bytes);                                                    \
        if (rps > small_stage_rows(WT, MT)) rps = small_stage_rows(WT, MT);                             \
        if (rps < 1) rps = 1;                                                                           \
        const int slot = rl * rps * row_bytes;                                                          \
        /* (fused: the quantized activations after the ring) */                                       \
        const int act_bytes = FUSED ? small_act_bytes(MT, nb) : 0;                                       \
        int nsb = (SM_RING_BYTES - act_bytes) / slot;                                                   \
        if (nsb > SM_MAX_SLOTS) nsb = SM_MAX_SLOTS;                                                     \
        if (nsb < 2) return cudaErrorInvalidValue;                                                      \
        cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(k), SM_RING_BYTES);             \
        if (e != cudaSuccess) return e;                                                                 \
        return launch_dependent(k, grid, 32 * (rl * wpr + 1), static_cast<size_t>(nsb) * slot + act_bytes, st, w, ldw, N, \
                                nb, act, y, ldy, epi, wpr, rl, rps, nsb, status, wcfg);                 \
    }
    if constexpr (FUSED) {
        switch (M) {
            QG_SMALL_CASE(1)
            QG_SMALL_CASE(2)
            default:
                return cudaErrorInvalidValue;
        }
    } else {
        switch (M) {
            QG_SMALL_CASE(1)
            QG_SMALL_CASE(2)
            QG_SMALL_CASE(3)
            QG_SMALL_CASE(4)
            QG_SMALL_CASE(5)
            QG_SMALL_CASE(6)
            QG_SMALL_CASE(7)
            QG_SMALL_CASE(8)
            default:
                return cudaErrorInvalidValue;
        }
    }
#undef QG_SMALL_CASE
}

}  // namespace

bool small_supported(int wtype, int64_t M, int64_t K) {
    (void)wtype;
    const int64_t nb = K / 256;
    return M >= 1 && M <= SMALL_M_LIMIT && (nb + 3) / 4 <= SM_MAX_WPR;
}

cudaError_t launch_small(const SmallLaunch& a, cudaStream_t st) {
    const int nb = static_cast<int>(a.K / 256);
    const uint8_t* w = static_cast<const uint8_t*>(a.w);
    const int M = static_cast<int>(a.M), N = static_cast<int>(a.N);
    if (a.act.x) {
        if (M > SMALL_FUSED_M_MAX) return cudaErrorInvalidValue;
        return a.wtype == 4 ? launch_small_wt<4, true>(w, a.ldw, N, nb, a.act, M, a.y, a.ldy, a.epi, a.sm_count,
                                                       a.status, a.wait, st)
                            : launch_small_wt<6, true>(w, a.ldw, N, nb, a.act, M, a.y, a.ldy, a.epi, a.sm_count,
                                                       a.status, a.wait, st);
    }
    return a.wtype == 4 ? launch_small_wt<4, false>(w, a.ldw, N, nb, a.act, M, a.y, a.ldy, a.epi, a.sm_count,
                                                    a.status, a.wait, st)
                        : launch_small_wt<6, false>(w, a.ldw, N, nb, a.act, M, a.y, a.ldy, a.epi, a.sm_count,
                                                    a.status, a.wait, st);
}

}  // namespace qg
