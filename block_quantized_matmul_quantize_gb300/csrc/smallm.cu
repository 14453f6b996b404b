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
//   * Each CTA owns a contiguous range of weight rows; thread = a fixed
//     32-weight slice of K (warp w covers blocks 4w .. 4w+3, 8 threads per
//     block), so one row is read by the CTA as a few fully used 512-B runs.
//   * The weights are staged in shared memory by every thread copying its own
//     16-byte pieces with cp.async, a stage of several rows at a time, double
//     buffered: the whole stage is in flight at once from all threads.
//     (Measured on GB300: 1D bulk copies from one producer thread per CTA
//     moved a DRAM-resident row range at ~3 B/clk per CTA, and register
//     prefetch a couple of rows ahead kept too few bytes in flight.)
//   * The slice's Q8_K activations of all M tokens (int8 values, the two
//     bsums it needs, the block scale dx) stay in registers for the whole
//     kernel.
//   * Integer part with dp4a, exact: per block and token the slice adds
//       Q4_K: dx * (d * (sc_lo*I_lo + sc_hi*I_hi) - dmin * (m_lo*B_lo + m_hi*B_hi))
//       Q6_K: dx * d * (sc_a*(I_a - 32*B_a) + sc_b*(I_b - 32*B_b))
//     with I the int dot of unsigned weight codes and int8 activations and B
//     the activation sums over the slice's 16-value groups (the bsums).
//     Every integer partial stays below 2^24, so its fp32 conversion is exact.
//   * Rows go in batches: per batch one reduce-scatter over the warp (about
//     one shuffle per output value), one barrier, and warp 0 adds the warps'
//     partials and stores the batch (consecutive lanes -> consecutive rows).
// There are no waits other than the CTA barrier, which every thread reaches
// the same number of times.
#include <cuda_fp16.h>

#include <mutex>
#include <unordered_map>

#include "internal.h"
#include "epilogue.cuh"
#include "ptx.cuh"

namespace qg {
namespace {

constexpr int SM_MAX_WARPS = 15;              // warps per CTA: K <= 15360
constexpr int SM_STAGE_BYTES = 24 * 1024;     // weight bytes per staging buffer (whole rows)

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

template <int WT, int MT>
__global__ void __launch_bounds__(32 * SM_MAX_WARPS)
    smallm_kernel(const uint8_t* __restrict__ w, int64_t ldw, int N, int nb, const int8_t* __restrict__ xqs,
                  const float* __restrict__ xd, const int16_t* __restrict__ xbs, void* __restrict__ y,
                  int64_t ldy, const Epi epi, int stage_rows) {
    constexpr int BLK = SmallTraits<WT>::BLOCK;
    constexpr int P = pow2_at_least(MT);      // token slots per row
    constexpr int VALS = 16;                  // values per thread per reduction batch
    constexpr int RB = VALS / P;              // rows per batch
    __shared__ float red[2][SM_MAX_WARPS][32];
    extern __shared__ __align__(16) uint8_t stage_mem[];   // [2][stage_rows][row_bytes]

    const int K = nb * 256;
    const int nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = static_cast<int>(static_cast<int64_t>(N) * blockIdx.x / gridDim.x);
    const int r1 = static_cast<int>(static_cast<int64_t>(N) * (blockIdx.x + 1) / gridDim.x);

    const int b = 4 * warp + (lane >> 3);   // this thread's block
    const int sub = lane & 7;               // and its 32-weight slice in it
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

    // ---- weight staging: stage g holds rows r0 + g*S .. + S of this CTA
    const int row_bytes = nb * BLK;
    const int S = stage_rows;
    const int nstage = (r1 - r0 + S - 1) / S;
    // this thread's 16-byte pieces of a row (offsets inside its block)
    const bool hdr_copier = WT == 4 ? sub == 0 : sub < 2;   // Q4_K header / Q6_K scales+d
    const int hdr_off = WT == 4 ? 0 : 192 + 16 * sub;
    auto issue_stage = [&](int g) {
        uint8_t* buf = stage_mem + (g & 1) * S * row_bytes;
        const int ra = r0 + g * S, nr = min(S, r1 - ra);
        if (active) {
            for (int q = 0; q < nr; ++q) {
                const uint8_t* src = w + static_cast<int64_t>(ra + q) * ldw + b * BLK;
                uint8_t* dst = buf + q * row_bytes + b * BLK;
                cp_async16(dst + wq0, src + wq0);
                if constexpr (WT == 6) cp_async16(dst + wq1, src + wq1);
                if (hdr_copier) cp_async16(dst + hdr_off, src + hdr_off);
            }
        }
        cp_async_commit();
    };

    // both stage buffers are in flight before the activations load: the
    // weights do not depend on the preceding grid, so with a programmatic
    // dependent launch they stream while that grid finishes (measured on
    // GB300: loading the activations first did not shorten the kernel, and
    // lost that overlap)
    issue_stage(0);
    if (nstage > 1) issue_stage(1);
    griddep_wait();   // the activations come from the preceding grid

    // the slice's activations, all tokens, in registers
    uint32_t xa[MT][4], xb[MT][4];
    int bsa[MT], bsb[MT];
    float dx[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (active) {
            const int8_t* xr = xqs + static_cast<int64_t>(m) * K + 256 * b;
            const uint4 va = *reinterpret_cast<const uint4*>(xr + ka);
            const uint4 vb = *reinterpret_cast<const uint4*>(xr + kb);
            xa[m][0] = va.x, xa[m][1] = va.y, xa[m][2] = va.z, xa[m][3] = va.w;
            xb[m][0] = vb.x, xb[m][1] = vb.y, xb[m][2] = vb.z, xb[m][3] = vb.w;
            const int16_t* br = xbs + static_cast<int64_t>(m) * (K / 16) + 16 * b;
            bsa[m] = br[ka / 16];
            bsb[m] = br[kb / 16];
            dx[m] = xd[static_cast<int64_t>(m) * nb + b];
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) xa[m][k] = xb[m][k] = 0u;
            bsa[m] = bsb[m] = 0;
            dx[m] = 0.0f;
        }
    }

    int it = 0;   // reduction batch counter (parity of the red buffer)
    for (int g = 0; g < nstage; ++g) {
        // committed so far: stages 0 .. min(g + 1, nstage - 1)
        if (g + 1 < nstage)
            cp_async_wait<1>();
        else
            cp_async_wait<0>();
        __syncthreads();   // every thread's pieces of stage g have landed
        const uint8_t* buf = stage_mem + (g & 1) * S * row_bytes;
        const int ra = r0 + g * S, nr = min(S, r1 - ra);
        for (int q0 = 0; q0 < nr; q0 += RB, ++it) {
            float v[VALS];
#pragma unroll
            for (int t = 0; t < VALS; ++t) v[t] = 0.0f;
#pragma unroll
            for (int rr = 0; rr < RB; ++rr) {
                if (q0 + rr >= nr || !active) break;   // nr uniform over the CTA
                const uint8_t* blk = buf + (q0 + rr) * row_bytes + b * BLK;
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
            // lane l now holds the warp total of value t = l / (32 / VALS), i.e.
            // row t / P, token t % P of the batch
            const float tot = reduce_scatter<VALS>(v, lane);
            float (*rbuf)[32] = red[it & 1];
            if ((lane & (32 / VALS - 1)) == 0) rbuf[warp][lane / (32 / VALS)] = tot;
            __syncthreads();
            if (warp == 0 && lane < VALS) {
                const int rr = lane / P, m = lane % P, n = ra + q0 + rr;
                if (m < MT && q0 + rr < nr) {
                    float sum = 0.0f;
                    for (int u = 0; u < nw; ++u) sum += rbuf[u][lane];
                    epi_store(y, static_cast<int64_t>(m) * ldy + n,
                              epi_value(sum, epi.bias ? epi.bias[n] : 0.0f, epi.act), epi.out);
                }
            }
        }
        __syncthreads();   // stage buffer g & 1 is refilled next
        if (g + 2 < nstage) issue_stage(g + 2);
    }
}

// Resident CTAs per SM of one kernel instantiation and shape, looked up once
// per device (the dynamic shared-memory limit is raised on first use).
cudaError_t small_occupancy(const void* kernel, int wt, int mt, int nb, int threads, size_t smem, int* occ) {
    static std::mutex mtx;
    static std::unordered_map<uint64_t, int> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t key = (static_cast<uint64_t>(dev) << 32) | (static_cast<uint64_t>(wt) << 24) |
                         (static_cast<uint64_t>(mt) << 16) | static_cast<uint64_t>(nb);
    std::lock_guard<std::mutex> lk(mtx);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *occ = it->second;
        return cudaSuccess;
    }
    // the limit belongs to the kernel, shared by every shape: raise it to the
    // most any shape asks (two stages of at most SM_STAGE_BYTES whole rows)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * SM_STAGE_BYTES);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
    if (e != cudaSuccess) return e;
    *occ = n < 1 ? 1 : n;
    cache[key] = *occ;
    return cudaSuccess;
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

template <int WT>
cudaError_t launch_small_wt(const uint8_t* w, int64_t ldw, int N, int nb, const int8_t* xqs, const float* xd,
                            const int16_t* xbs, int M, void* y, int64_t ldy, const Epi& epi, int sm_count,
                            cudaStream_t st) {
    const int threads = 32 * ((nb + 3) / 4);
    const int row_bytes = nb * SmallTraits<WT>::BLOCK;
    // stage: whole rows, at most about SM_STAGE_BYTES; two stage buffers per CTA
    int max_rows = SM_STAGE_BYTES / row_bytes;   // >= 1: a row is at most 60 * 224 B
    if (max_rows < 1) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(2) * max_rows * row_bytes;
    // grid: as many CTAs as are resident at once, at most one per stage of rows
#define QG_SMALL_CASE(MT)                                                                               \
    case MT: {                                                                                          \
        auto k = smallm_kernel<WT, MT>;                                                                 \
        int occ = 0;                                                                                    \
        cudaError_t e = small_occupancy(reinterpret_cast<const void*>(k), WT, MT, nb, threads, smem, &occ); \
        if (e != cudaSuccess) return e;                                                                 \
        int64_t grid = static_cast<int64_t>(sm_count) * occ;                                            \
        if (grid > N) grid = N;                                                                         \
        /* at least two stages per CTA, so the second one loads while the first is used */             \
        const int64_t rpc = (N + grid - 1) / grid;                                                      \
        int stage_rows = static_cast<int>((rpc + 1) / 2);                                               \
        if (stage_rows > max_rows) stage_rows = max_rows;                                               \
        if (stage_rows < 1) stage_rows = 1;                                                             \
        return launch_dependent(k, static_cast<int>(grid), threads, smem, st, w,                        \
                                ldw, N, nb, xqs, xd, xbs, y, ldy, epi, stage_rows);                     \
    }
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
#undef QG_SMALL_CASE
}

}  // namespace

bool small_supported(int wtype, int64_t M, int64_t K) {
    (void)wtype;
    const int64_t nb = K / 256;
    return M >= 1 && M <= SMALL_M_LIMIT && (nb + 3) / 4 <= SM_MAX_WARPS;
}

cudaError_t launch_small(const SmallLaunch& a, cudaStream_t st) {
    const int nb = static_cast<int>(a.K / 256);
    const uint8_t* w = static_cast<const uint8_t*>(a.w);
    if (a.wtype == 4)
        return launch_small_wt<4>(w, a.ldw, static_cast<int>(a.N), nb, a.xqs, a.xd, a.xbs, static_cast<int>(a.M),
                                  a.y, a.ldy, a.epi, a.sm_count, st);
    return launch_small_wt<6>(w, a.ldw, static_cast<int>(a.N), nb, a.xqs, a.xd, a.xbs, static_cast<int>(a.M), a.y,
                              a.ldy, a.epi, a.sm_count, st);
}

}  // namespace qg
