// quantize.cu -- fp32 activations -> Q8_K, plus the small HBM-bound helper
// kernels around the GEMM (operand preparation, Q6_K repacking).
//
// Q8_K (q8k.cuh): per 256-element chunk of a row, d = amax/127 (fp32), q =
// round-half-away-from-zero(x/d) clamped to +-127, and 16 int16 sums of each
// 16 consecutive q.  Stored as three planes (qs [M][K] int8, d [M][K/256]
// fp32, bsums [M][K/16] int16) so that every plane row is 16-byte aligned.
// The int8 values, scales and sums are bit-exact with any IEEE implementation
// of the same definition.
#include <cuda_fp16.h>

#include "internal.h"
#include "q8k.cuh"

namespace {
// The kernel that follows in the stream (the tile GEMM, launched as a
// programmatic dependent) may start now: it loads and expands weights, which
// this kernel does not touch, and waits for this grid before reading its output.
__device__ __forceinline__ void allow_dependent_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Launched as a programmatic dependent of the Q4_K side-data kernel (whose
// output this kernel does not read), this kernel ends only after that one
// has: the GEMM that depends on this kernel then sees both outputs.  (A
// no-op without such a predecessor.)
__device__ __forceinline__ void join_predecessor() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// A launch of `kernel` that may start while the preceding kernel in the
// stream runs (programmatic stream serialization), or a plain launch.
template <typename... Params, typename... Args>
cudaError_t launch_maybe_dependent(bool dependent, void (*kernel)(Params...), dim3 grid, dim3 block, cudaStream_t st,
                                   Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}
}  // namespace

namespace qg {

namespace {

constexpr int QWARPS = 8;  // chunks (warps) per block

// The tile GEMM's operand planes (see xprep_kernel), written by the
// quantizer itself when asked to ("prepared workspace").
struct PrepOut {
    __half* xh;    // [M][K] fp16
    __half* xbs;   // [M][K/16] fp16
    float* dxT;    // [K/256][Mp] fp32, rows m >= M zero
    int64_t Mp;
    int* counters; // TC_COUNTERS cut-tile counters, zeroed
};

// One warp per 256-element chunk: each lane owns 8 consecutive elements
// (two 16-byte loads), so one chunk is one coalesced 1 KiB read.  The chunk
// index is 32-bit unless M * K/256 reaches 2^31 (WIDE).  At most 32 registers,
// so that 64 warps (64 chunks in flight) fit on an SM (measured on GB300,
// M=8192 K=5120 with the operand planes: 59.4 -> 57.2 us; two chunks per warp
// with both loads issued first: 65.4 us).
template <bool PREP, bool WIDE>
__global__ void __launch_bounds__(QWARPS * 32, 8) quantize_q8k_kernel(const float* __restrict__ x, int64_t M,
                                                                  int64_t K, int64_t ldx, int8_t* __restrict__ qs,
                                                                  float* __restrict__ dout,
                                                                  int16_t* __restrict__ bsums, PrepOut prep) {
    allow_dependent_launch();
    if constexpr (PREP) {
        // (by every thread of block 0, before any warp without a chunk leaves)
        if (blockIdx.x == 0)
            for (int i = threadIdx.x; i < TC_COUNTERS; i += blockDim.x) prep.counters[i] = 0;
    }
    const int lane = threadIdx.x & 31;
    const int64_t nb = K >> 8;
    int64_t m, b;
    if constexpr (WIDE) {
        const int64_t chunk = static_cast<int64_t>(blockIdx.x) * QWARPS + (threadIdx.x >> 5);
        if (chunk >= M * nb) return;
        m = chunk / nb;
        b = chunk - m * nb;
    } else {
        const uint32_t chunk = blockIdx.x * QWARPS + (threadIdx.x >> 5);
        if (chunk >= static_cast<uint32_t>(M * nb)) return;
        const uint32_t m32 = chunk / static_cast<uint32_t>(nb);
        m = m32;
        b = chunk - m32 * static_cast<uint32_t>(nb);
    }

    const float4* src = reinterpret_cast<const float4*>(x + m * ldx + b * 256) + lane * 2;
    const float4 v0 = __ldcs(src);
    const float4 v1 = __ldcs(src + 1);
    float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};

    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));

    int q[8];
    const float d = q8k_quantize<8>(v, amax, q);
    uint2 packed;
    packed.x = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) | (static_cast<uint32_t>(q[3] & 0xff) << 24);
    packed.y = (q[4] & 0xff) | ((q[5] & 0xff) << 8) | ((q[6] & 0xff) << 16) | (static_cast<uint32_t>(q[7] & 0xff) << 24);
    *reinterpret_cast<uint2*>(qs + m * K + b * 256 + lane * 8) = packed;

    int s = q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7];
    s += __shfl_xor_sync(0xffffffffu, s, 1);  // lanes 2g, 2g+1 hold group g's 16 values
    if ((lane & 1) == 0) bsums[m * (K >> 4) + b * 16 + (lane >> 1)] = static_cast<int16_t>(s);
    if (lane == 0) dout[m * nb + b] = d;
    if constexpr (PREP) {
        // the same values as fp16 (integers of at most 11 significant bits: exact),
        // each aligned group of 4 in the K order 0, 2, 1, 3 of the weight operand
        uint32_t o[4];
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            const __half2 a = __halves2half2(__int2half_rn(q[4 * g]), __int2half_rn(q[4 * g + 2]));
            const __half2 c = __halves2half2(__int2half_rn(q[4 * g + 1]), __int2half_rn(q[4 * g + 3]));
            o[2 * g] = *reinterpret_cast<const uint32_t*>(&a);
            o[2 * g + 1] = *reinterpret_cast<const uint32_t*>(&c);
        }
        *reinterpret_cast<uint4*>(prep.xh + m * K + b * 256 + lane * 8) = make_uint4(o[0], o[1], o[2], o[3]);
        if ((lane & 1) == 0) prep.xbs[m * (K >> 4) + b * 16 + (lane >> 1)] = __int2half_rn(s);
        if (lane == 0) prep.dxT[b * prep.Mp + m] = d;
        if (m == M - 1 && lane >= 1 && lane < 4 && m + lane < prep.Mp) prep.dxT[b * prep.Mp + m + lane] = 0.0f;
    }
    join_predecessor();
}

// Q8_K -> fp16 operand planes.  Every int8 value and every bsum (|bsum| <=
// 16*127) is an integer of at most 11 significant bits, so fp16 holds it exactly.
// xh keeps each aligned group of 4 values in the K order 0, 2, 1, 3, the order
// in which the tile GEMM expands the weights (no byte permutes there).
__global__ void xprep_kernel(const int8_t* __restrict__ qs, const float* __restrict__ d,
                             const int16_t* __restrict__ bsums, int64_t M, int64_t K, __half* __restrict__ xh,
                             __half* __restrict__ xbs, float* __restrict__ dxT, int64_t Mp,
                             int* __restrict__ counters) {
    allow_dependent_launch();
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < TC_COUNTERS; i += blockDim.x) counters[i] = 0;
    const int64_t nb = K >> 8;
    const int64_t n16 = M * (K >> 4);                 // 16-element groups of qs (= number of bsums)
    const int64_t ndx = nb * Mp;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16 + ndx; i += stride) {
        if (i < n16) {
            const int4 raw = __ldcs(reinterpret_cast<const int4*>(qs) + i);
            const int w[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t o[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // bytes 0..3 of word j are values 4j..4j+3: pairs (0, 2) and (1, 3)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int lo = static_cast<int8_t>((w[j] >> (8 * h)) & 0xff);
                    const int hi = static_cast<int8_t>((w[j] >> (8 * h + 16)) & 0xff);
                    const __half2 p = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
                    o[2 * j + h] = *reinterpret_cast<const uint32_t*>(&p);
                }
            }
            uint4* dst = reinterpret_cast<uint4*>(xh) + 2 * i;
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            xbs[i] = __int2half_rn(bsums[i]);
        } else {
            const int64_t j = i - n16;
            const int64_t b = j / Mp;
            const int64_t m = j - b * Mp;
            dxT[j] = (m < M) ? d[m * nb + b] : 0.0f;
        }
    }
    join_predecessor();
}

// SRC-byte blocks -> DST-byte blocks (the same bytes, zeros after), so that
// every block and every row starts on a 16-byte boundary: Q6_K 210 -> 224,
// PTQ1_0 28 -> 32.
template <int SRC, int DST>
__global__ void prepack_kernel(const uint8_t* __restrict__ w, int64_t N, int64_t nb, int64_t ldw,
                               uint8_t* __restrict__ out) {
    const int64_t total = N * nb * (DST / 16);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += stride) {
        const int64_t blk = i / (DST / 16);
        const int part = static_cast<int>(i - blk * (DST / 16));
        const int64_t n = blk / nb;
        const int64_t b = blk - n * nb;
        const uint8_t* src = w + n * ldw + b * SRC;
        uint8_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int off = part * 16 + j;
            v[j] = off < SRC ? src[off] : 0;
        }
        uint4 o;
        o.x = v[0] | (v[1] << 8) | (v[2] << 16) | (static_cast<uint32_t>(v[3]) << 24);
        o.y = v[4] | (v[5] << 8) | (v[6] << 16) | (static_cast<uint32_t>(v[7]) << 24);
        o.z = v[8] | (v[9] << 8) | (v[10] << 16) | (static_cast<uint32_t>(v[11]) << 24);
        o.w = v[12] | (v[13] << 8) | (v[14] << 16) | (static_cast<uint32_t>(v[15]) << 24);
        reinterpret_cast<uint4*>(out)[i] = o;
    }
}

// Q8_K planes <-> the pages' 292-byte block ("BlockQ8_K (292B/256 elements)",
// vllm.cpp PR #3036, commit 4), field order d (fp32), qs[256] (int8),
// bsums[16] (int16).  292 is a multiple of 4, so every field of every block
// starts on a 4-byte boundary: one warp per block moves its 73 32-bit words
// (word 0 = d, words 1..64 = qs, words 65..72 = bsums), no arithmetic.
constexpr int AOS_WORDS = 73;
template <bool TO_AOS>
__global__ void q8k_aos_kernel(int8_t* __restrict__ qs, float* __restrict__ d, int16_t* __restrict__ bsums,
                               int64_t M, int64_t K, uint32_t* __restrict__ aos) {
    const int64_t nb = K >> 8;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int lane = threadIdx.x & 31;
    for (int64_t blk = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); blk < M * nb;
         blk += warps) {
        const int64_t m = blk / nb, b = blk - m * nb;
        uint32_t* a = aos + blk * AOS_WORDS;
        uint32_t* q = reinterpret_cast<uint32_t*>(qs + m * K + b * 256);
        uint32_t* s = reinterpret_cast<uint32_t*>(bsums + m * (K >> 4) + b * 16);
        uint32_t* dd = reinterpret_cast<uint32_t*>(d + m * nb + b);
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int wd = lane + 32 * i;
            if (wd >= AOS_WORDS) break;
            uint32_t* plane = wd == 0 ? dd : wd <= 64 ? q + (wd - 1) : s + (wd - 65);
            if constexpr (TO_AOS)
                a[wd] = *plane;
            else
                *plane = a[wd];
        }
    }
}

int grid_for(int64_t work, int threads) {
    int64_t g = (work + threads - 1) / threads;
    const int64_t cap = 152 * 16;
    if (g > cap) g = cap;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_quantize_q8k(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs, float* d,
                                int16_t* bsums, cudaStream_t s, __half* xh, __half* xbs, float* dxT, int64_t Mp,
                                int* counters, bool dependent) {
    const int64_t chunks = M * (K >> 8);
    const int64_t blocks = (chunks + QWARPS - 1) / QWARPS;
    const PrepOut prep{xh, xbs, dxT, Mp, counters};
    const bool wide = chunks >= (int64_t(1) << 31);
    const dim3 grid(static_cast<unsigned>(blocks)), block(QWARPS * 32);
    cudaError_t e;
    if (xh)
        e = wide ? launch_maybe_dependent(dependent, quantize_q8k_kernel<true, true>, grid, block, s, x, M, K, ldx, qs,
                                          d, bsums, prep)
                 : launch_maybe_dependent(dependent, quantize_q8k_kernel<true, false>, grid, block, s, x, M, K, ldx,
                                          qs, d, bsums, prep);
    else
        e = wide ? launch_maybe_dependent(dependent, quantize_q8k_kernel<false, true>, grid, block, s, x, M, K, ldx,
                                          qs, d, bsums, prep)
                 : launch_maybe_dependent(dependent, quantize_q8k_kernel<false, false>, grid, block, s, x, M, K, ldx,
                                          qs, d, bsums, prep);
    return e;
}

cudaError_t launch_xprep(const int8_t* qs, const float* d, const int16_t* bsums, int64_t M, int64_t K,
                         __half* xh, __half* xbs, float* dxT, int64_t Mp, int* counters, cudaStream_t s,
                         bool dependent) {
    const int64_t work = M * (K >> 4) + (K >> 8) * Mp;
    return launch_maybe_dependent(dependent, xprep_kernel, dim3(grid_for(work, 256)), dim3(256), s, qs, d, bsums, M, K,
                                  xh, xbs, dxT, Mp, counters);
}

cudaError_t launch_q8k_aos(int8_t* qs, float* d, int16_t* bsums, int64_t M, int64_t K, void* aos, bool to_aos,
                           cudaStream_t s) {
    const int64_t blocks = M * (K >> 8);
    const int per_cta = 8;   // warps (blocks of Q8_K) per CTA
    int64_t grid = (blocks + per_cta - 1) / per_cta;
    if (grid > 152 * 16) grid = 152 * 16;
    if (to_aos)
        q8k_aos_kernel<true><<<static_cast<unsigned>(grid), 32 * per_cta, 0, s>>>(qs, d, bsums, M, K,
                                                                              static_cast<uint32_t*>(aos));
    else
        q8k_aos_kernel<false><<<static_cast<unsigned>(grid), 32 * per_cta, 0, s>>>(qs, d, bsums, M, K,
                                                                               static_cast<uint32_t*>(aos));
    return cudaGetLastError();
}

cudaError_t launch_q6k_prepack(const uint8_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* out,
                               cudaStream_t s) {
    const int64_t nb = K >> 8;
    const int64_t work = N * nb * (Q6K_PACKED / 16);
    prepack_kernel<Q6K_BLOCK, Q6K_PACKED><<<grid_for(work, 256), 256, 0, s>>>(w, N, nb, ldw, out);
    return cudaGetLastError();
}

cudaError_t launch_ptq1_prepack(const uint8_t* w, int64_t N, int64_t K, int64_t ldw, uint8_t* out,
                                cudaStream_t s) {
    const int64_t nb = K >> 7;   // 128-weight blocks
    const int64_t work = N * nb * (PTQ1_PACKED / 16);
    prepack_kernel<PTQ1_BLOCK, PTQ1_PACKED><<<grid_for(work, 256), 256, 0, s>>>(w, N, nb, ldw, out);
    return cudaGetLastError();
}

}  // namespace qg
