// route.cu -- expert routing for the routed GEMM (MUL_MAT_ID): group the
// (token, slot) pairs by expert and gather each routed row's operand planes.
//
// The pages test MUL_MAT_ID beside MUL_MAT ("cuda: branch-free PTQ1_0 MMQ
// tile loader ...", llama.cpp PR #214, test-backend-ops): for token i and
// slot s the expert ids[i][s] multiplies token i.  Here the pairs of one
// expert become consecutive "routed rows", so one launch of the tile GEMM
// covers every expert: a token tile never mixes experts, and each output
// row is scattered back to (i, s) by the epilogue.
#include <cuda_fp16.h>

#include "internal.h"

namespace qg {
namespace {

constexpr int RT_THREADS = 1024;

// Inclusive sum over the CTA of one int per thread (RT_THREADS threads).
__device__ int block_inclusive_sum(int v, int* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int r = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    __syncthreads();   // warp_sums is reused by the next call
    return r;
}

// One CTA: histogram of the ids, prefix sums (rows and bm-row tiles per
// expert), then each pair takes the next routed row of its expert.
__global__ void __launch_bounds__(RT_THREADS) route_kernel(const int32_t* __restrict__ ids, int64_t P, int E,
                                                          int bm, int* __restrict__ row_off,
                                                          int* __restrict__ row_end, int* __restrict__ tile_off,
                                                          int* __restrict__ perm, uint32_t* __restrict__ status) {
    __shared__ int cnt[ROUTE_MAX_EXPERTS];
    __shared__ int cursor[ROUTE_MAX_EXPERTS];
    __shared__ int warp_sums[32];
    for (int e = threadIdx.x; e < ROUTE_MAX_EXPERTS; e += RT_THREADS) cnt[e] = 0;
    __syncthreads();
    bool bad = false;
    for (int64_t q = threadIdx.x; q < P; q += RT_THREADS) {
        const int e = ids[q];
        if (e >= 0 && e < E)
            atomicAdd(&cnt[e], 1);
        else
            bad = true;
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(status, ST_BAD_EXPERT);
    // thread t owns expert t (E <= ROUTE_MAX_EXPERTS = RT_THREADS)
    const int e = threadIdx.x;
    const int c = e < E ? cnt[e] : 0;
    const int c4 = (c + 3) & ~3;   // the expert's rows, padded to a multiple of 4
    const int tiles = (c + bm - 1) / bm;
    const int rows_incl = block_inclusive_sum(c4, warp_sums);
    const int tiles_incl = block_inclusive_sum(tiles, warp_sums);
    if (e < E) {
        const int start = rows_incl - c4;
        row_off[e] = start;
        row_end[e] = start + c;
        tile_off[e + 1] = tiles_incl;
        cursor[e] = start;
        for (int p = start + c; p < start + c4; ++p) perm[p] = -1;   // padding rows
        if (e == E - 1) row_off[E] = rows_incl;
    }
    if (e == 0) tile_off[0] = 0;
    __syncthreads();
    for (int64_t q = threadIdx.x; q < P; q += RT_THREADS) {
        const int ex = ids[q];
        if (ex >= 0 && ex < E) perm[atomicAdd(&cursor[ex], 1)] = static_cast<int>(q);
    }
}

// Routed row p <- token perm[p] / top_k: fp16 operand planes as the plain
// preparation writes them (each aligned group of 4 values in the K order
// 0, 2, 1, 3; bsums in fp16; d transposed).  Padding rows (perm -1) and rows
// from row_off[E] on are zero.
__global__ void xgather_kernel(const int8_t* __restrict__ qs, const float* __restrict__ d,
                               const int16_t* __restrict__ bsums, int64_t K, int top_k, const int* __restrict__ perm,
                               const int* __restrict__ rows_valid, int64_t P, __half* __restrict__ xh,
                               __half* __restrict__ xbs, float* __restrict__ dxT, int64_t Pp) {
    const int64_t nb = K >> 8, g16 = K >> 4;   // blocks and 16-value groups per row
    const int64_t valid = *rows_valid;
    const int64_t n16 = P * g16;
    const int64_t ndx = nb * Pp;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16 + ndx; i += stride) {
        if (i < n16) {
            const int64_t p = i / g16, g = i - p * g16;
            uint4* dst = reinterpret_cast<uint4*>(xh) + 2 * i;
            if (p >= valid || perm[p] < 0) {
                dst[0] = make_uint4(0u, 0u, 0u, 0u);
                dst[1] = make_uint4(0u, 0u, 0u, 0u);
                xbs[i] = __float2half_rn(0.0f);
                continue;
            }
            const int64_t src = static_cast<int64_t>(perm[p] / top_k) * g16 + g;
            const int4 raw = *(reinterpret_cast<const int4*>(qs) + src);
            const int w[4] = {raw.x, raw.y, raw.z, raw.w};
            uint32_t o[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int lo = static_cast<int8_t>((w[j] >> (8 * h)) & 0xff);
                    const int hi = static_cast<int8_t>((w[j] >> (8 * h + 16)) & 0xff);
                    const __half2 pr = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
                    o[2 * j + h] = *reinterpret_cast<const uint32_t*>(&pr);
                }
            }
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            xbs[i] = __int2half_rn(bsums[src]);
        } else {
            const int64_t j = i - n16;
            const int64_t b = j / Pp;
            const int64_t p = j - b * Pp;
            dxT[j] = (p < valid && perm[p] >= 0) ? d[static_cast<int64_t>(perm[p] / top_k) * nb + b] : 0.0f;
        }
    }
}

int grid_for(int64_t work, int threads) {
    int64_t g = (work + threads - 1) / threads;
    if (g > 65535) g = 65535;
    if (g < 1) g = 1;
    return static_cast<int>(g);
}

}  // namespace

cudaError_t launch_route(const int32_t* ids, int64_t P, int E, int bm, int* row_off, int* row_end, int* tile_off,
                         int* perm, uint32_t* status, cudaStream_t s) {
    if (E < 1 || E > ROUTE_MAX_EXPERTS) return cudaErrorInvalidValue;
    route_kernel<<<1, RT_THREADS, 0, s>>>(ids, P, E, bm, row_off, row_end, tile_off, perm, status);
    return cudaGetLastError();
}

cudaError_t launch_xgather(const int8_t* qs, const float* d, const int16_t* bsums, int64_t K, int top_k,
                           const int* perm, const int* rows_valid, int64_t P, __half* xh, __half* xbs, float* dxT,
                           int64_t Pp, cudaStream_t s) {
    const int64_t work = P * (K >> 4) + (K >> 8) * Pp;
    xgather_kernel<<<grid_for(work, 256), 256, 0, s>>>(qs, d, bsums, K, top_k, perm, rows_valid, P, xh, xbs, dxT,
                                                      Pp);
    return cudaGetLastError();
}

}  // namespace qg
