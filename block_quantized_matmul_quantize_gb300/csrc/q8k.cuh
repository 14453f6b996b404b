// q8k.cuh -- the Q8_K value arithmetic, shared by the quantizer kernel and the
// small-M kernel's fused path (which quantizes its activations itself).
//
// Q8_K, as the library defines it (the block the pages call "BlockQ8_K,
// 292 B / 256 elements", vllm.cpp PR #3036, commit 4): per 256-element chunk
// of a row, d = amax/127 (fp32), q = round-half-away-from-zero(x/d) clamped to
// +-127.  d = 0 (amax = 0, or amax/127 underflowing to zero) gives all-zero q.
// x/d and amax/127 are IEEE fp32 divisions, correctly rounded (the library is
// built without fast-math; -prec-div=true), and roundf rounds halves away from
// zero, so every caller of these helpers gets the same bits.
#pragma once
#include <cuda_runtime.h>

namespace qg {

// round-half-away(x / d) of one element, by the IEEE definition: x / d
// correctly rounded, then halves away from zero, clamped to +-127.
__device__ __forceinline__ int q8_exact(float x, float d) {
    const float r = fminf(fmaxf(roundf(x / d), -127.0f), 127.0f);
    return static_cast<int>(r);
}

// The same value for a normal d (d >= 2^-126), cheaper: r = x * RN(1/d) is
// within 2^-23 * |x/d| <= 1.52e-5 of x/d, and the correctly rounded x / d
// within 7.6e-6 of it, so they round to the same integer unless r lies
// within 2.3e-5 of a half-integer.  a = |r| + 0.5 is rounded by at most
// 2^-18, so if a is more than 2^-14 from an integer, floor(a) is that
// integer and the result equals q8_exact; otherwise q8_exact decides (about
// one element in 10^4 of normal data).  |r| <= 127.00002 needs no clamp.
// (Products and sums with the _rn intrinsics: no contraction into an FMA.)
__device__ __forceinline__ int q8_fast(float x, float y, float d) {
    constexpr float TH = 6.103515625e-05f;   // 2^-14
    const float r = __fmul_rn(x, y);
    const float a = __fadd_rn(fabsf(r), 0.5f);
    const int qa = __float2int_rz(a);
    const float t = __fsub_rn(a, __int2float_rn(qa));
    if (t < TH || t > 1.0f - TH) return q8_exact(x, d);
    return r < 0.0f ? -qa : qa;
}

// d of a chunk from its amax (over all 256 values), and this thread's NV
// values of the chunk quantized with it; returns d.
template <int NV>
__device__ __forceinline__ float q8k_quantize(const float (&v)[NV], float amax, int (&q)[NV]) {
    const float d = amax / 127.0f;
    if (d >= 1.17549435e-38f) {
        // a normal scale (the usual case): one reciprocal
        const float y = __frcp_rn(d);
#pragma unroll
        for (int i = 0; i < NV; ++i) q[i] = q8_fast(v[i], y, d);
    } else if (d == 0.0f) {
        // amax == 0, or amax/127 underflows to zero: the chunk quantizes to zero
#pragma unroll
        for (int i = 0; i < NV; ++i) q[i] = 0;
    } else {
        // a subnormal scale: the division itself
#pragma unroll
        for (int i = 0; i < NV; ++i) q[i] = q8_exact(v[i], d);
    }
    return d;
}

}  // namespace qg
