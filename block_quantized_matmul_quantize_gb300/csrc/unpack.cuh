// unpack.cuh -- the branch-free weight expanders of the tile GEMM: one
// thread turns its weight row's block into the fp16 operand the tensor core
// multiplies (exact integers, or d-scaled exact values for PTQ1_0), plus the
// per-superblock side values (the Q4_K dmin-correction operands and the
// epilogue scale).  Shared by the GEMM kernel and by the test-only expansion
// kernel (unpack_check.cu), so that the tests check the very code the GEMM runs.
//
// The weight formats ("perf(KERNEL-QUANT-CIQ-GEMM-ROCM): cooperative-tile
// WMMA kernels", vllm.cpp PR #3036, commits 1 and 4; "cuda: branch-free
// PTQ1_0 MMQ tile loader ...", llama.cpp PR #214):
//   Q4_K: w = d*sc_j*q - dmin*m_j, sc_j, m_j 6-bit, q 4-bit;
//   Q6_K: w = d*sc_j*(q - 32), sc_j int8, q 6-bit;
//   PTQ1_0: w = d*(t - 1), t a base-3 digit.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace qg {
namespace {

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
__device__ __forceinline__ uint32_t hadd2u(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// Byte B of w as an exact fp16 in both halves, without a conversion
// instruction: the byte under the exponent byte 0x64 is the fp16 1024 + v,
// and subtracting 1024 leaves v.  Unsigned bytes (0..255); for a signed byte
// pass w ^ 0x80808080 and subtract 1152 (1024 + 128) instead.
template <int B>
__device__ __forceinline__ uint32_t byte_h2(uint32_t w, uint32_t minus_bias) {
    constexpr uint32_t sel = B | (4u << 4) | (B << 8) | (4u << 12);   // w[B], 0x64, w[B], 0x64
    return hadd2u(__byte_perm(w, 0x64646464u, sel), minus_bias);
}
constexpr uint32_t H2_M1024 = 0xE400E400u;   // fp16 -1024 in both halves
constexpr uint32_t H2_M1152 = 0xE480E480u;   // fp16 -1152
constexpr uint32_t H2_1_16 = 0x2C002C00u;    // fp16 1/16
constexpr uint32_t H2_M64 = 0xD400D400u;     // fp16 -64

__device__ __forceinline__ uint32_t h2dup(__half h) {
    const uint32_t u = __half_as_ushort(h);
    return u | (u << 16);
}

// ---------------------------------------------------------------- unpack
// Both expanders write the K positions of every aligned group of 4 in the
// order 0, 2, 1, 3 (fp16 pair (w[4k], w[4k+2]), then (w[4k+1], w[4k+3])):
// two weights two bytes apart sit in one 32-bit word with no byte permute.
// The activation operand (xh) is written in the same order, so the MMA's
// dot products are unchanged; groups of 4 never straddle a 16-value group,
// so the bsums are unchanged too.
//
// Q4_K: expand K64 chunk c of one 144-byte block into 64 fp16 values sc_j*q:
// words 0..15 from the low nibbles (sub-block 2c), words 16..31 from the high
// nibbles (sub-block 2c+1).
__device__ __forceinline__ void unpack_q4k_chunk(const uint8_t* blk, int c, uint32_t scL, uint32_t cL,
                                                 uint32_t scH, uint32_t cH, uint32_t (&o)[32]) {
    const uint4 q0 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c + 16);
    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    constexpr uint32_t MAGIC = 0x64006400u;  // fp16 1024 in both halves
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        // bytes 4k..4k+3 hold weights 4k..4k+3 (low nibbles) and 32+4k.. (high nibbles)
        const uint32_t wk = w[k], sk = w[k] >> 8;
        o[2 * k] = hfma2u((wk & 0x000F000Fu) | MAGIC, scL, cL);           // (1024+q)*sc - 1024*sc
        o[2 * k + 1] = hfma2u((sk & 0x000F000Fu) | MAGIC, scL, cL);
        o[16 + 2 * k] = hfma2u((wk & 0x00F000F0u) | MAGIC, scH, cH);      // (1024+16q)*sc/16 - 64*sc
        o[17 + 2 * k] = hfma2u((sk & 0x00F000F0u) | MAGIC, scH, cH);
    }
}

// Q4_K operand range.  The operand sc_j*q is exact in fp16, but the dmin
// correction operands m_j*r, r = -dmin/d, overflow fp16 (65504) once |r|
// passes about 1000.  A block whose ratio is that large is computed on a
// power-of-two shifted scale instead: operands sc_j*q*2^-s and m_j*r*2^-s,
// epilogue factor e = d*2^s.  The shifted main operand stays exact: sc_j*q
// is an integer below 2^10 and 2^-s >= 2^-14 keeps it a normal fp16.  The
// shift is a function of the exponents of d and dmin alone (integer
// operations on the fp16 fields, so that the unpack and the side-data writer
// agree on it bit for bit):
//   s = clamp(E(dmin) - E(d) - 8, 0, 14),  E = floor(log2 |x|),
// 0 when d or dmin is zero; it gives |r|*2^-s < 2^9 whenever the clamp does
// not bind.
__device__ __forceinline__ int h_floor_log2(uint32_t h) {   // fp16 bits, nonzero magnitude
    const int ex = static_cast<int>((h >> 10) & 0x1fu);
    return ex != 0 ? ex - 15 : (31 - __clz(static_cast<int>(h & 0x3ffu))) - 24;
}
__device__ __forceinline__ int q4k_shift_hdr(uint32_t hx) {   // hx: fp16 d in bits 0..15, dmin in 16..31
    const uint32_t hd = hx & 0x7fffu, hm = (hx >> 16) & 0x7fffu;
    if (hd == 0u || hm == 0u) return 0;
    const int s = h_floor_log2(hm) - h_floor_log2(hd) - 8;
    return s < 0 ? 0 : (s > 14 ? 14 : s);
}
// At the largest shift the correction can still leave fp16's range: the row
// is then declined.  Both the side-data writer (which makes its e NaN) and
// the unpack (which records the status bit) take this decision from the same
// fp32 arithmetic: 63 * |r * 2^-14| <= 65504, i.e. |r * 2^-14| <= 1039.
__device__ __forceinline__ float q4k_ratio(uint32_t hx, int s) {   // r * 2^-s, d != 0
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hx & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hx >> 16)));
    return (-dmin / d) * __uint_as_float(static_cast<uint32_t>(127 - s) << 23);
}
__device__ __forceinline__ bool q4k_in_range(int s, float ratio) { return s != 14 || fabsf(ratio) <= 1039.0f; }
// s can be nonzero only for a subnormal d or a dmin whose exponent field is 9
// or more above d's (d = 0 is caught here too, and gives s = 0): a test of
// the two exponent fields, so that the usual block pays for nothing
// more.
__device__ __forceinline__ bool q4k_maybe_shifted(uint32_t hx) {
    const uint32_t ed = (hx >> 10) & 0x1fu, em = (hx >> 26) & 0x1fu;
    return ed == 0u || em >= ed + 9u;
}
// fp16 2^-s in both halves (0 <= s <= 14: a normal fp16)
__device__ __forceinline__ uint32_t h2_pow2m(int s) {
    const uint32_t b = static_cast<uint32_t>(15 - s) << 10;
    return b | (b << 16);
}

// (e, r * 2^-s) of a block that q4k_maybe_shifted flags; (e0, r0) when its
// shift is 0; e = NaN when the row is declined.
static __device__ __noinline__ float2 q4k_shifted_side(uint32_t hx, float e0, float r0) {
    const int s = q4k_shift_hdr(hx);
    if (s == 0) return make_float2(e0, r0);
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hx & 0xffffu)));
    const float ratio = q4k_ratio(hx, s);
    const float e = q4k_in_range(s, ratio) ? d * __uint_as_float(static_cast<uint32_t>(127 + s) << 23)
                                           : __uint_as_float(0x7fc00000u);
    return make_float2(e, ratio);
}

// Q4_K side values of one block row, from its 16-byte header (fp16 d, fp16
// dmin, 12 scale bytes): the epilogue factor e = d * 2^s and the correction
// operands a1[j] + a2[j] = m_j * r * 2^-s (fp16 hi + lo, about 22
// significant bits; each duplicated into both halves, one per 16-value group
// of sub-block j), handed to put(j, a1[j], a2[j]).  d = 0: the main operand
// is zeroed, e = dmin and r = -1 (exact).  A declined row (q4k_in_range) gets
// e = NaN: its outputs become NaN rather than a wrong number.  (No status
// write here: in the tile GEMM this runs beside 64 live accumulators at the
// register limit; the unpack records the status bit instead.)
template <typename Put>
__device__ __forceinline__ void q4k_side(uint4 hdr, float& e, Put&& put) {
    const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x & 0xffffu)));
    const float dmin = __half2float(__ushort_as_half(static_cast<unsigned short>(hdr.x >> 16)));
    const uint32_t mn03 = hdr.z & 0x3f3f3f3fu;
    const uint32_t mn47 = ((hdr.w >> 4) & 0x0f0f0f0fu) | ((hdr.z >> 2) & 0x30303030u);
    const bool main_on = (d != 0.0f);
    e = main_on ? d : dmin;
    float ratio = main_on ? -dmin / d : -1.0f;
    if (q4k_maybe_shifted(hdr.x)) {   // rare: e and r for the row's shift (NaN e if declined)
        const float2 er = q4k_shifted_side(hdr.x, e, ratio);
        e = er.x;
        ratio = er.y;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int mj = ((j < 4 ? mn03 : mn47) >> (8 * (j & 3))) & 0xff;
        const float v = static_cast<float>(mj) * ratio;
        const __half h1 = __float2half_rn(v);
        const __half h2 = __float2half_rn(v - __half2float(h1));
        put(j, h2dup(h1), h2dup(h2));
    }
}

// Q6_K sub-scale split.  The operand sc_j*(q - 32) is an integer of up to
// 128*32 = 4096; fp16 holds every integer up to 2048 but only even ones
// above, so for |sc_j| > 64 an odd product would round.  The scale is split
// as sc_j = hi_j + lo_j with lo_j = 1 exactly when |sc_j| > 64 and sc_j is
// odd (else 0): hi_j*(q - 32) is then either at most 2048 or even and at most
// 4096, lo_j*(q - 32) at most 32, both exact, and the tensor core adds the
// two parts into the same accumulator.  Four int8 scales per word, bytewise.
// For an odd int8 byte, |sc| > 64 exactly when its bits 7 and 6 differ
// (65..127 is 01xxxxxx, -127..-65 is 10xxxxxx), so lo is bit 0 of
// sc & (sc >> 7 ^ sc >> 6) in each byte, and hi = sc - lo clears that bit.
__device__ __forceinline__ void q6k_split(uint32_t sw, uint32_t& hi, uint32_t& lo) {
    lo = sw & ((sw >> 7) ^ (sw >> 6)) & 0x01010101u;
    hi = sw & ~lo;
}
// Four int8 scales (one word) -> four fp16 pairs (each scale in both halves).
__device__ __forceinline__ void q6k_scales_h2(uint32_t scw, uint32_t (&s4)[4]) {
    const uint32_t u = scw ^ 0x80808080u;   // signed bytes, offset by 128
    s4[0] = byte_h2<0>(u, H2_M1152);
    s4[1] = byte_h2<1>(u, H2_M1152);
    s4[2] = byte_h2<2>(u, H2_M1152);
    s4[3] = byte_h2<3>(u, H2_M1152);
}

// Q6_K: K64 chunk c = weights 64c..64c+63 of a 224-byte packed block, as
// fp16 (q-32)*sc.  Half h = c/2; low nibbles for c even, high for c odd; qh
// bits 4*(c&1) + 2*pp for the first (pp = 0) and second (pp = 1) 32 weights.
__device__ __forceinline__ void unpack_q6k_chunk(const uint8_t* blk, int c, const uint32_t (&s4)[4],
                                                 uint32_t (&o)[32]) {
    const int h = c >> 1, hn = c & 1;
    const uint4* Lp = reinterpret_cast<const uint4*>(blk + 64 * h);
    const uint4* Hp = reinterpret_cast<const uint4*>(blk + 128 + 32 * h);
    const uint4 l0 = Lp[0], l1 = Lp[1], l2 = Lp[2], l3 = Lp[3];
    const uint4 h0 = Hp[0], h1 = Hp[1];
    const uint32_t Lw[16] = {l0.x, l0.y, l0.z, l0.w, l1.x, l1.y, l1.z, l1.w,
                             l2.x, l2.y, l2.z, l2.w, l3.x, l3.y, l3.z, l3.w};
    const uint32_t Hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    constexpr uint32_t MAGIC = 0x64006400u;
    constexpr uint32_t OFF = 0x64206420u;  // fp16 1056 = 1024 + 32 in both halves
    const int nsh = 4 * hn;                 // low or high nibble
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            // 6-bit codes of weights 32pp+4k .. +3, one per byte
            const uint32_t q6 = ((Lw[8 * pp + k] >> nsh) & 0x0F0F0F0Fu) |
                                (((Hw[k] >> (nsh + 2 * pp)) << 4) & 0x30303030u);
            const uint32_t sc = s4[2 * pp + (k >> 2)];
            // bytes 0, 2 (a) and 1, 3 (b) of q6 under the fp16 exponent byte 0x64:
            // 1024 + q, one byte permute each (measured on GB300: 3.5% off the
            // M=512 K=11008 N=2048 GEMM against a mask-and-or and a shift)
            const uint32_t a = __byte_perm(q6, MAGIC, 0x7250);
            const uint32_t b = __byte_perm(q6, MAGIC, 0x7351);
            o[16 * pp + 2 * k] = hmul2u(hsub2u(a, OFF), sc);        // (q - 32) * sc, exact
            o[16 * pp + 2 * k + 1] = hmul2u(hsub2u(b, OFF), sc);
        }
    }
}

// PTQ1_0 ("cuda: branch-free PTQ1_0 MMQ tile loader ...", llama.cpp PR
// #214): one 32-byte block (28 + 4 zero) -> its 128 weights as fp16
// (t - 1) * d, weights 0..63 in v0 and 64..127 in v1, each aligned group of 4
// in the K order 0, 2, 1, 3.  Weight 24 i + 4 w + b (b < 4) is base-3 digit i
// of qs byte 4 w + b, so a qs word and a digit give one aligned group of 4:
// bytes 0 and 2 of the word (16-bit lanes of w & 0x00ff00ff) hold weights b =
// 0 and 2, bytes 1 and 3 weights 1 and 3.  One division by 3 per digit and
// lane pair, x / 3 = (x * 171) >> 9 (exact for x < 256, no carry between the
// lanes); the digit lands in bits 0-1 of its lane, under the fp16 exponent
// 0x64 (1024 + t), and (1024 + t - 1025) * d is exact.  Weights 120 + r are
// digit r / 2 of qh byte r % 2.  No branch depends on the lane or the data.
// Expanded in two halves (v0 = weights 0..63, then v1 = 64..127), so that
// only one half and the words' lane pairs after two divisions (st) are live:
// weights 0..63 are digits 0 and 1 of every qs word and digit 2 of words 0..3.
struct Ptq1State {
    uint32_t xl[6], xh[6];   // each word's lane pairs divided by 9
    uint32_t tail, d2;
};
__device__ __forceinline__ uint32_t ptq1_val(uint32_t t2, uint32_t d2) {
    // (1024 + t - 1025) * d: exact in fp16 for t in {0, 1, 2}
    return hmul2u(hadd2u(t2 | 0x64006400u, 0xE401E401u), d2);
}
__device__ __forceinline__ void ptq1_div3(uint32_t x, uint32_t& q, uint32_t& t) {
    q = ((x * 171u) >> 9) & 0x007f007fu;   // x / 3 in both 16-bit lanes (x < 256)
    t = x - 3u * q;
}
__device__ __forceinline__ void unpack_ptq1_lo(const uint8_t* blk, Ptq1State& st, uint32_t (&v0)[32]) {
    const uint4 a = *reinterpret_cast<const uint4*>(blk);
    const uint4 b = *reinterpret_cast<const uint4*>(blk + 16);
    const uint32_t qw[6] = {a.x, a.y, a.z, a.w, b.x, b.y};
    st.tail = b.z;                                   // qh[0] | qh[1] << 8 | d << 16
    st.d2 = (st.tail >> 16) * 0x10001u;              // fp16 d in both halves
#pragma unroll
    for (int w = 0; w < 6; ++w) {
        uint32_t xl = qw[w] & 0x00ff00ffu, xh = (qw[w] >> 8) & 0x00ff00ffu, ql, qh, tl, th;
#pragma unroll
        for (int i = 0; i < 2; ++i) {                // weights 24 i + 4 w .. + 3
            ptq1_div3(xl, ql, tl);
            ptq1_div3(xh, qh, th);
            v0[12 * i + 2 * w] = ptq1_val(tl, st.d2);
            v0[12 * i + 2 * w + 1] = ptq1_val(th, st.d2);
            xl = ql;
            xh = qh;
        }
        st.xl[w] = xl;
        st.xh[w] = xh;
        if (w < 4) {                                 // digit 2 of words 0..3: weights 48 + 4 w
            ptq1_div3(xl, ql, tl);
            ptq1_div3(xh, qh, th);
            v0[24 + 2 * w] = ptq1_val(tl, st.d2);
            v0[25 + 2 * w] = ptq1_val(th, st.d2);
        }
    }
}
__device__ __forceinline__ void unpack_ptq1_hi(const Ptq1State& st, uint32_t (&v1)[32]) {
#pragma unroll
    for (int w = 0; w < 6; ++w) {
        uint32_t xl = st.xl[w], xh = st.xh[w], ql, qh, tl, th;
#pragma unroll
        for (int i = 2; i < 5; ++i) {
            ptq1_div3(xl, ql, tl);
            ptq1_div3(xh, qh, th);
            const int k = 24 * i + 4 * w;            // first weight of the group
            if (k >= 64) {                           // (digit 2 of words 0..3 went to v0)
                v1[(k - 64) >> 1] = ptq1_val(tl, st.d2);
                v1[((k - 64) >> 1) + 1] = ptq1_val(th, st.d2);
            }
            xl = ql;
            xh = qh;
        }
    }
    // qh[0] in lane 0, qh[1] in lane 1: digits i of both bytes per step
    uint32_t x = (st.tail & 0xffu) | ((st.tail & 0xff00u) << 8), dg[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t q;
        ptq1_div3(x, q, dg[i]);
        x = q;
    }
    // group 120..123: (qh0 digit 0, qh0 digit 1), (qh1 digit 0, qh1 digit 1); 124..127 with digits 2, 3
    v1[28] = ptq1_val(__byte_perm(dg[0], dg[1], 0x5410), st.d2);
    v1[29] = ptq1_val(__byte_perm(dg[0], dg[1], 0x7632), st.d2);
    v1[30] = ptq1_val(__byte_perm(dg[2], dg[3], 0x5410), st.d2);
    v1[31] = ptq1_val(__byte_perm(dg[2], dg[3], 0x7632), st.d2);
}


// ---- one K64 chunk of one block row, as the tile GEMM stores it in TMEM ----
// Column j (0..31) of chunk c holds the fp16 pair of weights k and k + 2 with
// k = 64c + 4*(j/2) + (j%2): each aligned group of four weights in the K order
// 0, 2, 1, 3 (the activation operand uses the same order).

// Q4_K: the scale words of chunks 0-1 (sc_0..sc_3) and 2-3 (sc_4..sc_7), zero
// when d = 0 (the main part vanishes), and the operand scale 2^-s.
struct Q4kScales {
    uint32_t sc03, sc47;
    uint32_t p2;       // fp16 2^-s in both halves
    bool shifted;      // s > 0 (rare)
    bool declined;     // the row is out of range even at the largest shift
};
// The rare branches below are out of line (the tile GEMM's role loops stay
// compact; measured on GB300, inlined they cost 4-5% on every call, not only
// on the rare blocks).  Bits 0-4: s; bit 5: declined.
static __device__ __noinline__ uint32_t q4k_shift_info(uint32_t hx) {
    const int s = q4k_shift_hdr(hx);
    const bool declined = s == 14 && (hx & 0x7fffu) != 0u && !q4k_in_range(s, q4k_ratio(hx, s));
    return static_cast<uint32_t>(s) | (declined ? 32u : 0u);
}
__device__ __forceinline__ Q4kScales q4k_scales(uint4 hdr) {
    const bool main_on = (hdr.x & 0x7fffu) != 0u;   // d != 0
    Q4kScales r;
    r.sc03 = main_on ? (hdr.y & 0x3f3f3f3fu) : 0u;
    r.sc47 = main_on ? ((hdr.w & 0x0f0f0f0fu) | ((hdr.y >> 2) & 0x30303030u)) : 0u;
    r.p2 = 0x3C003C00u;   // fp16 1
    r.shifted = false;
    r.declined = false;
    if (q4k_maybe_shifted(hdr.x)) {   // rare
        const uint32_t info = q4k_shift_info(hdr.x);
        r.p2 = h2_pow2m(static_cast<int>(info & 31u));
        r.shifted = (info & 31u) != 0u;
        r.declined = (info & 32u) != 0u;
    }
    return r;
}
// Chunk c (its parity CI = c % 2 picks bytes 2CI, 2CI+1 of the scale word):
// sc_j * q * 2^-s.  (The low nibbles take sc and -1024 sc, the high ones sc/16
// and -64 sc; every factor and result is exact in fp16.)
template <int CI>
__device__ __forceinline__ void q4k_expand(const uint8_t* blk, int c, uint32_t scw, const Q4kScales& qs4,
                                           uint32_t (&o)[32]) {
    uint32_t sl = byte_h2<2 * CI>(scw, H2_M1024);
    uint32_t sh = byte_h2<2 * CI + 1>(scw, H2_M1024);
    if (qs4.shifted) {
        sl = hmul2u(sl, qs4.p2);
        sh = hmul2u(sh, qs4.p2);
    }
    unpack_q4k_chunk(blk, c, sl, hmul2u(sl, H2_M1024), hmul2u(sh, H2_1_16), hmul2u(sh, H2_M64), o);
}
// Q6_K chunk c, scale word scw (the chunk's four int8 sub-scales): the hi
// part (q - 32) * hi_j; `slo` gets the lo scales (bytes 0 or 1).
__device__ __forceinline__ void q6k_expand_hi(const uint8_t* blk, int c, uint32_t scw, uint32_t& slo,
                                              uint32_t (&o)[32]) {
    uint32_t shi;
    q6k_split(scw, shi, slo);
    uint32_t s4[4];
    q6k_scales_h2(shi, s4);
    unpack_q6k_chunk(blk, c, s4, o);
}
// The lo part (q - 32) * lo_j of chunk c.
__device__ __forceinline__ void q6k_expand_lo(const uint8_t* blk, int c, uint32_t slo, uint32_t (&o)[32]) {
    uint32_t s4[4];   // unsigned bytes 0 or 1
    s4[0] = byte_h2<0>(slo, H2_M1024);
    s4[1] = byte_h2<1>(slo, H2_M1024);
    s4[2] = byte_h2<2>(slo, H2_M1024);
    s4[3] = byte_h2<3>(slo, H2_M1024);
    unpack_q6k_chunk(blk, c, s4, o);
}

}  // namespace
}  // namespace qg
