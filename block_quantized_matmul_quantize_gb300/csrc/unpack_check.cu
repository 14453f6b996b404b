// unpack_check.cu -- the tile GEMM's weight expansion on its own, for tests:
// qgemm_debug_expand runs the expanders of unpack.cuh (the very functions
// the GEMM's unpack warps call) over an array of blocks and writes what the
// GEMM would put into tensor memory and into its side data, so that the
// expansion can be compared with a CPU decoding of the same bytes block by
// block, without the multiply in between.
#include <cuda_fp16.h>

#include "internal.h"
#include "qgemm.h"
#include "unpack.cuh"

namespace qg {
namespace {

constexpr int REC_WORDS = QGEMM_DEBUG_EXPAND_BYTES / 4;

// One thread per superblock row.  Record layout (32-bit words):
//   [0, 128)    main (hi) operand, chunk c in words 32c..32c+31 (TMEM columns)
//   [128, 256)  Q6_K lo operand (zero elsewhere)
//   [256, 264)  Q4_K correction operands a1[j], [264, 272) a2[j]
//   [272]       epilogue factor e (fp32 bits)
//   [273]       bit 0: the block is in range; bits 8..15: the Q4_K shift s
template <int WT>
__global__ void expand_kernel(const uint8_t* __restrict__ blocks, int64_t n, uint32_t* __restrict__ out) {
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n) return;
    uint32_t* rec = out + i * REC_WORDS;
    uint32_t v[32];
    if constexpr (WT == 4) {
        const uint8_t* blk = blocks + i * Q4K_BLOCK;
        const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
        const Q4kScales qs4 = q4k_scales(hdr);
        for (int c = 0; c < 4; ++c) {
            const uint32_t scw = c < 2 ? qs4.sc03 : qs4.sc47;
            if (c & 1)
                q4k_expand<1>(blk, c, scw, qs4, v);
            else
                q4k_expand<0>(blk, c, scw, qs4, v);
            for (int k = 0; k < 32; ++k) rec[32 * c + k] = v[k];
        }
        for (int k = 0; k < 128; ++k) rec[128 + k] = 0u;
        float e;
        q4k_side(hdr, e, [&](int j, uint32_t w1, uint32_t w2) {
            rec[256 + j] = w1;
            rec[264 + j] = w2;
        });
        rec[272] = __float_as_uint(e);
        const bool ok = !qs4.declined;
        rec[273] = (ok ? 1u : 0u) | (static_cast<uint32_t>(q4k_shift_hdr(hdr.x)) << 8);
    } else if constexpr (WT == 6) {
        const uint8_t* blk = blocks + i * Q6K_PACKED;
        const uint4 scv = *reinterpret_cast<const uint4*>(blk + 192);
        for (int c = 0; c < 4; ++c) {
            uint32_t slo;
            q6k_expand_hi(blk, c, c == 0 ? scv.x : c == 1 ? scv.y : c == 2 ? scv.z : scv.w, slo, v);
            for (int k = 0; k < 32; ++k) rec[32 * c + k] = v[k];
            q6k_expand_lo(blk, c, slo, v);
            for (int k = 0; k < 32; ++k) rec[128 + 32 * c + k] = v[k];
        }
        for (int k = 256; k < 272; ++k) rec[k] = 0u;
        rec[272] = __float_as_uint(__half2float(*reinterpret_cast<const __half*>(blk + 208)));
        rec[273] = 1u;
    } else {
        // PTQ1_0: a superblock is two repacked 32-byte blocks; block j's 128
        // weights are chunks 2j (lo half) and 2j + 1 (hi half)
        const uint8_t* sb = blocks + i * 2 * PTQ1_PACKED;
        for (int j = 0; j < 2; ++j) {
            Ptq1State st;
            unpack_ptq1_lo(sb + PTQ1_PACKED * j, st, v);
            for (int k = 0; k < 32; ++k) rec[64 * j + k] = v[k];
            unpack_ptq1_hi(st, v);
            for (int k = 0; k < 32; ++k) rec[64 * j + 32 + k] = v[k];
        }
        for (int k = 128; k < 272; ++k) rec[k] = 0u;
        rec[272] = __float_as_uint(1.0f);
        rec[273] = 1u;
    }
    for (int k = 274; k < REC_WORDS; ++k) rec[k] = 0u;
}

}  // namespace
}  // namespace qg

extern "C" int qgemm_debug_expand(int wtype, const void* blocks, int64_t nblocks, void* out, qgemm_stream_t stream) {
    if (wtype != 4 && wtype != 6 && wtype != 1) return qg::set_last_error(QGEMM_EINVAL, "wtype must be 4, 6 or 1");
    if (nblocks < 0) return qg::set_last_error(QGEMM_EINVAL, "nblocks must be >= 0");
    if (nblocks == 0) return QGEMM_OK;
    if (!blocks || !out) return qg::set_last_error(QGEMM_EINVAL, "null pointer");
    if ((reinterpret_cast<uintptr_t>(blocks) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u))
        return qg::set_last_error(QGEMM_EALIGN, "blocks and out must be 16-byte aligned");
    const uint8_t* b = static_cast<const uint8_t*>(blocks);
    uint32_t* o = static_cast<uint32_t*>(out);
    const int threads = 128;
    const unsigned grid = static_cast<unsigned>((nblocks + threads - 1) / threads);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (wtype == 4)
        qg::expand_kernel<4><<<grid, threads, 0, s>>>(b, nblocks, o);
    else if (wtype == 6)
        qg::expand_kernel<6><<<grid, threads, 0, s>>>(b, nblocks, o);
    else
        qg::expand_kernel<1><<<grid, threads, 0, s>>>(b, nblocks, o);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return qg::set_last_error(QGEMM_ECUDA, cudaGetErrorString(e));
    return QGEMM_OK;
}
