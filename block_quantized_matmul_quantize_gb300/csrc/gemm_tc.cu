// gemm_tc.cu -- the tile GEMM's plain instantiations (fp32 output, no
// epilogue, host work list) and its host dispatch; the kernel is in
// gemm_tc_kernel.cuh, the epilogue, routed and Q4_K self-side instantiations
// in gemm_tc_epi.cu, gemm_tc_routed.cu, gemm_tc_self.cu and
// gemm_tc_epi_self.cu (built in parallel).
#include "gemm_tc_kernel.cuh"

namespace qg {

size_t tc_smem_bytes(int wtype, int bm) {
#define QG_CASE(W, B) \
    if (wtype == W && bm == B) return Layout<W, B>::TOTAL;
    QG_CASE(4, 16) QG_CASE(4, 32) QG_CASE(4, 64) QG_CASE(4, 128)
    QG_CASE(6, 16) QG_CASE(6, 32) QG_CASE(6, 64) QG_CASE(6, 128)
    QG_CASE(1, 16) QG_CASE(1, 32) QG_CASE(1, 64) QG_CASE(1, 128)
#undef QG_CASE
    return 0;
}

cudaError_t tc_prepare(int wtype, int bm) {
    if (wtype == 4 || wtype == 6) {   // (the epilogue and routed variants: Q4_K and Q6_K)
        cudaError_t e = tc_prepare_epi(wtype, bm);
        if (e == cudaSuccess) e = tc_prepare_routed(wtype, bm);
        if (e == cudaSuccess && wtype == 4) e = tc_prepare_self(bm);
        if (e == cudaSuccess && wtype == 4) e = tc_prepare_epi_self(bm);
        if (e != cudaSuccess) return e;
    }
#define QG_CASE(W, B) \
    if (wtype == W && bm == B) return prepare_t<W, B, VAR_PLAIN>();
    QG_CASE(4, 16) QG_CASE(4, 32) QG_CASE(4, 64) QG_CASE(4, 128)
    QG_CASE(6, 16) QG_CASE(6, 32) QG_CASE(6, 64) QG_CASE(6, 128)
    QG_CASE(1, 16) QG_CASE(1, 32) QG_CASE(1, 64) QG_CASE(1, 128)
#undef QG_CASE
    return cudaErrorInvalidValue;
}

// The Q4_K side words of every (row, superblock), computed as the side-data
// warps of the other variants compute them (q4k_side), for the plain and
// epilogue variants to load by TMA.  One thread per (superblock, row), rows fastest: each warp
// writes 32 consecutive 32-byte rows of a slab.
__global__ void q4k_side_kernel(const uint8_t* __restrict__ w, int64_t N, int64_t nb, int64_t ldw,
                                uint32_t* __restrict__ side, float* __restrict__ eout, int64_t Np) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= N * nb) return;
    const int64_t b = i / N, n = i - b * N;
    const uint4 hdr = *reinterpret_cast<const uint4*>(w + n * ldw + b * Q4K_BLOCK);
    uint32_t a1[8], a2[8];
    float e;
    q4k_side(hdr, e, [&](int j, uint32_t w1, uint32_t w2) {
        a1[j] = w1;
        a2[j] = w2;
    });
    uint4* s1 = reinterpret_cast<uint4*>(side + ((2 * b) * N + n) * 8);
    uint4* s2 = reinterpret_cast<uint4*>(side + ((2 * b + 1) * N + n) * 8);
    s1[0] = make_uint4(a1[0], a1[1], a1[2], a1[3]);
    s1[1] = make_uint4(a1[4], a1[5], a1[6], a1[7]);
    s2[0] = make_uint4(a2[0], a2[1], a2[2], a2[3]);
    s2[1] = make_uint4(a2[4], a2[5], a2[6], a2[7]);
    eout[b * Np + n] = e;
}

cudaError_t launch_q4k_side(const void* w, int64_t N, int64_t nb, int64_t ldw, uint32_t* side, float* e,
                            int64_t Np, cudaStream_t s) {
    const int64_t n = N * nb;
    q4k_side_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(static_cast<const uint8_t*>(w), N, nb,
                                                                           ldw, side, e, Np);
    return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const TcLaunch& a, cudaStream_t s) {
    if (a.work.experts > 0) return launch_gemm_tc_routed(a, s);
    const bool epi = a.epi.out != OUT_F32 || a.epi.act != ACT_NONE || a.epi.bias != nullptr;
    if (a.wtype == 4 && !a.tm_side) return epi ? launch_gemm_tc_epi_self(a, s) : launch_gemm_tc_self(a, s);
    if (epi) return launch_gemm_tc_epi(a, s);
#define QG_CASE(W, B) \
    if (a.wtype == W && a.bm == B) return launch_t<W, B, VAR_PLAIN>(a, s);
    QG_CASE(4, 16) QG_CASE(4, 32) QG_CASE(4, 64) QG_CASE(4, 128)
    QG_CASE(6, 16) QG_CASE(6, 32) QG_CASE(6, 64) QG_CASE(6, 128)
    QG_CASE(1, 16) QG_CASE(1, 32) QG_CASE(1, 64) QG_CASE(1, 128)
#undef QG_CASE
    return cudaErrorInvalidValue;
}

}  // namespace qg
