// gemm_tc.cu -- the tile GEMM's plain instantiations (fp32 output, no
// epilogue, host work list) and its host dispatch; the kernel is in
// gemm_tc_kernel.cuh, the epilogue and routed instantiations in
// gemm_tc_epi.cu and gemm_tc_routed.cu (built in parallel).
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

cudaError_t launch_gemm_tc(const TcLaunch& a, cudaStream_t s) {
    if (a.work.experts > 0) return launch_gemm_tc_routed(a, s);
    if (a.epi.out != OUT_F32 || a.epi.act != ACT_NONE || a.epi.bias != nullptr) return launch_gemm_tc_epi(a, s);
#define QG_CASE(W, B) \
    if (a.wtype == W && a.bm == B) return launch_t<W, B, VAR_PLAIN>(a, s);
    QG_CASE(4, 16) QG_CASE(4, 32) QG_CASE(4, 64) QG_CASE(4, 128)
    QG_CASE(6, 16) QG_CASE(6, 32) QG_CASE(6, 64) QG_CASE(6, 128)
    QG_CASE(1, 16) QG_CASE(1, 32) QG_CASE(1, 64) QG_CASE(1, 128)
#undef QG_CASE
    return cudaErrorInvalidValue;
}

}  // namespace qg
