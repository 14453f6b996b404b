// gemm_tc_epi.cu -- the tile GEMM with the output epilogue compiled in
// (bias, activation, fp16/bf16 output); a translation unit of its own so
// that the two sets of instantiations build in parallel.
#include "gemm_tc_kernel.cuh"

namespace qg {

cudaError_t tc_prepare_epi(int wtype, int bm) {
#define QG_CASE(W, B) \
    if (wtype == W && bm == B) return prepare_t<W, B, VAR_EPI>();
    QG_CASE(4, 16) QG_CASE(4, 32) QG_CASE(4, 64) QG_CASE(4, 128)
    QG_CASE(6, 16) QG_CASE(6, 32) QG_CASE(6, 64) QG_CASE(6, 128)
#undef QG_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc_epi(const TcLaunch& a, cudaStream_t s) {
#define QG_CASE(W, B) \
    if (a.wtype == W && a.bm == B) return launch_t<W, B, VAR_EPI>(a, s);
    QG_CASE(4, 16) QG_CASE(4, 32) QG_CASE(4, 64) QG_CASE(4, 128)
    QG_CASE(6, 16) QG_CASE(6, 32) QG_CASE(6, 64) QG_CASE(6, 128)
#undef QG_CASE
    return cudaErrorInvalidValue;
}

}  // namespace qg
