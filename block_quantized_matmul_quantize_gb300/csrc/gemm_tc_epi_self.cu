// gemm_tc_epi_self.cu -- the Q4_K tile GEMM with the output epilogue that
// makes each weight tile's side words itself (VAR_EPI_SELF); a translation
// unit of its own so that it builds in parallel with the other
// instantiations.
#include "gemm_tc_kernel.cuh"

namespace qg {

cudaError_t tc_prepare_epi_self(int bm) {
#define QG_CASE(B) \
    if (bm == B) return prepare_t<4, B, VAR_EPI_SELF>();
    QG_CASE(16) QG_CASE(32) QG_CASE(64) QG_CASE(128)
#undef QG_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemm_tc_epi_self(const TcLaunch& a, cudaStream_t s) {
#define QG_CASE(B) \
    if (a.wtype == 4 && a.bm == B) return launch_t<4, B, VAR_EPI_SELF>(a, s);
    QG_CASE(16) QG_CASE(32) QG_CASE(64) QG_CASE(128)
#undef QG_CASE
    return cudaErrorInvalidValue;
}

}  // namespace qg
