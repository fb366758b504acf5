// Entry points of the scaled-operand tcgen05 GEMM (dispatch over the tile
// widths instantiated in umma_dq_gemm_bn*.cu).
#include "kparams.h"

namespace qg {

cudaError_t launch_umma_dq_gemm(int bn, const GemmMaps& m, const GemmKernelParams& p, int grid,
                                cudaStream_t st) {
    switch (bn) {
#define QG_CASE(B) \
    case B: return launch_dq_bn<B>(m, p, grid, st);
        QG_FOR_EACH_DQ_BN(QG_CASE)
#undef QG_CASE
        default: return cudaErrorInvalidValue;
    }
}

int umma_dq_max_stages(int bn) {
    switch (bn) {
#define QG_CASE(B) \
    case B: return dq_stages_bn<B>();
        QG_FOR_EACH_DQ_BN(QG_CASE)
#undef QG_CASE
        default: return 0;
    }
}

}  // namespace qg
