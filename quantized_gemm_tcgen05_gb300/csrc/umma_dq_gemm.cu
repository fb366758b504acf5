// Placeholder until the scaled-operand kernel lands.
#include "kparams.h"
namespace qg {
cudaError_t launch_umma_dq_gemm(int, const CUtensorMap&, const CUtensorMap&, const GemmKernelParams&, int,
                                cudaStream_t) {
    return cudaErrorNotSupported;
}
int umma_dq_max_stages(int) { return 0; }
}  // namespace qg
