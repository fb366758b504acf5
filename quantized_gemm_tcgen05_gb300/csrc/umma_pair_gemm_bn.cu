// Instantiations of the CTA-pair tcgen05 GEMM kernel.
#include "umma_pair_gemm.cuh"

namespace qg {
#define QG_INST(B)                                                                                       \
    template cudaError_t launch_pair_bn<B>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t); \
    template int pair_stages_bn<B>(int);                                                                    \
    template int pair_max_clusters_bn<B>();
QG_FOR_EACH_PAIR_BN(QG_INST)
#undef QG_INST
}  // namespace qg
