// Instantiation of the CTA-pair tcgen05 GEMM kernel for tile width 224 (one
// width per translation unit, so they compile in parallel).
#include "umma_pair_gemm.cuh"

namespace qg {
template cudaError_t launch_pair_bn<224>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int pair_stages_bn<224>(int);
template int pair_max_clusters_bn<224>();
}  // namespace qg
