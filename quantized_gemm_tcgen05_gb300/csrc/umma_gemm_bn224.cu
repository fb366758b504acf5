// Instantiation of the dense tcgen05 GEMM kernel for tile width 224 (one
// width per translation unit, so they compile in parallel).
#include "umma_gemm.cuh"

namespace qg {
template cudaError_t launch_umma_bn<224>(const GemmMaps&, const GemmKernelParams&, int, cudaStream_t);
template int umma_stages_bn<224>(int);
}  // namespace qg
