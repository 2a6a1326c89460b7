// ge_gemm_epi_gelu_aux.cu -- the tensor-core GEMM kernels with the bias + tanh-GELU + pre-activation epilogue.
#include "ge_gemm_kernel.cuh"

namespace ge {

template cudaError_t launch_tc_gemm_epi<EPI_GELU_AUX_BIAS>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);

}  // namespace ge
