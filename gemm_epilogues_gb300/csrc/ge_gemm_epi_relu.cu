// ge_gemm_epi_relu.cu -- the tensor-core GEMM kernels with the bias + ReLU epilogue.
#include "ge_gemm_kernel.cuh"

namespace ge {

template cudaError_t launch_tc_gemm_epi<EPI_RELU_BIAS>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);

}  // namespace ge
