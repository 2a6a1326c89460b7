// ge_gemm_epi_dgelu.cu -- the tensor-core GEMM kernels with the DGELU_BGRAD epilogue.
#include "ge_gemm_kernel.cuh"

namespace ge {

template cudaError_t launch_tc_gemm_epi<EPI_DGELU_BGRAD>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);

}  // namespace ge
