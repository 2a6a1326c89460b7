// ge_gemm_epi_none.cu -- the tensor-core GEMM kernels with the no epilogue arithmetic (and the masked-operand weight gradient) epilogue.
#include "ge_gemm_kernel.cuh"

namespace ge {

template cudaError_t launch_tc_gemm_epi<EPI_NONE>(int, int, int, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                                   const GemmArgs&, int, cudaStream_t);

int tc_gemm_max_pairs(int block_n, int num_sms, int epi_warps) {
  if (epi_warps == 8)
    return block_n == 256 ? max_pairs<256, 8>(num_sms) : block_n == 224 ? max_pairs<224, 8>(num_sms) : max_pairs<128, 8>(num_sms);
  return block_n == 256 ? max_pairs<256, 4>(num_sms) : block_n == 224 ? max_pairs<224, 4>(num_sms) : max_pairs<128, 4>(num_sms);
}

}  // namespace ge
