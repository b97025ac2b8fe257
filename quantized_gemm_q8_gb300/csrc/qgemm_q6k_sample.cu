// Instantiations and launcher of the Q6_K GEMM whose LM-head epilogue also draws tokens by the
// Gumbel-max rule (temperature sampling); used only by the LM head with a temperature > 0.
#include "internal.h"
#include "qgemm.cuh"

namespace dllm {

template <int NT>
static int launch_one(const CUtensorMap& map, const QgemmParams& p, int grid, cudaStream_t s) {
  constexpr int SMEM = QCfg<TYPE_Q6K, NT>::SMEM;
  auto* k = &qgemm_kernel<TYPE_Q6K, NT, true>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(qgemm_q6k_sample)");
  e = launch_pdl(k, dim3(grid), dim3(QG_THREADS), SMEM, s, map, p);
  note_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch qgemm_q6k_sample");
  return DLLM_OK;
}

int launch_qgemm_q6k_sample(int nt, const CUtensorMap& map, const QgemmParams& p, int grid, cudaStream_t s) {
  switch (nt) {
    case 32: return launch_one<32>(map, p, grid, s);
    case 64: return launch_one<64>(map, p, grid, s);
    case 128: return launch_one<128>(map, p, grid, s);
    case 160: return launch_one<160>(map, p, grid, s);
    default: return fail(DLLM_E_SHAPE, "qgemm_q6k_sample: unsupported token tile %d", nt);
  }
}

}  // namespace dllm
