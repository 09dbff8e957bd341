// Instantiations and launcher of the GEMV kernel for NVFP4 weights (E2M1 + E4M3 per 16 k).
#include <atomic>

#include "bsgemv_kernel.cuh"

namespace bsg {

template <bool BF16, int MT>
static int go(const KParams& p, int ctas, int smem, cudaStream_t s) {
  auto k = bsgemv_mma_kernel<kNvfp4, BF16, MT, false, false>;
  static std::atomic<int> attr_smem{0};  // largest dynamic smem already granted to `k`
  if (smem > attr_smem.load()) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return BSGEMV_ERR_CUDA;
    attr_smem.store(smem);
  }
  k<<<ctas, kThreads, smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

int launch_nvfp4(const KParams& p, int mt, bool bf16, int ctas, int smem, cudaStream_t s) {
  if (bf16) return mt == 1 ? go<true, 1>(p, ctas, smem, s) : go<true, 2>(p, ctas, smem, s);
  return mt == 1 ? go<false, 1>(p, ctas, smem, s) : go<false, 2>(p, ctas, smem, s);
}

}  // namespace bsg
