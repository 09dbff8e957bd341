// Instantiations and launcher of the GEMV kernel for 8-bit integer weights.
#include <atomic>

#include "bsgemv_kernel.cuh"

namespace bsg {

template <bool BF16, int MT, bool ZP>
static int go(const KParams& p, int ctas, int smem, cudaStream_t s) {
  auto k = bsgemv_mma_kernel<kInt8, BF16, MT, ZP, false>;
  static std::atomic<int> attr_smem{0};  // largest dynamic smem already granted to `k`
  if (smem > attr_smem.load()) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return BSGEMV_ERR_CUDA;
    attr_smem.store(smem);
  }
  k<<<ctas, kThreads, smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

template <bool BF16, int MT>
static int go2(const KParams& p, bool zp, int ctas, int smem, cudaStream_t s) {
  return zp ? go<BF16, MT, true>(p, ctas, smem, s) : go<BF16, MT, false>(p, ctas, smem, s);
}

int launch_int8(const KParams& p, int mt, bool bf16, bool zp, int ctas, int smem, cudaStream_t s) {
  if (bf16) return mt == 1 ? go2<true, 1>(p, zp, ctas, smem, s) : go2<true, 2>(p, zp, ctas, smem, s);
  return mt == 1 ? go2<false, 1>(p, zp, ctas, smem, s) : go2<false, 2>(p, zp, ctas, smem, s);
}

}  // namespace bsg
