// Instantiations and launcher of the GEMV kernel for 4-bit integer weights.
#include <atomic>

#include "bsgemv_kernel.cuh"

namespace bsg {

template <bool BF16, int MT, bool ZP, bool SUB2>
static int go(const KParams& p, int ctas, int smem, cudaStream_t s) {
  auto k = bsgemv_mma_kernel<kInt4, BF16, MT, ZP, SUB2>;
  static std::atomic<int> attr_smem{0};  // largest dynamic smem already granted to `k`
  if (smem > attr_smem.load()) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return BSGEMV_ERR_CUDA;
    attr_smem.store(smem);
  }
  k<<<ctas, kThreads, smem, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

template <bool BF16, int MT, bool ZP>
static int go2(const KParams& p, bool sub2, int ctas, int smem, cudaStream_t s) {
  return sub2 ? go<BF16, MT, ZP, true>(p, ctas, smem, s) : go<BF16, MT, ZP, false>(p, ctas, smem, s);
}

template <bool BF16, int MT>
static int go3(const KParams& p, bool zp, bool sub2, int ctas, int smem, cudaStream_t s) {
  return zp ? go2<BF16, MT, true>(p, sub2, ctas, smem, s) : go2<BF16, MT, false>(p, sub2, ctas, smem, s);
}

int launch_int4(const KParams& p, int mt, bool bf16, bool zp, bool sub2, int ctas, int smem,
                cudaStream_t s) {
  if (bf16) return mt == 1 ? go3<true, 1>(p, zp, sub2, ctas, smem, s) : go3<true, 2>(p, zp, sub2, ctas, smem, s);
  return mt == 1 ? go3<false, 1>(p, zp, sub2, ctas, smem, s) : go3<false, 2>(p, zp, sub2, ctas, smem, s);
}

}  // namespace bsg
