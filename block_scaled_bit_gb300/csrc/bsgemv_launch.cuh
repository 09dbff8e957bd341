// bsgemv_launch.cuh -- launching one instantiation of the GEMV kernel.
#pragma once

#include <atomic>

#include "bsgemv_kernel.cuh"

namespace bsg {

template <int FMT, bool BF16, int MT, bool ZP, int BMODE>
int launch_one(const KParams& p, int ctas, int smem, cudaStream_t s) {
  auto k = bsgemv_mma_kernel<FMT, BF16, MT, ZP, BMODE>;
  static std::atomic<int> attr_smem{0};  // largest dynamic smem already granted to `k`
  if (smem > attr_smem.load()) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return BSGEMV_ERR_CUDA;
    attr_smem.store(smem);
  }
  // Programmatic dependent launch: the kernel may start while the previous kernel in the stream
  // drains; it waits (griddepcontrol.wait) before touching anything that kernel could write.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k, p) != cudaSuccess) return BSGEMV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

// Dispatch over the n8 tile count, zero points and block mode for one format / activation type.
template <int FMT, bool BF16>
int launch_fmt(const KParams& p, int mt, bool zp, int bmode, int ctas, int smem, cudaStream_t s) {
#define BSG_L(MTV, ZPV, BM) return launch_one<FMT, BF16, MTV, ZPV, BM>(p, ctas, smem, s)
#define BSG_ZP(MTV, BM) \
  if (zp) BSG_L(MTV, true, BM); \
  BSG_L(MTV, false, BM)
  if constexpr (FMT == kInt4) {
    if (mt == 1) {
      if (bmode == kBlockPerChunk) { BSG_ZP(1, kBlockPerChunk); }
      if (bmode == kBlockPerPair) { BSG_ZP(1, kBlockPerPair); }
      BSG_ZP(1, kTwoPerChunk);
    }
    if (bmode == kBlockPerChunk) { BSG_ZP(2, kBlockPerChunk); }
    if (bmode == kBlockPerPair) { BSG_ZP(2, kBlockPerPair); }
    BSG_ZP(2, kTwoPerChunk);
  } else if constexpr (FMT == kInt8) {
    if (mt == 1) {
      if (bmode == kBlockPerChunk) { BSG_ZP(1, kBlockPerChunk); }
      BSG_ZP(1, kBlockPerPair);
    }
    if (bmode == kBlockPerChunk) { BSG_ZP(2, kBlockPerChunk); }
    BSG_ZP(2, kBlockPerPair);
  } else if constexpr (FMT == kFp8) {
    if (mt == 1) BSG_L(1, false, kBlockPerPair);
    BSG_L(2, false, kBlockPerPair);
  } else {
    if (mt == 1) BSG_L(1, false, kBlockPerChunk);
    BSG_L(2, false, kBlockPerChunk);
  }
#undef BSG_ZP
#undef BSG_L
}

}  // namespace bsg
