// bsgemv_launch.cuh -- launching one instantiation of the GEMV kernel.
#pragma once

#include <atomic>

#include "bsgemv_kernel.cuh"

namespace bsg {

// Launch kernel `k` (one instantiation; `rec` is its own record of the attributes already set,
// per device and context).
template <class Kernel>
int launch_kernel(Kernel k, AttrRecord& rec, const KParams& p, int ctas, int smem, cudaStream_t s) {
  int dev = -1;
  uint64_t ctx = 0;
  if (!current_device_context(&dev, &ctx)) return BSGEMV_ERR_CUDA;
  const int d = rec.slot(dev, ctx);
  if (smem > rec.smem[d].load()) {
    // One shared-memory carveout (the largest) for every instantiation: an SM holds CTAs of
    // kernels with different carveouts only after draining, which would serialise consecutive
    // calls that programmatic dependent launch otherwise overlaps.
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared) != cudaSuccess)
      return BSGEMV_ERR_CUDA;
    rec.smem[d].store(smem);
  }
  if (p.cluster > 8 && rec.cluster[d].load() == 0) {
    if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return BSGEMV_ERR_CUDA;
    rec.cluster[d].store(1);
  }
  // Programmatic dependent launch: the kernel may start while the previous kernel in the stream
  // drains; it waits (griddepcontrol.wait) before touching anything that kernel could write.
  // Cluster split: the CTAs of a tile form one cluster (consecutive in x).
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int nattr = 1;
  if (p.cluster >= 2) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    nattr = 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  if (cudaLaunchKernelEx(&cfg, k, p) != cudaSuccess) return BSGEMV_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

template <int FMT, bool BF16, int MT, bool ZP, int CPB, int H>
int launch_one(const KParams& p, int ctas, int smem, cudaStream_t s) {
  // one kernel per source of the scales: the side ring, or global memory (unaligned pitches)
  static AttrRecord rec_side, rec_global;
  if (p.side_tma)
    return launch_kernel(bsgemv_mma_kernel<FMT, BF16, MT, ZP, CPB, H, true>, rec_side, p, ctas,
                         smem, s);
  return launch_kernel(bsgemv_mma_kernel<FMT, BF16, MT, ZP, CPB, H, false>, rec_global, p, ctas,
                       smem, s);
}

template <int FMT, bool BF16, bool ZP, int CPB, int COLS>
int launch_one_cc(const KParams& p, int ctas, int smem, cudaStream_t s) {
  static AttrRecord rec_side, rec_global;
  if (p.side_tma)
    return launch_kernel(bsgemv_fma_kernel<FMT, BF16, ZP, CPB, COLS, true>, rec_side, p, ctas,
                         smem, s);
  return launch_kernel(bsgemv_fma_kernel<FMT, BF16, ZP, CPB, COLS, false>, rec_global, p, ctas,
                       smem, s);
}

// CUDA-core variant (M <= 8): dispatch over zero points and chunks per scale block; COLS = 1
// for calls with M = 1, else 8 (the same arithmetic per activation row).
template <int FMT, bool BF16, int COLS>
int launch_fmt_cc_cols(const KParams& p, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
#define BSG_C(ZPV, C) return launch_one_cc<FMT, BF16, ZPV, C, COLS>(p, ctas, smem, s)
#define BSG_CZ(C) \
  if (zp) BSG_C(true, C); \
  BSG_C(false, C)
  if constexpr (FMT == kInt4) {
    switch (cpb) {
      case 0: BSG_CZ(0);
      case 1: BSG_CZ(1);
      case 2: BSG_CZ(2);
      case 4: BSG_CZ(4);
      default: BSG_CZ(8);
    }
  } else if constexpr (FMT == kInt8) {
    switch (cpb) {
      case 1: BSG_CZ(1);
      case 2: BSG_CZ(2);
      case 4: BSG_CZ(4);
      default: BSG_CZ(8);
    }
  } else if constexpr (FMT == kFp8) {
    BSG_C(false, 8);
  } else {
    BSG_C(false, 1);
  }
#undef BSG_CZ
#undef BSG_C
}

template <int FMT, bool BF16>
int launch_fmt_cc(const KParams& p, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
  if (p.M == 1) return launch_fmt_cc_cols<FMT, BF16, 1>(p, zp, cpb, ctas, smem, s);
  return launch_fmt_cc_cols<FMT, BF16, 8>(p, zp, cpb, ctas, smem, s);
}

// Dispatch over zero points and chunks per scale block (block_mode) for one format, activation
// type, n8 tile count MT (1 .. 4) and H halves per tile.
template <int FMT, bool BF16, int MT, int H = 1>
int launch_fmt_mt(const KParams& p, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
#define BSG_L(ZPV, C) return launch_one<FMT, BF16, MT, ZPV, C, H>(p, ctas, smem, s)
#define BSG_ZP(C) \
  if (zp) BSG_L(true, C); \
  BSG_L(false, C)
  if constexpr (FMT == kInt4) {
    switch (cpb) {
      case 0: BSG_ZP(0);
      case 1: BSG_ZP(1);
      case 2: BSG_ZP(2);
      case 4: BSG_ZP(4);
      default: BSG_ZP(8);
    }
  } else if constexpr (FMT == kInt8) {  // 8-bit chunks hold 16 k: no block is smaller
    switch (cpb) {
      case 1: BSG_ZP(1);
      case 2: BSG_ZP(2);
      case 4: BSG_ZP(4);
      default: BSG_ZP(8);
    }
  } else if constexpr (FMT == kFp8) {  // one 128-k block per stage
    BSG_L(false, 8);
  } else {  // NVFP4 folds its scales
    BSG_L(false, 1);
  }
#undef BSG_ZP
#undef BSG_L
}

}  // namespace bsg
