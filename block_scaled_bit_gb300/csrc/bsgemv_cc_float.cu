// Instantiations of the CUDA-core variant of the GEMV kernel for FP8 E4M3 and NVFP4 weights (see
// bsgemv_launch.cuh).
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_cc_fp8(const KParams& p, bool bf16, int ctas, int smem, cudaStream_t s) {
  return bf16 ? launch_fmt_cc<kFp8, true>(p, false, 8, ctas, smem, s)
              : launch_fmt_cc<kFp8, false>(p, false, 8, ctas, smem, s);
}

int launch_cc_nvfp4(const KParams& p, bool bf16, int ctas, int smem, cudaStream_t s) {
  return bf16 ? launch_fmt_cc<kNvfp4, true>(p, false, 1, ctas, smem, s)
              : launch_fmt_cc<kNvfp4, false>(p, false, 1, ctas, smem, s);
}

}  // namespace bsg
