// Instantiations of the GEMV kernel for fp8 weights (see bsgemv_launch.cuh).
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_fp8(const KParams& p, int mt, bool bf16, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
  return bf16 ? launch_fmt<kFp8, true>(p, mt, zp, cpb, ctas, smem, s)
              : launch_fmt<kFp8, false>(p, mt, zp, cpb, ctas, smem, s);
}

}  // namespace bsg
