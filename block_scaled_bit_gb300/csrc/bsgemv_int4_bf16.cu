// Instantiations of the GEMV kernel for int4_bf16 weights (see bsgemv_launch.cuh).
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_int4_bf16(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
  return launch_fmt<kInt4, true>(p, mt, zp, cpb, ctas, smem, s);
}

}  // namespace bsg
