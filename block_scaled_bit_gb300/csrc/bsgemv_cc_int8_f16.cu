// Instantiations of the CUDA-core variant of the GEMV kernel for int8 weights with fp16
// activations (see bsgemv_launch.cuh).
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_cc_int8_f16(const KParams& p, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
  return launch_fmt_cc<kInt8, false>(p, zp, cpb, ctas, smem, s);
}

}  // namespace bsg
