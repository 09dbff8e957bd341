// Instantiations of the GEMV kernel for int8 weights with bf16 activations (see
// bsgemv_launch.cuh).
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_int8_bf16(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
  return launch_fmt<kInt8, true>(p, mt, zp, cpb, ctas, smem, s);
}

}  // namespace bsg
