// Instantiations of the GEMV kernel for int8 weights with bf16 activations, calls with 17 to 32
// rows (three or four n8 tiles; see bsgemv_launch.cuh).
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_int8_bf16_wide(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                          cudaStream_t s) {
  if (mt == 3) return launch_fmt_mt<kInt8, true, 3>(p, zp, cpb, ctas, smem, s);
  return launch_fmt_mt<kInt8, true, 4>(p, zp, cpb, ctas, smem, s);
}

}  // namespace bsg
