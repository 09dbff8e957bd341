// Instantiations of the GEMV kernel for int4 weights with fp16 activations, 128-row
// tiles (two 64-row halves), calls with up to 16 rows (see bsgemv_launch.cuh).
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_int4_f16_tall(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                         cudaStream_t s) {
  if (mt == 1) return launch_fmt_mt<kInt4, false, 1, 2>(p, zp, cpb, ctas, smem, s);
  return launch_fmt_mt<kInt4, false, 2, 2>(p, zp, cpb, ctas, smem, s);
}

}  // namespace bsg
