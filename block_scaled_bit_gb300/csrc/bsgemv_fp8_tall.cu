// Instantiations of the GEMV kernel for fp8 weights, 128-row tiles (two 64-row halves), calls
// with up to 16 rows (see bsgemv_launch.cuh).
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_fp8_tall(const KParams& p, int mt, bool bf16, int ctas, int smem, cudaStream_t s) {
  if (bf16)
    return mt == 1 ? launch_fmt_mt<kFp8, true, 1, 2>(p, false, 0, ctas, smem, s)
                   : launch_fmt_mt<kFp8, true, 2, 2>(p, false, 0, ctas, smem, s);
  return mt == 1 ? launch_fmt_mt<kFp8, false, 1, 2>(p, false, 0, ctas, smem, s)
                 : launch_fmt_mt<kFp8, false, 2, 2>(p, false, 0, ctas, smem, s);
}

}  // namespace bsg
