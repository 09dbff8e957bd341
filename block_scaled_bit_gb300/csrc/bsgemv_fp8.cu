// Instantiations of the GEMV kernel for fp8 weights, 64-row tiles (see bsgemv_launch.cuh).
// 128-row tiles: bsgemv_fp8_tall.cu.
#include "bsgemv_launch.cuh"

namespace bsg {

// Tiles: 1 (M <= 8), 2 (M <= 16), 3 (M <= 24), 4 (M <= 32).
template <bool BF16>
int launch_fp8_act(const KParams& p, int mt, int ctas, int smem, cudaStream_t s) {
  switch (mt) {
    case 1: return launch_fmt_mt<kFp8, BF16, 1>(p, false, 0, ctas, smem, s);
    case 2: return launch_fmt_mt<kFp8, BF16, 2>(p, false, 0, ctas, smem, s);
    case 3: return launch_fmt_mt<kFp8, BF16, 3>(p, false, 0, ctas, smem, s);
    default: return launch_fmt_mt<kFp8, BF16, 4>(p, false, 0, ctas, smem, s);
  }
}

int launch_fp8(const KParams& p, int mt, int halves, bool bf16, int ctas, int smem,
               cudaStream_t s) {
  // (128-row tiles exist for calls of up to 16 rows only: plans for more rows never take them)
  if (halves == 2) return mt <= 2 ? launch_fp8_tall(p, mt, bf16, ctas, smem, s)
                                : BSGEMV_ERR_UNSUPPORTED;
  return bf16 ? launch_fp8_act<true>(p, mt, ctas, smem, s)
              : launch_fp8_act<false>(p, mt, ctas, smem, s);
}

}  // namespace bsg
