// Instantiations of the GEMV kernel for int4 weights with bf16 activations, 64-row
// tiles, calls with up to 16 rows (one or two n8 tiles; see bsgemv_launch.cuh).  128-row tiles:
// bsgemv_int4_bf16_tall.cu; calls of 17 to 32 rows: bsgemv_int4_bf16_wide.cu.
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_int4_bf16(const KParams& p, int mt, int halves, bool zp, int cpb, int ctas, int smem,
                     cudaStream_t s) {
  // (128-row tiles exist for calls of up to 16 rows only: plans for more rows never take them)
  if (halves == 2) return mt <= 2 ? launch_int4_bf16_tall(p, mt, zp, cpb, ctas, smem, s)
                                : BSGEMV_ERR_UNSUPPORTED;
  if (mt > 2) return launch_int4_bf16_wide(p, mt, zp, cpb, ctas, smem, s);
  if (mt == 1) return launch_fmt_mt<kInt4, true, 1>(p, zp, cpb, ctas, smem, s);
  return launch_fmt_mt<kInt4, true, 2>(p, zp, cpb, ctas, smem, s);
}

}  // namespace bsg
