// Instantiations of the GEMV kernel for int4 weights with fp16 activations, calls with up to 16
// rows (one or two n8 tiles; see bsgemv_launch.cuh).  Wider calls: bsgemv_int4_f16_wide.cu.
#include "bsgemv_launch.cuh"

namespace bsg {

int launch_int4_f16(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
  switch (mt) {
    case 1: return launch_fmt_mt<kInt4, false, 1>(p, zp, cpb, ctas, smem, s);
    case 2: return launch_fmt_mt<kInt4, false, 2>(p, zp, cpb, ctas, smem, s);
    default: return launch_int4_f16_wide(p, mt, zp, cpb, ctas, smem, s);
  }
}

}  // namespace bsg
