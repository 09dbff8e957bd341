// Instantiations of the GEMV kernel for nvfp4 weights (see bsgemv_launch.cuh).
#include "bsgemv_launch.cuh"

namespace bsg {

// Tiles: 1 (M <= 8), 2 (M <= 16), 3 (M <= 24), 4 (M <= 32).
template <bool BF16>
int launch_nvfp4_act(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
  switch (mt) {
    case 1: return launch_fmt_mt<kNvfp4, BF16, 1>(p, zp, cpb, ctas, smem, s);
    case 2: return launch_fmt_mt<kNvfp4, BF16, 2>(p, zp, cpb, ctas, smem, s);
    case 3: return launch_fmt_mt<kNvfp4, BF16, 3>(p, zp, cpb, ctas, smem, s);
    default: return launch_fmt_mt<kNvfp4, BF16, 4>(p, zp, cpb, ctas, smem, s);
  }
}

int launch_nvfp4(const KParams& p, int mt, bool bf16, bool zp, int cpb, int ctas, int smem, cudaStream_t s) {
  return bf16 ? launch_nvfp4_act<true>(p, mt, zp, cpb, ctas, smem, s)
              : launch_nvfp4_act<false>(p, mt, zp, cpb, ctas, smem, s);
}

}  // namespace bsg
