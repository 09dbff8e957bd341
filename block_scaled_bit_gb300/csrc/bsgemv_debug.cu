// bsgemv_debug.cu -- test hook: the dequantised weight through the GEMV's own register decoders.
//
// One warp per (16-row group, 16-byte chunk).  Lane (g, t) reads the same 32-bit words the
// GEMV's ldmatrix hands it (bytes [4t, 4t+4) of the chunk of rows g and g+8), runs the same
// decoder, and scatters every 16-bit operand half back to its physical k with the same phys_k
// mapping, times the fp32 block scale (int, FP8) or the global scale (NVFP4, whose E4M3 block
// scale is already folded into the operand).
#include "bsgemv_kernel.cuh"

namespace bsg {

template <int FMT, bool BF16, bool ZP>
__global__ void __launch_bounds__(128) debug_dequant_kernel(const uint8_t* __restrict__ W,
                                                            const uint8_t* __restrict__ scales,
                                                            const uint8_t* __restrict__ zp,
                                                            const float* __restrict__ gscale,
                                                            int64_t N, int64_t K, int bs_log2,
                                                            float* __restrict__ out) {
  constexpr bool kFour = (FMT == kInt4 || FMT == kNvfp4);
  constexpr int kKpc = kFour ? 32 : 16;
  constexpr int kSteps = kKpc / 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int64_t nchunks = K / kKpc;
  const int64_t c = int64_t(blockIdx.y) * 4 + warp;
  if (c >= nchunks) return;
  const int64_t row_bytes = kFour ? K / 2 : K;
  const int64_t n_lo = int64_t(blockIdx.x) * 16 + g, n_hi = n_lo + 8;
  const int64_t nb = K >> bs_log2;
  const int64_t k_lane = c * kKpc + (kFour ? 8 * t : 4 * t);  // first k of the lane's word
  const int64_t blk = k_lane >> bs_log2;

  auto word = [&](int64_t n) -> uint32_t {
    return n < N ? *reinterpret_cast<const uint32_t*>(W + n * row_bytes + c * 16 + 4 * t) : 0u;
  };
  const uint32_t lo = word(n_lo), hi = word(n_hi);
  const int64_t rlo = n_lo < N ? n_lo : N - 1, rhi = n_hi < N ? n_hi : N - 1;

  uint32_t a[kSteps][4];
  float s_lo = 1.f, s_hi = 1.f;
  if constexpr (FMT == kInt4 || FMT == kInt8) {
    uint32_t zv_lo = (FMT == kInt4) ? 8u : 128u, zv_hi = zv_lo;
    if constexpr (ZP) {
      if constexpr (FMT == kInt4) {
        const int64_t zrow = (nb + 1) / 2;
        const uint32_t b_lo = zp[rlo * zrow + (blk >> 1)], b_hi = zp[rhi * zrow + (blk >> 1)];
        zv_lo = (blk & 1) ? (b_lo >> 4) : (b_lo & 0xFu);
        zv_hi = (blk & 1) ? (b_hi >> 4) : (b_hi & 0xFu);
      } else {
        zv_lo = zp[rlo * nb + blk];
        zv_hi = zp[rhi * nb + blk];
      }
    }
    uint32_t zl_lo, zh_lo, zl_hi, zh_hi;
    zp_consts<FMT, BF16>(zv_lo, zl_lo, zh_lo);
    zp_consts<FMT, BF16>(zv_hi, zl_hi, zh_hi);
    if constexpr (FMT == kInt4) {
      decode_int4<BF16>(lo, hi, zl_lo, zh_lo, zl_hi, zh_hi, a);
    } else {
      decode_int8<BF16>(lo, hi, zl_lo, zl_hi, a);
    }
    const __half* s = reinterpret_cast<const __half*>(scales);
    s_lo = __half2float(s[rlo * nb + blk]);
    s_hi = __half2float(s[rhi * nb + blk]);
  } else if constexpr (FMT == kFp8) {
    decode_fp8<BF16>(lo, hi, a);
    const float* s = reinterpret_cast<const float*>(scales);
    s_lo = s[rlo * nb + blk];
    s_hi = s[rhi * nb + blk];
  } else {
    const uint32_t f_lo = e4m3x2_to_f16x2(uint32_t(scales[rlo * nb + blk]) * 0x0101u);
    const uint32_t f_hi = e4m3x2_to_f16x2(uint32_t(scales[rhi * nb + blk]) * 0x0101u);
    decode_nvfp4<BF16>(lo, hi, f_lo, f_hi, a);
    s_lo = s_hi = *gscale;
  }

#pragma unroll
  for (int st = 0; st < kSteps; ++st) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const bool upper = (r & 1) != 0;
      const int64_t n = upper ? n_hi : n_lo;
      if (n >= N) continue;
      const int rp = r >> 1;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint16_t bits = static_cast<uint16_t>(a[st][r] >> (16 * h));
        float v;
        if constexpr (BF16) v = __bfloat162float(__ushort_as_bfloat16(bits));
        else v = __half2float(__ushort_as_half(bits));
        const int64_t k = c * kKpc + phys_k<FMT>(st, rp, h, t);
        out[n * K + k] = v * (upper ? s_hi : s_lo);
      }
    }
  }
}

template <int FMT, bool BF16, bool ZP>
static int go(int bs, int64_t N, int64_t K, const uint8_t* W, const uint8_t* scales,
              const uint8_t* zp, const float* gscale, float* out, cudaStream_t s) {
  constexpr int kKpc = (FMT == kInt4 || FMT == kNvfp4) ? 32 : 16;
  const int64_t nchunks = K / kKpc;
  const dim3 grid(static_cast<unsigned>((N + 15) / 16), static_cast<unsigned>((nchunks + 3) / 4));
  int bs_log2 = 0;
  while ((1 << bs_log2) < bs) ++bs_log2;
  debug_dequant_kernel<FMT, BF16, ZP><<<grid, 128, 0, s>>>(W, scales, zp, gscale, N, K, bs_log2, out);
  return cudaGetLastError() == cudaSuccess ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

int launch_debug_dequant(int fmt, bool bf16, bool has_zp, int bs, int64_t N, int64_t K,
                         const uint8_t* W, const uint8_t* scales, const uint8_t* zp,
                         const float* gscale, float* out, cudaStream_t s) {
#define BSG_DBG(F, B, Z) return go<F, B, Z>(bs, N, K, W, scales, zp, gscale, out, s)
  switch (fmt) {
    case kInt4:
      if (bf16) { if (has_zp) BSG_DBG(kInt4, true, true); BSG_DBG(kInt4, true, false); }
      if (has_zp) BSG_DBG(kInt4, false, true);
      BSG_DBG(kInt4, false, false);
    case kInt8:
      if (bf16) { if (has_zp) BSG_DBG(kInt8, true, true); BSG_DBG(kInt8, true, false); }
      if (has_zp) BSG_DBG(kInt8, false, true);
      BSG_DBG(kInt8, false, false);
    case kFp8:
      if (bf16) BSG_DBG(kFp8, true, false);
      BSG_DBG(kFp8, false, false);
    case kNvfp4:
      if (bf16) BSG_DBG(kNvfp4, true, false);
      BSG_DBG(kNvfp4, false, false);
  }
#undef BSG_DBG
  return BSGEMV_ERR_INVALID_ARG;
}

}  // namespace bsg
