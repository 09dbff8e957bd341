// bsgemv_internal.h -- host/device shared definitions of the block-scaled GEMV library.
//
// Work decomposition (one persistent kernel per call):
//   * a CTA tile is kRowsPerTile consecutive output columns n (rows of W) over a k-range;
//   * k is walked in "stages" of 128 weight bytes per row (one 128-byte-swizzled TMA box, plus
//     the stage's activations, scales and zero points copied with cp.async):
//     256 k for the 4-bit formats, 128 k for the 8-bit formats;
//   * the tiles x stages grid is cut into `ctas` equal contiguous ranges (stream-K); a tile whose
//     stages fall into several CTAs is finished by the last CTA to arrive, which adds the
//     partial sums in CTA order (a fixed order, so results are deterministic).
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

#include "bsgemv.h"

namespace bsg {

enum Fmt : int { kInt4 = 1, kInt8 = 2, kFp8 = 3, kNvfp4 = 4 };

constexpr int kRowsPerTile = 64;      // output columns per CTA tile (4 mma row groups of 16)
constexpr int kConsumerWarps = 8;     // decode + mma warps; warp 0 issues the copies
constexpr int kRgPerWarp = 2;         // 16-row mma groups per consumer warp (2 of the tile's 4)
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kChunksPerStage = 8;    // 16-byte chunks of a weight row per stage (128 B)
constexpr int kStageRowBytes = 16 * kChunksPerStage;
constexpr int kMaxStages = 12;

// Error word bits written by kernels that abandon a bounded wait.
constexpr unsigned kErrTimeoutFull = 1u;
constexpr unsigned kErrTimeoutEmpty = 2u;

// Kernel parameters (passed by value as a __grid_constant__; the tensor maps must be 64-byte
// aligned in parameter space).
struct KParams {
  CUtensorMap tm_w;   // W  as uint8 [N][row_bytes], box [kRowsPerTile][128], 128B swizzle
  const uint16_t* A;       // activations [M][K] (fp16 / bf16 bits)
  const uint8_t* W;
  const uint8_t* scales;   // global copy, used when the scale tensor cannot be TMA-tiled
  const uint8_t* zp;       // idem for zero points
  const float* gscale;     // NVFP4 global scale
  void* y;
  float* partials;         // [ctas][2][slot_floats] cross-CTA partial sums
  unsigned* counters;      // [tiles] arrival counters, left at zero by every call
  unsigned* err;           // error word
  int64_t N, K;
  int64_t total_stages;    // tiles * spt
  int64_t spt;             // stages per tile
  int M;
  int nb_s;                // scale elements per row (K/bs, or K/16 for nvfp4)
  int bs_log2;
  int scale_pitch;         // bytes per scale row (global)
  int zp_pitch;            // bytes per zero-point row (global)
  int stages;              // ring depth
  int slot_bytes, act_off, sc_off, zp_off;  // offsets inside one ring slot
  int act_box_bytes;       // smem bytes per activation box (MPAD * 128)
  int ring_bytes, red_off, bar_off;
  int tx_bytes;            // bytes landing per stage
  int sbw;                 // scale box width in elements (blocks)
  int zbw_bytes;           // zero-point box width in bytes
  int zblk;                // blocks covered by one zero-point box
  int side_scale_tma;      // 1: scales are staged into the ring; 0: read from global memory
  int side_zp_tma;         // idem for zero points
  int slot_floats;         // floats per partial slot
};

struct Geometry {
  bsgemv_geometry pub;
  int fmt, bf16, has_zp, block_size, max_M;
  int64_t N, K;
  int kpc;                 // k per 16-byte chunk
  int kc;                  // k per stage
  int nbox;                // activation boxes per stage
  int mpad;                // activation rows reserved per box (8 or 16)
  int mt_max;              // 1 or 2 n8 mma tiles
  int scale_es;            // bytes per scale element
  int nb_s;
  int sbw, zbw_bytes, zblk;
  int slot_bytes, act_off, sc_off, zp_off, act_box_bytes, red_bytes, ring_bytes, red_off,
      bar_off;
  int slot_floats;
};

// Validates the problem and fills the geometry for `sm_count` SMs.  Pure host code.
int compute_geometry(int format, int block_size, int has_zp, int64_t N, int64_t K, int max_M,
                     int sm_count, int ctas_override, int stages_override, Geometry* g);

// Kernel launchers (one translation unit per weight format; int4 split by activation type).
// bmode: 0 = one scale block per 16-byte chunk, 1 = a consumer warp's chunk pair in one block,
// 2 = two blocks per chunk (int4 with 16-element blocks).
int launch_int4_f16(const KParams& p, int mt, bool zp, int bmode, int ctas, int smem,
                    cudaStream_t s);
int launch_int4_bf16(const KParams& p, int mt, bool zp, int bmode, int ctas, int smem,
                     cudaStream_t s);
int launch_int8(const KParams& p, int mt, bool bf16, bool zp, int bmode, int ctas, int smem,
                cudaStream_t s);
int launch_fp8(const KParams& p, int mt, bool bf16, bool zp, int bmode, int ctas, int smem,
               cudaStream_t s);
int launch_nvfp4(const KParams& p, int mt, bool bf16, bool zp, int bmode, int ctas, int smem,
                 cudaStream_t s);

// Block mode of a problem (see above).
inline int block_mode(int fmt, int block_size) {
  if (fmt == kInt4) return block_size == 16 ? 2 : (block_size == 32 ? 0 : 1);
  if (fmt == kInt8) return block_size == 16 ? 0 : 1;
  if (fmt == kFp8) return 1;
  return 0;
}

int launch_debug_dequant(int fmt, bool bf16, bool has_zp, int bs, int64_t N, int64_t K,
                         const uint8_t* W, const uint8_t* scales, const uint8_t* zp,
                         const float* gscale, float* out, cudaStream_t s);

}  // namespace bsg
