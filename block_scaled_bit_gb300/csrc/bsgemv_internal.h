// bsgemv_internal.h -- host/device shared definitions of the block-scaled GEMV library.
//
// Work decomposition (one persistent kernel per call):
//   * a CTA tile is 64 or 128 consecutive output columns n (rows of W) over a k-range: one or
//     two "halves" of kBoxRows = 64 rows.  Consumer warp w owns mma row group w (16 rows) of
//     every half, so with two halves every activation fragment it loads and every stage's
//     bookkeeping serve 32 rows.  Plans for up to 16 rows whose 128-row tiles would each be
//     shared by few resident CTAs take two halves; plans whose tiles are shared by many CTAs keep
//     one (a finer split of the work; see compute_geometry);
//   * k is walked in "stages" of 256 k for the 4-bit formats (128 weight bytes per row), of 256 k
//     (two k-boxes) for the 8-bit formats with one half and 128 k with two: one 128-byte-swizzled
//     TMA box [64 rows][128 B] per half and k-box (8 KB of weight per stage for the 4-bit formats
//     with one half, else 16 KB), plus the stage's activations (cp.async) -- scales and zero
//     points arrive per several stages on a side ring;
//   * the tiles x stages grid is cut into `ctas` equal contiguous ranges (stream-K), and a tile
//     whose stages fall into several CTAs is finished by the last CTA to arrive, which adds the
//     partial sums in CTA order; or, for shapes with few tiles, each tile's stages are split
//     evenly over the CTAs of one thread-block cluster and added in rank order in the leader's
//     shared memory.  Either way the order is fixed, so results are deterministic.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <stdint.h>

#include <atomic>

#include "bsgemv.h"

namespace bsg {

enum Fmt : int { kInt4 = 1, kInt8 = 2, kFp8 = 3, kNvfp4 = 4 };

constexpr int kBoxRows = 64;          // rows of one weight TMA box (one half of a tile)
constexpr int kMaxHalves = 2;         // halves per tile: 1 (64 rows) or 2 (128 rows)
constexpr int kMaxRowsPerTile = kMaxHalves * kBoxRows;
constexpr int kConsumerWarps = 4;     // decode + mma warps (row group w of every half); warp 0
                                      // copies
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxM = 32;             // activation rows per call: up to four n8 mma tiles
// CTAs per SM the kernels are built for (their register and shared-memory budget).  One half:
// 4 with one n8 activation tile (M <= 8), 3 with two or three (M <= 24; 128 registers, no
// spills), 2 with four (M <= 32).  Two halves (M <= 16 only): 3 -- twice the accumulators, and a
// CTA's two 16 KB stages, activations and side ring fill a third of the SM's shared memory.
constexpr int ctas_per_sm_for(int mt, int halves) {
  return halves == 2 ? 3 : (mt == 1 ? 4 : mt <= 3 ? 3 : 2);
}
// n8 activation tiles of the kernel a plan is sized for (and of the kernel a call with M rows
// runs).
constexpr int mt_for_m(int m) { return m <= 8 ? 1 : m <= 16 ? 2 : m <= 24 ? 3 : 4; }
constexpr int kBoxRowBytes = 128;     // bytes per row of one weight TMA box (128-byte swizzle)
// Weight boxes along k per stage: two for the 8-bit formats with one half (so that a stage is
// 16 KB of weight, 256 k, as for every other case), else one.
constexpr int stage_kboxes(int fmt, int halves) {
  return (fmt == kInt4 || fmt == kNvfp4 || halves == 2) ? 1 : 2;
}
// k per stage: 128 weight bytes per row and k-box, i.e. 256 k of the 4-bit formats, 128 k of the
// 8-bit ones per k-box.
constexpr int stage_k(int fmt, int halves) {
  return stage_kboxes(fmt, halves) * ((fmt == kInt4 || fmt == kNvfp4) ? 256 : 128);
}
constexpr int kMaxStages = 12;

// Error word bits written by kernels that abandon a bounded wait.
constexpr unsigned kErrTimeoutFull = 1u;
constexpr unsigned kErrTimeoutEmpty = 2u;
constexpr uint64_t kDefaultWaitNs = 4000000000ull;  // 4 s: far above any legitimate stall

// Kernel parameters (passed by value as a __grid_constant__; the tensor maps must be 64-byte
// aligned in parameter space).
struct KParams {
  CUtensorMap tm_w;   // W as uint8 [N][row_bytes], box [kBoxRows][128], 128B swizzle
  CUtensorMap tm_s;   // scales as uint8 [N][scale_pitch], box [tile rows][kSideScaleBytes]
  CUtensorMap tm_z;   // zero points as uint8 [N][zp_pitch], box [tile rows][zbox_bytes]
  const uint16_t* A;       // activations [M][K] (fp16 / bf16 bits)
  const uint8_t* W;
  const uint8_t* scales;   // global copy, read directly when side_tma == 0
  const uint8_t* zp;       // idem for zero points
  const float* gscale;     // NVFP4 global scale
  const uint16_t* bias;    // [N] bias in the activation dtype added before the rounding, or null
  void* y;
  float* partials;         // [ctas][2][kConsumerWarps][slot_floats] cross-CTA partial sums
                           // (a slot: every half's fragments of one warp)
  unsigned* counters;      // [tiles][kConsumerWarps] arrival counters, left at zero by every call
  unsigned* err;           // error word
  int64_t N, K;
  int64_t total_stages;    // tiles * spt
  uint64_t wait_ns;        // limit of every bounded wait (kWaitLimitNs unless a test lowers it)
  int spt;                 // stages per tile
  int M;
  int nb_s;                // scale elements per row (K/bs, or K/16 for nvfp4)
  int bs_log2;
  int scale_pitch;         // bytes per scale row (global)
  int zp_pitch;            // bytes per zero-point row (global)
  int stages;              // weight / activation ring depth
  int act_off;             // activation ring: stages x act_bytes
  int act_bytes;           // activation bytes per stage (max_M padded rows)
  int side_tma;            // 1: scales / zero points staged by TMA into the side ring
  int side_off;            // side ring: side_slots x side_bytes
  int side_bytes;          // one side box: scales [64][kSideScaleBytes], zero points after
  int side_slots;
  int side_tx;             // bytes one side box lands (scales + zero points)
  int zbox_bytes;          // zero-point box width in bytes
  int rs_log2;             // log2(stages per side box)
  int bar_off;
  int slot_floats;         // floats per partial slot (one warp's fragments)
  int cluster;             // 0: stream-K; C >= 1: C CTAs per tile in one cluster
  int red_off;             // cluster split: [C][kConsumerWarps][MT][8 * red_tq] float4 in the
  int red_tq;              //   leader; quad lanes t < red_tq hold output columns < max_M
  int skip_stage;          // test hook: CTA 0's producer leaves out this stage of its range
                           // (its consumers' wait then runs out); -1 = none
};

struct Geometry {
  bsgemv_geometry pub;
  int fmt, bf16, has_zp, block_size, max_M;
  int64_t N, K;
  int kpc;                 // k per 16-byte chunk
  int kc;                  // k per stage (stage_k)
  int stage_bytes;         // weight bytes per stage
  int mt_max;              // n8 mma tiles of the kernel sized for max_M (1 .. 4)
  int halves;              // 64-row halves per tile (1 or 2): pub.rows_per_tile / kBoxRows
  int scale_es;            // bytes per scale element
  int nb_s;
  int scale_pitch, zp_pitch;
  int act_bytes, act_off;
  int rs_log2, side_slots, side_bytes, zbox_bytes, side_off;
  int bar_off;
  int slot_floats;
  int red_off, red_bytes;  // cluster split: the leader's reduction buffer
  int red_tq;              // cluster split: quad lanes t < red_tq hold output columns < max_M
};

// Weight bytes of one stage (one [64 rows][128 B] box per half and k-box: 8 or 16 KB), and scale
// bytes per row of one side box.
inline int stage_bytes(int fmt, int halves) {
  return halves * stage_kboxes(fmt, halves) * kBoxRows * kBoxRowBytes;
}
constexpr int kSideScaleBytes = 64;

// Validates the problem and fills the geometry for `sm_count` SMs.  Pure host code.
// split = enum bsgemv_split, cluster = CTAs per tile for BSGEMV_SPLIT_CLUSTER (0 = chosen).
// rows (1 .. max_M, 0 = max_M): the layout of the shared-memory ring for a call with that many
// activation rows; the split, CTA count and residency are those of max_M whatever `rows` is.
// tile_rows: 64 or 128 output columns per tile, 0 = chosen (128 only for max_M <= 16).
int compute_geometry(int format, int block_size, int has_zp, int64_t N, int64_t K, int max_M,
                     int sm_count, int ctas_override, int stages_override, int split, int cluster,
                     Geometry* g, int rows = 0, int tile_rows = 0);

constexpr int kMaxCluster = 16;     // CTAs per cluster (above 8: non-portable cluster size)
constexpr int kMaxAutoCluster = 8;  // largest cluster the automatic split picks

// Kernel launchers (one translation unit per weight format; int4 and int8 split by activation
// type; "wide": calls of 17 to 32 rows; "tall": 128-row tiles, calls of up to 16 rows).
// cpb: see block_mode.  halves: the plan's 64-row halves per tile.
int launch_int4_f16(const KParams& p, int mt, int halves, bool zp, int cpb, int ctas, int smem,
                    cudaStream_t s);
int launch_int4_bf16(const KParams& p, int mt, int halves, bool zp, int cpb, int ctas, int smem,
                     cudaStream_t s);
int launch_int8_f16(const KParams& p, int mt, int halves, bool zp, int cpb, int ctas, int smem,
                    cudaStream_t s);
int launch_int8_bf16(const KParams& p, int mt, int halves, bool zp, int cpb, int ctas, int smem,
                     cudaStream_t s);
int launch_fp8(const KParams& p, int mt, int halves, bool bf16, int ctas, int smem,
               cudaStream_t s);
int launch_nvfp4(const KParams& p, int mt, int halves, bool bf16, int ctas, int smem,
                 cudaStream_t s);
int launch_int4_f16_wide(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                         cudaStream_t s);
int launch_int4_bf16_wide(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                          cudaStream_t s);
int launch_int8_f16_wide(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                         cudaStream_t s);
int launch_int8_bf16_wide(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                          cudaStream_t s);
int launch_int4_f16_tall(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                         cudaStream_t s);
int launch_int4_bf16_tall(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                          cudaStream_t s);
int launch_int8_f16_tall(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                         cudaStream_t s);
int launch_int8_bf16_tall(const KParams& p, int mt, bool zp, int cpb, int ctas, int smem,
                          cudaStream_t s);
int launch_fp8_tall(const KParams& p, int mt, bool bf16, int ctas, int smem, cudaStream_t s);
int launch_nvfp4_tall(const KParams& p, int mt, bool bf16, int ctas, int smem, cudaStream_t s);
// The CUDA-core variant (BSGEMV_VARIANT_CUDA_CORE; M <= 8).
int launch_cc_int4_f16(const KParams& p, bool zp, int cpb, int ctas, int smem, cudaStream_t s);
int launch_cc_int4_bf16(const KParams& p, bool zp, int cpb, int ctas, int smem, cudaStream_t s);
int launch_cc_int8_f16(const KParams& p, bool zp, int cpb, int ctas, int smem, cudaStream_t s);
int launch_cc_int8_bf16(const KParams& p, bool zp, int cpb, int ctas, int smem, cudaStream_t s);
int launch_cc_fp8(const KParams& p, bool bf16, int ctas, int smem, cudaStream_t s);
int launch_cc_nvfp4(const KParams& p, bool bf16, int ctas, int smem, cudaStream_t s);

// Chunks (16 bytes of a weight row) per scale block, the kernel's CPB: 0 when a chunk holds two
// blocks, else bs / k-per-chunk capped at 8 (a block spanning a whole stage or more).  NVFP4
// folds its scales and uses 1.
inline int block_mode(int fmt, int block_size) {
  if (fmt == kNvfp4) return 1;
  const int k_per_chunk = (fmt == kInt4) ? 32 : 16;
  if (block_size < k_per_chunk) return 0;
  const int c = block_size / k_per_chunk;
  return c >= 8 ? 8 : c;
}

// TMA tensor maps of one call's operands.  side_tma: the scales (and zero points) could be
// tiled (16-byte aligned base and pitch), so the kernel stages them through its side ring.
struct OperandMaps {
  CUtensorMap tm_w, tm_s, tm_z;
  bool side_tma;
};

// Host helpers shared by the entry points (bsgemv_host.cpp).
int encode_maps(const Geometry& g, const void* W, const void* scales, const void* zp,
                OperandMaps* m);
void fill_params(const Geometry& g, const OperandMaps& m, const void* A, const void* W,
                 const void* scales, const void* zp, void* y, int M, float* partials,
                 unsigned* counters, unsigned* err, KParams* k);
int launch_gemv(const Geometry& g, const KParams& k, cudaStream_t s);

// The current device and the id of its current context (unique for the life of the process,
// never reused, unlike a context's handle); false if either cannot be read.  Function
// attributes (dynamic shared-memory size, carveout, non-portable cluster sizes) and symbol
// addresses belong to a context, so every record of them is keyed by both.
bool current_device_context(int* dev, uint64_t* ctx_id);
constexpr int kMaxDevices = 64;

// The launch attributes already set for one kernel, per device: a record made under another
// context (another device's, or one destroyed by a device reset) counts as nothing set.
struct AttrRecord {
  std::atomic<uint64_t> ctx[kMaxDevices];
  std::atomic<int> smem[kMaxDevices];     // largest dynamic shared memory granted
  std::atomic<int> cluster[kMaxDevices];  // non-portable cluster sizes allowed
  // Slot of device `dev` under context `ctx`, cleared when the context changed.
  int slot(int dev, uint64_t ctx_id) {
    if (ctx[dev].load() != ctx_id) {
      smem[dev].store(0);
      cluster[dev].store(0);
      ctx[dev].store(ctx_id);
    }
    return dev;
  }
};

// The error word of bsgemv_run_noalloc's scratch area on the current device.
int noalloc_error_word(unsigned** out);

// Copy `bytes` from src to dst with a kernel on stream s (programmatic dependent launch: it waits
// for the previous kernel in the stream before touching either buffer).  Both 16-byte aligned
// (else BSGEMV_ERR_MISALIGNED); either may be pinned host memory seen through its device mapping.
int launch_host_copy(void* dst, const void* src, size_t bytes, int sm_count, cudaStream_t s);

int launch_debug_dequant(int fmt, bool bf16, bool has_zp, int bs, int64_t N, int64_t K,
                         const uint8_t* W, const uint8_t* scales, const uint8_t* zp,
                         const float* gscale, float* out, cudaStream_t s);

}  // namespace bsg
