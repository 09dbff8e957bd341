// bsgemv_geometry.cpp -- pure host code: argument validation and the launch geometry.
//
// Everything here depends only on the problem (format, block size, zero points, N, K, max_M)
// and the SM count, never on M of a call, so every M run through one plan takes the same
// per-row summation order (rows are bit-identical across M).
//
// Choices (the reasons are measurements on GB300; see the design notes):
//   * 64 output columns per CTA tile, 8 consumer warps + 1 copy warp, 2 CTAs per SM;
//   * a ring of up to 12 stages of 128 weight bytes per row, as deep as the shared-memory share
//     of a CTA allows (2 CTAs per SM), so that every SM keeps tens of KB of weight in flight;
//   * stream-K: the tiles x stages work is split into equal contiguous ranges over
//     min(total stages, 2 x SMs) persistent CTAs, which balances every shape to within one
//     stage per CTA without a wave tail.
#include <algorithm>
#include <cstdint>
#include <cstring>

#include "bsgemv_internal.h"

namespace bsg {

namespace {
constexpr int kSmemPerSm = 233472;       // 228 KB shared memory per SM on sm_100-class parts
constexpr int kSmemPerBlockMax = 232448; // 227 KB opt-in maximum per CTA
constexpr int kReservedPerBlock = 1024;  // reserved by the system per resident CTA
constexpr int kCtasPerSm = 2;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool is_pow2_block(int bs) {
  return bs == 16 || bs == 32 || bs == 64 || bs == 128 || bs == 256;
}
}  // namespace

int compute_geometry(int format, int block_size, int has_zp, int64_t N, int64_t K, int max_M,
                     int sm_count, int ctas_override, int stages_override, Geometry* g) {
  if (g == nullptr) return BSGEMV_ERR_INVALID_ARG;
  std::memset(g, 0, sizeof(*g));
  if ((format & ~(0xFF | BSGEMV_ACT_BF16)) != 0) return BSGEMV_ERR_INVALID_ARG;
  const int fmt = format & 0xFF;
  if (fmt < kInt4 || fmt > kNvfp4) return BSGEMV_ERR_INVALID_ARG;
  if (has_zp != 0 && has_zp != 1) return BSGEMV_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || max_M < 1 || max_M > 16 || sm_count < 1 || block_size < 1)
    return BSGEMV_ERR_INVALID_ARG;
  if (ctas_override < 0 || stages_override < 0 || stages_override > kMaxStages)
    return BSGEMV_ERR_INVALID_ARG;
  switch (fmt) {
    case kInt4:
    case kInt8:
      if (!is_pow2_block(block_size)) return BSGEMV_ERR_UNSUPPORTED;
      break;
    case kFp8:
      if (block_size != 128 || has_zp) return BSGEMV_ERR_UNSUPPORTED;
      break;
    case kNvfp4:
      if (block_size != 16 || has_zp) return BSGEMV_ERR_UNSUPPORTED;
      break;
  }
  if (K % 64 != 0 || K % block_size != 0) return BSGEMV_ERR_UNSUPPORTED;
  // TMA coordinates are signed 32-bit; y indices are 64-bit.
  if (N > (int64_t(1) << 31) - kRowsPerTile || K > (int64_t(1) << 30)) return BSGEMV_ERR_UNSUPPORTED;

  const bool four = (fmt == kInt4 || fmt == kNvfp4);
  g->fmt = fmt;
  g->bf16 = (format & BSGEMV_ACT_BF16) ? 1 : 0;
  g->has_zp = has_zp;
  g->block_size = block_size;
  g->max_M = max_M;
  g->N = N;
  g->K = K;
  g->kpc = four ? 32 : 16;
  g->kc = kChunksPerStage * g->kpc;
  g->nbox = g->kc / 64;
  g->mpad = max_M <= 8 ? 8 : 16;
  g->mt_max = g->mpad / 8;
  g->scale_es = (fmt == kFp8) ? 4 : (fmt == kNvfp4 ? 1 : 2);
  g->nb_s = static_cast<int>(K / block_size);
  const int bps = std::max(1, g->kc / block_size);  // scale blocks per stage
  g->sbw = std::max(16 / g->scale_es, bps);
  if (fmt == kInt4) {
    g->zbw_bytes = std::max(16, bps / 2);
    g->zblk = 2 * g->zbw_bytes;
  } else {
    g->zbw_bytes = std::max(16, bps);
    g->zblk = g->zbw_bytes;
  }

  // one ring slot: [W 64 x 128 B][activation boxes][scales][zero points]
  g->act_box_bytes = g->mpad * 128;
  g->act_off = kRowsPerTile * kStageRowBytes;
  g->sc_off = g->act_off + g->nbox * g->act_box_bytes;
  g->zp_off = g->sc_off + kRowsPerTile * g->sbw * g->scale_es;
  const int slot_end = g->zp_off + (has_zp ? kRowsPerTile * g->zbw_bytes : 0);
  g->slot_bytes = static_cast<int>(ceil_div(slot_end, 1024) * 1024);
  g->red_bytes = kConsumerWarps * kRgPerWarp * g->mt_max * 32 * 16;
  g->slot_floats = 4 * g->mt_max * 32 * 4;

  auto smem_for = [&](int stages) {
    return stages * g->slot_bytes + g->red_bytes + 16 * stages + 16 + 1024;
  };
  int ctas_per_sm = kCtasPerSm;
  const int budget = kSmemPerSm / ctas_per_sm - kReservedPerBlock;
  int stages = kMaxStages;
  while (stages > 2 && smem_for(stages) > budget) --stages;
  if (smem_for(stages) > budget) {
    ctas_per_sm = 1;
    stages = kMaxStages;
    while (stages > 2 && smem_for(stages) > kSmemPerBlockMax) --stages;
  }
  if (stages_override > 0) {
    if (smem_for(stages_override) > kSmemPerBlockMax) return BSGEMV_ERR_UNSUPPORTED;
    stages = stages_override;
    if (smem_for(stages) > budget) ctas_per_sm = 1;
  }
  g->ring_bytes = stages * g->slot_bytes;
  g->red_off = g->ring_bytes;
  g->bar_off = g->red_off + g->red_bytes;

  bsgemv_geometry& pub = g->pub;
  pub.variant = BSGEMV_VARIANT_MMA;
  pub.rows_per_tile = kRowsPerTile;
  pub.k_per_stage = g->kc;
  pub.stages = stages;
  pub.consumer_warps = kConsumerWarps;
  pub.ctas_per_sm = ctas_per_sm;
  pub.sm_count = sm_count;
  pub.tiles = ceil_div(N, kRowsPerTile);
  pub.stages_per_tile = ceil_div(K, g->kc);
  pub.total_stages = pub.tiles * pub.stages_per_tile;
  int64_t ctas = std::min<int64_t>(pub.total_stages, int64_t(sm_count) * ctas_per_sm);
  if (ctas_override > 0) ctas = std::min<int64_t>(pub.total_stages, ctas_override);
  pub.ctas = static_cast<int>(ctas);
  pub.smem_bytes = smem_for(stages);
  // workspace: partial slots [ctas][2], counters [tiles], error word
  pub.workspace_bytes = int64_t(pub.ctas) * 2 * g->slot_floats * 4 + pub.tiles * 4 + 256;
  return BSGEMV_OK;
}

}  // namespace bsg

extern "C" int bsgemv_geometry_for(int format, int block_size, int has_zp, int64_t N, int64_t K,
                                   int max_M, int sm_count, bsgemv_geometry* g) {
  if (g == nullptr) return BSGEMV_ERR_INVALID_ARG;
  bsg::Geometry geo;
  const int rc = bsg::compute_geometry(format, block_size, has_zp, N, K, max_M, sm_count, 0, 0, &geo);
  if (rc != BSGEMV_OK) return rc;
  *g = geo.pub;
  return BSGEMV_OK;
}
