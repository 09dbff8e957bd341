// bsgemv_geometry.cpp -- pure host code: argument validation and the launch geometry.
//
// Everything here depends only on the problem (format, block size, zero points, N, K, max_M)
// and the SM count, never on M of a call, so every M run through one plan takes the same
// per-row summation order (rows are bit-identical across M).
//
// Choices (each one the faster of the alternatives measured on GB300, as stated below):
//   * 64 or 128 output columns per CTA tile (one or two 64-row halves), 4 consumer warps (each
//     one 16-row group of every half, over a whole stage) + 1 copy warp.  Two halves halve the
//     per-row cost of everything a warp does once per stage and chunk (activation fragments,
//     barrier waits, side loads, ring bookkeeping) but halve the tiles.  Plans for up to 16 rows
//     take them when, with 128-row tiles, at most kTallMaxCtasPerTile resident CTAs share a tile
//     on average and there are at least kTallMinStages stages per resident CTA (measured on
//     GB300, calls of 1 to 8 rows: int4 151936 x 4096 16 % and 12288 x 4096 22 % faster, NVFP4
//     248320 x 2048 7 %, int8 12288 x 4096 2-4 %; with 9 to 40 resident CTAs per tile -- int4
//     4096 x 4096 and 4096 x 12288, int8 / FP8 shapes of 4096 to 8192 columns, FP8 5120 x 17408
//     -- 3 to 65 % slower: a coarser split with more partial sums per tile);
//   * 4 CTAs per SM for one half and one n8 activation tile, 3 for up to three n8 tiles or two
//     halves, 2 for four n8 tiles (accumulator registers and shared memory);
//   * a ring of up to 12 stages of 128 weight bytes per row (256 k of the 4-bit formats, 128 k of
//     the 8-bit ones) plus the stage's activations, as deep as the shared-memory share of a CTA
//     allows, so that every SM keeps tens of KB of weight in flight;
//   * a side ring of scale / zero-point boxes, each covering 64 bytes of scales per row (4 to
//     64 stages), so that side data costs one TMA per box instead of copies every stage;
//   * stream-K: the tiles x stages work is split into equal contiguous ranges over
//     min(total stages, CTAs per SM x SMs) persistent CTAs, which balances every shape to within one
//     stage per CTA without a wave tail.
#include <algorithm>
#include <cstdint>
#include <cstring>

#include "bsgemv_internal.h"

namespace bsg {

namespace {
// 128-row tiles: when at most this many resident CTAs share a tile on average, and the tiles
// hold at least this many stages per resident CTA
constexpr int kTallMaxCtasPerTile = 5;
constexpr int kTallMinStages = 2;
constexpr int kSmemPerSm = 233472;       // 228 KB shared memory per SM on sm_100-class parts
constexpr int kSmemPerBlockMax = 232448; // 227 KB opt-in maximum per CTA
constexpr int kReservedPerBlock = 1024;  // reserved by the system per resident CTA

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool is_pow2_block(int bs) {
  return bs == 16 || bs == 32 || bs == 64 || bs == 128 || bs == 256;
}
}  // namespace

namespace {

// The geometry for a kernel of `mt` n8 activation tiles (mt >= mt_for_m(max_M)) and `halves`
// 64-row halves per tile.
int geometry_for_tiles(int format, int block_size, int has_zp, int64_t N, int64_t K, int max_M,
                       int sm_count, int ctas_override, int stages_override, int split,
                       int cluster, int mt, int halves, int rows, Geometry* g) {
  if (g == nullptr) return BSGEMV_ERR_INVALID_ARG;
  std::memset(g, 0, sizeof(*g));
  if ((format & ~(0xFF | BSGEMV_ACT_BF16)) != 0) return BSGEMV_ERR_INVALID_ARG;
  const int fmt = format & 0xFF;
  if (fmt < kInt4 || fmt > kNvfp4) return BSGEMV_ERR_INVALID_ARG;
  if (has_zp != 0 && has_zp != 1) return BSGEMV_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || max_M < 1 || max_M > kMaxM || sm_count < 1 || block_size < 1)
    return BSGEMV_ERR_INVALID_ARG;
  if (rows < 1 || rows > max_M) return BSGEMV_ERR_INVALID_ARG;
  if (ctas_override < 0 || stages_override < 0 || stages_override > kMaxStages)
    return BSGEMV_ERR_INVALID_ARG;
  if (split < BSGEMV_SPLIT_AUTO || split > BSGEMV_SPLIT_CLUSTER || cluster < 0 ||
      cluster > kMaxCluster)
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
  if (N > (int64_t(1) << 31) - kMaxRowsPerTile || K > (int64_t(1) << 30))
    return BSGEMV_ERR_UNSUPPORTED;
  const int rpt = halves * kBoxRows;  // output columns per tile

  const bool four = (fmt == kInt4 || fmt == kNvfp4);
  g->fmt = fmt;
  g->bf16 = (format & BSGEMV_ACT_BF16) ? 1 : 0;
  g->has_zp = has_zp;
  g->block_size = block_size;
  g->max_M = max_M;
  g->N = N;
  g->K = K;
  g->kpc = four ? 32 : 16;
  g->kc = stage_k(fmt, halves);
  g->stage_bytes = stage_bytes(fmt, halves);
  g->mt_max = mt;
  g->halves = halves;
  g->scale_es = (fmt == kFp8) ? 4 : (fmt == kNvfp4 ? 1 : 2);
  g->nb_s = static_cast<int>(K / block_size);
  g->scale_pitch = g->nb_s * g->scale_es;
  g->zp_pitch = (fmt == kInt4) ? (g->nb_s + 1) / 2 : g->nb_s;

  // activation ring: per stage, max_M rows of the stage's k (2 kc bytes) padded by one chunk's
  // activation bytes (32 or 64: consecutive rows start in different banks)
  const int act_pitch = 2 * g->kc + (four ? 64 : 32);
  g->act_bytes = max_M * act_pitch;
  // side ring: one box holds kSideScaleBytes of scales per row (64 / es blocks), i.e.
  // 2^rs_log2 stages, and the zero points of the same blocks
  const int blocks_per_box = kSideScaleBytes / g->scale_es;
  const int64_t stages_per_box = int64_t(blocks_per_box) * block_size / g->kc;
  g->rs_log2 = 0;
  while ((int64_t(1) << (g->rs_log2 + 1)) <= stages_per_box) ++g->rs_log2;
  g->zbox_bytes = (fmt == kInt4) ? blocks_per_box / 2 : blocks_per_box;
  const bool side_possible = (g->scale_pitch % 16 == 0) && (!has_zp || g->zp_pitch % 16 == 0);
  g->side_bytes = side_possible
                      ? static_cast<int>(ceil_div(rpt * (kSideScaleBytes +
                                                                  (has_zp ? g->zbox_bytes : 0)),
                                                  128) * 128)
                      : 0;
  g->slot_floats = halves * g->mt_max * 32 * 4;

  const int64_t spt = ceil_div(K, g->kc);
  const int64_t tiles = ceil_div(N, rpt);
  const int64_t total = tiles * spt;

  // activation ring bytes, rounded up so that the side ring after it starts 128-byte aligned
  auto act_ring = [&](int stages) { return (stages * g->act_bytes + 127) / 128 * 128; };
  // side boxes in flight over a ring of `stages`: a box spans min(2^rs, stages per tile) stages
  auto side_slots_for = [&](int stages) {
    if (g->side_bytes == 0) return 0;
    const int64_t span = std::min<int64_t>(int64_t(1) << g->rs_log2, spt);
    return static_cast<int>(std::min<int64_t>(4, std::max<int64_t>(2, ceil_div(stages, span) + 1)));
  };
  auto smem_with = [&](int stages, int red) {
    const int ss = side_slots_for(stages);
    return 1024 + stages * g->stage_bytes + act_ring(stages) + ss * g->side_bytes + red +
           8 * (2 * stages + 9);
  };
  const int slots_per_sm = ctas_per_sm_for(g->mt_max, halves);
  const int64_t slots = int64_t(sm_count) * slots_per_sm;
  const int budget_slots = kSmemPerSm / slots_per_sm - kReservedPerBlock;

  // K split.  Stream-K gives every CTA ceil(T / slots) stages of the tiles x stages space T but
  // ends every call with a global last-arriver reduction; a cluster of C CTAs per tile gives each
  // ceil(spt / C) stages and reduces in the leader's shared memory (no atomics, no global
  // round trips).  Automatic choice: the cluster split with the fewest stages per CTA (the
  // smallest such C) among clusters of at most 8 CTAs that divide the tile's stages evenly (or
  // split it unevenly where that cuts the largest share by a quarter), when that is within one
  // stage of stream-K's, the tiles x C CTAs fit one wave and the leader's reduction buffer
  // leaves room for a ring of two stages.
  // Reduction buffer: per CTA of the cluster and consumer warp, the fragment lanes that hold
  // output columns below max_M (quad lanes t < red_tq) of each n8 tile.
  g->red_tq = (g->mt_max >= 2) ? 4 : static_cast<int>(std::min<int64_t>(4, ceil_div(max_M, 2)));
  const int red_warp = halves * g->mt_max * 8 * g->red_tq * 16;
  auto red_for = [&](int c) { return c >= 2 ? c * kConsumerWarps * red_warp : 0; };
  // Cluster split with an even share per CTA: the ring needs no more stages than the share, and
  // one side box when the share never crosses a box boundary (it divides the box's stages)
  auto cluster_stages = [&](int64_t c) {
    return static_cast<int>(std::min<int64_t>(kMaxStages, ceil_div(spt, c)));
  };
  auto cluster_one_box = [&](int64_t c) {
    const int64_t share = spt / c;
    return spt % c == 0 && ((int64_t(1) << g->rs_log2) % share == 0);
  };
  // (a single side slot only when that is what makes the split fit: measured on GB300, the
  // smaller footprint was otherwise slower for back-to-back calls)
  auto cluster_smem_ss = [&](int64_t c, int stages, bool one) {
    const int ss = (g->side_bytes == 0) ? 0 : (one ? 1 : side_slots_for(stages));
    return 1024 + stages * g->stage_bytes + act_ring(stages) + ss * g->side_bytes +
           red_for(static_cast<int>(c)) + 8 * (2 * stages + 9);
  };
  auto cluster_one_slot = [&](int64_t c) {
    const int st = std::min(2, cluster_stages(c));
    return cluster_one_box(c) && cluster_smem_ss(c, st, false) > budget_slots;
  };
  auto cluster_smem = [&](int64_t c, int stages) {
    return cluster_smem_ss(c, stages, cluster_one_slot(c));
  };
  auto cluster_fits = [&](int64_t c) {
    return c <= kMaxCluster && c <= spt && tiles * c <= slots &&
           cluster_smem(c, std::min(2, cluster_stages(c))) <= budget_slots;
  };
  int C = 0;
  if (split == BSGEMV_SPLIT_CLUSTER && cluster > 0) {
    if (!cluster_fits(cluster)) return BSGEMV_ERR_UNSUPPORTED;
    C = cluster;
  } else if (split == BSGEMV_SPLIT_CLUSTER || (split == BSGEMV_SPLIT_AUTO && ctas_override == 0)) {
    // (a CTA-count override describes a stream-K grid: it implies stream-K)
    const int64_t sk = ceil_div(total, std::min<int64_t>(total, slots));  // stream-K stages/CTA
    int64_t best = -1, best_uneven = -1;
    int C_uneven = 0;
    for (int c = 1; c <= kMaxCluster; ++c) {
      // (a size that does not fit does not end the search: a larger one can still fit, as a
      // share that lies inside one side box needs a single side slot)
      if (!cluster_fits(c)) continue;
      // automatic: clusters of at most 8 CTAs (measured on GB300: 16-CTA clusters were slower
      // than stream-K)
      if (split == BSGEMV_SPLIT_AUTO && c > kMaxAutoCluster) continue;
      const int64_t st = ceil_div(spt, c);
      // automatic: a one-stage share only while the grid stays within half the resident slots
      // (measured on GB300: FP8 4096 x 2048, 512 CTAs of one stage each, 8-17 % slower than 256
      // of two; FP8 512 x 2048 and NVFP4 2048 x 2048, 64 and 256 CTAs, fastest at one stage)
      if (split == BSGEMV_SPLIT_AUTO && st == 1 && tiles * c > slots / 2) continue;
      if (split == BSGEMV_SPLIT_AUTO && spt % c != 0) {
        if (best_uneven < 0 || st < best_uneven) {
          best_uneven = st;
          C_uneven = c;
        }
        continue;
      }
      if (best < 0 || st < best) {
        best = st;
        C = c;
      }
    }
    // taken when a CTA's share is within one stage of stream-K's, or at most 4 stages (stream-K
    // with a share of one or two stages has many partial sums per tile to add: measured slower)
    if (split == BSGEMV_SPLIT_AUTO && (C == 0 || best > std::max<int64_t>(sk + 1, 4))) C = 0;
    // automatic: an even cluster split of 4 or more CTAs so taken gives way to a cluster whose
    // CTAs' shares differ by one stage (the CTA with the extra stage sets the pace) only where
    // that cuts the largest share by a quarter or more.  Measured on GB300: 4-CTA clusters of 4
    // stages against 6-CTA clusters of 2-3, where 8-CTA clusters exceed the resident slots: int4
    // 4096 x 4096 in plans for 16 rows 4-15 % faster at every M, FP8 2048 x 4096 in plans for 9
    // rows 9 %; 2-CTA clusters of 4 stages against 3-CTA clusters of 2-3 (FP8 8192 x 2048, plans
    // for 16 rows): up to 33 % slower.  Plans for up to 16 rows only: the residency of plans for
    // 17 to 24 rows is chosen by the split it keeps, and was measured with even splits.
    if (split == BSGEMV_SPLIT_AUTO && g->mt_max <= 2 && C >= 4 && C_uneven > 0 &&
        best_uneven * 4 <= best * 3) {
      best = best_uneven;
      C = C_uneven;
    }
    if (split == BSGEMV_SPLIT_CLUSTER && C == 0) return BSGEMV_ERR_UNSUPPORTED;
  }
  g->red_bytes = red_for(C);
  auto smem_for = [&](int stages) {
    return C > 0 ? cluster_smem(C, stages) : smem_with(stages, g->red_bytes);
  };
  int ctas_per_sm = slots_per_sm;
  const int budget = budget_slots;
  // the ring: as deep as fits (at most the CTA's share of a tile under the cluster split)
  const int max_stages = C > 0 ? cluster_stages(C) : kMaxStages;
  const int min_stages = std::min(2, max_stages);
  int stages = max_stages;
  while (stages > min_stages && smem_for(stages) > budget) --stages;
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
  // Everything above is decided for max_M rows (and so is the same for every call of a plan).
  // The ring of a call with fewer rows holds fewer activation bytes per stage, so the same
  // per-CTA budget takes more stages: the ring depth changes nothing that a row's summation
  // order depends on (which CTA sums which stages, and in what order), only how many stages
  // are in flight.
  if (rows < max_M) {
    g->act_bytes = rows * act_pitch;
    if (stages_override == 0) {
      const int b = ctas_per_sm == 1 ? kSmemPerBlockMax : budget;
      stages = max_stages;
      while (stages > min_stages && smem_for(stages) > b) --stages;
    }
  }
  g->side_slots = (C > 0 && g->side_bytes != 0 && cluster_one_slot(C)) ? 1 : side_slots_for(stages);
  g->act_off = stages * g->stage_bytes;
  g->side_off = g->act_off + act_ring(stages);  // side boxes are TMA destinations: 128-aligned
  g->red_off = g->side_off + g->side_slots * g->side_bytes;
  g->bar_off = g->red_off + g->red_bytes;
  // Alignment the kernel relies on (checked here, on the host, rather than found on the device):
  // weight boxes 1024 (128-byte swizzle atoms), activation rows 16 (cp.async, 16-byte loads),
  // side boxes 128 (TMA destinations), the reduction buffer 16 (v4 stores), mbarriers 8.
  if (g->act_off % 1024 != 0 || g->act_bytes % 16 != 0 || g->side_off % 128 != 0 ||
      g->side_bytes % 128 != 0 || g->red_off % 16 != 0 || g->bar_off % 8 != 0)
    return BSGEMV_ERR_UNSUPPORTED;

  bsgemv_geometry& pub = g->pub;
  pub.variant = BSGEMV_VARIANT_MMA;
  pub.rows_per_tile = rpt;
  pub.k_per_stage = g->kc;
  pub.stages = stages;
  pub.consumer_warps = kConsumerWarps;
  pub.ctas_per_sm = ctas_per_sm;
  pub.sm_count = sm_count;
  pub.tiles = tiles;
  pub.stages_per_tile = spt;
  pub.total_stages = total;
  pub.cluster = C;
  const int64_t resident = int64_t(sm_count) * ctas_per_sm;
  int64_t ctas = std::min<int64_t>(pub.total_stages, resident);
  // Stream-K over fewer tiles than resident CTAs: a whole number (>= 2) of CTAs per tile, so
  // that the CTAs' ranges meet the tile boundaries (each CTA holds part of one tile: one
  // partial sum, no tile crossing).  Measured faster than filling every slot.
  if (C == 0 && pub.total_stages > resident && resident / tiles >= 2)
    ctas = tiles * (resident / tiles);
  if (ctas_override > 0) ctas = std::min<int64_t>(pub.total_stages, ctas_override);
  if (C > 0) ctas = tiles * C;
  pub.ctas = static_cast<int>(ctas);
  pub.smem_bytes = smem_for(stages);
  // workspace: partial slots [ctas][2][warps], counters [tiles][warps], error word
  pub.workspace_bytes = int64_t(pub.ctas) * 2 * kConsumerWarps * g->slot_floats * 4 +
                        pub.tiles * kConsumerWarps * 4 + 256;
  return BSGEMV_OK;
}

}  // namespace

int compute_geometry(int format, int block_size, int has_zp, int64_t N, int64_t K, int max_M,
                     int sm_count, int ctas_override, int stages_override, int split, int cluster,
                     Geometry* g, int rows, int tile_rows) {
  const int mt = (max_M >= 1 && max_M <= kMaxM) ? mt_for_m(max_M) : 1;
  if (rows == 0) rows = max_M;
  if (tile_rows != 0 && tile_rows != kBoxRows && tile_rows != kMaxRowsPerTile)
    return BSGEMV_ERR_INVALID_ARG;
  // (128-row tiles: kernels for calls of up to 16 rows only)
  if (tile_rows == kMaxRowsPerTile && mt > 2) return BSGEMV_ERR_UNSUPPORTED;
  if (tile_rows == kMaxRowsPerTile)
    return geometry_for_tiles(format, block_size, has_zp, N, K, max_M, sm_count, ctas_override,
                              stages_override, split, cluster, mt, 2, rows, g);
  int rc = geometry_for_tiles(format, block_size, has_zp, N, K, max_M, sm_count, ctas_override,
                              stages_override, split, cluster, mt, 1, rows, g);
  if (rc != BSGEMV_OK) return rc;
  if (tile_rows == 0 && mt <= 2) {
    // Two halves when the plan's work per resident CTA is long (see the header); decided on the
    // plan's geometry (rows = max_M) and so the same for every call of the plan.
    Geometry tall;
    if (geometry_for_tiles(format, block_size, has_zp, N, K, max_M, sm_count, ctas_override,
                           stages_override, split, cluster, mt, 2, max_M, &tall) == BSGEMV_OK &&
        tall.pub.tiles * kTallMaxCtasPerTile >= int64_t(sm_count) * tall.pub.ctas_per_sm &&
        tall.pub.total_stages >= int64_t(kTallMinStages) * sm_count * tall.pub.ctas_per_sm &&
        // ... unless 128-row tiles lose the cluster split that 64-row tiles keep, leaving several
        // CTAs per tile to a stream-K reduction (measured on GB300, 12288 x 4096 in plans for 16
        // rows: 64-row tiles in 2-CTA clusters 2-9 % faster than 128-row stream-K for int4, 13-17 %
        // for int8 at M = 9 and 16)
        !(tall.pub.cluster == 0 && tall.pub.ctas > tall.pub.tiles && g->pub.cluster >= 2)) {
      if (rows == max_M) {
        *g = tall;
        return BSGEMV_OK;
      }
      return geometry_for_tiles(format, block_size, has_zp, N, K, max_M, sm_count, ctas_override,
                                stages_override, split, cluster, mt, 2, rows, g);
    }
  }
  if (mt != 3 || split != BSGEMV_SPLIT_AUTO || ctas_override != 0 || stages_override != 0)
    return rc;
  // Plans for 17..24 rows: three n8 tiles at 3 CTAs per SM, unless that residency's shared
  // memory (activation ring of 24 rows, reduction buffer) costs the cluster split that four
  // tiles at 2 CTAs per SM keep, with shares of at most 4 stages (measured on GB300: such small
  // shapes ran 15-25 % faster at 2 CTAs per SM; larger shapes 13-22 % faster at 3).
  Geometry four;
  if (geometry_for_tiles(format, block_size, has_zp, N, K, max_M, sm_count, 0, 0, split, 0, 4, 1,
                         rows, &four) != BSGEMV_OK)
    return rc;
  const int C4 = four.pub.cluster, C3 = g->pub.cluster;
  if (C4 >= 2 && C3 < C4 && (four.pub.stages_per_tile + C4 - 1) / C4 <= 4) *g = four;
  return BSGEMV_OK;
}

}  // namespace bsg

extern "C" int bsgemv_geometry_for(int format, int block_size, int has_zp, int64_t N, int64_t K,
                                   int max_M, int sm_count, bsgemv_geometry* g) {
  if (g == nullptr) return BSGEMV_ERR_INVALID_ARG;
  bsg::Geometry geo;
  const int rc = bsg::compute_geometry(format, block_size, has_zp, N, K, max_M, sm_count, 0, 0,
                                       BSGEMV_SPLIT_AUTO, 0, &geo);
  if (rc != BSGEMV_OK) return rc;
  *g = geo.pub;
  return BSGEMV_OK;
}
