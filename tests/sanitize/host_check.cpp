// Host code of the library under -fsanitize=address,undefined, without a GPU: the launch geometry
// over a sweep of problems and SM counts (every split, override, tile height, max_M and per-call
// row count), the kernel parameters filled from each geometry, and the C ABI's host-side paths
// (argument errors, NULL handles, the no-device path of bsgemv_plan).  Exits 0 and prints "ok" when every
// invariant holds; a sanitizer report makes it fail.  (Compiled and run by
// tests/test_sanitizers.py; the host code of "[CUDA] Pin FP8 GEMV residency for grids just past
// two blocks per SM" is tested under UBSan in the same spirit, its Tests section.)
#include <cstdio>
#include <cstring>

#include "../../block_scaled_bit_gb300/csrc/bsgemv_internal.h"

#define CHECK(cond)                                                              \
  do {                                                                           \
    if (!(cond)) {                                                               \
      std::fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond);    \
      return 1;                                                                  \
    }                                                                            \
  } while (0)

namespace {
uint64_t g_state = 0x9E3779B97F4A7C15ull;
uint64_t next() {  // xorshift64*
  g_state ^= g_state >> 12;
  g_state ^= g_state << 25;
  g_state ^= g_state >> 27;
  return g_state * 2685821657736338717ull;
}
int pick(const int* v, int n) { return v[next() % n]; }
}  // namespace

int main() {
  const int fmts[] = {bsg::kInt4, bsg::kInt8, bsg::kFp8, bsg::kNvfp4};
  const int int_bs[] = {16, 32, 64, 128, 256};
  const int sms[] = {132, 148, 152};
  long checked = 0;
  for (int it = 0; it < 4000; ++it) {
    const int fmt = pick(fmts, 4);
    const int bs = fmt == bsg::kFp8 ? 128 : fmt == bsg::kNvfp4 ? 16 : pick(int_bs, 5);
    const int zp = (fmt == bsg::kInt4 || fmt == bsg::kInt8) ? int(next() % 2) : 0;
    const int act = (next() % 2) ? BSGEMV_ACT_BF16 : 0;
    const int64_t N = 1 + int64_t(next() % (it % 10 == 0 ? 300000 : 20000));
    const int64_t K = 256 * (1 + int64_t(next() % 64));
    const int max_M = 1 + int(next() % 32);
    const int sm = pick(sms, 3);
    const int split = int(next() % 3);
    const int cluster = split == BSGEMV_SPLIT_CLUSTER ? int(next() % 9) : 0;
    const int ctas = (split == BSGEMV_SPLIT_AUTO && next() % 4 == 0) ? 1 + int(next() % 2000) : 0;
    const int stages = next() % 8 == 0 ? 1 + int(next() % bsg::kMaxStages) : 0;
    const int tile_rows_v[] = {0, 0, 64, 128};
    const int tile_rows = pick(tile_rows_v, 4);
    bsg::Geometry g;
    const int rc = bsg::compute_geometry(fmt | act, bs, zp, N, K, max_M, sm, ctas, stages, split,
                                         cluster, &g, 0, tile_rows);
    if (rc != BSGEMV_OK) {
      CHECK(rc == BSGEMV_ERR_UNSUPPORTED);
      continue;
    }
    CHECK(g.pub.ctas >= 1 && g.pub.ctas <= g.pub.total_stages);
    CHECK(g.pub.stages >= 1 && g.pub.stages <= bsg::kMaxStages);
    CHECK(g.pub.smem_bytes <= 232448 && g.act_off % 1024 == 0 && g.side_off % 128 == 0);
    CHECK(g.pub.cluster == 0 || g.pub.ctas == g.pub.tiles * g.pub.cluster);
    // tiles of one or two 64-row halves; two only for kernels of up to two n8 tiles
    CHECK(g.pub.rows_per_tile == 64 * g.halves && (g.halves == 1 || g.halves == 2));
    CHECK(tile_rows == 0 || g.pub.rows_per_tile == tile_rows);
    CHECK(g.halves == 1 || g.mt_max <= 2);
    CHECK(g.pub.tiles * g.pub.rows_per_tile >= N && (g.pub.tiles - 1) * g.pub.rows_per_tile < N);
    // a stage: one 8 KB box per half and k-box (two k-boxes for 8-bit weights with one half)
    const bool four = fmt == bsg::kInt4 || fmt == bsg::kNvfp4;
    CHECK(g.stage_bytes == ((four && g.halves == 1) ? 8192 : 16384));
    CHECK(g.pub.k_per_stage == ((!four && g.halves == 2) ? 128 : 256));
    CHECK(g.slot_floats == g.halves * g.mt_max * 128);
    // every call's ring layout keeps the plan's split, CTA count and residency
    for (int rows = 1; rows <= max_M; rows += 1 + int(next() % 5)) {
      bsg::Geometry r;
      CHECK(bsg::compute_geometry(fmt | act, bs, zp, N, K, max_M, sm, ctas, stages, split, cluster,
                                  &r, rows, tile_rows) == BSGEMV_OK);
      CHECK(r.pub.rows_per_tile == g.pub.rows_per_tile && r.halves == g.halves);
      CHECK(r.pub.ctas == g.pub.ctas && r.pub.cluster == g.pub.cluster &&
            r.pub.ctas_per_sm == g.pub.ctas_per_sm && r.pub.total_stages == g.pub.total_stages);
      CHECK(r.pub.stages >= g.pub.stages && r.pub.smem_bytes <= 232448);
      CHECK(r.bar_off % 8 == 0 && r.red_off % 16 == 0 && r.act_bytes % 16 == 0);
      bsg::OperandMaps maps;
      std::memset(&maps, 0, sizeof(maps));
      bsg::KParams k;
      bsg::fill_params(r, maps, nullptr, nullptr, nullptr, nullptr, nullptr, rows, nullptr,
                       nullptr, nullptr, &k);
      CHECK(k.M == rows && k.stages == r.pub.stages && k.skip_stage == -1 && k.wait_ns > 0);
      CHECK(k.side_tx % r.pub.rows_per_tile == 0);
      ++checked;
    }
    bsgemv_geometry pub;
    if (split == BSGEMV_SPLIT_AUTO && ctas == 0 && stages == 0 && tile_rows == 0) {
      CHECK(bsgemv_geometry_for(fmt | act, bs, zp, N, K, max_M, sm, &pub) == BSGEMV_OK);
      CHECK(std::memcmp(&pub, &g.pub, sizeof(pub)) == 0);
    }
  }
  // C ABI host paths
  bsgemv_plan_t plan = nullptr;
  CHECK(bsgemv_plan(&plan, BSGEMV_INT8, 48, 1, 64, 512, 1) == BSGEMV_ERR_UNSUPPORTED && !plan);
  CHECK(bsgemv_plan(&plan, BSGEMV_INT4, 32, 0, 0, 512, 1) == BSGEMV_ERR_INVALID_ARG && !plan);
  CHECK(bsgemv_plan(nullptr, BSGEMV_INT4, 32, 0, 64, 512, 1) == BSGEMV_ERR_INVALID_ARG);
  // a valid problem on a machine without a GPU: refused, nothing leaked or written
  const int rc = bsgemv_plan(&plan, BSGEMV_INT4, 32, 0, 4096, 4096, 16);
  CHECK(rc != BSGEMV_OK && plan == nullptr);
  CHECK(bsgemv_run(nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 1, nullptr) ==
        BSGEMV_ERR_INVALID_ARG);
  CHECK(bsgemv_plan_set_test_fault(nullptr, -1, 0) == BSGEMV_ERR_INVALID_ARG);
  CHECK(bsgemv_plan_describe(nullptr, nullptr) == BSGEMV_ERR_INVALID_ARG);
  CHECK(bsgemv_device_status(nullptr, nullptr) != BSGEMV_OK);
  CHECK(bsgemv_destroy(nullptr) == BSGEMV_OK);
  for (int s = -9; s <= 1; ++s) CHECK(bsgemv_status_string(s) != nullptr);
  std::printf("ok: %ld geometries\n", checked);
  return 0;
}
