// bsgemv_api.cu -- the C ABI declared in include/bsgemv.h (host code).
//
// A plan holds the geometry (fixed per problem and device), the device workspace of the
// stream-K reduction (partials, arrival counters, error word) and a small cache of the operands'
// TMA tensor maps.  bsgemv_run validates, encodes the tensor maps when W, scales or zp change,
// and launches one kernel on the caller's stream.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "bsgemv_internal.h"

struct bsgemv_plan_s {
  bsg::Geometry geo;                 // the plan's geometry (ring laid out for max_M rows)
  std::vector<bsg::Geometry> rows;   // [M - 1]: the same split, the ring laid out for M rows
  int format = 0;
  int device = -1;
  int sm_count = 0;
  int variant_override = 0, ctas_override = 0, stages_override = 0, rows_override = 0;
  int split = BSGEMV_SPLIT_AUTO, cluster = 0;
  int fault_skip = -1;            // bsgemv_plan_set_test_fault
  uint64_t fault_wait_ns = 0;
  void* ws = nullptr;         // one allocation: partials | counters | error word
  size_t ws_bytes = 0;
  float* partials = nullptr;
  unsigned* counters = nullptr;
  unsigned* err = nullptr;
  void* stage = nullptr;      // bsgemv_run_host staging for A and y
  size_t stage_bytes = 0;
  // tensor-map cache: the last few (W, scales, zp) pointer triples seen (e.g. rotating weight
  // copies)
  struct MapEntry {
    bool valid = false;
    const void* W = nullptr;
    const void* scales = nullptr;
    const void* zp = nullptr;
    unsigned last_use = 0;
    bsg::OperandMaps maps;
  };
  static constexpr int kMapCache = 4;
  MapEntry maps[kMapCache];
  unsigned use_clock = 0;
  bsg::KParams params;
};

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int query_device(int* dev, int* sms) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_UNSUPPORTED;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  // The kernels are built for sm_103a only.
  if (major != 10 || minor != 3) return BSGEMV_ERR_UNSUPPORTED;
  return BSGEMV_OK;
}

// The workspace for geometry `geo`, zeroed: the plan's own buffer while it is large enough,
// else a new one, and the old one is freed only once the new one exists -- so that a failed
// allocation leaves the plan with its previous geometry and workspace, still usable.  A failed
// clear leaves the plan without a workspace (its calls return BSGEMV_ERR_CUDA) until a later
// geometry change succeeds.
int alloc_workspace(bsgemv_plan_s* p, const bsg::Geometry& geo) {
  const bsgemv_geometry& g = geo.pub;
  const size_t partial_bytes =
      size_t(g.ctas) * 2 * bsg::kConsumerWarps * geo.slot_floats * sizeof(float);
  const size_t counter_bytes = size_t(g.tiles) * bsg::kConsumerWarps * sizeof(unsigned);
  const size_t need = partial_bytes + counter_bytes + 256;
  if (need > p->ws_bytes) {
    void* fresh = nullptr;
    if (cudaMalloc(&fresh, need) != cudaSuccess) {
      cudaGetLastError();
      return BSGEMV_ERR_CUDA;
    }
    if (p->ws) {
      cudaDeviceSynchronize();
      cudaFree(p->ws);
    }
    p->ws = fresh;
    p->ws_bytes = need;
  }
  p->partials = nullptr;
  p->counters = nullptr;
  p->err = nullptr;
  if (cudaMemset(p->ws, 0, p->ws_bytes) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  p->partials = static_cast<float*>(p->ws);
  p->counters = reinterpret_cast<unsigned*>(static_cast<char*>(p->ws) + partial_bytes);
  p->err = reinterpret_cast<unsigned*>(static_cast<char*>(p->ws) + partial_bytes + counter_bytes);
  return BSGEMV_OK;
}

int rebuild_geometry(bsgemv_plan_s* p) {
  bsg::Geometry geo;
  const int max_M = p->geo.max_M;
  // the CUDA-core variant runs 64-row tiles
  const int tile_rows = p->variant_override == BSGEMV_VARIANT_CUDA_CORE
                            ? (p->rows_override == bsg::kMaxRowsPerTile ? -1 : bsg::kBoxRows)
                            : p->rows_override;
  if (tile_rows < 0) return BSGEMV_ERR_UNSUPPORTED;
  int rc = bsg::compute_geometry(p->format, p->geo.block_size, p->geo.has_zp, p->geo.N, p->geo.K,
                                 max_M, p->sm_count, p->ctas_override, p->stages_override,
                                 p->split, p->cluster, &geo, max_M, tile_rows);
  if (rc != BSGEMV_OK) return rc;
  std::vector<bsg::Geometry> rows(max_M);
  for (int m = 1; m <= max_M && rc == BSGEMV_OK; ++m)
    rc = bsg::compute_geometry(p->format, p->geo.block_size, p->geo.has_zp, p->geo.N, p->geo.K,
                               max_M, p->sm_count, p->ctas_override, p->stages_override, p->split,
                               p->cluster, &rows[m - 1], m, tile_rows);
  if (rc != BSGEMV_OK) return rc;
  if (p->variant_override == BSGEMV_VARIANT_CUDA_CORE) {
    geo.pub.variant = BSGEMV_VARIANT_CUDA_CORE;
    for (auto& r : rows) r.pub.variant = BSGEMV_VARIANT_CUDA_CORE;
  }
  // the workspace first: the geometry is taken only once its workspace exists
  if ((rc = alloc_workspace(p, geo)) != BSGEMV_OK) return rc;
  // the side boxes' tensor maps are shaped by the tile's rows: encode them again
  for (auto& e : p->maps) e.valid = false;
  p->geo = geo;
  p->rows.swap(rows);
  return BSGEMV_OK;
}

// Fill p->params for this call.  The tensor maps are re-encoded only for a new (W, scales, zp).
int prepare_params(bsgemv_plan_s* p, const void* A, const void* W, const void* scales,
                   const void* zp, void* y, int M) {
  bsgemv_plan_s::MapEntry* hit = nullptr;
  for (auto& e : p->maps)
    if (e.valid && e.W == W && e.scales == scales && e.zp == zp) hit = &e;
  if (hit == nullptr) {
    // an empty entry if there is one, else the least recently used
    for (auto& e : p->maps)
      if (!e.valid) { hit = &e; break; }
    if (hit == nullptr) {
      hit = &p->maps[0];
      for (auto& e : p->maps)
        if (e.last_use < hit->last_use) hit = &e;
    }
    hit->valid = false;
    const int rc = bsg::encode_maps(p->geo, W, scales, zp, &hit->maps);
    if (rc != BSGEMV_OK) return rc;
    hit->valid = true;
    hit->W = W;
    hit->scales = scales;
    hit->zp = zp;
  }
  hit->last_use = ++p->use_clock;
  bsg::fill_params(p->rows[M - 1], hit->maps, A, W, scales, zp, y, M, p->partials, p->counters,
                   p->err, &p->params);
  p->params.skip_stage = p->fault_skip;
  if (p->fault_wait_ns > 0) p->params.wait_ns = p->fault_wait_ns;
  return BSGEMV_OK;
}

int check_device(const bsgemv_plan_s* p) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  return cur == p->device ? BSGEMV_OK : BSGEMV_ERR_WRONG_DEVICE;
}

int validate_run(const bsgemv_plan_s* p, const void* A, const void* W, const void* scales,
                 const void* zp, const void* y, int M) {
  if (p == nullptr) return BSGEMV_ERR_INVALID_ARG;
  if (p->err == nullptr) return BSGEMV_ERR_CUDA;  // no workspace (a failed clear)
  const bsg::Geometry& g = p->geo;
  if (M < 1) return BSGEMV_ERR_INVALID_ARG;
  if (M > g.max_M) return BSGEMV_ERR_M_TOO_LARGE;
  if (!A || !W || !scales || !y) return BSGEMV_ERR_INVALID_ARG;
  if (g.fmt == bsg::kNvfp4 && zp == nullptr) return BSGEMV_ERR_INVALID_ARG;  // global scale
  if ((g.fmt == bsg::kInt4 || g.fmt == bsg::kInt8) && g.has_zp && zp == nullptr)
    return BSGEMV_ERR_INVALID_ARG;
  if ((g.fmt == bsg::kInt4 || g.fmt == bsg::kInt8) && !g.has_zp && zp != nullptr)
    return BSGEMV_ERR_INVALID_ARG;
  if (g.fmt == bsg::kFp8 && zp != nullptr) return BSGEMV_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(W, 16) || !aligned(y, 16)) return BSGEMV_ERR_MISALIGNED;
  if (!aligned(scales, g.scale_es)) return BSGEMV_ERR_MISALIGNED;
  if (g.fmt == bsg::kNvfp4 && !aligned(zp, 4)) return BSGEMV_ERR_MISALIGNED;
  return BSGEMV_OK;
}

// The geometry of the prepared call (its ring laid out for the call's M).
int launch(bsgemv_plan_s* p, cudaStream_t s) {
  return bsg::launch_gemv(p->rows[p->params.M - 1], p->params, s);
}

}  // namespace

extern "C" {

int bsgemv_version(void) { return 200; }

const char* bsgemv_status_string(int status) {
  switch (status) {
    case BSGEMV_OK: return "ok";
    case BSGEMV_ERR_INVALID_ARG: return "invalid argument";
    case BSGEMV_ERR_UNSUPPORTED: return "unsupported problem or device";
    case BSGEMV_ERR_MISALIGNED: return "misaligned pointer";
    case BSGEMV_ERR_M_TOO_LARGE: return "M exceeds the plan's max_M";
    case BSGEMV_ERR_CUDA: return "CUDA error";
    case BSGEMV_ERR_WRONG_DEVICE: return "current device is not the plan's device";
    case BSGEMV_ERR_DEVICE_TIMEOUT: return "a kernel abandoned a bounded wait";
    case BSGEMV_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed scratch area of bsgemv_run_noalloc";
  }
  return "unknown status";
}

int bsgemv_plan(bsgemv_plan_t* out, int format, int block_size, int has_zp, int64_t N, int64_t K,
                int max_M) {
  if (out == nullptr) return BSGEMV_ERR_INVALID_ARG;
  *out = nullptr;
  bsg::Geometry probe;
  int rc = bsg::compute_geometry(format, block_size, has_zp, N, K, max_M, 1, 0, 0,
                                 BSGEMV_SPLIT_AUTO, 0, &probe);
  if (rc != BSGEMV_OK) return rc;  // argument errors need no GPU
  int dev = -1, sms = 0;
  rc = query_device(&dev, &sms);
  if (rc != BSGEMV_OK) return rc;
  bsgemv_plan_s* p = new (std::nothrow) bsgemv_plan_s();
  if (!p) return BSGEMV_ERR_CUDA;
  p->format = format;
  p->device = dev;
  p->sm_count = sms;
  p->geo = probe;
  rc = rebuild_geometry(p);
  if (rc != BSGEMV_OK) {
    if (p->ws) cudaFree(p->ws);
    delete p;
    return rc;
  }
  *out = p;
  return BSGEMV_OK;
}

int bsgemv_run(bsgemv_plan_t plan, const void* A, const void* W, const void* scales,
               const void* zp, void* y, int M, void* stream) {
  int rc = validate_run(plan, A, W, scales, zp, y, M);
  if (rc != BSGEMV_OK) return rc;
  rc = check_device(plan);
  if (rc != BSGEMV_OK) return rc;
  rc = prepare_params(plan, A, W, scales, zp, y, M);
  if (rc != BSGEMV_OK) return rc;
  return launch(plan, static_cast<cudaStream_t>(stream));
}

int bsgemv_run_bias(bsgemv_plan_t plan, const void* A, const void* W, const void* scales,
                    const void* zp, const void* bias, void* y, int M, void* stream) {
  int rc = validate_run(plan, A, W, scales, zp, y, M);
  if (rc != BSGEMV_OK) return rc;
  if (bias == nullptr) return BSGEMV_ERR_INVALID_ARG;
  if (!aligned(bias, 2)) return BSGEMV_ERR_MISALIGNED;
  rc = check_device(plan);
  if (rc != BSGEMV_OK) return rc;
  rc = prepare_params(plan, A, W, scales, zp, y, M);
  if (rc != BSGEMV_OK) return rc;
  plan->params.bias = static_cast<const uint16_t*>(bias);
  return launch(plan, static_cast<cudaStream_t>(stream));
}

namespace {

// A host -> device into the plan's staging buffer, the GEMV, y device -> host, all on `stream`;
// waits for the stream when `sync`.
// The device address of pinned host memory (nullptr for pageable memory, device memory, or a
// mapping the current device cannot use).
void* host_mapping(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

int run_host_impl(bsgemv_plan_t plan, const void* A_host, const void* W, const void* scales,
                  const void* zp, void* y_host, int M, void* stream, bool sync) {
  if (plan == nullptr || A_host == nullptr || y_host == nullptr) return BSGEMV_ERR_INVALID_ARG;
  const bsg::Geometry& g = plan->geo;
  if (M < 1) return BSGEMV_ERR_INVALID_ARG;
  if (M > g.max_M) return BSGEMV_ERR_M_TOO_LARGE;
  int rc = check_device(plan);
  if (rc != BSGEMV_OK) return rc;
  const size_t a_bytes = size_t(g.max_M) * g.K * 2;
  const size_t a_pad = (a_bytes + 255) / 256 * 256;
  const size_t need = a_pad + size_t(g.max_M) * g.N * 2;
  if (plan->stage_bytes < need) {
    if (plan->stage) cudaFree(plan->stage);
    plan->stage = nullptr;
    plan->stage_bytes = 0;
    if (cudaMalloc(&plan->stage, need) != cudaSuccess) {
      cudaGetLastError();
      return BSGEMV_ERR_CUDA;
    }
    plan->stage_bytes = need;
  }
  void* dA = plan->stage;
  void* dy = static_cast<char*>(plan->stage) + a_pad;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t a_call = size_t(M) * g.K * 2, y_call = size_t(M) * g.N * 2;
  // Pinned host buffers (16-byte aligned) are used through their device mapping: A is copied
  // into the staging buffer by a kernel (whose start-up overlaps the neighbouring kernels, where
  // a copy-engine transfer adds latency of its own) and the GEMV writes y straight into the host
  // buffer.  Other host memory goes by copy-engine transfers through the staging buffer.
  void* A_map = host_mapping(A_host);
  void* y_map = host_mapping(y_host);
  const bool by_kernel = A_map != nullptr && y_map != nullptr && aligned(A_map, 16) &&
                         aligned(y_map, 16);
  if (by_kernel) {
    if ((rc = bsg::launch_host_copy(dA, A_map, a_call, plan->sm_count, s)) != BSGEMV_OK) return rc;
  } else if (cudaMemcpyAsync(dA, A_host, a_call, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    return BSGEMV_ERR_CUDA;
  }
  rc = bsgemv_run(plan, dA, W, scales, zp, by_kernel ? y_map : dy, M, stream);
  if (rc != BSGEMV_OK) return rc;
  if (!by_kernel && cudaMemcpyAsync(y_host, dy, y_call, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return BSGEMV_ERR_CUDA;
  if (!sync) return BSGEMV_OK;
  return cudaStreamSynchronize(s) == cudaSuccess ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

}  // namespace

int bsgemv_run_host(bsgemv_plan_t plan, const void* A_host, const void* W, const void* scales,
                    const void* zp, void* y_host, int M, void* stream) {
  return run_host_impl(plan, A_host, W, scales, zp, y_host, M, stream, true);
}

int bsgemv_run_host_async(bsgemv_plan_t plan, const void* A_host, const void* W,
                          const void* scales, const void* zp, void* y_host, int M, void* stream) {
  return run_host_impl(plan, A_host, W, scales, zp, y_host, M, stream, false);
}

int bsgemv_destroy(bsgemv_plan_t plan) {
  if (plan == nullptr) return BSGEMV_OK;
  int rc = BSGEMV_OK;
  if (plan->ws || plan->stage) {
    if (cudaDeviceSynchronize() != cudaSuccess) rc = BSGEMV_ERR_CUDA;
    if (plan->ws) cudaFree(plan->ws);
    if (plan->stage) cudaFree(plan->stage);
  }
  delete plan;
  return rc;
}

int bsgemv_debug_dequant(bsgemv_plan_t plan, const void* W, const void* scales, const void* zp,
                         float* out, void* stream) {
  if (plan == nullptr || W == nullptr || scales == nullptr || out == nullptr)
    return BSGEMV_ERR_INVALID_ARG;
  const bsg::Geometry& g = plan->geo;
  if ((g.fmt == bsg::kNvfp4 || g.has_zp) && zp == nullptr) return BSGEMV_ERR_INVALID_ARG;
  if (!aligned(W, 16) || !aligned(scales, g.scale_es)) return BSGEMV_ERR_MISALIGNED;
  const int rc = check_device(plan);
  if (rc != BSGEMV_OK) return rc;
  return bsg::launch_debug_dequant(
      g.fmt, g.bf16, g.has_zp, g.block_size, g.N, g.K, static_cast<const uint8_t*>(W),
      static_cast<const uint8_t*>(scales),
      (g.fmt == bsg::kInt4 || g.fmt == bsg::kInt8) ? static_cast<const uint8_t*>(zp) : nullptr,
      g.fmt == bsg::kNvfp4 ? static_cast<const float*>(zp) : nullptr, out,
      static_cast<cudaStream_t>(stream));
}

int bsgemv_plan_set_override(bsgemv_plan_t plan, int variant, int ctas, int rows_per_tile,
                             int stages) {
  if (plan == nullptr || variant < 0 || ctas < 0 || stages < 0 ||
      (rows_per_tile != 0 && rows_per_tile != bsg::kBoxRows &&
       rows_per_tile != bsg::kMaxRowsPerTile))
    return BSGEMV_ERR_INVALID_ARG;
  if (variant > BSGEMV_VARIANT_CUDA_CORE) return BSGEMV_ERR_INVALID_ARG;
  // the CUDA-core variant accumulates at most 8 activation rows per lane
  if (variant == BSGEMV_VARIANT_CUDA_CORE && plan->geo.max_M > 8) return BSGEMV_ERR_UNSUPPORTED;
  const int old_c = plan->ctas_override, old_s = plan->stages_override;
  const int old_v = plan->variant_override, old_r = plan->rows_override;
  if (variant) plan->variant_override = variant;
  if (ctas) plan->ctas_override = ctas;
  if (stages) plan->stages_override = stages;
  if (rows_per_tile) plan->rows_override = rows_per_tile;
  const int rc = rebuild_geometry(plan);
  if (rc != BSGEMV_OK) {
    plan->ctas_override = old_c;
    plan->stages_override = old_s;
    plan->variant_override = old_v;
    plan->rows_override = old_r;
    rebuild_geometry(plan);
  }
  return rc;
}

int bsgemv_plan_set_split(bsgemv_plan_t plan, int split, int cluster_size) {
  if (plan == nullptr || split < BSGEMV_SPLIT_AUTO || split > BSGEMV_SPLIT_CLUSTER ||
      cluster_size < 0 || cluster_size > bsg::kMaxCluster ||
      (cluster_size != 0 && split != BSGEMV_SPLIT_CLUSTER))
    return BSGEMV_ERR_INVALID_ARG;
  const int old_s = plan->split, old_c = plan->cluster;
  plan->split = split;
  plan->cluster = cluster_size;
  const int rc = rebuild_geometry(plan);
  if (rc != BSGEMV_OK) {
    plan->split = old_s;
    plan->cluster = old_c;
    rebuild_geometry(plan);
  }
  return rc;
}

int bsgemv_plan_autotune(bsgemv_plan_t plan, const void* A, const void* W, const void* scales,
                         const void* zp, void* y, int M, int reps, void* stream) {
  int rc = validate_run(plan, A, W, scales, zp, y, M);
  if (rc != BSGEMV_OK) return rc;
  if (reps < 1 || reps > 100) return BSGEMV_ERR_INVALID_ARG;
  rc = check_device(plan);
  if (rc != BSGEMV_OK) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  const bsg::Geometry& g = plan->geo;

  // Candidates, in two rounds.  First the K split under each tile height (the automatic one,
  // 64 and 128 rows): the plan's automatic choice first, stream-K over the default grid and
  // over 1 .. 4 CTAs per SM, and a thread-block cluster of each size 2 .. 8 per tile.  Then the
  // ring depth of the fastest of those: 2, 3, 4, 6, 8 and 12 stages, where the CTAs per SM stay
  // as they were.  Candidates the plan cannot run (a cluster or a ring that does not fit, 128-row
  // tiles in a plan for more than 16 rows) are skipped, and so are repeats of a geometry already
  // measured.
  struct Cand {
    int split, cluster, ctas, rows, stages;
  };
  std::vector<Cand> cands;
  for (int rows : {0, bsg::kBoxRows, bsg::kMaxRowsPerTile}) {
    cands.push_back({BSGEMV_SPLIT_AUTO, 0, 0, rows, 0});
    cands.push_back({BSGEMV_SPLIT_STREAM_K, 0, 0, rows, 0});
    for (int k = 1; k <= 4; ++k) cands.push_back({BSGEMV_SPLIT_STREAM_K, 0, k * plan->sm_count, rows, 0});
    for (int c = 2; c <= bsg::kMaxAutoCluster; ++c) cands.push_back({BSGEMV_SPLIT_CLUSTER, c, 0, rows, 0});
  }
  const int kRingDepths[] = {2, 3, 4, 6, 8, 12};

  // The regime the calls run in: back to back on one stream, each on weights that are not in L2.
  // The caller's weight, scales and zero points are copied R - 1 times (R copies >= 3x the L2,
  // at most 8); a CUDA graph of reps rounds over the R copies is timed per candidate.
  int l2 = 0;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, plan->device) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  const bool int_zp = (g.fmt == bsg::kInt4 || g.fmt == bsg::kInt8) && g.has_zp;
  const size_t w_bytes = static_cast<size_t>(g.N) * ((g.fmt == bsg::kInt4 || g.fmt == bsg::kNvfp4) ? g.K / 2 : g.K);
  const size_t s_bytes = static_cast<size_t>(g.N) * g.scale_pitch;
  const size_t z_bytes = int_zp ? static_cast<size_t>(g.N) * g.zp_pitch : 0;
  auto up = [](size_t b) { return (b + 255) / 256 * 256; };
  const size_t copy_bytes = up(w_bytes) + up(s_bytes) + up(z_bytes);
  const int R = static_cast<int>(std::min<size_t>(8, std::max<size_t>(1, (3 * static_cast<size_t>(l2) + copy_bytes - 1) / copy_bytes)));
  struct Ops {
    const void *W, *s, *z;
  };
  std::vector<Ops> ops(R, Ops{W, scales, zp});
  void* pool = nullptr;
  cudaStream_t ts = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  bool ok = cudaStreamCreateWithFlags(&ts, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess &&
            (R == 1 || cudaMalloc(&pool, copy_bytes * (R - 1)) == cudaSuccess);
  for (int r = 1; ok && r < R; ++r) {
    char* base = static_cast<char*>(pool) + copy_bytes * (r - 1);
    ops[r].W = base;
    ops[r].s = base + up(w_bytes);
    ops[r].z = int_zp ? base + up(w_bytes) + up(s_bytes) : zp;  // NVFP4: the global scale
    ok = cudaMemcpyAsync(base, W, w_bytes, cudaMemcpyDeviceToDevice, ts) == cudaSuccess &&
         cudaMemcpyAsync(base + up(w_bytes), scales, s_bytes, cudaMemcpyDeviceToDevice, ts) == cudaSuccess &&
         (!int_zp || cudaMemcpyAsync(base + up(w_bytes) + up(s_bytes), zp, z_bytes,
                                     cudaMemcpyDeviceToDevice, ts) == cudaSuccess);
  }
  if (ok) ok = cudaStreamSynchronize(ts) == cudaSuccess;
  rc = ok ? BSGEMV_OK : BSGEMV_ERR_CUDA;

  const Cand keep = {plan->split, plan->cluster, plan->ctas_override, plan->rows_override,
                     plan->stages_override};
  float best_us = -1.f;
  Cand best = keep;
  int best_per_sm = 0;
  struct Key {
    int rows, cluster, ctas, stages;
    bool operator==(const Key& o) const {
      return rows == o.rows && cluster == o.cluster && ctas == o.ctas && stages == o.stages;
    }
  };
  std::vector<Key> seen;  // geometries measured
  const int calls = R * reps;
  // Put candidate c in place; false if the plan cannot run it.
  auto apply = [&](const Cand& c) {
    plan->split = c.split;
    plan->cluster = c.cluster;
    plan->ctas_override = c.ctas;
    plan->rows_override = c.rows;
    plan->stages_override = c.stages;
    return rebuild_geometry(plan) == BSGEMV_OK;
  };
  // Time the plan's current geometry on calls of m rows (back to back, cold weights): µs per
  // call in *us.
  auto time_rows = [&](int m, float* us) {
    // one eager call first: kernel attributes (shared-memory size) are set outside the capture
    if ((rc = prepare_params(plan, A, W, scales, zp, y, m)) != BSGEMV_OK) return;
    if ((rc = launch(plan, ts)) != BSGEMV_OK) return;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    if (cudaStreamBeginCapture(ts, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      rc = BSGEMV_ERR_CUDA;
      return;
    }
    for (int i = 0; i < calls && rc == BSGEMV_OK; ++i) {
      const Ops& o = ops[i % R];
      rc = prepare_params(plan, A, o.W, o.s, o.z, y, m);
      if (rc == BSGEMV_OK) rc = launch(plan, ts);
    }
    const bool captured = cudaStreamEndCapture(ts, &graph) == cudaSuccess;
    if (rc == BSGEMV_OK && !captured) rc = BSGEMV_ERR_CUDA;
    if (rc == BSGEMV_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) rc = BSGEMV_ERR_CUDA;
    float ms = 0.f;
    if (rc == BSGEMV_OK &&
        (cudaGraphLaunch(exec, ts) != cudaSuccess ||  // warm-up
         cudaEventRecord(e0, ts) != cudaSuccess || cudaGraphLaunch(exec, ts) != cudaSuccess ||
         cudaGraphLaunch(exec, ts) != cudaSuccess || cudaEventRecord(e1, ts) != cudaSuccess ||
         cudaEventSynchronize(e1) != cudaSuccess || cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
      rc = BSGEMV_ERR_CUDA;
    if (exec) cudaGraphExecDestroy(exec);
    if (graph) cudaGraphDestroy(graph);
    *us = ms * 1000.f / (2.f * calls);
  };
  // The objective: calls of M rows plus, when M > 1, calls of one row, each timed in a graph of
  // their own -- the geometry serves every M of the plan, and one tuned on its largest M alone
  // can be slower on the smallest (calls of the two sizes alternating in one graph instead
  // favour geometries whose ring is the same at every M: a ring fixed at 2 stages won there on
  // the NVFP4 lm_head, 4 % slower than the automatic one at each M alone).
  auto time_current = [&](float* us) {
    time_rows(M, us);
    if (rc != BSGEMV_OK || M == 1) return;
    float u1 = 0.f;
    time_rows(1, &u1);
    *us += u1;
  };
  // Time candidate c; a candidate that cannot run or repeats a measured geometry is skipped.
  // Keeps the fastest: another geometry must beat the automatic choice (measured first) by
  // more than 1 %.
  auto measure = [&](const Cand& c) {
    if (!apply(c)) return;  // this candidate does not fit
    const bsgemv_geometry& pg = plan->geo.pub;
    const Key key{pg.rows_per_tile, pg.cluster, pg.ctas, pg.stages};
    if (std::find(seen.begin(), seen.end(), key) != seen.end()) return;
    seen.push_back(key);
    float us = 0.f;
    time_current(&us);
    if (rc != BSGEMV_OK) return;
    if (best_us < 0.f || us < 0.99f * best_us) {
      best_us = us;
      best = c;
      best_per_sm = pg.ctas_per_sm;
    }
  };
  for (size_t ci = 0; rc == BSGEMV_OK && ci < cands.size(); ++ci) measure(cands[ci]);
  if (rc == BSGEMV_OK && best_us >= 0.f) {
    const Cand base = best;
    const int base_per_sm = best_per_sm;
    for (int st : kRingDepths) {
      if (rc != BSGEMV_OK) break;
      Cand c = base;
      c.stages = st;
      // a ring that only fits at fewer CTAs per SM changes the residency as well: not a candidate
      if (!apply(c) || plan->geo.pub.ctas_per_sm != base_per_sm) continue;
      measure(c);
    }
  }
  // Confirmation: a winner other than the automatic choice is timed again against it, in turn,
  // twice each, and kept only if it is still more than 1 % faster (one timing of a few tens of
  // calls can be off by more than that).
  const Cand& automatic = cands[0];
  const bool other = best.split != automatic.split || best.cluster != automatic.cluster ||
                     best.ctas != automatic.ctas || best.rows != automatic.rows ||
                     best.stages != automatic.stages;
  if (rc == BSGEMV_OK && best_us >= 0.f && other) {
    float t_auto = 0.f, t_best = 0.f;
    int pairs = 0;
    for (int r = 0; r < 2 && rc == BSGEMV_OK; ++r) {
      float ua = 0.f, ub = 0.f;
      if (!apply(automatic)) break;
      time_current(&ua);
      if (rc != BSGEMV_OK || !apply(best)) break;
      time_current(&ub);
      if (rc != BSGEMV_OK) break;
      t_auto += ua;
      t_best += ub;
      ++pairs;
    }
    if (rc == BSGEMV_OK && !(pairs == 2 && t_best < 0.99f * t_auto)) best = automatic;
  }
  if (rc != BSGEMV_OK) cudaGetLastError();
  if (ts) {
    cudaStreamSynchronize(ts);
    cudaStreamDestroy(ts);
  }
  if (pool) cudaFree(pool);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  // the fastest candidate (or, after an error, the settings the plan had)
  if (rc != BSGEMV_OK || best_us < 0.f) best = keep;
  plan->split = best.split;
  plan->cluster = best.cluster;
  plan->ctas_override = best.ctas;
  plan->rows_override = best.rows;
  plan->stages_override = best.stages;
  const int rc2 = rebuild_geometry(plan);
  if (rc != BSGEMV_OK) return rc;
  if (best_us < 0.f) return BSGEMV_ERR_UNSUPPORTED;
  return rc2;
}

int bsgemv_plan_describe(bsgemv_plan_t plan, bsgemv_geometry* g) {
  if (plan == nullptr || g == nullptr) return BSGEMV_ERR_INVALID_ARG;
  *g = plan->geo.pub;
  return BSGEMV_OK;
}

int bsgemv_plan_set_test_fault(bsgemv_plan_t plan, int skip_stage, int64_t wait_ns) {
  if (plan == nullptr || skip_stage < -1 || wait_ns < 0) return BSGEMV_ERR_INVALID_ARG;
  plan->fault_skip = skip_stage;
  plan->fault_wait_ns = static_cast<uint64_t>(wait_ns);
  return BSGEMV_OK;
}

int bsgemv_device_status(bsgemv_plan_t plan, void* stream) {
  unsigned* err = nullptr;
  if (plan != nullptr) {
    err = plan->err;
    if (err == nullptr) return BSGEMV_ERR_CUDA;  // no workspace (a failed clear)
  } else {
    const int rc = bsg::noalloc_error_word(&err);  // bsgemv_run_noalloc's, current device
    if (rc != BSGEMV_OK) return rc;
  }
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  unsigned word = 0;
  if (cudaMemcpy(&word, err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  if (word != 0) {
    const unsigned zero = 0;
    cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    return BSGEMV_ERR_DEVICE_TIMEOUT;
  }
  return BSGEMV_OK;
}

}  // extern "C"
