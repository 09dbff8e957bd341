// bsgemv_noalloc.cu -- bsgemv_run_noalloc: one GEMV call that allocates nothing.
//
// Who needs this: code that must not allocate device memory on its own -- allocator-free
// inference runtimes and embedded deployments that own all device memory up front, callers that
// run inside another framework's memory pool and may not call cudaMalloc behind its back, and
// code paths where an allocation could fail or synchronise at the wrong moment.  bsgemv_plan
// allocates the cross-CTA reduction workspace with cudaMalloc; this entry point instead uses one
// fixed scratch area that is part of the library's device image.
//
// The scratch area is the file-scope array below.  Every GPU that loads the library holds it
// (kScratchBytes, about 2.6 MiB) until the process exits.  Its device address is looked up once
// per device, on the first call made with that device current; that first call should happen
// before any stream capture.  All calls on a device share the one array: two calls that overlap
// on the GPU (different streams, or different host threads) race on it and give wrong results,
// so callers serialise them.  Each call clears the arrival counters and the error word it uses
// before its kernel runs; the partial sums need no clearing (each is written before it is read).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "bsgemv_internal.h"

namespace {

// Largest problem the fixed scratch area serves: up to kMaxCtas persistent CTAs (twice the SM
// count of a 152-SM GB300 fits) and up to kMaxTiles tiles of 64 output columns (N <= 524288).
constexpr int kMaxCtas = 320;
constexpr int kMaxTiles = 8192;
constexpr int kMaxSlotFloats = 4 * 2 * 32 * 4;  // one partial slot with two n8 tiles
constexpr size_t kHeaderBytes = 256;            // error word, padded
constexpr size_t kCounterBytes = size_t(kMaxTiles) * sizeof(unsigned);
constexpr size_t kPartialBytes = size_t(kMaxCtas) * 2 * kMaxSlotFloats * sizeof(float);
constexpr size_t kScratchBytes = kHeaderBytes + kCounterBytes + kPartialBytes;

// [error word][arrival counters][partial sums]
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of the scratch array on the current device `dev` (looked up on first use).
int scratch_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return BSGEMV_ERR_UNSUPPORTED;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return BSGEMV_ERR_CUDA;
      }
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = static_cast<unsigned char*>(p);
  return BSGEMV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" int bsgemv_run_noalloc(int format, int block_size, int has_zp, int64_t N, int64_t K,
                                  const void* A, const void* W, const void* scales,
                                  const void* zp, void* y, int M, void* stream) {
  // The problem: same rules as bsgemv_plan, with max_M = M.
  if (M < 1 || M > 16) return BSGEMV_ERR_INVALID_ARG;
  int dev = -1, sms = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_UNSUPPORTED;
  }
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return BSGEMV_ERR_UNSUPPORTED;
  bsg::Geometry g;
  int rc = bsg::compute_geometry(format, block_size, has_zp, N, K, M, sms, 0, 0, &g);
  if (rc != BSGEMV_OK) return rc;
  if (g.pub.ctas > kMaxCtas || g.pub.tiles > kMaxTiles || g.slot_floats > kMaxSlotFloats)
    return BSGEMV_ERR_SCRATCH_LIMIT;

  // The call's arguments: same rules as bsgemv_run.
  const bool int_fmt = (g.fmt == bsg::kInt4 || g.fmt == bsg::kInt8);
  if (!A || !W || !scales || !y) return BSGEMV_ERR_INVALID_ARG;
  if (g.fmt == bsg::kNvfp4 && zp == nullptr) return BSGEMV_ERR_INVALID_ARG;
  if (int_fmt && (g.has_zp != 0) != (zp != nullptr)) return BSGEMV_ERR_INVALID_ARG;
  if (g.fmt == bsg::kFp8 && zp != nullptr) return BSGEMV_ERR_INVALID_ARG;
  if (!aligned(A, 16) || !aligned(W, 16) || !aligned(y, 16)) return BSGEMV_ERR_MISALIGNED;
  if (!aligned(scales, g.scale_es)) return BSGEMV_ERR_MISALIGNED;
  if (g.fmt == bsg::kNvfp4 && !aligned(zp, 4)) return BSGEMV_ERR_MISALIGNED;

  unsigned char* scratch = nullptr;
  rc = scratch_address(dev, &scratch);
  if (rc != BSGEMV_OK) return rc;
  unsigned* err = reinterpret_cast<unsigned*>(scratch);
  unsigned* counters = reinterpret_cast<unsigned*>(scratch + kHeaderBytes);
  float* partials = reinterpret_cast<float*>(scratch + kHeaderBytes + kCounterBytes);

  bsg::KParams k{};
  auto fn = encode_fn();
  if (!fn) return BSGEMV_ERR_CUDA;
  const int64_t row_bytes = (g.fmt == bsg::kInt4 || g.fmt == bsg::kNvfp4) ? g.K / 2 : g.K;
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(g.N)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {bsg::kStageRowBytes, bsg::kRowsPerTile};
    const cuuint32_t estr[2] = {1, 1};
    if (fn(&k.tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(W), dims, strides, box,
           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return BSGEMV_ERR_CUDA;
  }
  const int scale_pitch = g.nb_s * g.scale_es;
  const int zp_pitch = (g.fmt == bsg::kInt4) ? (g.nb_s + 1) / 2 : g.nb_s;
  k.A = static_cast<const uint16_t*>(A);
  k.W = static_cast<const uint8_t*>(W);
  k.scales = static_cast<const uint8_t*>(scales);
  k.zp = int_fmt ? static_cast<const uint8_t*>(zp) : nullptr;
  k.gscale = (g.fmt == bsg::kNvfp4) ? static_cast<const float*>(zp) : nullptr;
  k.y = y;
  k.partials = partials;
  k.counters = counters;
  k.err = err;
  k.N = g.N;
  k.K = g.K;
  k.total_stages = g.pub.total_stages;
  k.spt = g.pub.stages_per_tile;
  k.M = M;
  k.nb_s = g.nb_s;
  int l2 = 0;
  while ((1 << l2) < g.block_size) ++l2;
  k.bs_log2 = l2;
  k.scale_pitch = scale_pitch;
  k.zp_pitch = zp_pitch;
  k.stages = g.pub.stages;
  k.slot_bytes = g.slot_bytes;
  k.act_off = g.act_off;
  k.sc_off = g.sc_off;
  k.zp_off = g.zp_off;
  k.act_box_bytes = g.act_box_bytes;
  k.ring_bytes = g.ring_bytes;
  k.red_off = g.red_off;
  k.bar_off = g.bar_off;
  k.tx_bytes = bsg::kRowsPerTile * bsg::kStageRowBytes;
  k.sbw = g.sbw;
  k.zbw_bytes = g.zbw_bytes;
  k.zblk = g.zblk;
  k.side_scale_tma = (scale_pitch % 16 == 0 && aligned(scales, 16)) ? 1 : 0;
  k.side_zp_tma = (int_fmt && g.has_zp && zp_pitch % 16 == 0 && aligned(zp, 16)) ? 1 : 0;
  k.slot_floats = g.slot_floats;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // clear the error word and the arrival counters this call uses (stream-ordered, no allocation)
  if (cudaMemsetAsync(scratch, 0, kHeaderBytes + size_t(g.pub.tiles) * sizeof(unsigned), s) !=
      cudaSuccess)
    return BSGEMV_ERR_CUDA;
  const int mt = M > 8 ? 2 : 1;
  const int bm = bsg::block_mode(g.fmt, g.block_size);
  switch (g.fmt) {
    case bsg::kInt4:
      return g.bf16 ? bsg::launch_int4_bf16(k, mt, g.has_zp, bm, g.pub.ctas, g.pub.smem_bytes, s)
                    : bsg::launch_int4_f16(k, mt, g.has_zp, bm, g.pub.ctas, g.pub.smem_bytes, s);
    case bsg::kInt8:
      return bsg::launch_int8(k, mt, g.bf16, g.has_zp, bm, g.pub.ctas, g.pub.smem_bytes, s);
    case bsg::kFp8:
      return bsg::launch_fp8(k, mt, g.bf16, false, bm, g.pub.ctas, g.pub.smem_bytes, s);
    case bsg::kNvfp4:
      return bsg::launch_nvfp4(k, mt, g.bf16, false, bm, g.pub.ctas, g.pub.smem_bytes, s);
  }
  return BSGEMV_ERR_INVALID_ARG;
}
