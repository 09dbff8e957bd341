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
// (kScratchBytes, about 7.6 MiB) until the process exits.  Its device address is looked up on
// the first call made with a device current, and again on the first call after that device's
// context changed (a device reset ends the context the address belonged to); such a first call
// should happen before any stream capture.  All calls on a device share the one array: two calls
// that overlap on the GPU (different streams, or different host threads) race on it and give
// wrong results, so callers serialise them.  Each call clears the arrival counters it uses
// before its kernel runs; the partial sums need no clearing (each is written before it is
// read).  The error word is not cleared by a call: a bounded wait that ran out stays recorded
// until bsgemv_device_status(NULL, stream) reads and clears it.
//
// Every call runs the geometry of a plan sized for 16 rows, whatever its M, so that a row comes
// out bit-identical for every M (the summation order of a row is fixed by the geometry), and
// equal to what bsgemv_plan(..., max_M = 16) + bsgemv_run gives.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "bsgemv_internal.h"

namespace {

// Largest problem the fixed scratch area serves: up to kMaxCtas persistent CTAs (the three per SM
// of a geometry for 16 rows on a 152-SM GB300 fit) and N <= kMaxN output columns (kMaxTiles
// tiles of 64 columns, or half as many of 128).
constexpr int kMaxCtas = 480;
constexpr int64_t kMaxN = 524288;
constexpr int kMaxTiles = static_cast<int>(kMaxN / bsg::kBoxRows);
// one warp's slot: two n8 tiles of two halves
constexpr int kMaxSlotFloats = bsg::kMaxHalves * 2 * 32 * 4;
constexpr size_t kHeaderBytes = 256;        // error word, padded
constexpr size_t kCounterBytes = size_t(kMaxTiles) * bsg::kConsumerWarps * sizeof(unsigned);
constexpr size_t kPartialBytes =
    size_t(kMaxCtas) * 2 * bsg::kConsumerWarps * kMaxSlotFloats * sizeof(float);
constexpr size_t kScratchBytes = kHeaderBytes + kCounterBytes + kPartialBytes;

// [error word][arrival counters][partial sums]
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kRows = 16;  // the geometry's max_M, for every call

// Per device: the context the scratch address was looked up under, and the address.
struct ScratchRecord {
  std::atomic<uint64_t> ctx{0};
  std::atomic<void*> addr{nullptr};
};
ScratchRecord g_scratch[bsg::kMaxDevices];
std::mutex g_setup_mutex;

// Device address of the scratch array for the current device and context (looked up once per
// device and context, with that device current).
int scratch_address(unsigned char** out) {
  int dev = -1;
  uint64_t ctx = 0;
  if (!bsg::current_device_context(&dev, &ctx)) return BSGEMV_ERR_CUDA;
  ScratchRecord& r = g_scratch[dev];
  void* p = r.addr.load(std::memory_order_acquire);
  if (p == nullptr || r.ctx.load(std::memory_order_acquire) != ctx) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = r.addr.load(std::memory_order_acquire);
    if (p == nullptr || r.ctx.load(std::memory_order_acquire) != ctx) {
      p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return BSGEMV_ERR_CUDA;
      }
      r.addr.store(nullptr, std::memory_order_release);
      r.ctx.store(ctx, std::memory_order_release);
      r.addr.store(p, std::memory_order_release);
    }
  }
  *out = static_cast<unsigned char*>(p);
  return BSGEMV_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace bsg {

// The no-allocation path's error word on the current device (bsgemv_device_status(NULL, ...)).
int noalloc_error_word(unsigned** out) {
  unsigned char* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != BSGEMV_OK) return rc;
  *out = reinterpret_cast<unsigned*>(scratch);
  return BSGEMV_OK;
}

}  // namespace bsg

extern "C" int bsgemv_run_noalloc(int format, int block_size, int has_zp, int64_t N, int64_t K,
                                  const void* A, const void* W, const void* scales,
                                  const void* zp, void* y, int M, void* stream) {
  // The problem: same rules as bsgemv_plan with max_M = 16.
  if (M < 1 || M > kRows) return BSGEMV_ERR_INVALID_ARG;
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
  int rc = bsg::compute_geometry(format, block_size, has_zp, N, K, kRows, sms, 0, 0,
                                 BSGEMV_SPLIT_AUTO, 0, &g, M);
  if (rc != BSGEMV_OK) return rc;
  if (N > kMaxN || g.pub.ctas > kMaxCtas || g.pub.tiles > kMaxTiles ||
      g.slot_floats > kMaxSlotFloats)
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
  rc = scratch_address(&scratch);
  if (rc != BSGEMV_OK) return rc;
  unsigned* err = reinterpret_cast<unsigned*>(scratch);
  unsigned* counters = reinterpret_cast<unsigned*>(scratch + kHeaderBytes);
  float* partials = reinterpret_cast<float*>(scratch + kHeaderBytes + kCounterBytes);

  bsg::OperandMaps maps;
  rc = bsg::encode_maps(g, W, scales, zp, &maps);
  if (rc != BSGEMV_OK) return rc;
  bsg::KParams k;
  bsg::fill_params(g, maps, A, W, scales, zp, y, M, partials, counters, err, &k);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // clear the arrival counters this call uses (stream-ordered, no allocation); the error word
  // keeps what earlier calls recorded until it is read
  if (cudaMemsetAsync(counters, 0, size_t(g.pub.tiles) * bsg::kConsumerWarps * sizeof(unsigned),
                      s) != cudaSuccess)
    return BSGEMV_ERR_CUDA;
  return bsg::launch_gemv(g, k, s);
}
