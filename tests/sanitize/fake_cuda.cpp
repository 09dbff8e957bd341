// A fake CUDA runtime for host-only tests of the planned entry points (plan, run, run_host,
// set_override, autotune, device_status): one sm_103 device with 152 SMs whose "device memory"
// comes from the host heap, streams / events / graphs as plain objects, and kernel launchers
// that check the pointers they are handed and charge a test-chosen time per launch to a fake
// clock.  Linked instead of libcudart (every runtime call the library makes is defined here), so
// the library's host code runs under the sanitizers exactly as it runs on a GPU, with failures
// injected where the test asks (a cudaMalloc or cudaMemset that fails).
#include "fake_cuda.h"

#include <cudaTypedefs.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>

namespace fake {

State g;

namespace {
std::map<uintptr_t, size_t> live;    // device allocations: base -> bytes
std::map<uintptr_t, size_t> pinned;  // host ranges registered as pinned (mapped)

bool inside(const std::map<uintptr_t, size_t>& m, const void* p, size_t n) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  auto it = m.upper_bound(a);
  if (it == m.begin()) return false;
  --it;
  return a >= it->first && a + n <= it->first + it->second;
}

struct Graph {
  double cost_us;
};
struct Event {
  double t_us;
};
int stream_obj, default_ctx_obj;
}  // namespace

bool device_range(const void* p, size_t n) { return inside(live, p, n); }
bool pinned_range(const void* p, size_t n) { return inside(pinned, p, n); }
size_t live_allocations() { return live.size(); }
void register_pinned(const void* p, size_t n) { pinned[reinterpret_cast<uintptr_t>(p)] = n; }

void* device_alloc(size_t n) {
  void* p = nullptr;
  return cudaMalloc(&p, n) == cudaSuccess ? p : nullptr;
}

void charge(const Launch& l) {
  ++g.launches;
  g.last = l;
  const double us = g.cost ? g.cost(l) : 1.0;
  if (g.capturing) g.capture_cost += us;
  else g.clock_us += us;
}

void violation(const char* what) {
  ++g.violations;
  std::fprintf(stderr, "fake device: %s\n", what);
}

}  // namespace fake

using fake::g;

extern "C" {

cudaError_t cudaGetDevice(int* device) {
  *device = g.current_device;
  return cudaSuccess;
}

cudaError_t cudaDeviceGetAttribute(int* value, enum cudaDeviceAttr attr, int device) {
  if (device != 0) return cudaErrorInvalidDevice;
  switch (attr) {
    case cudaDevAttrComputeCapabilityMajor: *value = 10; break;
    case cudaDevAttrComputeCapabilityMinor: *value = 3; break;
    case cudaDevAttrMultiProcessorCount: *value = 152; break;
    case cudaDevAttrL2CacheSize: *value = 8 * 1024 * 1024; break;  // small: few weight copies
    default: *value = 0;
  }
  return cudaSuccess;
}

cudaError_t cudaMalloc(void** p, size_t size) {
  if (g.fail_malloc > 0 && --g.fail_malloc == 0) {
    *p = nullptr;
    return cudaErrorMemoryAllocation;
  }
  const size_t n = (size + 255) / 256 * 256;
  *p = std::aligned_alloc(256, n == 0 ? 256 : n);
  if (*p == nullptr) return cudaErrorMemoryAllocation;
  fake::live[reinterpret_cast<uintptr_t>(*p)] = size;
  return cudaSuccess;
}

cudaError_t cudaFree(void* p) {
  if (p == nullptr) return cudaSuccess;
  auto it = fake::live.find(reinterpret_cast<uintptr_t>(p));
  if (it == fake::live.end()) {
    fake::violation("cudaFree of a pointer that is not a live allocation");
    return cudaErrorInvalidValue;
  }
  fake::live.erase(it);
  std::free(p);
  return cudaSuccess;
}

cudaError_t cudaMemset(void* p, int v, size_t n) {
  if (g.memset_broken || (g.fail_memset > 0 && --g.fail_memset == 0)) return cudaErrorUnknown;
  if (!fake::device_range(p, n)) {
    fake::violation("cudaMemset outside a live allocation");
    return cudaErrorInvalidValue;
  }
  std::memset(p, v, n);
  return cudaSuccess;
}

cudaError_t cudaMemcpy(void* dst, const void* src, size_t n, enum cudaMemcpyKind) {
  std::memcpy(dst, src, n);
  return cudaSuccess;
}

cudaError_t cudaMemcpyAsync(void* dst, const void* src, size_t n, enum cudaMemcpyKind kind,
                            cudaStream_t) {
  ++g.memcpy_calls;
  return cudaMemcpy(dst, src, n, kind);
}

cudaError_t cudaPointerGetAttributes(struct cudaPointerAttributes* a, const void* p) {
  std::memset(a, 0, sizeof(*a));
  if (fake::device_range(p, 1)) {
    a->type = cudaMemoryTypeDevice;
    a->devicePointer = const_cast<void*>(p);
  } else if (fake::pinned_range(p, 1)) {
    a->type = cudaMemoryTypeHost;
    a->devicePointer = const_cast<void*>(p);  // mapped at the same address (unified addressing)
    a->hostPointer = const_cast<void*>(p);
  } else {
    a->type = cudaMemoryTypeUnregistered;
  }
  return cudaSuccess;
}

cudaError_t cudaDeviceSynchronize(void) { return cudaSuccess; }
cudaError_t cudaStreamSynchronize(cudaStream_t) { return cudaSuccess; }
cudaError_t cudaGetLastError(void) { return cudaSuccess; }

cudaError_t cudaStreamCreateWithFlags(cudaStream_t* s, unsigned int) {
  *s = reinterpret_cast<cudaStream_t>(&fake::stream_obj);
  return cudaSuccess;
}
cudaError_t cudaStreamDestroy(cudaStream_t) { return cudaSuccess; }

cudaError_t cudaEventCreate(cudaEvent_t* e) {
  *e = reinterpret_cast<cudaEvent_t>(new fake::Event{0.0});
  return cudaSuccess;
}
cudaError_t cudaEventDestroy(cudaEvent_t e) {
  delete reinterpret_cast<fake::Event*>(e);
  return cudaSuccess;
}
cudaError_t cudaEventRecord(cudaEvent_t e, cudaStream_t) {
  reinterpret_cast<fake::Event*>(e)->t_us = g.clock_us;
  return cudaSuccess;
}
cudaError_t cudaEventSynchronize(cudaEvent_t) { return cudaSuccess; }
cudaError_t cudaEventElapsedTime(float* ms, cudaEvent_t a, cudaEvent_t b) {
  *ms = static_cast<float>((reinterpret_cast<fake::Event*>(b)->t_us -
                            reinterpret_cast<fake::Event*>(a)->t_us) / 1000.0);
  return cudaSuccess;
}

cudaError_t cudaStreamBeginCapture(cudaStream_t, enum cudaStreamCaptureMode) {
  if (g.capturing) return cudaErrorIllegalState;
  g.capturing = true;
  g.capture_cost = 0.0;
  ++g.capture_sessions;
  return cudaSuccess;
}
cudaError_t cudaStreamEndCapture(cudaStream_t, cudaGraph_t* graph) {
  if (!g.capturing) return cudaErrorIllegalState;
  g.capturing = false;
  *graph = reinterpret_cast<cudaGraph_t>(new fake::Graph{g.capture_cost});
  return cudaSuccess;
}
cudaError_t cudaGraphInstantiate(cudaGraphExec_t* exec, cudaGraph_t graph, unsigned long long) {
  *exec = reinterpret_cast<cudaGraphExec_t>(
      new fake::Graph{reinterpret_cast<fake::Graph*>(graph)->cost_us});
  return cudaSuccess;
}
cudaError_t cudaGraphLaunch(cudaGraphExec_t exec, cudaStream_t) {
  g.clock_us += reinterpret_cast<fake::Graph*>(exec)->cost_us;
  return cudaSuccess;
}
cudaError_t cudaGraphDestroy(cudaGraph_t graph) {
  delete reinterpret_cast<fake::Graph*>(graph);
  return cudaSuccess;
}
cudaError_t cudaGraphExecDestroy(cudaGraphExec_t exec) {
  delete reinterpret_cast<fake::Graph*>(exec);
  return cudaSuccess;
}

}  // extern "C"

// Driver entry points the library looks up: tensor-map encoding (fills the map with a marker)
// and the current context (one context for the whole run).
namespace {
CUresult encode_tiled(CUtensorMap* tm, CUtensorMapDataType, cuuint32_t, void* base,
                      const cuuint64_t*, const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                      CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                      CUtensorMapFloatOOBfill) {
  std::memset(tm, 0, sizeof(*tm));
  std::memcpy(tm, &base, sizeof(base));
  ++g.maps_encoded;
  return CUDA_SUCCESS;
}
CUresult ctx_current(CUcontext* c) {
  *c = reinterpret_cast<CUcontext>(&fake::default_ctx_obj);
  return CUDA_SUCCESS;
}
CUresult ctx_id(CUcontext, unsigned long long* id) {
  *id = 1;
  return CUDA_SUCCESS;
}
const PFN_cuTensorMapEncodeTiled_v12000 kEncode = encode_tiled;
const PFN_cuCtxGetCurrent_v4000 kCtxCurrent = ctx_current;
const PFN_cuCtxGetId_v12000 kCtxId = ctx_id;
}  // namespace

extern "C" cudaError_t cudaGetDriverEntryPointByVersion(const char* symbol, void** fn,
                                                        unsigned int, unsigned long long,
                                                        enum cudaDriverEntryPointQueryResult* q) {
  void* p = nullptr;
  if (std::strcmp(symbol, "cuTensorMapEncodeTiled") == 0) p = reinterpret_cast<void*>(kEncode);
  if (std::strcmp(symbol, "cuCtxGetCurrent") == 0) p = reinterpret_cast<void*>(kCtxCurrent);
  if (std::strcmp(symbol, "cuCtxGetId") == 0) p = reinterpret_cast<void*>(kCtxId);
  *fn = p;
  if (q) *q = p ? cudaDriverEntryPointSuccess : cudaDriverEntryPointSymbolNotFound;
  return cudaSuccess;
}

// The kernel launchers: each checks that every pointer it is handed lies in memory the fake
// device can reach (a live allocation, or a registered pinned host range for the outputs), that
// the workspace holds the partial slots of its grid, and charges the launch to the clock.
namespace bsg {
namespace {
int gemv(const KParams& k, int mt, int halves, int ctas, int smem) {
  const size_t slots = size_t(ctas) * 2 * kConsumerWarps * size_t(k.slot_floats) * sizeof(float);
  if (!fake::device_range(k.partials, slots)) fake::violation("partial slots outside the workspace");
  if (!fake::device_range(k.err, sizeof(unsigned))) fake::violation("error word outside the workspace");
  if (!fake::device_range(k.counters, sizeof(unsigned))) fake::violation("counters outside the workspace");
  if (!fake::device_range(k.A, size_t(k.M) * k.K * 2)) fake::violation("A not in device memory");
  const size_t yb = size_t(k.M) * k.N * 2;
  if (!fake::device_range(k.y, yb) && !fake::pinned_range(k.y, yb)) fake::violation("y unreachable");
  if (smem <= 0 || smem > 232448) fake::violation("shared memory out of range");
  if (k.bias && !fake::device_range(k.bias, size_t(k.N) * 2)) fake::violation("bias unreachable");
  fake::Launch l{k.M, mt, halves, ctas, k.cluster, k.stages, k.A, k.y, k.partials, k.bias};
  fake::charge(l);
  return BSGEMV_OK;
}
}  // namespace

#define FAKE_MTH(name) \
  int name(const KParams& k, int mt, int h, bool, int, int ctas, int smem, cudaStream_t) { \
    return gemv(k, mt, h, ctas, smem); \
  }
FAKE_MTH(launch_int4_f16)
FAKE_MTH(launch_int4_bf16)
FAKE_MTH(launch_int8_f16)
FAKE_MTH(launch_int8_bf16)
#undef FAKE_MTH
int launch_fp8(const KParams& k, int mt, int h, bool, int ctas, int smem, cudaStream_t) {
  return gemv(k, mt, h, ctas, smem);
}
int launch_nvfp4(const KParams& k, int mt, int h, bool, int ctas, int smem, cudaStream_t) {
  return gemv(k, mt, h, ctas, smem);
}
#define FAKE_CC(name) \
  int name(const KParams& k, bool, int, int ctas, int smem, cudaStream_t) { \
    return gemv(k, 1, 1, ctas, smem); \
  }
FAKE_CC(launch_cc_int4_f16)
FAKE_CC(launch_cc_int4_bf16)
FAKE_CC(launch_cc_int8_f16)
FAKE_CC(launch_cc_int8_bf16)
#undef FAKE_CC
int launch_cc_fp8(const KParams& k, bool, int ctas, int smem, cudaStream_t) {
  return gemv(k, 1, 1, ctas, smem);
}
int launch_cc_nvfp4(const KParams& k, bool, int ctas, int smem, cudaStream_t) {
  return gemv(k, 1, 1, ctas, smem);
}
int launch_debug_dequant(int, bool, bool, int, int64_t, int64_t, const uint8_t*, const uint8_t*,
                         const uint8_t*, const float*, float*, cudaStream_t) {
  return BSGEMV_ERR_CUDA;
}
int noalloc_error_word(unsigned**) { return BSGEMV_ERR_CUDA; }
int launch_host_copy(void* dst, const void* src, size_t bytes, int, cudaStream_t) {
  ++g.host_copies;
  if (!fake::device_range(dst, bytes)) fake::violation("host copy into memory that is not the device's");
  if (!fake::pinned_range(src, bytes)) fake::violation("host copy from memory that is not pinned");
  std::memcpy(dst, src, bytes);
  return BSGEMV_OK;
}
}  // namespace bsg
