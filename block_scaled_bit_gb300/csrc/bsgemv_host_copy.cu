// bsgemv_host_copy.cu -- copies between pinned host memory and device memory by a kernel, for
// bsgemv_run_host / bsgemv_run_host_async: the activations of a call into the plan's staging
// buffer (the GEMV writes the outputs into the host buffer itself).  A kernel in the stream
// instead of a copy-engine transfer: consecutive kernels overlap their start-up through
// programmatic dependent launch, while each copy-engine transfer between kernels costs a few
// microseconds of its own latency.  The host buffer is read or written through its device mapping (pinned host
// memory is addressable from the GPU under unified addressing).
#include <cuda_runtime.h>

#include <cstdint>

#include "bsgemv_internal.h"

namespace {

__global__ void __launch_bounds__(256) host_copy_kernel(const uint4* __restrict__ src,
                                                       uint4* __restrict__ dst, int64_t n16,
                                                       const uint8_t* __restrict__ src_tail,
                                                       uint8_t* __restrict__ dst_tail, int tail) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the previous kernel in the stream may produce `src` or still read `dst`
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride)
    dst[i] = src[i];
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail)
    dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

}  // namespace

namespace bsg {

int launch_host_copy(void* dst, const void* src, size_t bytes, int sm_count, cudaStream_t s) {
  if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) % 16 != 0)
    return BSGEMV_ERR_MISALIGNED;
  const int64_t n16 = static_cast<int64_t>(bytes / 16);
  const int tail = static_cast<int>(bytes % 16);
  int64_t blocks = (n16 + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > int64_t(4) * sm_count) blocks = int64_t(4) * sm_count;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint8_t* st = static_cast<const uint8_t*>(src) + n16 * 16;
  uint8_t* dt = static_cast<uint8_t*>(dst) + n16 * 16;
  if (cudaLaunchKernelEx(&cfg, host_copy_kernel, static_cast<const uint4*>(src),
                         static_cast<uint4*>(dst), n16, st, dt, tail) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  return BSGEMV_OK;
}

}  // namespace bsg
