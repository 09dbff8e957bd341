// Stand-ins for the device-code entry points that the host-only sanitizer build links against:
// the kernels themselves are not built into that program (it runs without a GPU), so every
// launcher reports a CUDA error, which the host code must pass on without touching memory.
#include "../../block_scaled_bit_gb300/csrc/bsgemv_internal.h"

namespace bsg {

#define BSG_STUB_MTH(name) \
  int name(const KParams&, int, int, bool, int, int, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }
BSG_STUB_MTH(launch_int4_f16)
BSG_STUB_MTH(launch_int4_bf16)
BSG_STUB_MTH(launch_int8_f16)
BSG_STUB_MTH(launch_int8_bf16)
#undef BSG_STUB_MTH
#define BSG_STUB_MT(name) \
  int name(const KParams&, int, bool, int, int, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }
BSG_STUB_MT(launch_int4_f16_wide)
BSG_STUB_MT(launch_int4_bf16_wide)
BSG_STUB_MT(launch_int8_f16_wide)
BSG_STUB_MT(launch_int8_bf16_wide)
BSG_STUB_MT(launch_int4_f16_tall)
BSG_STUB_MT(launch_int4_bf16_tall)
BSG_STUB_MT(launch_int8_f16_tall)
BSG_STUB_MT(launch_int8_bf16_tall)
#undef BSG_STUB_MT
int launch_fp8(const KParams&, int, int, bool, int, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }
int launch_nvfp4(const KParams&, int, int, bool, int, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }
int launch_fp8_tall(const KParams&, int, bool, int, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }
int launch_nvfp4_tall(const KParams&, int, bool, int, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }
#define BSG_STUB_CC(name) \
  int name(const KParams&, bool, int, int, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }
BSG_STUB_CC(launch_cc_int4_f16)
BSG_STUB_CC(launch_cc_int4_bf16)
BSG_STUB_CC(launch_cc_int8_f16)
BSG_STUB_CC(launch_cc_int8_bf16)
#undef BSG_STUB_CC
int launch_cc_fp8(const KParams&, bool, int, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }
int launch_cc_nvfp4(const KParams&, bool, int, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }
int launch_debug_dequant(int, bool, bool, int, int64_t, int64_t, const uint8_t*, const uint8_t*,
                         const uint8_t*, const float*, float*, cudaStream_t) {
  return BSGEMV_ERR_CUDA;
}
int noalloc_error_word(unsigned**) { return BSGEMV_ERR_CUDA; }
int launch_host_copy(void*, const void*, size_t, int, cudaStream_t) { return BSGEMV_ERR_CUDA; }

}  // namespace bsg
