// bsgemv_host.cpp -- host code shared by the planned entry points (bsgemv_api.cu) and the
// allocation-free one (bsgemv_noalloc.cu): TMA tensor maps of a call's operands, the kernel
// parameters, and the dispatch to one kernel instantiation.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "bsgemv_internal.h"

namespace bsg {

namespace {

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

struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns& ctx_fns() {
  static CtxFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return f;
}

// 2D uint8 tensor [rows][row_bytes] with row pitch `pitch`, box [box_rows][box_bytes].
int encode_u8(CUtensorMap* tm, const void* base, uint64_t row_bytes, uint64_t rows,
              uint64_t pitch, uint32_t box_bytes, uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return BSGEMV_ERR_CUDA;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

}  // namespace

bool current_device_context(int* dev, uint64_t* ctx_id) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (*dev < 0 || *dev >= kMaxDevices) return false;
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return false;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return false;
  if (ctx == nullptr) {
    // a thread that has not used the device yet: the runtime binds its primary context on the
    // first call that needs one
    if (cudaFree(nullptr) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  }
  unsigned long long id = 0;
  if (f.get_id(ctx, &id) != CUDA_SUCCESS) return false;
  *ctx_id = id;
  return true;
}

int encode_maps(const Geometry& g, const void* W, const void* scales, const void* zp,
                OperandMaps* m) {
  std::memset(m, 0, sizeof(*m));
  const int64_t row_bytes = (g.fmt == kInt4 || g.fmt == kNvfp4) ? g.K / 2 : g.K;
  int rc = encode_u8(&m->tm_w, W, row_bytes, g.N, row_bytes, kBoxRowBytes, kBoxRows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != BSGEMV_OK) return rc;
  const bool int_zp = (g.fmt == kInt4 || g.fmt == kInt8) && g.has_zp;
  m->side_tma = g.side_bytes > 0 && aligned16(scales) && (!int_zp || aligned16(zp));
  if (m->side_tma) {
    rc = encode_u8(&m->tm_s, scales, g.scale_pitch, g.N, g.scale_pitch, kSideScaleBytes,
                   g.pub.rows_per_tile, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc == BSGEMV_OK && int_zp)
      rc = encode_u8(&m->tm_z, zp, g.zp_pitch, g.N, g.zp_pitch, g.zbox_bytes, g.pub.rows_per_tile,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc != BSGEMV_OK) m->side_tma = false;  // fall back to direct reads
  }
  return BSGEMV_OK;
}

void fill_params(const Geometry& g, const OperandMaps& m, const void* A, const void* W,
                 const void* scales, const void* zp, void* y, int M, float* partials,
                 unsigned* counters, unsigned* err, KParams* k) {
  std::memset(k, 0, sizeof(*k));
  const bool int_fmt = (g.fmt == kInt4 || g.fmt == kInt8);
  k->tm_w = m.tm_w;
  k->tm_s = m.tm_s;
  k->tm_z = m.tm_z;
  k->A = static_cast<const uint16_t*>(A);
  k->W = static_cast<const uint8_t*>(W);
  k->scales = static_cast<const uint8_t*>(scales);
  k->zp = int_fmt ? static_cast<const uint8_t*>(zp) : nullptr;
  k->gscale = (g.fmt == kNvfp4) ? static_cast<const float*>(zp) : nullptr;
  k->y = y;
  k->partials = partials;
  k->counters = counters;
  k->err = err;
  k->N = g.N;
  k->K = g.K;
  k->total_stages = g.pub.total_stages;
  k->spt = static_cast<int>(g.pub.stages_per_tile);
  k->M = M;
  k->nb_s = g.nb_s;
  int l2 = 0;
  while ((1 << l2) < g.block_size) ++l2;
  k->bs_log2 = l2;
  k->scale_pitch = g.scale_pitch;
  k->zp_pitch = g.zp_pitch;
  k->stages = g.pub.stages;
  k->act_off = g.act_off;
  k->act_bytes = g.act_bytes;
  k->side_tma = m.side_tma ? 1 : 0;
  k->side_off = g.side_off;
  k->side_bytes = g.side_bytes;
  k->side_slots = g.side_slots;
  k->side_tx =
      g.pub.rows_per_tile * (kSideScaleBytes + ((int_fmt && g.has_zp) ? g.zbox_bytes : 0));
  k->zbox_bytes = g.zbox_bytes;
  k->rs_log2 = g.rs_log2;
  k->bar_off = g.bar_off;
  k->slot_floats = g.slot_floats;
  k->cluster = g.pub.cluster;
  k->red_off = g.red_off;
  k->red_tq = g.red_tq;
  k->wait_ns = kDefaultWaitNs;
  k->skip_stage = -1;
}

int launch_gemv(const Geometry& g, const KParams& k, cudaStream_t s) {
  if (g.pub.variant == BSGEMV_VARIANT_CUDA_CORE) {
    if (k.M > 8) return BSGEMV_ERR_UNSUPPORTED;
    const int bm = block_mode(g.fmt, g.block_size);
    const int ctas = g.pub.ctas, smem = g.pub.smem_bytes;
    switch (g.fmt) {
      case kInt4:
        return g.bf16 ? launch_cc_int4_bf16(k, g.has_zp, bm, ctas, smem, s)
                      : launch_cc_int4_f16(k, g.has_zp, bm, ctas, smem, s);
      case kInt8:
        return g.bf16 ? launch_cc_int8_bf16(k, g.has_zp, bm, ctas, smem, s)
                      : launch_cc_int8_f16(k, g.has_zp, bm, ctas, smem, s);
      case kFp8: return launch_cc_fp8(k, g.bf16, ctas, smem, s);
      case kNvfp4: return launch_cc_nvfp4(k, g.bf16, ctas, smem, s);
    }
    return BSGEMV_ERR_INVALID_ARG;
  }
  // n8 activation tiles per call: calls with more than 16 rows run the tile count their plan
  // was sized for (3 or 4)
  const int mt = k.M > 16 ? g.mt_max : k.M > 8 ? 2 : 1;
  const int ctas = g.pub.ctas, smem = g.pub.smem_bytes;
  const int bm = block_mode(g.fmt, g.block_size);
  switch (g.fmt) {
    case kInt4:
      return g.bf16 ? launch_int4_bf16(k, mt, g.halves, g.has_zp, bm, ctas, smem, s)
                    : launch_int4_f16(k, mt, g.halves, g.has_zp, bm, ctas, smem, s);
    case kInt8:
      return g.bf16 ? launch_int8_bf16(k, mt, g.halves, g.has_zp, bm, ctas, smem, s)
                    : launch_int8_f16(k, mt, g.halves, g.has_zp, bm, ctas, smem, s);
    case kFp8:
      return launch_fp8(k, mt, g.halves, g.bf16, ctas, smem, s);
    case kNvfp4:
      return launch_nvfp4(k, mt, g.halves, g.bf16, ctas, smem, s);
  }
  return BSGEMV_ERR_INVALID_ARG;
}

}  // namespace bsg
