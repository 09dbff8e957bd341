// bsgemv_kernel.cuh -- the sm_103a GEMV kernel template
//
//     y[M, N] = A[M, K] . deq(W)[N, K]^T,  M <= 16
//
// Data path per CTA (one persistent CTA per ring of stages, 2 per SM):
//   warp 0, lane 0   producer: for every stage of its stream-K range, waits for a free ring slot
//                    and issues cp.async.bulk.tensor copies of the weight box [64 rows][128 B]
//                    (128-byte swizzle), the activation boxes [M][64 halves] (swizzled), and the
//                    scale / zero-point boxes, all completing on the slot's mbarrier.
//   warps 1..4       consumers: each owns 2 of the 8 16-byte chunks of every stage.  ldmatrix
//                    hands every lane one 32-bit word of each of the 16 rows of an mma tile;
//                    the word is decoded in registers to exact fp16/bf16 operand pairs
//                    ((q - zp), e4m3, or e2m1 * e4m3), fed to mma.sync.m16n8k16 with the
//                    weight as the A operand (16 output columns) and the activations as the B
//                    operand (8 rows of A per n8 tile), accumulating in fp32.  Int and FP8
//                    scales multiply the fp32 partial of each scale block; NVFP4's E4M3 scale is
//                    folded into the 16-bit operand (exact: 2 + 4 significand bits).
//   epilogue         the 4 consumer warps' partials are added in warp order through shared
//                    memory; a tile finished inside one CTA is rounded and stored, otherwise its
//                    fp32 partial goes to the plan's workspace and the last CTA to arrive adds
//                    all partials of the tile in CTA order and stores y.
//
// K permutation.  K is a reduction axis, so any permutation applied to both operands gives the
// same sum ("[CUDA] Block-scaled MatMul decode GEMV: tensor cores, packed FP4 decode and
// M-tiling", FP8 and NVFP4 tensor-core paragraphs).  Inside each 16-byte chunk lane t of a quad
// owns bytes [4t, 4t+4): 8 codes (4-bit formats, 2 mma k-steps) or 4 codes (8-bit formats,
// 1 k-step).  The mma columns {2t, 2t+1, 2t+8, 2t+9} of each k-step are mapped to physical k so
// that the register decoders' natural pairs line up; the activation fragment is permuted to
// match (see act_fragment).  Every k-step lies inside one scale block for the int and FP8
// formats (block >= 32 for int4, >= 16 for int8), except int4 with 16-element blocks, where the
// two halves of a quad use separate accumulators (SUB2).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "bsgemv_internal.h"

#define BSG_DEV __device__ __forceinline__

namespace bsg {

// Polls of mbarrier.try_wait before a wait is abandoned (each poll may suspend the thread for a
// hardware-defined interval); at least seconds, far above any legitimate stall.
constexpr uint32_t kWaitPolls = 1u << 24;

// ------------------------------------------------------------------------------ PTX wrappers
BSG_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

BSG_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

BSG_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

BSG_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

BSG_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

BSG_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: returns false (and records `code` in the error word) if the phase never
// completes.  Nothing in a correct launch waits anywhere near the limit.
BSG_DEV bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* err, unsigned code) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
  }
  atomicOr(err, code);
  return false;
}

BSG_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

BSG_DEV void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

BSG_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

BSG_DEV uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

BSG_DEV uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

BSG_DEV uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

BSG_DEV uint32_t lds16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

BSG_DEV uint32_t lds8(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}

BSG_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

BSG_DEV void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// D += A * B on the tensor cores: m16n8k16, fp16 or bf16 operands, fp32 accumulate.
template <bool BF16>
BSG_DEV void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// ------------------------------------------------------------------------------ 16-bit pairs
BSG_DEV uint32_t h2_sub(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
BSG_DEV uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b),
                      *reinterpret_cast<__half2*>(&c));
  return *reinterpret_cast<uint32_t*>(&r);
}
BSG_DEV uint32_t h2_mul(uint32_t a, uint32_t b) {
  __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
BSG_DEV uint32_t bf2_sub(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&a),
                             *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}
BSG_DEV uint32_t bf2_mul(uint32_t a, uint32_t b) {
  __nv_bfloat162 r = __hmul2(*reinterpret_cast<__nv_bfloat162*>(&a),
                             *reinterpret_cast<__nv_bfloat162*>(&b));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Two E4M3 codes (low byte -> low half) to an exact f16 pair.
BSG_DEV uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
  uint32_t d;
  const unsigned short v = static_cast<unsigned short>(two_codes);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
  return d;
}

// Two E2M1 codes in one byte (low nibble -> low half) to an exact f16 pair.
BSG_DEV uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t d;
  const unsigned short v = static_cast<unsigned short>(byte);
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(d)
      : "h"(v));
  return d;
}

// An f16 pair whose values are exact in bf16 and normal (or zero) in f16, re-encoded as a bf16
// pair: keep the sign, shift exponent and top mantissa bits into bf16 position (the value is
// then 2^-112 of the original) and scale back by 2^112, which is exact.  Used for E4M3 values
// and E2M1 x E4M3 products, which have at most 6 significand bits, so the 3 bits shifted out of
// each half are zero.
BSG_DEV uint32_t f16x2_exact_to_bf16x2(uint32_t h) {
  const uint32_t mag = ((h & 0x7FFF7FFFu) >> 3);
  const uint32_t bits = (mag & 0x0FFF0FFFu) | (h & 0x80008000u);
  return bf2_mul(bits, 0x77807780u);  // 2^112 in each bf16 half
}

// ------------------------------------------------------------------------------ decoders
// Each decoder turns the ldmatrix words of one mma row pair -- `lo` for tile row g, `hi` for row
// g + 8 -- into the A fragments of every k-step of the chunk:
//   a[s][0] = (row g,   cols 2t, 2t+1)   a[s][1] = (row g+8, cols 2t, 2t+1)
//   a[s][2] = (row g,   cols 2t+8, 2t+9) a[s][3] = (row g+8, cols 2t+8, 2t+9)
// The physical k of each half is given by phys_k below; the activation fragment follows it.

// int4: nibble j of the lane's word holds k = 8t + j.  (1024 + q) in f16 is the nibble OR-ed
// under the exponent of 1024; (1024 + 16 q) for the high nibble of a byte, which an fma with
// 1/16 brings back.  Both give the exact small integer q - zp
// ("[CUDA] MatMulNBits 8-bit: wide fp16 M=1 kernel for decode GEMVs", Description: exact
// (q - zp) in fp16).  zl = (1024 + zp) and zh = -(64 + zp) replicated in both halves.
// For bf16 the exponent of 128 holds 7 mantissa bits, so each nibble is shifted to the bottom
// first and zl = (128 + zp).
template <bool BF16>
BSG_DEV void decode_int4(uint32_t lo, uint32_t hi, uint32_t zl_lo, uint32_t zh_lo, uint32_t zl_hi,
                         uint32_t zh_hi, uint32_t (&a)[2][4]) {
  if constexpr (!BF16) {
    const uint32_t k16 = 0x2C002C00u;  // 1/16 in each f16 half
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t wl = lo >> (8 * s), wh = hi >> (8 * s);
      a[s][0] = h2_sub((wl & 0x000F000Fu) | 0x64006400u, zl_lo);
      a[s][1] = h2_sub((wh & 0x000F000Fu) | 0x64006400u, zl_hi);
      a[s][2] = h2_fma((wl & 0x00F000F0u) | 0x64006400u, k16, zh_lo);
      a[s][3] = h2_fma((wh & 0x00F000F0u) | 0x64006400u, k16, zh_hi);
    }
  } else {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t wl = lo >> (8 * s), wh = hi >> (8 * s);
      a[s][0] = bf2_sub((wl & 0x000F000Fu) | 0x43004300u, zl_lo);
      a[s][1] = bf2_sub((wh & 0x000F000Fu) | 0x43004300u, zl_hi);
      a[s][2] = bf2_sub(((wl >> 4) & 0x000F000Fu) | 0x43004300u, zl_lo);
      a[s][3] = bf2_sub(((wh >> 4) & 0x000F000Fu) | 0x43004300u, zl_hi);
    }
  }
  (void)zh_lo;
  (void)zh_hi;
}

// int8: byte j of the lane's word holds k = 4t + j.  f16: prmt places byte j under the
// exponent of 1024 (exact 1024 + q), minus (1024 + zp).  bf16 (7 mantissa bits cannot hold
// 0..255 above one exponent): 2^23 + q in fp32, minus (2^23 + zp), packed by an exact cvt.
template <bool BF16>
BSG_DEV void decode_int8(uint32_t lo, uint32_t hi, uint32_t z_lo, uint32_t z_hi,
                         uint32_t (&a)[1][4]) {
  if constexpr (!BF16) {
    a[0][0] = h2_sub(prmt(lo, 0x64646464u, 0x4140u), z_lo);
    a[0][1] = h2_sub(prmt(hi, 0x64646464u, 0x4140u), z_hi);
    a[0][2] = h2_sub(prmt(lo, 0x64646464u, 0x4342u), z_lo);
    a[0][3] = h2_sub(prmt(hi, 0x64646464u, 0x4342u), z_hi);
  } else {
    const float zf_lo = __uint_as_float(z_lo), zf_hi = __uint_as_float(z_hi);  // 2^23 + zp
    auto pair = [](uint32_t w, uint32_t sel0, uint32_t sel1, float z) -> uint32_t {
      const float x0 = __uint_as_float(prmt(w, 0x4B000000u, sel0)) - z;
      const float x1 = __uint_as_float(prmt(w, 0x4B000000u, sel1)) - z;
      uint32_t d;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(x1), "f"(x0));
      return d;
    };
    a[0][0] = pair(lo, 0x7440u, 0x7441u, zf_lo);
    a[0][1] = pair(hi, 0x7440u, 0x7441u, zf_hi);
    a[0][2] = pair(lo, 0x7442u, 0x7443u, zf_lo);
    a[0][3] = pair(hi, 0x7442u, 0x7443u, zf_hi);
  }
}

// FP8 E4M3: byte j of the lane's word holds k = 4t + j; E4M3 is exact in f16 and bf16
// (decode-GEMV page, FP8 tensor-core paragraph).
template <bool BF16>
BSG_DEV void decode_fp8(uint32_t lo, uint32_t hi, uint32_t (&a)[1][4]) {
  a[0][0] = e4m3x2_to_f16x2(lo & 0xFFFFu);
  a[0][1] = e4m3x2_to_f16x2(hi & 0xFFFFu);
  a[0][2] = e4m3x2_to_f16x2(lo >> 16);
  a[0][3] = e4m3x2_to_f16x2(hi >> 16);
  if constexpr (BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) a[0][i] = f16x2_exact_to_bf16x2(a[0][i]);
  }
}

// NVFP4: byte b of the lane's word holds k = 8t + 2b (low nibble) and 8t + 2b + 1.  The E4M3
// block scale (sc_lo for row g, sc_hi for row g+8, as f16 pairs) is folded into the decoded
// E2M1 value: exact in f16 and bf16 (decode-GEMV page, NVFP4 tensor-core paragraph).
template <bool BF16>
BSG_DEV void decode_nvfp4(uint32_t lo, uint32_t hi, uint32_t sc_lo, uint32_t sc_hi,
                          uint32_t (&a)[2][4]) {
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    a[s][0] = h2_mul(e2m1x2_to_f16x2((lo >> (16 * s)) & 0xFFu), sc_lo);
    a[s][1] = h2_mul(e2m1x2_to_f16x2((hi >> (16 * s)) & 0xFFu), sc_hi);
    a[s][2] = h2_mul(e2m1x2_to_f16x2((lo >> (16 * s + 8)) & 0xFFu), sc_lo);
    a[s][3] = h2_mul(e2m1x2_to_f16x2((hi >> (16 * s + 8)) & 0xFFu), sc_hi);
    if constexpr (BF16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) a[s][i] = f16x2_exact_to_bf16x2(a[s][i]);
    }
  }
}

// Physical k (inside the 16-byte chunk of lane t) of half h of the A fragment register pair
// rp (0: cols 2t/2t+1, 1: cols 2t+8/2t+9) in k-step s.
template <int FMT>
BSG_DEV int phys_k(int s, int rp, int h, int t) {
  if constexpr (FMT == kInt4) return 8 * t + 2 * s + rp + 4 * h;
  if constexpr (FMT == kNvfp4) return 8 * t + 2 * (2 * s + rp) + h;
  return 4 * t + 2 * rp + h;  // int8, fp8
}

// Zero-point operand constants of one row (see decode_int4 / decode_int8).
template <int FMT, bool BF16>
BSG_DEV void zp_consts(uint32_t zp, uint32_t& zl, uint32_t& zh) {
  const uint32_t rep = zp * 0x00010001u;
  if constexpr (FMT == kInt4) {
    zl = rep | (BF16 ? 0x43004300u : 0x64006400u);
    zh = (rep << 4) | 0xD400D400u;  // -(64 + zp) in f16
  } else if constexpr (!BF16) {
    zl = rep | 0x64006400u;
    zh = 0;
  } else {
    zl = __float_as_uint(8388608.0f + static_cast<float>(zp));  // 2^23 + zp
    zh = 0;
  }
}

// ------------------------------------------------------------------------------ the kernel
template <int FMT, bool BF16, int MT, bool ZP, bool SUB2>
struct Gemv {
  static constexpr bool kFour = (FMT == kInt4 || FMT == kNvfp4);
  static constexpr int kKpc = kFour ? 32 : 16;  // k per 16-byte chunk
  static constexpr int kSteps = kKpc / 16;      // mma k-steps per chunk
  static constexpr int kKc = kChunksPerStage * kKpc;
  static constexpr int kNbox = kKc / 64;        // activation boxes per stage
  static constexpr bool kFold = (FMT == kNvfp4);
  static constexpr int kSub = SUB2 ? 2 : 1;

  // ---- shared-memory layout helpers
  struct Smem {
    uint8_t* base;
    const KParams& p;
    BSG_DEV uint32_t slot(int i) const { return smem_u32(base) + i * p.slot_bytes; }
    BSG_DEV uint32_t full(int i) const { return smem_u32(base) + p.bar_off + 8 * i; }
    BSG_DEV uint32_t empty(int i) const { return smem_u32(base) + p.bar_off + 8 * (p.stages + i); }
    BSG_DEV float4* red() const { return reinterpret_cast<float4*>(base + p.red_off); }
    BSG_DEV int* flag() const { return reinterpret_cast<int*>(base + p.bar_off + 16 * p.stages); }
  };

  // ---- producer: one thread
  static BSG_DEV void produce(const KParams& p, const Smem& sm, int64_t s0, int64_t s1) {
    prefetch_tmap(&p.tm_w);
    prefetch_tmap(&p.tm_a);
    if (p.side_scale_tma) prefetch_tmap(&p.tm_s);
    if (p.side_zp_tma) prefetch_tmap(&p.tm_z);
    int64_t it = 0;
    for (int64_t s = s0; s < s1; ++s, ++it) {
      const int slot = static_cast<int>(it % p.stages);
      const uint32_t par = static_cast<uint32_t>((it / p.stages) & 1) ^ 1u;
      if (!mbar_wait(sm.empty(slot), par, p.err, kErrTimeoutEmpty)) return;
      const uint32_t full = sm.full(slot);
      mbar_arrive_expect_tx(full, static_cast<uint32_t>(p.tx_bytes));
      const int64_t tile = s / p.spt;
      const int ks = static_cast<int>(s % p.spt);
      const int row0 = static_cast<int>(tile * kRowsPerTile);
      const uint32_t dst = sm.slot(slot);
      tma_load_2d(dst, &p.tm_w, ks * kStageRowBytes, row0, full);
#pragma unroll
      for (int j = 0; j < kNbox; ++j)
        tma_load_2d(dst + p.act_off + j * p.act_box_bytes, &p.tm_a, ks * kKc + 64 * j, 0, full);
      const int blk0 = (ks * kKc) >> p.bs_log2;
      if (p.side_scale_tma) {
        const int x = (blk0 / p.sbw) * p.sbw;
        tma_load_2d(dst + p.sc_off, &p.tm_s, x, row0, full);
      }
      if (ZP && p.side_zp_tma) {
        const int xb = (blk0 / p.zblk) * p.zblk;
        tma_load_2d(dst + p.zp_off, &p.tm_z, (FMT == kInt4) ? xb / 2 : xb, row0, full);
      }
    }
  }

  // ---- consumer helpers
  // Activation B fragments of chunk c for n8 tile mt: b[st][0] = (k 2t, 2t+1), b[st][1] =
  // (k 2t+8, 2t+9) of activation row mt*8 + g, permuted like the weight (phys_k).
  static BSG_DEV void act_fragment(const KParams& p, uint32_t act_base, int c, int mt, int g, int t,
                                   uint32_t (&b)[kSteps][2]) {
    const int m = mt * 8 + g;
    if constexpr (kFour) {
      const int box = c >> 1;
      const int q = ((c & 1) << 2) + t;  // 16-byte chunk inside the 128-byte activation row
      const uint4 v = lds128(act_base + box * p.act_box_bytes + m * 128 + ((q ^ (m & 7)) << 4));
      if constexpr (FMT == kInt4) {  // pairs (8t+j, 8t+j+4)
        b[0][0] = prmt(v.x, v.z, 0x5410u);
        b[0][1] = prmt(v.x, v.z, 0x7632u);
        b[1][0] = prmt(v.y, v.w, 0x5410u);
        b[1][1] = prmt(v.y, v.w, 0x7632u);
      } else {  // nvfp4: natural pairs
        b[0][0] = v.x;
        b[0][1] = v.y;
        b[1][0] = v.z;
        b[1][1] = v.w;
      }
    } else {
      const int box = c >> 2;
      const int q = ((c & 3) << 1) + (t >> 1);
      const uint2 v = lds64(act_base + box * p.act_box_bytes + m * 128 + ((q ^ (m & 7)) << 4) +
                            ((t & 1) << 3));
      b[0][0] = v.x;
      b[0][1] = v.y;
    }
  }

  // fp32 scale of (tile row r, block blk); blk relative to the stage's scale box when staged.
  static BSG_DEV float scale_at(const KParams& p, uint32_t sc_base, int64_t tile, int r,
                                int blk, int box0) {
    if (p.side_scale_tma) {
      const int es = (FMT == kFp8) ? 4 : 2;
      const uint32_t a = sc_base + (r * p.sbw + (blk - box0)) * es;
      if constexpr (FMT == kFp8) return __uint_as_float(lds32(a));
      else return __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(a))));
    }
    if (blk >= p.nb_s) return 0.f;  // chunk past K in the ragged last stage: weight is zero
    int64_t n = tile * kRowsPerTile + r;
    if (n >= p.N) n = p.N - 1;
    const uint8_t* src = p.scales + n * p.scale_pitch;
    if constexpr (FMT == kFp8) return __ldg(reinterpret_cast<const float*>(src) + blk);
    else return __half2float(__ldg(reinterpret_cast<const __half*>(src) + blk));
  }

  static BSG_DEV uint32_t zp_at(const KParams& p, uint32_t zp_base, int64_t tile, int r, int blk,
                                int zbox0) {
    uint32_t byte;
    int rel;
    if (p.side_zp_tma) {
      rel = blk - zbox0;
      byte = lds8(zp_base + r * p.zbw_bytes + ((FMT == kInt4) ? (rel >> 1) : rel));
    } else {
      if (blk >= p.nb_s) return 0u;  // past K: the weight and activation there are zero
      int64_t n = tile * kRowsPerTile + r;
      if (n >= p.N) n = p.N - 1;
      rel = blk;
      byte = __ldg(p.zp + n * p.zp_pitch + ((FMT == kInt4) ? (blk >> 1) : blk));
    }
    if constexpr (FMT == kInt4) return (rel & 1) ? (byte >> 4) : (byte & 0xFu);
    return byte;
  }

  // NVFP4 E4M3 scale code of (tile row r, 16-block blk of the row) as a replicated f16 pair.
  static BSG_DEV uint32_t fold_scale(const KParams& p, uint32_t sc_base, int64_t tile, int r,
                                     int blk, int box0) {
    uint32_t code;
    if (p.side_scale_tma) {
      code = lds8(sc_base + r * p.sbw + (blk - box0));
    } else if (blk >= p.nb_s) {
      code = 0;  // past K
    } else {
      int64_t n = tile * kRowsPerTile + r;
      if (n >= p.N) n = p.N - 1;
      code = __ldg(p.scales + n * p.scale_pitch + blk);
    }
    return e4m3x2_to_f16x2(code * 0x0101u);
  }

  // Consume one ring slot: chunks 2*cw and 2*cw+1 of stage ks of `tile`.
  static BSG_DEV void consume_stage(const KParams& p, uint32_t slot, int64_t tile, int ks, int cw,
                                    int lane, float (&acc)[4][MT][4]) {
    const int g = lane >> 2, t = lane & 3;
    const uint32_t w_base = slot, act_base = slot + p.act_off, sc_base = slot + p.sc_off,
                   zp_base = slot + p.zp_off;
    const int blk_stage0 = (ks * kKc) >> p.bs_log2;
    const int sbox0 = (blk_stage0 / p.sbw) * p.sbw;
    const int zbox0 = ZP ? (blk_stage0 / p.zblk) * p.zblk : 0;

    float tmp[kSub][4][MT][4];
    if constexpr (!kFold) {
#pragma unroll
      for (int u = 0; u < kSub; ++u)
#pragma unroll
        for (int rg = 0; rg < 4; ++rg)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) tmp[u][rg][mt][i] = 0.f;
    }

#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * cw + cc;
      const int kchunk = ks * kKc + c * kKpc;  // first k of the chunk
      const int blk = kchunk >> p.bs_log2;     // scale block of the chunk (first half for SUB2)

      // activation fragments
      uint32_t b[MT][kSteps][2];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) act_fragment(p, act_base, c, mt, g, t, b[mt]);
      uint32_t bsub[kSub][MT][kSteps][2];
#pragma unroll
      for (int u = 0; u < kSub; ++u)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int st = 0; st < kSteps; ++st) {
            // SUB2: quad lanes t < 2 hold block blk, t >= 2 block blk + 1
            const bool keep = !SUB2 || ((t >> 1) == u);
            bsub[u][mt][st][0] = keep ? b[mt][st][0] : 0u;
            bsub[u][mt][st][1] = keep ? b[mt][st][1] : 0u;
          }

      // weight words: wv[2*rg] = row 16*rg + g, wv[2*rg + 1] = row 16*rg + g + 8
      uint32_t wv[8];
      {
        const int r0 = lane, r1 = 32 + lane;
        ldsm_x4(w_base + r0 * 128 + ((c ^ (r0 & 7)) << 4), wv[0], wv[1], wv[2], wv[3]);
        ldsm_x4(w_base + r1 * 128 + ((c ^ (r1 & 7)) << 4), wv[4], wv[5], wv[6], wv[7]);
      }

#pragma unroll
      for (int rg = 0; rg < 4; ++rg) {
        const int rlo = 16 * rg + g, rhi = rlo + 8;
        uint32_t a[kSteps][4];
        if constexpr (FMT == kInt4) {
          // zero point of the lane's own block (for SUB2: block blk + (t >> 1))
          uint32_t zl_lo, zh_lo, zl_hi, zh_hi;
          if constexpr (ZP) {
            const int zb = SUB2 ? blk + (t >> 1) : blk;
            zp_consts<FMT, BF16>(zp_at(p, zp_base, tile, rlo, zb, zbox0), zl_lo, zh_lo);
            zp_consts<FMT, BF16>(zp_at(p, zp_base, tile, rhi, zb, zbox0), zl_hi, zh_hi);
          } else {
            zp_consts<FMT, BF16>(8u, zl_lo, zh_lo);
            zl_hi = zl_lo;
            zh_hi = zh_lo;
          }
          decode_int4<BF16>(wv[2 * rg], wv[2 * rg + 1], zl_lo, zh_lo, zl_hi, zh_hi, a);
        } else if constexpr (FMT == kInt8) {
          uint32_t z_lo, z_hi, unused;
          if constexpr (ZP) {
            zp_consts<FMT, BF16>(zp_at(p, zp_base, tile, rlo, blk, zbox0), z_lo, unused);
            zp_consts<FMT, BF16>(zp_at(p, zp_base, tile, rhi, blk, zbox0), z_hi, unused);
          } else {
            zp_consts<FMT, BF16>(128u, z_lo, unused);
            z_hi = z_lo;
          }
          decode_int8<BF16>(wv[2 * rg], wv[2 * rg + 1], z_lo, z_hi, a);
        } else if constexpr (FMT == kFp8) {
          decode_fp8<BF16>(wv[2 * rg], wv[2 * rg + 1], a);
        } else {
          // NVFP4: the lane's 8 codes lie in 16-block (k_chunk + 8t) / 16
          const int fb = (kchunk >> 4) + (t >> 1);
          const uint32_t s_lo = fold_scale(p, sc_base, tile, rlo, fb, sbox0);
          const uint32_t s_hi = fold_scale(p, sc_base, tile, rhi, fb, sbox0);
          decode_nvfp4<BF16>(wv[2 * rg], wv[2 * rg + 1], s_lo, s_hi, a);
        }
#pragma unroll
        for (int st = 0; st < kSteps; ++st)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            if constexpr (kFold) {
              mma16816<BF16>(acc[rg][mt], a[st], b[mt][st][0], b[mt][st][1]);
            } else {
#pragma unroll
              for (int u = 0; u < kSub; ++u)
                mma16816<BF16>(tmp[u][rg][mt], a[st], bsub[u][mt][st][0], bsub[u][mt][st][1]);
            }
          }
      }

      // per-block fp32 scale: after every chunk, or after the pair when both chunks share it
      if constexpr (!kFold) {
        if (cc == 1 || !p.merge_pair) {
#pragma unroll
          for (int u = 0; u < kSub; ++u) {
#pragma unroll
            for (int rg = 0; rg < 4; ++rg) {
              const int rlo = 16 * rg + g, rhi = rlo + 8;
              const float s_lo = scale_at(p, sc_base, tile, rlo, blk + u, sbox0);
              const float s_hi = scale_at(p, sc_base, tile, rhi, blk + u, sbox0);
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) {
                acc[rg][mt][0] = fmaf(tmp[u][rg][mt][0], s_lo, acc[rg][mt][0]);
                acc[rg][mt][1] = fmaf(tmp[u][rg][mt][1], s_lo, acc[rg][mt][1]);
                acc[rg][mt][2] = fmaf(tmp[u][rg][mt][2], s_hi, acc[rg][mt][2]);
                acc[rg][mt][3] = fmaf(tmp[u][rg][mt][3], s_hi, acc[rg][mt][3]);
#pragma unroll
                for (int i = 0; i < 4; ++i) tmp[u][rg][mt][i] = 0.f;
              }
            }
          }
        }
      }
    }
  }

  // Store 4 fp32 results of a fragment slot (rg, mt, lane) of `tile` as rounded y.
  static BSG_DEV void store_y(const KParams& p, int64_t tile, int rg, int mt, int ln, float4 v,
                              float gs) {
    const int g = ln >> 2, t = ln & 3;
    const int64_t n0 = tile * kRowsPerTile + 16 * rg + g;
    const int m0 = mt * 8 + 2 * t;
    const float vals[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t n = n0 + ((i & 2) ? 8 : 0);
      const int m = m0 + (i & 1);
      if (m < p.M && n < p.N) {
        const float r = vals[i] * gs;
        if constexpr (BF16)
          reinterpret_cast<__nv_bfloat16*>(p.y)[m * p.N + n] = __float2bfloat16_rn(r);
        else
          reinterpret_cast<__half*>(p.y)[m * p.N + n] = __float2half_rn(r);
      }
    }
  }

  // CTA whose stream-K range contains stage x: the largest i with floor(i*T/G) <= x.
  static BSG_DEV int64_t cta_of_stage(int64_t x, int64_t T, int64_t G) {
    return ((x + 1) * G + T - 1) / T - 1;
  }

  // End of a tile segment: reduce the consumer warps, then store or publish a partial.
  static BSG_DEV void epilogue(const KParams& p, const Smem& sm, int64_t tile, bool whole,
                               int64_t s0, int cw, int lane, float (&acc)[4][MT][4], float gs) {
    const int tid = cw * 32 + lane;  // 0 .. 127
    constexpr int kSlots = 4 * MT * 32;  // float4 slots per warp
    float4* red = sm.red();
#pragma unroll
    for (int rg = 0; rg < 4; ++rg)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        red[cw * kSlots + (rg * MT + mt) * 32 + lane] =
            make_float4(acc[rg][mt][0], acc[rg][mt][1], acc[rg][mt][2], acc[rg][mt][3]);
    named_bar_sync(1, kConsumerWarps * 32);

    const int64_t G = gridDim.x, T = p.total_stages;
    const int64_t me = blockIdx.x;
    float4 sum[MT];
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      const int slot = tid + j * kConsumerWarps * 32;
      float4 v = red[slot];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) {
        const float4 u = red[w * kSlots + slot];
        v.x += u.x;
        v.y += u.y;
        v.z += u.z;
        v.w += u.w;
      }
      sum[j] = v;
    }
    if (whole) {
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        const int slot = tid + j * kConsumerWarps * 32;
        store_y(p, tile, slot / (MT * 32), (slot / 32) % MT, slot % 32, sum[j], gs);
      }
    } else {
      const int seg = (tile == (me * T / G) / p.spt) ? 0 : 1;
      float4* mine = reinterpret_cast<float4*>(p.partials) + (me * 2 + seg) * (p.slot_floats / 4);
#pragma unroll
      for (int j = 0; j < MT; ++j) __stcg(mine + tid + j * kConsumerWarps * 32, sum[j]);
      __threadfence();
      named_bar_sync(1, kConsumerWarps * 32);
      const int64_t first = cta_of_stage(tile * p.spt, T, G);
      const int64_t last = cta_of_stage((tile + 1) * p.spt - 1, T, G);
      if (tid == 0) {
        const unsigned old = atomicAdd(p.counters + tile, 1u);
        *sm.flag() = (old == static_cast<unsigned>(last - first)) ? 1 : 0;
      }
      named_bar_sync(1, kConsumerWarps * 32);
      if (*sm.flag()) {
        __threadfence();
#pragma unroll
        for (int j = 0; j < MT; ++j) {
          const int slot = tid + j * kConsumerWarps * 32;
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int64_t i = first; i <= last; ++i) {
            const int sg = (tile == (i * T / G) / p.spt) ? 0 : 1;
            const float4 u =
                __ldcg(reinterpret_cast<const float4*>(p.partials) + (i * 2 + sg) * (p.slot_floats / 4) + slot);
            v.x += u.x;
            v.y += u.y;
            v.z += u.z;
            v.w += u.w;
          }
          store_y(p, tile, slot / (MT * 32), (slot / 32) % MT, slot % 32, v, gs);
        }
        if (tid == 0) p.counters[tile] = 0u;  // every contributor has arrived: reset for reuse
      }
    }
    named_bar_sync(1, kConsumerWarps * 32);  // `red` and the flag are reused by the next segment
    (void)s0;
  }

  static BSG_DEV void consume(const KParams& p, const Smem& sm, int64_t s0, int64_t s1, int cw,
                              int lane) {
    float acc[4][MT][4];
#pragma unroll
    for (int rg = 0; rg < 4; ++rg)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[rg][mt][i] = 0.f;
    const float gs = kFold ? __ldg(p.gscale) : 1.0f;

    int64_t it = 0;
    bool ok = true;
    for (int64_t s = s0; s < s1; ++s, ++it) {
      const int slot = static_cast<int>(it % p.stages);
      const uint32_t par = static_cast<uint32_t>((it / p.stages) & 1);
      if (ok) ok = mbar_wait(sm.full(slot), par, p.err, kErrTimeoutFull);
      const int64_t tile = s / p.spt;
      const int ks = static_cast<int>(s % p.spt);
      if (ok) consume_stage(p, sm.slot(slot), tile, ks, cw, lane, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty(slot));
      if (ks == p.spt - 1 || s == s1 - 1) {
        const bool whole = (s0 <= tile * p.spt) && (s1 >= (tile + 1) * p.spt);
        epilogue(p, sm, tile, whole, s0, cw, lane, acc, gs);
#pragma unroll
        for (int rg = 0; rg < 4; ++rg)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[rg][mt][i] = 0.f;
      }
    }
  }
};

template <int FMT, bool BF16, int MT, bool ZP, bool SUB2>
__global__ void __launch_bounds__(kThreads, 2) bsgemv_mma_kernel(const __grid_constant__ KParams p) {
  using K = Gemv<FMT, BF16, MT, ZP, SUB2>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const typename K::Smem sm{base, p};

  const int64_t G = gridDim.x, T = p.total_stages;
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * T / G;
  const int64_t s1 = (static_cast<int64_t>(blockIdx.x) + 1) * T / G;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(sm.full(i), 1);
      mbar_init(sm.empty(i), kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    if (lane == 0) K::produce(p, sm, s0, s1);
  } else {
    K::consume(p, sm, s0, s1, warp - 1, lane);
  }
}

}  // namespace bsg
