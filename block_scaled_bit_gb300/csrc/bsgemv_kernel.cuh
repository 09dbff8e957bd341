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

// Bounded waits: a waiting thread sleeps in mbarrier.try_wait (suspend-time hint, woken when the
// phase completes) and gives up after kWaitLimitNs of wall time, far above any legitimate stall.
constexpr uint32_t kSuspendHintNs = 1000000;
constexpr uint64_t kWaitLimitNs = 4000000000ull;

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

// Raise the barrier's expected transaction bytes without arriving.
BSG_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

BSG_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

BSG_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

BSG_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: returns false (and records `code` in the error word) if the phase does not
// complete within kWaitLimitNs.
BSG_DEV bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* err, unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, code);
      return false;
    }
  }
}

BSG_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Same as tma_load_2d with an L2 eviction-priority policy (evict_first for stream-once data).
BSG_DEV void tma_load_2d_hint(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar,
                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

BSG_DEV uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 16-byte asynchronous global -> shared copy through L2; `bytes` < 16 zero-fills the rest
// (0 copies nothing and only writes zeros).
BSG_DEV void cp_async16(uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes)
               : "memory");
}

// Make `bar` wait for this thread's prior cp.async copies: its pending count is raised now
// and an arrival is performed when the copies have landed.
BSG_DEV void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Prefetch one TMA box of a 2D tensor into L2 (no shared memory, no barrier).
BSG_DEV void tma_prefetch_l2_2d(const CUtensorMap* tm, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tm)),
               "r"(x), "r"(y)
               : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream be scheduled now, and wait
// until the previous kernel has completed with its memory visible.  Both are no-ops for a
// launch without the programmatic-serialization attribute.
BSG_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
BSG_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

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

// D = A * B (the accumulator input is zero): starts a scale group without zeroing registers.
template <bool BF16>
BSG_DEV void mma16816_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  const float z = 0.f;
  if constexpr (BF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  }
}

// (acc0, acc1) += (x0, x1) * s, two fp32 FMAs in one packed instruction.
BSG_DEV void ffma2(float& acc0, float& acc1, float x0, float x1, float s) {
  uint64_t a, x, ss;
  asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(acc0), "f"(acc1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
  asm("mov.b64 %0, {%1, %1};" : "=l"(ss) : "f"(s));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x), "l"(ss));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(acc0), "=f"(acc1) : "l"(a));
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
// Scale-block grouping of a consumer warp's two chunks (k = 32 per chunk for the 4-bit formats,
// 16 for the 8-bit formats):
//   kBlockPerChunk  block == chunk k-range: scale after every chunk       (int4 bs32, int8 bs16)
//   kBlockPerPair   both chunks in one block: scale once per stage        (bs >= 2 chunks, fp8)
//   kTwoPerChunk    a chunk holds two blocks, quad lanes t < 2 and t >= 2 (int4 bs16)
enum BlockMode : int { kBlockPerChunk = 0, kBlockPerPair = 1, kTwoPerChunk = 2 };

template <int FMT, bool BF16, int MT, bool ZP, int BMODE>
struct Gemv {
  static constexpr bool kFour = (FMT == kInt4 || FMT == kNvfp4);
  static constexpr int kKpc = kFour ? 32 : 16;  // k per 16-byte chunk
  static constexpr int kSteps = kKpc / 16;      // mma k-steps per chunk
  static constexpr int kKc = kChunksPerStage * kKpc;
  static constexpr int kNbox = kKc / 64;        // activation boxes per stage
  static constexpr bool kFold = (FMT == kNvfp4);
  static constexpr int kSub = (BMODE == kTwoPerChunk) ? 2 : 1;
  static constexpr int kScaleEs = (FMT == kFp8) ? 4 : (FMT == kNvfp4 ? 1 : 2);
  // scale box width in blocks (16 bytes, or 32 bytes when a stage holds 16 int4 blocks)
  static constexpr int kSbw = (FMT == kFp8) ? 4 : ((FMT == kNvfp4 || BMODE == kTwoPerChunk) ? 16 : 8);
  static constexpr int kSpitch = kSbw * kScaleEs;  // bytes per row of the scale box
  static constexpr int kZblk = (FMT == kInt4) ? 32 : 16;  // blocks per 16-byte zero-point box row

  struct Smem {
    uint8_t* base;
    int stages, slot_bytes, bar_off, red_off;
    BSG_DEV uint32_t slot(int i) const { return smem_u32(base) + i * slot_bytes; }
    BSG_DEV uint32_t full(int i) const { return smem_u32(base) + bar_off + 8 * i; }
    BSG_DEV uint32_t empty(int i) const { return smem_u32(base) + bar_off + 8 * (stages + i); }
    BSG_DEV float4* red() const { return reinterpret_cast<float4*>(base + red_off); }
    BSG_DEV int* flag() const { return reinterpret_cast<int*>(base + bar_off + 16 * stages); }
  };

  // ---- producer: warp 0.  Lane 0 copies the stage's weight box [64 rows][128 B] with one TMA
  // (L2 evict-first: the weight is read once).  All 32 lanes copy the small pieces -- the
  // activations [M][k of the stage] into the same 128-byte-swizzled layout TMA would write,
  // the scale box and the zero-point box -- with 16-byte cp.async, whose completion is tracked
  // by the same full barrier (cp.async.mbarrier.arrive).  One TMA request stream per stage
  // keeps the TMA unit on the bulk data; rows past N and k past K are zero-filled.
  // Copies of one stage issued by the producer warp (`dst` = the slot, `full` = its barrier).
  struct Stager {
    const KParams& p;
    int lane;
    uint64_t pol;
    int act_units, act_off, abox, sc_off, zp_off, bs_log2, spitch_g, zpitch_g;
    bool side_s, side_z;
    static constexpr int kUpr = kKc / 8;      // 16-byte activation units per row per stage
    static constexpr int kSu = kSpitch / 16;  // 16-byte units per scale box row

    // activations [M][k-range of the stage], written in the 128-byte-swizzled layout
    BSG_DEV void act(uint32_t dst, int ks) const {
      const int64_t k0 = static_cast<int64_t>(ks) * kKc, K = p.K;
      for (int u = lane; u < act_units; u += 32) {
        const int m = u / kUpr, qg = u % kUpr;
        const int q = qg & 7;
        const uint32_t d = dst + act_off + (qg >> 3) * abox + m * 128 + ((q ^ (m & 7)) << 4);
        const int64_t k = k0 + qg * 8;
        const bool in = k < K;
        cp_async16(d, p.A + m * K + (in ? k : 0), in ? 16u : 0u);
      }
    }
    // scale box and zero-point box of the stage (weights: never written by a preceding GEMV)
    BSG_DEV void side(uint32_t dst, int64_t tile, int ks) const {
      const int64_t row0 = tile * kRowsPerTile, N = p.N;
      const int blk0 = (ks * kKc) >> bs_log2;
      if (side_s) {
        const int sx = (blk0 & ~(kSbw - 1)) * kScaleEs;  // byte offset of the box in a scale row
        for (int u = lane; u < kRowsPerTile * kSu; u += 32) {
          const int r = u / kSu, v = u % kSu;
          const int64_t n = row0 + r;
          const bool in = n < N && sx + v * 16 < spitch_g;
          cp_async16(dst + sc_off + r * kSpitch + v * 16,
                     p.scales + (in ? n * spitch_g + sx + v * 16 : 0), in ? 16u : 0u);
        }
      }
      if (side_z) {
        const int xb = blk0 & ~(kZblk - 1);
        const int zx = (FMT == kInt4) ? xb / 2 : xb;
        for (int r = lane; r < kRowsPerTile; r += 32) {
          const int64_t n = row0 + r;
          const bool in = n < N && zx < zpitch_g;
          cp_async16(dst + zp_off + r * 16, p.zp + (in ? n * zpitch_g + zx : 0), in ? 16u : 0u);
        }
      }
    }
    // the weight box (lane 0)
    BSG_DEV void weight(uint32_t dst, uint32_t full, int64_t tile, int ks) const {
      tma_load_2d_hint(dst, &p.tm_w, ks * kStageRowBytes, static_cast<int>(tile * kRowsPerTile),
                       full, pol);
    }
  };

  // ---- producer: warp 0.  Lane 0 copies each stage's weight box [64 rows][128 B] with one TMA
  // (L2 evict-first: the weight is read once).  All 32 lanes copy the small pieces -- the
  // activations [M][k of the stage] into the same 128-byte-swizzled layout TMA would write, the
  // scale box and the zero-point box -- with 16-byte cp.async, whose completion is tracked by the
  // same full barrier (cp.async.mbarrier.arrive).  One TMA request stream per stage keeps the
  // TMA unit on the bulk data; rows past N and k past K are zero-filled.
  //
  // Programmatic dependent launch: while the previous kernel in the stream is still finishing,
  // the first ring slots are filled with everything that is weight (W box, scales, zero points);
  // only after pdl_wait are their activations copied and the slots released to the consumers.
  static BSG_DEV void produce(const KParams& p, const Smem& sm, int64_t s0, int64_t s1, int lane) {
    if (lane == 0) prefetch_tmap(&p.tm_w);
    constexpr uint32_t kTx = kRowsPerTile * kStageRowBytes;
    const Stager st{p, lane, policy_evict_first(), p.M * Stager::kUpr, p.act_off,
                    p.act_box_bytes, p.sc_off, p.zp_off, p.bs_log2, p.scale_pitch, p.zp_pitch,
                    p.side_scale_tma != 0, ZP && p.side_zp_tma != 0};
    const int64_t spt = p.spt;
    int64_t tile0 = s0 / spt;
    const int ks0 = static_cast<int>(s0 - tile0 * spt);

    // phase 1: weight of the first `pre` stages (fresh slots need no empty-barrier wait); the
    // full barrier keeps its one pending arrival (lane 0, phase 2) until the activations land
    const int pre = static_cast<int>((s1 - s0) < sm.stages ? (s1 - s0) : sm.stages);
    {
      int64_t tile = tile0;
      int ks = ks0;
      for (int i = 0; i < pre; ++i) {
        const uint32_t dst = sm.slot(i), full = sm.full(i);
        st.side(dst, tile, ks);
        cp_async_mbar_arrive(full);
        if (lane == 0) {
          mbar_expect_tx(full, kTx);
          st.weight(dst, full, tile, ks);
        }
        if (++ks == spt) {
          ks = 0;
          ++tile;
        }
      }
    }
    pdl_wait();
    // phase 2: activations of those stages, then lane 0's arrival releases each slot
    {
      int64_t tile = tile0;
      int ks = ks0;
      for (int i = 0; i < pre; ++i) {
        const uint32_t dst = sm.slot(i), full = sm.full(i);
        st.act(dst, ks);
        cp_async_mbar_arrive(full);
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
        if (++ks == spt) {
          ks = 0;
          ++tile;
        }
      }
    }
    // steady state
    int slot = pre % sm.stages;
    uint32_t phase = (pre == sm.stages) ? 1u : 0u;
    int64_t tile = tile0;
    int ks = ks0;
    for (int i = 0; i < pre; ++i) {
      if (++ks == spt) {
        ks = 0;
        ++tile;
      }
    }
    for (int64_t s = s0 + pre; s < s1; ++s) {
      if (!mbar_wait(sm.empty(slot), phase ^ 1u, p.err, kErrTimeoutEmpty)) break;
      const uint32_t dst = sm.slot(slot), full = sm.full(slot);
      st.act(dst, ks);
      st.side(dst, tile, ks);
      cp_async_mbar_arrive(full);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(full, kTx);
        st.weight(dst, full, tile, ks);
      }
      if (++slot == sm.stages) {
        slot = 0;
        phase ^= 1u;
      }
      if (++ks == spt) {
        ks = 0;
        ++tile;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  }

  // Register copies of the launch parameters the consumer's stage loop reads (same names as
  // in KParams, so the helpers below read them from registers instead of parameter memory).
  struct Run {
    int64_t N;
    int nb_s, bs_log2, scale_pitch, zp_pitch, side_scale_tma, side_zp_tma;
    const uint8_t* scales;
    const uint8_t* zp;
  };

  static BSG_DEV Run make_run(const KParams& p) {
    return Run{p.N, p.nb_s, p.bs_log2, p.scale_pitch, p.zp_pitch, p.side_scale_tma,
               p.side_zp_tma, p.scales, p.zp};
  }

  // ---- per-lane constants.  Consumer warp cw owns the chunk pair cp = cw & 3 (chunks 2cp and
  // 2cp+1 of every stage) and the row half rh = cw >> 2 (tile rows 32 rh .. 32 rh + 31, i.e.
  // mma row groups 2 rh and 2 rh + 1).  Lane (g, t) holds fragment rows g + 8 rr, rr = 0..3
  // (rr = 2 * local group + upper half), of that row half.
  struct Lane {
    int cp, rh, lane, g, t;
    uint32_t w[2];        // ldmatrix row address of chunk cc (rows 32 rh + lane)
    uint32_t act[2][MT];  // activation fragment address of chunk cc, n8 tile mt
    uint32_t srow;        // scale box row 32 rh + g; row rr adds rr * 8 * kSpitch
    uint32_t zrow;        // zero-point box row 32 rh + g; row rr adds rr * 8 * 16
  };

  static BSG_DEV Lane make_lane(const KParams& p, int cw, int lane) {
    Lane L;
    L.cp = cw & 3;
    L.rh = cw >> 2;
    L.lane = lane;
    L.g = lane >> 2;
    L.t = lane & 3;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = 2 * L.cp + cc;
      const int r = 32 * L.rh + lane;
      L.w[cc] = r * kStageRowBytes + ((c ^ (r & 7)) << 4);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const int m = mt * 8 + L.g;
        if constexpr (kFour) {
          const int q = ((c & 1) << 2) + L.t;
          L.act[cc][mt] = p.act_off + (c >> 1) * p.act_box_bytes + m * 128 + ((q ^ (m & 7)) << 4);
        } else {
          const int q = ((c & 3) << 1) + (L.t >> 1);
          L.act[cc][mt] = p.act_off + (c >> 2) * p.act_box_bytes + m * 128 +
                          ((q ^ (m & 7)) << 4) + ((L.t & 1) << 3);
        }
      }
    }
    L.srow = p.sc_off + (32 * L.rh + L.g) * kSpitch;
    L.zrow = p.zp_off + (32 * L.rh + L.g) * 16;
    return L;
  }

  static BSG_DEV int64_t row_of(const Run& p, const Lane& L, int64_t tile, int rr) {
    const int64_t n = tile * kRowsPerTile + 32 * L.rh + L.g + 8 * rr;
    return n < p.N ? n : p.N - 1;
  }

  // fp32 scales of the lane's 4 rows for NB consecutive blocks starting at `blk` (box-relative
  // index `rel`); NB = 2 only for 2-byte scales at an even `rel` (one 32-bit load per row).
  template <int NB>
  static BSG_DEV void load_scales(const Run& p, const Lane& L, uint32_t slot, int64_t tile,
                                  int blk, int rel, float (&s)[NB][4]) {
    if (p.side_scale_tma) {
      const uint32_t a = slot + L.srow + rel * kScaleEs;
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const uint32_t ar = a + rr * 8 * kSpitch;
        if constexpr (FMT == kFp8) {
#pragma unroll
          for (int u = 0; u < NB; ++u) s[u][rr] = __uint_as_float(lds32(ar + 4 * u));
        } else if constexpr (NB == 2) {
          const uint32_t two = lds32(ar);
          s[0][rr] = __half2float(__ushort_as_half(static_cast<unsigned short>(two & 0xFFFFu)));
          s[1][rr] = __half2float(__ushort_as_half(static_cast<unsigned short>(two >> 16)));
        } else {
          s[0][rr] = __half2float(__ushort_as_half(static_cast<unsigned short>(lds16(ar))));
        }
      }
    } else {
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const uint8_t* src = p.scales + row_of(p, L, tile, rr) * p.scale_pitch;
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          const int b = blk + u;
          if (b >= p.nb_s) {  // chunk past K in the ragged last stage: its weight is zero
            s[u][rr] = 0.f;
          } else if constexpr (FMT == kFp8) {
            s[u][rr] = __ldg(reinterpret_cast<const float*>(src) + b);
          } else {
            s[u][rr] = __half2float(__ldg(reinterpret_cast<const __half*>(src) + b));
          }
        }
      }
    }
  }

  // Zero-point operand constants (see zp_consts) of the lane's 4 rows for block `blk`.
  static BSG_DEV void load_zp(const Run& p, const Lane& L, uint32_t slot, int64_t tile,
                              int blk, int rel, uint32_t (&zl)[4], uint32_t (&zh)[4]) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      uint32_t z;
      if constexpr (!ZP) {
        z = (FMT == kInt4) ? 8u : 128u;
      } else if (p.side_zp_tma) {
        const uint32_t byte = lds8(slot + L.zrow + rr * 8 * 16 + ((FMT == kInt4) ? (rel >> 1) : rel));
        z = (FMT == kInt4) ? ((rel & 1) ? (byte >> 4) : (byte & 0xFu)) : byte;
      } else {
        uint32_t byte = 0;
        if (blk < p.nb_s)
          byte = __ldg(p.zp + row_of(p, L, tile, rr) * p.zp_pitch + ((FMT == kInt4) ? (blk >> 1) : blk));
        z = (FMT == kInt4) ? ((blk & 1) ? (byte >> 4) : (byte & 0xFu)) : byte;
      }
      zp_consts<FMT, BF16>(z, zl[rr], zh[rr]);
    }
  }

  // NVFP4: the replicated f16 E4M3 block scale of the lane's 4 rows for 16-block `blk`.
  static BSG_DEV void load_fold(const Run& p, const Lane& L, uint32_t slot, int64_t tile,
                                int blk, int rel, uint32_t (&f)[4]) {
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      uint32_t code;
      if (p.side_scale_tma) {
        code = lds8(slot + L.srow + rr * 8 * kSpitch + rel);
      } else {
        code = (blk < p.nb_s) ? __ldg(p.scales + row_of(p, L, tile, rr) * p.scale_pitch + blk) : 0u;
      }
      f[rr] = e4m3x2_to_f16x2(code * 0x0101u);
    }
  }

  // Activation B fragments of chunk cc: b[mt][st][0] = (k 2t, 2t+1), b[mt][st][1] = (k 2t+8,
  // 2t+9) of activation row mt*8 + g, permuted like the weight (phys_k).
  static BSG_DEV void act_fragment(const Lane& L, uint32_t slot, int cc, uint32_t (&b)[MT][kSteps][2]) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      if constexpr (kFour) {
        const uint4 v = lds128(slot + L.act[cc][mt]);
        if constexpr (FMT == kInt4) {  // pairs (8t+j, 8t+j+4)
          b[mt][0][0] = prmt(v.x, v.z, 0x5410u);
          b[mt][0][1] = prmt(v.x, v.z, 0x7632u);
          b[mt][1][0] = prmt(v.y, v.w, 0x5410u);
          b[mt][1][1] = prmt(v.y, v.w, 0x7632u);
        } else {  // nvfp4: natural pairs
          b[mt][0][0] = v.x;
          b[mt][0][1] = v.y;
          b[mt][1][0] = v.z;
          b[mt][1][1] = v.w;
        }
      } else {
        const uint2 v = lds64(slot + L.act[cc][mt]);
        b[mt][0][0] = v.x;
        b[mt][0][1] = v.y;
      }
    }
  }

  // Decode the lane's 2 row groups of chunk cc and multiply into d[u] (u: sub-block for
  // kTwoPerChunk).  ZC: the first k-step starts from zero instead of accumulating.
  template <bool ZC>
  static BSG_DEV void chunk_mma(const Lane& L, uint32_t slot, int cc, const uint32_t (&zl)[4],
                                const uint32_t (&zh)[4], float (&d)[kSub][2][MT][4]) {
    uint32_t b[MT][kSteps][2];
    act_fragment(L, slot, cc, b);
    uint32_t wv[4];
    ldsm_x4(slot + L.w[cc], wv[0], wv[1], wv[2], wv[3]);
#pragma unroll
    for (int lg = 0; lg < 2; ++lg) {
      uint32_t a[kSteps][4];
      if constexpr (FMT == kInt4) {
        decode_int4<BF16>(wv[2 * lg], wv[2 * lg + 1], zl[2 * lg], zh[2 * lg], zl[2 * lg + 1],
                          zh[2 * lg + 1], a);
      } else if constexpr (FMT == kInt8) {
        decode_int8<BF16>(wv[2 * lg], wv[2 * lg + 1], zl[2 * lg], zl[2 * lg + 1], a);
      } else if constexpr (FMT == kFp8) {
        decode_fp8<BF16>(wv[2 * lg], wv[2 * lg + 1], a);
      } else {
        decode_nvfp4<BF16>(wv[2 * lg], wv[2 * lg + 1], zl[2 * lg], zl[2 * lg + 1], a);
      }
#pragma unroll
      for (int st = 0; st < kSteps; ++st)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const bool zc = ZC && st == 0;
#pragma unroll
          for (int u = 0; u < kSub; ++u) {
            uint32_t b0 = b[mt][st][0], b1 = b[mt][st][1];
            if constexpr (kSub == 2) {
              // quad lanes t < 2 hold the chunk's first block, t >= 2 the second
              const bool mine = (L.t >> 1) == u;
              b0 = mine ? b0 : 0u;
              b1 = mine ? b1 : 0u;
            }
            if (zc) mma16816_zc<BF16>(d[u][lg][mt], a[st], b0, b1);
            else mma16816<BF16>(d[u][lg][mt], a[st], b0, b1);
          }
        }
    }
  }

  // acc += tmp * s (per fragment row: s[2*lg] for row g, s[2*lg+1] for row g+8).
  static BSG_DEV void apply_scales(const float (&s)[4], const float (&tmp)[2][MT][4],
                                   float (&acc)[2][MT][4]) {
#pragma unroll
    for (int lg = 0; lg < 2; ++lg)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        acc[lg][mt][0] = fmaf(tmp[lg][mt][0], s[2 * lg], acc[lg][mt][0]);
        acc[lg][mt][1] = fmaf(tmp[lg][mt][1], s[2 * lg], acc[lg][mt][1]);
        acc[lg][mt][2] = fmaf(tmp[lg][mt][2], s[2 * lg + 1], acc[lg][mt][2]);
        acc[lg][mt][3] = fmaf(tmp[lg][mt][3], s[2 * lg + 1], acc[lg][mt][3]);
      }
  }

  template <int U>
  static BSG_DEV void zero(float (&x)[U][2][MT][4]) {
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int lg = 0; lg < 2; ++lg)
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int i = 0; i < 4; ++i) x[u][lg][mt][i] = 0.f;
  }

  // Consume one ring slot: chunks 2cp and 2cp+1, row half rh, of stage ks of `tile`.
  static BSG_DEV void consume_stage(const Run& p, const Lane& L, uint32_t slot, int64_t tile,
                                    int ks, float (&acc)[1][2][MT][4]) {
    const int bs_log2 = p.bs_log2;
    const int blk0 = (ks * kKc) >> bs_log2;  // first scale block of the stage
    const int sbox0 = blk0 & ~(kSbw - 1);     // first block of the staged scale box
    const int zbox0 = blk0 & ~(kZblk - 1);
    uint32_t zl[4], zh[4];
    if constexpr (kFold) {
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        // the lane's 8 codes lie in 16-block (k of chunk + 8t) / 16
        const int fb = ((ks * kKc + (2 * L.cp + cc) * kKpc) >> 4) + (L.t >> 1);
        load_fold(p, L, slot, tile, fb, fb - sbox0, zl);
        chunk_mma<false>(L, slot, cc, zl, zh, acc);
      }
    } else if constexpr (BMODE == kBlockPerPair) {
      const int blk = blk0 + ((2 * L.cp * kKpc) >> bs_log2);
      load_zp(p, L, slot, tile, blk, blk - zbox0, zl, zh);
      float tmp[1][2][MT][4];
      chunk_mma<true>(L, slot, 0, zl, zh, tmp);
      chunk_mma<false>(L, slot, 1, zl, zh, tmp);
      float s[1][4];
      load_scales<1>(p, L, slot, tile, blk, blk - sbox0, s);
      apply_scales(s[0], tmp[0], acc[0]);
    } else if constexpr (BMODE == kBlockPerChunk) {
      const int blk = blk0 + 2 * L.cp;  // chunk cc is block blk + cc
      float s[2][4];
      if constexpr (kScaleEs == 2) {
        load_scales<2>(p, L, slot, tile, blk, blk - sbox0, s);
      } else {
        float s1[1][4];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          load_scales<1>(p, L, slot, tile, blk + cc, blk + cc - sbox0, s1);
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) s[cc][rr] = s1[0][rr];
        }
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        load_zp(p, L, slot, tile, blk + cc, blk + cc - zbox0, zl, zh);
        float tmp[1][2][MT][4];
        chunk_mma<true>(L, slot, cc, zl, zh, tmp);
        apply_scales(s[cc], tmp[0], acc[0]);
      }
    } else {  // kTwoPerChunk: chunk cc holds blocks blk, blk + 1 (int4, 16-element blocks)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int blk = blk0 + 2 * (2 * L.cp + cc);
        const int zb = blk + (L.t >> 1);
        load_zp(p, L, slot, tile, zb, zb - zbox0, zl, zh);
        float tmp[2][2][MT][4];
        chunk_mma<true>(L, slot, cc, zl, zh, tmp);
        float s[2][4];
        load_scales<2>(p, L, slot, tile, blk, blk - sbox0, s);
        apply_scales(s[0], tmp[0], acc[0]);
        apply_scales(s[1], tmp[1], acc[0]);
      }
    }
  }

  // Store the 4 fp32 results of fragment slot (tile row group rg, tile mt, lane ln) as y.
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

  // End of a tile segment: add the 4 chunk-pair warps of each row half (fixed order), then
  // store, or publish a partial and let the last CTA of the tile add the partials in CTA order.
  // Partial slots: CTA i writes slot 0 for the first tile of its range and slot 1 for its last
  // tile, so among a tile's contributors only the first can hold it in slot 1 (when its range
  // began in an earlier tile).
  static BSG_DEV void epilogue(const KParams& p, const Smem& sm, int64_t tile, bool whole,
                               int64_t my_first_tile, int cw, int lane, float (&acc)[1][2][MT][4],
                               float gs) {
    constexpr int kNT = kConsumerWarps * 32;   // 256 consumer threads
    constexpr int kSlots = 2 * MT * 32;        // float4 slots per warp
    constexpr int kOut = 4 * MT * 32;          // float4 slots per tile (4 row groups)
    const int tid = cw * 32 + lane;
    float4* red = sm.red();
#pragma unroll
    for (int lg = 0; lg < 2; ++lg)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        red[cw * kSlots + (lg * MT + mt) * 32 + lane] =
            make_float4(acc[0][lg][mt][0], acc[0][lg][mt][1], acc[0][lg][mt][2], acc[0][lg][mt][3]);
    named_bar_sync(1, kNT);

    // output slot tid = ((rh * 2 + lg) * MT + mt) * 32 + ln, tile row group rg = 2 rh + lg
    const bool active = tid < kOut;
    const int ln = tid & 31;
    const int q = tid >> 5;
    const int mt = q % MT, rg = q / MT;
    const int rh = rg >> 1, lg = rg & 1;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) {
#pragma unroll
      for (int cp = 0; cp < 4; ++cp) {
        const float4 u = red[(rh * 4 + cp) * kSlots + (lg * MT + mt) * 32 + ln];
        sum.x += u.x;
        sum.y += u.y;
        sum.z += u.z;
        sum.w += u.w;
      }
    }
    if (whole) {
      if (active) store_y(p, tile, rg, mt, ln, sum, gs);
    } else {
      const int slot_floats4 = p.slot_floats / 4;
      const int seg = (tile == my_first_tile) ? 0 : 1;
      float4* mine = reinterpret_cast<float4*>(p.partials) +
                     (static_cast<int64_t>(blockIdx.x) * 2 + seg) * slot_floats4;
      if (active) __stcg(mine + tid, sum);
      named_bar_sync(1, kNT);
      int* info = sm.flag();  // [0] last arriver?  [1] first CTA  [2] last CTA  [3] first's slot
      if (tid == 0) {
        const int64_t G = gridDim.x, T = p.total_stages;
        const int64_t x0 = tile * p.spt;
        const int64_t first = cta_of_stage(x0, T, G);
        const int64_t last = cta_of_stage(x0 + p.spt - 1, T, G);
        // the barrier orders every thread's partial store before this fence (fences are
        // cumulative), which publishes them at GPU scope before the arrival count
        __threadfence();
        const unsigned old = atomicAdd(p.counters + tile, 1u);
        info[0] = (old == static_cast<unsigned>(last - first)) ? 1 : 0;
        info[1] = static_cast<int>(first);
        info[2] = static_cast<int>(last);
        info[3] = (first * T < x0 * G) ? 1 : 0;  // first CTA's range began before this tile
      }
      named_bar_sync(1, kNT);
      if (info[0]) {
        __threadfence();  // acquire side: order the partial loads after the observed count
        const int first = info[1], last = info[2], fseg = info[3];
        if (active) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          const float4* part = reinterpret_cast<const float4*>(p.partials) + tid;
          for (int i = first; i <= last; ++i) {
            const int sg = (i == first) ? fseg : 0;
            const float4 u = __ldcg(part + (static_cast<int64_t>(i) * 2 + sg) * slot_floats4);
            v.x += u.x;
            v.y += u.y;
            v.z += u.z;
            v.w += u.w;
          }
          store_y(p, tile, rg, mt, ln, v, gs);
        }
        if (tid == 0) p.counters[tile] = 0u;  // every contributor has arrived: reset for reuse
      }
    }
    named_bar_sync(1, kNT);  // `red` and the info words are reused by the next segment
  }

  static BSG_DEV void consume(const KParams& p, const Smem& sm, int64_t s0, int64_t s1, int cw,
                              int lane) {
    pdl_wait();  // the epilogues write y and the plan's workspace
    const Lane L = make_lane(p, cw, lane);
    const Run R = make_run(p);
    float acc[1][2][MT][4];
    zero(acc);
    const float gs = kFold ? __ldg(p.gscale) : 1.0f;
    const int64_t spt = p.spt;
    int slot = 0;
    uint32_t phase = 0;
    int64_t tile = s0 / spt;
    int ks = static_cast<int>(s0 - tile * spt);
    const int64_t first_tile = tile;
    bool ok = true;
    for (int64_t s = s0; s < s1; ++s) {
      if (ok) ok = mbar_wait(sm.full(slot), phase, p.err, kErrTimeoutFull);
      if (ok) consume_stage(R, L, sm.slot(slot), tile, ks, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.empty(slot));
      if (ks == spt - 1 || s == s1 - 1) {
        const bool whole = (s0 <= tile * spt) && (s1 >= (tile + 1) * spt);
        epilogue(p, sm, tile, whole, first_tile, cw, lane, acc, gs);
        zero(acc);
      }
      if (++slot == sm.stages) {
        slot = 0;
        phase ^= 1u;
      }
      if (++ks == spt) {
        ks = 0;
        ++tile;
      }
    }
  }
};

template <int FMT, bool BF16, int MT, bool ZP, int BMODE>
__global__ void __launch_bounds__(kThreads, 2) bsgemv_mma_kernel(const __grid_constant__ KParams p) {
  using K = Gemv<FMT, BF16, MT, ZP, BMODE>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const typename K::Smem sm{base, p.stages, p.slot_bytes, p.bar_off, p.red_off};

  const int64_t G = gridDim.x, T = p.total_stages;
  const int64_t s0 = static_cast<int64_t>(blockIdx.x) * T / G;
  const int64_t s1 = (static_cast<int64_t>(blockIdx.x) + 1) * T / G;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < sm.stages; ++i) {
      mbar_init(sm.full(i), 1);
      mbar_init(sm.empty(i), kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 0) {
    K::produce(p, sm, s0, s1, lane);
  } else {
    K::consume(p, sm, s0, s1, warp - 1, lane);
  }
}

}  // namespace bsg
