// bsgemv_kernel.cuh -- the sm_103a GEMV kernel template
//
//     y[M, N] = A[M, K] . deq(W)[N, K]^T,  M <= 32
//
// Data path per CTA (a persistent grid, 4 CTAs of 160 threads per SM; 3 for plans with M up to
// 24, 2 for M up to 32):
//   warp 0           producer: for every stage (256 k of a 64-row tile) of the CTA's range, lane
//                    0 waits for a free ring slot and issues the stage's weight box(es)
//                    [64 rows][128 B] with cp.async.bulk.tensor (128-byte swizzle, L2
//                    evict-first); all 32 lanes copy the stage's activations [M][256 k] with
//                    16-byte cp.async into padded rows.  Scales and zero points travel on a
//                    side ring, one TMA box [64 rows][64 B of scales] per 2..64 stages.
//   warps 1..4       consumers: warp w owns rows 16w .. 16w + 15 of the tile over the whole
//                    stage.  ldmatrix hands every lane the 32-bit words of its two rows (g and
//                    g + 8) in every 16-byte chunk; the words are decoded in registers to exact
//                    fp16/bf16 operand pairs ((q - zp), e4m3, or e2m1 * e4m3), fed to
//                    mma.sync.m16n8k16 with the weight as the A operand (16 output columns)
//                    and the activations as the B operand (8 rows of A per n8 tile), summed in
//                    fp32.  Int and FP8 scales multiply the fp32 partial of each scale block;
//                    NVFP4's E4M3 scale is folded into the 16-bit operand (exact: 2 + 4
//                    significand bits).  The CUDA-core variant (template parameter CC) forms
//                    the same products with packed fp32 FMAs instead (chunk_cc).
//   epilogue         a tile consumed whole by the CTA is rounded and stored; a tile shared with
//                    other CTAs is finished either by the last CTA to arrive (stream-K: fp32
//                    partials in the plan's workspace, added in CTA order) or by the leader of
//                    the tile's thread-block cluster (partials in its shared memory, added in
//                    rank order).  The optional bias is added in fp32 before the one rounding.
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

// Bounded waits: a waiting thread blocks in mbarrier.try_wait (the hardware's own time window,
// no suspend-time hint: measured faster to wake than a hinted wait) and gives up after a limit
// of wall time -- kWaitLimitNs unless the launch sets another (KParams::wait_ns), far above any
// legitimate stall.
constexpr uint64_t kWaitLimitNs = kDefaultWaitNs;

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

// Arrive on `bar` if `pred` (a predicated instruction: no branch around it).
BSG_DEV void mbar_arrive_if(uint32_t bar, bool pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar),
      "r"(static_cast<uint32_t>(pred))
      : "memory");
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

BSG_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: returns false (and records `code` in the error word) if the phase does not
// complete within limit_ns.
BSG_DEV bool mbar_wait(uint32_t bar, uint32_t parity, unsigned* err, unsigned code,
                       uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) {
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

// Programmatic dependent launch: let the next kernel in the stream be scheduled now, and wait
// until the previous kernel has completed with its memory visible.  Both are no-ops for a
// launch without the programmatic-serialization attribute.
BSG_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
BSG_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Arrival on a global counter with release (publishes what this thread has observed, e.g. its
// warp's stores ordered by __syncwarp) and acquire (a last arriver sees every contributor's
// stores) semantics at GPU scope.  Returns the old value.
BSG_DEV unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Thread-block clusters: this CTA's rank, the shared-window address of `addr` in CTA `rank` of
// the cluster, a 16-byte store there, and a cluster-wide barrier (release / acquire: shared
// memory written before it by any CTA of the cluster is visible after it).
BSG_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

BSG_DEV uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t d;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(addr), "r"(rank));
  return d;
}

BSG_DEV void st_cluster_f32x4(uint32_t addr, float x, float y, float z, float w) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(x), "f"(y),
               "f"(z), "f"(w)
               : "memory");
}

BSG_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}

BSG_DEV void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// ldmatrix at addr + OFF (a compile-time offset in the instruction's immediate field).
template <int OFF>
BSG_DEV void ldsm_x4_at(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4+%5];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr), "n"(OFF));
}

BSG_DEV uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// Plain shared-memory load of a T at p (p derived from the kernel's shared array).  Unlike an
// asm statement, the compiler may reorder these among themselves and hoist them to cover
// latency; the "memory" clobbers of the barrier waits and arrivals keep them inside the slot's
// ownership window.
template <typename T>
BSG_DEV T lsh(const uint8_t* p) {
  return *reinterpret_cast<const T*>(p);
}

// Bits of a where MASK is set, bits of c elsewhere: one LOP3 with the mask as its immediate.
// The decoders take the constant part of an operand (exponent bits) from the zero-point
// registers they hold anyway, so no constant has to be kept in (or re-created into) a register
// per use.
template <uint32_t MASK>
BSG_DEV uint32_t select_bits(uint32_t a, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xE2;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
  return d;
}

// prmt with a compile-time selector (the instruction's immediate field).
template <uint32_t SEL>
BSG_DEV uint32_t prmt(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "n"(SEL));
  return d;
}

// D += A * B on the tensor cores: m16n8k16, fp16 or bf16 operands, fp32 accumulate.
template <bool BF16>
BSG_DEV void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm(
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
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  } else {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  }
}

// Packed fp32 pairs (low word = first element) for the CUDA-core variant's FMAs.
BSG_DEV uint64_t f32x2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
BSG_DEV float f32x2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
BSG_DEV float f32x2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
// acc += a * b on both fp32 halves (one packed CUDA-core FMA).
BSG_DEV void fma_f32x2(uint64_t& acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
BSG_DEV uint64_t mul_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// ------------------------------------------------------------------------------ 16-bit pairs
// Half h of a 16-bit pair (f16 or bf16) as fp32 (exact).
template <bool BF16>
BSG_DEV float half_to_f32(uint32_t pair, int h) {
  if constexpr (BF16) return __uint_as_float(h ? (pair & 0xFFFF0000u) : (pair << 16));
  const __half2 v = *reinterpret_cast<const __half2*>(&pair);
  return h ? __high2float(v) : __low2float(v);
}

BSG_DEV uint32_t h2_sub(uint32_t a, uint32_t b) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
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

// The four E2M1 code pairs of a word (byte b -> out[b], low nibble -> low half), unpacked from
// the register's bytes inside the conversion.
BSG_DEV void e2m1x8_to_f16x2x4(uint32_t w, uint32_t (&out)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3])
      : "r"(w));
}

// The E4M3 code in byte `sel & 3` of w, replicated as an exact f16 pair (sel = 0x11 * byte).
BSG_DEV uint32_t e4m3_byte_to_f16x2(uint32_t w, uint32_t sel) {
  uint32_t d;
  asm("{\n\t.reg .b32 t;\n\t.reg .b16 l, h;\n\t"
      "prmt.b32 t, %1, %1, %2;\n\t"
      "mov.b32 {l, h}, t;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t}"
      : "=r"(d)
      : "r"(w), "r"(sel));
  return d;
}

// The two E4M3 code pairs of a word (low half -> lo, high half -> hi).
BSG_DEV void e4m3x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// An f16 pair as a bf16 pair: each half widened to fp32 (exact) and the two packed by one
// round-to-nearest-even conversion, which is exact for values bf16 holds -- E4M3 values and
// E2M1 x E4M3 products have at most 6 significand bits and lie in [2^-10, 2688] -- and keeps a
// NaN a NaN (E4M3 codes 0x7F / 0xFF decode to an f16 NaN; as a weight, or as an NVFP4 block
// scale, the product must stay NaN, as the format's definition and the oracle have it).
BSG_DEV uint32_t f16x2_to_bf16x2(uint32_t h) {
  uint32_t d;
  asm("{\n\t.reg .b16 l, u;\n\t.reg .f32 fl, fu;\n\t"
      "mov.b32 {l, u}, %1;\n\t"
      "cvt.f32.f16 fl, l;\n\t"
      "cvt.f32.f16 fu, u;\n\t"
      "cvt.rn.bf16x2.f32 %0, fu, fl;\n\t}"
      : "=r"(d)
      : "r"(h));
  return d;
}

// ------------------------------------------------------------------------------ decoders
// Each decoder turns the ldmatrix words of one mma row pair -- `lo` for tile row g, `hi` for row
// g + 8 -- into the A fragments of every k-step of the chunk:
//   a[s][0] = (row g,   cols 2t, 2t+1)   a[s][1] = (row g+8, cols 2t, 2t+1)
//   a[s][2] = (row g,   cols 2t+8, 2t+9) a[s][3] = (row g+8, cols 2t+8, 2t+9)
// The physical k of each half is given by phys_k below; the activation fragment follows it.

// int4: nibble j of the lane's word holds k = 8t + j.  Put under the exponent bits of
// zl = (1024 + zp) (zp sits in the low nibble, which the nibble replaces), the low nibble of a
// byte gives the f16 value 1024 + q; put under the sign and exponent of zh = -(64 + zp) (zp in
// bits 4..7, replaced), the high nibble gives -(64 + q), so that zh minus it is q - zp.  Both
// results are the exact small integer q - zp ("[CUDA] MatMulNBits 8-bit: wide fp16 M=1 kernel
// for decode GEMVs", Description: exact (q - zp) in fp16).  For bf16 the exponent of 128 holds
// 7 mantissa bits, so each nibble is shifted to the bottom first and zl = (128 + zp).
template <bool BF16>
BSG_DEV void decode_int4(uint32_t lo, uint32_t hi, uint32_t zl_lo, uint32_t zh_lo, uint32_t zl_hi,
                         uint32_t zh_hi, uint32_t (&a)[2][4]) {
  if constexpr (!BF16) {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t wl = lo >> (8 * s), wh = hi >> (8 * s);
      a[s][0] = h2_sub(select_bits<0x000F000Fu>(wl, zl_lo), zl_lo);
      a[s][1] = h2_sub(select_bits<0x000F000Fu>(wh, zl_hi), zl_hi);
      a[s][2] = h2_sub(zh_lo, select_bits<0x00F000F0u>(wl, zh_lo));
      a[s][3] = h2_sub(zh_hi, select_bits<0x00F000F0u>(wh, zh_hi));
    }
  } else {
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t wl = lo >> (8 * s), wh = hi >> (8 * s);
      a[s][0] = bf2_sub(select_bits<0x000F000Fu>(wl, zl_lo), zl_lo);
      a[s][1] = bf2_sub(select_bits<0x000F000Fu>(wh, zl_hi), zl_hi);
      a[s][2] = bf2_sub(select_bits<0x000F000Fu>(wl >> 4, zl_lo), zl_lo);
      a[s][3] = bf2_sub(select_bits<0x000F000Fu>(wh >> 4, zl_hi), zl_hi);
    }
  }
  (void)zh_lo;
  (void)zh_hi;
}

// int8: byte j of the lane's word holds k = 4t + j.  f16: prmt places byte j under the
// exponent byte of 1024, taken from z = (1024 + zp) itself (its bytes 1 and 3), giving the
// exact 1024 + q, minus z.  bf16 (7 mantissa bits cannot hold 0..255 above one exponent):
// 2^23 + q in fp32 (the high bytes again from z = 2^23 + zp: bytes 1, 2 are zero, byte 3 the
// exponent), minus z, packed by an exact cvt.
template <bool BF16>
BSG_DEV void decode_int8(uint32_t lo, uint32_t hi, uint32_t z_lo, uint32_t z_hi,
                         uint32_t (&a)[1][4]) {
  if constexpr (!BF16) {
    a[0][0] = h2_sub(prmt<0x5150u>(lo, z_lo), z_lo);
    a[0][1] = h2_sub(prmt<0x5150u>(hi, z_hi), z_hi);
    a[0][2] = h2_sub(prmt<0x5352u>(lo, z_lo), z_lo);
    a[0][3] = h2_sub(prmt<0x5352u>(hi, z_hi), z_hi);
  } else {
    auto pack = [](float x0, float x1) -> uint32_t {
      uint32_t d;
      asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(x1), "f"(x0));
      return d;
    };
    const float zl = __uint_as_float(z_lo), zh = __uint_as_float(z_hi);  // 2^23 + zp
    a[0][0] = pack(__uint_as_float(prmt<0x7550u>(lo, z_lo)) - zl,
                   __uint_as_float(prmt<0x7551u>(lo, z_lo)) - zl);
    a[0][1] = pack(__uint_as_float(prmt<0x7550u>(hi, z_hi)) - zh,
                   __uint_as_float(prmt<0x7551u>(hi, z_hi)) - zh);
    a[0][2] = pack(__uint_as_float(prmt<0x7552u>(lo, z_lo)) - zl,
                   __uint_as_float(prmt<0x7553u>(lo, z_lo)) - zl);
    a[0][3] = pack(__uint_as_float(prmt<0x7552u>(hi, z_hi)) - zh,
                   __uint_as_float(prmt<0x7553u>(hi, z_hi)) - zh);
  }
}

// FP8 E4M3: byte j of the lane's word holds k = 4t + j; E4M3 is exact in f16 and bf16
// (decode-GEMV page, FP8 tensor-core paragraph).
template <bool BF16>
BSG_DEV void decode_fp8(uint32_t lo, uint32_t hi, uint32_t (&a)[1][4]) {
  e4m3x4_to_f16x2x2(lo, a[0][0], a[0][2]);
  e4m3x4_to_f16x2x2(hi, a[0][1], a[0][3]);
  if constexpr (BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) a[0][i] = f16x2_to_bf16x2(a[0][i]);
  }
}

// NVFP4: byte b of the lane's word holds k = 8t + 2b (low nibble) and 8t + 2b + 1.  The E4M3
// block scale (sc_lo for row g, sc_hi for row g+8, as f16 pairs) is folded into the decoded
// E2M1 value: exact in f16 and bf16 (decode-GEMV page, NVFP4 tensor-core paragraph).
template <bool BF16>
BSG_DEV void decode_nvfp4(uint32_t lo, uint32_t hi, uint32_t sc_lo, uint32_t sc_hi,
                          uint32_t (&a)[2][4]) {
  uint32_t l[4], h[4];  // byte b of the word as an f16 pair
  e2m1x8_to_f16x2x4(lo, l);
  e2m1x8_to_f16x2x4(hi, h);
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    a[s][0] = h2_mul(l[2 * s], sc_lo);
    a[s][1] = h2_mul(h[2 * s], sc_hi);
    a[s][2] = h2_mul(l[2 * s + 1], sc_lo);
    a[s][3] = h2_mul(h[2 * s + 1], sc_hi);
    if constexpr (BF16) {
#pragma unroll
      for (int i = 0; i < 4; ++i) a[s][i] = f16x2_to_bf16x2(a[s][i]);
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
// Scale blocks of the weight formats, per 16-byte chunk of a row (k = 32 per chunk for the 4-bit
// formats, 16 for the 8-bit formats): the kernel's CPB template parameter is the number of
// chunks per scale block -- 0 when a chunk holds two blocks (int4 with 16-element blocks), 1, 2,
// 4, or 8 for a block of a whole 128-byte box or more (larger blocks, fp8).  NVFP4 folds its scales
// into the decoded values and uses 1.

// CC > 0 selects the CUDA-core variant: the same copies, rings, decoders and epilogues, but the
// products are formed by fp32 FMAs on the CUDA cores (each lane over its own k positions of
// the tile rows it holds, for CC = 1 or 8 activation rows: calls with M = 1, or M <= 8)
// instead of mma.sync.
template <int FMT, bool BF16, int MT, bool ZP, int CPB, int H, int CC = 0>
struct Gemv {
  static_assert(H == 1 || H == 2, "one or two 64-row halves per tile");
  static_assert(CC == 0 || ((CC == 1 || CC == 8) && MT == 1),
                "CUDA-core variant: 1 or 8 activation rows, natural activation order");
  static constexpr int kCcCols = CC > 0 ? CC : 1;  // activation rows a CUDA-core lane accumulates
  static constexpr bool kFour = (FMT == kInt4 || FMT == kNvfp4);
  static constexpr int kKpc = kFour ? 32 : 16;  // k per 16-byte chunk
  static constexpr int kSteps = kKpc / 16;      // mma k-steps per chunk
  static constexpr int kKb = stage_kboxes(FMT, H);  // weight boxes along k per stage (1 or 2)
  static constexpr int kKc = stage_k(FMT, H);        // k per stage: 256, or 128 (8-bit, 2 halves)
  static constexpr int kBoxK = kKc / kKb;            // k per box
  static constexpr int kCps = kBoxK / kKpc;          // 16-byte chunks per row per box: 8
  static constexpr int kSrb = kKb * kBoxRowBytes;    // weight bytes per row per stage
  static_assert(kCps * 16 == kBoxRowBytes, "a box is 128 bytes of a row");
  static constexpr int kH = H;                              // 64-row halves per tile
  static constexpr int kRows = kH * kBoxRows;               // output columns per tile
  static constexpr int kBoxB = kBoxRows * kBoxRowBytes;     // bytes per weight box (8 KB)
  static constexpr int kStageB = kKb * kH * kBoxB;          // weight bytes per stage (8 or 16 KB)
  static constexpr bool kFold = (FMT == kNvfp4);
  static constexpr int kSub = (CPB == 0) ? 2 : 1;  // scale blocks per chunk (int4, 16-element blocks)
  static constexpr int kScaleEs = (FMT == kFp8) ? 4 : (FMT == kNvfp4 ? 1 : 2);
  static constexpr int kZpW = (FMT == kInt4) ? 4 : 8;  // zero-point bits per block
  // Activation slot of a stage: max_M rows of the stage's k, each padded by one chunk's
  // activation bytes, so that the 8 rows a B-fragment load touches start in different banks
  // (conflict-free without a swizzle, and every chunk's offset is a compile-time constant).
  static constexpr int kActChunkB = 2 * kKpc;               // activation bytes of one chunk
  static constexpr int kActPitch = 2 * kKc + kActChunkB;    // bytes per activation row
  // zero-point bytes per side-box row: the box's 64 bytes of f16 scales are 32 blocks
  static constexpr int kZboxB = 32 * kZpW / 8;
  // log2 of the block size where the kernel variant fixes it (CPB < 8), else -1 (read from
  // the launch: int8 blocks of 128 or 256, one or half a block per weight box)
  static constexpr int kBsLog2 = (kFold || CPB == 0) ? 4
                                : CPB == 8 ? -1
                                           : (CPB == 1 ? 0 : CPB == 2 ? 1 : 2) + (kFour ? 5 : 4);

  // Shared memory: [W ring: stages x kStageB (box (k-box j, half h) at (j kH + h) kBoxB)]
  // [activation ring][side ring]
  // [cluster reduction buffer][barriers].
  // The weight boxes are 1024-byte aligned (128-byte swizzle atoms).
  struct Smem {
    uint8_t* base;    // generic pointer into the kernel's shared array
    uint32_t base_u;  // the same address in the shared window
    int stages, act_off, act_bytes, side_off, side_bytes, side_slots, bar_off;
    BSG_DEV uint32_t w(int i) const { return base_u + i * kStageB; }
    BSG_DEV uint32_t act_u(int i) const { return base_u + act_off + i * act_bytes; }
    BSG_DEV uint32_t side_u(int j) const { return base_u + side_off + j * side_bytes; }
    BSG_DEV uint32_t full(int i) const { return base_u + bar_off + 8 * i; }
    BSG_DEV uint32_t empty(int i) const { return base_u + bar_off + 8 * (stages + i); }
    BSG_DEV uint32_t sfull(int j) const { return base_u + bar_off + 8 * (2 * stages + j); }
    BSG_DEV uint32_t sempty(int j) const { return base_u + bar_off + 8 * (2 * stages + 4 + j); }
    // failure word: set by a warp whose bounded wait ran out (read once, at the CTA's end)
    BSG_DEV volatile uint32_t* abort_word() const {
      return reinterpret_cast<volatile uint32_t*>(base + bar_off + 8 * (2 * stages + 8));
    }
  };

  // Position in a CTA's stream-K range: stage ks of `tile`.  The side ring holds one box of
  // scales / zero points per 2^rs_log2 stages of a tile; a stage opens a box when it is the
  // first of the CTA's segment on that tile or the first of its box, and closes it when it is
  // the last of the segment or of the box.  Producer and consumers walk the same sequence.
  struct Walk {
    int64_t tile;
    int ks, spt, rsm;
    BSG_DEV bool opens(bool seg_first) const { return seg_first || (ks & rsm) == 0; }
    BSG_DEV bool closes(bool seg_last) const { return seg_last || ((ks + 1) & rsm) == 0; }
    BSG_DEV void next() {
      if (++ks == spt) {
        ks = 0;
        ++tile;
      }
    }
  };

  // Ring position: slot index and the parity of its current use.
  struct Ring {
    int slot;
    uint32_t phase;
    int size;
    BSG_DEV void next() {
      if (++slot == size) {
        slot = 0;
        phase ^= 1u;
      }
    }
  };

  // ---- producer: warp 0.  Lane 0 copies each stage's weight boxes [64 rows][128 B] (one TMA
  // per half of the tile and k-box; L2 evict-first: the weight is read once) and, once per side
  // box, the scale box [tile rows][64 B] and zero-point box [tile rows][16 or 32 B] (two more
  // TMAs on the side ring).  All 32 lanes copy the
  // stage's activations [M][k of the stage] with 16-byte cp.async, tracked by the stage's full
  // barrier (cp.async.mbarrier.arrive).  Rows past N and k past K are zero-filled.
  //
  // Programmatic dependent launch: while the previous kernel in the stream is still finishing,
  // the first ring slots are filled with everything that is weight (W boxes, side boxes); only
  // after pdl_wait are their activations copied and the slots released to the consumers.  That
  // prefill never waits on a consumer release (which could not come before pdl_wait).
  static BSG_DEV void act_copy(const KParams& p, uint32_t dst, int ks, int lane) {
    constexpr int kUpr = kKc / 8;  // 16-byte activation units per row per stage
    const int units = p.M * kUpr;
    const int64_t k0 = static_cast<int64_t>(ks) * kKc, K = p.K;
    for (int u = lane; u < units; u += 32) {
      const int m = u / kUpr, qg = u % kUpr;
      const uint32_t d = dst + m * kActPitch + qg * 16;
      const int64_t k = k0 + qg * 8;
      const bool in = k < K;
      cp_async16(d, p.A + m * K + (in ? k : 0), in ? 16u : 0u);
    }
  }

  // The weight boxes of stage (tile, ks) into ring slot i (lane 0): one [64 rows][128 B] box
  // per half of the tile and k-box of the stage.  (A k-box wholly past the row, in the ragged
  // last stage, is filled with zeros like any out-of-range part of a box.)
  static BSG_DEV void weight_copy(const KParams& p, const Smem& sm, int i, const Walk& w,
                                  uint64_t pol) {
    const int row = static_cast<int>(w.tile * kRows);
#pragma unroll
    for (int j = 0; j < kKb; ++j)
#pragma unroll
      for (int h = 0; h < kH; ++h)
        tma_load_2d_hint(sm.w(i) + (j * kH + h) * kBoxB, &p.tm_w,
                         w.ks * kSrb + j * kBoxRowBytes, row + h * kBoxRows, sm.full(i), pol);
  }

  // The side boxes of the box holding stage (tile, ks) into side slot j (lane 0).  With one half
  // they keep the normal L2 policy: a box reads 64 bytes of a row's scales (16 or 32 of its zero
  // points), and the rest of the row's L2 line, fetched from DRAM with them, is what the next box
  // of the same rows reads a few stages later (measured on GB300: 1-4 % faster than evict-first,
  // which loses that rest to the streaming weights and reads it again).  With two halves they are
  // evict-first like the weights (the normal policy measured 2-4 % slower on the int4 lm_head,
  // though its DRAM reads fell from 1.055 to 1.011 of the algorithmic bytes).
  static BSG_DEV void side_copy(const KParams& p, const Smem& sm, int j, const Walk& w,
                                uint64_t pol) {
    const uint32_t full = sm.sfull(j), dst = sm.side_u(j);
    const int bx = w.ks >> p.rs_log2;
    const int row = static_cast<int>(w.tile * kRows);
    mbar_arrive_expect_tx(full, static_cast<uint32_t>(p.side_tx));
    if constexpr (kH == 1) {
      tma_load_2d(dst, &p.tm_s, bx * kSideScaleBytes, row, full);
      if constexpr (ZP)
        tma_load_2d(dst + kRows * kSideScaleBytes, &p.tm_z, bx * p.zbox_bytes, row, full);
    } else {
      tma_load_2d_hint(dst, &p.tm_s, bx * kSideScaleBytes, row, full, pol);
      if constexpr (ZP)
        tma_load_2d_hint(dst + kRows * kSideScaleBytes, &p.tm_z, bx * p.zbox_bytes, row, full,
                         pol);
    }
  }

  // Failure handling.  Every wait is bounded (KParams::wait_ns).  A consumer warp that gives up
  // records it in the CTA's failure word and from then on neither reads nor releases its ring
  // slots, so the copy warp's own wait for a free slot runs out in turn and it stops issuing
  // (a slot is never refilled while a copy into it may be in flight).  After both roles have
  // returned, the CTA's copy warp -- only when the failure word is set -- waits, bounded again,
  // until every copy it issued has landed (pending weight and side boxes are tracked per ring
  // slot with the parity of their use), so that no asynchronous copy outlives the CTA; on the
  // normal path the consumers have waited for every copy already.  A test hook
  // (KParams::skip_stage) makes CTA 0's copy warp leave out one stage of its range entirely, so
  // that the consumers' wait on it runs out.
  struct Pending {
    uint32_t wmask = 0, wpar = 0, smask = 0, spar = 0;  // weight / side slots, parity of the use
    BSG_DEV void weight(int slot, uint32_t phase) {
      wmask |= 1u << slot;
      wpar = (wpar & ~(1u << slot)) | (phase << slot);
    }
    BSG_DEV void side(int slot, uint32_t phase) {
      smask |= 1u << slot;
      spar = (spar & ~(1u << slot)) | (phase << slot);
    }
  };

  // Lane 0 (which issued them) waits until the tracked weight and side copies have landed.
  static BSG_DEV void drain(const KParams& p, const Smem& sm, const Pending& pd, int lane) {
    if (lane != 0) return;
    for (int s = 0; s < sm.stages; ++s)
      if ((pd.wmask >> s) & 1u)
        mbar_wait(sm.full(s), (pd.wpar >> s) & 1u, p.err, kErrTimeoutFull, p.wait_ns);
    for (int j = 0; j < sm.side_slots; ++j)
      if ((pd.smask >> j) & 1u)
        mbar_wait(sm.sfull(j), (pd.spar >> j) & 1u, p.err, kErrTimeoutFull, p.wait_ns);
  }

  // Returns with the copy warp's record of what it issued (for the end-of-CTA drain).
  static BSG_DEV Pending produce(const KParams& p, const Smem& sm, int64_t s0, int64_t s1,
                                 int lane) {
    const bool side = p.side_tma != 0;
    if (lane == 0) {
      prefetch_tmap(&p.tm_w);
      if (side) {
        prefetch_tmap(&p.tm_s);
        if constexpr (ZP) prefetch_tmap(&p.tm_z);
      }
    }
    const uint64_t pol = policy_evict_first();
    const int spt = p.spt;
    const int n = static_cast<int>(s1 - s0);
    const int64_t tile0 = s0 / spt;
    const Walk start{tile0, static_cast<int>(s0 - tile0 * spt), spt, (1 << p.rs_log2) - 1};
    Ring sr{sm.side_slots - 1, 1u, sm.side_slots};  // side ring: advanced before each use
    const int skip = blockIdx.x == 0 ? p.skip_stage : -1;  // test hook (-1: none)
    Pending pd;

    // phase 1: weights (and side boxes) of the first `pre` stages; fresh slots, no waits
    int pre = 0;
    {
      Walk w = start;
      int boxes = 0;
      const int lim = n < sm.stages ? n : sm.stages;
      for (int i = 0; i < lim; ++i) {
        const bool seg_first = (i == 0) || (w.ks == 0);
        if (side && w.opens(seg_first)) {
          if (boxes == sm.side_slots) break;  // the next box would reuse a slot: wait for phase 3
          ++boxes;
          sr.next();
          if (lane == 0) side_copy(p, sm, sr.slot, w, pol);
          pd.side(sr.slot, sr.phase);
        }
        if (i != skip) {
          if (lane == 0) {
            mbar_expect_tx(sm.full(i), kStageB);
            weight_copy(p, sm, i, w, pol);
          }
          pd.weight(i, 0u);
        }
        pre = i + 1;
        w.next();
      }
    }
    pdl_wait();
    // phase 2: activations of those stages; lane 0's arrival then releases each slot
    Walk w = start;
    for (int i = 0; i < pre; ++i) {
      if (i != skip) {
        act_copy(p, sm.act_u(i), w.ks, lane);
        cp_async_mbar_arrive(sm.full(i));
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.full(i));
      }
      w.next();
    }
    // phase 3: steady state
    Ring r{pre % sm.stages, pre == sm.stages ? 1u : 0u, sm.stages};
    bool ok = true;
    for (int i = pre; i < n; ++i) {
      const bool seg_first = (i == 0) || (w.ks == 0);
      if (side && w.opens(seg_first)) {
        sr.next();
        ok = mbar_wait(sm.sempty(sr.slot), sr.phase ^ 1u, p.err, kErrTimeoutEmpty, p.wait_ns);
        if (!ok) break;
        if (lane == 0) side_copy(p, sm, sr.slot, w, pol);
        pd.side(sr.slot, sr.phase);
      }
      ok = mbar_wait(sm.empty(r.slot), r.phase ^ 1u, p.err, kErrTimeoutEmpty, p.wait_ns);
      if (!ok) break;
      const uint32_t full = sm.full(r.slot);
      if (i != skip) {
        act_copy(p, sm.act_u(r.slot), w.ks, lane);
        cp_async_mbar_arrive(full);
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(full, kStageB);
          weight_copy(p, sm, r.slot, w, pol);
        }
        pd.weight(r.slot, r.phase);
      }
      r.next();
      w.next();
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (!ok && lane == 0) *sm.abort_word() = 1u;
    return pd;
  }

  // ---- per-lane constants.  Consumer warp cw owns mma row group rg = cw of every half of the
  // tile (rows 64 h + 16 rg .. 64 h + 16 rg + 15, h < kH) over the whole stage (kCps = 8 chunks
  // of 16 bytes per row and k-box); lane (g, t) holds rows g and g + 8 of the group (rr = 0, 1).
  struct Lane {
    int rg, lane, g, t;
    uint32_t w[4];             // ldmatrix.x4 row address of chunk pair j (chunks 2j, 2j + 1) in
                               // the weight box of half 0; half h adds h * kBoxB
    uint32_t act[MT];          // activation fragment offset of chunk 0 (n8 tile mt) in a stage's
                               // activation slot; chunk c adds c * kActChunkB
    uint32_t fsel[2];          // NVFP4: prmt selector of the lane's scale code, chunk parity 0/1
    uint32_t srow;             // side box: scale row 16 rg + g (half 0); row g + 8 adds
                               // 8 * kSideScaleBytes, half h adds h * kBoxRows * kSideScaleBytes
    uint32_t zrow;             // side box: zero-point row 16 rg + g (half 0); row g + 8 adds
                               // 8 * kZboxB, half h adds h * kBoxRows * kZboxB
    uint32_t cact;             // CUDA-core variant: the lane's k positions of a chunk in an
                               // activation row (4 or 8 halves from byte t * kActChunkB / 4)
  };

  static BSG_DEV Lane make_lane(const KParams& p, int cw, int lane) {
    Lane L;
    L.rg = cw;
    L.lane = lane;
    L.g = lane >> 2;
    L.t = lane & 3;
    // ldmatrix.x4: lanes 8i .. 8i + 7 address matrix i = (rows +8 if i odd) x (chunk +1 if i >= 2)
    const int i = lane >> 3;
    const int r = 16 * L.rg + 8 * (i & 1) + (lane & 7);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = 2 * j + (i >> 1);
      L.w[j] = r * kBoxRowBytes + ((c ^ (r & 7)) << 4);
    }
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      // activation row of the B fragment column; columns past M read row 0 (their results are
      // never stored), so the slot holds only the call's M rows.  Lane t reads k 8t .. 8t + 7
      // (4-bit formats) or 4t .. 4t + 3 (8-bit) of the chunk.
      const int m0 = mt * 8 + L.g;
      const int m = m0 < p.M ? m0 : 0;
      L.act[mt] = m * kActPitch + L.t * (kActChunkB / 4);
    }
    // chunk c's codes lie in 16-block 2c + t/2 of the stage: byte 2 (c & 1) + t/2 of word c / 2
    L.fsel[0] = 0x11u * static_cast<uint32_t>(L.t >> 1);
    L.fsel[1] = 0x11u * static_cast<uint32_t>(2 + (L.t >> 1));
    L.srow = (16 * L.rg + L.g) * kSideScaleBytes;
    L.zrow = kRows * kSideScaleBytes + (16 * L.rg + L.g) * kZboxB;
    L.cact = L.t * (kActChunkB / 4);
    return L;
  }

  // Offset of chunk c's activation fragment (n8 tile mt) in a stage's activation slot.
  static BSG_DEV uint32_t act_off(const Lane& L, int c, int mt) {
    return L.act[mt] + c * kActChunkB;
  }

  // Launch parameters the stage loop reads, as registers.  SIDE (fixed per launch, taken out of
  // the loop): scales and zero points come from the side ring, else straight from global memory.
  template <bool SIDE>
  struct Run {
    static constexpr bool side = SIDE;
    int bs_log2, rs_log2, zbox_bytes;
    const KParams& k;  // the rest, read where used (global-memory path)
  };

  template <class R>
  static BSG_DEV int64_t row_of(const R& p, const Lane& L, int64_t tile, int h, int rr) {
    const int64_t n = tile * kRows + h * kBoxRows + 16 * L.rg + L.g + 8 * rr;
    return n < p.k.N ? n : p.k.N - 1;
  }

  // fp32 scales of the lane's 2 rows for NB consecutive blocks from global memory, at absolute
  // block `blk` (the path for scale arrays whose pitch a tensor map cannot describe).
  template <int NB, class R>
  static BSG_DEV void load_scales(const R& p, const Lane& L, int64_t tile, int h, int blk,
                                  float (&s)[NB][2]) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const uint8_t* src = p.k.scales + row_of(p, L, tile, h, rr) * p.k.scale_pitch;
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const int b = blk + u;
        if (b >= p.k.nb_s) {  // chunk past K in the ragged last stage: its weight is zero
          s[u][rr] = 0.f;
        } else if constexpr (FMT == kFp8) {
          s[u][rr] = __ldg(reinterpret_cast<const float*>(src) + b);
        } else {
          s[u][rr] = __half2float(__ldg(reinterpret_cast<const __half*>(src) + b));
        }
      }
    }
  }

  // Zero points of the lane's 2 rows for NB consecutive blocks from global memory (same
  // addressing as load_scales), packed: block u at bit u * kZpW.  Without zero points: the
  // implicit 2^(bits-1) of every block.
  static constexpr uint32_t kNoZp = (FMT == kInt4) ? 0x88888888u : 0x80808080u;

  template <int NB, class R>
  static BSG_DEV void load_zp(const R& p, const Lane& L, int64_t tile, int h, int blk,
                              uint32_t (&z)[2]) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      if constexpr (!ZP) {
        z[rr] = kNoZp;
      } else {
        uint32_t v = 0;
        const uint8_t* src = p.k.zp + row_of(p, L, tile, h, rr) * p.k.zp_pitch;
#pragma unroll
        for (int u = 0; u < NB; ++u) {
          const int b = blk + u;
          uint32_t q = 0;
          if (b < p.k.nb_s) {
            const uint32_t byte = __ldg(src + ((FMT == kInt4) ? (b >> 1) : b));
            q = (FMT == kInt4) ? ((b & 1) ? (byte >> 4) : (byte & 0xFu)) : byte;
          }
          v |= q << (u * kZpW);
        }
        z[rr] = v;
      }
    }
  }

  // A stage's shared-memory operands: the kernel's shared array (generic pointer, so that plain
  // loads through it stay shared-memory loads) and 32-bit offsets into it of the stage's
  // activation slot and side box.
  struct Sh {
    const uint8_t* base;
    uint32_t a, s;
  };

  // Scales and zero points of the lane's 2 rows for NB consecutive blocks of a side box, in one
  // shared load per row each (NB a power of two; the first block `rel` a multiple of NB, so the
  // loads are aligned): f16 scale pairs (or the fp32 scale of FP8, NB = 1) and zero points
  // packed at kZpW bits per block, as stored.
  template <int NB>
  struct SideLoad {
    uint32_t s[2][(NB + 1) / 2];
    uint32_t z[2][(NB * kZpW + 31) / 32];
  };

  template <int NB>
  static BSG_DEV void load_side(const Lane& L, const Sh& sh, int h, int rel, SideLoad<NB>& v) {
    const uint32_t sa = sh.s + L.srow + h * (kBoxRows * kSideScaleBytes) + rel * kScaleEs;
    const uint32_t za0 = sh.s + L.zrow + h * (kBoxRows * kZboxB) + ((rel * kZpW) >> 3);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const uint8_t* a = sh.base + (sa + rr * 8 * kSideScaleBytes);
      if constexpr (FMT == kFp8) {
        static_assert(NB == 1, "one fp32 scale per weight box");
        v.s[rr][0] = lsh<uint32_t>(a);
      } else if constexpr (NB == 1) {
        v.s[rr][0] = lsh<uint16_t>(a);
      } else if constexpr (NB == 2) {
        v.s[rr][0] = lsh<uint32_t>(a);
      } else if constexpr (NB == 4) {
        const uint2 x = lsh<uint2>(a);
        v.s[rr][0] = x.x;
        v.s[rr][1] = x.y;
      } else {
        static_assert(NB == 8, "at most 8 blocks per side load");
        const uint4 x = lsh<uint4>(a);
        v.s[rr][0] = x.x;
        v.s[rr][1] = x.y;
        v.s[rr][2] = x.z;
        v.s[rr][3] = x.w;
      }
      if constexpr (ZP) {
        const uint8_t* za = sh.base + (za0 + rr * 8 * kZboxB);
        constexpr int kBits = NB * kZpW;
        if constexpr (kBits == 4) {
          v.z[rr][0] = static_cast<uint32_t>(lsh<uint8_t>(za)) >> ((rel & 1) * 4);
        } else if constexpr (kBits == 8) {
          v.z[rr][0] = lsh<uint8_t>(za);
        } else if constexpr (kBits == 16) {
          v.z[rr][0] = lsh<uint16_t>(za);
        } else if constexpr (kBits == 32) {
          v.z[rr][0] = lsh<uint32_t>(za);
        } else {
          const uint2 x = lsh<uint2>(za);
          v.z[rr][0] = x.x;
          v.z[rr][1] = x.y;
        }
      }
    }
  }

  // The scales (fp32) and packed zero points of blocks b0 .. b0 + NG - 1 of a side load.
  template <int NG, int NB>
  static BSG_DEV void side_group(const SideLoad<NB>& v, int b0, uint32_t (&z)[2],
                                 float (&s)[NG][2]) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
#pragma unroll
      for (int u = 0; u < NG; ++u) {
        const int b = b0 + u;
        if constexpr (FMT == kFp8) {
          s[u][rr] = __uint_as_float(v.s[rr][0]);
        } else {
          const __half2 two = *reinterpret_cast<const __half2*>(&v.s[rr][b >> 1]);
          s[u][rr] = (b & 1) ? __high2float(two) : __low2float(two);
        }
      }
      if constexpr (ZP) {
        const int bit = b0 * kZpW;  // a group's zero points never straddle a word
        z[rr] = v.z[rr][bit >> 5] >> (bit & 31);
      } else {
        z[rr] = kNoZp;
      }
    }
  }

  // Zero-point operand constants (see zp_consts) of the lane's 2 rows for block u of `z`.
  static BSG_DEV void zp_of(const uint32_t (&z)[2], int u, uint32_t (&zl)[2], uint32_t (&zh)[2]) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
      zp_consts<FMT, BF16>((z[rr] >> (u * kZpW)) & ((1u << kZpW) - 1u), zl[rr], zh[rr]);
  }

  // NVFP4: the replicated f16 E4M3 block scale of the lane's 2 rows for 16-block `blk` (side
  // box block `rel`).
  template <class R>
  static BSG_DEV void load_fold(const R& p, const Lane& L, const Sh& sh, int64_t tile, int h,
                                int blk, int rel, uint32_t (&f)[2]) {
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      uint32_t code;
      if constexpr (R::side) {
        code = lsh<uint8_t>(sh.base + (sh.s + L.srow + h * (kBoxRows * kSideScaleBytes) +
                                       rr * 8 * kSideScaleBytes + rel));
      } else {
        code = (blk < p.k.nb_s)
                   ? __ldg(p.k.scales + row_of(p, L, tile, h, rr) * p.k.scale_pitch + blk)
                   : 0u;
      }
      f[rr] = e4m3x2_to_f16x2(code * 0x0101u);
    }
  }

  // Activation B fragments of chunk c: b[mt][st][0] = (k 2t, 2t+1), b[mt][st][1] = (k 2t+8,
  // 2t+9) of activation row mt*8 + g, permuted like the weight (phys_k).
  static BSG_DEV void act_fragment(const Lane& L, const Sh& sh, int c,
                                   uint32_t (&b)[MT][kSteps][2]) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      if constexpr (kFour) {
        const uint4 v = lsh<uint4>(sh.base + (sh.a + act_off(L, c, mt)));
        if constexpr (FMT == kInt4) {  // pairs (8t+j, 8t+j+4)
          b[mt][0][0] = prmt<0x5410u>(v.x, v.z);
          b[mt][0][1] = prmt<0x7632u>(v.x, v.z);
          b[mt][1][0] = prmt<0x5410u>(v.y, v.w);
          b[mt][1][1] = prmt<0x7632u>(v.y, v.w);
        } else {  // nvfp4: natural pairs
          b[mt][0][0] = v.x;
          b[mt][0][1] = v.y;
          b[mt][1][0] = v.z;
          b[mt][1][1] = v.w;
        }
      } else {
        const uint2 v = lsh<uint2>(sh.base + (sh.a + act_off(L, c, mt)));
        b[mt][0][0] = v.x;
        b[mt][0][1] = v.y;
      }
    }
  }

  // Decode chunk words lo (row g), hi (row g + 8) and multiply them with the chunk's activation
  // fragments b into d[u] (u: sub-block when a chunk holds two scale blocks).  ZC: the first
  // k-step starts from zero instead of accumulating.  zl/zh: zero-point constants (int formats)
  // or the fold scales (NVFP4) of rows g, g + 8.
  template <bool ZC, int NS>
  static BSG_DEV void chunk_mma(const Lane& L, const uint32_t (&b)[MT][kSteps][2], uint32_t lo,
                                uint32_t hi, const uint32_t (&zl)[2], const uint32_t (&zh)[2],
                                float (&d)[NS][MT][4]) {
    static_assert(NS == kSub, "one accumulator per scale block of the chunk");
    uint32_t a[kSteps][4];
    if constexpr (FMT == kInt4) {
      decode_int4<BF16>(lo, hi, zl[0], zh[0], zl[1], zh[1], a);
    } else if constexpr (FMT == kInt8) {
      decode_int8<BF16>(lo, hi, zl[0], zl[1], a);
    } else if constexpr (FMT == kFp8) {
      decode_fp8<BF16>(lo, hi, a);
    } else {
      decode_nvfp4<BF16>(lo, hi, zl[0], zl[1], a);
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
          if (zc) mma16816_zc<BF16>(d[u][mt], a[st], b0, b1);
          else mma16816<BF16>(d[u][mt], a[st], b0, b1);
        }
      }
  }

  // acc += tmp * s (fragment entries 0, 1: row g; 2, 3: row g + 8).  With two or more n8 tiles
  // the row's pairs go through packed fp32 FMAs (fma.rn.f32x2: the same rounding per element,
  // half the instructions once the scale pair is built).
  static BSG_DEV void apply_scales(float s0, float s1, const float (&tmp)[MT][4], float (&acc)[MT][4]) {
    if constexpr (MT >= 2) {
      const uint64_t p0 = f32x2(s0, s0), p1 = f32x2(s1, s1);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint64_t a01 = f32x2(acc[mt][0], acc[mt][1]), a23 = f32x2(acc[mt][2], acc[mt][3]);
        fma_f32x2(a01, f32x2(tmp[mt][0], tmp[mt][1]), p0);
        fma_f32x2(a23, f32x2(tmp[mt][2], tmp[mt][3]), p1);
        acc[mt][0] = f32x2_lo(a01);
        acc[mt][1] = f32x2_hi(a01);
        acc[mt][2] = f32x2_lo(a23);
        acc[mt][3] = f32x2_hi(a23);
      }
    } else {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        acc[mt][0] = fmaf(tmp[mt][0], s0, acc[mt][0]);
        acc[mt][1] = fmaf(tmp[mt][1], s0, acc[mt][1]);
        acc[mt][2] = fmaf(tmp[mt][2], s1, acc[mt][2]);
        acc[mt][3] = fmaf(tmp[mt][3], s1, acc[mt][3]);
      }
    }
  }

  static BSG_DEV void zero(float (&x)[MT][4]) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) x[mt][i] = 0.f;
  }

  // Consume one stage, stage ks of `tile`: per k-box, the kCps = 8 chunks of row group rg in
  // every half (consume_box; `wa` is the box's weight slot, a shared-window address for ldmatrix,
  // half h's box at wa + h * kBoxB; `ap` the activation slot and side box; k0 and kb the box's
  // first k in the row and in the side box).  Each chunk's activation fragment is loaded once
  // and multiplied with the weights of every half.
  //
  // Scale groups (CPB = chunks per scale block): the chunks are taken in groups that share one
  // shared-memory load of scales and zero points per row -- a pair of chunks for CPB = 1 and 2,
  // four for CPB = 4, the whole box for CPB = 8 (blocks of eight chunks or longer), one chunk
  // holding two blocks for CPB = 0.  Within a block the chunk products are summed on the tensor
  // cores and then scaled into acc.
  static constexpr int kGC = (CPB == 0) ? 1 : (CPB <= 2 ? 2 : CPB);  // chunks per group
  static constexpr int kGB = (CPB == 0 || CPB == 1) ? 2 : 1;          // blocks per group

  template <class R>
  static BSG_DEV void consume_stage(const R& p, const Lane& L, uint32_t wa, const Sh& ap,
                                    int64_t tile, int ks, float (&acc)[kH][MT][4],
                                    uint64_t (&cacc)[kH][2][kCcCols]) {
    const int k0 = ks * kKc;                                // first k of the stage in the row
    const int kb = (ks & ((1 << p.rs_log2) - 1)) * kKc;    // ... in the side box
    uint32_t wv[kH][4][4];  // ldmatrix words: chunk c, row g in wv[h][c >> 1][2 (c & 1)]
    // k-box j of the stage: its boxes at wa + j kH kBoxB, its activations kCps chunks further
#pragma unroll
    for (int j = 0; j < kKb; ++j) {
      const uint32_t wj = wa + j * kH * kBoxB;
      const Sh aj{ap.base, ap.a + j * kCps * kActChunkB, ap.s};
      if constexpr (CC > 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) load_pair(L, wj, q, wv);
        consume_box_cc(p, L, wv, aj, tile, k0 + j * kBoxK, kb + j * kBoxK, cacc);
      } else {
        consume_box(p, L, wj, wv, aj, tile, k0 + j * kBoxK, kb + j * kBoxK, acc);
      }
    }
  }

  // The ldmatrix words of chunk pair j (chunks 2j, 2j + 1, rows g and g + 8) of every half.
  // (ldmatrix is a volatile asm: the loads stay where they are written, so the consumer loop
  // issues each pair's loads one pair ahead of its use and keeps two pairs of registers live.)
  static BSG_DEV void load_pair(const Lane& L, uint32_t wa, int j, uint32_t (&wv)[kH][4][4]) {
    const uint32_t wl = wa + L.w[j];
    ldsm_x4_at<0>(wl, wv[0][j][0], wv[0][j][1], wv[0][j][2], wv[0][j][3]);
    if constexpr (kH == 2)
      ldsm_x4_at<kBoxB>(wl, wv[1][j][0], wv[1][j][1], wv[1][j][2], wv[1][j][3]);
  }

  // The box's first ldmatrix words: with one half all four pairs at once (16 registers, the
  // most loads in flight); with two halves the first pair, the others one pair ahead of their use
  // (prefetch), which keeps 16 registers live instead of 32.
  static BSG_DEV void first_pairs(const Lane& L, uint32_t wa, uint32_t (&wv)[kH][4][4]) {
    if constexpr (kH == 1) {
#pragma unroll
      for (int j = 0; j < 4; ++j) load_pair(L, wa, j, wv);
    } else {
      load_pair(L, wa, 0, wv);
    }
  }

  // Chunk c is about to be multiplied: with two halves, when it opens a chunk pair, load the next
  // pair's words.
  static BSG_DEV void prefetch(const Lane& L, uint32_t wa, int c, uint32_t (&wv)[kH][4][4]) {
    if constexpr (kH == 2)
      if ((c & 1) == 0 && (c >> 1) + 1 < 4) load_pair(L, wa, (c >> 1) + 1, wv);
  }

  template <class R>
  static BSG_DEV void consume_box(const R& p, const Lane& L, uint32_t wa,
                                  uint32_t (&wv)[kH][4][4], const Sh& ap, int64_t tile,
                                  int k0, int kb, float (&acc)[kH][MT][4]) {
#define BSG_LO(h, c) wv[h][(c) >> 1][2 * ((c) & 1)]
#define BSG_HI(h, c) wv[h][(c) >> 1][2 * ((c) & 1) + 1]
    uint32_t zh[2] = {0u, 0u};
    first_pairs(L, wa, wv);
    if constexpr (kFold) {
      // the lane's 8 codes of chunk c lie in 16-block (k of the chunk + 8t) / 16 = 2c + t/2
      if constexpr (R::side) {
        // the box's 16 scale codes per row (2 per chunk) in one load per half; the lane's code
        // picked by prmt
        uint4 cv[kH][2];
#pragma unroll
        for (int h = 0; h < kH; ++h)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr)
            cv[h][rr] = lsh<uint4>(ap.base + (ap.s + L.srow + h * (kBoxRows * kSideScaleBytes) +
                                              rr * 8 * kSideScaleBytes + (kb >> 4)));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          prefetch(L, wa, c, wv);
          uint32_t b[MT][kSteps][2];
          act_fragment(L, ap, c, b);
#pragma unroll
          for (int h = 0; h < kH; ++h) {
            uint32_t f[2];
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const uint32_t wd = (c >> 1) == 0 ? cv[h][rr].x
                                : (c >> 1) == 1 ? cv[h][rr].y
                                : (c >> 1) == 2 ? cv[h][rr].z : cv[h][rr].w;
              f[rr] = e4m3_byte_to_f16x2(wd, L.fsel[c & 1]);
            }
            chunk_mma<false>(L, b, BSG_LO(h, c), BSG_HI(h, c), f, zh,
                             reinterpret_cast<float (&)[1][MT][4]>(acc[h]));
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          prefetch(L, wa, c, wv);
          uint32_t b[MT][kSteps][2];
          act_fragment(L, ap, c, b);
          const int d = 2 * c + (L.t >> 1);
#pragma unroll
          for (int h = 0; h < kH; ++h) {
            uint32_t f[2];
            load_fold(p, L, ap, tile, h, (k0 >> 4) + d, (kb >> 4) + d, f);
            chunk_mma<false>(L, b, BSG_LO(h, c), BSG_HI(h, c), f, zh,
                             reinterpret_cast<float (&)[1][MT][4]>(acc[h]));
          }
        }
      }
    } else {
      // side ring: one load per row and half of the scales and zero points of up to 8 blocks
      // (the whole box, or half of it for 16-element int4 blocks)
      constexpr int kBB = (8 / kGC) * kGB;         // scale blocks per box
      constexpr int kSL = kBB < 8 ? kBB : 8;       // blocks per side load
      constexpr int kGpl = kSL / kGB;              // groups per side load
      SideLoad<kSL> sl[kH];
#pragma unroll
      for (int grp = 0; grp < 8 / kGC; ++grp) {
        const int kg = grp * kGC * kKpc;  // k of the group in the box
        uint32_t z[kH][2];
        float s[kH][kGB][2];
#pragma unroll
        for (int h = 0; h < kH; ++h) {
          if constexpr (R::side) {
            if (grp % kGpl == 0) {
              int rel;
              if constexpr (kBsLog2 >= 0) rel = (kb + kg) >> kBsLog2;
              else rel = (kb + kg) >> p.bs_log2;
              load_side<kSL>(L, ap, h, rel, sl[h]);
            }
            side_group<kGB>(sl[h], (grp % kGpl) * kGB, z[h], s[h]);
          } else {
            const int blk = (k0 + kg) >> p.bs_log2;
            load_zp<kGB>(p, L, tile, h, blk, z[h]);
            load_scales<kGB>(p, L, tile, h, blk, s[h]);
          }
        }
        uint32_t zl[2], zhh[2];
        if constexpr (CPB == 0) {  // one chunk, two blocks: the lane's codes are in block t/2
          prefetch(L, wa, grp, wv);
          uint32_t b[MT][kSteps][2];
          act_fragment(L, ap, grp, b);
#pragma unroll
          for (int h = 0; h < kH; ++h) {
            zp_of(z[h], L.t >> 1, zl, zhh);
            float tmp[2][MT][4];
            chunk_mma<true>(L, b, BSG_LO(h, grp), BSG_HI(h, grp), zl, zhh, tmp);
            apply_scales(s[h][0][0], s[h][0][1], tmp[0], acc[h]);
            apply_scales(s[h][1][0], s[h][1][1], tmp[1], acc[h]);
          }
        } else if constexpr (CPB == 1) {  // two chunks, one block each
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c = grp * 2 + u;
            prefetch(L, wa, c, wv);
            uint32_t b[MT][kSteps][2];
            act_fragment(L, ap, c, b);
#pragma unroll
            for (int h = 0; h < kH; ++h) {
              zp_of(z[h], u, zl, zhh);
              float tmp[1][MT][4];
              chunk_mma<true>(L, b, BSG_LO(h, c), BSG_HI(h, c), zl, zhh, tmp);
              apply_scales(s[h][u][0], s[h][u][1], tmp[0], acc[h]);
            }
          }
        } else {  // CPB 2, 4 or 8: kGC chunks in one block, one mma chain per half
          float t[kH][1][MT][4];
#pragma unroll
          for (int u = 0; u < kGC; ++u) {
            const int c = grp * kGC + u;
            prefetch(L, wa, c, wv);
            uint32_t b[MT][kSteps][2];
            act_fragment(L, ap, c, b);
#pragma unroll
            for (int h = 0; h < kH; ++h) {
              zp_of(z[h], 0, zl, zhh);
              if (u == 0) chunk_mma<true>(L, b, BSG_LO(h, c), BSG_HI(h, c), zl, zhh, t[h]);
              else chunk_mma<false>(L, b, BSG_LO(h, c), BSG_HI(h, c), zl, zhh, t[h]);
            }
          }
#pragma unroll
          for (int h = 0; h < kH; ++h) apply_scales(s[h][0][0], s[h][0][1], t[h][0], acc[h]);
        }
      }
    }
#undef BSG_LO
#undef BSG_HI
  }

  // ---- CUDA-core variant.  Lane (g, t) holds, for tile rows g and g + 8, the codes of its own k
  // positions of every chunk (the words ldmatrix hands it), decoded by the same exact decoders
  // as the mma path.  Each decoded 16-bit pair becomes an fp32 pair times the row's block scale
  // (exact for the int formats: at most 9 + 11 significand bits) and is multiplied into the
  // packed partial sums cacc[rr][m] -- one per tile row rr and activation row m, its halves the
  // pair's two k -- with the activations of the same k of row m: one fma.rn.f32x2 per pair, tile
  // row and activation row.  The quad's four lanes cover the chunk's k; their sums are added at
  // the end of a tile segment (cc_fragment).
  template <class R>
  static BSG_DEV void chunk_cc(const R& p, const Lane& L, const Sh& ap, int c, uint32_t lo,
                               uint32_t hi, const uint32_t (&zl)[2], const uint32_t (&zh)[2],
                               const float (&sc)[2], uint64_t (&cacc)[2][kCcCols]) {
    uint32_t a[kSteps][4];
    if constexpr (FMT == kInt4) {
      decode_int4<BF16>(lo, hi, zl[0], zh[0], zl[1], zh[1], a);
    } else if constexpr (FMT == kInt8) {
      decode_int8<BF16>(lo, hi, zl[0], zl[1], a);
    } else if constexpr (FMT == kFp8) {
      decode_fp8<BF16>(lo, hi, a);
    } else {
      decode_nvfp4<BF16>(lo, hi, zl[0], zl[1], a);
    }
    constexpr int kP = 2 * kSteps;  // k pairs of a lane per tile row and chunk
    uint64_t w[2][kP];
#pragma unroll
    for (int s = 0; s < kSteps; ++s)
#pragma unroll
      for (int rp = 0; rp < 2; ++rp)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const uint32_t h = a[s][2 * rp + rr];
          uint64_t v = f32x2(half_to_f32<BF16>(h, 0), half_to_f32<BF16>(h, 1));
          if constexpr (!kFold) v = mul_f32x2(v, f32x2(sc[rr], sc[rr]));
          w[rr][2 * s + rp] = v;
        }
#pragma unroll
    for (int m = 0; m < kCcCols; ++m) {
      if (m > 0 && m >= p.k.M) break;
      // the lane's 8 (4-bit formats) or 4 (8-bit) activation halves of chunk c, row m
      const uint8_t* src = ap.base + (ap.a + m * kActPitch + c * kActChunkB + L.cact);
      uint32_t x[kFour ? 4 : 2];
      if constexpr (kFour) {
        const uint4 v = lsh<uint4>(src);
        x[0] = v.x;
        x[1] = v.y;
        x[2] = v.z;
        x[3] = v.w;
      } else {
        const uint2 v = lsh<uint2>(src);
        x[0] = v.x;
        x[1] = v.y;
      }
#pragma unroll
      for (int s = 0; s < kSteps; ++s)
#pragma unroll
        for (int rp = 0; rp < 2; ++rp) {
          // halves j0, j1 of x hold the pair's two k (phys_k, relative to the lane's first k)
          const int j0 = phys_k<FMT>(s, rp, 0, 0), j1 = phys_k<FMT>(s, rp, 1, 0);
          const uint64_t xa = f32x2(half_to_f32<BF16>(x[j0 >> 1], j0 & 1),
                                    half_to_f32<BF16>(x[j1 >> 1], j1 & 1));
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) fma_f32x2(cacc[rr][m], w[rr][2 * s + rp], xa);
        }
    }
  }

  // Zero points and scales of scale group `grp` of half h of a box (the same sources and
  // order as consume_box).
  template <int NS, class R>
  static BSG_DEV void group_side(const R& p, const Lane& L, const Sh& ap, int64_t tile, int h,
                                 int k0, int kb, int grp, SideLoad<NS>& sl, uint32_t (&z)[2],
                                 float (&s)[kGB][2]) {
    const int kg = grp * kGC * kKpc;  // k of the group in the box
    if constexpr (R::side) {
      constexpr int kGpl = NS / kGB;  // groups per side load
      if (grp % kGpl == 0) {
        int rel;
        if constexpr (kBsLog2 >= 0) rel = (kb + kg) >> kBsLog2;
        else rel = (kb + kg) >> p.bs_log2;
        load_side<NS>(L, ap, h, rel, sl);
      }
      side_group<kGB>(sl, (grp % kGpl) * kGB, z, s);
    } else {
      const int blk = (k0 + kg) >> p.bs_log2;
      load_zp<kGB>(p, L, tile, h, blk, z);
      load_scales<kGB>(p, L, tile, h, blk, s);
    }
  }

  // A box's chunks of every half on the CUDA cores (see chunk_cc), half by half.  Every
  // lane's codes of a chunk lie in one scale block: block t/2 of the chunk when it holds two
  // (16-element int4 blocks).
  template <class R>
  static BSG_DEV void consume_box_cc(const R& p, const Lane& L,
                                     const uint32_t (&wv)[kH][4][4], const Sh& ap,
                                     int64_t tile, int k0, int kb,
                                     uint64_t (&cacc)[kH][2][kCcCols]) {
#define BSG_LO(c) wv[h][(c) >> 1][2 * ((c) & 1)]
#define BSG_HI(c) wv[h][(c) >> 1][2 * ((c) & 1) + 1]
#pragma unroll
    for (int h = 0; h < kH; ++h) {
      uint32_t zl[2], zh[2] = {0u, 0u};
      if constexpr (kFold) {
        const float one[2] = {1.f, 1.f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int d = 2 * c + (L.t >> 1);
          load_fold(p, L, ap, tile, h, (k0 >> 4) + d, (kb >> 4) + d, zl);
          chunk_cc(p, L, ap, c, BSG_LO(c), BSG_HI(c), zl, zh, one, cacc[h]);
        }
      } else {
        constexpr int kBB = (8 / kGC) * kGB;    // scale blocks per box
        constexpr int kSL = kBB < 8 ? kBB : 8;  // blocks per side load
        SideLoad<kSL> sl;
#pragma unroll
        for (int grp = 0; grp < 8 / kGC; ++grp) {
          uint32_t z[2];
          float s[kGB][2];
          group_side<kSL>(p, L, ap, tile, h, k0, kb, grp, sl, z, s);
          if constexpr (CPB == 0) {  // one chunk, two blocks: the lane's codes are in block t/2
            const int u = L.t >> 1;
            zp_of(z, u, zl, zh);
            const float sc[2] = {u ? s[1][0] : s[0][0], u ? s[1][1] : s[0][1]};
            chunk_cc(p, L, ap, grp, BSG_LO(grp), BSG_HI(grp), zl, zh, sc, cacc[h]);
          } else if constexpr (CPB == 1) {  // two chunks, one block each
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int c = grp * 2 + u;
              zp_of(z, u, zl, zh);
              const float sc[2] = {s[u][0], s[u][1]};
              chunk_cc(p, L, ap, c, BSG_LO(c), BSG_HI(c), zl, zh, sc, cacc[h]);
            }
          } else {  // CPB 2, 4 or 8: kGC chunks in one block
            zp_of(z, 0, zl, zh);
            const float sc[2] = {s[0][0], s[0][1]};
#pragma unroll
            for (int u = 0; u < kGC; ++u) {
              const int c = grp * kGC + u;
              chunk_cc(p, L, ap, c, BSG_LO(c), BSG_HI(c), zl, zh, sc, cacc[h]);
            }
          }
        }
      }
    }
#undef BSG_LO
#undef BSG_HI
  }

  // End of a tile segment (CUDA-core variant): add each pair's halves, then the quad's four
  // lanes by a butterfly (every lane of the quad gets bit-identical sums, as fp32 addition
  // commutes), and leave in acc the mma fragment layout the epilogues take (tile rows g, g + 8;
  // activation rows 2t, 2t + 1).  The partial sums are cleared for the next segment.
  static BSG_DEV void cc_fragment(const Lane& L, uint64_t (&cacc)[2][kCcCols],
                                  float (&acc)[MT][4]) {
    float v[2][kCcCols];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr)
#pragma unroll
      for (int m = 0; m < kCcCols; ++m) {
        float x = f32x2_lo(cacc[rr][m]) + f32x2_hi(cacc[rr][m]);
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 1);
        x += __shfl_xor_sync(0xFFFFFFFFu, x, 2);
        v[rr][m] = x;
        cacc[rr][m] = 0ull;
      }
    if constexpr (kCcCols == 8) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          acc[0][2 * rr + e] = L.t == 0   ? v[rr][e]
                                  : L.t == 1 ? v[rr][2 + e]
                                  : L.t == 2 ? v[rr][4 + e]
                                             : v[rr][6 + e];
    } else {  // one activation row: column 0 is entry 0 (row g) and 2 (row g + 8) of lane t = 0
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        acc[0][2 * rr] = L.t == 0 ? v[rr][0] : 0.f;
        acc[0][2 * rr + 1] = 0.f;
      }
    }
  }

  // Store the 4 fp32 results of lane ln's fragment (half h, row group rg, n8 tile mt) as y,
  // after adding the bias of the output column when the call has one (in fp32, before the one
  // rounding to the activation dtype).
  static BSG_DEV void store_y(const KParams& p, int64_t tile, int h, int rg, int mt, int ln,
                              const float (&v)[4], float gs) {
    const int g = ln >> 2, t = ln & 3;
    const int64_t n0 = tile * kRows + h * kBoxRows + 16 * rg + g;
    const int m0 = mt * 8 + 2 * t;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t n = n0 + ((i & 2) ? 8 : 0);
      const int m = m0 + (i & 1);
      if (m < p.M && n < p.N) {
        float r = v[i] * gs;
        if (p.bias != nullptr) {
          const uint32_t b = __ldg(p.bias + n);
          r += BF16 ? __uint_as_float(b << 16) : __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
        }
        if constexpr (BF16)
          reinterpret_cast<__nv_bfloat16*>(p.y)[m * p.N + n] = __float2bfloat16_rn(r);
        else
          reinterpret_cast<__half*>(p.y)[m * p.N + n] = __float2half_rn(r);
      }
    }
  }

  // CTA whose stream-K range contains stage x: the largest i with floor(i*T/G) <= x, i.e. with
  // i*T < (x+1)*G.  A single-precision estimate (off by at most one: i <= G < 2^16) is
  // corrected with exact 64-bit products.
  static BSG_DEV int cta_of_stage(int64_t x, int64_t T, int G) {
    const int64_t lim = (x + 1) * G;
    int i = static_cast<int>(static_cast<float>(lim - 1) / static_cast<float>(T));
    while (static_cast<int64_t>(i + 1) * T < lim) ++i;
    while (i > 0 && static_cast<int64_t>(i) * T >= lim) --i;
    return i;
  }

  // ---- stream-K epilogue.  A tile the CTA consumed whole is rounded and stored at once.  For
  // a tile shared with other CTAs the warp writes its fp32 fragments to its partial slot
  // (st.cg) and goes on with its range; the arrivals on the tiles' (tile, row group) counters
  // are deferred to the end of the range and made together (one lane per pending tile, one
  // acquire-release atomic each: the release publishes all of the warp's partial stores,
  // which __syncwarp ordered before it).  The last arriver of a tile adds the contributors'
  // partials in CTA order and stores y -- P4's visibility protocol, without its per-call memset.
  // Deferring keeps the mid-range tile boundary off the consumer's critical path.
  // Partial slots [cta][seg][rg]: a CTA writes seg 0 for the first tile of its range and seg 1
  // for its last tile, so among a tile's contributors only the first can hold it in seg 1 (when
  // its range began in an earlier tile).
  static BSG_DEV void store_partial(const KParams& p, int64_t tile, int64_t my_first_tile, int rg,
                                    int lane, const float (&acc)[kH][MT][4]) {
    const int slot4 = p.slot_floats / 4;  // float4 per (cta, seg, rg) slot: every half
    const int seg = (tile == my_first_tile) ? 0 : 1;
    float4* mine = reinterpret_cast<float4*>(p.partials) +
                   ((static_cast<int64_t>(blockIdx.x) * 2 + seg) * kConsumerWarps + rg) * slot4;
#pragma unroll
    for (int h = 0; h < kH; ++h)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        __stcg(mine + (h * MT + mt) * 32 + lane,
               make_float4(acc[h][mt][0], acc[h][mt][1], acc[h][mt][2], acc[h][mt][3]));
  }

  // First and last CTA holding stages of `tile`.
  static BSG_DEV void tile_owners(const KParams& p, int64_t tile, int& first, int& last) {
    const int G = gridDim.x;
    const int64_t T = p.total_stages, x0 = tile * p.spt;
    first = cta_of_stage(x0, T, G);
    last = cta_of_stage(x0 + p.spt - 1, T, G);
  }

  // Arrive on the np (1 or 2) pending shared tiles; reduce and store each one this warp was the
  // last to arrive on.
  static BSG_DEV void arrive_and_reduce(const KParams& p, const int64_t (&pend)[2], int np,
                                        int rg, int lane, float gs) {
    __syncwarp();  // the warp's partial stores before the arrivals' release
    unsigned mine_last = 0;
    if (lane < np) {
      const int64_t tile = lane == 0 ? pend[0] : pend[1];
      int first, last;
      tile_owners(p, tile, first, last);
      const unsigned old = atom_add_acq_rel_gpu(p.counters + tile * kConsumerWarps + rg, 1u);
      mine_last = (old == static_cast<unsigned>(last - first)) ? 1u : 0u;
    }
    const unsigned last_mask = __ballot_sync(0xFFFFFFFFu, mine_last != 0);
    if (last_mask == 0) return;
    __syncwarp();  // order the warp's partial loads after the arriving lanes' acquire
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (j < np && ((last_mask >> j) & 1u)) reduce_tile(p, pend[j], rg, lane, gs);
  }

  static BSG_DEV void reduce_tile(const KParams& p, int64_t tile, int rg, int lane, float gs) {
    const int slot4 = p.slot_floats / 4;
    const int G = gridDim.x;
    const int64_t T = p.total_stages, x0 = tile * p.spt;
    int first, last;
    tile_owners(p, tile, first, last);
    const int fseg = (static_cast<int64_t>(first) * T < x0 * G) ? 1 : 0;  // first began earlier
    const float4* part = reinterpret_cast<const float4*>(p.partials);
    // contributors' partials in batches of kBatch independent loads, added in CTA order
    constexpr int kF = kH * MT;  // float4 per lane and slot
    constexpr int kBatch = 8 / kF > 0 ? 8 / kF : 1;
    float v[kF][4];
#pragma unroll
    for (int f = 0; f < kF; ++f)
#pragma unroll
      for (int e = 0; e < 4; ++e) v[f][e] = 0.f;
    for (int i0 = first; i0 <= last; i0 += kBatch) {
      float4 u[kBatch][kF];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int i = i0 + j;
        const int sg = (i == first) ? fseg : 0;
        const float4* src =
            part + ((static_cast<int64_t>(i) * 2 + sg) * kConsumerWarps + rg) * slot4 + lane;
#pragma unroll
        for (int f = 0; f < kF; ++f)
          u[j][f] = (i <= last) ? __ldcg(src + f * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        if (i0 + j > last) break;
#pragma unroll
        for (int f = 0; f < kF; ++f) {
          v[f][0] += u[j][f].x;
          v[f][1] += u[j][f].y;
          v[f][2] += u[j][f].z;
          v[f][3] += u[j][f].w;
        }
      }
    }
#pragma unroll
    for (int h = 0; h < kH; ++h)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) store_y(p, tile, h, rg, mt, lane, v[h * MT + mt], gs);
    if (lane == 0) p.counters[tile * kConsumerWarps + rg] = 0u;  // all arrived: reset for reuse
  }

  // ---- cluster split: the CTAs of a cluster each hold a K-range of the same tile.  Every
  // consumer warp stores the fragment lanes that hold output columns below max_M (quad lanes
  // t < red_tq) into the leader's (rank 0) reduction buffer slot [rank][warp], through
  // distributed shared memory; after the cluster barrier the leader's warps add the slots in rank
  // order (fixed: deterministic) and store y.
  static BSG_DEV uint32_t red_slot(const KParams& p, const Smem& sm, int rank, int cw, int h,
                                   int mt, int li) {
    const int per_mt = 8 * p.red_tq;
    return sm.base_u + p.red_off +
           (((((rank * kConsumerWarps + cw) * kH + h) * MT + mt) * per_mt) + li) * 16;
  }

  static BSG_DEV void cluster_publish(const KParams& p, const Smem& sm, int cw, const Lane& L,
                                      const float (&acc)[kH][MT][4]) {
    if (L.t >= p.red_tq) return;
    const int rank = static_cast<int>(cluster_ctarank());
    const int li = L.g * p.red_tq + L.t;
#pragma unroll
    for (int h = 0; h < kH; ++h)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
        st_cluster_f32x4(mapa_shared(red_slot(p, sm, rank, cw, h, mt, li), 0), acc[h][mt][0],
                         acc[h][mt][1], acc[h][mt][2], acc[h][mt][3]);
  }

  static BSG_DEV void cluster_reduce(const KParams& p, const Smem& sm, int cw, int lane) {
    const int g = lane >> 2, t = lane & 3;
    if (t >= p.red_tq) return;
    const int li = g * p.red_tq + t;
    const int64_t tile = blockIdx.x / p.cluster;
    const float gs = kFold ? __ldg(p.gscale) : 1.0f;
#pragma unroll
    for (int h = 0; h < kH; ++h)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int r = 0; r < p.cluster; ++r) {
          const float4 u = *reinterpret_cast<const float4*>(
              sm.base + (red_slot(p, sm, r, cw, h, mt, li) - sm.base_u));
          v[0] += u.x;
          v[1] += u.y;
          v[2] += u.z;
          v[3] += u.w;
        }
        store_y(p, tile, h, cw, mt, lane, v, gs);
      }
  }

  // ---- consumers: warps 1..4.  The CTA's range is walked tile segment by tile segment; within
  // a segment every stage waits for its slot (and, when it opens one, its side box), is
  // multiplied in, and is released; the segment ends with the epilogue.
  // SIDE: scales and zero points from the side ring (KParams::side_tma), else from global memory;
  // a template parameter of the kernel, so that each kernel holds one consumer loop.
  template <bool SIDE>
  static BSG_DEV void consume(const KParams& p, const Smem& sm, int64_t s0, int64_t s1, int cw,
                              int lane) {
    pdl_wait();  // the epilogues write y and the plan's workspace
    consume_range<SIDE>(p, sm, s0, s1, cw, lane);
  }

  template <bool SIDE>
  static BSG_DEV void consume_range(const KParams& p, const Smem& sm, int64_t s0, int64_t s1,
                                    int cw, int lane) {
    const Lane L = make_lane(p, cw, lane);
    const Run<SIDE> R{p.bs_log2, p.rs_log2, p.zbox_bytes, p};
    float acc[kH][MT][4];
#pragma unroll
    for (int h = 0; h < kH; ++h) zero(acc[h]);
    uint64_t cacc[kH][2][kCcCols];  // CUDA-core variant's partial sums (unused by the mma
                                         // variant)
#pragma unroll
    for (int h = 0; h < kH; ++h)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int m = 0; m < kCcCols; ++m) cacc[h][rr][m] = 0ull;
    const float gs = kFold ? __ldg(p.gscale) : 1.0f;
    const int spt = p.spt;
    const int n = static_cast<int>(s1 - s0);
    const int64_t first_tile = s0 / spt;
    Walk w{first_tile, static_cast<int>(s0 - first_tile * spt), spt, (1 << p.rs_log2) - 1};
    Ring r{0, 0u, sm.stages};
    Ring sr{sm.side_slots - 1, 1u, sm.side_slots};
    bool ok = true;  // false once a wait of this warp has run out (see produce)
    int64_t pend[2] = {0, 0};  // shared tiles whose arrival is deferred to the end of the range
    int np = 0;
    for (int i = 0; i < n;) {
      const int seg = (spt - w.ks) < (n - i) ? (spt - w.ks) : (n - i);  // stages of this segment
      const int64_t tile = w.tile;
      for (int q = 0; q < seg; ++q) {
        // (every lane of the converged warp sees the same barrier state and the same
        // %globaltimer value at each step of the wait, so `ok` is the same in all lanes)
        if (SIDE && w.opens(q == 0)) {
          sr.next();
          if (ok) ok = mbar_wait(sm.sfull(sr.slot), sr.phase, p.err, kErrTimeoutFull, p.wait_ns);
        }
        if (ok) ok = mbar_wait(sm.full(r.slot), r.phase, p.err, kErrTimeoutFull, p.wait_ns);
        if (ok) {
          const Sh sh{sm.base, static_cast<uint32_t>(sm.act_off + r.slot * sm.act_bytes),
                      static_cast<uint32_t>(sm.side_off + sr.slot * sm.side_bytes)};
          consume_stage(R, L, sm.w(r.slot), sh, tile, w.ks, acc, cacc);
        }
        __syncwarp();
        // after a wait ran out, the warp releases nothing more (see produce)
        mbar_arrive_if(sm.empty(r.slot), ok && lane == 0);
        if (SIDE && w.closes(q == seg - 1)) mbar_arrive_if(sm.sempty(sr.slot), ok && lane == 0);
        r.next();
        w.next();
      }
      i += seg;
      if constexpr (CC > 0) {
#pragma unroll
        for (int h = 0; h < kH; ++h) cc_fragment(L, cacc[h], acc[h]);
      }
      if (p.cluster >= 2) {
        cluster_publish(p, sm, cw, L, acc);  // the cluster's leader adds and stores
      } else if (seg == spt) {  // whole: this CTA consumed every stage of the tile
#pragma unroll
        for (int h = 0; h < kH; ++h)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) store_y(p, tile, h, cw, mt, lane, acc[h][mt], gs);
      } else {  // shared with other CTAs (at most the first and the last segment of the range)
        store_partial(p, tile, first_tile, cw, lane, acc);
        pend[np++ & 1] = tile;
      }
#pragma unroll
      for (int h = 0; h < kH; ++h) zero(acc[h]);
    }
    if (np > 0) arrive_and_reduce(p, pend, np, cw, lane, gs);
    if (!ok && lane == 0) *sm.abort_word() = 1u;
  }
};

// The body shared by both kernels: one CTA of the persistent grid.
template <class K, bool SIDE>
BSG_DEV void gemv_cta(const KParams& p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned (128-byte swizzle atoms), derived from the shared array so that plain
  // loads through it stay shared-memory loads
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const typename K::Smem sm{base, smem_u32(base), p.stages, p.act_off, p.act_bytes,
                            p.side_off, p.side_bytes, p.side_slots, p.bar_off};

  // stream-K: an equal share of the tiles x stages space; cluster split: an equal share of the
  // stages of tile blockIdx.x / cluster (the cluster's CTAs are consecutive in x)
  int64_t s0, s1;
  if (p.cluster > 0) {
    const int64_t C = p.cluster, tile = blockIdx.x / C, r = blockIdx.x % C;
    s0 = tile * p.spt + r * p.spt / C;
    s1 = tile * p.spt + (r + 1) * p.spt / C;
  } else {
    const int64_t G = gridDim.x, T = p.total_stages;
    s0 = static_cast<int64_t>(blockIdx.x) * T / G;
    s1 = (static_cast<int64_t>(blockIdx.x) + 1) * T / G;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < sm.stages; ++i) {
      mbar_init(sm.full(i), 1);
      mbar_init(sm.empty(i), kConsumerWarps);
    }
    for (int j = 0; j < sm.side_slots; ++j) {
      mbar_init(sm.sfull(j), 1);
      mbar_init(sm.sempty(j), kConsumerWarps);
    }
    *sm.abort_word() = 0u;
    fence_mbar_init();
  }
  __syncthreads();

  typename K::Pending pd;
  if (warp == 0) {
    pd = K::produce(p, sm, s0, s1, lane);
  } else {
    K::template consume<SIDE>(p, sm, s0, s1, warp - 1, lane);
  }
  // A wait that ran out anywhere in the CTA: the copy warp waits for what it issued (see
  // produce) before the CTA's shared memory is given up.
  __syncthreads();
  if (warp == 0 && *sm.abort_word() != 0u) {
    K::drain(p, sm, pd, lane);
    __syncwarp();  // lane 0's waits end before the warp's aligned cluster barrier
  }
  if (p.cluster >= 2) {
    cluster_sync();  // every CTA of the cluster has stored its partials in the leader
    if (cluster_ctarank() == 0 && warp > 0) K::cluster_reduce(p, sm, warp - 1, lane);
  }
}

// Tensor-core kernel (the default): products on mma.sync.m16n8k16.
template <int FMT, bool BF16, int MT, bool ZP, int CPB, int H, bool SIDE>
__global__ void __launch_bounds__(kThreads, ctas_per_sm_for(MT, H))
    bsgemv_mma_kernel(const __grid_constant__ KParams p) {
  gemv_cta<Gemv<FMT, BF16, MT, ZP, CPB, H>, SIDE>(p);
}

// CUDA-core kernel (BSGEMV_VARIANT_CUDA_CORE): products on fp32 FMAs, COLS = 1 (calls with
// M = 1) or 8 (M <= 8) activation rows per lane.
template <int FMT, bool BF16, bool ZP, int CPB, int COLS, bool SIDE>
__global__ void __launch_bounds__(kThreads, ctas_per_sm_for(1, 1))
    bsgemv_fma_kernel(const __grid_constant__ KParams p) {
  gemv_cta<Gemv<FMT, BF16, 1, ZP, CPB, 1, COLS>, SIDE>(p);
}

}  // namespace bsg
