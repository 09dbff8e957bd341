// bsgemv_dense.cu -- the dense small-N split-K GEMV ("[CUDA] MatMul: add an opt-in split-K GEMV
// for small-N fp16 shapes"): y[M, N] = A[M, K] . B[K, N], fp16 or bf16, B row-major (the
// MatMul right-hand side), M <= 8, fp32 accumulation, one rounding.
//
// Decode-time projections with small N leave most SMs idle when each CTA owns a whole column
// range, so K is split too.  On GB300:
//   * a CTA tile is 64 output columns n over a contiguous K-slice; the S K-slices of a tile are
//     the S CTAs of one thread-block cluster (S <= 8);
//   * warp 0 streams stages of 64 k: one TMA box of B [64 k][64 n] (128-byte swizzle) and one of
//     A [8 rows][64 k] (rows past M and k past K zero-filled) into a ring of mbarrier slots;
//   * warps 1..4 each own 16 columns: ldmatrix.trans turns the [k][n] tile into the A operand of
//     mma.sync.m16n8k16 (rows = n), the activations are the B operand (8 columns = the M rows);
//   * the cluster's CTAs publish their fp32 fragments into the leader's shared memory
//     (st.shared::cluster), and the leader adds them in rank order -- the page's fixed-order
//     reduction, without global workspace, counters or a per-call memset.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <new>

#include "bsgemv_kernel.cuh"

namespace bsg {

constexpr int kDenseTileN = 64;       // output columns per CTA (4 consumer warps x 16)
constexpr int kDenseStageK = 64;      // k per stage: B box [64][64] (8 KB), A box [8][64] (1 KB)
constexpr int kDenseMaxStages = 8;
constexpr int kDenseMaxSplit = 8;     // CTAs per tile (portable cluster size)
constexpr int kDenseMaxM = 8;
constexpr int kDenseBBox = kDenseStageK * kDenseTileN * 2;
constexpr int kDenseABox = kDenseMaxM * kDenseStageK * 2;

struct DParams {
  CUtensorMap tm_b;  // B as 16-bit [K][N], box [64 k][64 n], 128-byte swizzle
  CUtensorMap tm_a;  // A as 16-bit [M][K], box [8 m][64 k], 128-byte swizzle
  void* y;
  unsigned* err;
  int64_t N, K;
  int M, spt, splits, stages, red_off, bar_off;
};

template <bool BF16>
BSG_DEV void dense_store(const DParams& p, int64_t n0, int lane, const float (&v)[4]) {
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int64_t n = n0 + g + ((i & 2) ? 8 : 0);
    const int m = 2 * t + (i & 1);
    if (m < p.M && n < p.N) {
      if constexpr (BF16)
        reinterpret_cast<__nv_bfloat16*>(p.y)[m * p.N + n] = __float2bfloat16_rn(v[i]);
      else
        reinterpret_cast<__half*>(p.y)[m * p.N + n] = __float2half_rn(v[i]);
    }
  }
}

template <bool BF16>
__global__ void __launch_bounds__(32 * 5, 1) bsgemv_dense_kernel(const __grid_constant__ DParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base_u = smem_u32(base);
  const int S = p.splits, R = p.stages;
  const int64_t tile = blockIdx.x / S;
  const int rank = static_cast<int>(blockIdx.x % S);
  const int s0 = rank * p.spt / S, s1 = (rank + 1) * p.spt / S;  // this CTA's stages of the tile
  const int n = s1 - s0;
  auto bslot = [&](int i) { return base_u + i * kDenseBBox; };
  auto aslot = [&](int i) { return base_u + R * kDenseBBox + i * kDenseABox; };
  auto full = [&](int i) { return base_u + p.bar_off + 8 * i; };
  auto empty = [&](int i) { return base_u + p.bar_off + 8 * (R + i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 4);
    }
    fence_mbar_init();
  }
  __syncthreads();

  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (warp == 0) {
    // producer: B (the weight, never written by a preceding kernel) for the first ring slots
    // before the dependency wait, A after it
    if (lane == 0) {
      prefetch_tmap(&p.tm_b);
      prefetch_tmap(&p.tm_a);
      const uint64_t pol = policy_evict_first();
      const int x_n = static_cast<int>(tile * kDenseTileN);
      const int pre = n < R ? n : R;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(full(i), kDenseBBox + kDenseABox);
        tma_load_2d_hint(bslot(i), &p.tm_b, x_n, (s0 + i) * kDenseStageK, full(i), pol);
      }
      pdl_wait();
      for (int i = 0; i < pre; ++i) tma_load_2d(aslot(i), &p.tm_a, (s0 + i) * kDenseStageK, 0, full(i));
      int slot = pre % R;
      uint32_t phase = pre == R ? 1u : 0u;
      for (int i = pre; i < n; ++i) {
        if (!mbar_wait(empty(slot), phase ^ 1u, p.err, kErrTimeoutEmpty)) break;
        mbar_arrive_expect_tx(full(slot), kDenseBBox + kDenseABox);
        tma_load_2d_hint(bslot(slot), &p.tm_b, x_n, (s0 + i) * kDenseStageK, full(slot), pol);
        tma_load_2d(aslot(slot), &p.tm_a, (s0 + i) * kDenseStageK, 0, full(slot));
        if (++slot == R) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    pdl_wait();  // y is written below
    const int wn = warp - 1;  // columns 16 wn .. 16 wn + 15 of the tile
    // ldmatrix.x4.trans: lanes 8q .. 8q + 7 address matrix q = (k rows +8 if q >= 2) x (n +8 if
    // q odd); row r = lane & 7 of the stage's 16-k step; 128-byte swizzle: chunk c of row k is
    // stored at chunk c ^ (k & 7)
    const int q = lane >> 3, r = lane & 7;
    const uint32_t b_off = ((q >> 1) * 8 + r) * 128 + (((2 * wn + (q & 1)) ^ r) << 4);
    const int g = lane >> 2, t = lane & 3;
    int slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int i = 0; i < n; ++i) {
      if (ok) ok = mbar_wait(full(slot), phase, p.err, kErrTimeoutFull);
      if (ok) {
        const uint32_t bs = bslot(slot), as = aslot(slot);
#pragma unroll
        for (int ks = 0; ks < kDenseStageK / 16; ++ks) {
          uint32_t a[4];
          asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                       : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                       : "r"(bs + ks * 16 * 128 + b_off));
          // activations: row g, k = 16 ks + 2t (+ 8), chunk 2 ks (+ 1) swizzled by the row
          const uint32_t b0 = lds32(as + g * 128 + (((2 * ks) ^ g) << 4) + 4 * t);
          const uint32_t b1 = lds32(as + g * 128 + (((2 * ks + 1) ^ g) << 4) + 4 * t);
          mma16816<BF16>(acc, a, b0, b1);
        }
      }
      __syncwarp();
      mbar_arrive_if(empty(slot), lane == 0);
      if (++slot == R) {
        slot = 0;
        phase ^= 1u;
      }
    }
    if (S == 1) dense_store<BF16>(p, tile * kDenseTileN + 16 * wn, lane, acc);
  }
  if (S >= 2) {
    // every CTA's consumer warps publish into slot [rank][warp] of the leader's buffer
    if (warp > 0) {
      const uint32_t dst = base_u + p.red_off + ((rank * 4 + (warp - 1)) * 32 + lane) * 16;
      st_cluster_f32x4(mapa_shared(dst, 0), acc[0], acc[1], acc[2], acc[3]);
    }
    cluster_sync();
    if (rank == 0 && warp > 0) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      for (int rr = 0; rr < S; ++rr) {  // rank order: deterministic
        const float4 u = *reinterpret_cast<const float4*>(
            base + p.red_off + ((rr * 4 + (warp - 1)) * 32 + lane) * 16);
        v[0] += u.x;
        v[1] += u.y;
        v[2] += u.z;
        v[3] += u.w;
      }
      dense_store<BF16>(p, tile * kDenseTileN + 16 * (warp - 1), lane, v);
    }
  }
}

// ---- N not a multiple of 8 (B's rows are not 16-byte aligned, so no TMA): CUDA-core kernel.
// A CTA owns kNarrowN columns and a K-slice; its 256 threads stride over k (thread t takes
// k = k0 + t, k0 + t + 256, ...), each keeping fp32 sums for the 8 columns and up to 8 rows.
// Then, in a fixed order: a butterfly over the warp's lanes, the 8 warps in order, and (K
// split over a cluster) the CTAs of the cluster in rank order in the leader's shared memory.
constexpr int kNarrowN = 8;
constexpr int kNarrowThreads = 256;

struct NParams {
  const uint16_t* A;
  const uint16_t* B;
  void* y;
  int64_t N, K;
  int M, splits;
};

template <bool BF16>
BSG_DEV float bits_to_f32(uint16_t b) {
  if constexpr (BF16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
  return __half2float(__ushort_as_half(b));
}

template <bool BF16>
__global__ void __launch_bounds__(kNarrowThreads, 1)
    bsgemv_dense_narrow_kernel(const __grid_constant__ NParams p) {
  __shared__ float part[kNarrowThreads / 32][kDenseMaxM * kNarrowN];  // per warp
  __shared__ __align__(16) float red[kDenseMaxSplit][kDenseMaxM * kNarrowN];  // leader: per rank
  const int S = p.splits;
  const int64_t tile = blockIdx.x / S;
  const int rank = static_cast<int>(blockIdx.x % S);
  const int64_t n0 = tile * kNarrowN;
  const int nn = static_cast<int>(p.N - n0 < kNarrowN ? p.N - n0 : kNarrowN);
  const int64_t k0 = rank * p.K / S, k1 = (rank + 1) * p.K / S;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  pdl_wait();  // A may be the previous kernel's output
  float acc[kDenseMaxM][kNarrowN];
#pragma unroll
  for (int m = 0; m < kDenseMaxM; ++m)
#pragma unroll
    for (int n = 0; n < kNarrowN; ++n) acc[m][n] = 0.f;
  for (int64_t k = k0 + threadIdx.x; k < k1; k += kNarrowThreads) {
    float b[kNarrowN];
    const uint16_t* row = p.B + k * p.N + n0;
#pragma unroll
    for (int n = 0; n < kNarrowN; ++n) b[n] = n < nn ? bits_to_f32<BF16>(__ldg(row + n)) : 0.f;
#pragma unroll
    for (int m = 0; m < kDenseMaxM; ++m) {
      if (m < p.M) {
        const float a = bits_to_f32<BF16>(__ldg(p.A + m * p.K + k));
#pragma unroll
        for (int n = 0; n < kNarrowN; ++n) acc[m][n] = fmaf(a, b[n], acc[m][n]);
      }
    }
  }
  // lanes: butterfly (every lane ends with the same sum: fp32 addition commutes)
#pragma unroll
  for (int m = 0; m < kDenseMaxM; ++m)
#pragma unroll
    for (int n = 0; n < kNarrowN; ++n) {
      float v = acc[m][n];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      acc[m][n] = v;
    }
  if (lane == 0) {
#pragma unroll
    for (int m = 0; m < kDenseMaxM; ++m)
#pragma unroll
      for (int n = 0; n < kNarrowN; ++n) part[warp][m * kNarrowN + n] = acc[m][n];
  }
  __syncthreads();
  // warps in order; then the cluster's CTAs in rank order
  const int e = threadIdx.x;  // one (m, n) per thread for e < 64
  float v = 0.f;
  if (e < kDenseMaxM * kNarrowN) {
    for (int w = 0; w < kNarrowThreads / 32; ++w) v += part[w][e];
  }
  if (S >= 2) {
    if (e < kDenseMaxM * kNarrowN) {
      const uint32_t dst = smem_u32(&red[rank][e]);
      asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(mapa_shared(dst, 0)), "f"(v) : "memory");
    }
    cluster_sync();
    if (rank != 0) return;
    v = 0.f;
    if (e < kDenseMaxM * kNarrowN)
      for (int r = 0; r < S; ++r) v += red[r][e];
  }
  if (e < kDenseMaxM * kNarrowN) {
    const int m = e / kNarrowN, n = e % kNarrowN;
    if (m < p.M && n < nn) {
      if constexpr (BF16)
        reinterpret_cast<__nv_bfloat16*>(p.y)[m * p.N + n0 + n] = __float2bfloat16_rn(v);
      else
        reinterpret_cast<__half*>(p.y)[m * p.N + n0 + n] = __float2half_rn(v);
    }
  }
}

namespace {

constexpr int kDenseThreads = 32 * 5;

struct DenseGeo {
  bsgemv_geometry pub;
  int bf16, max_M, narrow;
  int64_t N, K;
  int red_off, bar_off;
};

// Validation and geometry (pure host code).  Split: as many CTAs per tile (a cluster of at
// most 8) as keep tiles x S within two CTAs per SM and give each CTA at least one stage.
int dense_geometry(int act_bf16, int64_t N, int64_t K, int max_M, int sm_count, DenseGeo* g) {
  if (g == nullptr) return BSGEMV_ERR_INVALID_ARG;
  std::memset(g, 0, sizeof(*g));
  if ((act_bf16 != 0 && act_bf16 != 1) || N < 1 || K < 1 || max_M < 1 || max_M > kDenseMaxM ||
      sm_count < 1)
    return BSGEMV_ERR_INVALID_ARG;
  if (N > (int64_t(1) << 31) - kDenseTileN || K > (int64_t(1) << 30)) return BSGEMV_ERR_UNSUPPORTED;
  g->bf16 = act_bf16;
  g->max_M = max_M;
  g->N = N;
  g->K = K;
  // TMA needs row pitches of B (N) and A (K) in multiples of 16 bytes; otherwise the CUDA-core
  // kernel (8 columns per CTA, 256 threads striding over k, K split over a cluster)
  g->narrow = (N % 8 != 0 || K % 8 != 0 || K < 16) ? 1 : 0;
  if (g->narrow) {
    const int64_t tiles = (N + kNarrowN - 1) / kNarrowN;
    const int64_t kslices = (K + kNarrowThreads - 1) / kNarrowThreads;
    const int64_t cap = std::max<int64_t>(1, (2 * int64_t(sm_count)) / tiles);
    const int S = static_cast<int>(std::min<int64_t>({kDenseMaxSplit, kslices, cap}));
    bsgemv_geometry& q = g->pub;
    q.variant = BSGEMV_VARIANT_CUDA_CORE;
    q.rows_per_tile = kNarrowN;
    q.k_per_stage = kNarrowThreads;
    q.stages = 1;
    q.consumer_warps = kNarrowThreads / 32;
    q.ctas = static_cast<int>(tiles * S);
    q.ctas_per_sm = 2;
    q.sm_count = sm_count;
    q.tiles = tiles;
    q.stages_per_tile = kslices;
    q.total_stages = tiles * kslices;
    q.smem_bytes = 0;
    q.workspace_bytes = 256;
    q.cluster = S;
    return BSGEMV_OK;
  }
  const int64_t tiles = (N + kDenseTileN - 1) / kDenseTileN;
  const int64_t spt = (K + kDenseStageK - 1) / kDenseStageK;
  const int64_t cap = std::max<int64_t>(1, (2 * int64_t(sm_count)) / tiles);
  const int S = static_cast<int>(std::min<int64_t>({kDenseMaxSplit, spt, cap}));
  const int share = static_cast<int>((spt + S - 1) / S);
  const int stages = std::min(kDenseMaxStages, share);
  const int red = S >= 2 ? S * 4 * 32 * 16 : 0;
  g->red_off = stages * (kDenseBBox + kDenseABox);
  g->bar_off = g->red_off + red;
  bsgemv_geometry& p = g->pub;
  p.variant = BSGEMV_VARIANT_MMA;
  p.rows_per_tile = kDenseTileN;
  p.k_per_stage = kDenseStageK;
  p.stages = stages;
  p.consumer_warps = 4;
  p.ctas = static_cast<int>(tiles * S);
  p.ctas_per_sm = 2;
  p.sm_count = sm_count;
  p.tiles = tiles;
  p.stages_per_tile = spt;
  p.total_stages = tiles * spt;
  p.smem_bytes = 1024 + g->bar_off + 16 * stages;
  p.workspace_bytes = 256;
  p.cluster = S;
  return BSGEMV_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 dense_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 16-bit 2D tensor [rows][cols], box [box_rows][box_cols], 128-byte swizzle, zero fill.
int encode_u16(CUtensorMap* tm, const void* ptr, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows) {
  auto fn = dense_encode_fn();
  if (!fn) return BSGEMV_ERR_CUDA;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) % 16) == 0; }
bool aligned2(const void* p) { return (reinterpret_cast<uintptr_t>(p) % 2) == 0; }

int launch_dense_narrow(const DenseGeo& g, const void* A, const void* B, void* y, int M,
                        cudaStream_t s) {
  NParams k;
  k.A = static_cast<const uint16_t*>(A);
  k.B = static_cast<const uint16_t*>(B);
  k.y = y;
  k.N = g.N;
  k.K = g.K;
  k.M = M;
  k.splits = g.pub.cluster;
  auto kern = g.bf16 ? bsgemv_dense_narrow_kernel<true> : bsgemv_dense_narrow_kernel<false>;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  int na = 1;
  if (g.pub.cluster >= 2) {
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = static_cast<unsigned>(g.pub.cluster);
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    na = 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(g.pub.ctas));
  cfg.blockDim = dim3(kNarrowThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kern, k) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

}  // namespace
}  // namespace bsg

struct bsgemv_dense_plan_s {
  bsg::DenseGeo geo;
  int device = -1;
  unsigned* err = nullptr;
  const void* b_ptr = nullptr;  // tensor maps of the last B and (A, M)
  CUtensorMap tm_b;
  const void* a_ptr = nullptr;
  int a_m = 0;
  CUtensorMap tm_a;
};

extern "C" {

int bsgemv_dense_geometry_for(int act_bf16, int64_t N, int64_t K, int max_M, int sm_count,
                              bsgemv_geometry* g) {
  if (g == nullptr) return BSGEMV_ERR_INVALID_ARG;
  bsg::DenseGeo geo;
  const int rc = bsg::dense_geometry(act_bf16, N, K, max_M, sm_count, &geo);
  if (rc == BSGEMV_OK) *g = geo.pub;
  return rc;
}

int bsgemv_dense_plan(bsgemv_dense_plan_t* out, int act_bf16, int64_t N, int64_t K, int max_M) {
  if (out == nullptr) return BSGEMV_ERR_INVALID_ARG;
  *out = nullptr;
  bsg::DenseGeo probe;
  int rc = bsg::dense_geometry(act_bf16, N, K, max_M, 1, &probe);
  if (rc != BSGEMV_OK) return rc;  // argument errors need no GPU
  int dev = -1, major = 0, minor = 0, sms = 0;
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
  auto* p = new (std::nothrow) bsgemv_dense_plan_s();
  if (!p) return BSGEMV_ERR_CUDA;
  rc = bsg::dense_geometry(act_bf16, N, K, max_M, sms, &p->geo);
  if (rc == BSGEMV_OK && (cudaMalloc(&p->err, 256) != cudaSuccess ||
                          cudaMemset(p->err, 0, 256) != cudaSuccess)) {
    cudaGetLastError();
    rc = BSGEMV_ERR_CUDA;
  }
  if (rc != BSGEMV_OK) {
    if (p->err) cudaFree(p->err);
    delete p;
    return rc;
  }
  p->device = dev;
  *out = p;
  return BSGEMV_OK;
}

int bsgemv_dense_run(bsgemv_dense_plan_t plan, const void* A, const void* B, void* y, int M,
                     void* stream) {
  if (plan == nullptr || A == nullptr || B == nullptr || y == nullptr || M < 1)
    return BSGEMV_ERR_INVALID_ARG;
  const bsg::DenseGeo& g = plan->geo;
  if (M > g.max_M) return BSGEMV_ERR_M_TOO_LARGE;
  const bool narrow = g.narrow != 0;
  if (narrow ? (!bsg::aligned2(A) || !bsg::aligned2(B) || !bsg::aligned2(y))
             : (!bsg::aligned16(A) || !bsg::aligned16(B) || !bsg::aligned16(y)))
    return BSGEMV_ERR_MISALIGNED;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  if (cur != plan->device) return BSGEMV_ERR_WRONG_DEVICE;
  if (narrow) return bsg::launch_dense_narrow(g, A, B, y, M, static_cast<cudaStream_t>(stream));
  if (B != plan->b_ptr) {
    plan->b_ptr = nullptr;
    if (bsg::encode_u16(&plan->tm_b, B, g.N, g.K, bsg::kDenseTileN, bsg::kDenseStageK) != BSGEMV_OK)
      return BSGEMV_ERR_CUDA;
    plan->b_ptr = B;
  }
  if (A != plan->a_ptr || M != plan->a_m) {
    plan->a_ptr = nullptr;
    if (bsg::encode_u16(&plan->tm_a, A, g.K, M, bsg::kDenseStageK, bsg::kDenseMaxM) != BSGEMV_OK)
      return BSGEMV_ERR_CUDA;
    plan->a_ptr = A;
    plan->a_m = M;
  }
  bsg::DParams k;
  std::memset(&k, 0, sizeof(k));
  k.tm_b = plan->tm_b;
  k.tm_a = plan->tm_a;
  k.y = y;
  k.err = plan->err;
  k.N = g.N;
  k.K = g.K;
  k.M = M;
  k.spt = static_cast<int>(g.pub.stages_per_tile);
  k.splits = g.pub.cluster;
  k.stages = g.pub.stages;
  k.red_off = g.red_off;
  k.bar_off = g.bar_off;
  auto kern = g.bf16 ? bsg::bsgemv_dense_kernel<true> : bsg::bsgemv_dense_kernel<false>;
  static bsg::AttrRecord rec_bf16, rec_f16;  // per device and context
  bsg::AttrRecord& rec = g.bf16 ? rec_bf16 : rec_f16;
  int dev = -1;
  uint64_t ctx = 0;
  if (!bsg::current_device_context(&dev, &ctx)) return BSGEMV_ERR_CUDA;
  const int d = rec.slot(dev, ctx);
  if (g.pub.smem_bytes > rec.smem[d].load()) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             g.pub.smem_bytes) != cudaSuccess)
      return BSGEMV_ERR_CUDA;
    rec.smem[d].store(g.pub.smem_bytes);
  }
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  int na = 1;
  if (g.pub.cluster >= 2) {
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = static_cast<unsigned>(g.pub.cluster);
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    na = 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(g.pub.ctas));
  cfg.blockDim = dim3(bsg::kDenseThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(g.pub.smem_bytes);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = at;
  cfg.numAttrs = na;
  if (cudaLaunchKernelEx(&cfg, kern, k) != cudaSuccess) {
    cudaGetLastError();
    return BSGEMV_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? BSGEMV_OK : BSGEMV_ERR_CUDA;
}

int bsgemv_dense_describe(bsgemv_dense_plan_t plan, bsgemv_geometry* g) {
  if (plan == nullptr || g == nullptr) return BSGEMV_ERR_INVALID_ARG;
  *g = plan->geo.pub;
  return BSGEMV_OK;
}

int bsgemv_dense_device_status(bsgemv_dense_plan_t plan, void* stream) {
  if (plan == nullptr) return BSGEMV_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return BSGEMV_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, plan->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return BSGEMV_ERR_CUDA;
  if (word != 0) {
    cudaMemset(plan->err, 0, sizeof(unsigned));
    return BSGEMV_ERR_DEVICE_TIMEOUT;
  }
  return BSGEMV_OK;
}

int bsgemv_dense_destroy(bsgemv_dense_plan_t plan) {
  if (plan == nullptr) return BSGEMV_OK;
  int rc = BSGEMV_OK;
  if (plan->err) {
    if (cudaDeviceSynchronize() != cudaSuccess) rc = BSGEMV_ERR_CUDA;
    cudaFree(plan->err);
  }
  delete plan;
  return rc;
}

}  // extern "C"
