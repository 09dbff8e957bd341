/*
 * bsgemv.h -- C ABI of the fused dequantize-and-multiply small-M GEMV for one NVIDIA GB300
 * (sm_103a):
 *
 *     y[M, N] = A[M, K] . deq(W)[N, K]^T,        1 <= M <= 32
 *
 * A is fp16 or bf16.  W is block-quantised along K and stored in the [N, blocks, blob] layout
 * ("[CUDA] Batched small-M GEMV for MatMulNBits (4-bit/8-bit)", Description), in one of:
 *
 *   BSGEMV_INT4      4-bit codes, two per byte (low nibble = even k); deq = (q - zp) * s with an
 *                    fp16 scale per (row, block) and an optional packed 4-bit zero point
 *                    ("[CUDA] MatMulNBits 8-bit: wide fp16 M=1 kernel for decode GEMVs",
 *                    Description; batched small-M page, Description and review)
 *   BSGEMV_INT8      8-bit codes; deq = (q - zp) * s, fp16 scale, optional 8-bit zero point
 *                    (wide M=1 page, Description)
 *   BSGEMV_FP8_E4M3  E4M3 codes; deq = e4m3 * s with one fp32 scale per 128 k
 *                    ("[CUDA] Block-scaled MatMul decode GEMV: tensor cores, packed FP4 decode
 *                    and M-tiling", description, FP8 tensor-core paragraph)
 *   BSGEMV_NVFP4     E2M1 codes two per byte (low nibble = even k), one E4M3 scale per 16 k and
 *                    one fp32 global scale g; deq = e2m1 * e4m3 * g (same page, NVFP4
 *                    tensor-core paragraph)
 *
 * Every call accumulates in fp32 and rounds the result once, round-to-nearest-even, to the
 * activation dtype.  The library has no CPU fallback: without an sm_103a device every entry
 * point that needs one returns an error.
 *
 * Layouts (all row-major, all tensors caller-owned):
 *   A       [M, K] fp16/bf16, device memory, 16-byte aligned
 *   W       int4/nvfp4: [N, K/2] bytes; int8/fp8: [N, K] bytes; device, 16-byte aligned
 *   scales  int4/int8: fp16 [N, K/bs]; fp8: fp32 [N, K/128]; nvfp4: E4M3 bytes [N, K/16]
 *   zp      int4: [N, ceil((K/bs)/2)] bytes, block b in nibble (b & 1) of byte b/2 (low nibble =
 *           even block); int8: [N, K/bs] bytes; NULL when has_zp == 0 (implicit zero point 8
 *           for int4, 128 for int8).  For NVFP4 this slot carries the device pointer of the one
 *           fp32 global scale.  For FP8 it must be NULL.
 *   y       [M, N] in the activation dtype, device memory, 16-byte aligned
 *
 * Streams are passed as `void*` holding a cudaStream_t (NULL = the legacy default stream).
 * All entry points are host functions; bsgemv_run only enqueues work and never synchronises.
 * A plan may be used by one stream at a time: its cross-CTA reduction workspace is shared by
 * every call made with it.  Status codes are returned; no exception crosses the ABI.
 */
#ifndef BSGEMV_H_
#define BSGEMV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct bsgemv_plan_s* bsgemv_plan_t; /* opaque; owned by the library */

enum bsgemv_format {
  BSGEMV_INT4 = 1,
  BSGEMV_INT8 = 2,
  BSGEMV_FP8_E4M3 = 3,
  BSGEMV_NVFP4 = 4
};
/* OR-ed into `format`: the activations (and the output) are bf16 instead of fp16. */
#define BSGEMV_ACT_BF16 0x100

enum bsgemv_status {
  BSGEMV_OK = 0,
  BSGEMV_ERR_INVALID_ARG = -1,    /* NULL pointer, M out of range for the call, bad enum ... */
  BSGEMV_ERR_UNSUPPORTED = -2,    /* shape / block size / format combination not provided,
                                     or no sm_103a device */
  BSGEMV_ERR_MISALIGNED = -3,     /* A, W or y not 16-byte aligned */
  BSGEMV_ERR_M_TOO_LARGE = -4,    /* M > the plan's max_M */
  BSGEMV_ERR_CUDA = -5,           /* a CUDA runtime/driver call failed */
  BSGEMV_ERR_WRONG_DEVICE = -6,   /* the current device is not the plan's device */
  BSGEMV_ERR_DEVICE_TIMEOUT = -7, /* a kernel gave up a bounded wait (reported by
                                     bsgemv_device_status) */
  BSGEMV_ERR_SCRATCH_LIMIT = -8   /* bsgemv_run_noalloc: the problem needs more than the fixed
                                     scratch area holds */
};

/* Variants a plan can run (bsgemv_geometry.variant, bsgemv_plan_set_override). */
enum bsgemv_variant {
  BSGEMV_VARIANT_AUTO = 0,
  BSGEMV_VARIANT_MMA = 1,        /* tensor-core mma.sync m16n8k16, fp32 accumulate */
  BSGEMV_VARIANT_CUDA_CORE = 2   /* CUDA-core packed fp32 FMA (fma.rn.f32x2) over the same
                                    copies, decoders and reductions; plans with max_M <= 8.  A
                                    measured alternative: the tensor-core variant is faster for
                                    every format and M */
};

/* What a plan chose.  Filled by bsgemv_plan_describe / bsgemv_geometry_for. */
typedef struct {
  int variant;           /* enum bsgemv_variant */
  int rows_per_tile;     /* output columns n per CTA tile */
  int k_per_stage;       /* k elements per pipeline stage */
  int stages;            /* depth of the shared-memory ring */
  int consumer_warps;    /* warps that decode and multiply; one more warp issues the copies */
  int ctas;              /* persistent CTAs launched */
  int ctas_per_sm;       /* CTAs resident per SM the geometry was sized for */
  int sm_count;          /* SM count the geometry was derived for */
  int64_t tiles;         /* ceil(N / rows_per_tile) */
  int64_t stages_per_tile;
  int64_t total_stages;  /* tiles * stages_per_tile: the work split evenly over the CTAs */
  int smem_bytes;        /* dynamic shared memory per CTA */
  int64_t workspace_bytes;
  int cluster;           /* how a tile's K is split: 0 = stream-K over all CTAs with a global
                            last-arriver reduction; C >= 1 = C CTAs per tile in one thread-block
                            cluster, reduced in the cluster leader's shared memory */
} bsgemv_geometry;

/* How a plan splits the K of a tile over CTAs (bsgemv_plan_set_split). */
enum bsgemv_split {
  BSGEMV_SPLIT_AUTO = 0,      /* cluster split where its per-CTA work is within one stage of
                                 stream-K's, else stream-K */
  BSGEMV_SPLIT_STREAM_K = 1,  /* the tiles x stages space cut into equal ranges over all CTAs */
  BSGEMV_SPLIT_CLUSTER = 2    /* each tile split over the CTAs of one cluster, shares differing
                                 by at most one stage */
};

/*
 * Create a plan for one weight shape.  format = enum bsgemv_format, optionally | BSGEMV_ACT_BF16.
 * block_size: int4/int8 one of 16, 32, 64, 128, 256; fp8 128; nvfp4 16.
 * has_zp: 0 or 1 (int formats only; must be 0 for fp8 and nvfp4).
 * N >= 1 (any tail); K >= 64 with K % 64 == 0 and K % block_size == 0; 1 <= max_M <= 32 (the
 * pages' decode GEMVs take M <= 16; a plan for up to 24 rows runs three n8 activation tiles at
 * 3 CTAs per SM, or four at 2 CTAs per SM where that keeps a cluster split of its tiles; a plan
 * for up to 32 rows runs four at 2 CTAs per SM.  Size a plan for the largest M it serves).
 * Uses the current CUDA device, which must be sm_103 (GB300).  Allocates the plan's own device
 * workspace (cross-CTA partial sums, arrival counters and an error word, all zeroed here) with
 * cudaMalloc; every call reuses it and the kernels leave the counters at zero.
 * On success *out holds the plan; on error *out is NULL and a status < 0 is returned.
 */
int bsgemv_plan(bsgemv_plan_t* out, int format, int block_size, int has_zp, int64_t N, int64_t K,
                int max_M);

/*
 * Enqueue y = A . deq(W)^T for the first M (1 <= M <= max_M) rows of A on `stream`.
 * Pointers as in the layout table above (device memory).  Checks arguments, alignment and the
 * current device, launches one kernel and returns cudaGetLastError's result; it does not wait.
 * Results depend only on the plan and the inputs: the same row of A gives bit-identical
 * output for every M, and repeated calls are bit-identical.
 */
int bsgemv_run(bsgemv_plan_t plan, const void* A, const void* W, const void* scales,
               const void* zp, void* y, int M, void* stream);

/*
 * y = A . deq(W)^T + bias: as bsgemv_run, plus `bias`, N values in the activation dtype (device
 * memory, 2-byte aligned, caller-owned), added to every row's fp32 sum before the one rounding.
 * ("[CUDA] Block-scaled MatMul decode GEMV: tensor cores, packed FP4 decode and M-tiling",
 * Tests: the FP8 and FP4 operators take an optional bias; "[CUDA] Pin FP8 GEMV residency for
 * grids just past two blocks per SM", Tests.)  NULL bias: BSGEMV_ERR_INVALID_ARG (call
 * bsgemv_run instead).  Same determinism as bsgemv_run: rows are bit-identical across M.
 */
int bsgemv_run_bias(bsgemv_plan_t plan, const void* A, const void* W, const void* scales,
                    const void* zp, const void* bias, void* y, int M, void* stream);

/*
 * Same as bsgemv_run, but A and y are HOST memory (pinned memory gives asynchronous copies):
 * A is copied into the plan's device staging buffer, the GEMV runs, y is copied back, and the
 * call returns after the stream has finished (the host buffers are ready on return).  W,
 * scales and zp stay device pointers.  The staging buffer (max_M * (K + N) activation
 * elements) is allocated by the first call and freed by bsgemv_destroy.  When both host
 * buffers are pinned and 16-byte aligned they are used through their device mapping: a small
 * kernel copies A into the staging buffer (its start-up overlaps the neighbouring kernels like
 * the GEMV's own) and the GEMV writes y straight into y_host; otherwise A and y go through the
 * staging buffer by copy-engine transfers (cudaMemcpyAsync).
 */
int bsgemv_run_host(bsgemv_plan_t plan, const void* A_host, const void* W, const void* scales,
                    const void* zp, void* y_host, int M, void* stream);

/*
 * bsgemv_run_host without the final wait: the copy of A in, the GEMV and the copy of y out are
 * enqueued on `stream` and the call returns.  y_host holds the result once the stream has been
 * synchronised, and A_host must not change before then.  With pinned host memory the copies are
 * asynchronous, so a step of several GEMVs costs one synchronisation, not one per GEMV.  Calls
 * on one plan share its staging buffer: issue them on one stream (stream order keeps each
 * call's copy of A after the previous call's copy of y).
 */
int bsgemv_run_host_async(bsgemv_plan_t plan, const void* A_host, const void* W,
                          const void* scales, const void* zp, void* y_host, int M, void* stream);

/* Free the plan and its device memory (synchronises the device first).  NULL is a no-op. */
int bsgemv_destroy(bsgemv_plan_t plan);

/* Static, human-readable name of a status code. */
const char* bsgemv_status_string(int status);

/*
 * Test hook: write the dequantised weight deq(W) as fp32 [N, K] to `out` (device, caller-owned,
 * N * K floats), through the same register decoders and fragment mapping as the GEMV.  Each
 * value is the exact dequantised weight rounded once to fp32 (exact for int4/int8; for fp8 and
 * nvfp4 one rounding of the exact product).  Enqueued on `stream`.
 */
int bsgemv_debug_dequant(bsgemv_plan_t plan, const void* W, const void* scales, const void* zp,
                         float* out, void* stream);

/*
 * Choose how the plan splits each tile's K over CTAs (no counterpart on the pages, whose kernels
 * use a fixed split-K or none: an A/B and testing aid like bsgemv_plan_set_override).
 * split = enum bsgemv_split; cluster_size (CLUSTER only) = CTAs per tile, 1..16, 0 = chosen by
 * the plan from the SM count.  Returns BSGEMV_ERR_UNSUPPORTED when the tiles x cluster_size
 * CTAs do not fit one wave of the device or cluster_size exceeds the stages of a tile; the plan
 * is then unchanged.  Not thread-safe with bsgemv_run on the same plan.
 */
int bsgemv_plan_set_split(bsgemv_plan_t plan, int split, int cluster_size);

/*
 * A/B override for measurements: variant (enum bsgemv_variant, 0 = keep; CUDA_CORE needs a plan
 * with max_M <= 8, else BSGEMV_ERR_UNSUPPORTED), ctas (persistent
 * CTAs of a stream-K split, 0 = keep; under BSGEMV_SPLIT_AUTO a CTA count selects stream-K),
 * rows_per_tile (output columns per CTA tile: 64 or 128, 0 = keep; 128 needs a plan with
 * max_M <= 16 and the tensor-core variant, else BSGEMV_ERR_UNSUPPORTED), stages (ring depth,
 * 0 = keep).
 * Changes the summation order, so results are bit-identical only between calls made under the
 * same settings.  Returns BSGEMV_ERR_UNSUPPORTED for a setting the plan cannot run.
 */
int bsgemv_plan_set_override(bsgemv_plan_t plan, int variant, int ctas, int rows_per_tile,
                             int stages);

/*
 * Measure this plan's candidate geometries on the device and keep the fastest (the "online
 * profiler" that "[CUDA] Batched small-M GEMV for MatMulNBits (4-bit/8-bit)", review, proposes
 * instead of thresholds tuned on one GPU).  Candidates, in two rounds: first the K split under
 * each tile height (the automatic one, 64 and 128 rows) -- the automatic choice, stream-K over the
 * default grid and over 1 .. 4 CTAs per SM, and thread-block clusters of 2 .. 8 CTAs per tile --
 * then the ring depth of the fastest (2, 3, 4, 6, 8 or 12 stages, at the same CTAs per SM);
 * candidates the plan cannot run are skipped.  They are timed in the regime the calls run in:
 * back to back on one stream (a CUDA graph of `reps` (1 .. 100) rounds over R copies of W,
 * scales and zp, R copies >= 3x the L2, at most 8, so that no call finds its weights in L2),
 * with the caller's A and y (y is overwritten): calls of M rows plus, when M > 1, calls of one
 * row in a graph of their own (the chosen geometry serves every M of the plan).  The copies, a private
 * stream and the graphs are made and freed here.  Another geometry replaces the automatic
 * choice only if it is more than 1 % faster, in the search and again when the two are timed in
 * turn, twice each, at the end.
 * Synchronises `stream` first and returns when done; not for use inside stream capture.
 * Afterwards every call of the plan runs the chosen geometry, so rows stay bit-identical across
 * M from then on (results may differ in the last bits from calls made before, as the
 * summation order can change).  On an error the plan keeps its previous settings.
 */
int bsgemv_plan_autotune(bsgemv_plan_t plan, const void* A, const void* W, const void* scales,
                         const void* zp, void* y, int M, int reps, void* stream);

/* Copy the plan's current geometry into *g. */
int bsgemv_plan_describe(bsgemv_plan_t plan, bsgemv_geometry* g);

/*
 * Pure host function, no CUDA call: the geometry bsgemv_plan would choose for this problem on a
 * device with `sm_count` SMs (and the sm_103 shared-memory budget).  Returns the same status
 * bsgemv_plan would return for invalid arguments.
 */
int bsgemv_geometry_for(int format, int block_size, int has_zp, int64_t N, int64_t K, int max_M,
                        int sm_count, bsgemv_geometry* g);

/*
 * Synchronise `stream`, then read and clear the plan's device error word.  Returns BSGEMV_OK,
 * BSGEMV_ERR_DEVICE_TIMEOUT if a kernel of this plan abandoned a bounded wait since the last
 * check, or BSGEMV_ERR_CUDA if the synchronisation failed.  plan = NULL reads and clears the
 * error word of bsgemv_run_noalloc on the current device instead (kept across its calls until
 * read here).  Every wait of the kernels is bounded (4 s): a kernel that gives one up stops
 * reading its copies, waits (bounded again) for the copies it issued to land, completes its
 * partial sums so that the plan stays usable, and returns; its output is not valid.
 */
int bsgemv_device_status(bsgemv_plan_t plan, void* stream);

/*
 * Test hook of the failure path above (the method's pages have no counterpart; it exercises this
 * library's bounded waits without faulting the GPU).  skip_stage >= 0: in the plan's next calls
 * the copy warp of CTA 0 leaves out stage `skip_stage` of that CTA's range (nothing is copied
 * for it, so its consumer warps' wait on it runs out); -1: none.  wait_ns > 0: the calls' waits
 * give up after wait_ns nanoseconds instead of 4 s; 0: the default.  Host only, no CUDA call;
 * returns BSGEMV_ERR_INVALID_ARG for NULL, skip_stage < -1 or wait_ns < 0.
 * bsgemv_plan_set_test_fault(plan, -1, 0) restores normal calls.
 */
int bsgemv_plan_set_test_fault(bsgemv_plan_t plan, int skip_stage, int64_t wait_ns);

/*
 * The GEMV without any allocation, for callers that cannot call cudaMalloc: runtimes that own
 * all device memory up front, code running inside another framework's memory pool, paths where
 * an allocation could fail or synchronise at the wrong moment.  (The method's pages have no
 * counterpart; this is a property of this library's interface.)
 *
 * Arguments as bsgemv_plan plus bsgemv_run; no plan is created.  Every call runs the geometry of
 * a plan sized for 16 rows, whatever its M: a row's result is bit-identical for every M and
 * equal to bsgemv_plan(..., max_M = 16) + bsgemv_run.  Instead of a plan's cudaMalloc'd
 * workspace the cross-CTA reduction uses one fixed scratch area compiled into the library (a
 * file-scope device array of about 7.6 MiB that every GPU loading the library holds until the
 * process exits).  Limits: M <= 16 (BSGEMV_ERR_INVALID_ARG beyond), N <= 524288 output columns
 * and at most 480 persistent CTAs (a 152-SM GB300 uses 456); beyond them the call returns
 * BSGEMV_ERR_SCRATCH_LIMIT and does nothing.  The first call on a device looks up the scratch
 * area's device address (with that device current), and so does the first call after the
 * device's context changed (e.g. after cudaDeviceReset); make such a first call before any
 * stream capture.  Every call on a device shares the one scratch area: calls that overlap on
 * the GPU (other streams, other host threads) race on it and give wrong results, so serialise
 * them.  Each call clears the counters it uses with cudaMemsetAsync on `stream` before its
 * kernel; it calls no cudaMalloc, cudaFree or allocating routine.  A bounded wait that ran out
 * in one of these calls is reported by bsgemv_device_status(NULL, stream).  Enqueue only; no
 * synchronisation.
 */
int bsgemv_run_noalloc(int format, int block_size, int has_zp, int64_t N, int64_t K,
                       const void* A, const void* W, const void* scales, const void* zp, void* y,
                       int M, void* stream);

/*
 * Dense small-N GEMV ("[CUDA] MatMul: add an opt-in split-K GEMV for small-N fp16 shapes",
 * Description): y[M, N] = A[M, K] . B[K, N] with A, B and y fp16 (act_bf16 = 0) or bf16
 * (act_bf16 = 1), B row-major [K, N] (the MatMul right-hand side), 1 <= M <= max_M <= 8.
 * K is split over the CTAs of a thread-block cluster per 64-column tile and the partial sums
 * are added in a fixed order (results are deterministic and rows bit-identical across M).
 * N % 8 == 0, K % 8 == 0 and K >= 16 (16-byte row pitches) run the TMA / tensor-core kernel, with
 * A, B and y 16-byte aligned; any other N >= 1, K >= 1 (the page's tests include N = 1) runs a
 * CUDA-core kernel (8 columns per CTA, K split over a cluster, the same fixed-order reduction),
 * with A, B and y 2-byte aligned.  Device memory.  The plan allocates only an error word.  Same
 * status conventions as above.
 */
typedef struct bsgemv_dense_plan_s* bsgemv_dense_plan_t;

int bsgemv_dense_plan(bsgemv_dense_plan_t* out, int act_bf16, int64_t N, int64_t K, int max_M);

/* Enqueue y = A . B for the first M rows of A on `stream` (one kernel; no synchronisation). */
int bsgemv_dense_run(bsgemv_dense_plan_t plan, const void* A, const void* B, void* y, int M,
                     void* stream);

/* The plan's geometry: rows_per_tile = 64 columns, k_per_stage = 64, cluster = CTAs per tile. */
int bsgemv_dense_describe(bsgemv_dense_plan_t plan, bsgemv_geometry* g);

/* Pure host function: the geometry bsgemv_dense_plan would choose with `sm_count` SMs. */
int bsgemv_dense_geometry_for(int act_bf16, int64_t N, int64_t K, int max_M, int sm_count,
                              bsgemv_geometry* g);

/* Synchronise `stream`, then read and clear the plan's error word (as bsgemv_device_status). */
int bsgemv_dense_device_status(bsgemv_dense_plan_t plan, void* stream);

/* Free the plan (synchronises the device first).  NULL is a no-op. */
int bsgemv_dense_destroy(bsgemv_dense_plan_t plan);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int bsgemv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* BSGEMV_H_ */
