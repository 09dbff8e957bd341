// The planned entry points' host code on a fake device (fake_cuda.cpp), under
// -fsanitize=address,undefined: plan creation, calls, failed workspace allocations and clears,
// the autotuner's choice, the host-buffer entry point's two paths, and destruction.  Every kernel
// launch checks the pointers it is handed; the program exits 0 and prints "ok" when every check
// holds.  (Compiled and run by tests/test_sanitizers.py.)
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "fake_cuda.h"

#define CHECK(cond)                                                              \
  do {                                                                           \
    if (!(cond)) {                                                               \
      std::fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond);    \
      return 1;                                                                  \
    }                                                                            \
  } while (0)

namespace {

using fake::g;

// int4, block 32, no zero points, fp16 activations, N = K = 4096 (plans for 16 rows take
// 64-row tiles in 6-CTA clusters, 384 CTAs, on 152 SMs)
constexpr int64_t kN = 4096, kK = 4096;

struct Buffers {
  void *A, *W, *s, *y;
};

Buffers device_buffers() {
  return {fake::device_alloc(16 * kK * 2), fake::device_alloc(kN * kK / 2),
          fake::device_alloc(kN * (kK / 32) * 2), fake::device_alloc(16 * kN * 2)};
}

bool same(const bsgemv_geometry& a, const bsgemv_geometry& b) {
  return std::memcmp(&a, &b, sizeof(a)) == 0;
}

int run(bsgemv_plan_t p, const Buffers& b, int M) {
  return bsgemv_run(p, b.A, b.W, b.s, nullptr, b.y, M, nullptr);
}

// Autotune a fresh int4 plan for 16 rows under `cost`; returns its geometry afterwards.
int tuned(const Buffers& b, std::function<double(const fake::Launch&)> cost, bsgemv_geometry* out) {
  bsgemv_plan_t p = nullptr;
  if (bsgemv_plan(&p, BSGEMV_INT4, 32, 0, kN, kK, 16) != BSGEMV_OK) return -1;
  const size_t live = fake::live_allocations();
  g.cost = std::move(cost);
  const int rc = bsgemv_plan_autotune(p, b.A, b.W, b.s, nullptr, b.y, 16, 2, nullptr);
  g.cost = nullptr;
  bsgemv_plan_describe(p, out);
  // the tuner's weight copies, stream, events and graphs are gone; the plan still runs
  const bool clean = fake::live_allocations() == live;
  const long v0 = g.violations;
  const int rr = run(p, b, 16);
  bsgemv_destroy(p);
  if (rc != BSGEMV_OK || rr != BSGEMV_OK || !clean || g.violations != v0) return -2;
  return 0;
}

bool is_auto(const bsgemv_geometry& t) {
  return t.rows_per_tile == 64 && t.cluster == 6 && t.ctas == 384;
}

}  // namespace

int main() {
  const Buffers b = device_buffers();
  CHECK(b.A && b.W && b.s && b.y);
  const size_t own = fake::live_allocations();

  // 1. a plan on the device takes the host predicate's geometry, for every format
  struct P {
    int fmt, bs, zp;
    int64_t N, K;
    int max_M;
  };
  const P probs[] = {{BSGEMV_INT4, 32, 0, 4096, 4096, 16}, {BSGEMV_INT4, 32, 1, 151936, 4096, 8},
                     {BSGEMV_INT8 | BSGEMV_ACT_BF16, 128, 1, 12288, 4096, 1},
                     {BSGEMV_FP8_E4M3, 128, 0, 5120, 17408, 8}, {BSGEMV_NVFP4, 16, 0, 2048, 2048, 4},
                     {BSGEMV_INT8, 64, 0, 333, 2048, 32}};
  for (const P& q : probs) {
    bsgemv_plan_t p = nullptr;
    CHECK(bsgemv_plan(&p, q.fmt, q.bs, q.zp, q.N, q.K, q.max_M) == BSGEMV_OK && p);
    bsgemv_geometry a, e;
    CHECK(bsgemv_plan_describe(p, &a) == BSGEMV_OK);
    CHECK(bsgemv_geometry_for(q.fmt, q.bs, q.zp, q.N, q.K, q.max_M, 152, &e) == BSGEMV_OK);
    CHECK(same(a, e));
    CHECK(bsgemv_destroy(p) == BSGEMV_OK);
  }
  CHECK(fake::live_allocations() == own && g.violations == 0);

  // 2. a workspace allocation that fails leaves the plan with its geometry and workspace
  bsgemv_plan_t p = nullptr;
  CHECK(bsgemv_plan(&p, BSGEMV_INT4, 32, 0, kN, kK, 16) == BSGEMV_OK);
  bsgemv_geometry g0, cur;
  bsgemv_plan_describe(p, &g0);
  CHECK(is_auto(g0));
  CHECK(run(p, b, 16) == BSGEMV_OK && g.launches == 1 && g.violations == 0);
  CHECK(g.last.ctas == 384 && g.last.cluster == 6);
  g.fail_malloc = 1;  // stream-K over 4 x 152 CTAs needs more partial slots
  CHECK(bsgemv_plan_set_override(p, 0, 4 * 152, 0, 0) == BSGEMV_ERR_CUDA);
  CHECK(g.fail_malloc == 0);
  bsgemv_plan_describe(p, &cur);
  CHECK(same(cur, g0));
  CHECK(run(p, b, 9) == BSGEMV_OK && g.launches == 2 && g.violations == 0);
  CHECK(g.last.ctas == 384 && g.last.M == 9);
  CHECK(bsgemv_device_status(p, nullptr) == BSGEMV_OK);

  // 3. a clear that fails leaves no workspace: calls are refused until a change succeeds
  g.memset_broken = true;
  CHECK(bsgemv_plan_set_override(p, 0, 4 * 152, 0, 0) == BSGEMV_ERR_CUDA);
  CHECK(run(p, b, 16) == BSGEMV_ERR_CUDA && g.launches == 2);
  CHECK(bsgemv_device_status(p, nullptr) == BSGEMV_ERR_CUDA);
  g.memset_broken = false;
  CHECK(bsgemv_plan_set_override(p, 0, 2 * 152, 0, 0) == BSGEMV_OK);
  CHECK(run(p, b, 16) == BSGEMV_OK && g.launches == 3 && g.violations == 0);
  CHECK(g.last.ctas == 304 && g.last.cluster == 0);
  CHECK(bsgemv_device_status(p, nullptr) == BSGEMV_OK);

  // splits and the bias epilogue: a forced split shows in the geometry and the launch; a bias
  // reaches only the call that passes it; a call from another device is refused
  CHECK(bsgemv_plan_set_split(p, BSGEMV_SPLIT_CLUSTER, 4) == BSGEMV_OK);
  bsgemv_plan_describe(p, &cur);
  CHECK(cur.cluster == 4 && cur.ctas == cur.tiles * 4);
  CHECK(bsgemv_plan_set_split(p, BSGEMV_SPLIT_STREAM_K, 4) == BSGEMV_ERR_INVALID_ARG);
  CHECK(bsgemv_plan_set_split(p, 7, 0) == BSGEMV_ERR_INVALID_ARG);
  bsgemv_plan_describe(p, &g0);
  CHECK(same(cur, g0));  // refused settings change nothing
  void* bias = fake::device_alloc(kN * 2);
  CHECK(bias != nullptr);
  CHECK(bsgemv_run_bias(p, b.A, b.W, b.s, nullptr, bias, b.y, 3, nullptr) == BSGEMV_OK);
  CHECK(g.last.bias == bias && g.last.cluster == 4 && g.last.M == 3);
  CHECK(bsgemv_run_bias(p, b.A, b.W, b.s, nullptr, static_cast<char*>(bias) + 1, b.y, 3,
                        nullptr) == BSGEMV_ERR_MISALIGNED);
  CHECK(bsgemv_run_bias(p, b.A, b.W, b.s, nullptr, nullptr, b.y, 3, nullptr) ==
        BSGEMV_ERR_INVALID_ARG);
  CHECK(run(p, b, 3) == BSGEMV_OK && g.last.bias == nullptr);
  g.current_device = 1;
  const long before = g.launches;
  CHECK(run(p, b, 3) == BSGEMV_ERR_WRONG_DEVICE && g.launches == before);
  g.current_device = 0;
  CHECK(bsgemv_plan_set_split(p, BSGEMV_SPLIT_AUTO, 0) == BSGEMV_OK);
  CHECK(bsgemv_plan_set_override(p, 0, 0, 64, 0) == BSGEMV_OK);
  CHECK(bsgemv_destroy(p) == BSGEMV_OK);
  CHECK(cudaFree(bias) == cudaSuccess);
  CHECK(fake::live_allocations() == own && g.violations == 0);

  // 4. the autotuner: a clearly faster geometry is kept ...
  auto streamk304 = [](const fake::Launch& l) { return l.cluster == 0 && l.ctas == 304; };
  bsgemv_geometry t;
  CHECK(tuned(b, [&](const fake::Launch& l) { return streamk304(l) ? 8.0 : 10.0; }, &t) == 0);
  CHECK(t.cluster == 0 && t.ctas == 304 && t.rows_per_tile == 64);
  // ... one within 1 % is not ...
  CHECK(tuned(b, [&](const fake::Launch& l) { return streamk304(l) ? 9.95 : 10.0; }, &t) == 0);
  CHECK(is_auto(t));
  // ... nor one faster on calls of M rows but slower on calls of one row ...
  CHECK(tuned(b, [&](const fake::Launch& l) {
          return streamk304(l) ? (l.M == 16 ? 9.0 : 12.0) : 10.0;
        }, &t) == 0);
  CHECK(is_auto(t));
  // ... nor one that was fast only the first time it was timed (the confirmation round)
  long first = -1;
  CHECK(tuned(b, [&](const fake::Launch& l) {
          if (!streamk304(l) || !g.capturing) return 10.0;  // (untimed eager calls)
          if (first < 0) first = g.capture_sessions;
          return g.capture_sessions == first ? 8.0 : 10.2;
        }, &t) == 0);
  CHECK(first > 0 && is_auto(t));
  CHECK(fake::live_allocations() == own && g.violations == 0);

  // 5. host buffers: pinned and 16-byte aligned ones through their mapping (a copy kernel for
  // A, the outputs stored straight into y_host), others through copy-engine transfers
  CHECK(bsgemv_plan(&p, BSGEMV_INT4, 32, 0, kN, kK, 4) == BSGEMV_OK);
  void* Ah = std::aligned_alloc(256, 4 * kK * 2);
  void* yh = std::aligned_alloc(256, 4 * kN * 2 + 256);
  CHECK(Ah && yh);
  std::memset(Ah, 0, 4 * kK * 2);
  const long copies0 = g.host_copies, memcpys0 = g.memcpy_calls;
  CHECK(bsgemv_run_host(p, Ah, b.W, b.s, nullptr, yh, 4, nullptr) == BSGEMV_OK);  // pageable
  CHECK(g.host_copies == copies0 && g.memcpy_calls == memcpys0 + 2);
  CHECK(g.last.y != yh && fake::device_range(g.last.y, 4 * kN * 2));
  fake::register_pinned(Ah, 4 * kK * 2);
  fake::register_pinned(yh, 4 * kN * 2 + 256);
  CHECK(bsgemv_run_host(p, Ah, b.W, b.s, nullptr, yh, 4, nullptr) == BSGEMV_OK);  // pinned
  CHECK(g.host_copies == copies0 + 1 && g.memcpy_calls == memcpys0 + 2);
  CHECK(g.last.y == yh && fake::device_range(g.last.A, 4 * kK * 2));
  void* yh_odd = static_cast<char*>(yh) + 2;  // pinned, but not 16-byte aligned
  CHECK(bsgemv_run_host(p, Ah, b.W, b.s, nullptr, yh_odd, 4, nullptr) == BSGEMV_OK);
  CHECK(g.host_copies == copies0 + 1 && g.memcpy_calls == memcpys0 + 4 && g.last.y != yh_odd);
  CHECK(bsgemv_run_host(p, Ah, b.W, b.s, nullptr, yh, 5, nullptr) == BSGEMV_ERR_M_TOO_LARGE);
  CHECK(bsgemv_destroy(p) == BSGEMV_OK);
  CHECK(g.violations == 0);
  std::free(Ah);
  std::free(yh);

  for (void* q : {b.A, b.W, b.s, b.y}) CHECK(cudaFree(q) == cudaSuccess);
  CHECK(fake::live_allocations() == 0 && g.violations == 0);
  std::printf("ok %ld launches\n", g.launches);
  return 0;
}
