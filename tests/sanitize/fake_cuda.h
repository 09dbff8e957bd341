// The fake CUDA device of the host-only plan tests (fake_cuda.cpp): its state, which the test
// reads and steers.
#pragma once
#include <cstddef>
#include <cstdint>
#include <functional>

#include "../../block_scaled_bit_gb300/csrc/bsgemv_internal.h"

namespace fake {

// One kernel launch as the launchers saw it.
struct Launch {
  int M, mt, halves, ctas, cluster, stages;
  const void* A;
  const void* y;
  const void* partials;
  const void* bias;
};

struct State {
  // steering
  int fail_malloc = 0;   // > 0: the fail_malloc-th cudaMalloc from now fails
  int fail_memset = 0;   // > 0: the fail_memset-th cudaMemset from now fails
  bool memset_broken = false;  // every cudaMemset fails
  int current_device = 0;      // what cudaGetDevice reports (the fake device is 0)
  std::function<double(const Launch&)> cost;  // µs charged per launch (1 if unset)
  // observation
  long launches = 0, violations = 0, host_copies = 0, memcpy_calls = 0, maps_encoded = 0;
  long capture_sessions = 0;
  Launch last{};
  // clock and capture
  double clock_us = 0.0, capture_cost = 0.0;
  bool capturing = false;
};
extern State g;

bool device_range(const void* p, size_t n);
bool pinned_range(const void* p, size_t n);
size_t live_allocations();
void register_pinned(const void* p, size_t n);
void* device_alloc(size_t n);
void charge(const Launch& l);
void violation(const char* what);

}  // namespace fake
