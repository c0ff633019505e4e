// Device helpers shared by the persistent pipelines: bounded mbarrier waits
// (timeouts recorded in the CTA's error bits, an abort flag every role polls)
// and a block-wide scan.
#pragma once
#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace gmmfr {

struct Ctl {
  volatile int* abort;
  uint32_t* err;  // shared-memory error bits of this CTA
  int64_t timeout_ns;
};

// The polling loop of a bounded wait: gives up when another role aborted or after
// timeout_ns (then records the timeout and aborts).
__device__ __forceinline__ bool wait_bar_loop(uint32_t bar, uint32_t parity, const Ctl& c) {
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*c.abort) return false;
    if (ptx::globaltimer() - t0 > (uint64_t)c.timeout_ns) {
      *c.abort = 1;
      atomicOr(c.err, kErrTimeout);
      return false;
    }
  }
}
static __device__ __noinline__ bool wait_bar_poll(uint32_t bar, uint32_t parity, Ctl c) {
  return wait_bar_loop(bar, parity, c);
}

// Bounded wait for the phase of `parity` to complete.  kOutOfLine: only the first try_wait is
// inlined and the polling loop is one shared out-of-line function, which keeps the role loops
// that call it small (the persistent kernels' instruction caches are their scarce resource:
// atomic-mode C1 37.9 -> 37.5 us, C5 1082.4 -> 1081.7 us per call); the deterministic
// instantiations, whose register budget the call disturbs (C5 1150 -> 1156 us), inline it.
template <bool kOutOfLine = true>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  if constexpr (kOutOfLine) return wait_bar_poll(bar, parity, c);
  else return wait_bar_loop(bar, parity, c);
}

// wait_bar for a whole warp: every lane waits in hardware (the warp stays
// converged and sleeps in try_wait), then a vote makes the outcome uniform, so
// a timeout seen by one lane can never split the warp.
template <bool kOutOfLine = true>
__device__ __forceinline__ bool warp_wait_bar(uint32_t bar, uint32_t parity, const Ctl& c) {
  const bool ok = wait_bar<kOutOfLine>(bar, parity, c);
  return __all_sync(0xffffffffu, ok) != 0;
}

// Wait used while draining after an abort: ignores the abort flag, fixed 1 s limit.
__device__ __forceinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > 1000000000ull) return false;
  }
  return true;
}

// Block-wide inclusive scan (sum or max) over kThreads threads; `total`
// gets the last value.  Every thread must call it.
template <bool kMax, int kThreads>
__device__ int64_t cta_scan(int64_t v, int64_t* scratch, int64_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kThreads / 32;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int64_t u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = kMax ? (u > v ? u : v) : v + u;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  int64_t carry = kMax ? INT64_MIN : 0, all = kMax ? INT64_MIN : 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int64_t u = scratch[w];
    if (w < warp) carry = kMax ? (u > carry ? u : carry) : carry + u;
    all = kMax ? (u > all ? u : all) : all + u;
  }
  if (warp > 0) v = kMax ? (carry > v ? carry : v) : v + carry;
  total = all;
  __syncthreads();
  return v;
}

}  // namespace gmmfr
