// wst_common.cuh -- pieces shared by the three kernels and the host launcher:
// the workspace layout, device-side error latching, and bounded waits.
#pragma once

#include <cstdint>
#include "sm103.cuh"

namespace wst {

// Device status codes (same values as wst_status in include/wst.h).
enum : uint32_t {
  kOk = 0,
  kErrTimeout = 5,
  kErrBadOffsets = 6,
};

// First 256 bytes of every workspace.
struct WsHeader {
  uint32_t error;       // first latched device error (0 = none)
  uint32_t error_info;  // where it happened (role << 16 | detail)
  uint32_t reserved0;   // (unused; the flags' per-call value comes from the host)
  uint32_t reserved1;
  uint32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

constexpr size_t kWsHeaderBytes = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// IKBO workspace: header | flags[num_users] (256-B padded) | P[num_users][O][D] fp32
__host__ __device__ inline size_t ikbo_flags_offset() { return kWsHeaderBytes; }
__host__ __device__ inline size_t ikbo_partials_offset(int num_users) {
  return kWsHeaderBytes + align_up((size_t)num_users * 4, 256);
}
__host__ __device__ inline size_t workspace_bytes(int num_users, int O, int D) {
  if (num_users <= 0) return kWsHeaderBytes;
  return ikbo_partials_offset(num_users) + (size_t)num_users * O * D * 4;
}

// Roles, for error_info.
enum : uint32_t { kRoleProducer = 1, kRoleMma = 2, kRoleEpilogue = 3, kRoleFlag = 4 };

__device__ __forceinline__ void latch_error(WsHeader* ws, uint32_t code, uint32_t info) {
  if (atomicCAS(&ws->error, 0u, code) == 0u) atomicExch(&ws->error_info, info);
}

// Per-CTA guard for bounded waits: a CTA-wide abort flag in shared memory,
// the workspace (for latching) and the time limit.
struct Guard {
  WsHeader* ws;
  volatile uint32_t* abort;  // shared memory
  uint64_t limit_ns;
};

// Wait for completion of the mbarrier phase with parity `parity`.  Returns
// false if the CTA is aborting or the limit ran out (which latches
// kErrTimeout and raises the CTA abort flag).  Never spins without bound.
static __device__ __noinline__ bool wait_slow(const Guard& g, uint32_t bar, uint32_t parity,
                                       uint32_t info, bool cluster_scope) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (true) {
    bool done = cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    if (done) return true;
    if ((++it & 31u) == 0u) {
      if (*g.abort) return false;
      if (globaltimer_ns() - t0 > g.limit_ns || it > (1u << 28)) {
        *g.abort = 1u;
        latch_error(g.ws, kErrTimeout, info);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_phase(const Guard& g, uint32_t bar, uint32_t parity,
                                           uint32_t info) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(g, bar, parity, info, false);
}

__device__ __forceinline__ bool wait_phase_cluster(const Guard& g, uint32_t bar, uint32_t parity,
                                                   uint32_t info) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  return wait_slow(g, bar, parity, info, true);
}

// Warp-collective form: lane 0 waits, the outcome is broadcast to the warp.
__device__ __forceinline__ bool warp_wait_phase(const Guard& g, uint32_t bar, uint32_t parity,
                                                uint32_t info) {
  uint32_t ok = 0;
  if (lane_id() == 0) ok = wait_phase(g, bar, parity, info) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

__device__ __forceinline__ bool warp_wait_phase_cluster(const Guard& g, uint32_t bar,
                                                        uint32_t parity, uint32_t info) {
  uint32_t ok = 0;
  if (lane_id() == 0) ok = wait_phase_cluster(g, bar, parity, info) ? 1u : 0u;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// Bounded spin until *flag == want (acquire, gpu scope).
static __device__ __noinline__ bool wait_flag(const Guard& g, const uint32_t* flag, uint32_t want,
                                       uint32_t info) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t it = 0;
  while (ld_acquire_gpu(flag) != want) {
    __nanosleep(64);
    if ((++it & 15u) == 0u) {
      if (*g.abort) return false;
      if (globaltimer_ns() - t0 > g.limit_ns || it > (1u << 26)) {
        *g.abort = 1u;
        latch_error(g.ws, kErrTimeout, info);
        return false;
      }
    }
  }
  return true;
}

}  // namespace wst
