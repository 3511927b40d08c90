// Device helpers of the fused prefill kernel (fused2.cu): per-CTA control
// word, optional tracing, bounded waits that record an error instead of hanging, and the
// ring and tile bookkeeping of a job.
#pragma once

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace fused_common {

struct Ctl {
  int group;       // written by cluster rank 0 into both CTAs
  int abort;
  uint32_t tmem;
};

// Optional tracing: per role slot (group * 2 + cluster rank) kTraceWords words
//   [0] start ns  [1] end ns  [2] cta << 32 | producer << 31 | job
//   [3] ns waiting on the other role kind (consumer: `ready` flags; producer: `consumed`)
//   [4] ns the MMA thread waited for operands (kv_full / prod_full)
//   [5] ns the MMA thread waited for softmax (p_full) or conversion (acc_empty)
//   [6] ns softmax warp 0 waited for S (s_full)   [7] stages / passes
struct TraceAcc {
  unsigned long long t = 0;
  __device__ __forceinline__ uint64_t begin(const FusedParams& p) const { return p.trace ? global_timer_ns() : 0; }
  __device__ __forceinline__ void end(const FusedParams& p, uint64_t t0) { if (p.trace) t += global_timer_ns() - t0; }
};
__device__ __forceinline__ void trace_put(const FusedParams& p, int role, int word, unsigned long long v) {
  if (p.trace) p.trace[(size_t)role * kTraceWords + word] = v;
}
// Per-stage timestamps of one role (after the per-role words): 8 words per stage
//   [0] K load issued  [1] V load issued  [2] MMA saw K  [3] MMA issued S
//   [4] MMA saw P  [5] MMA saw V (PV issued next)  [6] softmax saw S  [7] softmax published P
// Stage kTraceOnce holds one-off stamps of the role (consumer: Q load start,
// Q landed, Q ready, last PV seen, epilogue done).
constexpr int kTraceOnce = 4000;
__device__ __forceinline__ void trace_stage(const FusedParams& p, int role, int stage, int word) {
  if (p.trace && role == p.trace_detail_role && stage < 4096)
    p.trace[(size_t)p.n_groups * 2 * kTraceWords + (size_t)stage * 8 + word] = global_timer_ns();
}

__device__ __forceinline__ bool aborted_global(const FusedParams& p) { return ld_volatile_u32(p.err) != 0u; }

// Bounded mbarrier wait; on timeout records the error and returns false.
__device__ __forceinline__ bool wait_bar(const FusedParams& p, uint32_t bar, uint32_t parity) {
  if (mbar_wait(bar, parity, p.wait_limit_ns)) return true;
  atomicOr(p.err, kErrTimeout);
  return false;
}

// Same, decided once for the whole warp (every lane must call it together), so a
// timeout never splits a warp before a warp-collective tcgen05.ld/st.
__device__ __forceinline__ bool wait_bar_warp(const FusedParams& p, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_bar(p, bar, parity));
}

// Bounded wait until *flag >= target (acquire).  Gives up early when another
// CTA has already recorded an error.
__device__ inline bool wait_flag_geq(const FusedParams& p, const uint32_t* flag, uint32_t target) {
  if (ld_acquire_gpu(flag) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_gpu(flag) < target) {
    if (global_timer_ns() - t0 > p.wait_limit_ns || aborted_global(p)) {
      atomicOr(p.err, kErrTimeout);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

// Number of 128-key tiles consumer `ci` (queries 128 ci .. 128 ci + 127 of the
// request) of job `J` attends to (causal clip).
__device__ __forceinline__ int consumer_tiles(const Job& J, int ci) {
  const int q0 = ci * 128;
  const int nq = min(128, J.q_count - q0);
  if (nq <= 0) return 0;
  const int last_tok = J.q_tok ? J.q_tok[J.q_begin + q0 + nq - 1] : J.q_tok0 + q0 + nq - 1;
  const int k_end = min(J.k_end, last_tok + 1);
  if (k_end <= J.k_begin) return 0;
  return (k_end - J.t0 + 127) >> 7;
}

// Token index of query row q (within the job's rows; rows past the job's
// last are padding and take its last row's token).
__device__ __forceinline__ int query_token(const Job& J, int q) {
  return J.q_tok ? J.q_tok[J.q_begin + min(q, J.q_count - 1)] : J.q_tok0 + q;
}

// Ring slot of tile t (the depth is a power of two).
__device__ __forceinline__ int ring_slot(const FusedParams& p, int t) { return t & (p.ring_depth - 1); }

__device__ __forceinline__ uint32_t* ready_flag(const FusedParams& p, int job, int slot) {
  return p.flags + (size_t)job * (2 * (size_t)p.ring_depth) + slot;
}
__device__ __forceinline__ uint32_t* consumed_flag(const FusedParams& p, int job, int slot) {
  return p.flags + (size_t)job * (2 * (size_t)p.ring_depth) + p.ring_depth + slot;
}

// Ring tiles [t, end) (end - t <= 8) that are produced, polled together: the
// relaxed reads of their ready flags go out at once and one fence makes the
// ones seen an acquire.  Returns the first tile of the range not yet seen
// produced (> t), waiting (bounded) until tile t is; -1 after a timeout or
// another CTA's error.
__device__ inline int wait_ready_window(const FusedParams& p, int job, int t, int end) {
  uint64_t t0 = 0;
  for (;;) {
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = t + i < end ? ld_relaxed_gpu(ready_flag(p, job, ring_slot(p, t + i))) : 0u;
    int k = t;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (k == t + i && t + i < end && v[i] >= (uint32_t)(t + i + 1)) k = t + i + 1;
    if (k > t) {
      fence_acq_rel_gpu();
      return k;
    }
    if (t0 == 0) t0 = global_timer_ns();
    else if (global_timer_ns() - t0 > p.wait_limit_ns || aborted_global(p)) {
      atomicOr(p.err, kErrTimeout);
      return -1;
    }
    __nanosleep(32);
  }
}

// Adds 1 to the consumed counts of ring tiles [t, t + n), whose reads (async
// proxy) are complete, behind a single release fence.
__device__ inline void release_tiles(const FusedParams& p, int job, int t, int n) {
  fence_proxy_async_global();
  fence_acq_rel_gpu();
  for (int i = 0; i < n; ++i) red_relaxed_gpu_add(consumed_flag(p, job, ring_slot(p, t + i)), 1u);
}

// Row of logical block `lb` of the job's request in the gathered rows (the
// gather pass copied the request's blocks in logical order from row_block0 on;
// it also reported any bad block id).  Rows past the request's blocks are
// read but belong to keys outside the job's range, which are masked.
__device__ __forceinline__ int block_row(const Job& J, int lb) { return (J.row_block0 + lb) * kBlock; }

}  // namespace fused_common
}  // namespace mla
