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
  int lane_ok;     // producer role: passes whose ring slot the lane's previous job is done with
};

// Optional tracing: per role slot (group * 2 + cluster rank) kTraceWords words
//   [0] start ns  [1] end ns  [2] cta << 32 | producer << 31 | job
//   [3] ns waiting on the other role kind (consumer: `ready` flags; producer: `consumed`)
//   [4] ns the MMA thread waited for operands (kv_full / prod_full)
//   [5] ns the MMA thread waited for softmax (p_full) or conversion (acc_empty)
//   [6] consumer: ns softmax warp 0 waited for S (s_full); producer: ns its row
//       loader waited for the ring lane's previous job   [7] stages / passes
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

// Bounded wait until the shared word *w >= target (acquire, CTA scope);
// gives up when this CTA aborts or another CTA records an error.
__device__ inline bool wait_shared_geq(const FusedParams& p, volatile Ctl* ctl, const int* w, int target) {
  if (ld_acquire_cta_s32(w) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_cta_s32(w) < target) {
    if (ctl->abort || global_timer_ns() - t0 > p.wait_limit_ns || aborted_global(p)) {
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

// Device view of job (piece, head) of the launch; its index is piece * H + head.
__device__ __forceinline__ Job make_job(const FusedParams& p, int piece, int head) {
  const Piece& P = p.pieces[piece];
  Job J;
  J.req = P.req;
  J.head = head;
  J.q_begin = P.q_begin;
  J.q_count = P.q_count;
  J.q_tok0 = P.q_tok0;
  J.q_tok = p.q_tok;
  J.k_begin = P.k_begin;
  J.k_end = P.k_end;
  J.t0 = P.k_begin & ~(kBlock - 1);
  J.n_tiles = (P.k_end - J.t0 + 127) >> 7;
  J.n_cons = P.n_cons;
  J.n_prod = P.n_prod;
  J.slot = P.slot;
  J.row_block0 = P.row_block0;
  J.rope_offset = P.rope_offset;
  J.n_exact_tiles = P.exact & 255;
  J.n_exact_pairs = P.exact >> 8;
  return J;
}

// Ring slot of tile t (the depth is a power of two).
__device__ __forceinline__ int ring_slot(const FusedParams& p, int t) { return t & (p.ring_depth - 1); }

// First of the four [128 x 64] bf16 blocks of ring slot `slot` of job `job`
// (K_nope cols 0-63, 64-127, V cols 0-63, 64-127).  Jobs take turns on
// ring_lanes lanes of ring_depth slots: job j writes a slot of lane
// j mod ring_lanes once job j - ring_lanes is done with it, so the rings of a
// launch span a fixed number of lanes, whatever its number of jobs, and a
// lane's slots are rewritten soon enough to be still in L2.
__device__ __forceinline__ int ring_block(const FusedParams& p, int job, int slot) {
  return ((job % p.ring_lanes) * p.ring_depth + slot) * 4;
}
// First of the two [128 x 64] bf16 blocks (cols 0-63, 64-127) of the K_nope
// residual K - bf16(K) of ring slot `slot` (< kExactSlots) of job `job`,
// after all the lanes' slots.
__device__ __forceinline__ int residual_block(const FusedParams& p, int job, int slot) {
  return p.ring_lanes * p.ring_depth * 4 + ((job % p.ring_lanes) * min(p.ring_depth, kExactSlots) + slot) * 2;
}

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
