// Persistent fused MLA prefill kernel on CTA pairs (tcgen05 cta_group::2).
//
// What it computes ("DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析",
// sections 4.2-4.4, with the query relocation of "RedKnot-MLA: Multi-Head
// Offline-Online Reuse for DeepSeek-V4 Long-Context Serving", section 2): per
// job (request, head, key range with one RoPE offset) the keys are
// up-projected once, K_nope | V = c_kv * kv_b_proj[:, head], and every query of
// the request attends to them with an online softmax that yields (out, lse).
//
// A queue of roles feeds the persistent grid.  Clusters of two CTAs run every
// role together and the pair's tensor-core work is issued by the first CTA
// (the leader) as M = 256 MMAs: rows 0..127 of A and of the accumulator live in
// the leader, rows 128..255 in its peer, and each CTA holds half of B.  So each
// CTA stores half of every key tile, which frees shared memory for Q and TMEM
// for a third score buffer:
//   producer pair  up-projects passes of 256 tokens (128 per CTA); CTA r holds
//                  the head's K_nope (r = 0) or V (r = 1) columns of
//                  kv_b_proj; the accumulators (all 256 columns of the 128
//                  tokens of the CTA) are double-buffered in TMEM, so the next
//                  pass runs while 256 threads convert the previous one to
//                  bf16 and store it into the job's ring (in L2);
//   consumer pair  two 128-query tiles of the job (CTA r owns tile 2k + r;
//                  Q, RoPE-rotated, in shared memory).  Per 128-key tile CTA r
//                  loads keys 64r..64r+63 of K (K_nope and k_rope) and columns
//                  64r..64r+63 of V; S = Q K^T lands in one of three TMEM
//                  buffers of each CTA, so the MMA can run two tiles ahead of
//                  the softmax; P is written back over S as bf16 and
//                  O += P V reads it from TMEM.
// Barriers the leader's MMA thread waits on (operands landed in both CTAs,
// P written in both) live in the leader and count both CTAs; barriers of MMA
// completion are signalled in both CTAs by multicast commits.
#include <cuda.h>

#include "fused_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {
using namespace fused_common;

constexpr int kThreads = 384;
constexpr uint32_t kAtomQ = 16384;                  // [128 rows x 128 B] swizzled block
constexpr uint32_t kAtom64 = 8192;                  // [64 rows x 128 B] swizzled block

// ---------------------------------------------------------------- shared memory (per CTA)
// consumer
constexpr int kKStages = 4, kVStages = 4, kSBufs = 3;
constexpr uint32_t kQBase = 0;                                     // q_nope lo | q_nope hi | rotated q_rope
constexpr uint32_t kKStageBytes = 3 * kAtom64;                     // this CTA's 64 keys: K_nope lo | hi | k_rope
constexpr uint32_t kVStageBytes = kAtomQ;                          // 128 keys x this CTA's 64 columns of V
constexpr uint32_t kKBase = 3 * kAtomQ;                            // 49152
constexpr uint32_t kVBase = kKBase + kKStages * kKStageBytes;      // 147456
constexpr uint32_t kXchgBase = kVBase + kVStages * kVStageBytes;   // 212992: row maxima / sums of the two halves
constexpr uint32_t kQResBase = kVBase + 3 * kVStageBytes;           // exact pairs: rotated q_rope residual (V stage 3)
constexpr uint32_t kConsumerEnd = kXchgBase + 6 * 128 * 4;
// producer: this CTA's 128 kv_b_proj columns stay resident for the role
constexpr int kPStages = 6;
constexpr uint32_t kPWBase = 0;                                    // W: 8 k-slices [64 x 128 columns]
constexpr uint32_t kPCBase = 8 * kAtomQ;                           // 131072: latent rows, [128 tokens x 64] a stage
constexpr uint32_t kPStageBytes = kAtomQ;
constexpr uint32_t kProducerEnd = kPCBase + kPStages * kPStageBytes;   // 229376
constexpr uint32_t kBarBase = kConsumerEnd > kProducerEnd ? kConsumerEnd : kProducerEnd;
constexpr uint32_t kNumBars = 27;
constexpr uint32_t kSmemBytes = kBarBase + 8 * kNumBars + 64 + 1024;
static_assert(kSmemBytes <= 232448, "more than 227 KB of shared memory per CTA");

// consumer barriers ("leader": only the leader's copy is used, it counts both CTAs)
constexpr uint32_t kBQReady = 0;          // leader, 8 arrivals (the 4 Q-loading warps of each CTA)
constexpr uint32_t kBKFull = 1;           // leader, 4: both halves of a K stage landed
constexpr uint32_t kBKEmpty = 5;          // both, 4: the MMAs reading a K stage are done
constexpr uint32_t kBVFull = 9;           // leader, 4
constexpr uint32_t kBVEmpty = 13;         // both, 4
constexpr uint32_t kBSFull = 17;          // both, 3: S of a buffer computed
constexpr uint32_t kBPFull = 20;          // leader, 3: P of a buffer written, one arrival per softmax warp
constexpr uint32_t kBPvDone = 23;         // both, 3: PV reading a buffer done
constexpr uint32_t kBQLand = 26;          // both, own: this CTA's Q rows landed (TMA)
// producer barriers
constexpr uint32_t kBProdFull = 0;                     // leader, kPStages
constexpr uint32_t kBProdEmpty = kPStages;             // both, kPStages
constexpr uint32_t kBAccFull = 2 * kPStages;           // both, 2
constexpr uint32_t kBAccEmpty = 2 * kPStages + 2;      // leader, 2: one arrival per conversion warp
constexpr uint32_t kBWFull = 2 * kPStages + 4;         // leader: the resident kv_b_proj columns of both CTAs landed
static_assert(kBWFull < kNumBars, "producer barriers");

// TMEM columns (per CTA)
constexpr uint32_t kTmO = 0;              // consumer: O [128 x 128] fp32
constexpr uint32_t kTmS = 128;            // consumer: S buffer b at 128 + 128 b (P as bf16 pairs in its first 64)
constexpr uint32_t kTmAcc = 0;            // producer: accumulator b at 256 b

constexpr uint32_t kIdescS = idesc_bf16(256, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(256, 128, false, true);
constexpr uint32_t kIdescUp = idesc_bf16(256, 256, false, true);
constexpr uint32_t kIdescUp8 = idesc_e4m3(256, 256);   // FP8 up-projection: E4M3 rows x E4M3 kv_b_proj, K-major

constexpr float kRescaleThreshold = 8.f;   // log2 units: P stays <= 256

// L2 policies: ring tiles are kept (evict_last: written, read by every
// consumer pair of the job, rewritten by the lane's next job), what streams
// through once (q, kv_b_proj columns, out and partial states) goes first.
// With p.l2_hints = 0 both are evict_normal.
__device__ __forceinline__ uint64_t policy_keep(const FusedParams& p) {
  return p.l2_hints ? l2_policy_evict_last() : l2_policy_evict_normal();
}
__device__ __forceinline__ uint64_t policy_stream(const FusedParams& p) {
  return p.l2_hints ? l2_policy_evict_first() : l2_policy_evict_normal();
}

__device__ __forceinline__ uint32_t bar_addr(uint32_t sbase, uint32_t i) { return sbase + kBarBase + 8u * i; }

// Key tiles of consumer pair k (query tiles 2k and 2k+1; the second may be past
// the last one).  Both CTAs load and process all of them.
__device__ __forceinline__ int pair_tiles(const Job& J, int k) {
  int n = consumer_tiles(J, 2 * k);
  if (2 * k + 1 < J.n_cons) n = max(n, consumer_tiles(J, 2 * k + 1));
  return n;
}
// Consumer CTAs that load tile t (each adds 2 to the slot's consumed count).
__device__ __forceinline__ int consumers_needing_tile(const Job& J, int t) {
  int n = 0;
  for (int k = 0; 2 * k < J.n_cons; ++k) n += 2 * (pair_tiles(J, k) > t);
  return n;
}

// Exact scores: K-side tiles of consumer pair k that also take the K_nope
// residual (a second stage use each, right after the tile's own).
__device__ __forceinline__ int exact_tiles_produced(const FusedParams& p, const Job& J) {
  return J.n_exact_pairs > 0 ? min(J.n_exact_tiles, p.ring_depth) : 0;
}
__device__ __forceinline__ int exact_tiles(const FusedParams& p, const Job& J, int k, int n_tiles) {
  return k < J.n_exact_pairs ? min(exact_tiles_produced(p, J), n_tiles) : 0;
}
__device__ __forceinline__ int use_tile(int u, int ex) { return u < 2 * ex ? (u >> 1) : u - ex; }
__device__ __forceinline__ bool use_is_residual(int u, int ex) { return u < 2 * ex && (u & 1); }
__device__ __forceinline__ bool last_use_of_tile(int u, int ex) { return u >= 2 * ex || (u & 1); }

// =============================================================== consumer pair
// Warps: 0-7 softmax (warpgroup w owns key columns 64w..64w+63 of every row of
// this CTA's S; warpgroup 0 first loads and rotates Q into shared memory),
// 8 K loader, 10 V loader (each also releases ring slots once their stage is
// consumed), 9 MMA issuer (leader only).
template <bool kCompute, bool kExact>
__device__ void run_consumer(const FusedParams& p, const Job& J, int job, int k, int role, uint32_t sbase,
                             uint8_t* sgen, uint32_t tmem, volatile Ctl* ctl, uint32_t rank) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ci = 2 * k + (int)rank;
  const int q0 = ci * 128;
  const int nq = max(0, min(128, J.q_count - q0));
  const int grow0 = J.q_begin + q0;
  const int n_tiles = pair_tiles(J, k);
  const int H = p.num_heads;
  const bool leader = rank == 0;

  if constexpr (!kCompute) {
    if (warp == 8 || warp == 10) {
      // ---------------------------------------------------------- TMA loads of this CTA's half
      if (lane != 0) return;
      const bool is_k = warp == 8;
      if (!is_k) {
        // this CTA's 128 query rows of the head, rotated in place by warps 0-3
        const uint32_t qb = bar_addr(sbase, kBQLand);
        mbar_arrive_expect_tx(qb, 3 * kAtomQ);
        for (int part = 0; part < 3; ++part)
          tma_load_3d_hint(sbase + kQBase + part * kAtomQ, &p.tm_q, 64 * part, J.head, grow0, qb, policy_stream(p));
      }
      // an exact pair keeps its rotated q_rope residual in V stage 3, so its V side runs 3 stages
      const int ns = is_k ? kKStages : (kExact && exact_tiles(p, J, k, n_tiles) > 0 ? kVStages - 1 : kVStages);
      const uint32_t full0 = is_k ? kBKFull : kBVFull, empty0 = is_k ? kBKEmpty : kBVEmpty;
      const uint64_t pol_ring = policy_keep(p);
      TraceAcc tr;
      // A tile's ring slot is released once the pair's MMAs have read its
      // stage, before the next tile is waited for, in batches behind one fence
      // when the ring is deep enough; produced tiles are polled a window at a
      // time.  Per-tile flag round trips would otherwise pace the loads.
      const int batch = p.ring_depth >= ns + 4 ? 4 : 1;
      // Stage uses: one per tile, and on the K side a second one for the
      // K_nope residual of the first `ex` tiles when this pair takes exact scores.
      const int ex = kExact && is_k ? exact_tiles(p, J, k, n_tiles) : 0;
      const int n_uses = n_tiles + ex;
      int rel0 = 0;             // tiles below are released
      int done_to = 0;          // tiles below are read completely (every stage use consumed)
      int ready_to = 0;         // tiles below are known to be produced
      for (int u = 0; u < n_uses; ++u) {
        const int s = u % ns;
        const int j = use_tile(u, ex);
        if (u >= ns) {
          // the stage is free once the pair's MMAs read it
          if (!wait_bar(p, bar_addr(sbase, empty0 + s), ((u / ns) - 1) & 1)) { ctl->abort = 1; return; }
          if (last_use_of_tile(u - ns, ex)) {
            done_to = use_tile(u - ns, ex) + 1;
            if (done_to - rel0 == batch) {
              release_tiles(p, job, rel0, done_to - rel0);
              rel0 = done_to;
            }
          }
        }
        const bool res = use_is_residual(u, ex);
        if (!res && j >= ready_to) {
          const uint64_t w0 = tr.begin(p);
          ready_to = wait_ready_window(p, job, j, min(n_tiles, j + min(8, p.ring_depth)));
          tr.end(p, w0);
          if (ready_to < 0) { ctl->abort = 1; return; }
          fence_proxy_async_global();   // the acquired tiles, to the TMA reads below
        }
        const uint32_t full = bar_addr(sbase, full0 + s);
        const uint32_t full_leader = mapa_shared(full, 0u);
        const int zb = ring_block(p, job, ring_slot(p, j));   // first ring block of the tile
        if (is_k && res) {
          const uint32_t st = sbase + kKBase + s * kKStageBytes;
          if (leader) mbar_arrive_expect_tx(full, 2 * 2 * kAtom64);
          tma_load_3d_pair_hint(st, &p.tm_ring64, 0, 64 * (int)rank, residual_block(p, job, ring_slot(p, j)),
                                full_leader, pol_ring);                                              // K_nope residual
        } else if (is_k) {
          const uint32_t st = sbase + kKBase + s * kKStageBytes;
          if (leader) mbar_arrive_expect_tx(full, 2 * kKStageBytes);     // both halves land on the leader's count
          const int kt0 = J.t0 + 128 * j;
          tma_load_3d_pair_hint(st, &p.tm_ring64, 0, 64 * (int)rank, zb, full_leader, pol_ring);       // K_nope lo | hi
          tma_load_2d_pair(st + 2 * kAtom64, &p.tm_kr, p.krope_col, block_row(J, (kt0 >> 6) + (int)rank), full_leader);
          trace_stage(p, role, j, 0);
        } else {
          const uint32_t st = sbase + kVBase + s * kVStageBytes;
          if (leader) mbar_arrive_expect_tx(full, 2 * kVStageBytes);
          tma_load_3d_pair_hint(st, &p.tm_ring1, 0, 0, zb + 2 + (int)rank, full_leader, pol_ring);     // V columns
          trace_stage(p, role, j, 1);
        }
      }
      // the last stages: wait for their MMAs (this also takes the leader's last
      // commits into this CTA's barriers before they are reset), release the slots
      for (int u = max(0, n_uses - ns); u < n_uses; ++u) {
        if (!wait_bar(p, bar_addr(sbase, empty0 + u % ns), (u / ns) & 1)) { ctl->abort = 1; return; }
        if (last_use_of_tile(u, ex)) done_to = use_tile(u, ex) + 1;
      }
      if (done_to > rel0) release_tiles(p, job, rel0, done_to - rel0);
      if (is_k) {
        trace_put(p, role, 3, tr.t);
        trace_put(p, role, 7, (unsigned long long)n_tiles);
      }
    } else if ((warp == 9 || warp == 11) && leader) {
      // ---------------------------------------------------------- MMA issue (leader)
      // Two issuing threads, so neither kind of MMA waits behind the other in
      // a blocked issue: warp 9 issues S(j) once K stage j has landed and its
      // score buffer is free (PV(j-3) complete: the threads' MMAs are not
      // ordered with each other), warp 11 issues PV(j) once P(j) of both CTAs
      // and V stage j are there.
      if (lane != 0) return;
      const bool s_side = warp == 9;
      if (!wait_bar(p, bar_addr(sbase, kBQReady), 0)) { ctl->abort = 1; return; }
      tc_fence_after();
      const uint64_t t_start = p.trace ? global_timer_ns() : 0;
      const int ex = kExact ? exact_tiles(p, J, k, n_tiles) : 0;
      const int nv = ex > 0 ? kVStages - 1 : kVStages;
      for (int j = 0; j < n_tiles; ++j) {
        const int b = j % kSBufs;
        if (s_side) {
          const int g = j + min(j, ex);   // stage use of the tile (its residual, when exact, is the next one)
          const int sk = g % kKStages;
          if (!wait_bar(p, bar_addr(sbase, kBKFull + sk), (g / kKStages) & 1)) { ctl->abort = 1; return; }
          if (j >= kSBufs && !wait_bar(p, bar_addr(sbase, kBPvDone + b), ((j / kSBufs) - 1) & 1)) {
            ctl->abort = 1;
            return;
          }
          const bool res = kExact && j < ex;
          const int sr = (g + 1) % kKStages;
          if (res && !wait_bar(p, bar_addr(sbase, kBKFull + sr), ((g + 1) / kKStages) & 1)) { ctl->abort = 1; return; }
          trace_stage(p, role, j, 2);
          tc_fence_after();
          const uint32_t kst = sbase + kKBase + sk * kKStageBytes;
          const uint32_t d = tmem + kTmS + 128 * b;
#pragma unroll
          for (int kk = 0; kk < 12; ++kk)
            mma2_ss(d, sdesc_sw128(sbase + kQBase + (kk >> 2) * kAtomQ + (kk & 3) * 32, 16, 1024),
                    sdesc_sw128(kst + (kk >> 2) * kAtom64 + (kk & 3) * 32, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
          if (res) {
            // exact scores, added to the same accumulator: q_nope . (K_nope - bf16(K_nope))
            // and (rotated q_rope - its bf16) . k_rope
            const uint32_t krs = sbase + kKBase + sr * kKStageBytes;
#pragma unroll 1
            for (int kk = 0; kk < 8; ++kk)
              mma2_ss(d, sdesc_sw128(sbase + kQBase + (kk >> 2) * kAtomQ + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(krs + (kk >> 2) * kAtom64 + (kk & 3) * 32, 16, 1024), kIdescS, 1u);
#pragma unroll 1
            for (int kk = 0; kk < 4; ++kk)
              mma2_ss(d, sdesc_sw128(sbase + kQResBase + kk * 32, 16, 1024),
                      sdesc_sw128(kst + 2 * kAtom64 + kk * 32, 16, 1024), kIdescS, 1u);
          }
          mma2_commit_both(bar_addr(sbase, kBSFull + b));
          mma2_commit_both(bar_addr(sbase, kBKEmpty + sk));
          if (res) mma2_commit_both(bar_addr(sbase, kBKEmpty + sr));
          trace_stage(p, role, j, 3);
        } else {
          const int sv = j % nv;
          const uint32_t vpar = (j / nv) & 1;
          if (!wait_bar(p, bar_addr(sbase, kBPFull + b), (j / kSBufs) & 1)) { ctl->abort = 1; return; }
          trace_stage(p, role, j, 4);
          if (!wait_bar(p, bar_addr(sbase, kBVFull + sv), vpar)) { ctl->abort = 1; return; }
          trace_stage(p, role, j, 5);
          tc_fence_after();
          const uint32_t v = sbase + kVBase + sv * kVStageBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma2_ts(tmem + kTmO, tmem + kTmS + 128 * b + kk * 8, sdesc_sw128(v + kk * 2048, kAtomQ, 1024), kIdescPV,
                    (j > 0 || kk > 0) ? 1u : 0u);
          mma2_commit_both(bar_addr(sbase, kBPvDone + b));
          mma2_commit_both(bar_addr(sbase, kBVEmpty + sv));
        }
      }
      if (s_side) trace_put(p, role, 4, p.trace ? global_timer_ns() - t_start : 0);
    }
  } else {
    if (warp < 4) {
      // ---------------------------------------------------------- Q: RoPE of the landed rows (warpgroup 0)
      // q_nope and q_rope arrive by TMA (rows past the piece's queries are
      // other rows or zeros, and their results are not written); q_rope is
      // rotated by q_pos - offset in place while the angles are computed
      // during the load.
      const int r = tid & 127;
      const int64_t delta = r < nq ? (int64_t)__ldg(p.q_pos + grow0 + r) - J.rope_offset : 0;
      if (tid == 0) trace_stage(p, role, kTraceOnce, 0);
      float sn[32], cs[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) rope_sincos_sfu(delta, p.rope_frac[i], &sn[i], &cs[i]);
      const bool landed = wait_bar_warp(p, bar_addr(sbase, kBQLand), 0);
      if (tid == 0) trace_stage(p, role, kTraceOnce, 1);
      if (landed && !(kExact && exact_tiles(p, J, k, n_tiles) > 0)) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t addr = sbase + kQBase + 2 * kAtomQ + sw128_off(r, c);
          uint32_t w4[4];
          lds128(addr, w4);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float x0 = __uint_as_float(w4[i] << 16), x1 = __uint_as_float(w4[i] & 0xFFFF0000u);
            w4[i] = pack_bf16(x0 * cs[4 * c + i] - x1 * sn[4 * c + i], x0 * sn[4 * c + i] + x1 * cs[4 * c + i]);
          }
          sts128(addr, w4[0], w4[1], w4[2], w4[3]);
        }
      } else if (landed) {
        // exact scores: the rotation's bf16 residual too, in the layout of a Q block
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t addr = sbase + kQBase + 2 * kAtomQ + sw128_off(r, c);
          uint32_t w4[4], x4[4];
          lds128(addr, w4);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float x0 = __uint_as_float(w4[i] << 16), x1 = __uint_as_float(w4[i] & 0xFFFF0000u);
            const float y0 = x0 * cs[4 * c + i] - x1 * sn[4 * c + i], y1 = x0 * sn[4 * c + i] + x1 * cs[4 * c + i];
            w4[i] = pack_bf16(y0, y1);
            x4[i] = pack_bf16(y0 - __uint_as_float(w4[i] << 16), y1 - __uint_as_float(w4[i] & 0xFFFF0000u));
          }
          sts128(addr, w4[0], w4[1], w4[2], w4[3]);
          sts128(sbase + kQResBase + sw128_off(r, c), x4[0], x4[1], x4[2], x4[3]);
        }
      }
      fence_proxy_async_smem();   // visible to the tensor core before the leader issues S
      __syncwarp();
      if (tid == 0) trace_stage(p, role, kTraceOnce, 2);
      if (lane == 0) mbar_arrive_cluster(mapa_shared(bar_addr(sbase, kBQReady), 0u));   // one arrival per warp
    }
    // ------------------------------------------------------------ softmax / epilogue (warps 0..7)
    const int w = warp >> 2;           // key half
    const int r = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float* xchg = reinterpret_cast<float*>(sgen + kXchgBase);   // [2 slots][2 halves][128] maxima, then sums
    const int qtok = query_token(J, q0 + r);
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l_part = 0.f;
    bool ok = true;
    TraceAcc tr_s;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j % kSBufs, x = j & 1;
      const uint64_t w0 = tr_s.begin(p);
      if (ok && !wait_bar_warp(p, bar_addr(sbase, kBSFull + b), (j / kSBufs) & 1)) ok = false;
      tr_s.end(p, w0);
      if (tid == 0) trace_stage(p, role, j, 6);
      tc_fence_after();
      const uint32_t scol = tmem + lane_off + kTmS + 128 * b + 64 * w;
      uint32_t v[64];
      float mx = -INFINITY;
      if (ok) mx = tmem_ld64_max(scol, v);   // the half-row maximum comes with the load
      const int kt0 = J.t0 + 128 * j + 64 * w;
      const bool full = kt0 >= J.k_begin && kt0 + 63 < J.k_end && kt0 + 63 <= qtok;
      if (!full) {
        // visible columns form one range [lo, lo + span] of the half tile
        const int lo = max(J.k_begin - kt0, 0);
        const int span = min(J.k_end - 1, qtok) - kt0 - lo;   // negative: none
        float m8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const bool okc = span >= 0 && (uint32_t)(c - lo) <= (uint32_t)span;
          const float xv = okc ? __uint_as_float(v[c]) : -INFINITY;
          v[c] = __float_as_uint(xv);
          m8[c & 7] = fmaxf(m8[c & 7], xv);
        }
        mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      }
      // row maximum over both key halves; the barrier also orders both
      // warpgroups' S loads before either overwrites S with P
      xchg[(x * 2 + w) * 128 + r] = mx;
      tc_fence_before();
      named_bar_sync(1, 256);
      tc_fence_after();
      mx = fmaxf(mx, xchg[(x * 2 + (1 - w)) * 128 + r]);
      const float m_tile = mx * sl2;
      float alpha = 1.f;
      const bool rescale = m_tile > m_used + kRescaleThreshold;
      if (rescale) {
        alpha = ex2(m_used - m_tile);   // 0 when m_used = -inf
        m_used = m_tile;
      }
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      // P packed in place over the scores and stored in two 16-column halves
      const uint64_t sc2 = f2pack(sl2, sl2), nm2 = f2pack(-mref, -mref);
      uint64_t s4[4] = {0ull, 0ull, 0ull, 0ull};
      const uint32_t pcol = tmem + lane_off + kTmS + 128 * b + 32 * w;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float x0, x1;
        f2unpack(ffma2(f2pack(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1])), sc2, nm2), x0, x1);
        const float a = ex2(x0), bb = ex2(x1);
        s4[c & 3] = fadd2(s4[c & 3], f2pack(a, bb));
        v[c] = pack_bf16(a, bb);
        if (c == 15 && ok) tmem_st16(pcol, v);
      }
      if (ok) tmem_st16(pcol + 16, v + 16);
      float s8[4];
      f2unpack(fadd2(s4[0], s4[1]), s8[0], s8[1]);
      f2unpack(fadd2(s4[2], s4[3]), s8[2], s8[3]);
      l_part = l_part * alpha + ((s8[0] + s8[2]) + (s8[1] + s8[3]));
      if (j >= 1 && ok && __any_sync(0xffffffffu, rescale)) {
        // O holds PV of tiles < j: PV(j-1) must be done before O is rescaled.
        // PV(j-4) finished before S(j) did, so the barrier is at most one phase behind.
        if (!wait_bar_warp(p, bar_addr(sbase, kBPvDone + (j - 1) % kSBufs), ((j - 1) / kSBufs) & 1)) ok = false;
        tc_fence_after();
        if (ok) {
          const uint32_t ocol = tmem + lane_off + kTmO + 64 * w;
#pragma unroll 1
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t o[32];
            tmem_ld32(ocol + cc * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(ocol + cc * 32, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(bar_addr(sbase, kBPFull + b), 0u));   // leader issues PV
      if (tid == 0) trace_stage(p, role, j, 7);
    }
    // every PV done: O is final, and the leader's last commits reached this CTA's barriers
    if (ok && n_tiles > 0 &&
        !wait_bar_warp(p, bar_addr(sbase, kBPvDone + (n_tiles - 1) % kSBufs), ((n_tiles - 1) / kSBufs) & 1))
      ok = false;
    if (tid == 0) trace_put(p, role, 6, tr_s.t);
    if (tid == 0) trace_stage(p, role, kTraceOnce, 3);
    xchg[(4 + w) * 128 + r] = l_part;
    named_bar_sync(1, 256);
    const float l_run = l_part + xchg[(4 + (1 - w)) * 128 + r];
    if (!ok) { ctl->abort = 1; return; }
    if (tid == 0) trace_stage(p, role, kTraceOnce, 5);
    tc_fence_after();
    // ---- epilogue: this warpgroup writes output columns 64w .. 64w+63 of this CTA's rows
    const bool empty = n_tiles == 0 || !(l_run > 0.f);
    const float inv_l = empty ? 0.f : 1.f / l_run;
    const bool live = r < nq;
    const int grow = grow0 + r;
    const int64_t orow = J.slot < 0 ? (int64_t)grow : (int64_t)J.slot * p.slot_stride_rows + grow;
    const uint32_t ocol = tmem + lane_off + kTmO + 64 * w;
    if (nq == 128 && n_tiles > 0) {
      // A whole tile: the warpgroup stages its 64 columns in the idle K stages
      // (128-byte swizzled boxes) and one thread stores them by TMA, instead
      // of 32 scattered 16-byte pieces per warp store.
      const bool ob = J.slot < 0 && p.out_bf16;
      const uint32_t stg = sbase + kKBase + (uint32_t)w * 2 * kAtomQ;
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t o[32];
        tmem_ld32(ocol + cc * 32, o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(empty ? 0.f : __uint_as_float(o[i]) * inv_l);
        if (ob) {
#pragma unroll
          for (int g = 0; g < 4; ++g)
            sts128(stg + sw128_off(r, 4 * cc + g), pack_bf16(__uint_as_float(o[8 * g]), __uint_as_float(o[8 * g + 1])),
                   pack_bf16(__uint_as_float(o[8 * g + 2]), __uint_as_float(o[8 * g + 3])),
                   pack_bf16(__uint_as_float(o[8 * g + 4]), __uint_as_float(o[8 * g + 5])),
                   pack_bf16(__uint_as_float(o[8 * g + 6]), __uint_as_float(o[8 * g + 7])));
        } else {
#pragma unroll
          for (int g = 0; g < 8; ++g)
            sts128(stg + cc * kAtomQ + sw128_off(r, g), o[4 * g], o[4 * g + 1], o[4 * g + 2], o[4 * g + 3]);
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(2 + w, 128);
      if (r == 0) {
        const int row0 = J.slot < 0 ? grow0 : J.slot * p.slot_stride_rows + grow0;
        const uint64_t pol = policy_stream(p);
        if (ob) {
          tma_store_3d_hint(&p.tm_out, stg, 64 * w, J.head, row0, pol);
        } else {
          const CUtensorMap* m = J.slot < 0 ? &p.tm_out : &p.tm_part;
          tma_store_3d_hint(m, stg, 64 * w, J.head, row0, pol);
          tma_store_3d_hint(m, stg + kAtomQ, 64 * w + 32, J.head, row0, pol);
        }
        bulk_commit();
        bulk_wait_read0();   // the stages are free again before the role ends
      }
    } else {
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t o[32];
        if (n_tiles > 0) tmem_ld32(ocol + cc * 32, o);
        if (!live) continue;
        const int col0 = 64 * w + 32 * cc;
        if (J.slot < 0 && p.out_bf16) {
          uint16_t* dst = static_cast<uint16_t*>(p.out) + (orow * H + J.head) * kDv + col0;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 q;
            q.x = pack_bf16(empty ? 0.f : __uint_as_float(o[i + 0]) * inv_l, empty ? 0.f : __uint_as_float(o[i + 1]) * inv_l);
            q.y = pack_bf16(empty ? 0.f : __uint_as_float(o[i + 2]) * inv_l, empty ? 0.f : __uint_as_float(o[i + 3]) * inv_l);
            q.z = pack_bf16(empty ? 0.f : __uint_as_float(o[i + 4]) * inv_l, empty ? 0.f : __uint_as_float(o[i + 5]) * inv_l);
            q.w = pack_bf16(empty ? 0.f : __uint_as_float(o[i + 6]) * inv_l, empty ? 0.f : __uint_as_float(o[i + 7]) * inv_l);
            *reinterpret_cast<uint4*>(dst + i) = q;
          }
        } else {
          float* dst = (J.slot < 0 ? static_cast<float*>(p.out) : p.part_out) + (orow * H + J.head) * kDv + col0;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            float4 q;
            q.x = empty ? 0.f : __uint_as_float(o[i + 0]) * inv_l;
            q.y = empty ? 0.f : __uint_as_float(o[i + 1]) * inv_l;
            q.z = empty ? 0.f : __uint_as_float(o[i + 2]) * inv_l;
            q.w = empty ? 0.f : __uint_as_float(o[i + 3]) * inv_l;
            *reinterpret_cast<float4*>(dst + i) = q;
          }
        }
      }
    }
    if (live && w == 0) {
      const float lse = empty ? -INFINITY : m_used * 0.69314718055994531f + logf(l_run);
      (J.slot < 0 ? p.lse : p.part_lse)[orow * H + J.head] = lse;
    }
    if (tid == 0) trace_stage(p, role, kTraceOnce, 4);
  }
}

// Two ring blocks [128 tokens x 64 columns] from a thread's 128 packed bf16
// values of its row (pk[0..31]: block 0, pk[32..63]: block 1): after an 8x8
// transpose of 16-byte chunks across lanes, each warp store covers four whole
// 128-byte rows.
__device__ __forceinline__ void store_ring_blocks(uint16_t* dst, const uint32_t (&pk)[64], int lane, int st_row,
                                                  int st_chunk, uint64_t pol) {
#pragma unroll
  for (int hb = 0; hb < 2; ++hb) {
    uint4 c[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      c[e] = make_uint4(pk[32 * hb + 4 * e], pk[32 * hb + 4 * e + 1], pk[32 * hb + 4 * e + 2], pk[32 * hb + 4 * e + 3]);
    transpose8x16B(c, lane);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      st_global_v4_hint(dst + (size_t)hb * (128 * 64) + (size_t)(st_row + e) * 64 + st_chunk * 8, c[e], pol);
  }
}

// The K_nope residual K - bf16(K) of a thread's row (128 accumulator columns
// at `acc`, scaled by oscale), rounded to bf16 and stored as two ring blocks,
// one 64-column block at a time (32 words live, so the rare tiles that take
// it cost the common path no registers).
__device__ __forceinline__ void store_residual(uint32_t acc, float oscale, bool valid, uint16_t* dst, int lane,
                                              int st_row, int st_chunk, uint64_t pol) {
#pragma unroll 1
  for (int hb = 0; hb < 2; ++hb) {
    uint32_t w[32];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t a[32];
      tmem_ld32(acc + (2 * hb + cc) * 32, a);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float x0 = __uint_as_float(a[2 * i]) * oscale, x1 = __uint_as_float(a[2 * i + 1]) * oscale;
        const uint32_t h = pack_bf16(x0, x1);
        w[16 * cc + i] = valid ? pack_bf16(x0 - __uint_as_float(h << 16), x1 - __uint_as_float(h & 0xFFFF0000u)) : 0u;
      }
    }
    uint4 c[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) c[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
    transpose8x16B(c, lane);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      st_global_v4_hint(dst + (size_t)hb * (128 * 64) + (size_t)(st_row + e) * 64 + st_chunk * 8, c[e], pol);
  }
}

// =============================================================== producer pair
// Passes pi, pi + n_prod, ... of 256 tokens; CTA r up-projects tokens
// 128r..128r+127 of a pass (ring tile 2 pass + r).  Warps: 10 loads this CTA's
// half of the head's kv_b_proj columns once for the role, 8 streams its latent
// rows through the stages (waiting for each to be free), 9 MMA (leader), 0-7
// conversion: warpgroup 0 the K_nope columns, warpgroup 1 the V columns of the
// CTA's tile, stored from registers into the ring.
template <bool kCompute, bool kExact, bool kFp8W>
__device__ void run_producer(const FusedParams& p, const Job& J, int job, int pi, int role, uint32_t sbase,
                             uint32_t tmem, volatile Ctl* ctl, uint32_t rank) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_pass = (J.n_tiles + 1) >> 1;
  const int H = p.num_heads;
  const int h = J.head;
  const bool leader = rank == 0;
  int my_passes = 0;
  for (int pp = pi; pp < n_pass; pp += J.n_prod) ++my_passes;
  if (my_passes == 0) return;
  constexpr int kSlices = kFp8W ? kDc / 128 : kDc / 64;   // k-slices (stages) of a pass

  if constexpr (!kCompute) {
    if (warp == 10) {
      // the head's K_nope (CTA 0) or V (CTA 1) columns, once for every pass of the role
      if (lane != 0) return;
      const uint32_t full = bar_addr(sbase, kBWFull);
      const uint32_t full_leader = mapa_shared(full, 0u);
      const uint64_t pol = policy_stream(p);
      if constexpr (kFp8W) {
        // E4M3 columns, K-major (the transposed copy [H*256][512]): 4 k-slices of [128 columns x 128 B]
        if (leader) mbar_arrive_expect_tx(full, 2 * 4 * kAtomQ);
        const int wrow = rank == 0 ? h * kDnope : H * kDnope + h * kDv;
        for (int kx = 0; kx < kDc / 128; ++kx)
          tma_load_2d_pair_hint(sbase + kPWBase + kx * kAtomQ, &p.tm_w8, 128 * kx, wrow, full_leader, pol);
      } else {
        if (leader) mbar_arrive_expect_tx(full, 2 * 8 * kAtomQ);
        const int blk = rank == 0 ? 2 * h : (H * kDnope + h * kDv) / 64;
        for (int kx = 0; kx < kDc / 64; ++kx)
          tma_load_3d_pair_hint(sbase + kPWBase + kx * kAtomQ, &p.tm_w, 0, 64 * kx, blk, full_leader, pol);
      }
      trace_stage(p, role, 0, 7);
      // This CTA writes tile t = 2 pass + rank of each pass into ring slot
      // t mod depth of lane job mod ring_lanes.  On the first lap the lane's
      // previous job, job - ring_lanes, must be done with that slot: its last
      // tile there published and read by every consumer that needs it.  Its
      // roles precede this one in the queue (ring_lanes > prod_ahead) and never
      // wait on it, so the wait ends.  This thread checks pass by pass and
      // releases lane_ok to the row loader, which loads a pass's rows only
      // after its check; the pass's stores follow through the loads, the MMAs
      // and their barriers.  The checks stay off the loads' and MMAs' path.
      const int prev = job - p.ring_lanes;
      if (prev < 0) return;
      const Job Jp = make_job(p, prev / p.num_heads, prev % p.num_heads);
      int* ok = const_cast<int*>(&ctl->lane_ok);
      TraceAcc tr_lane;
      for (int n = 0; n < my_passes; ++n) {
        const int t = 2 * (pi + n * J.n_prod) + (int)rank;
        if (t < J.n_tiles && t < p.ring_depth && t < Jp.n_tiles) {
          const int tl = t + ((Jp.n_tiles - 1 - t) / p.ring_depth) * p.ring_depth;   // its last tile in slot t
          const uint64_t w0 = tr_lane.begin(p);
          if (!(wait_flag_geq(p, ready_flag(p, prev, t), (uint32_t)tl + 1) &&
                wait_flag_geq(p, consumed_flag(p, prev, t), 2u * (uint32_t)consumers_needing_tile(Jp, tl)))) {
            ctl->abort = 1;
            return;
          }
          tr_lane.end(p, w0);
        }
        st_release_cta_s32(ok, n + 1);
      }
      trace_put(p, role, 6, tr_lane.t);
    } else if (warp == 8) {
      if (lane != 0) return;
      const bool lane_wait = job >= p.ring_lanes;
      int g = 0;
      for (int n = 0; n < my_passes; ++n) {
        const int pass = pi + n * J.n_prod;
        const int row0 = block_row(J, (J.t0 >> 6) + 4 * pass) + 128 * (int)rank;
        // the ring slot of this pass's tile is free (checked by warp 10)
        if (lane_wait && !wait_shared_geq(p, ctl, const_cast<const int*>(&ctl->lane_ok), n + 1)) {
          ctl->abort = 1;
          return;
        }
        // a stage is one k-slice of the pass's rows: 64 bf16 values, or 128 E4M3 codes, of 128 tokens
        for (int kx = 0; kx < kSlices; ++kx, ++g) {
          const int s = g % kPStages;
          if (g >= kPStages && !wait_bar(p, bar_addr(sbase, kBProdEmpty + s), ((g / kPStages) - 1) & 1)) {
            ctl->abort = 1;
            return;
          }
          const uint32_t full = bar_addr(sbase, kBProdFull + s);
          if (leader) mbar_arrive_expect_tx(full, 2 * kPStageBytes);     // both CTAs' rows
          if constexpr (kFp8W)
            tma_load_2d_pair(sbase + kPCBase + s * kPStageBytes, &p.tm_c8, 128 * kx, row0, mapa_shared(full, 0u));
          else
            tma_load_2d_pair(sbase + kPCBase + s * kPStageBytes, &p.tm_kr128, 64 * kx, row0, mapa_shared(full, 0u));
          if (kx == 0) trace_stage(p, role, n, 6);
        }
      }
      // the stages' last MMAs: take the leader's commits before the barriers are reset
      for (int gx = max(0, g - kPStages); gx < g; ++gx)
        if (!wait_bar(p, bar_addr(sbase, kBProdEmpty + gx % kPStages), (gx / kPStages) & 1)) {
          ctl->abort = 1;
          return;
        }
    } else if (warp == 9 && leader) {
      if (lane != 0) return;
      TraceAcc tr_op, tr_acc;
      if (!wait_bar(p, bar_addr(sbase, kBWFull), 0)) { ctl->abort = 1; return; }
      int g = 0;
      for (int n = 0; n < my_passes; ++n) {
        const int b = n & 1;
        const uint64_t wa = tr_acc.begin(p);
        if (n >= 2 && !wait_bar(p, bar_addr(sbase, kBAccEmpty + b), ((n >> 1) - 1) & 1)) { ctl->abort = 1; return; }
        tr_acc.end(p, wa);
        trace_stage(p, role, n, 0);
        tc_fence_after();
        for (int kx = 0; kx < kSlices; ++kx, ++g) {
          const int s = g % kPStages;
          const uint64_t w0 = tr_op.begin(p);
          if (!wait_bar(p, bar_addr(sbase, kBProdFull + s), (g / kPStages) & 1)) { ctl->abort = 1; return; }
          tr_op.end(p, w0);
          tc_fence_after();
          const uint32_t st = sbase + kPCBase + s * kPStageBytes;
          const uint32_t wst = sbase + kPWBase + kx * kAtomQ;
          if constexpr (kFp8W) {
            // K = 32 E4M3 values (32 bytes) per MMA, both operands K-major
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma2_ss_e4m3(tmem + kTmAcc + 256 * b, sdesc_sw128(st + kk * 32, 16, 1024),
                           sdesc_sw128(wst + kk * 32, 16, 1024), kIdescUp8, (kx | kk) ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma2_ss(tmem + kTmAcc + 256 * b, sdesc_sw128(st + kk * 32, 16, 1024),
                      sdesc_sw128(wst + kk * 2048, kAtom64, 1024), kIdescUp, (kx | kk) ? 1u : 0u);
          }
          mma2_commit_both(bar_addr(sbase, kBProdEmpty + s));
        }
        mma2_commit_both(bar_addr(sbase, kBAccFull + b));
        trace_stage(p, role, n, 1);
      }
      trace_put(p, role, 4, tr_op.t);
      trace_put(p, role, 5, tr_acc.t);
      trace_put(p, role, 7, (unsigned long long)my_passes);
    }
  } else {
    // conversion: warpgroup wg converts accumulator columns 128 wg .. 128 wg + 127
    // (wg 0: K_nope, wg 1: V) of this CTA's 128 tokens into ring blocks 2 wg, 2 wg + 1
    const int wg = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float oscale = p.out_scale;
    // after the transpose lane l holds 16-byte chunk l % 8 of rows 8 (l / 8) + e of the warp's 32
    const int st_row = (warp & 3) * 32 + 8 * (lane >> 3), st_chunk = lane & 7;
    TraceAcc tr_c;
    // A pass's tile is stored straight from registers and published at the
    // next pass's barrier (which orders every thread's stores before the
    // release), so neither the stores' completion nor the release fence
    // delays the next accumulator.
    bool pend = false;        // the previous pass stored a tile not yet published
    int pend_t = 0, pend_slot = 0;
    const uint64_t pol_ring = policy_keep(p);
    for (int n = 0; n < my_passes; ++n) {
      const int pass = pi + n * J.n_prod;
      const int b = n & 1;
      const int t = 2 * pass + (int)rank;
      const bool live_tile = t < J.n_tiles;
      const int slot = ring_slot(p, t);
      const int tok = J.t0 + 128 * t + r;
      const bool valid = tok >= J.k_begin && tok < J.k_end;
      if (!wait_bar_warp(p, bar_addr(sbase, kBAccFull + b), (n >> 1) & 1)) ctl->abort = 1;
      if (tid == 0) trace_stage(p, role, n, 2);
      tc_fence_after();
      const uint32_t acc = tmem + lane_off + kTmAcc + 256 * b + 128 * wg;
      if (kExact && wg == 0 && live_tile && t < exact_tiles_produced(p, J) && !ctl->abort) {
        // a tile that a query row with few keys sees: its K_nope residual too,
        // stored first, before this thread holds the tile's bf16 values.  Such
        // tiles are on the lane's first lap (t < ring_depth), whose slot the
        // lane check cleared before this pass's MMAs began.
        store_residual(acc, oscale, valid, p.ring + (size_t)residual_block(p, job, slot) * (128 * 64), lane, st_row,
                       st_chunk, pol_ring);
      }
      uint32_t pk[64];
      if (live_tile && !ctl->abort) {
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t a[32];
          tmem_ld32(acc + cc * 32, a);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[16 * cc + i] = valid ? pack_bf16(__uint_as_float(a[2 * i]) * oscale, __uint_as_float(a[2 * i + 1]) * oscale) : 0u;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(mapa_shared(bar_addr(sbase, kBAccEmpty + b), 0u));   // accumulator free
      // every thread's stores of the previous tile are behind this barrier;
      // the stop decision is taken here for both warpgroups
      if (named_bar_or(1, 256, ctl->abort != 0)) return;
      // publish the previous tile before waiting for this tile's slot: a
      // consumer may need it to get to the release that frees the slot
      if (pend && tid == 0) {
        trace_stage(p, role, n, 4);
        st_release_gpu(ready_flag(p, job, pend_slot), (uint32_t)pend_t + 1);
        trace_stage(p, role, n, 5);
      }
      if (live_tile && t >= p.ring_depth) {
        // the slot's previous occupant (tile t - ring) must be published and
        // fully consumed before anyone writes it
        if (tid == 0 && !ctl->abort) {
          const uint64_t w0 = tr_c.begin(p);
          if (!(wait_flag_geq(p, ready_flag(p, job, slot), (uint32_t)(t - p.ring_depth + 1)) &&
                wait_flag_geq(p, consumed_flag(p, job, slot), 2u * (uint32_t)consumers_needing_tile(J, t - p.ring_depth))))
            ctl->abort = 1;
          tr_c.end(p, w0);
        }
        if (named_bar_or(1, 256, ctl->abort != 0)) return;
      }
      if (live_tile && tid == 0) *consumed_flag(p, job, slot) = 0u;   // ordered before the release of `ready`
      if (live_tile) {
        store_ring_blocks(p.ring + ((size_t)ring_block(p, job, slot) + 2 * wg) * (128 * 64), pk, lane, st_row, st_chunk,
                          pol_ring);
        if (tid == 0) trace_stage(p, role, n, 3);
      }
      pend = live_tile;
      pend_t = t;
      pend_slot = slot;
    }
    if (pend) {
      named_bar_sync(1, 256);
      if (tid == 0) st_release_gpu(ready_flag(p, job, pend_slot), (uint32_t)pend_t + 1);
    }
    if (tid == 0) trace_put(p, role, 3, tr_c.t);
  }
}

// The role loop of the pair, instantiated for the compute warps (0-7) and the
// control warps (8-11).  Cluster rank 0 takes the next role from the queue
// and writes it into both CTAs; every exit decision is made there, so both
// CTAs run the same sequence of cluster barriers.
template <bool kCompute, bool kExact, bool kFp8W>
__device__ __forceinline__ void role_loop(const FusedParams& p, uint32_t sbase, uint8_t* sgen, volatile Ctl* ctl,
                                          uint32_t tmem, uint32_t rank) {
  const int tid = threadIdx.x;
  for (;;) {
    if (kCompute && tid == 0 && rank == 0) {
      const int g = (ctl->abort || aborted_global(p)) ? p.n_groups : (int)atomicAdd(p.queue, 1u);
      ctl->group = g;
      st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(&ctl->group)), 1u), (uint32_t)g);
    }
    tc_fence_before();
    cluster_sync_all();   // also: both CTAs are done with the previous role
    tc_fence_after();
    const int g = ctl->group;
    if (g >= p.n_groups) break;
    int lo = 0, hi = p.n_pieces - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.pieces[mid].group_begin <= g) lo = mid; else hi = mid - 1;
    }
    const Piece& P = p.pieces[lo];
    const int n_pairs = (P.n_cons + 1) >> 1;
    const int local = g - P.group_begin;
    // Roles of a piece in queue order: the producers of heads 0 .. L-1, then
    // per head h the producers of head h + L followed by the consumers of head
    // h (the longest first), L = p.prod_ahead.  A head's producers thus run L
    // heads ahead of its consumers, which find their first tiles ready, and
    // still precede them in the queue.
    const int np = P.n_prod, la = min(p.prod_ahead, p.num_heads);
    int head, idx;
    bool producer;
    if (local < np * la) {
      producer = true;
      head = local / np;
      idx = local - head * np;
    } else {
      const int l = local - np * la, seg = np + n_pairs, n_full = p.num_heads - la;
      if (l < n_full * seg) {
        const int h = l / seg, r = l - h * seg;
        producer = r < np;
        head = producer ? h + la : h;
        idx = producer ? r : n_pairs - 1 - (r - np);
      } else {
        const int l2 = l - n_full * seg;
        producer = false;
        head = n_full + l2 / n_pairs;
        idx = n_pairs - 1 - (l2 - (l2 / n_pairs) * n_pairs);
      }
    }
    const Job J = make_job(p, lo, head);
    const int job = lo * p.num_heads + J.head;
    const int slot = g * 2 + (int)rank;   // trace slot
    if (kCompute && tid >= 32 && tid < 32 + (int)kNumBars) {
      // fresh barriers for this role (every barrier is idle here), one per lane of warp 1
      const uint32_t i = (uint32_t)(tid - 32);
      mbar_inval(bar_addr(sbase, i));
      uint32_t cnt = 1;
      // barriers the leader waits on count one arrival per warp of both CTAs
      if (!producer && i == kBQReady) cnt = 2 * 4;
      if (!producer && i >= kBPFull && i < kBPFull + kSBufs) cnt = 2 * 8;
      if (producer && (i == kBAccEmpty || i == kBAccEmpty + 1)) cnt = 2 * 8;
      mbar_init(bar_addr(sbase, i), cnt);
      fence_mbar_init();
    }
    if (kCompute && tid == 0) ctl->lane_ok = 0;
    cluster_sync_all();   // the peer's barriers exist before anything reaches them
    if (kCompute && p.trace && tid == 0) {
      trace_put(p, slot, 0, global_timer_ns());
      trace_put(p, slot, 2, ((unsigned long long)blockIdx.x << 32) | ((unsigned long long)producer << 31) | (unsigned)job);
    }
    if (!ctl->abort && !(producer && job == p.withhold_job)) {
      if (producer) run_producer<kCompute, kExact, kFp8W>(p, J, job, idx, slot, sbase, tmem, ctl, rank);
      else run_consumer<kCompute, kExact>(p, J, job, idx, slot, sbase, sgen, tmem, ctl, rank);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (kCompute && p.trace && tid == 0) trace_put(p, slot, 1, global_timer_ns());
  }
}

// kExact: some job of the launch has query rows that see fewer than
// kExactKeys keys (exact scores for them); the launches without such rows run
// the instantiation that has none of that code.
// kFp8W: the up-projection takes the cache's E4M3 codes as stored and an E4M3
// copy of kv_b_proj on the FP8 tensor cores.
template <bool kExact, bool kFp8W>
__global__ void __launch_bounds__(kThreads, 1) fused2_prefill_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  volatile Ctl* ctl = reinterpret_cast<volatile Ctl*>(sgen + kBarBase + 8 * kNumBars);
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_rank();

  if (tid == 0) {
    prefetch_tensormap(&p.tm_kr);
    if (kFp8W) {
      prefetch_tensormap(&p.tm_c8);
      prefetch_tensormap(&p.tm_w8);
    } else {
      prefetch_tensormap(&p.tm_kr128);
      prefetch_tensormap(&p.tm_w);
    }
    prefetch_tensormap(&p.tm_ring);
    prefetch_tensormap(&p.tm_ring1);
    prefetch_tensormap(&p.tm_ring64);
    prefetch_tensormap(&p.tm_q);
    prefetch_tensormap(&p.tm_out);
  }
  if (tid == 32) {
    ctl->abort = 0;
    for (uint32_t i = 0; i < kNumBars; ++i) mbar_init(bar_addr(sbase, i), 1);
    fence_mbar_init();
  }
  cluster_sync_all();   // both CTAs run before the pair allocates TMEM or touches the other's memory
  if ((tid >> 5) == 0) {
    tmem_alloc2(sbase + kBarBase + 8 * kNumBars + offsetof(Ctl, tmem), 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;

  // Registers: 384 x 168 at launch; warpgroup 2 gives back 112 each (128 x 112),
  // warpgroups 0 and 1 take 56 more each (256 x 56): the same total.
  if ((tid >> 5) >= 8) {
    setmaxnreg_dec<56>();
    role_loop<false, kExact, kFp8W>(p, sbase, sgen, ctl, tmem, rank);
  } else {
    setmaxnreg_inc<224>();
    role_loop<true, kExact, kFp8W>(p, sbase, sgen, ctl, tmem, rank);
  }
  tc_fence_before();
  cluster_sync_all();   // neither CTA releases TMEM while the pair's MMAs could still use it
  if ((tid >> 5) == 0) tmem_dealloc2(tmem, 512);
}

}  // namespace

int fused2_smem_bytes() { return (int)kSmemBytes; }

static cudaError_t configure2(int dev) {
  static int configured_device = -1;
  if (configured_device == dev) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fused2_prefill_kernel<false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused2_prefill_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused2_prefill_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused2_prefill_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
  if (e == cudaSuccess) configured_device = dev;
  return e;
}

static void cluster_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int grid, cudaStream_t s) {
  *cfg = {};
  cfg->gridDim = dim3(grid);
  cfg->blockDim = dim3(kThreads);
  cfg->dynamicSmemBytes = kSmemBytes;
  cfg->stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg->attrs = attr;
  cfg->numAttrs = 1;
}

// Clusters of two CTAs, no cooperative attribute: a role only ever waits on
// roles dequeued before it, which run on resident CTAs.
cudaError_t launch_fused2(const FusedParams& p, int grid, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = configure2(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  cluster_config(&cfg, attr, grid, s);
  bool exact = false;
  for (int i = 0; i < p.n_pieces; ++i) exact |= p.pieces[i].exact != 0;
  if (p.fp8w)
    e = exact ? cudaLaunchKernelEx(&cfg, fused2_prefill_kernel<true, true>, p)
              : cudaLaunchKernelEx(&cfg, fused2_prefill_kernel<false, true>, p);
  else
    e = exact ? cudaLaunchKernelEx(&cfg, fused2_prefill_kernel<true, false>, p)
              : cudaLaunchKernelEx(&cfg, fused2_prefill_kernel<false, false>, p);
  count_launch();
  return e;
}

cudaError_t fused2_grid_size(int* grid) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = configure2(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  cluster_config(&cfg, attr, 2 * ((sms + 1) / 2), nullptr);
  int clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&clusters, fused2_prefill_kernel<false, false>, &cfg);
  if (e != cudaSuccess) return e;
  *grid = 2 * clusters;
  return *grid > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

}  // namespace mla
