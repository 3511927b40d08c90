// Persistent fused MLA prefill kernel for sm_103a.
//
// What it computes ("DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析",
// section 4.4; query relocation from "RedKnot-MLA: Multi-Head Offline-Online
// Reuse for DeepSeek-V4 Long-Context Serving", section 2): for every job (one
// request, one head, one key range with one RoPE offset) and every query of
// the request, attention over the keys of the range, where
//   K_nope | V = c_kv * kv_b_proj[:, columns of the head]   (up-projection)
//   s = scale * (q_nope . K_nope + R(q_pos - offset) q_rope . k_rope).
//
// How it is organised.  The up-projection of a key tile is shared by every
// query of the request, so it is computed once per job, not once per query
// tile.  One cooperative grid of one CTA per SM pulls *roles* from a FIFO
// queue in global memory (an atomic counter):
//   producer role  up-projects passes of 256 key tokens: TMA loads the latent
//                  rows of four cache blocks (gathered through the block
//                  table) and kv_b_proj slices, tcgen05.mma accumulates
//                  [K_nope | V] for 2 x 128 tokens in TMEM (all 512 columns),
//                  then 256 threads convert to bf16 and store the tiles into a
//                  small per-job ring in global memory (it stays in L2) and
//                  publish each tile with a release flag;
//   consumer role  owns 256 queries (two 128-row tiles) of the job: TMA loads
//                  Q once, rotates q_rope by (q_pos - offset) in shared memory,
//                  then streams 64-key stages (K_nope and V from the ring,
//                  k_rope straight from the cache) through a 3-stage ring;
//                  per stage and query tile: S = Q K^T into TMEM, one thread
//                  per row does the online softmax (base 2, lazy rescaling),
//                  writes P back into TMEM as bf16, and O += P V reads P from
//                  TMEM.  Finally out = O / l and lse = ln(sum e^s).
// A job's producer roles precede its consumer roles in the queue, so every
// role that waits on another role of the same job waits on one that already
// runs; all waits are bounded and set an error bit instead of hanging.
#include <cuda.h>

#include "fused_common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {
using namespace fused_common;

constexpr int kThreads = 384;

// ---------------------------------------------------------------- shared memory
constexpr uint32_t kAtomQ = 16384;                  // [128 rows x 128 B] swizzled block
constexpr uint32_t kAtom64 = 8192;                  // [64 rows x 128 B] swizzled block
// consumer: K ring (K_nope 2 blocks + k_rope 1 block per 128 keys) and V ring (2 blocks)
constexpr int kKStages = 3, kVStages = 2;
constexpr uint32_t kKStageBytes = 3 * kAtomQ;       // 49152
constexpr uint32_t kVStageBytes = 2 * kAtomQ;       // 32768
constexpr uint32_t kKBase = 0;
constexpr uint32_t kVBase = kKBase + kKStages * kKStageBytes;      // 147456
constexpr uint32_t kXchgBase = kVBase + kVStages * kVStageBytes;   // 212992: row-max / row-sum exchange
constexpr uint32_t kConsumerEnd = kXchgBase + 6 * 128 * 4;         // max x2 buffers x2 halves, sum x2 halves
// producer
constexpr uint32_t kPStageBytes = 65536;            // C_A 16K | C_B 16K | W 32K
constexpr uint32_t kPCA = 0, kPCB = 16384, kPW = 32768;
constexpr uint32_t kPOutBase = 2 * kPStageBytes;    // bf16 output staging: 32 KB per warpgroup
constexpr uint32_t kProducerEnd = kPOutBase + 2 * 32768;             // 196608
constexpr uint32_t kBarBase = kConsumerEnd > kProducerEnd ? kConsumerEnd : kProducerEnd;
constexpr uint32_t kSmemBytes = kBarBase + 256 + 1024;
static_assert(kSmemBytes <= 232448, "more than 227 KB of shared memory per CTA");

// consumer barriers
constexpr uint32_t kBQReady = 0, kBKFull = 1, kBKEmpty = 4, kBVFull = 7, kBVEmpty = 9, kBSFull = 11, kBPFull = 13,
                   kBPvDone = 15 /* 2: PV of even / odd tiles */;
// producer barriers
constexpr uint32_t kBProdFull = 0, kBProdEmpty = 2, kBAccFull = 4, kBAccEmpty = 5;
constexpr uint32_t kNumBars = 24;

// TMEM columns
constexpr uint32_t kTmQ = 0;        // consumer: Q as bf16 pairs, 96 columns
constexpr uint32_t kTmO = 128;      // consumer: O [128 x 128] fp32
constexpr uint32_t kTmS = 256;      // consumer: S buffer b at 256 + 128 b (P as bf16 pairs in its first 64)
constexpr uint32_t kTmAccA = 0, kTmAccB = 256;   // producer

constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdescUp = idesc_bf16(128, 256, false, true);

constexpr float kRescaleThreshold = 8.f;   // log2 units: P stays <= 256

__device__ __forceinline__ uint32_t bar_addr(uint32_t sbase, uint32_t i) { return sbase + kBarBase + 8u * i; }

// Tiles consumer `ci` loads: a paired consumer (ci and ci^1 in one cluster)
// loads the tiles of both, since each CTA of the pair brings half of every
// tile into both shared memories.
__device__ __forceinline__ int consumer_load_tiles(const Job& J, int ci, int pair) {
  int n = consumer_tiles(J, ci);
  if (pair && (ci ^ 1) < J.n_cons) n = max(n, consumer_tiles(J, ci ^ 1));
  return n;
}

// Consumer CTAs that load tile t (each adds 2 to the slot's consumed count).
__device__ __forceinline__ int consumers_needing_tile(const Job& J, int t, int pair) {
  int n = 0;
  for (int ci = 0; ci < J.n_cons; ++ci) n += consumer_load_tiles(J, ci, pair) > t;
  return n;
}

// =============================================================== consumer
// One 128-query tile of a job.  Warps: 0-7 softmax (warpgroup w owns key
// columns 64w..64w+63 of every row; warpgroup 0 first loads and rotates Q into
// TMEM), 8 K loader, 9 MMA issuer, 10 V loader (the loaders also release the
// ring slots of the tiles that leave their stages).
// `paired`: this CTA and its cluster peer own query tiles ci and ci^1 of the
// same job and run the same key tiles; each CTA loads half of every K and V
// stage (block `rank`) with multicast into both, and both MMAs must release a
// stage (commits to both CTAs' empty barriers) before either refills it.
template <bool kCompute>
__device__ void run_consumer(const FusedParams& p, const Job& J, int job, int ci, int role, uint32_t sbase,
                             uint8_t* sgen, uint32_t tmem, volatile Ctl* ctl, bool paired, uint32_t rank) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q0 = ci * 128;
  const int nq = min(128, J.q_count - q0);
  const int grow0 = J.q_begin + q0;
  const int n_tiles = consumer_load_tiles(J, ci, paired ? 1 : 0);
  const uint16_t kBoth = 3;
  const int H = p.num_heads;

  if constexpr (!kCompute) {
  if (warp == 11 && !paired) {
    // ------------------------------------------------------------ second K issuer
    // K_nope hi and k_rope of every stage, so the K stage's boxes leave from
    // two warps (the per-SM TMA rate grows with the number of issuing warps);
    // warp 8 arms the stage's barrier and loads K_nope lo.
    if (lane != 0) return;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kKStages;
      if (!wait_flag_geq(p, ready_flag(p, job, ring_slot(p, j)), (uint32_t)j + 1)) { ctl->abort = 1; return; }
      if (j >= kKStages && !wait_bar(p, bar_addr(sbase, kBKEmpty + s), ((j / kKStages) - 1) & 1)) {
        ctl->abort = 1;
        return;
      }
      fence_proxy_async_global();
      const uint32_t st = sbase + kKBase + s * kKStageBytes;
      const uint32_t full = bar_addr(sbase, kBKFull + s);
      const int zb = (job * p.ring_depth + ring_slot(p, j)) * 4;
      tma_load_3d(st + kAtomQ, &p.tm_ring1, 0, 0, zb + 1, full);                               // K_nope hi
      tma_load_2d(st + 2 * kAtomQ, &p.tm_kr128, kDc, block_row(J, (J.t0 + 128 * j) >> 6), full);   // k_rope
    }
    // the last stages' MMAs: their commits land before the barriers are reset
    for (int j = max(0, n_tiles - kKStages); j < n_tiles; ++j)
      if (!wait_bar(p, bar_addr(sbase, kBKEmpty + j % kKStages), (j / kKStages) & 1)) { ctl->abort = 1; return; }
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ TMA loads (K or V)
    if (lane != 0) return;
    const bool is_k = warp == 8;
    TraceAcc tr;
    for (int j = 0; j < n_tiles; ++j) {
      const int ns = is_k ? kKStages : kVStages;
      const int s = j % ns;
      // The tile must be published.  Checked before the stage wait: producers
      // run ahead, so the flag is normally set already, and the round trip to
      // L2 overlaps the wait for the stage instead of following it.
      const uint64_t w0 = tr.begin(p);
      if (!wait_flag_geq(p, ready_flag(p, job, ring_slot(p, j)), (uint32_t)j + 1)) { ctl->abort = 1; return; }
      tr.end(p, w0);
      // stage reusable: the MMAs reading its previous tile are done
      if (j >= ns && !wait_bar(p, bar_addr(sbase, (is_k ? kBKEmpty : kBVEmpty) + s), ((j / ns) - 1) & 1)) {
        ctl->abort = 1;
        return;
      }
      fence_proxy_async_global();
      const int zb = (job * p.ring_depth + ring_slot(p, j)) * 4;   // first ring block of the tile
      if (is_k) {
        const uint32_t st = sbase + kKBase + s * kKStageBytes;
        const uint32_t full = bar_addr(sbase, kBKFull + s);
        mbar_arrive_expect_tx(full, kKStageBytes);       // both halves land here, the peer's by multicast
        const int kt0 = J.t0 + 128 * j;
        if (paired) {
          const int h = (int)rank;
          tma_load_3d_mc(st + h * kAtomQ, &p.tm_ring1, 0, 0, zb + h, full, kBoth);          // K_nope block h
          tma_load_2d_mc(st + 2 * kAtomQ + h * kAtom64, &p.tm_kr, kDc, block_row(J, (kt0 >> 6) + h), full,
                         kBoth);                                                             // k_rope, 64 keys
        } else {
          tma_load_3d(st, &p.tm_ring1, 0, 0, zb, full);                     // K_nope lo (warp 11: hi, k_rope)
          (void)kt0;
        }
        trace_stage(p, role, j, 0);
      } else {
        const uint32_t st = sbase + kVBase + s * kVStageBytes;
        const uint32_t full = bar_addr(sbase, kBVFull + s);
        mbar_arrive_expect_tx(full, kVStageBytes);
        if (paired)
          tma_load_3d_mc(st + rank * kAtomQ, &p.tm_ring1, 0, 0, zb + 2 + (int)rank, full, kBoth);  // V block
        else
          tma_load_3d(st, &p.tm_ring, 0, 0, zb + 2, full);                  // V, 32 KB
        trace_stage(p, role, j, 1);
      }
      // The tile that left the stage is consumed here: add one to its slot's
      // count (a slot is free again after 2 per consumer).  Done after the
      // next load is issued, so the release is off the path to the MMA.
      if (j >= ns) {
        fence_proxy_async_global();
        red_release_gpu_add(consumed_flag(p, job, ring_slot(p, j - ns)), 1u);
      }
    }
    // the last stages: once their MMAs are done, release their tiles' slots
    // (this also takes the last commits' arrivals before the barriers are reset)
    const int ns = is_k ? kKStages : kVStages;
    for (int j = max(0, n_tiles - ns); j < n_tiles; ++j) {
      if (!wait_bar(p, bar_addr(sbase, (is_k ? kBKEmpty : kBVEmpty) + j % ns), (j / ns) & 1)) { ctl->abort = 1; return; }
      fence_proxy_async_global();
      red_release_gpu_add(consumed_flag(p, job, ring_slot(p, j)), 1u);
    }
    if (is_k) trace_put(p, role, 3, tr.t);
    if (is_k) trace_put(p, role, 7, (unsigned long long)n_tiles);
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issue
    if (lane != 0) return;
    TraceAcc tr_kv, tr_p;
    bool ok = wait_bar(p, bar_addr(sbase, kBQReady), 0);
    auto issue_s = [&](int j) {
      const int sk = j % kKStages, b = j & 1;
      trace_stage(p, role, j, 2);
      tc_fence_after();
      const uint32_t k = sbase + kKBase + sk * kKStageBytes;
      const uint32_t d = tmem + kTmS + 128 * b;
#pragma unroll
      for (int kk = 0; kk < 12; ++kk)
        mma_bf16_ts(d, tmem + kTmQ + kk * 8, sdesc_sw128(k + (kk >> 2) * kAtomQ + (kk & 3) * 32, 16, 1024), kIdescS,
                    kk > 0 ? 1u : 0u);
      mma_commit(bar_addr(sbase, kBSFull + b));
      if (paired) mma_commit_mc(bar_addr(sbase, kBKEmpty + sk), kBoth);
      else mma_commit(bar_addr(sbase, kBKEmpty + sk));
      trace_stage(p, role, j, 3);
    };
    auto issue_pv = [&](int jj) {
      const int b = jj & 1, sv = jj % kVStages;
      trace_stage(p, role, jj, 4);
      if (!wait_bar(p, bar_addr(sbase, kBVFull + sv), (jj / kVStages) & 1)) { ok = false; return; }
      trace_stage(p, role, jj, 5);
      tc_fence_after();
      const uint32_t v = sbase + kVBase + sv * kVStageBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16_ts(tmem + kTmO, tmem + kTmS + 128 * b + kk * 8, sdesc_sw128(v + kk * 2048, kAtomQ, 1024), kIdescPV,
                    (jj > 0 || kk > 0) ? 1u : 0u);
      mma_commit(bar_addr(sbase, kBPvDone + b));
      if (paired) mma_commit_mc(bar_addr(sbase, kBVEmpty + sv), kBoth);
      else mma_commit(bar_addr(sbase, kBVEmpty + sv));
    };
    // S(j) needs K(j); PV(j-1) needs P(j-1) and V(j-1).  S(j) may run before
    // PV(j-1) (its S buffer's previous P was consumed by PV(j-2), issued
    // earlier), so issue whichever becomes ready first; S(j+1) always waits
    // for PV(j-1) to have been issued.
    int js = 0, jp = 0;           // next S to issue, next PV to issue
    const uint64_t t_start = p.trace ? global_timer_ns() : 0;
    uint64_t t_last = global_timer_ns();
    uint32_t polls = 0;
    while (ok && (js < n_tiles || jp < n_tiles)) {
      bool progressed = false;
      const bool want_s = js < n_tiles && js <= jp + 1;
      const bool want_p = jp < js;
      // sleep on the barrier of the older outstanding work; peek at the other one
      const uint32_t hint = (want_s && want_p) ? 200u : 20000u;
      if (want_s && mbar_try_wait_hint(bar_addr(sbase, kBKFull + js % kKStages), (js / kKStages) & 1,
                                       want_p ? 0u : hint)) {
        issue_s(js++);
        progressed = true;
      }
      if (want_p && mbar_try_wait_hint(bar_addr(sbase, kBPFull + (jp & 1)), (jp >> 1) & 1, hint)) {
        issue_pv(jp++);
        progressed = true;
      }
      if (progressed) {
        polls = 0;
      } else if ((++polls & 255u) == 0u) {
        const uint64_t now = global_timer_ns();
        if (polls == 256u) t_last = now;
        else if (now - t_last > kWaitLimitNs) {
          atomicOr(p.err, kErrTimeout);
          ok = false;
        }
      }
    }
    tr_kv.t = p.trace ? global_timer_ns() - t_start : 0;
    if (ok && n_tiles > 0) {
      // the last commits' arrivals must land before the barriers are reset for the next role
      const int jl = n_tiles - 1;
      if (ok && !wait_bar(p, bar_addr(sbase, kBVEmpty + jl % kVStages), (jl / kVStages) & 1)) ok = false;
      if (ok && !wait_bar(p, bar_addr(sbase, kBKEmpty + jl % kKStages), (jl / kKStages) & 1)) ok = false;
    }
    if (!ok) ctl->abort = 1;
    trace_put(p, role, 4, tr_kv.t);
    trace_put(p, role, 5, tr_p.t);
  }
  } else {
    if (warp < 4) {
      // ---------------------------------------------------------- Q -> TMEM (warpgroup 0)
    const int r = tid & 127;
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      const bool live = r < nq;
      const int grow = grow0 + r;
      const uint4* src = reinterpret_cast<const uint4*>(p.q_bf16 + ((int64_t)(live ? grow : 0) * H + J.head) * kDqk);
      const int64_t delta = live ? (int64_t)__ldg(p.q_pos + grow) - J.rope_offset : 0;
      // 32 TMEM columns (64 bf16) at a time: q_nope 0..63, q_nope 64..127, rotated q_rope
#pragma unroll 1
      for (int part = 0; part < 3; ++part) {
        uint32_t qv[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 a = live ? __ldg(src + 8 * part + c) : make_uint4(0, 0, 0, 0);
          uint32_t w4[4] = {a.x, a.y, a.z, a.w};
          if (part == 2) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float sn, cs;
              rope_sincos(delta, p.rope_frac[4 * c + i], &sn, &cs);
              const float x0 = __uint_as_float(w4[i] << 16), x1 = __uint_as_float(w4[i] & 0xFFFF0000u);
              w4[i] = pack_bf16(x0 * cs - x1 * sn, x0 * sn + x1 * cs);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) qv[4 * c + i] = w4[i];
        }
        tmem_st32(tmem + lane_off + kTmQ + 32 * part, qv);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, kBQReady));
    }
    // ------------------------------------------------------------ softmax / epilogue (warps 0..7)
    const int w = warp >> 2;           // key half
    const int r = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float* xchg = reinterpret_cast<float*>(sgen + kXchgBase);   // [2 buffers][2 halves][128] maxima, then sums
    const int qtok = query_token(J, q0 + r);
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l_part = 0.f;
    bool ok = true;
    TraceAcc tr_s;
    for (int j = 0; j < n_tiles; ++j) {
      const int b = j & 1;
      const uint64_t w0 = tr_s.begin(p);
      if (ok && !wait_bar_warp(p, bar_addr(sbase, kBSFull + b), (j >> 1) & 1)) ok = false;
      tr_s.end(p, w0);
      if (tid == 0) trace_stage(p, role, j, 6);
      tc_fence_after();
      const uint32_t scol = tmem + lane_off + kTmS + 128 * b + 64 * w;
      uint32_t v[64];
      if (ok) tmem_ld64(scol, v);
      const int kt0 = J.t0 + 128 * j + 64 * w;
      const bool full = kt0 >= J.k_begin && kt0 + 63 < J.k_end && kt0 + 63 <= qtok;
      float m8[8];
      if (full) {
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = __uint_as_float(v[i]);
#pragma unroll
        for (int c = 8; c < 64; c += 2)
          m8[(c >> 1) & 7] = fmax3(m8[(c >> 1) & 7], __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int kt = kt0 + c;
          const bool okc = kt >= J.k_begin && kt < J.k_end && kt <= qtok;
          const float x = okc ? __uint_as_float(v[c]) : -INFINITY;
          v[c] = __float_as_uint(x);
          m8[c & 7] = fmaxf(m8[c & 7], x);
        }
      }
      float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      // row maximum over both key halves; the barrier also orders both
      // warpgroups' S loads before either overwrites S with P
      xchg[(b * 2 + w) * 128 + r] = mx;
      tc_fence_before();
      named_bar_sync(1, 256);
      tc_fence_after();
      mx = fmaxf(mx, xchg[(b * 2 + (1 - w)) * 128 + r]);
      const float m_tile = mx * sl2;
      float alpha = 1.f;
      const bool rescale = m_tile > m_used + kRescaleThreshold;
      if (rescale) {
        alpha = ex2(m_used - m_tile);   // 0 when m_used = -inf
        m_used = m_tile;
      }
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      // exponent arguments and row sums on packed pairs: s * scale - m, then 2^x
      // P is packed in place over the scores (pair c lands in v[c], whose score
      // was consumed at pair c/2) and stored in two 16-column halves, so the
      // first half's store overlaps the second half's exponentials.
      const uint64_t sc2 = f2pack(sl2, sl2), nm2 = f2pack(-mref, -mref);
      uint64_t s4[4] = {0ull, 0ull, 0ull, 0ull};
      const uint32_t pcol = tmem + lane_off + kTmS + 128 * b + 32 * w;   // P over S's first 64 columns
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
      float s8[8];
      f2unpack(fadd2(s4[0], s4[1]), s8[0], s8[1]);
      f2unpack(fadd2(s4[2], s4[3]), s8[2], s8[3]);
      l_part = l_part * alpha + ((s8[0] + s8[2]) + (s8[1] + s8[3]));
      if (j >= 1 && ok && __any_sync(0xffffffffu, rescale)) {
        // O holds PV of tiles < j: PV(j-1) must be done before O is rescaled.  PV(j-2)
        // finished before S(j) did, so this barrier is at most one phase behind.
        if (!wait_bar_warp(p, bar_addr(sbase, kBPvDone + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) ok = false;
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
      mbar_arrive(bar_addr(sbase, kBPFull + b));
      if (tid == 0) trace_stage(p, role, j, 7);
    }
    if (ok && n_tiles > 0 &&
        !wait_bar_warp(p, bar_addr(sbase, kBPvDone + ((n_tiles - 1) & 1)), ((n_tiles - 1) >> 1) & 1))
      ok = false;
    if (tid == 0) trace_put(p, role, 6, tr_s.t);
    // row sum over both key halves (its own region: a slow partner may still read the maxima)
    xchg[(4 + w) * 128 + r] = l_part;
    named_bar_sync(1, 256);
    const float l_run = l_part + xchg[(4 + (1 - w)) * 128 + r];
    if (!ok) { ctl->abort = 1; return; }
    tc_fence_after();
    // ---- epilogue: this warpgroup writes output columns 64w .. 64w+63
    const bool empty = n_tiles == 0 || !(l_run > 0.f);
    const float inv_l = empty ? 0.f : 1.f / l_run;
    const bool live = r < nq;
    const int grow = grow0 + r;
    const int64_t orow = J.slot < 0 ? (int64_t)grow : (int64_t)J.slot * p.slot_stride_rows + grow;
    const uint32_t ocol = tmem + lane_off + kTmO + 64 * w;
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
    if (live && w == 0) {
      const float lse = empty ? -INFINITY : m_used * 0.69314718055994531f + logf(l_run);
      (J.slot < 0 ? p.lse : p.part_lse)[orow * H + J.head] = lse;
    }
  }
}

// =============================================================== producer
template <bool kCompute>
__device__ void run_producer(const FusedParams& p, const Job& J, int job, int pi, int role, uint32_t sbase,
                             uint32_t tmem, volatile Ctl* ctl) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_pass = (J.n_tiles + 1) >> 1;
  const int H = p.num_heads;
  const int h = J.head;
  int my_passes = 0;
  for (int pp = pi; pp < n_pass; pp += J.n_prod) ++my_passes;
  if (my_passes == 0) return;

  if constexpr (!kCompute) {
  if (warp == 8 || warp == 10) {
    // TMA issue, split over two warps: warp 8 loads the pass's 256 latent rows
    // (one 256-row box per 64-wide slice) and arms the stage, warp 10 the
    // head's kv_b_proj slices (K_nope columns, V columns).
    if (lane == 0) {
      const bool primary = warp == 8;
      int g = 0;
      for (int n = 0; n < my_passes; ++n) {
        const int pass = pi + n * J.n_prod;
        const int row0 = block_row(J, (J.t0 >> 6) + 4 * pass);
        for (int k = 0; k < kDc / 64; ++k, ++g) {
          const int s = g & 1;
          if (g >= 2 && !wait_bar(p, bar_addr(sbase, kBProdEmpty + s), ((g >> 1) - 1) & 1)) { ctl->abort = 1; return; }
          const uint32_t st = sbase + s * kPStageBytes;
          const uint32_t bar = bar_addr(sbase, kBProdFull + s);
          if (primary) {
            mbar_arrive_expect_tx(bar, kPStageBytes);
            tma_load_2d(st + kPCA, &p.tm_c, 64 * k, row0, bar);                                        // C_A | C_B
          } else {
            tma_load_3d(st + kPW, &p.tm_w, 0, 64 * k, 2 * h, bar);                                   // K_nope cols
            tma_load_3d(st + kPW + 2 * kAtom64, &p.tm_w, 0, 64 * k, (H * kDnope + h * kDv) / 64, bar); // V cols
          }
        }
      }
    }
  } else if (warp == 9) {
    if (lane == 0) {
      TraceAcc tr_op, tr_acc;
      int g = 0;
      for (int n = 0; n < my_passes; ++n) {
        const uint64_t wa = tr_acc.begin(p);
        if (n >= 1 && !wait_bar(p, bar_addr(sbase, kBAccEmpty), (n - 1) & 1)) { ctl->abort = 1; return; }
        tr_acc.end(p, wa);
        for (int k = 0; k < kDc / 64; ++k, ++g) {
          const int s = g & 1;
          const uint64_t w0 = tr_op.begin(p);
          if (!wait_bar(p, bar_addr(sbase, kBProdFull + s), (g >> 1) & 1)) { ctl->abort = 1; return; }
          tr_op.end(p, w0);
          tc_fence_after();
          const uint32_t st = sbase + s * kPStageBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = sdesc_sw128(st + kPW + kk * 2048, kAtom64, 1024);
            mma_bf16(tmem + kTmAccA, sdesc_sw128(st + kPCA + kk * 32, 16, 1024), bdesc, kIdescUp, (k | kk) ? 1u : 0u);
            mma_bf16(tmem + kTmAccB, sdesc_sw128(st + kPCB + kk * 32, 16, 1024), bdesc, kIdescUp, (k | kk) ? 1u : 0u);
          }
          mma_commit(bar_addr(sbase, kBProdEmpty + s));
        }
        mma_commit(bar_addr(sbase, kBAccFull));
      }
      trace_put(p, role, 4, tr_op.t);
      trace_put(p, role, 5, tr_acc.t);
      trace_put(p, role, 7, (unsigned long long)my_passes);
    }
  }
  } else {
  {
    // conversion: warpgroup 0 -> tile 2*pass, warpgroup 1 -> tile 2*pass + 1
    const int wg = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float oscale = p.out_scale;
    const uint32_t stage_out = sbase + kPOutBase + wg * 32768;   // [128 rows x 128 cols] bf16, 2 SW128 blocks
    TraceAcc tr_c;
    for (int n = 0; n < my_passes; ++n) {
      const int pass = pi + n * J.n_prod;
      const int t = 2 * pass + wg;
      const bool live_tile = t < J.n_tiles;
      const int slot = ring_slot(p, t);
      const int tok = J.t0 + 128 * t + r;
      const bool valid = tok >= J.k_begin && tok < J.k_end;
      const uint32_t acc = tmem + lane_off + (wg ? kTmAccB : kTmAccA);
      if (!wait_bar_warp(p, bar_addr(sbase, kBAccFull), n & 1)) ctl->abort = 1;
      tc_fence_after();
      // staging is free: thread 0 waited for the previous tile's stores to read it
      named_bar_sync(1 + wg, 128);
      uint32_t vpk[64];
      if (live_tile && !ctl->abort) {
        // K_nope half (accumulator columns 0..127) -> shared staging
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t a[32];
          tmem_ld32(acc + cc * 32, a);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              w[i] = valid ? pack_bf16(__uint_as_float(a[8 * g + 2 * i]) * oscale,
                                       __uint_as_float(a[8 * g + 2 * i + 1]) * oscale) : 0u;
            sts128(stage_out + (cc >> 1) * kAtomQ + sw128_off(r, (cc & 1) * 4 + g), w[0], w[1], w[2], w[3]);
          }
        }
        // V half (columns 128..255) -> registers, so the accumulators can be released now
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t a[32];
          tmem_ld32(acc + 128 + cc * 32, a);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            vpk[16 * cc + i] = valid ? pack_bf16(__uint_as_float(a[2 * i]) * oscale, __uint_as_float(a[2 * i + 1]) * oscale) : 0u;
        }
      }
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, kBAccEmpty));     // the next pass may overwrite the accumulators
      if (live_tile) {
        fence_proxy_async_smem();
        named_bar_sync(1 + wg, 128);
        const int zb = (job * p.ring_depth + slot) * 4;
        if (r == 0 && !ctl->abort) {
          const uint64_t w0 = tr_c.begin(p);
          // the slot's previous occupant (tile t - ring) must be published and fully consumed
          if (t >= p.ring_depth &&
              !(wait_flag_geq(p, ready_flag(p, job, slot), (uint32_t)(t - p.ring_depth + 1)) &&
                wait_flag_geq(p, consumed_flag(p, job, slot), 2u * (uint32_t)consumers_needing_tile(J, t - p.ring_depth, p.pair))))
            ctl->abort = 1;
          tr_c.end(p, w0);
          *consumed_flag(p, job, slot) = 0u;    // ordered before the release of `ready` below
          tma_store_3d(&p.tm_ring, stage_out, 0, 0, zb);               // K_nope lo | hi
          bulk_commit();
          bulk_wait_read0();                    // staging free for the V half
        }
        named_bar_sync(1 + wg, 128);
        if (ctl->abort) return;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int g = 0; g < 4; ++g)
            sts128(stage_out + (cc >> 1) * kAtomQ + sw128_off(r, (cc & 1) * 4 + g), vpk[16 * cc + 4 * g],
                   vpk[16 * cc + 4 * g + 1], vpk[16 * cc + 4 * g + 2], vpk[16 * cc + 4 * g + 3]);
        fence_proxy_async_smem();
        named_bar_sync(1 + wg, 128);
        if (r == 0) {
          tma_store_3d(&p.tm_ring, stage_out, 0, 0, zb + 2);           // V lo | hi
          bulk_commit();
          bulk_wait0();                         // both halves have landed
          fence_proxy_async_global();
          __threadfence();
          st_release_gpu(ready_flag(p, job, slot), (uint32_t)t + 1);
        }
      }
      if (ctl->abort) return;
    }
    if (tid == 0) trace_put(p, role, 3, tr_c.t);
  }
  }
}

// The role loop, instantiated once for the compute warps (0-7: softmax,
// conversion, Q load) and once for the control warps (8-11: TMA, MMA issue,
// ring release), which run it with different register budgets.
template <bool kCompute>
__device__ __forceinline__ void role_loop(const FusedParams& p, uint32_t sbase, uint8_t* sgen, volatile Ctl* ctl,
                                          uint32_t tmem) {
  const int tid = threadIdx.x;
  // Role groups: cluster rank 0 takes the next group from the queue and
  // writes it into both CTAs; every exit decision is made there, so both CTAs
  // of a cluster run the same sequence of cluster barriers.  A group holds up
  // to two producer roles of one job (independent) or a consumer pair (query
  // tiles 2k and 2k+1 of one job, sharing K/V loads); without pairing it holds
  // one role.
  const uint32_t rank = p.pair ? cluster_rank() : 0u;
  const int width = p.pair ? 2 : 1;
  cluster_sync_all();   // every CTA of the cluster has started before any shared::cluster access
  for (;;) {
    if (kCompute && tid == 0 && rank == 0) {
      const int g = (ctl->abort || aborted_global(p)) ? p.n_groups : (int)atomicAdd(p.queue, 1u);
      ctl->group = g;
      if (p.pair) st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(&ctl->group)), 1u), (uint32_t)g);
    }
    tc_fence_before();
    cluster_sync_all();   // also: both CTAs are done with the previous group
    tc_fence_after();
    const int g = ctl->group;
    if (g >= p.n_groups) break;
    int lo = 0, hi = p.n_pieces - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.pieces[mid].group_begin <= g) lo = mid; else hi = mid - 1;
    }
    const Piece& P = p.pieces[lo];
    const int gp = (P.n_prod + width - 1) / width, gc = (P.n_cons + width - 1) / width;
    const int local = g - P.group_begin;
    Job J;
    J.req = P.req;
    J.head = local / (gp + gc);
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
    const int job = lo * p.num_heads + J.head;
    const int gi = local - J.head * (gp + gc);
    const bool producer = gi < gp;
    const int idx = (producer ? gi : gi - gp) * width + (int)rank;
    const bool valid = idx < (producer ? J.n_prod : J.n_cons);
    const bool paired = !producer && p.pair && ((gi - gp) * 2 + 1) < J.n_cons;
    const int slot = g * 2 + (int)rank;   // trace slot
    if (kCompute && tid == 32) {
      // fresh barriers for this role (every barrier is idle here)
      for (uint32_t i = 0; i < kNumBars; ++i) {
        mbar_inval(bar_addr(sbase, i));
        uint32_t cnt = 1;
        if (!producer && (i == kBPFull || i == kBPFull + 1)) cnt = 256;
        if (!producer && i == kBQReady) cnt = 128;
        if (producer && i == kBAccEmpty) cnt = 256;
        if (paired && ((i >= kBKEmpty && i < kBKEmpty + kKStages) || (i >= kBVEmpty && i < kBVEmpty + kVStages)))
          cnt = 2;   // both MMAs of the pair release a stage
        mbar_init(bar_addr(sbase, i), cnt);
      }
      fence_mbar_init();
    }
    cluster_sync_all();   // the peer's barriers exist before any multicast or commit reaches them
    if (valid) {
      if (kCompute && p.trace && tid == 0) {
        trace_put(p, slot, 0, global_timer_ns());
        trace_put(p, slot, 2, ((unsigned long long)blockIdx.x << 32) | ((unsigned long long)producer << 31) | (unsigned)job);
      }
      if (!ctl->abort) {
        if (producer) run_producer<kCompute>(p, J, job, idx, slot, sbase, tmem, ctl);
        else run_consumer<kCompute>(p, J, job, idx, slot, sbase, sgen, tmem, ctl, paired, rank);
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
      if (kCompute && p.trace && tid == 0) trace_put(p, slot, 1, global_timer_ns());
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) fused_prefill_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  volatile Ctl* ctl = reinterpret_cast<volatile Ctl*>(sgen + kBarBase + 8 * kNumBars);
  const int tid = threadIdx.x;

  if (tid == 0) {
    prefetch_tensormap(&p.tm_kr);
    prefetch_tensormap(&p.tm_c);
    prefetch_tensormap(&p.tm_w);
    prefetch_tensormap(&p.tm_ring);
  }
  if ((tid >> 5) == 0) {
    tmem_alloc(sbase + kBarBase + 8 * kNumBars + offsetof(Ctl, tmem), 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    ctl->abort = 0;
    for (uint32_t i = 0; i < kNumBars; ++i) mbar_init(bar_addr(sbase, i), 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;

  // Registers: the control warps need few, the compute warps many.  At
  // launch every thread has 168 (384 x 168 = 64512); warpgroup 2 gives back
  // 112 each (128 x 112) and warpgroups 0 and 1 take 56 more each (256 x 56):
  // the same total, so the increase never waits on registers that are not there.
  if ((tid >> 5) >= 8) {
    setmaxnreg_dec<56>();
    role_loop<false>(p, sbase, sgen, ctl, tmem);
  } else {
    setmaxnreg_inc<224>();
    role_loop<true>(p, sbase, sgen, ctl, tmem);
  }
  tc_fence_before();
  __syncthreads();
  if ((tid >> 5) == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

int fused_smem_bytes() { return (int)kSmemBytes; }

static cudaError_t configure(int dev) {
  static int configured_device = -1;
  if (configured_device == dev) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fused_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e == cudaSuccess) configured_device = dev;
  return e;
}

// Pairs: clusters of two CTAs (no cooperative attribute: a role only ever
// waits on roles dequeued before it, which run on CTAs that are resident).
// Without pairs: a cooperative launch of single CTAs.
cudaError_t launch_fused(const FusedParams& p, int grid, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = configure(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (p.pair) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fused_prefill_kernel, p);
  count_launch();
  return e;
}

cudaError_t fused_grid_size(int* grid, int pair) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = configure(dev);
  if (e != cudaSuccess) return e;
  if (pair) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * ((sms + 1) / 2));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, fused_prefill_kernel, &cfg);
    if (e != cudaSuccess) return e;
    *grid = 2 * clusters;
  } else {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_prefill_kernel, kThreads, kSmemBytes);
    if (e != cudaSuccess) return e;
    *grid = sms * (per_sm > 0 ? per_sm : 0);
  }
  return *grid > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

}  // namespace mla
