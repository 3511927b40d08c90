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

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 512;
constexpr uint32_t kRing = kRingDepth;

// ---------------------------------------------------------------- shared memory
constexpr uint32_t kAtomQ = 16384;                  // [128 rows x 128 B]
constexpr uint32_t kAtom64 = 8192;                  // [64 rows x 128 B]
constexpr uint32_t kQBytes = 3 * kAtomQ;            // nope lo | nope hi | rope
constexpr uint32_t kStageBase = 2 * kQBytes;        // 98304
constexpr uint32_t kStageK = 0;                     // K_nope [64 x 128]: 2 atoms
constexpr uint32_t kStageKR = 2 * kAtom64;          // k_rope [64 x 64]
constexpr uint32_t kStageV = 3 * kAtom64;           // V [64 x 128]: 2 dv blocks
constexpr uint32_t kStageBytes = 5 * kAtom64;       // 40960
constexpr int kStages = 3;
// producer
constexpr uint32_t kPStageBytes = 65536;            // C_A 16K | C_B 16K | W 32K
constexpr uint32_t kPCA = 0, kPCB = 16384, kPW = 32768;
constexpr uint32_t kPRawBase = 2 * kPStageBytes;    // e4m3 staging, 16 KB per stage
constexpr uint32_t kBarBase = kStageBase + kStages * kStageBytes;  // 221184
constexpr uint32_t kSmemBytes = kBarBase + 256 + 1024;

// consumer barriers
constexpr uint32_t kBQFull = 0, kBQReady = 1, kBKvFull = 3, kBKvEmpty = 6, kBSFull = 9, kBPFull = 13, kBPvDone = 17;
// producer barriers
constexpr uint32_t kBProdFull = 0, kBProdEmpty = 2, kBRawFull = 4, kBAccFull = 6, kBAccEmpty = 7;
constexpr uint32_t kNumBars = 20;

// TMEM columns
constexpr uint32_t kTmO = 0;        // O of query tile u at u*128
constexpr uint32_t kTmS = 256;      // S of (u, b) at 256 + (2u + b) * 64
constexpr uint32_t kTmAccA = 0, kTmAccB = 256;

constexpr uint32_t kIdescS = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdescUp = idesc_bf16(128, 256, false, true);

constexpr float kRescaleThreshold = 8.f;   // log2 units: P stays <= 256

struct Ctl {
  int role;
  int abort;
  uint32_t tmem;
};

__device__ __forceinline__ uint32_t bar_addr(uint32_t sbase, uint32_t i) { return sbase + kBarBase + 8u * i; }

__device__ __forceinline__ bool aborted_global(const FusedParams& p) { return ld_volatile_u32(p.err) != 0u; }

// Bounded mbarrier wait; on timeout records the error and returns false.
__device__ __forceinline__ bool wait_bar(const FusedParams& p, uint32_t bar, uint32_t parity) {
  if (mbar_wait(bar, parity)) return true;
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
__device__ bool wait_flag_geq(const FusedParams& p, const uint32_t* flag, uint32_t target) {
  if (ld_acquire_gpu(flag) >= target) return true;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_gpu(flag) < target) {
    if (global_timer_ns() - t0 > kWaitLimitNs || aborted_global(p)) {
      atomicOr(p.err, kErrTimeout);
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

// Number of 64-key stages consumer `ci` of job `J` attends to (causal clip).
__device__ __forceinline__ int consumer_stages(const Job& J, int ci) {
  const int q0 = ci * 256;
  const int nq = min(256, J.q_count - q0);
  if (nq <= 0) return 0;
  const int last_tok = J.q_tok0 + q0 + nq - 1;
  const int k_end = min(J.k_end, last_tok + 1);
  if (k_end <= J.k_begin) return 0;
  return (k_end - J.t0 + 63) >> 6;
}

__device__ __forceinline__ int consumers_needing_tile(const Job& J, int t) {
  int n = 0;
  for (int ci = 0; ci < J.n_cons; ++ci) n += ((consumer_stages(J, ci) + 1) >> 1) > t;
  return n;
}

__device__ __forceinline__ uint32_t* ready_flag(const FusedParams& p, int job, int slot) {
  return p.flags + (size_t)job * (2 * kRing) + slot;
}
__device__ __forceinline__ uint32_t* consumed_flag(const FusedParams& p, int job, int slot) {
  return p.flags + (size_t)job * (2 * kRing) + kRing + slot;
}

// Physical cache row of logical block `lb` of request `req`, or a negative row
// (TMA fills zeros) when the block lies outside the table; a table entry
// outside [0, num_blocks) for a block holding live tokens is an error.
__device__ __forceinline__ int block_row(const FusedParams& p, int req, int lb, bool live) {
  if (lb < 0 || lb >= p.max_blocks) return -kBlock;
  const int blk = __ldg(p.block_table + (int64_t)req * p.max_blocks + lb);
  if (blk < 0 || blk >= p.num_blocks) {
    if (live) atomicOr(p.err, kErrBadBlock);
    return -kBlock;
  }
  return blk * kBlock;
}

// =============================================================== consumer
__device__ void run_consumer(const FusedParams& p, const Job& J, int job, int ci, uint32_t sbase, uint8_t* sgen,
                             uint32_t tmem, volatile Ctl* ctl) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q0 = ci * 256;
  const int nq_all = min(256, J.q_count - q0);
  const int nq0 = min(128, nq_all), nq1 = max(0, nq_all - 128);
  const int grow0 = J.q_begin + q0;
  const int n_stages = consumer_stages(J, ci);
  const int H = p.num_heads;
  const uint32_t sQ0 = sbase, sQ1 = sbase + kQBytes;

  if (warp == 12) {
    // ------------------------------------------------------------ TMA loads
    if (lane == 0) {
      const uint32_t qf = bar_addr(sbase, kBQFull);
      mbar_arrive_expect_tx(qf, 2 * kQBytes);
      for (int u = 0; u < 2; ++u)
        for (int a = 0; a < 3; ++a)
          tma_load_3d((u ? sQ1 : sQ0) + a * kAtomQ, &p.tm_q, 64 * a, J.head, grow0 + 128 * u, qf);
      const int ring_row0 = job * (int)kRing * 128;
      for (int j = 0; j < n_stages; ++j) {
        const int s = j % kStages;
        if (j >= kStages && !wait_bar(p, bar_addr(sbase, kBKvEmpty + s), ((j / kStages) - 1) & 1)) { ctl->abort = 1; break; }
        const int t = j >> 1, half = j & 1;
        if (half == 0) {
          if (!wait_flag_geq(p, ready_flag(p, job, t % kRing), (uint32_t)t + 1)) { ctl->abort = 1; break; }
          fence_proxy_async_global();
        }
        const int kt0 = J.t0 + 64 * j;
        const int yk = block_row(p, J.req, kt0 >> 6, true);
        const uint32_t st = sbase + kStageBase + s * kStageBytes;
        const uint32_t full = bar_addr(sbase, kBKvFull + s);
        mbar_arrive_expect_tx(full, kStageBytes);
        const int ry = ring_row0 + (t % kRing) * 128 + half * 64;
        tma_load_2d(st + kStageK, &p.tm_ring, 0, ry, full);
        tma_load_2d(st + kStageK + kAtom64, &p.tm_ring, 64, ry, full);
        tma_load_2d(st + kStageV, &p.tm_ring, 128, ry, full);
        tma_load_2d(st + kStageV + kAtom64, &p.tm_ring, 192, ry, full);
        tma_load_2d(st + kStageKR, &p.tm_kr, kDc, yk, full);   // element 512 (bf16) = byte 512 (fp8 row)
      }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      bool ok = wait_bar(p, bar_addr(sbase, kBQReady + 0), 0) && wait_bar(p, bar_addr(sbase, kBQReady + 1), 0);
      const bool act[2] = {nq0 > 0, nq1 > 0};
      auto issue_pv = [&](int jj) {
        const int sp = jj % kStages, bp = jj & 1;
        const uint32_t v = sbase + kStageBase + sp * kStageBytes + kStageV;
        for (int u = 0; u < 2; ++u) {
          if (!act[u]) continue;
          if (!wait_bar(p, bar_addr(sbase, kBPFull + 2 * u + bp), (jj >> 1) & 1)) { ok = false; return; }
          tc_fence_after();
          const uint32_t a = tmem + kTmS + (2 * u + bp) * 64;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(tmem + kTmO + 128 * u, a + kk * 8, sdesc_sw128(v + kk * 2048, kAtom64, 1024), kIdescPV,
                        (jj > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar_addr(sbase, kBPvDone + u));
        }
        mma_commit(bar_addr(sbase, kBKvEmpty + sp));
      };
      for (int j = 0; j < n_stages && ok; ++j) {
        const int s = j % kStages;
        if (!wait_bar(p, bar_addr(sbase, kBKvFull + s), (j / kStages) & 1)) { ok = false; break; }
        if ((j & 1) || j == n_stages - 1) {   // whole ring tile now in shared memory
          fence_proxy_async_global();
          red_release_gpu_add(consumed_flag(p, job, (j >> 1) % kRing), 1u);
        }
        tc_fence_after();
        const uint32_t st = sbase + kStageBase + s * kStageBytes;
        const int b = j & 1;
        for (int u = 0; u < 2; ++u) {
          if (!act[u]) continue;
          const uint32_t q = u ? sQ1 : sQ0;
          const uint32_t d = tmem + kTmS + (2 * u + b) * 64;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (uint32_t)(kk >> 2) * kAtomQ + (uint32_t)(kk & 3) * 32u;
            const uint32_t offk = (uint32_t)(kk >> 2) * kAtom64 + (uint32_t)(kk & 3) * 32u;
            mma_bf16(d, sdesc_sw128(q + off, 16, 1024), sdesc_sw128(st + kStageK + offk, 16, 1024), kIdescS,
                     kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16(d, sdesc_sw128(q + 2 * kAtomQ + kk * 32, 16, 1024), sdesc_sw128(st + kStageKR + kk * 32, 16, 1024),
                     kIdescS, 1u);
          mma_commit(bar_addr(sbase, kBSFull + 2 * u + b));
        }
        if (j >= 1) issue_pv(j - 1);
      }
      if (ok && n_stages > 0) {
        issue_pv(n_stages - 1);
        // the last commit's arrival must land before the barriers are reset for the next role
        const int jl = n_stages - 1;
        if (ok && !wait_bar(p, bar_addr(sbase, kBKvEmpty + jl % kStages), (jl / kStages) & 1)) ok = false;
      }
      if (!ok) ctl->abort = 1;
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax / epilogue
    const int u = warp >> 2;
    const int r = tid & 127;
    const int nq = u ? nq1 : nq0;
    const uint32_t q = u ? sQ1 : sQ0;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int grow = grow0 + 128 * u + r;
    // rotate q_rope of this row into the document frame: angle (q_pos - offset)
    if (!wait_bar_warp(p, bar_addr(sbase, kBQFull), 0)) ctl->abort = 1;
    if (r < nq) {
      const int64_t delta = (int64_t)__ldg(p.q_pos + grow) - J.rope_offset;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        const uint32_t addr = q + 2 * kAtomQ + sw128_off(r, c);
        uint32_t w[4];
        lds128(addr, w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float sn, cs;
          rope_sincos(delta, p.rope_frac[4 * c + i], &sn, &cs);
          const float x0 = __uint_as_float(w[i] << 16), x1 = __uint_as_float(w[i] & 0xFFFF0000u);
          w[i] = pack_bf16(x0 * cs - x1 * sn, x0 * sn + x1 * cs);
        }
        sts128(addr, w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1 + u, 128);
    if (r == 0) mbar_arrive(bar_addr(sbase, kBQReady + u));
    if (nq == 0) return;

    const int qtok = J.q_tok0 + q0 + 128 * u + r;
    const float sl2 = p.scale_log2;
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_stages; ++j) {
      const int b = j & 1;
      if (!wait_bar_warp(p, bar_addr(sbase, kBSFull + 2 * u + b), (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const uint32_t scol = tmem + lane_off + kTmS + (2 * u + b) * 64;
      uint32_t v[64];
      {
        uint32_t (&v0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[0]);
        uint32_t (&v1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32]);
        tmem_ld32(scol, v0);
        tmem_ld32(scol + 32, v1);
      }
      const int kt0 = J.t0 + 64 * j;
      const bool full = kt0 >= J.k_begin && kt0 + 63 < J.k_end && kt0 + 63 <= qtok;
      float mx = -INFINITY;
      if (full) {
#pragma unroll
        for (int c = 0; c < 64; ++c) mx = fmaxf(mx, __uint_as_float(v[c]));
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int kt = kt0 + c;
          const bool okc = kt >= J.k_begin && kt < J.k_end && kt <= qtok;
          const float x = okc ? __uint_as_float(v[c]) : -INFINITY;
          v[c] = __float_as_uint(x);
          mx = fmaxf(mx, x);
        }
      }
      const float m_tile = mx * sl2;
      float alpha = 1.f;
      const bool rescale = m_tile > m_used + kRescaleThreshold;
      if (rescale) {
        alpha = ex2(m_used - m_tile);   // 0 when m_used = -inf
        m_used = m_tile;
      }
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      float sum = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float a = ex2(fmaf(__uint_as_float(v[2 * c]), sl2, -mref));
        const float bb = ex2(fmaf(__uint_as_float(v[2 * c + 1]), sl2, -mref));
        sum += a + bb;
        pk[c] = pack_bf16(a, bb);
      }
      tmem_st32(scol, pk);
      l_run = l_run * alpha + sum;
      if (j >= 1) {
        // O holds PV of stages < j: wait for the last one before touching O
        if (!wait_bar_warp(p, bar_addr(sbase, kBPvDone + u), (j - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
          const uint32_t ocol = tmem + lane_off + kTmO + 128 * u;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
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
      mbar_arrive(bar_addr(sbase, kBPFull + 2 * u + b));
    }
    if (ok && n_stages > 0 && !wait_bar_warp(p, bar_addr(sbase, kBPvDone + u), (n_stages - 1) & 1)) ok = false;
    if (!ok) { ctl->abort = 1; return; }
    tc_fence_after();
    // ---- epilogue
    const bool empty = n_stages == 0 || !(l_run > 0.f);
    const float inv_l = empty ? 0.f : 1.f / l_run;
    const bool live = r < nq;
    const int64_t orow = J.slot < 0 ? (int64_t)grow : (int64_t)J.slot * p.slot_stride_rows + grow;
    const uint32_t ocol = tmem + lane_off + kTmO + 128 * u;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t o[32];
      if (n_stages > 0) tmem_ld32(ocol + cc * 32, o);
      if (!live) continue;
      if (J.slot < 0 && p.out_bf16) {
        uint16_t* dst = static_cast<uint16_t*>(p.out) + (orow * H + J.head) * kDv + cc * 32;
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          uint4 w;
          w.x = pack_bf16(empty ? 0.f : __uint_as_float(o[i + 0]) * inv_l, empty ? 0.f : __uint_as_float(o[i + 1]) * inv_l);
          w.y = pack_bf16(empty ? 0.f : __uint_as_float(o[i + 2]) * inv_l, empty ? 0.f : __uint_as_float(o[i + 3]) * inv_l);
          w.z = pack_bf16(empty ? 0.f : __uint_as_float(o[i + 4]) * inv_l, empty ? 0.f : __uint_as_float(o[i + 5]) * inv_l);
          w.w = pack_bf16(empty ? 0.f : __uint_as_float(o[i + 6]) * inv_l, empty ? 0.f : __uint_as_float(o[i + 7]) * inv_l);
          *reinterpret_cast<uint4*>(dst + i) = w;
        }
      } else {
        float* dst = (J.slot < 0 ? static_cast<float*>(p.out) : p.part_out) + (orow * H + J.head) * kDv + cc * 32;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          float4 w;
          w.x = empty ? 0.f : __uint_as_float(o[i + 0]) * inv_l;
          w.y = empty ? 0.f : __uint_as_float(o[i + 1]) * inv_l;
          w.z = empty ? 0.f : __uint_as_float(o[i + 2]) * inv_l;
          w.w = empty ? 0.f : __uint_as_float(o[i + 3]) * inv_l;
          *reinterpret_cast<float4*>(dst + i) = w;
        }
      }
    }
    if (live) {
      const float lse = empty ? -INFINITY : m_used * 0.69314718055994531f + logf(l_run);
      (J.slot < 0 ? p.lse : p.part_lse)[orow * H + J.head] = lse;
    }
  } else if (warp < 12) {
    // warpgroup 2 waits for Q so no TMA is in flight when the role ends
    if (!wait_bar(p, bar_addr(sbase, kBQFull), 0)) ctl->abort = 1;
  }
}

// =============================================================== producer
__device__ void run_producer(const FusedParams& p, const Job& J, int job, int pi, uint32_t sbase, uint32_t tmem,
                             volatile Ctl* ctl) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_pass = (J.n_tiles + 1) >> 1;
  const int H = p.num_heads;
  const int h = J.head;
  int my_passes = 0;
  for (int pp = pi; pp < n_pass; pp += J.n_prod) ++my_passes;
  if (my_passes == 0) return;

  if (warp == 12) {
    if (lane == 0) {
      int g = 0;
      for (int n = 0; n < my_passes; ++n) {
        const int pass = pi + n * J.n_prod;
        int rows[4];
        for (int i = 0; i < 4; ++i) {
          const int lb = (J.t0 >> 6) + 4 * pass + i;
          const int tok = lb * 64;
          const bool live = tok + 63 >= J.k_begin && tok < J.k_end;
          rows[i] = live ? block_row(p, J.req, lb, true) : -kBlock;
        }
        for (int k = 0; k < kDc / 64; ++k, ++g) {
          const int s = g & 1;
          if (g >= 2 && !wait_bar(p, bar_addr(sbase, kBProdEmpty + s), ((g >> 1) - 1) & 1)) { ctl->abort = 1; return; }
          const uint32_t st = sbase + s * kPStageBytes;
          const uint32_t bar = p.kv_fp8 ? bar_addr(sbase, kBRawFull + s) : bar_addr(sbase, kBProdFull + s);
          mbar_arrive_expect_tx(bar, p.kv_fp8 ? (16384u + 32768u) : kPStageBytes);
          for (int i = 0; i < 4; ++i) {
            if (p.kv_fp8)
              tma_load_2d(sbase + kPRawBase + s * 16384 + i * 4096, &p.tm_c, 64 * k, rows[i], bar);
            else
              tma_load_2d(st + (i < 2 ? kPCA : kPCB) + (i & 1) * kAtom64, &p.tm_c, 64 * k, rows[i], bar);
          }
          for (int w = 0; w < 4; ++w) {
            const int x = (w < 2) ? (h * kDnope + 64 * w) : (H * kDnope + h * kDv + 64 * (w - 2));
            tma_load_2d(st + kPW + w * kAtom64, &p.tm_w, x, 64 * k, bar);
          }
        }
      }
    }
  } else if (warp == 13) {
    if (lane == 0) {
      int g = 0;
      for (int n = 0; n < my_passes; ++n) {
        if (n >= 1 && !wait_bar(p, bar_addr(sbase, kBAccEmpty), (n - 1) & 1)) { ctl->abort = 1; return; }
        for (int k = 0; k < kDc / 64; ++k, ++g) {
          const int s = g & 1;
          if (!wait_bar(p, bar_addr(sbase, kBProdFull + s), (g >> 1) & 1)) { ctl->abort = 1; return; }
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
    }
  } else if (warp < 8) {
    // conversion: warpgroup 0 -> tile 2*pass, warpgroup 1 -> tile 2*pass + 1
    const int wg = warp >> 2;
    const int r = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const float oscale = p.kv_fp8 ? p.kv_scale : 1.f;
    for (int n = 0; n < my_passes; ++n) {
      const int pass = pi + n * J.n_prod;
      const int t = 2 * pass + wg;
      if (!wait_bar_warp(p, bar_addr(sbase, kBAccFull), n & 1)) ctl->abort = 1;
      tc_fence_after();
      if (t < J.n_tiles) {
        const int slot = t % kRing;
        if (r == 0 && !ctl->abort) {
          if (t >= (int)kRing &&
              !wait_flag_geq(p, consumed_flag(p, job, slot), (uint32_t)consumers_needing_tile(J, t - kRing)))
            ctl->abort = 1;
          *consumed_flag(p, job, slot) = 0u;   // ordered before the release of `ready` below
        }
        named_bar_sync(1 + wg, 128);
        if (ctl->abort) return;                // every thread of the warpgroup leaves here together
        const int tok = J.t0 + 128 * t + r;
        const bool valid = tok >= J.k_begin && tok < J.k_end;
        uint16_t* dst = p.ring + ((size_t)job * kRing * 128 + (size_t)slot * 128 + r) * 256;
        const uint32_t acc = tmem + lane_off + (wg ? kTmAccB : kTmAccA);
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t a[32];
          tmem_ld32(acc + cc * 32, a);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = valid ? pack_bf16(__uint_as_float(a[2 * i]) * oscale, __uint_as_float(a[2 * i + 1]) * oscale) : 0u;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(dst + cc * 32 + 8 * i) = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
        named_bar_sync(1 + wg, 128);
        if (r == 0) {
          __threadfence();
          st_release_gpu(ready_flag(p, job, slot), (uint32_t)t + 1);
        }
      } else {
        named_bar_sync(1 + wg, 128);
        if (ctl->abort) return;
      }
      tc_fence_before();
      mbar_arrive(bar_addr(sbase, kBAccEmpty));
    }
  } else if (warp < 12) {
    // e4m3 latent staging -> bf16 MMA operand (FP8 cache only)
    if (!p.kv_fp8) return;
    const int r = tid - 256;
    int g = 0;
    for (int n = 0; n < my_passes; ++n) {
      for (int k = 0; k < kDc / 64; ++k, ++g) {
        const int s = g & 1;
        const bool okw = wait_bar_warp(p, bar_addr(sbase, kBRawFull + s), (g >> 1) & 1);
        if (!okw) ctl->abort = 1;
        const uint32_t raw = sbase + kPRawBase + s * 16384;
        const uint32_t st = sbase + s * kPStageBytes;
#pragma unroll 4
        for (int idx = r; okw && idx < 256 * 8; idx += 128) {
          const int row = idx >> 3, c = idx & 7;   // row 0..255 of the pass, chunk of 8 values
          uint32_t lo, hi;
          asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(lo), "=r"(hi) : "r"(raw + row * 64 + c * 8));
          sts128(st + (row < 128 ? kPCA : kPCB) + sw128_off(row & 127, c), e4m3x2_to_bf16x2(lo & 0xFFFFu),
                 e4m3x2_to_bf16x2(lo >> 16), e4m3x2_to_bf16x2(hi & 0xFFFFu), e4m3x2_to_bf16x2(hi >> 16));
        }
        fence_proxy_async_smem();
        named_bar_sync(3, 128);
        if (ctl->abort) return;                // together, after the barrier
        if (r == 0) mbar_arrive(bar_addr(sbase, kBProdFull + s));
      }
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
    prefetch_tensormap(&p.tm_q);
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

  for (;;) {
    if (tid == 0) ctl->role = (ctl->abort || aborted_global(p)) ? p.n_roles : (int)atomicAdd(p.queue, 1u);
    __syncthreads();
    const int role = ctl->role;
    if (role >= p.n_roles) break;
    int lo = 0, hi = p.n_pieces - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.pieces[mid].role_begin <= role) lo = mid; else hi = mid - 1;
    }
    const Piece& P = p.pieces[lo];
    const int per_job = P.n_cons + P.n_prod;
    const int local = role - P.role_begin;
    Job J;
    J.req = P.req;
    J.head = local / per_job;
    J.q_begin = P.q_begin;
    J.q_count = P.q_count;
    J.q_tok0 = P.q_tok0;
    J.k_begin = P.k_begin;
    J.k_end = P.k_end;
    J.t0 = P.k_begin & ~(kBlock - 1);
    J.n_tiles = (P.k_end - J.t0 + 127) >> 7;
    J.n_cons = P.n_cons;
    J.n_prod = P.n_prod;
    J.slot = P.slot;
    J.rope_offset = P.rope_offset;
    const int job = lo * p.num_heads + J.head;
    const int idx = local - J.head * per_job;
    const bool producer = idx < J.n_prod;
    if (tid == 32) {
      // fresh barriers for this role (every barrier is idle here)
      for (uint32_t i = 0; i < kNumBars; ++i) {
        mbar_inval(bar_addr(sbase, i));
        uint32_t cnt = 1;
        if (!producer && (i >= kBPFull && i < kBPFull + 4)) cnt = 128;
        if (producer && i == kBAccEmpty) cnt = 256;
        mbar_init(bar_addr(sbase, i), cnt);
      }
      fence_mbar_init();
    }
    __syncthreads();
    if (producer) run_producer(p, J, job, idx, sbase, tmem, ctl);
    else run_consumer(p, J, job, idx - J.n_prod, sbase, sgen, tmem, ctl);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  tc_fence_before();
  __syncthreads();
  if ((tid >> 5) == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

int fused_smem_bytes() { return (int)kSmemBytes; }

cudaError_t launch_fused(const FusedParams& p, int grid, cudaStream_t s) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(fused_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, fused_prefill_kernel, p);
  count_launch();
  return e;
}

cudaError_t fused_grid_size(int* grid) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(fused_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fused_prefill_kernel, kThreads, kSmemBytes);
  if (e != cudaSuccess) return e;
  *grid = sms * (per_sm > 0 ? per_sm : 0);
  return *grid > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

}  // namespace mla
