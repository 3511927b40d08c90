// Absorbed (latent-space) MLA attention for short extends ("DeepSeek MLA —
// Prefix Cache 与 Chunked Prefill 深度解析", section 3, the absorbed path that
// the page pairs with decode): W_UK is folded into the query and W_UV applied
// after the attention, so the keys are the cached latent rows themselves,
// shared by every head:
//   qlat_h = q_nope_h W_UK,h^T                      [512]   (qabsorb_kernel, headproj.cu)
//   s_t    = scale (qlat_h . c_t + R q_rope_h . k_rope_t)
//   o_h    = sum_t softmax(s)_t c_t                  [512]   (absorb_attn_kernel)
//   out_h  = o_h W_UV,h                              [128]   (absorb_proj_kernel, headproj.cu)
// which equals the up-projected attention exactly, up to rounding.  Per
// (query, key, head) it costs 2 (576 + 512) FLOP against 2 (192 + 128) for the
// up-projected form, but it skips the 2 * 512 * 256 FLOP per (key, head) of the
// up-projection: cheaper while a request has fewer than about 170 queries.
//
// absorb_attn_kernel: clusters of two CTAs own one work item (128 rows of
// (token, head) pairs of one piece, one key split).  O [128 x 512] fp32 fills
// a CTA's whole tensor memory, so the item is split by operation:
//  - CTA 0 ("S side") keeps Q [128 x 576] bf16 in TMEM, computes
//    S = Q [c | k_rope]^T for 64 keys per tile (M = 128, N = 64), runs the
//    online softmax and sends P (bf16) and each row's rescale factor into CTA
//    1's shared memory with st.async;
//  - CTA 1 ("O side") accumulates O += P c (two N = 256 MMAs per 16 keys)
//    and writes O / l at the end.  With each P tile comes one flag per S-side
//    warp, set when one of its rows raised its maximum (the lazy rescale, so
//    rarely after the first tiles): only then does the MMA thread wait for the
//    previous PV and hand the tile to the correction warps, which rescale
//    those rows of O in TMEM before the tile's PV.
// Each CTA loads its own 64-key stages (the S side latent + k_rope, the O
// side latent only) and frees a stage as soon as its own MMA has read it: a
// stage loaded once for both CTAs would stay busy from its load until the O side's
// PV, a chain that three stages cannot cover.  The rows are read by every row
// tile of the piece and stay in L2.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kAThreads = 256;
constexpr int kAKeys = 64;
constexpr int kAStages = 3;                                    // O side
constexpr uint32_t kAAtom = 8192;                              // [64 rows x 128 B] swizzled block
constexpr uint32_t kACStage = 8 * kAAtom;                      // O side: bf16 latent part of 64 rows
constexpr uint32_t kACBase = 0;                                // both CTAs
constexpr uint32_t kAPBase = kAStages * kACStage;              // O side: two P tiles [128 x 64] bf16
constexpr uint32_t kAPBytes = 16384;
constexpr uint32_t kAAlphaBase = kAPBase + 2 * kAPBytes;       // O side: per P tile, 128 row factors
constexpr uint32_t kALBase = kAAlphaBase + 2 * 512;            // O side: 128 final row sums
constexpr uint32_t kAFlagBase = kALBase + 512;                 // O side: per P tile, 4 rescale flags; then
                                                               // the tile handed to the correction warps
constexpr uint32_t kABarBase = kAFlagBase + 2 * 16 + 16;
enum : uint32_t {
  kBFull = 0,      // 5, both: stage landed (S side: latent + k_rope; O side: latent)
  kBEmpty = 5,     // 5, both: the CTA's MMA that reads the stage is done
  kBSFull = 10,    // 2, S side: S buffer written
  kBSFree = 12,    // 2, S side: the 4 softmax warps read the S buffer
  kBPFree = 14,    // 2, S side: PV of the P tile done (commit from the O side)
  kBQReady = 16,   // S side: the 4 softmax warps copied Q into TMEM (stages 1-2 free again)
  kBPFull = 17,    // 2, O side: P tile, row factors and flags landed
  kBCNeed = 19,    // O side: the MMA thread handed a tile (or the end) to the correction warps
  kBCDone = 20,    // O side: the 4 correction warps rescaled the tile's rows
  kBPvDone = 21,   // 2, O side: PV of the tile done
  kBLFull = 23,    // O side: the final row sums landed
  kBQFull = 24,    // S side: the tile's absorbed queries landed in stages 1-2
  kANumBars = 25
};
constexpr uint32_t kATmemSlot = kABarBase + 8 * kANumBars;
constexpr uint32_t kASmemBytes = kATmemSlot + 16 + 1024;       // + alignment of the base to 1024
static_assert(kASmemBytes <= 232448, "more than 227 KB of shared memory per CTA");

// S side, by score precision: a stage is [latent | k_rope] of 64 keys
// (bf16: 8 + 1 swizzled [64 x 128 B] blocks; E4M3 latent: 4 + 1), and the
// tile's absorbed queries are staged over stages 1-2 at the start.
template <bool kF8>
struct SSide {
  static constexpr int kCAtoms = kF8 ? 4 : 8;
  static constexpr int kStages = kF8 ? 5 : 3;
  static constexpr uint32_t kStage = (kCAtoms + 1) * kAAtom;
  static constexpr uint32_t kKr = kCAtoms * kAAtom;           // k_rope block within a stage
  static constexpr uint32_t kTx = kStage;
  static constexpr int kQBoxes = kF8 ? 4 : 8;                 // [128 rows x 128 B] boxes of qlat
  static constexpr uint32_t kQStage = kStage;                 // stage 1 on
  static constexpr uint32_t kTmRope = kF8 ? 128 : 256;        // TMEM column of the rotated q_rope
  static_assert(kStages * kStage <= kABarBase, "S-side stages overlap the barriers");
  static_assert(kQStage + kQBoxes * 16384 <= 3 * kStage, "staged queries spill past stage 2");
};

constexpr uint32_t kATmS = 320;   // S side: S buffer b at 320 + 64 b (Q in columns 0..287)
constexpr uint32_t kIdescSA = idesc_bf16(128, 64, false, false);
constexpr uint32_t kIdescS8 = idesc_e4m3(128, 64);
constexpr uint32_t kIdescPVA = idesc_bf16(128, 256, false, true);
constexpr uint32_t kTxO = kACStage;
constexpr uint32_t kTxP = 128 * (128 + 4) + 16;   // per row: 64 bf16 of P and one fp32 factor; 4 flags
constexpr float kARescale = 8.f;             // log2 units: P stays <= 256

__device__ __forceinline__ uint32_t abar(uint32_t sbase, uint32_t i) { return sbase + kABarBase + 8u * i; }

// Bounded waits (a timeout records the error; the caller then skips its work).
__device__ __forceinline__ bool await(const AbsorbParams& p, uint32_t bar, uint32_t parity) {
  if (mbar_wait(bar, parity)) return true;
  atomicOr(p.err, kErrTimeout);
  return false;
}
__device__ __forceinline__ bool await_warp(const AbsorbParams& p, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, await(p, bar, parity));
}

// Optional tracing (p.trace non-null): %globaltimer of each tile j of work
// item p.trace_item (j < 4096) in words 8 j + k:
//   [0] S side: loads issued    [1] S MMA thread: stage landed   [2] S issued
//   [3] softmax saw S           [4] P computed (before waiting for its tile buffer)
//   [5] P sent                  [6] O side: PV issued            [7] O side: P landed
__device__ __forceinline__ void tstamp(const AbsorbParams& p, bool on, int j, int k) {
  if (on && j < 4096) p.trace[8 * j + k] = global_timer_ns();
}

struct AItem {
  const AbsPiece* P;
  int row0;      // first row of the tile within the piece (rows = token * H + head)
  int k_lo, k_hi, t0, n_tiles;
  int slot;
};

__device__ AItem decode_item(const AbsorbParams& p, int item) {
  int lo = 0, hi = p.n_pieces - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.pieces[mid].item_begin <= item) lo = mid; else hi = mid - 1;
  }
  const AbsPiece& P = p.pieces[lo];
  const int local = item - P.item_begin;
  const int tile = local / P.n_splits, split = local - tile * P.n_splits;
  AItem it;
  it.P = &P;
  it.row0 = tile * 128;
  it.slot = P.slot + split;
  // the tile's last query token bounds its causal keys
  const int rows = P.q_count * p.num_heads;
  const int last_t = min(rows - 1, it.row0 + 127) / p.num_heads;
  const int k_hi_tile = min(P.k_end, P.q_tok0 + last_t + 1);
  it.k_lo = P.k_begin + split * P.split_keys;
  it.k_hi = min(it.k_lo + P.split_keys, k_hi_tile);
  it.t0 = it.k_lo & ~(kAKeys - 1);
  it.n_tiles = it.k_hi > it.k_lo ? (it.k_hi - it.t0 + kAKeys - 1) / kAKeys : 0;
  return it;
}

template <bool kF8>
__global__ void __launch_bounds__(kAThreads, 1) absorb_attn_kernel(const __grid_constant__ AbsorbParams p) {
  using SS = SSide<kF8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const AItem it = decode_item(p, blockIdx.x >> 1);
  const AbsPiece& P = *it.P;
  const int H = p.num_heads;
  const int n = it.n_tiles;
  const bool tr = p.trace != nullptr && (int)(blockIdx.x >> 1) == p.trace_item;

  if (tid == 0) {
    prefetch_tensormap(&p.tm_c4);
    if (kF8) {
      prefetch_tensormap(&p.tm_f8);
      prefetch_tensormap(&p.tm_kr8);
      prefetch_tensormap(&p.tm_qlat8);
    } else {
      prefetch_tensormap(&p.tm_kr);
      prefetch_tensormap(&p.tm_qlat);
    }
    for (uint32_t i = 0; i < kANumBars; ++i) {
      uint32_t cnt = 1;
      if ((i >= kBSFree && i < kBSFree + 2) || i == kBQReady || i == kBCDone) cnt = 4;
      mbar_init(abar(sbase, i), cnt);
    }
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(sbase + kATmemSlot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers exist before either signals the other's
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + kATmemSlot);
  const int64_t row_base = (int64_t)P.row_block0 * kBlock;   // gathered row of key token 0

  if (rank == 0) {
    // ================================================================ S side
    if (warp == 0 || warp == 2 || warp == 3) {
      // ---------------------------------------------------------- TMA: a stage's boxes leave from up to
      // three warps (warp 0: latent blocks 0-3, warp 3: bf16 blocks 4-7, warp 2: k_rope); warp 0 arms the
      // stage's barrier and loads Q
      if (lane == 0) {
        bool ok = true;
        if (warp == 0 && n > 0) {
          // the tile's absorbed queries: rows q_begin H + row0 .. +127 of qlat, staged over stages 1-2
          mbar_arrive_expect_tx(abar(sbase, kBQFull), SS::kQBoxes * 16384);
          const int qrow = P.q_begin * H + it.row0;
#pragma unroll 1
          for (int cc = 0; cc < SS::kQBoxes; ++cc)
            tma_load_2d(sbase + SS::kQStage + cc * 16384, kF8 ? &p.tm_qlat8 : &p.tm_qlat, (kF8 ? 128 : 64) * cc, qrow,
                        abar(sbase, kBQFull));
        }
        for (int j = 0; j < n && ok; ++j) {
          const int s = j % SS::kStages;
          if (j >= SS::kStages && !await(p, abar(sbase, kBEmpty + s), ((j / SS::kStages) - 1) & 1)) { ok = false; break; }
          if (j == 1 && !await(p, abar(sbase, kBQReady), 0)) { ok = false; break; }   // Q copied out of stages 1-2
          const int row = (int)(row_base + it.t0 + kAKeys * j);
          const uint32_t full = abar(sbase, kBFull + s), st = sbase + s * SS::kStage;
          if (warp == 0) {
            mbar_arrive_expect_tx(full, SS::kTx);
            tstamp(p, tr, j, 0);
            tma_load_3d(st, kF8 ? &p.tm_f8 : &p.tm_c4, 0, row, 0, full);
          } else if (warp == 3) {
            if (!kF8) tma_load_3d(st + 4 * kAAtom, &p.tm_c4, 0, row, 4, full);
          } else if (kF8) {
            tma_load_2d(st + SS::kKr, &p.tm_kr8, kDc / 2, row, full);   // k_rope at byte 512 of a 640-byte row
          } else {
            tma_load_2d(st + SS::kKr, &p.tm_kr, kDc, row, full);
          }
        }
        // the last commits land on this CTA's barriers before it exits
        if (warp == 0)
          for (int j = max(0, n - SS::kStages); j < n && ok; ++j)
            if (!await(p, abar(sbase, kBEmpty + j % SS::kStages), (j / SS::kStages) & 1)) ok = false;
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- S = Q [c | k_rope]^T
      if (lane == 0 && n > 0) {
        bool ok = await(p, abar(sbase, kBQReady), 0);
        for (int j = 0; j < n && ok; ++j) {
          const int s = j % SS::kStages, b = j & 1;
          if (!await(p, abar(sbase, kBFull + s), (j / SS::kStages) & 1)) { ok = false; break; }
          tstamp(p, tr, j, 1);
          if (j >= 2 && !await(p, abar(sbase, kBSFree + b), ((j >> 1) - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint32_t c = sbase + s * SS::kStage, kr = c + SS::kKr;
          const uint32_t d = tmem + kATmS + 64 * b;
          // latent part: K = 16 (bf16) or 32 (E4M3) per MMA, four k-steps per 128-byte block
          constexpr int kLat = kF8 ? 16 : 32;
#pragma unroll
          for (int kk = 0; kk < kLat; ++kk) {
            const uint64_t bdesc = sdesc_sw128(c + (kk >> 2) * kAAtom + (kk & 3) * 32, 16, 1024);
            if (kF8) mma_e4m3_ts(d, tmem + kk * 8, bdesc, kIdescS8, kk > 0 ? 1u : 0u);
            else mma_bf16_ts(d, tmem + kk * 8, bdesc, kIdescSA, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(d, tmem + SS::kTmRope + kk * 8, sdesc_sw128(kr + kk * 32, 16, 1024), kIdescSA, 1u);
          mma_commit(abar(sbase, kBSFull + b));
          mma_commit(abar(sbase, kBEmpty + s));
          tstamp(p, tr, j, 2);
        }
      }
    } else if (warp >= 4) {
      // ---------------------------------------------------------- Q -> TMEM, then softmax
      const int r = tid - 128;
      const int prow = it.row0 + r;
      const bool live = prow < P.q_count * H;
      const int tl = live ? prow / H : 0, h = live ? prow - (prow / H) * H : 0;
      const int64_t grow = (int64_t)P.q_begin + tl;
      const int64_t orow = grow * H + h;
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      // E4M3 scores: the latent part of S counts in units of qscale[row] * kv_scale, so q_rope is divided
      // by it (the two parts share one accumulator) and the softmax multiplies it back
      const float qs = kF8 ? (live ? __ldg(p.qscale + orow) : 1.f) * p.kv_scale : 1.f;
      if (n > 0) {
        // rotated q_rope from global memory (its loads overlap the qlat TMA)
        const uint4* qr = reinterpret_cast<const uint4*>(p.q + orow * kDqk + kDnope);
        const int64_t delta = live ? (int64_t)__ldg(p.q_pos + grow) - P.rope_offset : 0;
        const float rq = 1.f / qs;
        uint4 qv[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) qv[c] = live ? __ldg(qr + c) : make_uint4(0, 0, 0, 0);
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t w4[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // (measured: the SFU form is 2% faster here with bf16 scores, the
            // accurate one 16% faster with E4M3 scores)
            float sn, cs;
            if constexpr (kF8) rope_sincos(delta, p.rope_frac[4 * c + i], &sn, &cs);
            else rope_sincos_sfu(delta, p.rope_frac[4 * c + i], &sn, &cs);
            const float x0 = __uint_as_float(w4[i] << 16), x1 = __uint_as_float(w4[i] & 0xFFFF0000u);
            w[4 * c + i] = pack_bf16((x0 * cs - x1 * sn) * rq, (x0 * sn + x1 * cs) * rq);
          }
        }
        tmem_st32(tmem + lane_off + SS::kTmRope, w);
        // qlat: shared memory (TMA, 128-byte swizzled [128 x 128 B] blocks) -> TMEM columns from 0
        const bool qok = await_warp(p, abar(sbase, kBQFull), 0);
#pragma unroll 1
        for (int cc = 0; cc < SS::kQBoxes; ++cc) {
          uint32_t u[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t v4[4];
            if (qok) lds128(sbase + SS::kQStage + cc * 16384 + sw128_off((uint32_t)r, (uint32_t)c), v4);
            else v4[0] = v4[1] = v4[2] = v4[3] = 0u;
            u[4 * c] = v4[0]; u[4 * c + 1] = v4[1]; u[4 * c + 2] = v4[2]; u[4 * c + 3] = v4[3];
          }
          tmem_st32(tmem + lane_off + 32 * cc, u);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(abar(sbase, kBQReady));
      }
      const int qk = live ? P.q_tok0 + tl : -1;   // last visible key token of the row
      const float sl2 = p.scale_log2 * qs;
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      const uint32_t peer_p = mapa_shared(sbase + kAPBase, 1u);
      const uint32_t peer_alpha = mapa_shared(sbase + kAAlphaBase, 1u);
      for (int j = 0; j < n; ++j) {
        const int b = j & 1;
        uint32_t v[64];
        float mx = -INFINITY;
        if (ok && !await_warp(p, abar(sbase, kBSFull + b), (j >> 1) & 1)) ok = false;
        tc_fence_after();
        if (ok) mx = tmem_ld64_max(tmem + lane_off + kATmS + 64 * b, v);   // the row maximum comes with the load
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(abar(sbase, kBSFree + b));
        if (!ok) break;
        if (tid == 128) tstamp(p, tr, j, 3);
        const int kt0 = it.t0 + kAKeys * j;
        if (!(kt0 >= it.k_lo && kt0 + kAKeys - 1 < it.k_hi && kt0 + kAKeys - 1 <= qk)) {
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int kt = kt0 + c;
            const bool vis = kt >= it.k_lo && kt < it.k_hi && kt <= qk;
            const float x = vis ? __uint_as_float(v[c]) : -INFINITY;
            v[c] = __float_as_uint(x);
            m8[c & 7] = fmaxf(m8[c & 7], x);
          }
          mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        }
        const float m_tile = mx * sl2;
        float alpha = 1.f;
        if (m_tile > m_used + kARescale) {
          alpha = ex2(m_used - m_tile);   // 0 when m_used = -inf
          m_used = m_tile;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t sc2 = f2pack(sl2, sl2), nm2 = f2pack(-mref, -mref);
        uint64_t s4[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x0, x1;
          f2unpack(ffma2(f2pack(__uint_as_float(v[2 * c]), __uint_as_float(v[2 * c + 1])), sc2, nm2), x0, x1);
          const float a = ex2(x0), bb = ex2(x1);
          s4[c & 3] = fadd2(s4[c & 3], f2pack(a, bb));
          pk[c] = pack_bf16(a, bb);
        }
        float s8[4];
        f2unpack(fadd2(s4[0], s4[1]), s8[0], s8[1]);
        f2unpack(fadd2(s4[2], s4[3]), s8[2], s8[3]);
        l = l * alpha + ((s8[0] + s8[2]) + (s8[1] + s8[3]));
        if (tid == 128) tstamp(p, tr, j, 4);
        // P tile b is free once the PV of tile j - 2 is done
        if (j >= 2 && !await_warp(p, abar(sbase, kBPFree + b), ((j - 2) >> 1) & 1)) { ok = false; break; }
        const uint32_t cbar = mapa_shared(abar(sbase, kBPFull + b), 1u);
        const uint32_t prow_addr = peer_p + b * kAPBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_async_v4(prow_addr + sw128_off((uint32_t)r, (uint32_t)c), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                      pk[4 * c + 3], cbar);
        st_async_b32(peer_alpha + b * 512 + 4 * r, __float_as_uint(alpha), cbar);
        const uint32_t any_rescale = __any_sync(0xffffffffu, alpha != 1.f) ? 1u : 0u;
        if (lane == 0) st_async_b32(mapa_shared(sbase + kAFlagBase + 16 * b + 4 * (warp & 3), 1u), any_rescale, cbar);
        if (tid == 128) tstamp(p, tr, j, 5);
      }
      // final row sums to the O side; lse of the item
      st_async_b32(mapa_shared(sbase + kALBase + 4 * r, 1u), __float_as_uint(ok ? l : 0.f),
                   mapa_shared(abar(sbase, kBLFull), 1u));
      if (live) {
        const float lse = (ok && l > 0.f) ? (m_used + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        p.lat_lse[(int64_t)it.slot * p.slot_stride_rows + orow] = lse;
      }
      // the last two PV commits land on this CTA's barriers before it exits
      for (int j = max(0, n - 2); j < n && ok; ++j)
        if (!await_warp(p, abar(sbase, kBPFree + (j & 1)), (j >> 1) & 1)) ok = false;
    }
  } else {
    // ================================================================ O side
    if (warp == 0 || warp == 3) {
      // ---------------------------------------------------------- TMA (latent rows; blocks 0-3 from warp 0,
      // which arms the barrier, blocks 4-7 from warp 3)
      if (lane == 0) {
        bool ok = true;
        for (int j = 0; j < n && ok; ++j) {
          const int s = j % kAStages;
          if (j >= kAStages && !await(p, abar(sbase, kBEmpty + s), ((j / kAStages) - 1) & 1)) { ok = false; break; }
          const int row = (int)(row_base + it.t0 + kAKeys * j);
          if (warp == 0) {
            mbar_arrive_expect_tx(abar(sbase, kBFull + s), kTxO);
            tma_load_3d(sbase + kACBase + s * kACStage, &p.tm_c4, 0, row, 0, abar(sbase, kBFull + s));
          } else {
            tma_load_3d(sbase + kACBase + s * kACStage + 4 * kAAtom, &p.tm_c4, 0, row, 4, abar(sbase, kBFull + s));
          }
        }
        if (warp == 0)
          for (int j = max(0, n - kAStages); j < n && ok; ++j)
            if (!await(p, abar(sbase, kBEmpty + j % kAStages), (j / kAStages) & 1)) ok = false;
      }
    } else if (warp == 1) {
      // ---------------------------------------------------------- O += P c
      if (lane == 0) {
        for (int b = 0; b < min(n, 2); ++b) mbar_arrive_expect_tx(abar(sbase, kBPFull + b), kTxP);
        mbar_arrive_expect_tx(abar(sbase, kBLFull), 512);
        bool ok = true;
        volatile int* hand = reinterpret_cast<volatile int*>(sgen + kAFlagBase + 32);
        int events = 0;
        for (int j = 0; j < n && ok; ++j) {
          const int s = j % kAStages, b = j & 1;
          if (!await(p, abar(sbase, kBFull + s), (j / kAStages) & 1)) { ok = false; break; }
          if (!await(p, abar(sbase, kBPFull + b), (j >> 1) & 1)) { ok = false; break; }
          tstamp(p, tr, j, 7);
          if (j > 0) {
            uint32_t f[4];
            lds128(sbase + kAFlagBase + 16 * b, f);
            if (f[0] | f[1] | f[2] | f[3]) {
              // O must hold PV of every earlier tile before its rows are rescaled
              if (!await(p, abar(sbase, kBPvDone + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) { ok = false; break; }
              *hand = b;
              mbar_arrive(abar(sbase, kBCNeed));
              if (!await(p, abar(sbase, kBCDone), events & 1)) { ok = false; break; }
              ++events;
            }
          }
          fence_proxy_async_smem();   // P was written by the peer's stores, the MMA reads it as an operand
          tc_fence_after();
          const uint32_t c = sbase + kACBase + s * kACStage, pt = sbase + kAPBase + b * kAPBytes;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = sdesc_sw128(pt + kk * 32, 16, 1024);
#pragma unroll
            for (int half = 0; half < 2; ++half)
              mma_bf16(tmem + 256 * half, adesc, sdesc_sw128(c + kk * 2048 + half * 4 * kAAtom, kAAtom, 1024),
                       kIdescPVA, (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(abar(sbase, kBPvDone + b));
          mma_commit(abar(sbase, kBEmpty + s));
          tstamp(p, tr, j, 6);
          mma_commit_mc(abar(sbase, kBPFree + b), 1);
          if (j + 2 < n) mbar_arrive_expect_tx(abar(sbase, kBPFull + b), kTxP);
        }
        *hand = -1;   // no more tiles: the correction warps go on to the epilogue
        mbar_arrive(abar(sbase, kBCNeed));
      }
    } else if (warp >= 4) {
      // ---------------------------------------------------------- rescale O rows; epilogue
      const int r = tid - 128;
      const int prow = it.row0 + r;
      const bool live = prow < P.q_count * H;
      const int tl = live ? prow / H : 0, h = live ? prow - (prow / H) * H : 0;
      const int64_t orow = ((int64_t)P.q_begin + tl) * H + h;
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      const float* alpha_s = reinterpret_cast<const float*>(sgen + kAAlphaBase);
      const volatile int* hand = reinterpret_cast<const volatile int*>(sgen + kAFlagBase + 32);
      bool ok = true;
      for (int ev = 0;; ++ev) {
        if (!await_warp(p, abar(sbase, kBCNeed), ev & 1)) { ok = false; break; }
        const int b = *hand;
        if (b < 0) break;
        tc_fence_after();
        const float a = alpha_s[b * 128 + r];
        if (__any_sync(0xffffffffu, a != 1.f)) {
#pragma unroll 1
          for (int cc = 0; cc < 16; ++cc) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_off + 32 * cc, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
            tmem_st32(tmem + lane_off + 32 * cc, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(abar(sbase, kBCDone));
      }
      if (ok && n > 0 && !await_warp(p, abar(sbase, kBPvDone + ((n - 1) & 1)), ((n - 1) >> 1) & 1)) ok = false;
      if (ok && !await_warp(p, abar(sbase, kBLFull), 0)) ok = false;
      tc_fence_after();
      const float lsum = ok ? reinterpret_cast<const float*>(sgen + kALBase)[r] : 0.f;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      float4* dst = reinterpret_cast<float4*>(p.lat_out + ((int64_t)it.slot * p.slot_stride_rows + orow) * kDc);
#pragma unroll 1
      for (int cc = 0; cc < 16; ++cc) {
        uint32_t o[32];
        if (ok && n > 0) tmem_ld32(tmem + lane_off + 32 * cc, o);
        else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        if (live) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[8 * cc + i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                          __uint_as_float(o[4 * i + 2]) * inv, __uint_as_float(o[4 * i + 3]) * inv);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // no peer operation targets this CTA's shared memory any more
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

static cudaError_t configure_absorb(int dev) {
  static int configured_device = -1;
  if (configured_device == dev) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(absorb_attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kASmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(absorb_attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmemBytes);
  if (e == cudaSuccess) configured_device = dev;
  return e;
}

cudaError_t launch_absorb_attn(const AbsorbParams& p, cudaStream_t s) {
  if (p.n_items == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = configure_absorb(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(2 * p.n_items);
  cfg.blockDim = dim3(kAThreads);
  cfg.dynamicSmemBytes = kASmemBytes;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = p.fp8_scores ? cudaLaunchKernelEx(&cfg, absorb_attn_kernel<true>, p)
                   : cudaLaunchKernelEx(&cfg, absorb_attn_kernel<false>, p);
  count_launch();
  return e;
}

}  // namespace mla
