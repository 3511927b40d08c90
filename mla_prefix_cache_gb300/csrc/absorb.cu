// Absorbed (latent-space) MLA attention for short extends ("DeepSeek MLA —
// Prefix Cache 与 Chunked Prefill 深度解析", section 3, the absorbed path that
// the page pairs with decode): W_UK is folded into the query and W_UV applied
// after the attention, so the keys are the cached latent rows [c | k_rope]
// themselves, shared by every head:
//   qlat_h = q_nope_h W_UK,h^T                      [512]   (qabsorb_kernel, headproj.cu)
//   s_t    = scale (qlat_h . c_t + R q_rope_h . k_rope_t)
//   o_h    = sum_t softmax(s)_t c_t                  [512]   (absorb_attn_kernel, here)
//   out_h  = o_h W_UV,h                              [128]   (absorb_proj_kernel, headproj.cu)
// which equals the up-projected attention exactly, up to rounding.  Per
// (query, key, head) it costs 2 (576 + 512) FLOP against 2 (192 + 128) for the
// up-projected form, but it skips the 2 * 512 * 256 FLOP per (key, head) of the
// up-projection: cheaper while a request has fewer than about 150 queries.
//
// A work item is 256 rows of (token, head) pairs of one piece and one key
// split.  Clusters of four CTAs own an item, as two CTA pairs whose tensor-core
// work is issued by the pair's first CTA as M = 256 MMAs (rows 0..127 of A
// and of the accumulator in the first CTA, rows 128..255 in its peer, each
// CTA holding half of B):
//  - S pair (ranks 0, 1): Q = [qlat | rotated q_rope] of its 128 rows
//    (qlat in TMEM, q_rope in shared memory); per 128-key tile
//    S = Q [c | k_rope]^T with N = 128, rank r loading keys 64 r .. 64 r + 63
//    of the tile (bf16 rows, or the FP8 rows as stored with E4M3 scores on
//    kind::f8f6f4); the online softmax of each CTA's rows writes P (bf16), the
//    rows' rescale factors and one "rescaled" flag per warp into one of two
//    staging buffers (alternate tiles), which one thread copies in bulk into
//    the shared memory of the O CTA that holds the same rows (2048 16-byte
//    stores into the other SM took a quarter of the time with E4M3 scores).
//  - O pair (ranks 2, 3): O [256 x 512] += P c with N = 256 per MMA, rank
//    2 + r loading latent columns 128 r .. 128 r + 127 of each 256-column half
//    of the keys; rows whose maximum rose are rescaled in TMEM by the CTA's
//    correction warps before the tile's PV; at the end O / l leaves as fp32
//    latent state.
// Each pair's MMAs are issued by a whole warp through one elected lane, and
// the per-tile signals between the CTAs are relaxed arrives (each says why
// no release is needed there).
// Each key is read from L2 once per 256 rows by the S pair and once by the O
// pair, half of it by each CTA.
#include "absorb.h"
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads2 = 256;   // warp 0: loads; 1: MMA; 2: TMEM; 3 (O): P landed; 4-7: softmax (S) or rescale and epilogue (O)
constexpr uint32_t kBlk = 8192;            // [64 rows x 128 B] swizzled block
constexpr uint32_t kBlk128 = 16384;        // [128 rows x 128 B] swizzled block

// S side, by score precision: the rotated q_rope, two P staging buffers (a P
// tile, its row factors and flags, in the O side's layout: one is filled while
// the other's copy into the O CTA is in flight), then the ring.  A stage is
// this CTA's 64 keys of a tile times kSBlocks blocks of 128 B of the row
// ([c | k_rope]: 9 blocks of bf16 or 5 of the FP8 row as stored).  The item's
// qlat is staged from the first P staging buffer on, over the first ring
// stages, before it is copied into TMEM.
template <bool kF8>
struct S2 {
  static constexpr int kSBlocks = kF8 ? 5 : 3;                // blocks per stage
  static constexpr int kStagesPerTile = kF8 ? 1 : 3;
  static constexpr int kLatBlocks = kF8 ? 4 : 8;              // latent blocks of a row (the last block is k_rope)
  static constexpr int kRing = kF8 ? 3 : 5;
  static constexpr uint32_t kStage = kSBlocks * kBlk;
  static constexpr uint32_t kQR = 0;                          // rotated q_rope [128 x 128 B]
  static constexpr uint32_t kPS = kBlk128;                    // P staging i at kPS + i kPSBuf: P [2 x 16 KB],
  static constexpr uint32_t kPSAlpha = 2 * kBlk128;           //   factors [512 B] and flags at these offsets
  static constexpr uint32_t kPSFlags = kPSAlpha + 512;
  static constexpr uint32_t kPSBuf = (kPSFlags + 16 + 1023) & ~1023u;
  static constexpr uint32_t kStage0 = kPS + 2 * kPSBuf;
  static constexpr int kQBoxes = kF8 ? 4 : 8;                 // [128 rows x 128 B] boxes of qlat
  static constexpr uint32_t kQBase = kPS;
  static constexpr uint32_t kQEnd = kQBase + kQBoxes * kBlk128;
  static constexpr uint32_t kEnd = kStage0 + kRing * kStage;
  static_assert(kQEnd <= kEnd, "staged queries spill past the ring");
  // ring stage s holds part of the staged queries until they are copied out
  static __device__ __forceinline__ bool holds_q(int s) { return kStage0 + s * kStage < kQEnd; }
};

// O side: two P tiles [128 rows x 128 keys] bf16, their row factors, the
// final row sums, per P tile four rescale flags (then the tile handed to the
// correction warps), then kORing stages of 64 keys x this CTA's 256 latent
// columns (blocks 2 r, 2 r + 1 of each half).
constexpr uint32_t kOP = 0;
constexpr uint32_t kOPBytes = 2 * kBlk128;
constexpr uint32_t kOAlpha = 2 * kOPBytes;
constexpr uint32_t kOL = kOAlpha + 2 * 512;
constexpr uint32_t kOFlags = kOL + 512;
constexpr uint32_t kOC = (kOFlags + 64 + 1023) & ~1023u;
constexpr int kORing = 4;
static_assert((kORing & (kORing - 1)) == 0, "the O ring's slot is a mask of the stage use");
constexpr uint32_t kOStage = 4 * kBlk;
constexpr uint32_t kOEnd = kOC + kORing * kOStage;
constexpr uint32_t kTxP2 = 128 * (256 + 4) + 16;   // per row: 128 bf16 of P and one factor; 4 flags

enum : uint32_t {
  // S side
  kSF = 0,     // 8: stage landed in both S CTAs (first CTA's count)
  kSE = 8,     // 8: the stage's MMAs are done (both S CTAs)
  kSSF = 16,   // 2: S buffer written (both S CTAs)
  kSSR = 18,   // 2: the 8 softmax warps of the pair read the S buffer (first CTA, count 8)
  kQF = 20,    // this CTA's qlat landed
  kQL = 21,    // this CTA's 4 softmax warps copied it out (count 4)
  kQR = 22,    // Q of both S CTAs in place (first CTA, count 8)
  kPFR = 23,   // 2: PV of the P tile done (both S CTAs, from the O pair)
  kSTF = 42,   // 2: a P staging buffer's last copy landed in the O CTA (S CTA, from its O CTA)
  // O side
  kCF = 25,    // 4: stage landed in both O CTAs (first CTA's count)
  kCE = 29,    // 4: the stage's MMAs are done (both O CTAs)
  kPF = 33,    // 2: P tile, factors and flags landed in this CTA
  kPR = 35,    // 2: P tile ready (and rows rescaled) in both O CTAs (first CTA, count 2)
  kPVD = 37,   // 2: PV of the tile done (both O CTAs)
  kCN = 39,    // this CTA's control thread handed a tile (or the end) to its correction warps
  kCD = 40,    // the 4 correction warps rescaled their rows (count 4)
  kLF = 41,    // the final row sums landed
  kNBars2 = 44
};

template <bool kF8>
struct L2 {
  static constexpr uint32_t kBars = (S2<kF8>::kEnd > kOEnd ? S2<kF8>::kEnd : kOEnd);
  static constexpr uint32_t kSlot = kBars + 8 * kNBars2;
  static constexpr uint32_t kSmem = kSlot + 16 + 1024;
  static_assert(kSmem <= 232448, "more than 227 KB of shared memory per CTA");
};

constexpr uint32_t kIdS2 = idesc_bf16(256, 128, false, false);
constexpr uint32_t kIdS2f8 = idesc_e4m3(256, 128);
constexpr uint32_t kIdPV2 = idesc_bf16(256, 256, false, true);
constexpr float kRescale2 = 8.f;   // log2 units: P stays <= 256
constexpr uint16_t kMaskS = 0x3, kMaskO = 0xC;

__device__ __forceinline__ uint32_t bar2(uint32_t sbase, uint32_t off_bars, uint32_t i) {
  return sbase + off_bars + 8u * i;
}
__device__ __forceinline__ bool await2(const AbsorbParams& p, uint32_t bar, uint32_t parity) {
  if (mbar_wait(bar, parity)) return true;
  atomicOr(p.err, kErrTimeout);
  return false;
}
__device__ __forceinline__ bool await2_warp(const AbsorbParams& p, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, await2(p, bar, parity));
}

// Row of the paged cache that holds the 64 keys from key token kt (a multiple
// of 64) of the piece's request, for a load that reads the cache in place.
// Keys past the request's last block, and a bad block id (reported), give a
// row before the map, which a TMA load reads as zeros.
__device__ __forceinline__ int cache_row(const AbsorbParams& p, const AbsPiece& P, int kt) {
  const int lb = kt >> 6;
  if (lb > P.last_lb) return -kBlock;
  const int id = lb < p.max_blocks ? __ldg(p.block_table + (int64_t)P.req * p.max_blocks + lb) : -1;
  if (id < 0 || id >= p.num_blocks) {
    atomicOr(p.err, kErrBadBlock);
    return -kBlock;
  }
  return id * kBlock;
}

struct AItem {
  const AbsPiece* P;
  int row0;      // first row of the item within the piece (rows = token * H + head)
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
  it.row0 = tile * 256;
  it.slot = P.slot + split;
  // the item's last query token bounds its causal keys
  const int rows = P.q_count * p.num_heads;
  const int last_t = min(rows - 1, it.row0 + 255) / p.num_heads;
  const int last_tok = p.q_tok ? __ldg(p.q_tok + P.q_begin + last_t) : P.q_tok0 + last_t;   // rows in token order
  const int k_hi_item = min(P.k_end, last_tok + 1);
  it.k_lo = P.k_begin + split * P.split_keys;
  it.k_hi = min(it.k_lo + P.split_keys, k_hi_item);
  it.t0 = it.k_lo & ~127;
  it.n_tiles = it.k_hi > it.k_lo ? (it.k_hi - it.t0 + 127) / 128 : 0;
  return it;
}

template <bool kF8>
__global__ void __launch_bounds__(kThreads2, 1) absorb_attn_kernel(const __grid_constant__ AbsorbParams p) {
  using SS = S2<kF8>;
  using LL = L2<kF8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const bool s_side = rank < 2;
  const uint32_t half = rank & 1;          // row half of the item (and key or column half of B)
  const bool first = half == 0;            // issues the pair's MMAs
  const AItem it = decode_item(p, blockIdx.x >> 2);
  const AbsPiece& P = *it.P;
  const int H = p.num_heads;
  const int n = it.n_tiles;
  const uint32_t B = LL::kBars;
  auto bar = [&](uint32_t i) { return bar2(sbase, B, i); };

  if (tid == 0) {
    if (s_side) {
      prefetch_tensormap(kF8 ? &p.tm_f5 : (p.s_in_place ? &p.tm_k3 : &p.tm_c3));
      prefetch_tensormap(kF8 ? &p.tm_qlat8 : &p.tm_qlat);
    } else {
      prefetch_tensormap(&p.tm_c2);
      if (p.o_in_place) prefetch_tensormap(&p.tm_k2);
    }
    for (uint32_t i = 0; i < kNBars2; ++i) {
      uint32_t cnt = 1;
      if (i == kSSR || i == kSSR + 1 || i == kQR) cnt = 8;
      else if (i == kQL || i == kCD) cnt = 4;
      else if (i == kPR || i == kPR + 1) cnt = 2;
      mbar_init(bar(i), cnt);
    }
    fence_mbar_init();
  }
  cluster_sync_all();   // every CTA's barriers exist before any is signalled; the pairs run before TMEM is allocated
  if (warp == 2) {
    tmem_alloc2(sbase + LL::kSlot, 512);
    tmem_relinquish2();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sgen + LL::kSlot);
  const int64_t row_base = (int64_t)P.row_block0 * kBlock;   // gathered row of key token 0 (rows read in place: the copy of the last block)

  if (s_side) {
    // ================================================================ S pair
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- loads: qlat, then this CTA's keys of each tile
      bool ok = true;
      const int U = n * SS::kStagesPerTile;
      if (n > 0) {
        mbar_arrive_expect_tx(bar(kQF), SS::kQBoxes * kBlk128);
        const int qrow = P.q_begin * H + it.row0 + 128 * (int)half;
#pragma unroll 1
        for (int cc = 0; cc < SS::kQBoxes; ++cc)
          tma_load_2d(sbase + SS::kQBase + cc * kBlk128, kF8 ? &p.tm_qlat8 : &p.tm_qlat, (kF8 ? 128 : 64) * cc, qrow,
                      bar(kQF));
      }
      const uint32_t full0 = mapa_shared(bar(kSF), 0u);
      bool q_copied = false;
      for (int u = 0; u < U && ok; ++u) {
        const int s = u % SS::kRing, j = u / SS::kStagesPerTile, m = u - j * SS::kStagesPerTile;
        // this CTA's 64 keys of the tile (looked up before the slot wait, which hides the table load): masked
        // past the item's keys, so read in place whatever they hold
        const int kt = it.t0 + 128 * j + 64 * (int)half;
        const int row = (kF8 || p.s_in_place) ? cache_row(p, P, kt) : (int)(row_base + kt);
        if (u >= SS::kRing && !await2(p, bar(kSE + s), ((u / SS::kRing) - 1) & 1)) { ok = false; break; }
        if (SS::holds_q(s) && !q_copied) {   // the staged queries are out of the stages before keys overwrite them
          if (!await2(p, bar(kQL), 0)) { ok = false; break; }
          q_copied = true;
        }
        if (first) mbar_arrive_expect_tx(bar(kSF + s), 2 * SS::kStage);
        if (kF8)
          tma_load_3d_pair(sbase + SS::kStage0 + s * SS::kStage, &p.tm_f5, 0, row, 0, full0 + 8u * s);
        else
          tma_load_3d_pair(sbase + SS::kStage0 + s * SS::kStage, p.s_in_place ? &p.tm_k3 : &p.tm_c3, 0, row, 3 * m,
                           full0 + 8u * s);
      }
      // the last commits land on this CTA's barriers before it exits
      for (int u = max(0, U - SS::kRing); u < U && ok; ++u)
        if (!await2(p, bar(kSE + u % SS::kRing), (u / SS::kRing) & 1)) ok = false;
    } else if (warp == 1 && first && n > 0) {
      // ---------------------------------------------------------- S = Q [c | k_rope]^T, N = 128 keys
      // (the whole warp runs the loop; one elected lane issues each MMA)
      bool ok = await2_warp(p, bar(kQR), 0);
      const uint64_t qd = sdesc_sw128(sbase + SS::kQR, 16, 1024);        // rotated q_rope
      const uint64_t sd0 = sdesc_sw128(sbase + SS::kStage0, 16, 1024);   // ring stage 0
      const uint32_t sf0 = bar(kSF), se0 = bar(kSE);
      int s = 0;          // ring slot of the next stage
      uint32_t ph = 0;    // and the parity of its fill
      for (int j = 0; j < n && ok; ++j) {
        const int b = j & 1;
        if (j >= 2 && !await2_warp(p, bar(kSSR + b), ((j >> 1) - 1) & 1)) { ok = false; break; }
        const uint32_t d = tmem + 256 + 128 * b;
#pragma unroll
        for (int m = 0; m < SS::kStagesPerTile; ++m) {
          if (!await2_warp(p, sf0 + 8u * s, ph)) { ok = false; break; }
          tc_fence_after();
          const uint64_t sd = sdesc_add(sd0, s * SS::kStage);
          const uint32_t ta = tmem + 32 * SS::kSBlocks * m;   // qlat columns of the stage's latent blocks
#pragma unroll
          for (int kb = 0; kb < SS::kSBlocks; ++kb) {
            if (m * SS::kSBlocks + kb < SS::kLatBlocks) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sdesc_add(sd, kb * kBlk + kk * 32);
                const uint32_t acc = (m | kb | kk) ? 1u : 0u;
                if (kF8) mma2_ts_e4m3_elect(d, ta + 32 * kb + 8 * kk, bd, kIdS2f8, acc);
                else mma2_ts_elect(d, ta + 32 * kb + 8 * kk, bd, kIdS2, acc);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma2_ss_elect(d, sdesc_add(qd, kk * 32), sdesc_add(sd, kb * kBlk + kk * 32), kIdS2, 1u);
            }
          }
          mma2_commit_mc_elect(se0 + 8u * s, kMaskS);
          if (++s == SS::kRing) { s = 0; ph ^= 1u; }
        }
        if (ok) mma2_commit_mc_elect(bar(kSSF + b), kMaskS);
      }
    } else if (warp >= 4) {
      // ---------------------------------------------------------- Q -> TMEM and shared memory, then softmax
      const int r = tid - 128;
      const int prow = it.row0 + 128 * (int)half + r;
      const bool live = prow < P.q_count * H;
      const int tl = live ? prow / H : 0, h = live ? prow - (prow / H) * H : 0;
      const int64_t grow = (int64_t)P.q_begin + tl;
      const int64_t orow = grow * H + h;
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      // E4M3 scores: the latent part of S counts in units of qscale[row] * kv_scale, so q_rope is divided
      // by it (the two parts share one accumulator) and the softmax multiplies it back
      const float qs = kF8 ? (live ? __ldg(p.qscale + orow) : 1.f) * p.kv_scale : 1.f;
      const uint32_t orank = 2u + half;   // the O CTA holding the same rows
      if (n > 0) {
        // rotated q_rope from global memory, into shared memory as a K-major swizzled block
        const uint4* qr = reinterpret_cast<const uint4*>(p.q + orow * kDqk + kDnope);
        const int64_t delta = live ? (int64_t)__ldg(p.q_pos + grow) - P.rope_offset : 0;
        const float rq = 1.f / qs;
        uint4 qv[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) qv[c] = live ? __ldg(qr + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t w4[4] = {qv[c].x, qv[c].y, qv[c].z, qv[c].w};
          uint32_t o4[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float sn, cs;
            if constexpr (kF8) rope_sincos(delta, p.rope_frac[4 * c + i], &sn, &cs);
            else rope_sincos_sfu(delta, p.rope_frac[4 * c + i], &sn, &cs);
            const float x0 = __uint_as_float(w4[i] << 16), x1 = __uint_as_float(w4[i] & 0xFFFF0000u);
            o4[i] = pack_bf16((x0 * cs - x1 * sn) * rq, (x0 * sn + x1 * cs) * rq);
          }
          sts128(sbase + SS::kQR + sw128_off((uint32_t)r, (uint32_t)c), o4[0], o4[1], o4[2], o4[3]);
        }
        // qlat: shared memory (TMA, swizzled [128 x 128 B] blocks) -> TMEM columns from 0
        const bool qok = await2_warp(p, bar(kQF), 0);
#pragma unroll 1
        for (int cc = 0; cc < SS::kQBoxes; ++cc) {
          uint32_t u[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t v4[4];
            if (qok) lds128(sbase + SS::kQBase + cc * kBlk128 + sw128_off((uint32_t)r, (uint32_t)c), v4);
            else v4[0] = v4[1] = v4[2] = v4[3] = 0u;
            u[4 * c] = v4[0]; u[4 * c + 1] = v4[1]; u[4 * c + 2] = v4[2]; u[4 * c + 3] = v4[3];
          }
          tmem_st32(tmem + lane_off + 32 * cc, u);
        }
        tmem_wait_st();
        fence_proxy_async_smem();   // q_rope, written here, is an MMA operand
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(kQL));
          mbar_arrive_cluster(mapa_shared(bar(kQR), 0u));   // release: this CTA's q_rope and TMEM rows
        }
      }
      // last visible key token of the row
      const int qk = live ? (p.q_tok ? __ldg(p.q_tok + grow) : P.q_tok0 + tl) : -1;
      const float sl2 = p.scale_log2 * qs;
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
      const uint32_t ssr0 = mapa_shared(bar(kSSR), 0u);
      for (int j = 0; j < n; ++j) {
        const int b = j & 1;
        uint32_t v0[64], v1[64];
        float mx = -INFINITY;
        bool wok = await2_warp(p, bar(kSSF + b), (j >> 1) & 1);
        tc_fence_after();
        if (wok) {
          const float m0 = tmem_ld64_max(tmem + lane_off + 256 + 128 * b, v0);   // keys 0..63 of the tile
          const float m1 = tmem_ld64_max(tmem + lane_off + 256 + 128 * b + 64, v1);
          mx = fmaxf(m0, m1);
        }
        tc_fence_before();
        __syncwarp();
        // relaxed: the S buffer's reads are ordered for the next MMAs by the tcgen05 fences around it
        if (lane == 0 && wok) mbar_arrive_cluster_relaxed(ssr0 + 8u * b);
        const int kt0 = it.t0 + 128 * j;
        const uint32_t stg = sbase + SS::kPS + b * SS::kPSBuf;   // this tile's staging buffer
        if (!(kt0 >= it.k_lo && kt0 + 127 < it.k_hi && kt0 + 127 <= qk)) {
          float m8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) m8[i] = -INFINITY;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int ka = kt0 + c, kb = kt0 + 64 + c;
            const float xa = (ka >= it.k_lo && ka < it.k_hi && ka <= qk) ? __uint_as_float(v0[c]) : -INFINITY;
            const float xb = (kb >= it.k_lo && kb < it.k_hi && kb <= qk) ? __uint_as_float(v1[c]) : -INFINITY;
            v0[c] = __float_as_uint(xa);
            v1[c] = __float_as_uint(xb);
            m8[c & 7] = fmax3(m8[c & 7], xa, xb);
          }
          mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])), fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        }
        const float m_tile = mx * sl2;
        float alpha = 1.f;
        if (m_tile > m_used + kRescale2) {
          alpha = ex2(m_used - m_tile);   // 0 when m_used = -inf
          m_used = m_tile;
        }
        const float mref = (m_used == -INFINITY) ? 0.f : m_used;
        const uint64_t sc2 = f2pack(sl2, sl2), nm2 = f2pack(-mref, -mref);
        // P of the tile in registers while the previous tile's copy is still in flight
        uint64_t s4[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[64];
        if (wok) {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const uint32_t x0u = c < 32 ? v0[2 * c] : v1[2 * c - 64], x1u = c < 32 ? v0[2 * c + 1] : v1[2 * c - 63];
            float x0, x1;
            f2unpack(ffma2(f2pack(__uint_as_float(x0u), __uint_as_float(x1u)), sc2, nm2), x0, x1);
            const float a = ex2(x0), bb = ex2(x1);
            s4[c & 3] = fadd2(s4[c & 3], f2pack(a, bb));
            pk[c] = pack_bf16(a, bb);
          }
        }
        // the tile's staging buffer is free once the copy it held two tiles ago landed; the four warps
        // go on, or leave, together
        if (wok && j >= 2) wok = await2_warp(p, bar(kSTF + b), ((j - 2) >> 1) & 1);
        if (named_bar_or(1, 128, !wok)) { ok = false; break; }
#pragma unroll
        for (int hk = 0; hk < 2; ++hk)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            sts128(stg + hk * kBlk128 + sw128_off((uint32_t)r, (uint32_t)c), pk[32 * hk + 4 * c],
                   pk[32 * hk + 4 * c + 1], pk[32 * hk + 4 * c + 2], pk[32 * hk + 4 * c + 3]);
        float s8[4];
        f2unpack(fadd2(s4[0], s4[1]), s8[0], s8[1]);
        f2unpack(fadd2(s4[2], s4[3]), s8[2], s8[3]);
        l = l * alpha + ((s8[0] + s8[2]) + (s8[1] + s8[3]));
        reinterpret_cast<float*>(sgen + SS::kPS + b * SS::kPSBuf + SS::kPSAlpha)[r] = alpha;
        const uint32_t any_rescale = __any_sync(0xffffffffu, alpha != 1.f) ? 1u : 0u;
        if (lane == 0) reinterpret_cast<uint32_t*>(sgen + SS::kPS + b * SS::kPSBuf + SS::kPSFlags)[warp & 3] = any_rescale;
        fence_proxy_async_smem();   // the staged tile is read by the bulk copy (async proxy)
        named_bar_sync(1, 128);
        if (r == 0) {
          // P tile b of the O CTA is free once the PV of tile j - 2 is done
          if (j >= 2 && !await2(p, bar(kPFR + b), ((j - 2) >> 1) & 1)) continue;   // the others time out next tile
          const uint32_t cbar = mapa_shared(bar(kPF + b), orank);
          bulk_copy_to_peer(mapa_shared(sbase + kOP + b * kOPBytes, orank), stg, kOPBytes, cbar);
          bulk_copy_to_peer(mapa_shared(sbase + kOAlpha + b * 512, orank), stg + SS::kPSAlpha, 512, cbar);
          bulk_copy_to_peer(mapa_shared(sbase + kOFlags + 16 * b, orank), stg + SS::kPSFlags, 16, cbar);
        }
      }
      // final row sums to the O CTA; lse of the item
      st_async_b32(mapa_shared(sbase + kOL + 4 * r, orank), __float_as_uint(ok ? l : 0.f),
                   mapa_shared(bar(kLF), orank));
      if (live) {
        const float lse = (ok && l > 0.f) ? (m_used + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        p.lat_lse[(int64_t)it.slot * p.slot_stride_rows + orow] = lse;
      }
      // the last two PV commits land on this CTA's barriers before it exits
      for (int j = max(0, n - 2); j < n && ok; ++j)
        if (!await2_warp(p, bar(kPFR + (j & 1)), (j >> 1) & 1)) ok = false;
    }
  } else {
    // ================================================================ O pair
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- loads: this CTA's latent columns of 64 keys a stage
      bool ok = true;
      const int U = 2 * n;
      const uint32_t full0 = mapa_shared(bar(kCF), 2u);
      for (int u = 0; u < U && ok; ++u) {
        const int s = u % kORing;
        // 64 keys: P is zero past the item's keys, so those rows must be finite: a request's last block comes
        // from its copy (zeros past the sequence), the others in place (looked up before the slot wait)
        const int kt = it.t0 + 64 * u;
        int row = (int)(row_base + kt);
        const void* map = &p.tm_c2;
        if (p.o_in_place) {
          if ((kt >> 6) == P.last_lb) {
            row = (int)row_base;
          } else {
            row = cache_row(p, P, kt);
            map = &p.tm_k2;
          }
        }
        if (u >= kORing && !await2(p, bar(kCE + s), ((u / kORing) - 1) & 1)) { ok = false; break; }
        if (first) mbar_arrive_expect_tx(bar(kCF + s), 2 * kOStage);
        const uint32_t st = sbase + kOC + s * kOStage;
        tma_load_3d_pair(st, map, 0, row, 2 * (int)half, full0 + 8u * s);              // columns 128 r ..
        tma_load_3d_pair(st + 2 * kBlk, map, 0, row, 4 + 2 * (int)half, full0 + 8u * s);   // 256 + 128 r ..
      }
      for (int u = max(0, U - kORing); u < U && ok; ++u)
        if (!await2(p, bar(kCE + u % kORing), (u / kORing) & 1)) ok = false;
    } else if (warp == 1) {
      // ---------------------------------------------------------- per tile: P landed, rows rescaled; then (first
      // CTA) O += P c for the pair.  The whole warp runs the loop: lane 0 arrives and arms the barriers, one
      // elected lane issues each MMA and commit.
      if (lane == 0) {
        for (int b = 0; b < min(n, 2); ++b) mbar_arrive_expect_tx(bar(kPF + b), kTxP2);
        mbar_arrive_expect_tx(bar(kLF), 512);
      }
      bool ok = true;
      volatile int* hand = reinterpret_cast<volatile int*>(sgen + kOFlags + 32);
      const uint32_t pr0 = mapa_shared(bar(kPR), 2u);
      const uint64_t pd0 = sdesc_sw128(sbase + kOP, 16, 1024);     // P tiles, K-major
      const uint64_t cd0 = sdesc_sw128(sbase + kOC, kBlk, 1024);   // latent stages, MN-major
      int events = 0;
      for (int j = 0; j < n && ok; ++j) {
        const int b = j & 1;
        if (!await2_warp(p, bar(kPF + b), (j >> 1) & 1)) { ok = false; break; }
        if (j > 0) {
          uint32_t f[4];
          lds128(sbase + kOFlags + 16 * b, f);
          if (f[0] | f[1] | f[2] | f[3]) {
            // O must hold PV of every earlier tile before its rows are rescaled
            if (!await2_warp(p, bar(kPVD + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) { ok = false; break; }
            if (lane == 0) {
              *hand = b;
              mbar_arrive(bar(kCN));
            }
            if (!await2_warp(p, bar(kCD), events & 1)) { ok = false; break; }
            ++events;
          }
        }
        fence_proxy_async_smem();   // P was written by the S CTA's stores, the MMA reads it as an operand
        tc_fence_before();
        __syncwarp();
        // P and the rescaled rows of this CTA are ready for the leader's MMAs.  Both arrives are relaxed: P
        // is in this CTA's shared memory once its copy's completion was observed above, and the MMAs the
        // leader issues after seeing this arrive read that memory directly; the rescaled rows were stored and
        // waited for (tcgen05.wait::st) and the tcgen05 fences around this arrive and the leader's wait order
        // them.  (A cluster-scope release here held the peer's thread 0.6 us a tile, on the path to each PV.)
        if (lane == 0) {
          if (first) mbar_arrive_relaxed(bar(kPR + b));
          else mbar_arrive_cluster_relaxed(pr0 + 8u * b);
          if (j + 2 < n) mbar_arrive_expect_tx_relaxed(bar(kPF + b), kTxP2);
        }
        if (first) {
          if (!await2_warp(p, bar(kPR + b), (j >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
            const int u = 2 * j + kh, s = u & (kORing - 1);
            if (!await2_warp(p, bar(kCF + s), (u / kORing) & 1)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sdesc_add(pd0, b * kOPBytes + kh * kBlk128 + kk * 32);
#pragma unroll
              for (int nh = 0; nh < 2; ++nh)
                mma2_ss_elect(tmem + 256 * nh, ad, sdesc_add(cd0, s * kOStage + nh * 2 * kBlk + kk * 2048), kIdPV2,
                              (j | kh | kk) ? 1u : 0u);
            }
            mma2_commit_mc_elect(bar(kCE + s), kMaskO);
          }
          if (!ok) break;
          mma2_commit_mc_elect(bar(kPVD + b), kMaskO);
          mma2_commit_mc_elect(bar(kPFR + b), kMaskS);
        }
      }
      if (lane == 0) {
        *hand = -1;   // no more tiles: the correction warps go on to the epilogue
        mbar_arrive(bar(kCN));
      }
    } else if (warp == 3 && lane == 0) {
      // ---------------------------------------------------------- each P tile landed: the S CTA that sent it
      // may stage the tile after next in that staging buffer.  A thread of its own, so that the control
      // thread's arrives never wait for this remote arrive to complete.  The copy of tile j + 2 into PF(b)'s
      // buffer waits for this thread's signal of tile j, so PF(b)'s phases never run ahead of this loop.
      const uint32_t stf_s = mapa_shared(bar(kSTF), half);
      for (int j = 0; j < n; ++j) {
        if (!await2(p, bar(kPF + (j & 1)), (j >> 1) & 1)) break;
        mbar_arrive_cluster_relaxed(stf_s + 8u * (j & 1));   // relaxed: a landed copy has read its source
      }
    } else if (warp >= 4) {
      // ---------------------------------------------------------- rescale O rows; epilogue
      const int r = tid - 128;
      const int prow = it.row0 + 128 * (int)half + r;
      const bool live = prow < P.q_count * H;
      const int tl = live ? prow / H : 0, h = live ? prow - (prow / H) * H : 0;
      const int64_t orow = ((int64_t)P.q_begin + tl) * H + h;
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      const float* alpha_s = reinterpret_cast<const float*>(sgen + kOAlpha);
      const volatile int* hand = reinterpret_cast<const volatile int*>(sgen + kOFlags + 32);
      bool ok = true;
      for (int ev = 0;; ++ev) {
        if (!await2_warp(p, bar(kCN), ev & 1)) { ok = false; break; }
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
        if (lane == 0) mbar_arrive(bar(kCD));
      }
      if (ok && n > 0 && !await2_warp(p, bar(kPVD + ((n - 1) & 1)), ((n - 1) >> 1) & 1)) ok = false;
      if (ok && !await2_warp(p, bar(kLF), 0)) ok = false;
      tc_fence_after();
      const float lsum = ok ? reinterpret_cast<const float*>(sgen + kOL)[r] : 0.f;
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      // every row of this CTA live (all but an item's last row tile): O / l leaves by TMA stores of
      // 32-column boxes staged in the latent stage ring, which the last PV has finished reading
      const bool full = ok && n > 0 && it.row0 + 128 * (int)half + 128 <= P.q_count * H;
      if (!named_bar_or(2, 128, !full)) {
        const int grow0 = (int)((int64_t)it.slot * p.slot_stride_rows + (int64_t)P.q_begin * H + it.row0 + 128 * (int)half);
#pragma unroll 1
        for (int cc = 0; cc < 16; ++cc) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_off + 32 * cc, o);
          const uint32_t box = sbase + kOC + (uint32_t)(cc & 7) * kBlk128;
          if (cc >= 8) {   // the box's store of 8 chunks ago has read it
            if (r == 0) bulk_wait_read<7>();
            named_bar_sync(2, 128);
          }
#pragma unroll
          for (int c = 0; c < 8; ++c)
            sts128(box + sw128_off((uint32_t)r, (uint32_t)c), __float_as_uint(__uint_as_float(o[4 * c]) * inv),
                   __float_as_uint(__uint_as_float(o[4 * c + 1]) * inv), __float_as_uint(__uint_as_float(o[4 * c + 2]) * inv),
                   __float_as_uint(__uint_as_float(o[4 * c + 3]) * inv));
          fence_proxy_async_smem();   // the box is read by the TMA store
          named_bar_sync(2, 128);
          if (r == 0) {
            tma_store_2d(&p.tm_lat, box, 32 * cc, grow0);
            bulk_commit();
          }
        }
        if (r == 0) bulk_wait0();
      } else {
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
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // no operation of another CTA targets this one's memory, and the pair's MMAs are done
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc2(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_absorb_attn(const AbsorbParams& p, cudaStream_t s) {
  if (p.n_items == 0) return cudaSuccess;
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(absorb_attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)L2<false>::kSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(absorb_attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)L2<true>::kSmem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(4 * p.n_items);
  cfg.blockDim = dim3(kThreads2);
  cfg.dynamicSmemBytes = p.fp8_scores ? L2<true>::kSmem : L2<false>::kSmem;
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;
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
