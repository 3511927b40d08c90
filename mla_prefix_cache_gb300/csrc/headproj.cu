// The two per-head projections of the absorbed (latent-space) path ("DeepSeek
// MLA — Prefix Cache 与 Chunked Prefill 深度解析", section 3: W_UK folded into
// the query, W_UV applied after the attention), on the tensor cores:
//   qabsorb_kernel<false>  qlat[t][h][:]  = bf16(scale q_nope[t][h] W_UK,h^T)   [512]
//   qabsorb_kernel<true>   qlat8[t][h][:] = e4m3(qlat / s), s = amax / 448 of the row
//   absorb_proj_kernel     out[t][h][:]   = scale o[t H + h] W_UV,h             [128]
// Both are one tcgen05 MMA chain per CTA (M = 128 rows of one head), operands
// staged in shared memory with 128-byte swizzle, the accumulator in TMEM.
//
// kv_b_proj is [512][H * 256]: W_UK,h[c][d] at column 128 h + d, W_UV,h[c][j]
// at column 128 H + 128 h + j.  So W_UK,h is K-major for the q absorption (K =
// d) and W_UV,h is MN-major for the projection (K = c, N = j contiguous).
#include "absorb.h"
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr uint32_t kAtomRows128 = 16384;   // [128 rows x 128 B] swizzled block

// Bounded wait; on timeout records the error.
__device__ __forceinline__ bool hwait(uint32_t* err, uint32_t bar, uint32_t parity) {
  if (mbar_wait(bar, parity)) return true;
  atomicOr(err, kErrTimeout);
  return false;
}

// ---------------------------------------------------------------- q absorption
// CTA (tile of 128 tokens, 256 latent columns (bf16) or all 512 (E4M3), head).
// Shared memory: A = q_nope [128 x 128] as two [128 x 64] blocks, then B = the
// CTA's rows of W_UK,h as [256 c x 64 d] blocks (d block, c half); after the
// MMAs the same memory stages the output rows for the TMA stores.
template <bool kF8>
struct QA {
  static constexpr int kCols = kF8 ? 512 : 256;           // latent columns of a CTA
  static constexpr int kHalves = kCols / 256;
  static constexpr uint32_t kA = 0;
  static constexpr uint32_t kB = 2 * kAtomRows128;
  static constexpr uint32_t kTx = 2 * kAtomRows128 + kHalves * 2 * 32768;
  static constexpr uint32_t kBars = kB + kHalves * 2 * 32768;
  static constexpr uint32_t kSmem = kBars + 64 + 1024;
};
constexpr uint32_t kIdescQA = idesc_bf16(128, 256, false, false);

template <bool kF8>
__global__ void __launch_bounds__(128, 1) qabsorb_kernel(const __grid_constant__ QAbsorbParams p) {
  using L = QA<kF8>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  const uint32_t bar_full = sbase + L::kBars, bar_done = bar_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + L::kBars + 16);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.z;
  const int c0 = blockIdx.y * L::kCols;
  const int t0 = p.row0 + blockIdx.x * 128;   // first token of the tile (TMA coordinates)

  if (threadIdx.x == 0) {
    mbar_init(bar_full, 1);
    mbar_init(bar_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), L::kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
  if (threadIdx.x == 0) {
    prefetch_tensormap(&p.tm_q);
    prefetch_tensormap(&p.tm_w);
    mbar_arrive_expect_tx(bar_full, L::kTx);
#pragma unroll
    for (int db = 0; db < 2; ++db) tma_load_3d(sbase + L::kA + db * kAtomRows128, &p.tm_q, 64 * db, h, t0, bar_full);
#pragma unroll
    for (int nh = 0; nh < L::kHalves; ++nh)
#pragma unroll
      for (int db = 0; db < 2; ++db)
        tma_load_2d(sbase + L::kB + (nh * 2 + db) * 32768, &p.tm_w, 128 * h + 64 * db, c0 + 256 * nh, bar_full);
    ok = hwait(p.err, bar_full, 0);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int nh = 0; nh < L::kHalves; ++nh)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16(tmem + 256 * nh, sdesc_sw128(sbase + L::kA + (kk >> 2) * kAtomRows128 + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(sbase + L::kB + (nh * 2 + (kk >> 2)) * 32768 + (kk & 3) * 32, 16, 1024), kIdescQA,
                   kk > 0 ? 1u : 0u);
      mma_commit(bar_done);
    }
  }
  ok = __syncthreads_and(ok);
  if (ok) ok = __all_sync(0xffffffffu, hwait(p.err, bar_done, 0));
  tc_fence_after();
  const int r = 32 * warp + lane;                 // row of the tile = TMEM lane
  const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
  if (ok) {
    if constexpr (!kF8) {
      // 32 columns a load: 64 B of bf16 = four 16-byte chunks of a [128 x 64] block
#pragma unroll 1
      for (int j = 0; j < 8; ++j) {
        uint32_t v[32];
        tmem_ld32(tl + 32 * j, v);
        const uint32_t blk = sbase + (j >> 1) * kAtomRows128;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t w0 = pack_bf16(__uint_as_float(v[8 * c]) * p.scale, __uint_as_float(v[8 * c + 1]) * p.scale);
          const uint32_t w1 = pack_bf16(__uint_as_float(v[8 * c + 2]) * p.scale, __uint_as_float(v[8 * c + 3]) * p.scale);
          const uint32_t w2 = pack_bf16(__uint_as_float(v[8 * c + 4]) * p.scale, __uint_as_float(v[8 * c + 5]) * p.scale);
          const uint32_t w3 = pack_bf16(__uint_as_float(v[8 * c + 6]) * p.scale, __uint_as_float(v[8 * c + 7]) * p.scale);
          sts128(blk + sw128_off(r, (j & 1) * 4 + c), w0, w1, w2, w3);
        }
      }
    } else {
      float m = 0.f;
#pragma unroll 1
      for (int j = 0; j < 16; ++j) {
        uint32_t v[32];
        tmem_ld32(tl + 32 * j, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(__uint_as_float(v[i])));
      }
      const float sc = m > 0.f ? m / 448.f : 1.f;
      const float inv = 1.f / sc;
      // 32 columns a load: 32 B of E4M3 = two 16-byte chunks of a [128 x 128 B] block
#pragma unroll 1
      for (int j = 0; j < 16; ++j) {
        uint32_t v[32];
        tmem_ld32(tl + 32 * j, v);
        const uint32_t blk = sbase + (j >> 2) * kAtomRows128;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int k = 16 * c + 4 * i;
            w[i] = (uint32_t)pack_e4m3x2(__uint_as_float(v[k]) * inv, __uint_as_float(v[k + 1]) * inv) |
                   ((uint32_t)pack_e4m3x2(__uint_as_float(v[k + 2]) * inv, __uint_as_float(v[k + 3]) * inv) << 16);
          }
          sts128(blk + sw128_off(r, (j & 3) * 2 + c), w[0], w[1], w[2], w[3]);
        }
      }
      const int t = t0 + r;
      if (t < p.row0 + p.tokens) p.qscale[(int64_t)t * p.num_heads + h] = sc;
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && ok) {
    // rows past the launch's last token are clipped by the map
#pragma unroll
    for (int b = 0; b < 4; ++b) tma_store_3d(&p.tm_out, sbase + b * kAtomRows128, c0 + (kF8 ? 128 : 64) * b, h, t0);
    bulk_commit();
    bulk_wait0();
  }
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kCols);
  }
}

// ---------------------------------------------------------------- output projection
// CTA (tile of 128 rows of the launch's ranges, head): K = 512 latent columns
// in four chunks of 128, double-buffered.  A chunk is A = o [128 rows x 128]
// (fp32 rounded to bf16 by the threads, two [128 x 64] K-major blocks) and
// B = W_UV,h [128 c x 128 j] (TMA, two MN-major [128 c x 64 j] blocks).
constexpr uint32_t kPChunk = 4 * kAtomRows128;      // A (2 blocks) + B (2 blocks)
constexpr uint32_t kPBars = 2 * kPChunk;             // 4 barriers, the TMEM address, then 128 row indices
constexpr uint32_t kPSmem = kPBars + 64 + 128 * 8 + 1024;
constexpr uint32_t kIdescPJ = idesc_bf16(128, 128, false, true);

__global__ void __launch_bounds__(256, 1) absorb_proj_kernel(const __grid_constant__ ProjParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - smem_u32(smem_raw));
  // bars: [0,1] B chunk landed (per buffer), [2,3] MMAs of the buffer's chunk done
  const uint32_t bars = sbase + kPBars;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + kPBars + 32);
  int64_t* grow_s = reinterpret_cast<int64_t*>(sgen + kPBars + 64);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.num_heads;
  const int h = blockIdx.z, r0 = blockIdx.x * 128;

  // global token row of each tile row (-1 past the launch's rows)
  for (int i = threadIdx.x; i < 128; i += 256) {
    const int x = r0 + i;
    int64_t g = -1;
    if (x < p.total_rows) {
      int lo = 0, hi = p.num_ranges - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.ranges[mid].prefix <= x) lo = mid; else hi = mid - 1;
      }
      g = p.ranges[lo].row_begin + (x - p.ranges[lo].prefix);
    }
    grow_s[i] = g;
  }
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) mbar_init(bars + 8 * i, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  bool ok = true;
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    const int b = ch & 1;
    const uint32_t abuf = sbase + b * kPChunk, bbuf = abuf + 2 * kAtomRows128;
    // (uniform) MMAs of chunk ch - 2 done, so its buffer is free
    ok = __syncthreads_and(ok && (ch < 2 || hwait(p.err, bars + 8 * (2 + b), 0)));
    if (!ok) break;
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(bars + 8 * b, 2 * kAtomRows128);
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
        tma_load_2d(bbuf + nb * kAtomRows128, &p.tm_w, 128 * H + 128 * h + 64 * nb, 128 * ch, bars + 8 * b);
    }
    // A: warp w converts rows 16 w .. 16 w + 15; lane l holds columns 4 l .. 4 l + 3 of the chunk
    {
      float4 a[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int64_t g = grow_s[16 * warp + i];
        a[i] = g >= 0 ? __ldg(reinterpret_cast<const float4*>(p.lat_out + (g * H + h) * kDc + 128 * ch) + lane)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const uint32_t blk = abuf + (lane >> 4) * kAtomRows128;
      const uint32_t c16 = (lane & 15) >> 1, sub = (lane & 1) * 8;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t rr = 16 * warp + i;
        const uint32_t addr = blk + rr * 128 + ((c16 ^ (rr & 7)) << 4) + sub;
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(pack_bf16(a[i].x, a[i].y)),
                     "r"(pack_bf16(a[i].z, a[i].w))
                     : "memory");
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      ok = hwait(p.err, bars + 8 * b, (ch >> 1) & 1);
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16(tmem, sdesc_sw128(abuf + (kk >> 2) * kAtomRows128 + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(bbuf + kk * 2048, kAtomRows128, 1024), kIdescPJ, (ch | kk) ? 1u : 0u);
        mma_commit(bars + 8 * (2 + b));
      }
    }
  }
  // the last chunk (3) used buffer 1 in its second round; chunk 2 buffer 0
  ok = __syncthreads_and(ok);
  if (ok) ok = __all_sync(0xffffffffu, hwait(p.err, bars + 8 * 3, 1) && hwait(p.err, bars + 8 * 2, 1));
  tc_fence_after();
  if (ok) {
    // warps w and w + 4 share TMEM lanes 32 (w mod 4) ..: columns 64 (w / 4) .. + 63
    const int r = 32 * (warp & 3) + lane;
    const int64_t g = grow_s[r];
    const int cb = 64 * (warp >> 2);
    uint32_t v[64];
    tmem_ld64(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + cb, v);
    if (g >= 0) {
      const int64_t o = (g * H + h) * kDv + cb;
      if (p.out_bf16) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + o);
        auto o2 = [&](int k) {
          return pack_bf16(__uint_as_float(v[k]) * p.scale, __uint_as_float(v[k + 1]) * p.scale);
        };
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_uint4(o2(8 * i), o2(8 * i + 2), o2(8 * i + 4), o2(8 * i + 6));
      } else {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + o);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          dst[i] = make_float4(__uint_as_float(v[4 * i]) * p.scale, __uint_as_float(v[4 * i + 1]) * p.scale,
                               __uint_as_float(v[4 * i + 2]) * p.scale, __uint_as_float(v[4 * i + 3]) * p.scale);
      }
      if (warp < 4) p.lse[g * H + h] = p.lat_lse[g * H + h];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, uint32_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t configure_headproj() {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || configured_device == dev) return e;
  e = set_smem(qabsorb_kernel<false>, QA<false>::kSmem);
  if (e == cudaSuccess) e = set_smem(qabsorb_kernel<true>, QA<true>::kSmem);
  if (e == cudaSuccess) e = set_smem(absorb_proj_kernel, kPSmem);
  if (e == cudaSuccess) configured_device = dev;
  return e;
}

}  // namespace

cudaError_t launch_qabsorb(const QAbsorbParams& p, cudaStream_t s) {
  if (p.tokens == 0) return cudaSuccess;
  cudaError_t e = configure_headproj();
  if (e != cudaSuccess) return e;
  const bool f8 = p.qscale != nullptr;
  const dim3 grid((p.tokens + 127) / 128, f8 ? 1 : kDc / 256, p.num_heads);
  if (f8) qabsorb_kernel<true><<<grid, 128, QA<true>::kSmem, s>>>(p);
  else qabsorb_kernel<false><<<grid, 128, QA<false>::kSmem, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_absorb_proj(const ProjParams& p, cudaStream_t s) {
  if (p.total_rows == 0) return cudaSuccess;
  cudaError_t e = configure_headproj();
  if (e != cudaSuccess) return e;
  const dim3 grid((p.total_rows + 127) / 128, 1, p.num_heads);
  absorb_proj_kernel<<<grid, 256, kPSmem, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
