// Fused MLA prefill tile kernel: paged latent gather (+FP8 dequant), kv_b_proj
// up-projection on tcgen05 into TMEM, QK^T with the broadcast k_rope, online
// softmax, PV, and (out, lse) per KV split.
//
// Follows "DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析", section 4.4
// (per chunk: gather c_kv and k_rope, kv_full = c_kv @ kv_b_proj, K = [K_nope |
// k_rope broadcast], flash attention giving (out, lse)) with the query RoPE
// relocation of "RedKnot-MLA: Multi-Head Offline-Online Reuse for DeepSeek-V4
// Long-Context Serving", section 2 ("Online position restoration and merge").
//
// One CTA = (split, 128-query tile, head).  Per 128-token KV tile:
//   1. 8 latent slices [128 tok x 64] and kv_b_proj slices [64 x 256] are staged
//      in 128B-swizzled shared memory; tcgen05.mma accumulates
//      [K_nope | V] = c_kv * W_h (M=128, N=256, K=512) in TMEM columns 0..255.
//   2. TMEM -> registers -> bf16 -> shared K_nope / V tiles (never global).
//   3. S = Q_nope K_nope^T + Q_rope k_rope^T (M=128, N=128, K=192) in TMEM.
//   4. One thread per query row: mask, online softmax (base 2), P -> shared bf16,
//      O rescale in TMEM.
//   5. O += P V (M=128, N=128, K=128) in TMEM.
// Epilogue: out = O / l, lse = ln(sum exp(s)), to the split's partial slot.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kTileQ = 128;
constexpr int kTileK = 128;

constexpr uint32_t kAtom = 16384;                 // [128 rows x 128 B] swizzled tile
constexpr uint32_t kSmQ = 0;                      // Q: nope[0:64], nope[64:128], rope
constexpr uint32_t kSmC = kSmQ + 3 * kAtom;       // latent slice [128 x 64]
constexpr uint32_t kSmW = kSmC + kAtom;           // W slice: 4 MN blocks [64 K-rows x 64]
constexpr uint32_t kSmK = kSmW + 2 * kAtom;       // K_nope [128 x 128]: 2 atom columns
constexpr uint32_t kSmV = kSmK + 2 * kAtom;       // V [128 keys x 128]: 2 dv halves
constexpr uint32_t kSmKR = kSmV + 2 * kAtom;      // k_rope [128 x 64]
constexpr uint32_t kSmP = kSmKR + kAtom;          // P [128 x 128]: 2 atom columns
constexpr uint32_t kSmCtl = kSmP + 2 * kAtom;     // mbarrier, TMEM base, flags
constexpr uint32_t kSmBytes = kSmCtl + 64 + 1024; // + alignment slack

constexpr uint32_t kTmemAcc = 0;    // 256 columns: K_nope 0..127, V 128..255
constexpr uint32_t kTmemS = 256;    // 128 columns
constexpr uint32_t kTmemO = 384;    // 128 columns

constexpr uint32_t kIdescUp = idesc_bf16(128, 256, false, true);
constexpr uint32_t kIdescS = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, false, true);

__device__ __forceinline__ uint4 ldg16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ldg8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ void sts16(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// OCP E4M3FN -> bf16 bits (exact: every finite e4m3 value is a bf16 value).
__device__ __forceinline__ uint32_t e4m3_to_bf16_bits(uint32_t c) {
  const uint32_t s = (c & 0x80u) << 8;
  const uint32_t e = (c >> 3) & 0xFu;
  const uint32_t m = c & 7u;
  if (e == 15u && m == 7u) return 0x7FC0u | s;
  if (e != 0u) return s | ((e + 120u) << 7) | (m << 4);  // rebias 7 -> 127
  if (m == 0u) return s;
  // subnormal m * 2^-9: leading one at bit lb of m gives 2^(lb-9) * (m / 2^lb)
  const uint32_t lb = (m >= 4u) ? 2u : ((m >= 2u) ? 1u : 0u);
  return s | ((118u + lb) << 7) | ((m - (1u << lb)) << (7u - lb));
}

__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint2 v) {
  uint32_t w[2] = {v.x, v.y};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t src = w[i >> 1] >> ((i & 1) * 16);
    o[i] = e4m3_to_bf16_bits(src & 0xFFu) | (e4m3_to_bf16_bits((src >> 8) & 0xFFu) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Physical row address of logical token t of request `req`, or nullptr (and an
// error bit) when the block-table entry is outside [0, num_blocks).
__device__ __forceinline__ const uint8_t* token_row(const PrefillParams& p, int req, int t) {
  const int blk = __ldg(p.block_table + (int64_t)req * p.max_blocks + (t >> 6));
  if (blk < 0 || blk >= p.num_blocks) {
    atomicOr(p.err, kErrBadBlock);
    return nullptr;
  }
  const int64_t row = (int64_t)blk * kBlock + (t & 63);
  return p.kv_cache + row * (p.kv_fp8 ? kRowBytesFp8 : kRowBytesBf16);
}

__global__ void __launch_bounds__(kThreads, 1) prefill_tile_kernel(const __grid_constant__ PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  const uint32_t sbase = (raw_base + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw_base);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h = blockIdx.y;
  const int H = p.num_heads;

  // ---- which split / q-tile
  int lo = 0, hi = p.num_splits - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.splits[mid].tile_begin <= (int)blockIdx.x) lo = mid; else hi = mid - 1;
  }
  const Split sp = p.splits[lo];
  const int q0 = ((int)blockIdx.x - sp.tile_begin) * kTileQ;
  const int nq = min(kTileQ, sp.q_count - q0);
  const int row0 = sp.q_begin + q0;
  const int tokq0 = sp.q_tok0 + q0;
  const int k_lo = sp.k_begin;
  const int k_hi = min(sp.k_end, tokq0 + nq);  // causal: key token <= last query token

  const uint32_t bar = sbase + kSmCtl;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sgen + kSmCtl + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sgen + kSmCtl + 12);

  if (warp == 0) {
    tmem_alloc(sbase + kSmCtl + 8, 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    mbar_init(bar, 1);
    fence_mbar_init();
    *abort_flag = 0;
  }

  // ---- Q tile: q_nope as is, q_rope rotated by (q_pos - rope_offset)
  for (int idx = tid; idx < kTileQ * 24; idx += kThreads) {
    const int r = idx / 24;
    const int c = idx - r * 24;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < nq) {
      const uint16_t* src = p.q + ((int64_t)(row0 + r) * H + h) * kDqk + c * 8;
      v = ldg16(src);
      if (c >= 16) {
        const int64_t delta = (int64_t)__ldg(p.q_pos + row0 + r) - sp.rope_offset;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int k = (c - 16) * 4 + i;
          float sn, cs;
          rope_sincos(delta, p.rope_frac[k], &sn, &cs);
          const float x0 = __uint_as_float(w[i] << 16);
          const float x1 = __uint_as_float(w[i] & 0xFFFF0000u);
          w[i] = pack_bf16(x0 * cs - x1 * sn, x0 * sn + x1 * cs);
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    const uint32_t atom = (uint32_t)(c >> 3);
    sts16(sbase + kSmQ + atom * kAtom + sw128_off(r, c & 7), v);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int row_q = (warp & 3) * 32 + lane;          // TMEM lane = query/token row
  const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
  float m_run = -INFINITY, l_run = 0.f;
  uint32_t phase = 0;
  bool first = true;
  bool aborted = false;

  const float out_scale = p.kv_fp8 ? p.kv_scale : 1.f;
  const int64_t wrow = (int64_t)H * (kDnope + kDv);

  for (int kt0 = k_lo; kt0 < k_hi && !aborted; kt0 += kTileK) {
    const int ntok = min(kTileK, k_hi - kt0);

    // ---------------- up-projection: 8 slices of 64 latent columns
    for (int ks = 0; ks < kDc / 64; ++ks) {
      // latent slice (+ k_rope on the first slice)
      for (int idx = tid; idx < kTileK * 8; idx += kThreads) {
        const int t = idx >> 3, c = idx & 7;
        uint4 v = make_uint4(0, 0, 0, 0), vr = make_uint4(0, 0, 0, 0);
        if (t < ntok) {
          const uint8_t* rp = token_row(p, sp.req, kt0 + t);
          if (rp) {
            if (p.kv_fp8) {
              v = e4m3x8_to_bf16x8(ldg8(rp + ks * 64 + c * 8));
              if (ks == 0) vr = ldg16(rp + kDc + c * 16);
            } else {
              v = ldg16(rp + ks * 128 + c * 16);
              if (ks == 0) vr = ldg16(rp + 2 * kDc + c * 16);
            }
          }
        }
        sts16(sbase + kSmC + sw128_off(t, c), v);
        if (ks == 0) sts16(sbase + kSmKR + sw128_off(t, c), vr);
      }
      // kv_b_proj slice: latent rows ks*64.., features K(h) then V(h)
      for (int idx = tid; idx < 64 * 32; idx += kThreads) {
        const int r = idx >> 5, c32 = idx & 31;
        const int j = c32 >> 3, c = c32 & 7;
        const int col = (j < 2) ? (h * kDnope + j * 64 + c * 8) : (H * kDnope + h * kDv + (j - 2) * 64 + c * 8);
        const uint4 v = ldg16(p.w + (int64_t)(ks * 64 + r) * wrow + col);
        sts16(sbase + kSmW + (uint32_t)j * 8192u + sw128_off(r, c), v);
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t a = sdesc_sw128(sbase + kSmC + kk * 32, 16, 1024);
          const uint64_t b = sdesc_sw128(sbase + kSmW + kk * 2048, 8192, 1024);
          mma_bf16(tmem + kTmemAcc, a, b, kIdescUp, (ks | kk) != 0);
        }
        mma_commit(bar);
      }
      if (!mbar_wait(bar, phase)) { atomicOr(p.err, kErrTimeout); *abort_flag = 1; }
      phase ^= 1;
      __syncthreads();
      if (*abort_flag) { aborted = true; break; }
    }
    if (aborted) break;

    // ---------------- TMEM accumulators -> bf16 K_nope / V tiles in shared memory
    tc_fence_after();
    {
      const bool is_v = warp >= 4;
      const uint32_t dst = sbase + (is_v ? kSmV : kSmK);
      const bool valid = row_q < ntok;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + kTmemAcc + (is_v ? 128u : 0u) + cc * 32, r);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (valid) {
            v.x = pack_bf16(__uint_as_float(r[g * 8 + 0]) * out_scale, __uint_as_float(r[g * 8 + 1]) * out_scale);
            v.y = pack_bf16(__uint_as_float(r[g * 8 + 2]) * out_scale, __uint_as_float(r[g * 8 + 3]) * out_scale);
            v.z = pack_bf16(__uint_as_float(r[g * 8 + 4]) * out_scale, __uint_as_float(r[g * 8 + 5]) * out_scale);
            v.w = pack_bf16(__uint_as_float(r[g * 8 + 6]) * out_scale, __uint_as_float(r[g * 8 + 7]) * out_scale);
          }
          const uint32_t atom = (uint32_t)(cc >> 1);
          const uint32_t chunk = (uint32_t)((cc & 1) * 4 + g);
          sts16(dst + atom * kAtom + sw128_off(row_q, chunk), v);
        }
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();

    // ---------------- S = Q K^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (uint32_t)(kk >> 2) * kAtom + (uint32_t)(kk & 3) * 32u;
        mma_bf16(tmem + kTmemS, sdesc_sw128(sbase + kSmQ + off, 16, 1024),
                 sdesc_sw128(sbase + kSmK + off, 16, 1024), kIdescS, kk != 0);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(tmem + kTmemS, sdesc_sw128(sbase + kSmQ + 2 * kAtom + kk * 32, 16, 1024),
                 sdesc_sw128(sbase + kSmKR + kk * 32, 16, 1024), kIdescS, 1);
      }
      mma_commit(bar);
    }
    if (!mbar_wait(bar, phase)) { atomicOr(p.err, kErrTimeout); *abort_flag = 1; }
    phase ^= 1;
    __syncthreads();
    if (*abort_flag) { aborted = true; break; }

    // ---------------- online softmax (warps 0..3, one query row per thread)
    tc_fence_after();
    if (warp < 4) {
      const int tok_q = tokq0 + row_q;
      uint32_t s[128];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_off + kTmemS + cc * 32, r);
#pragma unroll
        for (int j = 0; j < 32; ++j) s[cc * 32 + j] = r[j];
      }
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < kTileK; ++j) {
        const int kt = kt0 + j;
        const bool ok = (j < ntok) && (kt <= tok_q);
        const float x = ok ? __uint_as_float(s[j]) * p.scale_log2 : -INFINITY;
        s[j] = __float_as_uint(x);
        tmax = fmaxf(tmax, x);
      }
      const float m_new = fmaxf(m_run, tmax);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m_run - m_use);
      float lsum = 0.f;
#pragma unroll
      for (int cc = 0; cc < 16; ++cc) {
        uint32_t pk[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const float a = ex2(__uint_as_float(s[cc * 8 + 2 * g]) - m_use);
          const float b = ex2(__uint_as_float(s[cc * 8 + 2 * g + 1]) - m_use);
          lsum += a + b;
          pk[g] = pack_bf16(a, b);
        }
        sts16(sbase + kSmP + (uint32_t)(cc >> 3) * kAtom + sw128_off(row_q, cc & 7),
              make_uint4(pk[0], pk[1], pk[2], pk[3]));
      }
      l_run = l_run * alpha + lsum;
      m_run = m_new;
      if (!first && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + kTmemO + cc * 32, r);
#pragma unroll
          for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
          tmem_st32(tmem + lane_off + kTmemO + cc * 32, r);
        }
        tmem_wait_st();
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();

    // ---------------- O += P V
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t a = sdesc_sw128(sbase + kSmP + (uint32_t)(kk >> 2) * kAtom + (uint32_t)(kk & 3) * 32u, 16, 1024);
        const uint64_t b = sdesc_sw128(sbase + kSmV + (uint32_t)kk * 2048u, kAtom, 1024);
        mma_bf16(tmem + kTmemO, a, b, kIdescPV, (first && kk == 0) ? 0u : 1u);
      }
      mma_commit(bar);
    }
    if (!mbar_wait(bar, phase)) { atomicOr(p.err, kErrTimeout); *abort_flag = 1; }
    phase ^= 1;
    __syncthreads();
    if (*abort_flag) { aborted = true; break; }
    first = false;
  }

  // ---------------- epilogue: (out, lse) of this split
  tc_fence_after();
  if (warp < 4 && !aborted) {  // warp-uniform: every lane takes part in the TMEM loads
    const bool live = row_q < nq;
    const int64_t grow = (int64_t)sp.slot * p.slot_stride_rows + row0 + row_q;
    float* dst = p.part_out + (grow * H + h) * kDv;
    const bool empty = first || !(l_run > 0.f);
    const float inv_l = empty ? 0.f : 1.f / l_run;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t r[32];
      if (!first) tmem_ld32(tmem + lane_off + kTmemO + cc * 32, r);
      if (live) {
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float4 o;
          o.x = empty ? 0.f : __uint_as_float(r[j + 0]) * inv_l;
          o.y = empty ? 0.f : __uint_as_float(r[j + 1]) * inv_l;
          o.z = empty ? 0.f : __uint_as_float(r[j + 2]) * inv_l;
          o.w = empty ? 0.f : __uint_as_float(r[j + 3]) * inv_l;
          *reinterpret_cast<float4*>(dst + cc * 32 + j) = o;
        }
      }
    }
    if (live) p.part_lse[grow * H + h] = empty ? -INFINITY : m_run * 0.69314718055994531f + logf(l_run);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t s) {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(prefill_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmBytes);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  dim3 grid(p.num_tiles, p.num_heads);
  prefill_tile_kernel<<<grid, kThreads, kSmBytes, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
