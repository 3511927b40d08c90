// GPU steps of the content-addressed block store ("PagedAttention assumed MHA.
// DeepSeek-V4 says that assumption is broken", sections "Position independence
// beats prefix matching" and "The finding: content-addressed dedup needs byte
// verification"): the content hash of a sealed 64-token block, and the byte
// comparison that verifies a hash match.  The table, the sharing decision and
// the collision counter are host policy.
//
// Hash of a block of n 64-bit little-endian words w_i:
//   h = mix(n ^ sum_i mix(w_i + (i + 1) * 0x9e3779b97f4a7c15))   (mod 2^64)
// with mix the SplitMix64 output function (Steele, Lea and Flood, 2014,
// multipliers of Stafford's mix13).  The sum commutes, so a CTA reduces its
// block in any order and the bits do not depend on it.
//
// Both kernels read whole blocks (73728 B of bf16 rows or 40960 B of FP8
// rows) and are HBM-bound.  One CTA of 256 threads takes a block (or a block
// pair) and its threads load the block's 16-byte chunks straight into
// registers, eight CTAs (2048 threads) to an SM.  They use no dynamic shared
// memory: measured against copies through a 3-stage shared-memory ring filled
// by bulk copies, they are 15-20% faster per launch, partly because a kernel
// with a large shared-memory carve-out that follows one without it pays a
// reconfiguration.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr uint64_t kGamma = 0x9e3779b97f4a7c15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xbf58476d1ce4e5b9ull;
  z ^= z >> 27;
  z *= 0x94d049bb133111ebull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint64_t warp_sum64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
  return v;
}

// 16-byte read-only global load that is not kept in L1 (each byte is read once).
__device__ __forceinline__ uint4 ld_stream16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// kChunks: 16-byte chunks per thread in a block (18 for bf16 rows, 10 for FP8).
template <int kChunks>
__global__ void __launch_bounds__(256) block_hash_kernel(const uint8_t* __restrict__ cache, int num_blocks,
                                                         const int32_t* __restrict__ ids, int n,
                                                         uint64_t* __restrict__ hashes, uint32_t* err) {
  constexpr int kThreads = 256;
  constexpr uint64_t kWords = 2ull * kChunks * kThreads;   // words in a whole block
  __shared__ uint64_t part[kThreads / 32];
  const int it = blockIdx.x;
  const int b = __ldg(ids + it);
  const bool ok = b >= 0 && b < num_blocks;
  uint64_t acc = 0;
  if (ok) {
    const uint4* src = reinterpret_cast<const uint4*>(cache + (int64_t)b * (16 * kChunks * kThreads));
    uint4 v[kChunks];
#pragma unroll
    for (int k = 0; k < kChunks; ++k) v[k] = ld_stream16(src + threadIdx.x + k * kThreads);
    // chunk q of the block holds words 2q, 2q + 1; c = (2q + 1) gamma, stepped by 2 * kThreads * gamma
    uint64_t c = (2 * (uint64_t)threadIdx.x + 1) * kGamma;
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
      const uint64_t w0 = ((uint64_t)v[k].y << 32) | v[k].x, w1 = ((uint64_t)v[k].w << 32) | v[k].z;
      acc += mix64(w0 + c) + mix64(w1 + c + kGamma);
      c += 2 * kThreads * kGamma;
    }
  }
  acc = warp_sum64(acc);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint64_t t = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) t += part[w];
    hashes[it] = ok ? mix64(kWords ^ t) : 0ull;
    if (err != nullptr && !ok) atomicOr(err, kErrBadBlock);
  }
}

template <int kChunks>
__global__ void __launch_bounds__(256) block_compare_kernel(const uint8_t* __restrict__ cache, int num_blocks,
                                                            const int32_t* __restrict__ ia,
                                                            const int32_t* __restrict__ ib, int n,
                                                            int32_t* __restrict__ equal, uint32_t* err) {
  constexpr int kThreads = 256;
  const int it = blockIdx.x;
  const int a = __ldg(ia + it), b = __ldg(ib + it);
  const bool ok = a >= 0 && a < num_blocks && b >= 0 && b < num_blocks;
  uint32_t diff = 0;
  if (ok) {
    const uint4* pa = reinterpret_cast<const uint4*>(cache + (int64_t)a * (16 * kChunks * kThreads));
    const uint4* pb = reinterpret_cast<const uint4*>(cache + (int64_t)b * (16 * kChunks * kThreads));
    constexpr int kHalf = (kChunks + 1) / 2;
#pragma unroll
    for (int k0 = 0; k0 < kChunks; k0 += kHalf) {
      uint4 x[kHalf], y[kHalf];
#pragma unroll
      for (int k = 0; k < kHalf; ++k)
        if (k0 + k < kChunks) {
          x[k] = ld_stream16(pa + threadIdx.x + (k0 + k) * kThreads);
          y[k] = ld_stream16(pb + threadIdx.x + (k0 + k) * kThreads);
        }
#pragma unroll
      for (int k = 0; k < kHalf; ++k)
        if (k0 + k < kChunks) diff |= (x[k].x ^ y[k].x) | (x[k].y ^ y[k].y) | (x[k].z ^ y[k].z) | (x[k].w ^ y[k].w);
    }
  }
  const int any = __syncthreads_or(diff != 0u);
  if (threadIdx.x == 0) {
    equal[it] = ok ? (any ? 0 : 1) : -1;
    if (err != nullptr && !ok) atomicOr(err, kErrBadBlock);
  }
}

}  // namespace

cudaError_t launch_block_hash(const uint8_t* cache, int fp8, int num_blocks, const int32_t* ids, int n,
                              uint64_t* hashes, uint32_t* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (fp8) block_hash_kernel<10><<<n, 256, 0, s>>>(cache, num_blocks, ids, n, hashes, err);
  else block_hash_kernel<18><<<n, 256, 0, s>>>(cache, num_blocks, ids, n, hashes, err);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_block_compare(const uint8_t* cache, int fp8, int num_blocks, const int32_t* a, const int32_t* b,
                                 int n, int32_t* equal, uint32_t* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  if (fp8) block_compare_kernel<10><<<n, 256, 0, s>>>(cache, num_blocks, a, b, n, equal, err);
  else block_compare_kernel<18><<<n, 256, 0, s>>>(cache, num_blocks, a, b, n, equal, err);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
