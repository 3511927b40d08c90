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
// rows) and are HBM-bound.  They are persistent: each CTA walks its share of
// the blocks (or block pairs) one unit (half a block for the hash, a quarter
// for the comparison) at a time through a ring of three shared-memory stages,
// warps 0-3 keeping the bulk copies (a quarter of each unit from each warp)
// two stages ahead while all threads combine the current one.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kBStages = 3;
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

// The stage pipeline of one CTA over items blockIdx.x, +gridDim.x, ... < n,
// each item kSrc blocks read as kUnits equal units (the unit of a stage).
template <int kSrc, int kUnits>
struct Ring {
  uint32_t sbuf, bars;   // shared addresses: stages, then kBStages mbarriers
  uint32_t unit;         // bytes of one unit of a block
  int n;

  __device__ int item(int u) const { return blockIdx.x + (u / kUnits) * gridDim.x; }

  // Called by lane 0 of warps 0-3 (part = warp): each copies quarter `part`
  // of every source's unit; warp 0 also arms the stage's barrier.
  __device__ void issue(const uint8_t* cache, const int32_t* const* ids, int num_blocks, int u, int part) const {
    const int it = item(u);
    if (it >= n) return;
    const int s = u % kBStages;
    const uint32_t q = unit / 4;
    uint32_t bytes = 0;
    int blk[kSrc];
#pragma unroll
    for (int k = 0; k < kSrc; ++k) {
      blk[k] = __ldg(ids[k] + it);
      if (blk[k] >= 0 && blk[k] < num_blocks) bytes += unit;
    }
    if (part == 0) mbar_arrive_expect_tx(bars + 8 * s, bytes);
#pragma unroll
    for (int k = 0; k < kSrc; ++k)
      if (blk[k] >= 0 && blk[k] < num_blocks)
        bulk_load(sbuf + s * kSrc * unit + k * unit + part * q,
                  cache + (int64_t)blk[k] * kUnits * unit + (u % kUnits) * unit + part * q, q, bars + 8 * s);
  }
};

__device__ __forceinline__ int units_of_cta(int n, int units) {
  const int items = n > (int)blockIdx.x ? (n - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  return units * items;
}

// kChunks: 16-byte chunks per thread in half a block (2304 / 256 = 9 for bf16 rows, 1280 / 256 = 5 for FP8).
template <int kChunks>
__global__ void __launch_bounds__(256) block_hash_kernel(const uint8_t* __restrict__ cache, int num_blocks,
                                                         const int32_t* __restrict__ ids, int n,
                                                         uint64_t* __restrict__ hashes, uint32_t* err) {
  constexpr int kThreads = 256, kUnits = 2;
  extern __shared__ __align__(128) uint8_t sbuf[];
  __shared__ __align__(8) uint64_t bars[kBStages];
  __shared__ uint64_t part[kThreads / 32];
  constexpr uint32_t kUnit = 16u * kChunks * kThreads;
  constexpr uint64_t kWords = kUnits * kUnit / 8;   // words in a whole block
  Ring<1, kUnits> ring{smem_u32(sbuf), smem_u32(bars), kUnit, n};
  const int32_t* idp[1] = {ids};
  const int nu = units_of_cta(n, kUnits);
  const bool issuer = (threadIdx.x & 31) == 0 && threadIdx.x < 128;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBStages; ++s) mbar_init(smem_u32(bars) + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (issuer)
    for (int u = 0; u < kBStages && u < nu; ++u) ring.issue(cache, idp, num_blocks, u, threadIdx.x >> 5);
  uint64_t acc = 0;
  bool landed = true;
  for (int u = 0; u < nu; ++u) {
    const int s = u % kBStages;
    landed &= mbar_wait(smem_u32(bars) + 8 * s, (u / kBStages) & 1);
    const int it = ring.item(u);
    const int b = __ldg(ids + it);
    const bool ok = b >= 0 && b < num_blocks;
    if (ok) {
      // chunk q of the block holds words 2q, 2q + 1; c = (2q + 1) gamma, stepped by 2 * kThreads * gamma
      uint64_t c = (2 * (uint64_t)(threadIdx.x + (u % kUnits) * (kChunks * kThreads)) + 1) * kGamma;
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        uint32_t v[4];
        lds128(smem_u32(sbuf) + s * kUnit + 16 * (threadIdx.x + k * kThreads), v);
        const uint64_t w0 = ((uint64_t)v[1] << 32) | v[0], w1 = ((uint64_t)v[3] << 32) | v[2];
        acc += mix64(w0 + c) + mix64(w1 + c + kGamma);
        c += 2 * kThreads * kGamma;
      }
    }
    __syncthreads();   // every thread is done with stage s
    if (issuer && u + kBStages < nu) ring.issue(cache, idp, num_blocks, u + kBStages, threadIdx.x >> 5);
    if (u % kUnits == kUnits - 1) {
      acc = warp_sum64(acc);
      if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
      __syncthreads();
      if (threadIdx.x == 0) {
        uint64_t t = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) t += part[w];
        hashes[it] = (ok && landed) ? mix64(kWords ^ t) : 0ull;
        if (err != nullptr && !ok) atomicOr(err, kErrBadBlock);
        if (err != nullptr && ok && !landed) atomicOr(err, kErrTimeout);
      }
      acc = 0;
    }
  }
}

// kChunks: 16-byte chunks per thread in a quarter block (1152 / 128 = 9 for bf16 rows, 640 / 128 = 5 for FP8).
template <int kChunks>
__global__ void __launch_bounds__(128) block_compare_kernel(const uint8_t* __restrict__ cache, int num_blocks,
                                                            const int32_t* __restrict__ ia,
                                                            const int32_t* __restrict__ ib, int n,
                                                            int32_t* __restrict__ equal, uint32_t* err) {
  constexpr int kThreads = 128, kUnits = 4;
  extern __shared__ __align__(128) uint8_t sbuf[];
  __shared__ __align__(8) uint64_t bars[kBStages];
  constexpr uint32_t kUnit = 16u * kChunks * kThreads;
  Ring<2, kUnits> ring{smem_u32(sbuf), smem_u32(bars), kUnit, n};
  const int32_t* idp[2] = {ia, ib};
  const int nu = units_of_cta(n, kUnits);
  const bool issuer = (threadIdx.x & 31) == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kBStages; ++s) mbar_init(smem_u32(bars) + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (issuer)
    for (int u = 0; u < kBStages && u < nu; ++u) ring.issue(cache, idp, num_blocks, u, threadIdx.x >> 5);
  uint32_t diff = 0;
  bool landed = true;
  for (int u = 0; u < nu; ++u) {
    const int s = u % kBStages;
    landed &= mbar_wait(smem_u32(bars) + 8 * s, (u / kBStages) & 1);
    const int it = ring.item(u);
    const int a = __ldg(ia + it), b = __ldg(ib + it);
    const bool ok = a >= 0 && a < num_blocks && b >= 0 && b < num_blocks;
    if (ok) {
      const uint32_t base = smem_u32(sbuf) + s * 2 * kUnit;
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        const uint32_t off = 16u * (threadIdx.x + k * kThreads);
        uint32_t x[4], y[4];
        lds128(base + off, x);
        lds128(base + kUnit + off, y);
        diff |= (x[0] ^ y[0]) | (x[1] ^ y[1]) | (x[2] ^ y[2]) | (x[3] ^ y[3]);
      }
    }
    const int any = __syncthreads_or(diff != 0u);   // also: every thread is done with stage s
    if (issuer && u + kBStages < nu) ring.issue(cache, idp, num_blocks, u + kBStages, threadIdx.x >> 5);
    if (u % kUnits == kUnits - 1) {
      if (threadIdx.x == 0) {
        equal[it] = (ok && landed) ? (any ? 0 : 1) : -1;
        if (err != nullptr && !ok) atomicOr(err, kErrBadBlock);
        if (err != nullptr && ok && !landed) atomicOr(err, kErrTimeout);
      }
      diff = 0;
    }
  }
}

int persistent_grid(int n, int ctas_per_sm) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int cap = sms * ctas_per_sm;
  return n < cap ? n : cap;
}

// Opts the four kernels into their dynamic shared memory, once per device
// (the attribute call is not free, and it belongs outside a timed launch).
cudaError_t configure_blocks() {
  static int configured_device = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || configured_device == dev) return e;
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  if (e == cudaSuccess) e = cudaFuncSetAttribute(block_hash_kernel<5>, a, kBStages * 20480);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(block_hash_kernel<9>, a, kBStages * 36864);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(block_compare_kernel<5>, a, kBStages * 2 * 10240);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(block_compare_kernel<9>, a, kBStages * 2 * 18432);
  if (e == cudaSuccess) configured_device = dev;
  return e;
}

}  // namespace

cudaError_t launch_block_hash(const uint8_t* cache, int fp8, int num_blocks, const int32_t* ids, int n,
                              uint64_t* hashes, uint32_t* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const cudaError_t e = configure_blocks();
  if (e != cudaSuccess) return e;
  if (fp8) {
    constexpr int kSmem = kBStages * 20480;
    block_hash_kernel<5><<<persistent_grid(n, 3), 256, kSmem, s>>>(cache, num_blocks, ids, n, hashes, err);
  } else {
    constexpr int kSmem = kBStages * 36864;
    block_hash_kernel<9><<<persistent_grid(n, 2), 256, kSmem, s>>>(cache, num_blocks, ids, n, hashes, err);
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_block_compare(const uint8_t* cache, int fp8, int num_blocks, const int32_t* a, const int32_t* b,
                                 int n, int32_t* equal, uint32_t* err, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const cudaError_t e = configure_blocks();
  if (e != cudaSuccess) return e;
  if (fp8) {
    constexpr int kSmem = kBStages * 2 * 10240;
    block_compare_kernel<5><<<persistent_grid(n, 3), 128, kSmem, s>>>(cache, num_blocks, a, b, n, equal, err);
  } else {
    constexpr int kSmem = kBStages * 2 * 18432;
    block_compare_kernel<9><<<persistent_grid(n, 2), 128, kSmem, s>>>(cache, num_blocks, a, b, n, equal, err);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
