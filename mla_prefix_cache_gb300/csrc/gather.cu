// Paged latent gather, _gather_cache of "DeepSeek MLA — Prefix Cache 与 Chunked
// Prefill 深度解析", section 4.4 step 1: the rows of logical tokens
// [start, start+len) of one request, found through its block-table row (token t
// in block table[t/64], slot t%64; 64-token blocks per "PagedAttention assumed
// MHA. DeepSeek-V4 says that assumption is broken"), written contiguously as
// 576 bf16 values [c_kv | k_rope] (section 5.2 row layout).
//
// BF16 rows are copied bit-exactly.  FP8 rows (512 E4M3FN bytes + 64 bf16) are
// dequantised to bf16(e4m3 * scale), rounded to nearest even.
//
// Work is cut into tiles of 64 destination rows (72 KB of bf16 output).  One
// 256-thread CTA moves a tile: thread i owns chunks i, i+256, ..., i+17*256 of
// the tile's 4608 16-byte output chunks, issues all 18 loads before any store
// (about 73 KB in flight per CTA, which is what keeps HBM busy), and
// consecutive threads touch consecutive chunks, so every warp access is 512
// contiguous bytes.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kChunksPerRow = kRowBytesBf16 / 16;  // 72
constexpr int kGatherThreads = 256;
constexpr int kChunksPerThread = kBlock * kChunksPerRow / kGatherThreads;  // 18
static_assert(kChunksPerThread * kGatherThreads == kBlock * kChunksPerRow, "tile split");

// Chunk c (0..71) of a cache row: BF16 rows are 72 chunks of 16 bytes; an FP8
// row's chunk c < 64 is 8 e4m3 bytes (expanded to 16 bytes of bf16 later) and
// chunk c >= 64 is 16 bytes of its bf16 k_rope.
__device__ __forceinline__ uint4 load_chunk(const uint8_t* row, int c, int fp8) {
  if (!fp8) return __ldg(reinterpret_cast<const uint4*>(row) + c);
  if (c < 64) {
    const uint2 b = __ldg(reinterpret_cast<const uint2*>(row) + c);
    return make_uint4(b.x, b.y, 0u, 0u);
  }
  return __ldg(reinterpret_cast<const uint4*>(row + kDc) + (c - 64));
}

__device__ __forceinline__ uint4 finish_chunk(uint4 v, int c, int fp8, float scale) {
  if (!fp8 || c >= 64) return v;
  return make_uint4(e4m3x2_scaled_bf16x2(v.x, scale), e4m3x2_scaled_bf16x2(v.x >> 16, scale),
                    e4m3x2_scaled_bf16x2(v.y, scale), e4m3x2_scaled_bf16x2(v.y >> 16, scale));
}

// Tokens [start, start+len) of one request.  The tile's rows may straddle two
// cache blocks, so each chunk looks up its own block (the table row is cached).
__global__ void __launch_bounds__(kGatherThreads, 2) gather_kernel(const uint8_t* __restrict__ cache, int fp8,
                                                                   float scale, int num_blocks,
                                                                   const int32_t* __restrict__ table, int start,
                                                                   int len, uint16_t* __restrict__ dst,
                                                                   uint32_t* err) {
  const int64_t row_bytes = fp8 ? kRowBytesFp8 : kRowBytesBf16;
  const int tiles = (len + kBlock - 1) / kBlock;
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    uint4 v[kChunksPerThread];
    bool ok[kChunksPerThread];
#pragma unroll
    for (int j = 0; j < kChunksPerThread; ++j) {
      const int k = threadIdx.x + j * kGatherThreads;
      const int r = k / kChunksPerRow, c = k - r * kChunksPerRow;
      const int g = tile * kBlock + r;
      v[j] = make_uint4(0u, 0u, 0u, 0u);
      ok[j] = false;
      if (g < len) {
        const int t = start + g;
        const int blk = __ldg(table + (t >> 6));
        ok[j] = (blk >= 0 && blk < num_blocks);
        if (ok[j]) v[j] = load_chunk(cache + ((int64_t)blk * kBlock + (t & 63)) * row_bytes, c, fp8);
        else if (c == 0 && err != nullptr) atomicOr(err, kErrBadBlock);
      }
    }
#pragma unroll
    for (int j = 0; j < kChunksPerThread; ++j) {
      const int k = threadIdx.x + j * kGatherThreads;
      const int r = k / kChunksPerRow, c = k - r * kChunksPerRow;
      const int g = tile * kBlock + r;
      if (g < len)
        reinterpret_cast<uint4*>(dst + (int64_t)g * kRowBf16)[c] = ok[j] ? finish_chunk(v[j], c, fp8, scale) : v[j];
    }
  }
}

// Every block of several requests into one contiguous bf16 buffer: request i's
// logical block lb becomes rows (base_i + lb) * 64 .. +63 of dst.  A tile is
// one destination block, so it reads one whole cache block (72 KB of BF16 or
// 40 KB of FP8, contiguous in the pool) and the lookup is uniform over the CTA.
__global__ void __launch_bounds__(kGatherThreads, 2) gather_blocks_kernel(const __grid_constant__ GatherBlocksParams p) {
  const int64_t row_bytes = p.fp8 ? kRowBytesFp8 : kRowBytesBf16;
  for (int gb = blockIdx.x; gb < p.total_blocks; gb += gridDim.x) {
    int lo = 0, hi = p.n_reqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.reqs[mid].base_block <= gb) lo = mid; else hi = mid - 1;
    }
    const GatherReq rq = p.reqs[lo];
    const int lb = gb - rq.base_block;
    const int blk = (lb < p.max_blocks) ? __ldg(p.block_table + (int64_t)rq.req * p.max_blocks + lb) : -1;
    const bool ok = (blk >= 0 && blk < p.num_blocks);
    if (!ok && threadIdx.x == 0 && lb * kBlock < rq.seq_len) atomicOr(p.err, kErrBadBlock);
    const uint8_t* src = p.cache + (int64_t)(ok ? blk : 0) * kBlock * row_bytes;
    uint16_t* out = p.dst + (int64_t)gb * kBlock * kRowBf16;
    // slots past the request's length are zeroed: a kernel that reads a
    // whole block multiplies them by zero weights, which must stay zero
    const int live_rows = min(kBlock, rq.seq_len - lb * kBlock);
    uint4 v[kChunksPerThread];
#pragma unroll
    for (int j = 0; j < kChunksPerThread; ++j) {
      const int k = threadIdx.x + j * kGatherThreads;
      const int r = k / kChunksPerRow, c = k - r * kChunksPerRow;
      v[j] = (ok && r < live_rows) ? load_chunk(src + r * row_bytes, c, p.fp8) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kChunksPerThread; ++j) {
      const int k = threadIdx.x + j * kGatherThreads;
      const int r = k / kChunksPerRow, c = k - r * kChunksPerRow;
      reinterpret_cast<uint4*>(out)[k] = (ok && r < live_rows) ? finish_chunk(v[j], c, p.fp8, p.scale) : v[j];
    }
  }
}

// The FP8 rows of every block, as stored (640 B: 512 E4M3 codes, then k_rope
// as bf16), in the same logical order as gather_blocks_kernel; slots past a
// request's length and blocks with a bad id are zeroed, and a bad id of a
// block the request uses sets the error word.
__global__ void __launch_bounds__(kGatherThreads, 2) gather_blocks_raw_kernel(const __grid_constant__ GatherBlocksParams p) {
  constexpr int kChunks = kBlock * kRowBytesFp8 / 16;   // 2560 per block
  constexpr int kRowChunks = kRowBytesFp8 / 16;         // 40
  for (int gb = blockIdx.x; gb < p.total_blocks; gb += gridDim.x) {
    int lo = 0, hi = p.n_reqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.reqs[mid].base_block <= gb) lo = mid; else hi = mid - 1;
    }
    const GatherReq rq = p.reqs[lo];
    const int lb = gb - rq.base_block;
    const int blk = (lb < p.max_blocks) ? __ldg(p.block_table + (int64_t)rq.req * p.max_blocks + lb) : -1;
    const bool ok = (blk >= 0 && blk < p.num_blocks);
    if (!ok && threadIdx.x == 0 && lb * kBlock < rq.seq_len && p.err != nullptr) atomicOr(p.err, kErrBadBlock);
    const int live_rows = min(kBlock, rq.seq_len - lb * kBlock);
    const uint4* src = reinterpret_cast<const uint4*>(p.cache + (int64_t)(ok ? blk : 0) * kBlock * kRowBytesFp8);
    uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.dst) + (int64_t)gb * kBlock * kRowBytesFp8);
    for (int k = threadIdx.x; k < kChunks; k += kGatherThreads)
      dst[k] = (ok && k / kRowChunks < live_rows) ? __ldg(src + k) : make_uint4(0u, 0u, 0u, 0u);
  }
}

int gather_grid(int64_t tiles) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t cap = (int64_t)sms * 2;  // two resident CTAs per SM, each looping over tiles
  return (int)(tiles < cap ? tiles : cap);
}

}  // namespace

cudaError_t launch_gather_blocks(const GatherBlocksParams& p, cudaStream_t s) {
  if (p.total_blocks == 0) return cudaSuccess;
  gather_blocks_kernel<<<gather_grid(p.total_blocks), kGatherThreads, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather_blocks_raw(const GatherBlocksParams& p, cudaStream_t s) {
  if (p.total_blocks == 0) return cudaSuccess;
  gather_blocks_raw_kernel<<<gather_grid(p.total_blocks), kGatherThreads, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint8_t* cache, int fp8, float scale, int num_blocks, const int32_t* table_row,
                          int max_blocks, int start, int len, uint16_t* dst, uint32_t* err, cudaStream_t s) {
  (void)max_blocks;
  if (len == 0) return cudaSuccess;
  gather_kernel<<<gather_grid((len + kBlock - 1) / kBlock), kGatherThreads, 0, s>>>(cache, fp8, scale, num_blocks,
                                                                                      table_row, start, len, dst, err);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
