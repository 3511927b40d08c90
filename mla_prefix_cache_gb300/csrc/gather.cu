// Paged latent gather, _gather_cache of "DeepSeek MLA — Prefix Cache 与 Chunked
// Prefill 深度解析", section 4.4 step 1: the rows of logical tokens of a
// request, found through its block-table row (token t in block table[t/64],
// slot t%64; 64-token blocks per "PagedAttention assumed MHA. DeepSeek-V4 says
// that assumption is broken"), written contiguously ([c_kv | k_rope] rows,
// section 5.2).
//
// The copy is driven by the bulk-copy (TMA) engine.  A destination tile is 64
// rows; its rows come from at most two cache blocks, and each block's share is
// one contiguous range of rows, so a tile is one or two cp.async.bulk loads
// into a shared-memory stage.  BF16 rows (and FP8 rows copied as stored) go
// from the stage straight back out by one cp.async.bulk store; FP8 rows to be
// dequantised are converted by the CTA's threads from the stage and stored to
// global memory in 512-byte warp stores (bf16(e4m3 * scale), round to nearest
// even; k_rope copied).  Each CTA is persistent over its tiles, one thread
// keeping the loads of the next stages (3 of 72 KB, or 5 of 40 KB) in flight.
//
// Two callers: mla_gather_latent (one request's token range, any start) and
// the fused path's pass over every block of its requests in logical order
// (whole 64-row tiles, rows past a request's length zeroed: a kernel that reads
// whole blocks multiplies them by zero weights, which must stay zero).  Rows
// of a bad block id are zeroed and set the error word.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

// kMode 0: bf16 rows copied; 1: FP8 rows dequantised to bf16; 2: FP8 rows copied as stored.
template <int kMode>
struct Cfg {
  static constexpr int kSrcRow = kMode == 0 ? kRowBytesBf16 : kRowBytesFp8;
  static constexpr int kDstRow = kMode == 1 ? kRowBytesBf16 : kSrcRow;
  static constexpr int kInStages = kMode == 0 ? 3 : 5;
  static constexpr int kOutBufs = 0;
  static constexpr int kCtasPerSm = 1;
  static constexpr int kThreads = kMode == 1 ? 1024 : 256;   // the dequantisation takes every warp the SM has
  static constexpr uint32_t kInBytes = kBlock * kSrcRow;
  static constexpr uint32_t kOutBytes = kBlock * kDstRow;
  static constexpr uint32_t kSmem = kInStages * kInBytes + kOutBufs * kOutBytes;
  static_assert(kSmem + 64 <= 232448, "shared memory");
};

// One destination tile: rows [0, rows) of it are written; rows of segment g
// ([row0, row0 + n) of the tile) come from block blk, slots slot0.. ; the
// others (a bad block id, past a request's length) are zero.
struct Tile {
  int blk[2], slot0[2], row0[2], n[2];
  int rows;
  int64_t dst_row;
};

__device__ __forceinline__ bool valid_block(int blk, int num_blocks) { return blk >= 0 && blk < num_blocks; }

// Tokens [start, start + len) of one request (mla_gather_latent).
struct RangeSrc {
  const int32_t* table;
  int start, len;
  __device__ int tiles() const { return (len + kBlock - 1) / kBlock; }
  __device__ Tile tile(int i) const {
    Tile t;
    const int g0 = i * kBlock;
    t.rows = min(kBlock, len - g0);
    t.dst_row = g0;
    const int t0 = start + g0;
    const int lb = t0 >> 6, s0 = t0 & (kBlock - 1);
    t.blk[0] = __ldg(table + lb);
    t.slot0[0] = s0;
    t.row0[0] = 0;
    t.n[0] = min(kBlock - s0, t.rows);
    t.n[1] = t.rows - t.n[0];
    t.blk[1] = t.n[1] > 0 ? __ldg(table + lb + 1) : -1;
    t.slot0[1] = 0;
    t.row0[1] = t.n[0];
    return t;
  }
};

// Every block of several requests from each one's first_block on, in logical
// order (the fused path's pass; the absorbed path's copies of each request's
// last block); passed by value, so the request list sits in the kernel's
// parameter space.
struct BlocksSrc {
  GatherBlocksParams p;
  __device__ int tiles() const { return p.total_blocks; }
  __device__ Tile tile(int gb) const {
    int lo = 0, hi = p.n_reqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.reqs[mid].base_block <= gb) lo = mid; else hi = mid - 1;
    }
    const GatherReq rq = p.reqs[lo];
    const int lb = gb - rq.base_block + rq.first_block;
    Tile t;
    t.rows = kBlock;
    t.dst_row = (int64_t)gb * kBlock;
    t.blk[0] = lb < p.max_blocks ? __ldg(p.block_table + (int64_t)rq.req * p.max_blocks + lb) : -1;
    t.slot0[0] = 0;
    t.row0[0] = 0;
    t.n[0] = max(0, min(kBlock, rq.seq_len - lb * kBlock));
    t.blk[1] = -1;
    t.slot0[1] = t.row0[1] = t.n[1] = 0;
    return t;
  }
};

template <int kMode>
__device__ __forceinline__ void issue_tile(const Tile& t, const uint8_t* cache, int num_blocks, uint32_t stage,
                                           uint32_t bar) {
  using C = Cfg<kMode>;
  uint32_t bytes = 0;
#pragma unroll
  for (int g = 0; g < 2; ++g)
    if (t.n[g] > 0 && valid_block(t.blk[g], num_blocks)) bytes += (uint32_t)t.n[g] * C::kSrcRow;
  if (bytes == 0) {
    mbar_arrive(bar);
    return;
  }
  mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
  for (int g = 0; g < 2; ++g)
    if (t.n[g] > 0 && valid_block(t.blk[g], num_blocks))
      bulk_load(stage + (uint32_t)t.row0[g] * C::kSrcRow,
                cache + ((int64_t)t.blk[g] * kBlock + t.slot0[g]) * C::kSrcRow, (uint32_t)t.n[g] * C::kSrcRow, bar);
}

// Whether tile row r is read from the cache (else it is written as zeros).
__device__ __forceinline__ bool row_loaded(const Tile& t, int r, int num_blocks) {
#pragma unroll
  for (int g = 0; g < 2; ++g)
    if (r >= t.row0[g] && r < t.row0[g] + t.n[g]) return valid_block(t.blk[g], num_blocks);
  return false;
}

template <int kMode, class Src>
__global__ void __launch_bounds__(Cfg<kMode>::kThreads, 1)
    gather_tma_kernel(const __grid_constant__ Src src, const uint8_t* __restrict__ cache, int num_blocks, float scale,
                      uint8_t* dst, uint32_t* err) {
  using C = Cfg<kMode>;
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[C::kInStages];
  const int tid = threadIdx.x;
  const int n_tiles = src.tiles();
  const int mine = n_tiles > (int)blockIdx.x ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  const uint32_t sb = smem_u32(smem), bb = smem_u32(bars);
  if (tid == 0) {
    for (int s = 0; s < C::kInStages; ++s) mbar_init(bb + 8 * s, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int k = 0; k < C::kInStages && k < mine; ++k)
      issue_tile<kMode>(src.tile(blockIdx.x + k * gridDim.x), cache, num_blocks, sb + k * C::kInBytes, bb + 8 * k);
  bool landed = true;
  for (int k = 0; k < mine; ++k) {
    const int s = k % C::kInStages;
    const uint32_t stage = sb + s * C::kInBytes;
    const Tile t = src.tile(blockIdx.x + k * gridDim.x);
    landed &= mbar_wait(bb + 8 * s, (k / C::kInStages) & 1);
    if (tid == 0 && err != nullptr) {
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (t.n[g] > 0 && !valid_block(t.blk[g], num_blocks)) atomicOr(err, kErrBadBlock);
    }
    if constexpr (kMode == 1) {
      // dequantised from the stage straight to global memory: each warp store
      // is 512 contiguous bytes of the destination rows
      constexpr int kRowChunks = kRowBytesBf16 / 16;   // 72 output chunks of 16 bytes a row
      uint4* out = reinterpret_cast<uint4*>(dst + t.dst_row * kRowBytesBf16);
      for (int q = tid; q < t.rows * kRowChunks; q += C::kThreads) {
        const int r = q / kRowChunks, c = q - r * kRowChunks;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (row_loaded(t, r, num_blocks)) {
          const uint32_t row = stage + (uint32_t)r * kRowBytesFp8;
          if (c < kDc / 8) {
            const uint2 b = lds64(row + 8 * c);
            w[0] = e4m3x2_scaled_bf16x2(b.x, scale);
            w[1] = e4m3x2_scaled_bf16x2(b.x >> 16, scale);
            w[2] = e4m3x2_scaled_bf16x2(b.y, scale);
            w[3] = e4m3x2_scaled_bf16x2(b.y >> 16, scale);
          } else {
            lds128(row + kDc + 16 * (c - kDc / 8), w);
          }
        }
        out[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
      __syncthreads();   // every thread is done with the stage
      if (tid == 0 && k + C::kInStages < mine)
        issue_tile<kMode>(src.tile(blockIdx.x + (k + C::kInStages) * gridDim.x), cache, num_blocks, stage,
                          bb + 8 * s);
    } else {
      // rows not loaded are zeroed in the stage itself, which is then stored as it is
      constexpr int kRowChunks = C::kSrcRow / 16;
      for (int q = tid; q < kBlock * kRowChunks; q += C::kThreads) {
        const int r = q / kRowChunks;
        if (r < t.rows && !row_loaded(t, r, num_blocks)) sts128(stage + 16 * q, 0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();   // the threads' shared-memory writes, to the bulk store
      __syncthreads();
      if (tid == 0) {
        bulk_store(dst + t.dst_row * C::kDstRow, stage, (uint32_t)t.rows * C::kDstRow);
        bulk_commit();
        if (k + C::kInStages < mine) {
          bulk_wait_read0();   // the stage is free once its store has read it
          issue_tile<kMode>(src.tile(blockIdx.x + (k + C::kInStages) * gridDim.x), cache, num_blocks, stage,
                            bb + 8 * s);
        }
      }
    }
  }
  if (tid == 0) bulk_wait0();   // every store complete before the CTA's shared memory goes
  if (!landed && err != nullptr) atomicOr(err, kErrTimeout);
}

template <int kMode, class Src>
cudaError_t launch_tma(const Src& src, int tiles, const uint8_t* cache, int num_blocks, float scale, uint8_t* dst,
                       uint32_t* err, cudaStream_t s) {
  if (tiles == 0) return cudaSuccess;
  static int configured = -1;
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (configured != dev) {
    e = cudaFuncSetAttribute(gather_tma_kernel<kMode, Src>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Cfg<kMode>::kSmem);
    if (e != cudaSuccess) return e;
    configured = dev;
  }
  const int grid = tiles < sms * Cfg<kMode>::kCtasPerSm ? tiles : sms * Cfg<kMode>::kCtasPerSm;
  gather_tma_kernel<kMode, Src><<<grid, Cfg<kMode>::kThreads, Cfg<kMode>::kSmem, s>>>(src, cache, num_blocks, scale,
                                                                                    dst, err);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_blocks(const GatherBlocksParams& p, cudaStream_t s) {
  const BlocksSrc src{p};
  return p.fp8 ? launch_tma<1>(src, p.total_blocks, p.cache, p.num_blocks, p.scale, reinterpret_cast<uint8_t*>(p.dst),
                               p.err, s)
               : launch_tma<0>(src, p.total_blocks, p.cache, p.num_blocks, 1.f, reinterpret_cast<uint8_t*>(p.dst),
                               p.err, s);
}

cudaError_t launch_gather_blocks_raw(const GatherBlocksParams& p, cudaStream_t s) {
  const BlocksSrc src{p};
  return launch_tma<2>(src, p.total_blocks, p.cache, p.num_blocks, 1.f, reinterpret_cast<uint8_t*>(p.dst), p.err, s);
}

cudaError_t launch_gather(const uint8_t* cache, int fp8, float scale, int num_blocks, const int32_t* table_row,
                          int max_blocks, int start, int len, uint16_t* dst, uint32_t* err, cudaStream_t s) {
  (void)max_blocks;
  const RangeSrc src{table_row, start, len};
  const int tiles = (len + kBlock - 1) / kBlock;
  return fp8 ? launch_tma<1>(src, tiles, cache, num_blocks, scale, reinterpret_cast<uint8_t*>(dst), err, s)
             : launch_tma<0>(src, tiles, cache, num_blocks, 1.f, reinterpret_cast<uint8_t*>(dst), err, s);
}

}  // namespace mla
