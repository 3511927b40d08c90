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
// One thread per 16-byte output chunk (72 per row): consecutive threads write
// consecutive chunks, so each warp stores 512 contiguous bytes.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kChunksPerRow = kRowBytesBf16 / 16;  // 72

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
  float v;
  if (e == 15u && m == 7u) v = __int_as_float(0x7FC00000);
  else if (e == 0u) v = (float)m * 0.001953125f;  // m * 2^-9
  else v = __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (c & 0x80u) ? -v : v;
}

__global__ void __launch_bounds__(256) gather_kernel(const uint8_t* __restrict__ cache, int fp8, float scale,
                                                     int num_blocks, const int32_t* __restrict__ table,
                                                     int start, int len, uint16_t* __restrict__ dst,
                                                     uint32_t* err) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t i = gid / kChunksPerRow;
  const int c = (int)(gid - i * kChunksPerRow);
  if (i >= len) return;
  const int t = start + (int)i;
  const int blk = __ldg(table + (t >> 6));
  uint4 v = make_uint4(0, 0, 0, 0);
  if (blk < 0 || blk >= num_blocks) {
    if (err != nullptr && c == 0) atomicOr(err, kErrBadBlock);
  } else {
    const int64_t row = (int64_t)blk * kBlock + (t & 63);
    if (!fp8) {
      v = __ldg(reinterpret_cast<const uint4*>(cache + row * kRowBytesBf16) + c);
    } else {
      const uint8_t* rp = cache + row * kRowBytesFp8;
      if (c < 64) {  // 8 latent values from 8 bytes
        const uint2 b = __ldg(reinterpret_cast<const uint2*>(rp) + c);
        uint32_t w[2] = {b.x, b.y}, o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t src = w[k >> 1] >> ((k & 1) * 16);
          o[k] = pack_bf16(e4m3_value(src & 0xFFu) * scale, e4m3_value((src >> 8) & 0xFFu) * scale);
        }
        v = make_uint4(o[0], o[1], o[2], o[3]);
      } else {       // k_rope bf16, copied
        v = __ldg(reinterpret_cast<const uint4*>(rp + kDc) + (c - 64));
      }
    }
  }
  reinterpret_cast<uint4*>(dst + i * kRowBf16)[c] = v;
}

// Every block of several requests into one contiguous bf16 buffer: request i's
// logical block lb becomes rows (base_i + lb) * 64 .. +63 of dst.
__global__ void __launch_bounds__(256) gather_blocks_kernel(const __grid_constant__ GatherBlocksParams p) {
  const int64_t total_chunks = (int64_t)p.total_blocks * kBlock * kChunksPerRow;
  for (int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; gid < total_chunks;
       gid += (int64_t)gridDim.x * blockDim.x) {
    const int64_t g = gid / kChunksPerRow;              // destination row
    const int c = (int)(gid - g * kChunksPerRow);
    const int gb = (int)(g >> 6);                       // destination block
    int lo = 0, hi = p.n_reqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.reqs[mid].base_block <= gb) lo = mid; else hi = mid - 1;
    }
    const GatherReq rq = p.reqs[lo];
    const int lb = gb - rq.base_block;
    const int slot = (int)(g & 63);
    const int blk = (lb < p.max_blocks) ? __ldg(p.block_table + (int64_t)rq.req * p.max_blocks + lb) : -1;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (blk < 0 || blk >= p.num_blocks) {
      if (c == 0 && slot == 0 && lb * kBlock < rq.seq_len) atomicOr(p.err, kErrBadBlock);
    } else {
      const int64_t row = (int64_t)blk * kBlock + slot;
      if (!p.fp8) {
        v = __ldg(reinterpret_cast<const uint4*>(p.cache + row * kRowBytesBf16) + c);
      } else {
        const uint8_t* rp = p.cache + row * kRowBytesFp8;
        if (c < 64) {
          const uint2 b = __ldg(reinterpret_cast<const uint2*>(rp) + c);
          uint32_t w[2] = {b.x, b.y}, o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t src = w[k >> 1] >> ((k & 1) * 16);
            o[k] = pack_bf16(e4m3_value(src & 0xFFu) * p.scale, e4m3_value((src >> 8) & 0xFFu) * p.scale);
          }
          v = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
          v = __ldg(reinterpret_cast<const uint4*>(rp + kDc) + (c - 64));
        }
      }
    }
    reinterpret_cast<uint4*>(p.dst + g * kRowBf16)[c] = v;
  }
}

}  // namespace

cudaError_t launch_gather_blocks(const GatherBlocksParams& p, cudaStream_t s) {
  if (p.total_blocks == 0) return cudaSuccess;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t threads = (int64_t)p.total_blocks * kBlock * kChunksPerRow;
  const int64_t blocks = (threads + 255) / 256;
  const int grid = (int)(blocks < (int64_t)sms * 8 ? blocks : (int64_t)sms * 8);
  gather_blocks_kernel<<<grid, 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint8_t* cache, int fp8, float scale, int num_blocks, const int32_t* table_row,
                          int max_blocks, int start, int len, uint16_t* dst, uint32_t* err, cudaStream_t s) {
  (void)max_blocks;
  if (len == 0) return cudaSuccess;
  const int64_t threads = (int64_t)len * kChunksPerRow;
  const int blocks = (int)((threads + 255) / 256);
  gather_kernel<<<blocks, 256, 0, s>>>(cache, fp8, scale, num_blocks, table_row, start, len, dst, err);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
