// Query-side RoPE relocation ("RedKnot-MLA: Multi-Head Offline-Online Reuse for
// DeepSeek-V4 Long-Context Serving", section 2, "Online position restoration
// and merge"): the queries are rotated into a document's canonical frame so
// they can attend to k_rope cached at canonical positions.  Pair k of the 64
// RoPE columns, (x[2k], x[2k+1]), turns by (pos - offset) * theta^(-2k/64).
//
// One thread per (token, 8-column chunk, group of 4 heads): the thread
// computes its four angles once, loads its 16-byte chunk of each of the 4
// heads h, h+Q, h+2Q, h+3Q (Q = ceil(heads/4)) before storing any, and eight
// consecutive threads cover one (token, head) RoPE part = 128 contiguous
// bytes.  Each thread writes only the bytes it read, so y may equal x.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

struct RopeArgs {
  uint64_t frac[kDr / 2];
};

constexpr int kHeadsPerThread = 4;

__global__ void __launch_bounds__(256) rope_kernel(const uint16_t* x, const int32_t* __restrict__ pos,
                                                   int64_t offset, const __grid_constant__ RopeArgs a,
                                                   uint16_t* y, int tokens, int heads, int row_stride,
                                                   int rope_col) {
  const int hq = (heads + kHeadsPerThread - 1) / kHeadsPerThread;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int c = (int)(gid & 7);
  const int64_t th = gid >> 3;
  const int64_t t = th / hq;
  const int h0 = (int)(th - t * hq);
  if (t >= tokens) return;
  const int64_t delta = (int64_t)__ldg(pos + t) - offset;
  uint4 v[kHeadsPerThread];
#pragma unroll
  for (int j = 0; j < kHeadsPerThread; ++j) {
    const int h = h0 + j * hq;
    if (h < heads) v[j] = *reinterpret_cast<const uint4*>(x + (t * heads + h) * row_stride + rope_col + c * 8);
  }
  float sn[4], cs[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) rope_sincos(delta, a.frac[c * 4 + i], &sn[i], &cs[i]);
#pragma unroll
  for (int j = 0; j < kHeadsPerThread; ++j) {
    const int h = h0 + j * hq;
    if (h >= heads) continue;
    uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float x0 = __uint_as_float(w[i] << 16);
      const float x1 = __uint_as_float(w[i] & 0xFFFF0000u);
      w[i] = pack_bf16(x0 * cs[i] - x1 * sn[i], x0 * sn[i] + x1 * cs[i]);
    }
    *reinterpret_cast<uint4*>(y + (t * heads + h) * row_stride + rope_col + c * 8) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_rope(const uint16_t* x, const int32_t* pos, int64_t offset, const uint64_t* frac_host,
                        uint16_t* y, int tokens, int heads, int row_stride, int rope_col, cudaStream_t s) {
  if (tokens == 0 || heads == 0) return cudaSuccess;
  RopeArgs a;
  for (int k = 0; k < kDr / 2; ++k) a.frac[k] = frac_host[k];
  const int64_t threads = (int64_t)tokens * ((heads + kHeadsPerThread - 1) / kHeadsPerThread) * 8;
  const int blocks = (int)((threads + 255) / 256);
  rope_kernel<<<blocks, 256, 0, s>>>(x, pos, offset, a, y, tokens, heads, row_stride, rope_col);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
