// merge_attn_states ("DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析",
// section 4.3): the LSE-weighted average of partial attention states,
//   m = max_i lse_i;  w_i = e^(lse_i - m);  out = sum_i w_i out_i / sum_i w_i;
//   lse = m + ln(sum_i w_i),
// with (0, -inf) for a row whose every state is empty.  The two-state form is
// the pages' operation; the n-state form folds a request's KV splits (its
// context chunks and extend stage) in one pass, which equals the pages'
// sequential fold up to rounding.
//
// One warp per (row, head) of W values (W = 128 for attention outputs, 512 for
// the latent states of the absorbed path): lane i owns float4 columns
// i, i + 32, ..., so every load/store is a 16-byte vector and a warp moves 512
// contiguous bytes per access.  The output may alias slot 0 of the states:
// each lane writes only the columns it read, after a warp barrier.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kWarpsPerBlock = 8;

template <int W>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_slots_kernel(const __grid_constant__ MergeParams p) {
  constexpr int kV = W / 128;   // float4 columns per lane
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int H = p.num_heads;
  const int64_t total = (int64_t)p.total_rows * H;
  for (int64_t item = wid; item < total; item += (int64_t)gridDim.x * kWarpsPerBlock) {
    // item -> (range, row within range, head); ranges are consecutive in item space
    const int64_t local = item / H;
    const int h = (int)(item - local * H);
    int lo = 0, hi = p.num_ranges - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.ranges[mid].prefix <= local) lo = mid; else hi = mid - 1;
    }
    const int ri = lo;
    const int64_t row = p.ranges[ri].row_begin + (local - p.ranges[ri].prefix);
    const int ns = p.ranges[ri].nslots;

    float m = -INFINITY;
#pragma unroll 4
    for (int s = 0; s < ns; ++s) m = fmaxf(m, __ldg(p.part_lse + ((int64_t)s * p.slot_stride_rows + row) * H + h));
    float4 acc[kV];
#pragma unroll
    for (int v = 0; v < kV; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (m != -INFINITY) {
      // Predicated rather than branched, so the unrolled loads of several
      // slots are in flight together; an empty state (lse = -inf) adds 0.
#pragma unroll 4
      for (int s = 0; s < ns; ++s) {
        const int64_t g = ((int64_t)s * p.slot_stride_rows + row) * H + h;
        const float l = __ldg(p.part_lse + g);
        const bool live = (l != -INFINITY);
        const float w = live ? __expf(l - m) : 0.f;
#pragma unroll
        for (int v = 0; v < kV; ++v) {
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          if (live) o = reinterpret_cast<const float4*>(p.part_out + g * W)[lane + 32 * v];
          acc[v].x += w * o.x; acc[v].y += w * o.y; acc[v].z += w * o.z; acc[v].w += w * o.w;
        }
        wsum += w;
      }
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    const int64_t orow = row * H + h;
    __syncwarp();   // every lane has read the states (the output may alias slot 0)
#pragma unroll
    for (int v = 0; v < kV; ++v) {
      const float4 r = make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
      if (p.out_bf16) {
        uint2 b = make_uint2(pack_bf16(r.x, r.y), pack_bf16(r.z, r.w));
        reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + orow * W)[lane + 32 * v] = b;
      } else {
        reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * W)[lane + 32 * v] = r;
      }
    }
    if (lane == 0) p.lse[orow] = (wsum > 0.f) ? m + logf(wsum) : -INFINITY;
  }
}

// Two states, d_v = 128: a warp merges 4 rows at a time, an 8-lane group per
// row, each lane owning float4 columns l, l+8, l+16, l+24 of its row, so a
// lane has 8 independent 16-byte loads in flight.  out/lse may alias either
// input: each lane writes only the columns it read, and the group leader
// writes lse after the whole warp has read it.
__global__ void __launch_bounds__(256) merge2_d128_kernel(const float* oa, const float* la, const float* ob,
                                                          const float* lb, float* o, float* l, int64_t rows) {
  const int lane = threadIdx.x & 31, g = lane >> 3, q = lane & 7;
  const int64_t w0 = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  for (int64_t base = w0 * 4; base < rows; base += (int64_t)gridDim.x * 8 * 4) {
    const int64_t row = base + g;
    const bool live = row < rows;
    float a = -INFINITY, b = -INFINITY;
    float4 x[4], y[4];
    if (live) {
      a = la[row];
      b = lb[row];
      const float4* pa = reinterpret_cast<const float4*>(oa + row * kDv);
      const float4* pb = reinterpret_cast<const float4*>(ob + row * kDv);
#pragma unroll
      for (int k = 0; k < 4; ++k) { x[k] = pa[q + 8 * k]; y[k] = pb[q + 8 * k]; }
    }
    __syncwarp();
    if (live) {
      const float m = fmaxf(a, b);
      const bool empty = (m == -INFINITY);
      const float wa = (a == -INFINITY) ? 0.f : __expf(a - m);
      const float wb = (b == -INFINITY) ? 0.f : __expf(b - m);
      const float inv = empty ? 0.f : 1.f / (wa + wb);
      float4* po = reinterpret_cast<float4*>(o + row * kDv);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        po[q + 8 * k] = make_float4((wa * x[k].x + wb * y[k].x) * inv, (wa * x[k].y + wb * y[k].y) * inv,
                                    (wa * x[k].z + wb * y[k].z) * inv, (wa * x[k].w + wb * y[k].w) * inv);
      if (q == 0) l[row] = empty ? -INFINITY : m + logf(wa + wb);
    }
  }
}

// Two states, any d_v (multiple of 4): warp per row, lanes stride over float4
// columns; same aliasing rule as above.
__global__ void __launch_bounds__(256) merge2_kernel(const float* oa, const float* la,
                                                     const float* ob, const float* lb,
                                                     float* o, float* l, int64_t rows, int d_v) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  for (int64_t row = w0; row < rows; row += (int64_t)gridDim.x * 8) {
    const float a = la[row], b = lb[row];
    const float m = fmaxf(a, b);
    const bool empty = (m == -INFINITY);
    const float wa = (a == -INFINITY) ? 0.f : __expf(a - m);
    const float wb = (b == -INFINITY) ? 0.f : __expf(b - m);
    const float inv = empty ? 0.f : 1.f / (wa + wb);
    const float4* pa = reinterpret_cast<const float4*>(oa + row * d_v);
    const float4* pb = reinterpret_cast<const float4*>(ob + row * d_v);
    float4* po = reinterpret_cast<float4*>(o + row * d_v);
    __syncwarp();
    for (int c = lane; c < d_v / 4; c += 32) {
      const float4 x = pa[c], y = pb[c];
      po[c] = make_float4((wa * x.x + wb * y.x) * inv, (wa * x.y + wb * y.y) * inv,
                          (wa * x.z + wb * y.z) * inv, (wa * x.w + wb * y.w) * inv);
    }
    __syncwarp();
    if (lane == 0) l[row] = empty ? -INFINITY : m + logf(wa + wb);
  }
}

int grid_for(int64_t warps_needed, int warps_per_block) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (warps_needed + warps_per_block - 1) / warps_per_block;
  const int64_t cap = (int64_t)sms * 16;
  return (int)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_merge_slots(const MergeParams& p, cudaStream_t s) {
  const int64_t items = (int64_t)p.total_rows * p.num_heads;
  if (items == 0) return cudaSuccess;
  merge_slots_kernel<kDv><<<grid_for(items, kWarpsPerBlock), kWarpsPerBlock * 32, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge_slots_latent(const MergeParams& p, cudaStream_t s) {
  const int64_t items = (int64_t)p.total_rows * p.num_heads;
  if (items == 0) return cudaSuccess;
  merge_slots_kernel<kDc><<<grid_for(items, kWarpsPerBlock), kWarpsPerBlock * 32, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge2(const float* oa, const float* la, const float* ob, const float* lb, float* o,
                          float* l, int64_t rows, int d_v, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (d_v == kDv)
    merge2_d128_kernel<<<grid_for((rows + 3) / 4, 8), 256, 0, s>>>(oa, la, ob, lb, o, l, rows);
  else
    merge2_kernel<<<grid_for(rows, 8), 256, 0, s>>>(oa, la, ob, lb, o, l, rows, d_v);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
