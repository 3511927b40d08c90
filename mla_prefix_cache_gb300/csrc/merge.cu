// merge_attn_states ("DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析",
// section 4.3): the LSE-weighted average of partial attention states,
//   m = max_i lse_i;  w_i = e^(lse_i - m);  out = sum_i w_i out_i / sum_i w_i;
//   lse = m + ln(sum_i w_i),
// with (0, -inf) for a row whose every state is empty.  The two-state form is
// the pages' operation; the n-state form folds a request's KV splits (its
// context chunks and extend stage) in one pass, which equals the pages'
// sequential fold up to rounding.
//
// The n-state form: an 8-lane group per (row, head) of W values (W = 128 for
// attention outputs, 512 for the latent states of the absorbed path), four
// consecutive (row, head) items per warp, so a warp reads each slot as 4 W x 4
// contiguous bytes; the lse of a row's slots is read once, one slot per lane.
// The output may alias slot 0 of the states: each lane writes only the
// columns it read, after a warp barrier.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kWarpsPerBlock = 8;

template <int W>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_slots_kernel(const __grid_constant__ MergeParams p) {
  // an 8-lane group per (row, head) item, four consecutive items per warp: each slot is read as 4 x W x 4
  // contiguous bytes; lane q of a group owns float4 columns q, q + 8, ... of its item
  constexpr int kV = W / 32;                  // float4 columns per lane
  constexpr int kUnroll = W == 128 ? 4 : 1;   // slots whose loads are in flight together
  const int lane = threadIdx.x & 31, grp = lane >> 3, q = lane & 7;
  const int64_t wid = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const int H = p.num_heads;
  const int64_t total = (int64_t)p.total_rows * H;
  for (int64_t base = wid * 4; base < total; base += (int64_t)gridDim.x * kWarpsPerBlock * 4) {
    const int64_t item = base + grp;
    const bool live_item = item < total;
    // item -> (range, row within range, head); ranges are consecutive in item space
    const int64_t local = live_item ? item / H : 0;
    const int h = live_item ? (int)(item - local * H) : 0;
    int lo = 0, hi = p.num_ranges - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.ranges[mid].prefix <= local) lo = mid; else hi = mid - 1;
    }
    const int ri = lo;
    const int64_t row = p.ranges[ri].row_begin + (local - p.ranges[ri].prefix);
    const int ns = live_item ? p.ranges[ri].nslots : 0;
    auto lse_at = [&](int s) { return __ldg(p.part_lse + ((int64_t)s * p.slot_stride_rows + row) * H + h); };

    // lane q holds the lse of slots q, q + 8, ...: one round trip for all of them, then group maxima
    float m = -INFINITY;
    for (int s0 = 0; s0 < ns; s0 += 8) m = fmaxf(m, s0 + q < ns ? lse_at(s0 + q) : -INFINITY);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float4 acc[kV];
#pragma unroll
    for (int v = 0; v < kV; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    // every lane of the warp runs the same number of slot rounds (the groups' items may differ)
    int ns_max = ns;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ns_max = max(ns_max, __shfl_xor_sync(0xffffffffu, ns_max, o));
    for (int s0 = 0; s0 < ns_max; s0 += 8) {
      // this lane's slot weight (0 for an empty or absent state); the states are then read together,
      // each slot's weight taken from the lane of the group that holds it
      const float l = s0 + q < ns ? lse_at(s0 + q) : -INFINITY;
      const float w = (l == -INFINITY || m == -INFINITY) ? 0.f : __expf(l - m);
      float ws = w;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
      wsum += ws;
      const int n = min(8, ns_max - s0);
#pragma unroll kUnroll
      for (int i = 0; i < n; ++i) {
        const float wi = __shfl_sync(0xffffffffu, w, (lane & ~7) + i);
        const int64_t g = ((int64_t)(s0 + i) * p.slot_stride_rows + row) * H + h;
#pragma unroll
        for (int v = 0; v < kV; ++v) {
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          if (wi != 0.f) o = __ldg(reinterpret_cast<const float4*>(p.part_out + g * W) + q + 8 * v);
          acc[v].x += wi * o.x; acc[v].y += wi * o.y; acc[v].z += wi * o.z; acc[v].w += wi * o.w;
        }
      }
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    const int64_t orow = row * H + h;
    __syncwarp();   // every lane has read the states (the output may alias slot 0)
    if (live_item) {
#pragma unroll
      for (int v = 0; v < kV; ++v) {
        const float4 r = make_float4(acc[v].x * inv, acc[v].y * inv, acc[v].z * inv, acc[v].w * inv);
        if (p.out_bf16) {
          uint2 b = make_uint2(pack_bf16(r.x, r.y), pack_bf16(r.z, r.w));
          reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + orow * W)[q + 8 * v] = b;
        } else {
          reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow * W)[q + 8 * v] = r;
        }
      }
      if (q == 0) p.lse[orow] = (wsum > 0.f) ? m + logf(wsum) : -INFINITY;
    }
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
  merge_slots_kernel<kDv><<<grid_for((items + 3) / 4, kWarpsPerBlock), kWarpsPerBlock * 32, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_merge_slots_latent(const MergeParams& p, cudaStream_t s) {
  const int64_t items = (int64_t)p.total_rows * p.num_heads;
  if (items == 0) return cudaSuccess;
  merge_slots_kernel<kDc><<<grid_for((items + 3) / 4, kWarpsPerBlock), kWarpsPerBlock * 32, 0, s>>>(p);
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
