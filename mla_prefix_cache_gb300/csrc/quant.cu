// E4M3 copy of kv_b_proj for the FP8 up-projection (mla_prefill_ctx_fp8w):
// its largest magnitude, and its codes e4m3(W / scale), transposed so that
// each output column's 512 latent weights are contiguous (the K-major operand
// of the kind::f8f6f4 MMA).
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kAbsThreads = 1024;

// One CTA: the largest |x| of n bf16 values (16-byte loads when n % 8 == 0).
__global__ void __launch_bounds__(kAbsThreads) absmax_bf16_kernel(const uint16_t* x, int64_t n, float* out) {
  float m = 0.f;
  if ((n & 7) == 0) {
    const uint4* v = reinterpret_cast<const uint4*>(x);
    for (int64_t i = threadIdx.x; i < n / 8; i += kAbsThreads) {
      const uint4 w = __ldg(v + i);
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(u[k] << 16)), fabsf(__uint_as_float(u[k] & 0xFFFF0000u))));
    }
  } else {
    for (int64_t i = threadIdx.x; i < n; i += kAbsThreads) m = fmaxf(m, fabsf(__uint_as_float((uint32_t)x[i] << 16)));
  }
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[kAbsThreads / 32];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = red[threadIdx.x];
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) *out = m;
  }
}

// out[c][k] = e4m3(w[k][c] / scale) for the [512][cols] bf16 matrix w, by
// 64 x 64 tiles through shared memory (reads and writes coalesced).
__global__ void __launch_bounds__(256) quantize_t_kernel(const uint16_t* w, int cols, float scale, uint8_t* out) {
  __shared__ float tile[64][65];
  const int c0 = blockIdx.x * 64, k0 = blockIdx.y * 64;
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int k = i / 64, c = i % 64;
    tile[k][c] = c0 + c < cols ? __uint_as_float((uint32_t)w[(int64_t)(k0 + k) * cols + c0 + c] << 16) : 0.f;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 32; i += 256) {
    const int c = i / 32, k = 2 * (i % 32);
    if (c0 + c < cols) {
      const uint16_t v = pack_e4m3x2(tile[k][c] / scale, tile[k + 1][c] / scale);
      *reinterpret_cast<uint16_t*>(out + (int64_t)(c0 + c) * kDc + k0 + k) = v;
    }
  }
}

}  // namespace

cudaError_t launch_absmax_bf16(const uint16_t* x, int64_t n, float* out, cudaStream_t s) {
  absmax_bf16_kernel<<<1, kAbsThreads, 0, s>>>(x, n, out);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_quantize_t(const uint16_t* w, int cols, float scale, uint8_t* out, cudaStream_t s) {
  if (cols == 0) return cudaSuccess;
  quantize_t_kernel<<<dim3((cols + 63) / 64, kDc / 64), 256, 0, s>>>(w, cols, scale, out);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
