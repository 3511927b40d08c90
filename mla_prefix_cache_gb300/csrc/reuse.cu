// Head-split reuse with protected-row replacement ("RedKnot-MLA: Multi-Head
// Offline-Online Reuse for DeepSeek-V4 Long-Context Serving", section 2):
// Global heads are recomputed online for every query row, Local heads only
// for the protected rows, and every other (row, head) keeps its offline
// artifact state, replaced rather than added to.  The online parts run as two
// compacted sub-problems of the fused prefill (Global heads x all rows;
// Local heads x protected rows); these kernels build their inputs and merge
// the results.
#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

// q_sub[i][j][:] = q[rows ? rows[i] : i][heads[j]][:] (bf16 [.., 192]) and,
// for j == 0, pos_sub[i] = q_pos[row]; one thread per 16-byte chunk.
__global__ void __launch_bounds__(256) gather_q_kernel(const uint16_t* __restrict__ q, const int32_t* __restrict__ q_pos,
                                                       const int32_t* __restrict__ rows,
                                                       const int32_t* __restrict__ heads, int n_rows, int n_heads,
                                                       int H, uint16_t* __restrict__ q_sub, int32_t* __restrict__ pos_sub) {
  constexpr int kChunks = kDqk * 2 / 16;   // 24
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)n_rows * n_heads * kChunks;
  if (g >= total) return;
  const int c = (int)(g % kChunks);
  const int64_t ij = g / kChunks;
  const int j = (int)(ij % n_heads);
  const int64_t i = ij / n_heads;
  const int64_t row = rows ? __ldg(rows + i) : i;
  const int h = __ldg(heads + j);
  reinterpret_cast<uint4*>(q_sub)[ij * kChunks + c] = __ldg(reinterpret_cast<const uint4*>(q + (row * H + h) * kDqk) + c);
  if (j == 0 && c == 0 && pos_sub != nullptr) pos_sub[i] = __ldg(q_pos + row);
}

// w_sub [512][n_heads * 256]: the K_nope and V column blocks of heads[0..n_heads)
// in the layout of kv_b_proj (all K blocks, then all V blocks).
__global__ void __launch_bounds__(256) gather_w_kernel(const uint16_t* __restrict__ w, const int32_t* __restrict__ heads,
                                                       int n_heads, int H, uint16_t* __restrict__ w_sub) {
  constexpr int kChunks = 128 * 2 / 16;    // 16 per 128-column block
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)kDc * 2 * n_heads * kChunks;
  if (g >= total) return;
  const int c = (int)(g % kChunks);
  const int64_t t = g / kChunks;
  const int blk = (int)(t % (2 * n_heads));   // 0 .. n_heads-1: K blocks, then V blocks
  const int row = (int)(t / (2 * n_heads));
  const int kv = blk >= n_heads, j = kv ? blk - n_heads : blk;
  const int h = __ldg(heads + j);
  const int64_t src_col = (int64_t)kv * H * 128 + (int64_t)h * 128;
  const int64_t dst_col = (int64_t)kv * n_heads * 128 + (int64_t)j * 128;
  reinterpret_cast<uint4*>(w_sub + (int64_t)row * n_heads * 256 + dst_col)[c] =
      __ldg(reinterpret_cast<const uint4*>(w + (int64_t)row * H * 256 + src_col) + c);
}

// One warp per (row, head): the state comes from the Global sub-problem
// (gidx[h] >= 0), else from the protected-row sub-problem (pidx[row] >= 0,
// lidx[h]), else from the artifact.
__global__ void __launch_bounds__(256) assemble_kernel(const ReuseAssemble p) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t total = (int64_t)p.rows * p.H;
  if (wid >= total) return;
  const int64_t t = wid / p.H;
  const int h = (int)(wid - t * p.H);
  const int gi = __ldg(p.gidx + h);
  const int pi = __ldg(p.pidx + t);
  const float* so;
  float sl;
  if (gi >= 0) {
    const int64_t r = t * p.n_global + gi;
    so = p.out_g + r * kDv;
    sl = __ldg(p.lse_g + r);
  } else if (pi >= 0) {
    const int64_t r = (int64_t)pi * p.n_local + __ldg(p.lidx + h);
    so = p.out_p + r * kDv;
    sl = __ldg(p.lse_p + r);
  } else {
    so = p.art_out + wid * kDv;
    sl = __ldg(p.art_lse + wid);
  }
  const float4 v = __ldg(reinterpret_cast<const float4*>(so) + lane);
  if (p.out_bf16) {
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + wid * kDv)[lane] =
        make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w));
  } else {
    reinterpret_cast<float4*>(static_cast<float*>(p.out) + wid * kDv)[lane] = v;
  }
  if (lane == 0) p.lse[wid] = sl;
}

int blocks_for(int64_t threads) { return (int)((threads + 255) / 256); }

}  // namespace

cudaError_t launch_gather_q(const uint16_t* q, const int32_t* q_pos, const int32_t* rows, const int32_t* heads,
                            int n_rows, int n_heads, int H, uint16_t* q_sub, int32_t* pos_sub, cudaStream_t s) {
  const int64_t total = (int64_t)n_rows * n_heads * (kDqk * 2 / 16);
  if (total == 0) return cudaSuccess;
  gather_q_kernel<<<blocks_for(total), 256, 0, s>>>(q, q_pos, rows, heads, n_rows, n_heads, H, q_sub, pos_sub);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_gather_w(const uint16_t* w, const int32_t* heads, int n_heads, int H, uint16_t* w_sub,
                            cudaStream_t s) {
  const int64_t total = (int64_t)kDc * 2 * n_heads * 16;
  if (total == 0) return cudaSuccess;
  gather_w_kernel<<<blocks_for(total), 256, 0, s>>>(w, heads, n_heads, H, w_sub);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_reuse_assemble(const ReuseAssemble& p, cudaStream_t s) {
  const int64_t warps = (int64_t)p.rows * p.H;
  if (warps == 0) return cudaSuccess;
  assemble_kernel<<<(int)((warps + 7) / 8), 256, 0, s>>>(p);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
