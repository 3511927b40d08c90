// Internal structures shared by the C-ABI layer (host planner) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace mla {

constexpr int kDc = 512;
constexpr int kDr = 64;
constexpr int kDnope = 128;
constexpr int kDv = 128;
constexpr int kDqk = kDnope + kDr;
constexpr int kBlock = 64;
constexpr int kRowBf16 = kDc + kDr;          // elements
constexpr int kRowBytesBf16 = 2 * kRowBf16;  // 1152
constexpr int kRowBytesFp8 = kDc + 2 * kDr;  // 640
constexpr int kMaxHeads = 128;

// Device error word bits (kept in the caller's workspace).
constexpr uint32_t kErrBadBlock = 1u;
constexpr uint32_t kErrTimeout = 2u;

// One KV split of the plan: a contiguous key range of one request with one
// RoPE offset (a context chunk of a segment, or the extend stage).
struct Split {
  int32_t req;        // request index (block-table row)
  int32_t q_begin;    // global row of the request's first query
  int32_t q_count;    // E_r
  int32_t q_tok0;     // token index of the request's first query (= C_r)
  int32_t k_begin;    // first key token
  int32_t k_end;      // one past the last key token
  int32_t slot;       // index of this split within its request
  int32_t pad;
  int64_t rope_offset;
};

// Query rows [row_begin, row_end) whose partial states live in slots 0..nslots-1.
struct RowRange {
  int32_t row_begin;
  int32_t row_end;
  int32_t nslots;
  int32_t prefix;             // rows of the launch's earlier ranges
};

constexpr int kMaxRangesPerLaunch = 512;

struct MergeParams {
  const float* part_out;      // [slots, T_q, H, 128]
  const float* part_lse;      // [slots, T_q, H]
  int64_t slot_stride_rows;   // T_q
  void* out;                  // [T_q, H, 128] fp32 or bf16
  float* lse;                 // [T_q, H]
  int out_bf16;
  int num_heads;
  int num_ranges;
  int total_rows;             // sum of range lengths in this launch
  RowRange ranges[kMaxRangesPerLaunch];
};

// ------------------------------------------------------------ fused persistent kernel
constexpr int kRingDepth = 128;   // deepest ring lane: 128-token K/V tiles (8 MB); a small workspace gets less
constexpr int kRingLanes = 64;    // most ring lanes the jobs of a launch take turns on
constexpr int kLanePairs = 76;    // CTA pairs of a GB300's persistent grid (152 SMs), for the lane count
constexpr int kMaxPieces = 448;   // pieces per launch (kernel-parameter budget)

// One key range of one request attended with one RoPE offset, for every head.
// Each (piece, head) is a job: n_prod producer roles then n_cons consumer roles.
struct Piece {
  int32_t req;
  int32_t q_begin;     // global row of the request's first query
  int32_t q_count;     // E_r
  int32_t q_tok0;      // token index of the request's first query (C_r)
  int32_t k_begin;     // first key token
  int32_t k_end;       // one past the last key token
  int32_t slot;        // partial-state slot, or -1: write the final out/lse
  int32_t group_begin; // first role group of this piece in the launch's queue
  int32_t n_cons;      // consumer roles per head (128 queries each)
  int32_t n_prod;      // producer roles per head
  int32_t row_block0;  // the request's rows were gathered contiguously from this block on
  int32_t exact;       // exact scores: tiles [0, exact & 255) of the piece carry the bf16 residual of
                       // K_nope, used by consumer pairs below exact >> 8 (see kExactKeys)
  int64_t rope_offset;
};

// A query row that sees fewer than kExactKeys keys in all takes its scores
// with K_nope as bf16 + bf16 residual (exact to about 2^-16): its lse would
// otherwise carry the bf16 rounding of a handful of scores (about 1.4e-3 per
// unit-variance score), which many keys average out.  Such rows see at most
// kExactKeys + 63 keys of a piece from its aligned start: 9 tiles of 128.
constexpr int kExactKeys = 1024;
constexpr int kExactSlots = 16;   // ring slots per lane that hold residual tiles

// Device-side view of one job.
struct Job {
  int32_t req, head, q_begin, q_count, q_tok0, k_begin, k_end, t0, n_tiles, n_cons, n_prod, slot, row_block0;
  int32_t n_exact_tiles, n_exact_pairs;
  int64_t rope_offset;
  const int32_t* q_tok;   // FusedParams::q_tok
};

struct FusedParams {
  CUtensorMap tm_kr;     // gathered bf16 latent rows [rows][576], box 64 x 64 (k_rope at column 512)
  CUtensorMap tm_kr128;  // same rows, box 64 x 128 (the k_rope of one 128-key tile)
  CUtensorMap tm_c;      // same rows, box 64 x 256 (one 64-wide latent slice of a producer pass)
  CUtensorMap tm_w;      // bf16 kv_b_proj as [H*4 blocks][512 rows][64 cols], box 64 x 64 x 2
  CUtensorMap tm_ring;   // bf16 ring as [jobs*ring*4 blocks][128 rows][64 cols], box 64 x 128 x 2
  CUtensorMap tm_ring1;  // same ring, box 64 x 128 x 1 (one block: half of a paired consumer's stage)
  CUtensorMap tm_ring64; // same ring, box 64 x 64 x 2 (64 keys of K_nope lo | hi: a CTA pair's half tile)
  CUtensorMap tm_q;      // q as (column, head, row) of [T_q][H][192], box 64 x 1 x 128: 128 rows of one head
  CUtensorMap tm_out;    // out as (column, head, row) of [T_q][H][128], box 32 (fp32) or 64 (bf16) x 1 x 128
  CUtensorMap tm_part;   // partial states, fp32 [slots * T_q][H][128], box 32 x 1 x 128
  CUtensorMap tm_c8;     // FP8 up-projection: gathered 640-byte rows as bytes, box 128 B x 128 rows (E4M3 codes)
  CUtensorMap tm_w8;     // FP8 up-projection: E4M3 kv_b_proj transposed [H*256][512], box 128 B x 128 rows
  const uint16_t* q_bf16;  // q [T_q][H][192]
  const int32_t* q_tok;    // optional [T_q]: token index of each query row within its request (rows that are
                           // a sorted subset of the request's queries); nullptr: q_tok0 + row - q_begin
  uint32_t* err;
  uint32_t* queue;       // role-group counter
  uint32_t* flags;       // per job: ready[ring_depth], consumed[ring_depth]
  uint16_t* ring;
  const int32_t* block_table;
  const int32_t* q_pos;
  void* out;
  float* lse;
  float* part_out;
  float* part_lse;
  int64_t slot_stride_rows;
  int max_blocks;
  int num_blocks;
  int num_heads;
  int out_bf16;
  float out_scale;      // applied to the up-projection accumulators (FP8 dequant scale, else 1)
  float scale_log2;
  int n_pieces;
  int n_groups;         // role groups in the queue (one per cluster dequeue)
  int ring_depth;       // 128-token tiles per ring lane: a power of two <= kRingDepth (slots are t & (depth - 1))
  int ring_lanes;       // job j writes its tiles into lane j % ring_lanes
  int prod_ahead;       // heads by which a job's producers precede their consumers in the queue
  uint64_t wait_limit_ns;   // bound of every wait of the kernel (a timeout sets kErrTimeout)
  int l2_hints;         // 1: ring tiles evict_last, streamed data evict_first; 0: evict_normal
  int fp8w;             // 1: FP8 up-projection (E4M3 rows and kv_b_proj on kind::f8f6f4)
  int krope_col;        // element column of k_rope in the gathered rows seen as bf16 (512, or 256 for 640-byte rows)
  int withhold_job;     // test hook: this job's producer roles do nothing, so its consumers' waits run
                        // out (-1: none)
  unsigned long long* trace;   // optional, kTraceWords per role slot (group * 2 + cluster rank; see fused_common.cuh)
  int trace_detail_role;       // role slot whose stages are timed one by one (-1: none)
  uint64_t rope_frac[kDr / 2];
  Piece pieces[kMaxPieces];
};

constexpr int kTraceWords = 8;

static_assert(sizeof(FusedParams) <= 32000, "kernel parameter space");

// The persistent CTA-pair kernel (fused2.cu): pieces carry n_prod producer
// *pair* roles and group_begin counts pair roles (n_prod + ceil(n_cons / 2)
// per head).  The grid is the number of CTAs resident at once (a multiple of 2).
cudaError_t launch_fused2(const FusedParams& p, int grid, cudaStream_t s);
cudaError_t fused2_grid_size(int* grid);
int fused2_smem_bytes();

// Kernel launchers (return cudaError_t of the launch).
cudaError_t launch_merge_slots(const MergeParams& p, cudaStream_t s);
// The same merge over 512-wide fp32 latent states ([slots][T_q][H][512]).
cudaError_t launch_merge_slots_latent(const MergeParams& p, cudaStream_t s);
cudaError_t launch_merge2(const float* oa, const float* la, const float* ob, const float* lb,
                          float* o, float* l, int64_t rows, int d_v, cudaStream_t s);
cudaError_t launch_rope(const uint16_t* x, const int32_t* pos, int64_t offset, const uint64_t* frac_host,
                        uint16_t* y, int tokens, int heads, int row_stride, int rope_col,
                        cudaStream_t s);
cudaError_t launch_gather(const uint8_t* cache, int fp8, float scale, int num_blocks,
                          const int32_t* table_row, int max_blocks, int start, int len,
                          uint16_t* dst, uint32_t* err, cudaStream_t s);

struct GatherReq {
  int32_t req;
  int32_t base_block;   // first destination block
  int32_t seq_len;
  int32_t first_block;  // first logical block copied (blocks first_block .. of the request)
};
constexpr int kMaxGatherReqs = 1024;
struct GatherBlocksParams {
  const uint8_t* cache;
  const int32_t* block_table;
  uint16_t* dst;        // bf16 [total_blocks * 64][576]
  uint32_t* err;
  int fp8;
  float scale;
  int num_blocks;
  int max_blocks;
  int n_reqs;
  int total_blocks;
  GatherReq reqs[kMaxGatherReqs];
};
cudaError_t launch_gather_blocks(const GatherBlocksParams& p, cudaStream_t s);
// FP8 caches: the rows as stored (640 B), same order; dst is a byte buffer.
cudaError_t launch_gather_blocks_raw(const GatherBlocksParams& p, cudaStream_t s);

// Content-addressed block store (blocks.cu): content hash of whole cache
// blocks and byte comparison of block pairs.
cudaError_t launch_block_hash(const uint8_t* cache, int fp8, int num_blocks, const int32_t* ids, int n,
                              uint64_t* hashes, uint32_t* err, cudaStream_t s);
cudaError_t launch_block_compare(const uint8_t* cache, int fp8, int num_blocks, const int32_t* a, const int32_t* b,
                                 int n, int32_t* equal, uint32_t* err, cudaStream_t s);

// Head-split reuse (reuse.cu).
struct ReuseAssemble {
  const float* out_g;    // [rows][n_global][128]: Global heads, every row
  const float* lse_g;
  const float* out_p;    // [n_protected][n_local][128]: Local heads, protected rows
  const float* lse_p;
  const float* art_out;  // [rows][H][128]: the offline artifact
  const float* art_lse;
  const int32_t* gidx;   // [H]: index among the Global heads, or -1
  const int32_t* lidx;   // [H]: index among the Local heads, or -1
  const int32_t* pidx;   // [rows]: index among the protected rows, or -1
  void* out;             // [rows][H][128] fp32 or bf16
  float* lse;
  int out_bf16;
  int rows, H, n_global, n_local;
};
cudaError_t launch_gather_q(const uint16_t* q, const int32_t* q_pos, const int32_t* rows, const int32_t* heads,
                            int n_rows, int n_heads, int H, uint16_t* q_sub, int32_t* pos_sub, cudaStream_t s);
cudaError_t launch_gather_w(const uint16_t* w, const int32_t* heads, int n_heads, int H, uint16_t* w_sub,
                            cudaStream_t s);
cudaError_t launch_reuse_assemble(const ReuseAssemble& p, cudaStream_t s);

// E4M3 copy of kv_b_proj (quant.cu): the largest |x| of n bf16 values into
// *out (device), and out[c][k] = e4m3(w[k][c] / scale) of the [512][cols] matrix.
cudaError_t launch_absmax_bf16(const uint16_t* x, int64_t n, float* out, cudaStream_t s);
cudaError_t launch_quantize_t(const uint16_t* w, int cols, float scale, uint8_t* out, cudaStream_t s);

void count_launch(int n = 1);

}  // namespace mla
