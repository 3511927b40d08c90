// Declarations of the absorbed (latent-space) path: its work pieces, the
// parameters of the latent attention (absorb.cu) and of the two per-head
// projections (headproj.cu), and their launchers.
#pragma once

#include "internal.h"

namespace mla {

// ------------------------------------------------------------ absorbed (latent-space) path
// One piece of the absorbed path: a key range of one request with one RoPE
// offset, attended by all its (query, head) rows, which form 256-row tiles
// (row = token * H + head); each tile's keys are cut into n_splits work items.
struct AbsPiece {
  int32_t req;
  int32_t q_begin;     // global row of the request's first query
  int32_t q_count;     // E_r
  int32_t q_tok0;      // token index of the request's first query (C_r)
  int32_t k_begin;     // first key token
  int32_t k_end;       // one past the last key token
  int32_t row_block0;  // the request's rows were gathered contiguously from this block on (rows read in place:
                       // the block holding the copy of its last block)
  int32_t last_lb;     // the request's last logical block
  int32_t slot;        // partial-state slot of split 0 (split i uses slot + i)
  int32_t n_row_tiles; // ceil(q_count * H / 256)
  int32_t n_splits;    // key splits per row tile
  int32_t split_keys;  // keys per split (a multiple of 128)
  int32_t item_begin;  // first work item of this piece in the launch
  int64_t rope_offset;
};
constexpr int kMaxAbsPieces = 448;

// The latent attention (absorb.cu): items of 256 rows, 128-key tiles on two CTA pairs.
struct AbsorbParams {
  CUtensorMap tm_qlat;  // qlat as [T_q * H rows][512], box 64 x 128
  CUtensorMap tm_c3;    // gathered bf16 rows as 9 blocks of 64 columns ([c | k_rope]), box 64 cols x 64 rows x 3 blocks
  CUtensorMap tm_c2;    // gathered bf16 rows, latent blocks, box 64 x 64 x 2
  // E4M3 scores (fp8_scores): the paged FP8 cache's rows as stored (640 B, rows = num_blocks x 64)
  CUtensorMap tm_f5;    // as 5 blocks of 128 B (4 of E4M3 codes, k_rope as bf16), box 128 x 64 x 5
  CUtensorMap tm_qlat8; // E4M3 qlat as [T_q * H rows][512 B], box 128 x 128
  CUtensorMap tm_lat;   // lat_out as [slots * T_q * H rows][512] fp32, box 32 x 128
  // rows read in place: the paged BF16 cache itself (rows = num_blocks x 64), boxes as tm_c3 / tm_c2
  CUtensorMap tm_k3;
  CUtensorMap tm_k2;
  const int32_t* block_table;   // [num_reqs][max_blocks]
  int max_blocks;
  int num_blocks;
  int s_in_place;       // the score side reads the cache's blocks in place (always, with E4M3 scores)
  int o_in_place;       // the P c side reads them in place, a request's last block from its copy
  const float* qscale;  // [T_q * H]: the E4M3 qlat row's scale
  float kv_scale;
  int fp8_scores;
  const uint16_t* q;     // [T_q][H][192]: q_rope at 128..191, not rotated
  const uint16_t* qlat;  // [T_q][H][512] bf16: kv_scale * q_nope W_UK,h^T
  const int32_t* q_pos;
  const int32_t* q_tok;  // optional [T_q]: each row's token index (compacted rows); else q_tok0 + row
  float* lat_out;        // [slots][T_q * H][512] fp32, normalised by the row sum
  float* lat_lse;        // [slots][T_q * H], natural log
  int64_t slot_stride_rows;   // T_q * H
  uint32_t* err;
  int num_heads;
  int n_pieces;
  int n_items;
  float scale_log2;
  uint64_t rope_frac[kDr / 2];
  AbsPiece pieces[kMaxAbsPieces];
};
static_assert(sizeof(AbsorbParams) <= 32000, "kernel parameter space");

// q absorption (headproj.cu), over tokens row0 .. row0 + tokens - 1:
//   qlat[t][h][c] = bf16(scale sum_d q[t][h][d] W[c][128 h + d])        (qscale null)
//   qlat8[t][h][c] = e4m3(qlat / s), qscale[t H + h] = s = amax / 448  (qscale set; scale unused)
struct QAbsorbParams {
  CUtensorMap tm_q;        // q as (column, head, token) up to token row0 + tokens, box 64 x 1 x 128
  CUtensorMap tm_w;        // kv_b_proj as [512][H * 256], box 64 x 256
  CUtensorMap tm_out;      // qlat (bf16, box 64 x 1 x 128) or qlat8 (bytes, box 128 x 1 x 128) as
                           // (column, head, token) up to token row0 + tokens
  float* qscale;           // [T_q * H]: E4M3 row scales, or null for bf16 qlat
  uint32_t* err;
  float scale;
  int row0;                // first token row of this launch
  int tokens;              // rows row0 .. row0 + tokens - 1
  int num_heads;
};

// Output projection of the latent states (headproj.cu): for the rows of each
// request range, out[t][h][d] = scale * sum_c lat[t H + h][c] W[c][128 H + 128 h + d]
// and lse[t][h] = lat_lse[t H + h] (slot 0, where a request's splits were
// merged).
struct ProjParams {
  CUtensorMap tm_w;               // kv_b_proj as [512][H * 256], box 64 x 128
  const float* lat_out;           // [T_q * H][512]
  const float* lat_lse;           // [T_q * H]
  void* out;
  float* lse;
  uint32_t* err;
  int out_bf16;
  float scale;
  int num_heads;
  int num_ranges;
  int total_rows;                 // tokens of this launch's ranges
  RowRange ranges[kMaxRangesPerLaunch];
};

cudaError_t launch_absorb_attn(const AbsorbParams& p, cudaStream_t s);
cudaError_t launch_qabsorb(const QAbsorbParams& p, cudaStream_t s);
cudaError_t launch_absorb_proj(const ProjParams& p, cudaStream_t s);

}  // namespace mla
