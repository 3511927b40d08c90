/*
 * mla.h -- C ABI of libmla: MLA chunked prefill over a paged packed-latent KV
 * cache, hand-written for NVIDIA GB300 (sm_103a).
 *
 * Geometry (fixed): latent d_c = 512, RoPE width d_r = 64, per-head no-RoPE key
 * width d_nope = 128, value width d_v = 128, 64-token cache blocks.  One cached
 * token is one packed row [c_kv 0..511 | k_rope 0..63] ("DeepSeek MLA — Prefix
 * Cache 与 Chunked Prefill 深度解析", section 5.2; 64-token blocks from
 * "PagedAttention assumed MHA. DeepSeek-V4 says that assumption is broken",
 * section "Block size is not a tuning knob here").
 *
 * Conventions shared by every entry point
 *  - All tensors are contiguous, row-major, little-endian.  "device" pointers
 *    are CUDA device memory of the current device; "host" pointers are plain
 *    host memory read synchronously before the call returns.
 *  - The library never allocates and never frees; every buffer belongs to the
 *    caller.  Calls are asynchronous on `stream` (NULL = legacy default stream).
 *  - Host-side validation runs first and returns a status before anything is
 *    launched.  No C++ exception crosses the ABI.  Device-side faults that the
 *    kernels can detect (a block-table entry outside [0, num_blocks)) never
 *    trap: the affected rows are read as zeros and a bit is set in a device
 *    error word that the caller reads with mla_get_device_error().
 *  - Return value: an mla_status (0 = MLA_OK).
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* mla_stream_t; /* identical to cudaStream_t */

enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent lengths */
  MLA_ERR_UNSUPPORTED = 2,   /* a shape or mode the library does not implement */
  MLA_ERR_BAD_BLOCK_ID = 3,  /* device saw a block-table entry outside [0, num_blocks) */
  MLA_ERR_CUDA = 4,          /* a CUDA runtime call failed (see mla_last_cuda_error) */
  MLA_ERR_WORKSPACE = 5,     /* workspace missing or smaller than required */
  MLA_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up */
  MLA_ERR_TOO_LARGE = 7      /* needs more scratch than mla_prefill_ctx_noalloc holds */
};

enum mla_kv_dtype {
  MLA_KV_BF16 = 0,     /* rows of 576 bf16 = 1152 B */
  MLA_KV_FP8_E4M3 = 1  /* rows of 640 B: 512 OCP E4M3FN codes of c_kv / kv_scale,
                          then 64 bf16 k_rope values */
};

enum mla_out_dtype { MLA_OUT_FP32 = 0, MLA_OUT_BF16 = 1 };

enum mla_parts { MLA_PART_CONTEXT = 1, MLA_PART_EXTEND = 2, MLA_PART_ALL = 3 };

/* One relocated document segment of a request's cached context: key tokens
 * [start, start+len) of request `req`, whose k_rope was cached at canonical
 * positions so that token start+j carries position (rope_offset + j) - rope_offset
 * = j.  Queries attend to it with q_rope rotated by (q_pos - rope_offset)
 * ("RedKnot-MLA: Multi-Head Offline-Online Reuse for DeepSeek-V4 Long-Context
 * Serving", section 2, "Online position restoration and merge"). */
typedef struct {
  int32_t req;
  int32_t start;
  int32_t len;
  int32_t reserved; /* must be 0 */
  int64_t rope_offset;
} mla_segment;

/* ------------------------------------------------------------------------
 * mla_prefill_ctx -- the whole hot path of one layer's chunked prefill.
 *
 * Defines ("DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析",
 * sections 4.2-4.4): for request r with C_r = seq_lens[r] - E_r cached context
 * tokens and E_r = cu_q[r+1] - cu_q[r] new (extend) tokens, query i (global row
 * cu_q[r] + i, token index C_r + i, RoPE position q_pos[row]) and head h:
 *   context stage: keys = the request's segments (default one segment
 *     [0, C_r) with rope_offset 0), cut into chunks of `chunk` tokens;
 *   extend stage : keys C_r .. C_r + i (causal, diagonal included), offset 0;
 *   each key t: x_t = row of token t via block_table[r][t/64], slot t%64
 *     (FP8: c_kv = e4m3 * kv_scale); K_nope = c_kv * kv_b_proj[:, K cols of h],
 *     V = c_kv * kv_b_proj[:, V cols of h]; K = [K_nope | k_rope] (k_rope shared
 *     by all heads);
 *   s_t = softmax_scale * (q_nope . K_nope_t + R(q_pos - offset) q_rope . k_rope_t),
 *     R = rotation of interleaved pairs (2k, 2k+1) by theta^(-2k/64) per unit;
 *   every chunk and the extend stage give (out, lse = ln sum e^s); they are folded
 *   with merge_attn_states (see mla_merge_states).
 * The up-projection runs on the tensor cores inside the persistent attention
 * kernel, once per (key, head).  Its bf16 K_nope/V tiles pass from producer to
 * consumer CTAs through K/V ring lanes in the workspace (4 to 64 lanes of up
 * to 128 slots of 128 keys, whatever the number of pieces: enough lanes for
 * the jobs that run at once, and about 32 MiB of tiles when jobs have many
 * queries); the jobs of the call take turns on the lanes, and the tiles are
 * cached in L2 with an evict-last policy, so a lane's lines are rewritten
 * while they sit in the 126 MB L2: with long extends the up-projected K/V
 * is not written back to HBM (measured on GB300 with 128 heads: the fused
 * kernel writes 100 MB per call on 8K + 2K tokens, where the output alone is
 * 134 MB, and 5.5 GB on 256K + 4K tokens, where the partial states of the 17
 * pieces are 4.6 GB).
 *
 * Arguments
 *  q            device bf16 [T_q, H, 192]: [q_nope 0..127 | q_rope 128..191],
 *               q_rope NOT rotated.  T_q = cu_q[num_reqs].
 *  q_pos        device int32 [T_q]: true RoPE position of each query row.
 *  kv_cache     device [num_blocks, 64, row]: bf16 row of 576 (kv_dtype
 *               MLA_KV_BF16) or 640-byte FP8 row (MLA_KV_FP8_E4M3).
 *  kv_scale     FP8 per-tensor dequant scale (ignored for bf16).
 *  block_table  device int32 [num_reqs, max_blocks_per_req].  Entries that
 *               the request's tokens use must lie in [0, num_blocks).
 *  seq_lens     HOST int32 [num_reqs]: C_r + E_r (extend rows are in the cache).
 *  cu_q         HOST int32 [num_reqs + 1]: prefix sums of E_r, cu_q[0] = 0.
 *  segments     HOST, optional (NULL, num_segments = 0 for the default): every
 *               segment lies in [0, C_r) of its request; segments of a request
 *               must not overlap.  A request with no segment listed while
 *               segments != NULL has an empty context.
 *  chunk        context chunk length, a positive multiple of 64.
 *  kv_b_proj    device bf16 [512, H*256]: columns 0..H*128-1 are the K_nope
 *               blocks of heads 0..H-1, columns H*128.. are the V blocks.
 *  softmax_scale, rope_theta  scalars (rope_theta > 1).
 *  parts        MLA_PART_CONTEXT | MLA_PART_EXTEND.
 *  out          device [T_q, H, 128], fp32 or bf16 per out_dtype.
 *  lse          device fp32 [T_q, H], natural log, softmax scale included;
 *               -inf for a row with no visible key (its out row is 0).
 *  workspace    device, 256-B aligned; mla_prefill_workspace_size(...) bytes
 *               lets the whole call run as one kernel launch at full speed:
 *               the K/V ring lanes (up to 0.5 GiB), per-job ring flags, every block
 *               of the requests gathered in logical order as bf16 (1152 B per
 *               token; FP8 rows dequantised) and fp32 partial states
 *               (516 B per query row, head and piece of a request cut into
 *               several pieces: one per relocated segment and per 16384 keys).
 *               Any size down to mla_prefill_min_workspace_size(...) also
 *               works, with shallower and fewer lanes and, at the bottom, one
 *               piece per launch: more slowly.  Holds the device error word;
 *               must not be shared by calls that may overlap on the GPU.
 *  H            num_heads in [1, 128].
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_UNSUPPORTED (H > 128, chunk not a
 * multiple of 64), MLA_ERR_WORKSPACE, MLA_ERR_CUDA.  Bad block ids are reported
 * by mla_get_device_error(workspace, stream) after the call.
 * ---------------------------------------------------------------------- */
size_t mla_prefill_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q,
                                  int num_heads, const mla_segment* segments, int num_segments,
                                  int chunk, int parts);

/* The smallest workspace mla_prefill_ctx accepts for these arguments (two
 * ring lanes of 4 tiles, one piece per launch); 0 when the planner rejects
 * the arguments. */
size_t mla_prefill_min_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q,
                                      int num_heads, const mla_segment* segments, int num_segments,
                                      int chunk, int parts);

int mla_prefill_ctx(const void* q, const int32_t* q_pos,
                    const void* kv_cache, int kv_dtype, float kv_scale, int num_blocks,
                    const int32_t* block_table, int max_blocks_per_req,
                    const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                    const mla_segment* segments, int num_segments, int chunk,
                    const void* kv_b_proj, float softmax_scale, float rope_theta, int parts,
                    void* out, int out_dtype, float* lse,
                    void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_prefill_ctx_fp8w -- mla_prefill_ctx for an FP8 cache with the
 * up-projection on the FP8 tensor cores ("DeepSeek MLA — Prefix Cache 与
 * Chunked Prefill 深度解析", section 2.2, the FP8 cache; heading only there):
 * the cache's E4M3 codes are read as stored (640-byte rows, no bf16
 * dequantisation pass) and multiplied on tcgen05 kind::f8f6f4 by an E4M3 copy
 * of kv_b_proj; the fp32 products are scaled by kv_scale * w_scale.  The
 * attention that follows is that of mla_prefill_ctx (bf16 operands, exact
 * scores for rows with few keys).
 * The result is mla_prefill_ctx's with kv_b_proj replaced by
 * e4m3(kv_b_proj / w_scale) * w_scale: the weights' E4M3 rounding (relative
 * error up to 2^-4) moves each up-projected K_nope and V value by about 3%
 * RMS, which the softmax averages over the keys.
 *  kv_b_proj_e4m3_t  device uint8 [H*256][512]: E4M3 codes of kv_b_proj / w_scale,
 *                 transposed (row c holds column c's 512 latent weights), as
 *                 mla_kv_b_proj_to_e4m3 writes them; 16-byte aligned.
 *  w_scale        positive, finite (absmax / 448 uses the whole E4M3 range).
 *  kv_dtype       must be MLA_KV_FP8_E4M3 (MLA_KV_BF16: MLA_ERR_UNSUPPORTED).
 *  workspace      as mla_prefill_ctx (mla_prefill_workspace_size).
 *  other arguments, errors  as mla_prefill_ctx.
 * ---------------------------------------------------------------------- */
int mla_prefill_ctx_fp8w(const void* q, const int32_t* q_pos,
                         const void* kv_cache, int kv_dtype, float kv_scale, int num_blocks,
                         const int32_t* block_table, int max_blocks_per_req,
                         const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                         const mla_segment* segments, int num_segments, int chunk,
                         const void* kv_b_proj_e4m3_t, float w_scale,
                         float softmax_scale, float rope_theta, int parts,
                         void* out, int out_dtype, float* lse,
                         void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* The E4M3 copy of kv_b_proj for mla_prefill_ctx_fp8w, made once per model.
 * mla_kv_b_proj_absmax: *absmax (device fp32) = max |w| over the bf16
 *   kv_b_proj [512, H*256] (one CTA; asynchronous on `stream`).
 * mla_kv_b_proj_to_e4m3: out_e4m3_t[c][k] = e4m3(kv_b_proj[k][c] / w_scale),
 *   rounded to nearest even and saturated to +-448, for c < H*256, k < 512.
 *   out_e4m3_t: device uint8 [H*256][512].
 * Errors: MLA_ERR_INVALID_ARG (null pointer, H outside [1, 128], w_scale not
 * positive and finite), MLA_ERR_CUDA. */
int mla_kv_b_proj_absmax(const void* kv_b_proj, int num_heads, float* absmax, mla_stream_t stream);
int mla_kv_b_proj_to_e4m3(const void* kv_b_proj, int num_heads, float w_scale, void* out_e4m3_t,
                          mla_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_prefill_ctx_noalloc -- mla_prefill_ctx for callers that cannot allocate
 * device memory.  (No section of the pages has a counterpart: this is an
 * integration entry point.)
 *
 * Some callers may not call cudaMalloc: a host framework that owns every
 * device byte through its own pool, code that must not trigger the implicit
 * device synchronisation an allocation can cause, or a caller that is in the
 * middle of capturing a CUDA graph (allocation is refused under global
 * capture mode).  This entry point takes the same arguments as
 * mla_prefill_ctx minus the workspace and runs the same kernels, with their
 * scratch in a fixed array that the library holds in every GPU's memory from
 * the time the library is loaded on that device until the process exits:
 * MLA_NOALLOC_SCRATCH_BYTES (32 MiB).  It calls no cudaMalloc, cudaFree or
 * other device-allocating routine.
 *
 *  - The first call on a device looks up that device's address of the array
 *    (cudaGetSymbolAddress) with the device current and keeps it for the
 *    life of the process; make that first call before any stream capture
 *    begins.
 *  - Arguments are validated as by mla_prefill_ctx first (a call with no
 *    query rows returns MLA_OK without launching).  A problem whose
 *    mla_prefill_min_workspace_size exceeds the array returns
 *    MLA_ERR_TOO_LARGE before anything is launched.  That size is about
 *    0.6 MB of ring lanes plus 1152 B per cached token of the requests and,
 *    for a request cut into several pieces (more than about 16K keys, or
 *    relocated segments), 516 B per query row, head and piece: at 128 heads
 *    one request of up to 16K tokens fits, and little beyond that.
 *  - Every call shares the one array.  Each call re-zeroes the parts that must
 *    start at zero, but calls that may overlap on the GPU (different streams
 *    without ordering between them) race on it: order them.
 *  - mla_get_device_error() does not apply to this entry point's scratch; pass
 *    the same inputs to mla_prefill_ctx to diagnose a bad block table.
 * ---------------------------------------------------------------------- */
#define MLA_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

int mla_prefill_ctx_noalloc(const void* q, const int32_t* q_pos,
                            const void* kv_cache, int kv_dtype, float kv_scale, int num_blocks,
                            const int32_t* block_table, int max_blocks_per_req,
                            const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                            const mla_segment* segments, int num_segments, int chunk,
                            const void* kv_b_proj, float softmax_scale, float rope_theta, int parts,
                            void* out, int out_dtype, float* lse, mla_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_prefill_ctx_absorbed -- the same operation as mla_prefill_ctx (same
 * arguments, same out and lse up to rounding), computed in latent space
 * ("DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析", section 3, the
 * absorbed attention path, named there for decode):
 *   qlat = q_nope W_UK,h^T  (512 wide, per token and head);
 *   s_t  = softmax_scale * (qlat . c_t + R(q_pos - offset) q_rope . k_rope_t),
 *          with c_t, k_rope_t the cached latent row of key t itself, shared by
 *          every head;
 *   o    = sum_t softmax(s)_t c_t  (512 wide);  out = o W_UV,h;  lse as above.
 * No key is up-projected.  Per (query, key, head) it costs 2 * (576 + 512)
 * FLOP instead of 2 * (192 + 128), and it saves the 2 * 512 * 256 FLOP per
 * (key, head) of the up-projection: faster than mla_prefill_ctx while the
 * requests have few queries (about 170 or fewer per request), slower beyond.
 * The caller chooses the entry point.
 *  workspace    device, 256-B aligned, at least
 *               mla_prefill_absorbed_workspace_size(...) bytes (gathered rows,
 *               the absorbed queries [T_q, H, 512] bf16, and fp32 latent
 *               partial states [slots, T_q, H, 512] for the key splits);
 *               smaller -> MLA_ERR_WORKSPACE.  Holds the device error word
 *               read by mla_get_device_error().
 * Errors: as mla_prefill_ctx.
 * ---------------------------------------------------------------------- */
size_t mla_prefill_absorbed_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q,
                                           int num_heads, const mla_segment* segments, int num_segments,
                                           int chunk, int parts);

int mla_prefill_ctx_absorbed(const void* q, const int32_t* q_pos,
                             const void* kv_cache, int kv_dtype, float kv_scale, int num_blocks,
                             const int32_t* block_table, int max_blocks_per_req,
                             const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                             const mla_segment* segments, int num_segments, int chunk,
                             const void* kv_b_proj, float softmax_scale, float rope_theta, int parts,
                             void* out, int out_dtype, float* lse,
                             void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_prefill_ctx_auto -- mla_prefill_ctx with the path chosen per request:
 * a request with at most 208 queries (E_r <= 208) goes through the absorbed
 * path (mla_prefill_ctx_absorbed), the others through the up-projected one,
 * both writing their rows of the same out and lse.  On GB300 the absorbed
 * path is faster below about 230 queries per request (13x at one query,
 * 3.5x at 64, 1.85x at 128, 1.23x at 192, on 32K cached tokens and 128
 * heads) and slower above.
 *  workspace      at least mla_prefill_auto_workspace_size(...) bytes: the
 *                 two paths' workspaces side by side; holds the device error
 *                 word both report into.
 *  other arguments as mla_prefill_ctx.
 * ---------------------------------------------------------------------- */
size_t mla_prefill_auto_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q,
                                       int num_heads, const mla_segment* segments, int num_segments,
                                       int chunk, int parts);

int mla_prefill_ctx_auto(const void* q, const int32_t* q_pos,
                         const void* kv_cache, int kv_dtype, float kv_scale, int num_blocks,
                         const int32_t* block_table, int max_blocks_per_req,
                         const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                         const mla_segment* segments, int num_segments, int chunk,
                         const void* kv_b_proj, float softmax_scale, float rope_theta, int parts,
                         void* out, int out_dtype, float* lse,
                         void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_prefill_ctx_absorbed_fp8 -- mla_prefill_ctx_absorbed for an FP8 cache
 * with the latent part of every score on the FP8 tensor cores: the cache's
 * E4M3 codes are read as stored, and qlat is rounded to E4M3 with one scale
 * per (token, head) row (amax / 448); the k_rope part of the score, the
 * softmax and P c stay as in mla_prefill_ctx_absorbed.  The E4M3 rounding of
 * qlat (relative error up to 2^-4) makes the result an approximation of
 * mla_prefill_ctx's: about 2.5% noise on each score's latent part, which
 * averages over the keys (lse moves by about 0.03 / sqrt(visible keys)).
 *  kv_dtype       must be MLA_KV_FP8_E4M3 (MLA_KV_BF16: MLA_ERR_UNSUPPORTED).
 *  workspace      at least mla_prefill_absorbed_fp8_workspace_size(...) bytes.
 *  other arguments as mla_prefill_ctx.
 * ---------------------------------------------------------------------- */
size_t mla_prefill_absorbed_fp8_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q,
                                               int num_heads, const mla_segment* segments, int num_segments,
                                               int chunk, int parts);

int mla_prefill_ctx_absorbed_fp8(const void* q, const int32_t* q_pos,
                                 const void* kv_cache, int kv_dtype, float kv_scale, int num_blocks,
                                 const int32_t* block_table, int max_blocks_per_req,
                                 const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                                 const mla_segment* segments, int num_segments, int chunk,
                                 const void* kv_b_proj, float softmax_scale, float rope_theta, int parts,
                                 void* out, int out_dtype, float* lse,
                                 void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_prefill_reuse -- head-split reuse with protected-row replacement
 * ("RedKnot-MLA: Multi-Head Offline-Online Reuse for DeepSeek-V4 Long-Context
 * Serving", section 2: Local and Global heads over one packed latent stream;
 * the Global heads and the protected Local rows are recomputed online, the
 * other Local states come from the offline artifact, replaced rather than
 * double counted).  For query row t and head h:
 *   (out, lse)[t, h] = the state mla_prefill_ctx computes with the same
 *                      arguments, if h is a Global head or row t is protected;
 *                      (art_out, art_lse)[t, h] otherwise.
 * Only the recomputed (row, head) pairs are computed: the Global heads for
 * every row, and the Local heads for the protected rows.  The protected rows
 * go through the latent-space (absorbed) path when every request has at most
 * 128 of them and each sees at least 1024 keys (where that path is the
 * faster one), else through the up-projected kernel.
 *  global_heads   HOST int32 [n_global], head indices in [0, H) (repeats ignored).
 *  row_protected  HOST uint8 [T_q], nonzero for a protected row; NULL: none.
 *  art_out        device fp32 [T_q, H, 128];  art_lse  device fp32 [T_q, H].
 *  other arguments, out and lse as mla_prefill_ctx.
 *  workspace      device, 256-B aligned, at least
 *                 mla_prefill_reuse_workspace_size(...) bytes (a smaller one
 *                 returns MLA_ERR_WORKSPACE); holds the device error word.
 * Errors: as mla_prefill_ctx; MLA_ERR_INVALID_ARG for a head outside [0, H).
 * ---------------------------------------------------------------------- */
size_t mla_prefill_reuse_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q,
                                        int num_heads, const mla_segment* segments, int num_segments,
                                        int chunk, int parts, const int32_t* global_heads, int n_global,
                                        const uint8_t* row_protected);

int mla_prefill_reuse(const void* q, const int32_t* q_pos,
                      const void* kv_cache, int kv_dtype, float kv_scale, int num_blocks,
                      const int32_t* block_table, int max_blocks_per_req,
                      const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                      const mla_segment* segments, int num_segments, int chunk,
                      const void* kv_b_proj, float softmax_scale, float rope_theta, int parts,
                      const int32_t* global_heads, int n_global, const uint8_t* row_protected,
                      const float* art_out, const float* art_lse,
                      void* out, int out_dtype, float* lse,
                      void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* Reads and clears the device error word kept in `workspace` (synchronises
 * `stream`).  Returns MLA_OK, MLA_ERR_BAD_BLOCK_ID or MLA_ERR_TIMEOUT. */
int mla_get_device_error(void* workspace, mla_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_merge_states -- merge_attn_states ("DeepSeek MLA — Prefix Cache 与
 * Chunked Prefill 深度解析", section 4.3), one warp per row:
 *   m = max(lse_a, lse_b); wa = e^(lse_a - m); wb = e^(lse_b - m);
 *   out = (wa out_a + wb out_b) / (wa + wb);  lse = m + ln(wa + wb);
 * two rows with lse = -inf merge to (0, -inf).
 *  out_a, out_b, out   device fp32 [rows, d_v]; out may alias out_a or out_b.
 *  lse_a, lse_b, lse   device fp32 [rows]; lse may alias lse_a or lse_b.
 *  d_v                 a positive multiple of 4 (128 on the prefill path).
 * ---------------------------------------------------------------------- */
int mla_merge_states(const float* out_a, const float* lse_a, const float* out_b, const float* lse_b,
                     float* out, float* lse, int64_t rows, int d_v, mla_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_rope_relocate -- query-side RoPE relocation ("RedKnot-MLA ...", section
 * 2, "Online position restoration and merge"): rotate the 64 RoPE columns of
 * every (token, head) row of x by angle (pos[token] - offset) * theta^(-2k/64)
 * on interleaved pairs (2k, 2k+1), k = 0..31.
 *  x, y        device bf16 [tokens, heads, row_stride]; the RoPE part is
 *              columns rope_col .. rope_col+63 (rope_col a multiple of 8).
 *              Only those columns of y are written; y may equal x.
 *  pos         device int32 [tokens].
 * ---------------------------------------------------------------------- */
int mla_rope_relocate(const void* x, const int32_t* pos, int64_t offset, float theta, void* y,
                      int tokens, int heads, int row_stride, int rope_col, mla_stream_t stream);

/* ------------------------------------------------------------------------
 * mla_gather_latent -- _gather_cache of one request's token range
 * ("DeepSeek MLA — Prefix Cache 与 Chunked Prefill 深度解析", section 4.4,
 * step 1): dst[i] = row of token start+i (block_table_row[t/64], slot t%64),
 * as 576 bf16 values.  FP8 rows are dequantised to bf16(e4m3 * kv_scale),
 * rounded to nearest even; bf16 rows are copied bit-exactly.
 *  block_table_row  device int32 [max_blocks]: one request's row.
 *  dst              device bf16 [len, 576].
 *  dev_error        device uint32, optional: bit 0 is set when an entry is
 *                   outside [0, num_blocks) (that row of dst is zeroed).
 * ---------------------------------------------------------------------- */
int mla_gather_latent(const void* kv_cache, int kv_dtype, float kv_scale, int num_blocks,
                      const int32_t* block_table_row, int max_blocks, int start, int len,
                      void* dst, uint32_t* dev_error, mla_stream_t stream);

/* ------------------------------------------------------------------------
 * Content-addressed block store, GPU steps ("PagedAttention assumed MHA.
 * DeepSeek-V4 says that assumption is broken", sections "Position
 * independence beats prefix matching" and "The finding: content-addressed
 * dedup needs byte verification").  A sealed 64-token block is hashed and
 * looked up; on a hash match its bytes are compared with the installed
 * block's, and the candidate is shared only when they are equal (else it is
 * installed fresh and a collision is counted).  The table, that decision and
 * the counter are the caller's; these two calls are the parts that read
 * whole blocks.
 *
 * mla_block_hash: hashes[i] = h(block block_ids[i]) for i < n, where the
 * block's bytes as stored (64 rows of 1152 B bf16 or 640 B FP8) are read as
 * little-endian 64-bit words w_0 .. w_{m-1} and
 *   h = mix(m ^ sum_i mix(w_i + (i + 1) * 0x9e3779b97f4a7c15))  (mod 2^64),
 *   mix(z): z ^= z >> 30; z *= 0xbf58476d1ce4e5b9; z ^= z >> 27;
 *           z *= 0x94d049bb133111eb; z ^= z >> 31   (SplitMix64's output
 *           function).  The page's store uses xxh3; any non-cryptographic
 *           64-bit hash serves, since byte verification decides sharing.
 * mla_block_compare: equal[i] = 1 when blocks block_a[i] and block_b[i] hold
 * the same bytes, else 0.
 *  kv_cache            device, [num_blocks, 64, row] as for mla_prefill_ctx.
 *  block_ids, block_a, block_b   device int32 [n].
 *  hashes              device uint64 [n];  equal  device int32 [n].
 *  dev_error           device uint32, optional: bit 0 is set for an id
 *                      outside [0, num_blocks) (its hash is 0, its equal -1).
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_CUDA.
 * ---------------------------------------------------------------------- */
int mla_block_hash(const void* kv_cache, int kv_dtype, int num_blocks, const int32_t* block_ids, int n,
                   uint64_t* hashes, uint32_t* dev_error, mla_stream_t stream);
int mla_block_compare(const void* kv_cache, int kv_dtype, int num_blocks, const int32_t* block_a,
                      const int32_t* block_b, int n, int32_t* equal, uint32_t* dev_error, mla_stream_t stream);

/* Optional instrumentation.  With both arguments non-NULL (cudaEvent_t handles
 * created by the caller), every later mla_prefill_ctx call on this process
 * records `begin` on its stream just before its first fused prefill kernel
 * launch and `end` just after the last one (mla_prefill_ctx_absorbed: around
 * its latent attention kernel launches), so the caller can time the fused
 * kernel alone with cudaEventElapsedTime.  NULL, NULL turns it off.  The
 * setting is process-wide; the caller keeps the events alive while it is on. */
void mla_set_kernel_events(void* begin_event, void* end_event);

/* Optional tracing of the fused kernel.  With a non-NULL device buffer of at
 * least 64 bytes per role of a call, later mla_prefill_ctx calls write, per
 * role of the persistent kernel's queue, eight 64-bit words: start and end
 * (ns, %globaltimer), CTA / role kind / job, and the ns spent in its main
 * waits.  A call with more roles than the buffer holds is not traced.  NULL
 * turns it off.  Process-wide, like the kernel events. */
void mla_set_trace(void* device_buffer, size_t bytes);

/* Human-readable name of a status code (static storage). */
const char* mla_status_string(int status);

/* Text of the last CUDA runtime error seen by this thread's calls ("" if none). */
const char* mla_last_cuda_error(void);

/* Number of kernels this library has launched in this process (all threads). */
uint64_t mla_launch_count(void);

/* ABI version: 1. */
int mla_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
