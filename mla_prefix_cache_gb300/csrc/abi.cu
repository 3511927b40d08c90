// C-ABI entry points of libmla: argument validation, the host-side planner of
// KV splits, workspace layout and kernel launches.  See include/mla.h for the
// contract of each call.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "absorb.h"
#include "internal.h"
#include "mla.h"

namespace mla {

static std::atomic<uint64_t> g_launches{0};
static std::atomic<void*> g_ev_begin{nullptr};
static std::atomic<void*> g_ev_end{nullptr};
static std::atomic<void*> g_trace{nullptr};
static std::atomic<size_t> g_trace_bytes{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

static thread_local char g_cuda_err[256] = "";

static int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MLA_OK;
  std::snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return MLA_ERR_CUDA;
}

static bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// RoPE inverse frequencies theta^(-2k/64) as binary fractions of a turn per
// unit position (see rope_sincos).
static void rope_fracs(double theta, uint64_t* frac) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int k = 0; k < kDr / 2; ++k) {
    const double f = std::pow(theta, -2.0 * k / (double)kDr);
    const double turns = f / two_pi;                 // in (0, 1/(2 pi)]
    frac[k] = (uint64_t)std::ldexp(turns, 64);       // < 2^64
  }
}

// ------------------------------------------------------------------ planner
struct Plan {
  std::vector<Split> splits;
  std::vector<RowRange> ranges;
  std::vector<uint8_t> skip;   // per request, 1: left to another call (its rows are not touched)
  int max_slots = 0;
  int64_t total_q = 0;
};

// Step "plan" of the path: per request, context chunks of every segment and
// the extend stage become KV splits, each with its own partial-state slot.
// ctx_lens (optional): each request's context length C_r, its extend keys
// then being [C_r, seq_lens[r]) and its cu_q rows a sorted subset of those
// queries (their token indices given to the kernel); default C_r =
// seq_lens[r] - E_r with every query present.
// skip (optional): requests to leave out; their rows keep their places.
static int build_plan(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q, int num_heads,
                      const mla_segment* segs, int nseg, int chunk, int parts, Plan* plan,
                      const int32_t* ctx_lens = nullptr, const uint8_t* skip = nullptr) {
  if (num_reqs < 0 || num_heads < 1 || nseg < 0) return MLA_ERR_INVALID_ARG;
  if (num_heads > kMaxHeads) return MLA_ERR_UNSUPPORTED;
  if (chunk <= 0) return MLA_ERR_INVALID_ARG;
  if (chunk % kBlock != 0) return MLA_ERR_UNSUPPORTED;
  if (parts < 1 || parts > 3) return MLA_ERR_INVALID_ARG;
  if (num_reqs > 0 && (seq_lens == nullptr || cu_q == nullptr)) return MLA_ERR_INVALID_ARG;
  if (nseg > 0 && segs == nullptr) return MLA_ERR_INVALID_ARG;
  if (num_reqs > 0 && cu_q[0] != 0) return MLA_ERR_INVALID_ARG;
  for (int r = 0; r < num_reqs; ++r) {
    const int64_t e = (int64_t)cu_q[r + 1] - cu_q[r];
    if (e < 0 || seq_lens[r] < e) return MLA_ERR_INVALID_ARG;
    if (ctx_lens != nullptr && (ctx_lens[r] < 0 || seq_lens[r] - ctx_lens[r] < e)) return MLA_ERR_INVALID_ARG;
  }
  // segments: inside their request's context, non-overlapping per request
  std::vector<std::vector<const mla_segment*>> per_req(num_reqs);
  for (int i = 0; i < nseg; ++i) {
    const mla_segment& s = segs[i];
    if (s.req < 0 || s.req >= num_reqs || s.reserved != 0 || s.start < 0 || s.len < 0) return MLA_ERR_INVALID_ARG;
    const int64_t ctx = ctx_lens ? (int64_t)ctx_lens[s.req] : (int64_t)seq_lens[s.req] - (cu_q[s.req + 1] - cu_q[s.req]);
    if ((int64_t)s.start + s.len > ctx) return MLA_ERR_INVALID_ARG;
    per_req[s.req].push_back(&s);
  }
  for (auto& v : per_req) {
    std::vector<const mla_segment*> sorted(v);
    std::sort(sorted.begin(), sorted.end(), [](const mla_segment* a, const mla_segment* b) { return a->start < b->start; });
    for (size_t i = 1; i < sorted.size(); ++i)
      if (sorted[i - 1]->start + sorted[i - 1]->len > sorted[i]->start) return MLA_ERR_INVALID_ARG;
  }

  plan->splits.clear();
  plan->ranges.clear();
  plan->skip.assign(num_reqs, 0);
  if (skip != nullptr)
    for (int r = 0; r < num_reqs; ++r) plan->skip[r] = skip[r] ? 1 : 0;
  plan->max_slots = 0;
  plan->total_q = num_reqs > 0 ? cu_q[num_reqs] : 0;
  for (int r = 0; r < num_reqs; ++r) {
    const int E = cu_q[r + 1] - cu_q[r];
    const int C = ctx_lens ? ctx_lens[r] : seq_lens[r] - E;
    if (E == 0 || plan->skip[r]) continue;
    int slots = 0;
    auto add = [&](int k0, int k1, int64_t off) {
      Split sp{};
      sp.req = r;
      sp.q_begin = cu_q[r];
      sp.q_count = E;
      sp.q_tok0 = C;
      sp.k_begin = k0;
      sp.k_end = k1;
      sp.slot = slots++;
      sp.rope_offset = off;
      plan->splits.push_back(sp);
    };
    if (parts & MLA_PART_CONTEXT) {
      if (segs == nullptr) {
        for (int c0 = 0; c0 < C; c0 += chunk) add(c0, std::min(c0 + chunk, C), 0);
      } else {
        for (const mla_segment* s : per_req[r])
          for (int c0 = s->start; c0 < s->start + s->len; c0 += chunk)
            add(c0, std::min(c0 + chunk, s->start + s->len), s->rope_offset);
      }
    }
    if (parts & MLA_PART_EXTEND) add(C, seq_lens[r], 0);
    RowRange rr{};
    rr.row_begin = cu_q[r];
    rr.row_end = cu_q[r + 1];
    rr.nslots = slots;
    plan->ranges.push_back(rr);
    plan->max_slots = std::max(plan->max_slots, slots);
  }
  return MLA_OK;
}

static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }


// ------------------------------------------------------------------ fused path
static int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return (v && *v) ? std::atoi(v) : dflt;
}

struct FusedPlan {
  std::vector<uint8_t> skip;      // the plan's skipped requests
  std::vector<Piece> pieces;      // LPT order, group_begin unset
  std::vector<RowRange> merge;    // requests whose pieces go to partial slots
  std::vector<GatherReq> gather;  // FP8 caches: requests whose rows are dequantised up front
  int gather_blocks = 0;
  int max_slots = 0;
  int64_t total_q = 0;
};

// Pieces: each request's key ranges in order (segments / context chunks, then
// the extend stage); a range joins the previous piece when it continues it
// with the same RoPE offset and the piece is still below max(chunk, 16384)
// keys.  The online softmax inside a piece folds its chunks exactly as
// merge_attn_states would; pieces of one request are folded by the merge
// kernel.
// Exact-score fields of a request's pieces: its leading rows that see fewer
// than kExactKeys keys in all (context keys of every piece plus the causal
// extend keys), and per piece the tiles those rows see and the consumer
// pairs that hold them.  q_tok (host, optional): the token of each row.
static void set_exact(std::vector<Piece>& pr, int C, int E, const int32_t* q_tok) {
  int64_t ctx_keys = 0;
  bool has_ext = false;
  for (const Piece& pc : pr) {
    ctx_keys += std::max(0, std::min(pc.k_end, C) - pc.k_begin);
    has_ext |= pc.k_end > C;
  }
  auto tok = [&](int i) { return q_tok ? q_tok[i] : C + i; };
  int rows = 0;   // rows [0, rows) need exact scores
  while (rows < E && ctx_keys + (has_ext ? (int64_t)tok(rows) - C + 1 : 0) < kExactKeys) ++rows;
  for (Piece& pc : pr) {
    pc.exact = 0;
    if (rows == 0) continue;
    const int t0 = pc.k_begin & ~(kBlock - 1);
    const int vis_end = std::min(pc.k_end, std::max(C, tok(rows - 1) + 1));   // keys those rows see end here
    if (vis_end <= pc.k_begin) continue;
    const int tiles = std::min(kExactSlots, (vis_end - t0 + 127) / 128);
    const int pairs = (rows + 255) / 256;
    pc.exact = tiles | (pairs << 8);
  }
}

static int build_fused_plan(const Plan& splits, const int32_t* seq_lens, const int32_t* cu_q, int num_reqs,
                            int chunk, bool gather_rows, FusedPlan* fp, const int32_t* ctx_lens = nullptr,
                            const int32_t* q_tok = nullptr) {
  fp->skip = splits.skip;
  fp->pieces.clear();
  fp->merge.clear();
  fp->gather.clear();
  fp->gather_blocks = 0;
  fp->max_slots = 0;
  fp->total_q = splits.total_q;
  const int max_keys = std::max(chunk, env_int("MLA_MAX_PIECE_KEYS", 16384));
  // producer CTAs per job (the CTA-pair kernel runs them as pairs): two pairs
  // keep a head's consumers fed now that a pass runs at the MMA rate (on
  // GB300, 0.8% faster than three pairs and far faster than one)
  const int n_prod_cfg = std::max(1, env_int("MLA_PRODUCERS", 4));
  size_t si = 0;
  for (int r = 0; r < num_reqs; ++r) {
    const int E = cu_q[r + 1] - cu_q[r];
    if (E == 0 || (!fp->skip.empty() && fp->skip[r])) continue;
    const int C = ctx_lens ? ctx_lens[r] : seq_lens[r] - E;
    std::vector<Piece> pr;
    std::vector<Split> rs;
    while (si < splits.splits.size() && splits.splits[si].req == r) rs.push_back(splits.splits[si++]);
    std::stable_sort(rs.begin(), rs.end(), [](const Split& a, const Split& b) { return a.k_begin < b.k_begin; });
    for (const Split& sp : rs) {
      if (sp.k_end <= sp.k_begin) continue;
      if (!pr.empty() && pr.back().rope_offset == sp.rope_offset && pr.back().k_end == sp.k_begin &&
          pr.back().k_end - pr.back().k_begin < max_keys) {
        pr.back().k_end = sp.k_end;
        continue;
      }
      Piece pc{};
      pc.req = r;
      pc.q_begin = cu_q[r];
      pc.q_count = E;
      pc.q_tok0 = C;
      pc.k_begin = sp.k_begin;
      pc.k_end = sp.k_end;
      pc.rope_offset = sp.rope_offset;
      pr.push_back(pc);
    }
    set_exact(pr, C, E, q_tok ? q_tok + cu_q[r] : nullptr);
    const int np = (int)pr.size();
    int row_block0 = -1;
    if (gather_rows && np > 0) {
      GatherReq g{};
      g.req = r;
      g.base_block = fp->gather_blocks;
      g.seq_len = seq_lens[r];
      fp->gather.push_back(g);
      row_block0 = fp->gather_blocks;
      fp->gather_blocks += (seq_lens[r] + kBlock - 1) / kBlock;
    }
    for (int i = 0; i < np; ++i) {
      Piece& pc = pr[i];
      pc.row_block0 = row_block0;
      pc.slot = np == 1 ? -1 : i;
      pc.n_cons = (E + 127) / 128;
      const int t0 = pc.k_begin & ~(kBlock - 1);
      const int n_tiles = (pc.k_end - t0 + 127) / 128;
      pc.n_prod = std::max(1, std::min(n_prod_cfg, (n_tiles + 1) / 2));
      fp->pieces.push_back(pc);
    }
    if (np != 1) {
      RowRange rr{};
      rr.row_begin = cu_q[r];
      rr.row_end = cu_q[r + 1];
      rr.nslots = np;
      fp->merge.push_back(rr);
      fp->max_slots = std::max(fp->max_slots, np);
    }
  }
  // longest pieces first
  std::stable_sort(fp->pieces.begin(), fp->pieces.end(), [](const Piece& a, const Piece& b) {
    return (int64_t)a.n_cons * (a.k_end - a.k_begin) > (int64_t)b.n_cons * (b.k_end - b.k_begin);
  });
  return MLA_OK;
}

struct FusedWs {
  size_t err_off = 0, queue_off = 4, flags_off = 256, flags_bytes = 0, ring_off = 0, gath_off = 0, lse_off = 0,
         out_off = 0, total = 0;
  int pieces_per_launch = 0;
  int ring_depth = 0;
  int ring_lanes = 0;
};

// Workspace of the fused path when `ppl` pieces run per launch with `lanes`
// K/V ring lanes of `depth` tiles: header (error word, role queue), per-job
// ring flags, the ring lanes (jobs take turns on them), the gathered rows,
// partial states.
static FusedWs fused_ws_layout(const FusedPlan& fp, int num_heads, int ppl, int depth, int lanes) {
  FusedWs w;
  const size_t jobs = (size_t)ppl * num_heads;
  lanes = (int)std::min<size_t>((size_t)lanes, jobs);   // more lanes than jobs would stay unused
  w.pieces_per_launch = ppl;
  w.ring_depth = depth;
  w.ring_lanes = lanes;
  w.flags_bytes = jobs * 2 * (size_t)depth * sizeof(uint32_t);   // ready and consumed per ring slot
  w.ring_off = up256(w.flags_off + w.flags_bytes);
  // per lane: depth slots of [K_nope | V] tiles, then the K_nope residuals of its first kExactSlots slots
  const size_t ring_bytes = (size_t)lanes * ((size_t)depth * 128 * 256 + (size_t)std::min(depth, kExactSlots) * 128 * 128) *
                            sizeof(uint16_t);
  const size_t rows = (size_t)fp.max_slots * (size_t)fp.total_q * (size_t)num_heads;
  w.gath_off = up256(w.ring_off + ring_bytes);
  const size_t gath_bytes = (size_t)fp.gather_blocks * kBlock * kRowBytesBf16;
  w.lse_off = up256(w.gath_off + gath_bytes);
  w.out_off = up256(w.lse_off + rows * sizeof(float));
  w.total = w.out_off + rows * kDv * sizeof(float);
  return w;
}

// Deepest ring lane: 128 tiles (16384 keys, a whole piece of the default
// plan).  MLA_RING_DEPTH lowers it (a tuning knob; a power of two >= 4).
static int max_ring_depth() {
  int d = kRingDepth;
  const int cap = env_int("MLA_RING_DEPTH", kRingDepth);
  while (d > 4 && d > cap) d /= 2;
  return d;
}

// Heads by which a job's producers precede its consumers in the queue
// (measured best of 1-3); MLA_PRODUCER_LOOKAHEAD, at most 8.
static int producer_lookahead() { return std::min(8, std::max(1, env_int("MLA_PRODUCER_LOOKAHEAD", 2))); }

// Ring lanes.  Two needs set the count:
// - L2: the lanes' tiles stay in L2 while they hold about 32 MiB (measured on
//   GB300: 4 lanes of 16384-key pieces keep the fused kernel's DRAM traffic at
//   its compulsory bytes, 6 lanes of them write most tiles back), that is 32
//   MiB over the longest piece's tiles;
// - occupancy: about as many jobs as the grid's CTA pairs hold at once must
//   have a lane, or pairs go idle: the 76 pairs of a GB300 over the fewest
//   pairs (producers + consumers) a job has.  Jobs with few queries have few
//   consumer pairs each, and their lanes then outnumber what L2 holds.
// The count is the larger of the two, within [lookahead + 2, 64].  A producer
// waits for the lane's previous job, so lanes > lookahead is needed (its
// consumers then precede the producer in the queue), and one more lane keeps
// those waits short.  MLA_RING_LANES sets the count (at least lookahead + 1).
static int ring_lanes_cfg(const FusedPlan& fp, int depth) {
  const int ahead = producer_lookahead();
  const int forced = env_int("MLA_RING_LANES", 0);
  if (forced > 0) return std::max(ahead + 1, forced);
  int max_tiles = 1, min_pairs = 1 << 30;
  for (const Piece& pc : fp.pieces) {
    max_tiles = std::max(max_tiles, (pc.k_end - (pc.k_begin & ~(kBlock - 1)) + 127) / 128);
    min_pairs = std::min(min_pairs, std::max(1, (pc.n_prod + 1) / 2) + (pc.n_cons + 1) / 2);
  }
  const size_t tile_bytes = (size_t)128 * 256 * sizeof(uint16_t);
  const int fit = (int)(((size_t)32 << 20) / (tile_bytes * (size_t)std::min(max_tiles, depth)));
  const int busy = fp.pieces.empty() ? 0 : kLanePairs / min_pairs;
  return std::max(ahead + 2, std::min(kRingLanes, std::max(fit, busy)));
}

// The preferred layout: every piece in one launch (up to kMaxPieces), lanes
// as deep as the longest piece (a power of two, 4 to 128 tiles), so no job
// wraps around its lane; no lanes when there is no piece.
static FusedWs fused_ws_layout(const FusedPlan& fp, int num_heads) {
  const int ppl = std::max(1, std::min((int)fp.pieces.size(), kMaxPieces));
  int max_tiles = 1;
  for (const Piece& pc : fp.pieces)
    max_tiles = std::max(max_tiles, (pc.k_end - (pc.k_begin & ~(kBlock - 1)) + 127) / 128);
  int depth = 4;
  while (depth < max_tiles && depth < max_ring_depth()) depth *= 2;
  depth = std::min(depth, max_ring_depth());
  return fused_ws_layout(fp, num_heads, ppl, depth, fp.pieces.empty() ? 0 : ring_lanes_cfg(fp, depth));
}

// Layout for a workspace of `bytes`: the preferred one when it fits, else
// shallower lanes, then fewer lanes (down to 2, the producers then running
// one head ahead), then fewer pieces per launch; pieces_per_launch 0 when not
// even one piece with two 4-tile lanes fits.
static FusedWs fused_ws_fitting(const FusedPlan& fp, int num_heads, size_t bytes) {
  const FusedWs pref = fused_ws_layout(fp, num_heads);
  if (pref.total <= bytes) return pref;
  for (int depth = pref.ring_depth; depth >= 4; depth /= 2) {
    for (int lanes = pref.ring_lanes; lanes >= 2; --lanes) {
      int hi = pref.pieces_per_launch;
      while (hi >= 1 && fused_ws_layout(fp, num_heads, hi, depth, lanes).total > bytes) hi = hi > 8 ? hi - hi / 8 : hi - 1;
      if (hi >= 1) return fused_ws_layout(fp, num_heads, hi, depth, lanes);
    }
  }
  FusedWs none;
  none.pieces_per_launch = 0;
  return none;
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

static bool encode_map(CUtensorMap* m, CUtensorMapDataType dt, int rank, const void* base, const uint64_t* dims,
                       const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle sw) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides_bytes[i];
  return enc(m, dt, (cuuint32_t)rank, const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mla

using namespace mla;

// Scratch of mla_prefill_ctx_noalloc: one fixed array per device, part of the
// library image, so that entry point never allocates.
static __device__ __align__(256) uint8_t g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];
static void* g_noalloc_ptr[128];
static std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device, looked up once
// per device with that device current.
static int noalloc_scratch(void** out) {
  int dev = 0;
  int st = cuda_status(cudaGetDevice(&dev));
  if (st != MLA_OK) return st;
  if (dev < 0 || dev >= (int)(sizeof(g_noalloc_ptr) / sizeof(g_noalloc_ptr[0]))) return MLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_ptr[dev] == nullptr) {
    void* p = nullptr;
    st = cuda_status(cudaGetSymbolAddress(&p, g_noalloc_scratch));
    if (st != MLA_OK) return st;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return MLA_OK;
}

// The gather pass: every block of the plan's requests, in logical order, into
// `dst` (FP8 rows as exact bf16(e4m3) without the scale).
static int gather_rows(const FusedPlan& fp, const void* kv_cache, bool fp8, int num_blocks, const int32_t* block_table,
                       int max_blocks, uint8_t* dst, uint32_t* err, cudaStream_t s) {
  static GatherBlocksParams gp;   // large; built on the host under a lock
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  std::memset(&gp, 0, sizeof(gp));
  gp.cache = static_cast<const uint8_t*>(kv_cache);
  gp.block_table = block_table;
  gp.err = err;
  gp.fp8 = fp8 ? 1 : 0;
  gp.scale = 1.f;
  gp.num_blocks = num_blocks;
  gp.max_blocks = max_blocks;
  for (size_t g0 = 0; g0 < fp.gather.size(); g0 += kMaxGatherReqs) {
    const size_t n = std::min(fp.gather.size() - g0, (size_t)kMaxGatherReqs);
    int base = fp.gather[g0].base_block, end = base;
    for (size_t i = 0; i < n; ++i) {
      GatherReq g = fp.gather[g0 + i];
      end = g.base_block + (g.seq_len + kBlock - 1) / kBlock;
      g.base_block -= base;
      gp.reqs[i] = g;
    }
    gp.dst = reinterpret_cast<uint16_t*>(dst) + (size_t)base * kBlock * kRowBf16;
    gp.n_reqs = (int)n;
    gp.total_blocks = end - base;
    const int st = cuda_status(launch_gather_blocks(gp, s));
    if (st != MLA_OK) return st;
  }
  return MLA_OK;
}

// The FP8 rows of the plan's requests as stored (640 B), in the same order.
static int gather_rows_raw(const FusedPlan& fp, const void* kv_cache, int num_blocks, const int32_t* block_table,
                           int max_blocks, uint8_t* dst, uint32_t* err, cudaStream_t s) {
  static GatherBlocksParams gp;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  std::memset(&gp, 0, sizeof(gp));
  gp.cache = static_cast<const uint8_t*>(kv_cache);
  gp.block_table = block_table;
  gp.err = err;
  gp.fp8 = 1;
  gp.num_blocks = num_blocks;
  gp.max_blocks = max_blocks;
  for (size_t g0 = 0; g0 < fp.gather.size(); g0 += kMaxGatherReqs) {
    const size_t n = std::min(fp.gather.size() - g0, (size_t)kMaxGatherReqs);
    int base = fp.gather[g0].base_block, end = base;
    for (size_t i = 0; i < n; ++i) {
      GatherReq g = fp.gather[g0 + i];
      end = g.base_block + (g.seq_len + kBlock - 1) / kBlock;
      g.base_block -= base;
      gp.reqs[i] = g;
    }
    gp.dst = reinterpret_cast<uint16_t*>(dst + (size_t)base * kBlock * kRowBytesFp8);
    gp.n_reqs = (int)n;
    gp.total_blocks = end - base;
    const int st = cuda_status(launch_gather_blocks_raw(gp, s));
    if (st != MLA_OK) return st;
  }
  return MLA_OK;
}

// The last block of each of the plan's requests (rows past the sequence as
// zeros), request i of the plan's gather list into block i of `dst`: what the
// absorbed path's P c side reads for a request's last block while it reads
// the cache's other blocks in place.
static int gather_last_blocks(const FusedPlan& fp, const void* kv_cache, int num_blocks, const int32_t* block_table,
                              int max_blocks, uint8_t* dst, uint32_t* err, cudaStream_t s) {
  static GatherBlocksParams gp;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  std::memset(&gp, 0, sizeof(gp));
  gp.cache = static_cast<const uint8_t*>(kv_cache);
  gp.block_table = block_table;
  gp.err = err;
  gp.scale = 1.f;
  gp.num_blocks = num_blocks;
  gp.max_blocks = max_blocks;
  for (size_t g0 = 0; g0 < fp.gather.size(); g0 += kMaxGatherReqs) {
    const size_t n = std::min(fp.gather.size() - g0, (size_t)kMaxGatherReqs);
    for (size_t i = 0; i < n; ++i) {
      GatherReq g = fp.gather[g0 + i];
      g.first_block = std::max(0, (g.seq_len + kBlock - 1) / kBlock - 1);
      g.base_block = (int32_t)i;
      gp.reqs[i] = g;
    }
    gp.dst = reinterpret_cast<uint16_t*>(dst) + g0 * kBlock * kRowBf16;
    gp.n_reqs = (int)n;
    gp.total_blocks = (int)n;
    const int st = cuda_status(launch_gather_blocks(gp, s));
    if (st != MLA_OK) return st;
  }
  return MLA_OK;
}

static int prefill_fused(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                         int num_blocks, const int32_t* block_table, int max_blocks, int num_heads,
                         const void* kv_b_proj, float softmax_scale, float rope_theta, void* out, int out_dtype,
                         float* lse, void* workspace, const FusedPlan& fp, const FusedWs& fw, cudaStream_t s,
                         const int32_t* q_tok = nullptr, bool keep_err = false, const void* w8 = nullptr,
                         float w_scale = 1.f) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int H = num_heads;
  const int64_t T_q = fp.total_q;
  static FusedParams p;            // large; built on the host under a lock
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  std::memset(&p, 0, sizeof(p));

  const bool fp8 = kv_dtype == MLA_KV_FP8_E4M3;
  const bool fp8w = w8 != nullptr;   // FP8 up-projection: E4M3 rows as stored and the E4M3 kv_b_proj copy
  // The gather pass first copies every block the requests use, in logical
  // order, into the workspace (FP8 rows as exact bf16(e4m3), without the
  // scale, which is applied to the fp32 up-projection accumulators; with the
  // FP8 up-projection, the 640-byte rows as stored), so the kernel reads each
  // request's rows contiguously: one 128-row box per k-slice of a producer
  // CTA's pass, one 64-row box of k_rope per consumer CTA and tile.
  const void* rows_base = static_cast<const void*>(ws + fw.gath_off);
  const uint64_t rows_total = (uint64_t)std::max(fp.gather_blocks, 1) * kBlock;
  bool ok = true;
  p.q_bf16 = static_cast<const uint16_t*>(q);
  p.q_tok = q_tok;
  if (fp8w) {
    // the 640-byte rows: codes as bytes (one 128-code k-slice of 128 rows a box), k_rope as bf16 [rows][320]
    const uint64_t d[2] = {(uint64_t)kRowBytesFp8, rows_total};
    const uint64_t st[1] = {(uint64_t)kRowBytesFp8};
    const uint32_t b[2] = {128, 128};
    ok &= encode_map(&p.tm_c8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, rows_base, d, st, b, CU_TENSOR_MAP_SWIZZLE_128B);
    const uint64_t d2[2] = {(uint64_t)kRowBytesFp8 / 2, rows_total};
    const uint32_t b2[2] = {64, 64};
    ok &= encode_map(&p.tm_kr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows_base, d2, st, b2, CU_TENSOR_MAP_SWIZZLE_128B);
    // E4M3 kv_b_proj transposed [H*256][512]: 128 columns x one 128-code k-slice a box
    const uint64_t dw[2] = {(uint64_t)kDc, (uint64_t)H * (kDnope + kDv)};
    const uint64_t sw[1] = {(uint64_t)kDc};
    ok &= encode_map(&p.tm_w8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, w8, dw, sw, b, CU_TENSOR_MAP_SWIZZLE_128B);
    p.krope_col = kRowBytesFp8 / 2 - kDr;   // 256
  } else {
    const uint64_t d[2] = {(uint64_t)kRowBf16, rows_total};
    const uint64_t st[1] = {(uint64_t)kRowBytesBf16};
    const uint32_t b64[2] = {64, 64}, b128[2] = {64, 128}, b256[2] = {64, 256};
    ok &= encode_map(&p.tm_kr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows_base, d, st, b64, CU_TENSOR_MAP_SWIZZLE_128B);
    ok &= encode_map(&p.tm_kr128, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows_base, d, st, b128,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    ok &= encode_map(&p.tm_c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, rows_base, d, st, b256, CU_TENSOR_MAP_SWIZZLE_128B);
    // kv_b_proj [512][H*256] seen as 64-column blocks: (col in block, latent row, block)
    const uint64_t dw[3] = {64, (uint64_t)kDc, (uint64_t)H * (kDnope + kDv) / 64};
    const uint64_t sw[2] = {(uint64_t)H * (kDnope + kDv) * 2, 128};
    const uint32_t bw[3] = {64, 64, 2};
    ok &= encode_map(&p.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv_b_proj, dw, sw, bw, CU_TENSOR_MAP_SWIZZLE_128B);
    p.krope_col = kDc;
  }
  {
    // ring lanes: per lane and slot four contiguous [128 x 64] blocks K_nope cols 0-63, 64-127, V cols 0-63,
    // 64-127; after every lane's slots, per lane and residual slot two blocks of the K_nope residual
    const uint64_t d[3] = {64, 128, (uint64_t)fw.ring_lanes * ((uint64_t)fw.ring_depth * 4 +
                                                            (uint64_t)std::min(fw.ring_depth, kExactSlots) * 2)};
    const uint64_t st[2] = {128, 128 * 128};
    const uint32_t b[3] = {64, 128, 2};
    ok &= encode_map(&p.tm_ring, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ws + fw.ring_off, d, st, b,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    const uint32_t b1[3] = {64, 128, 1}, b64[3] = {64, 64, 2};
    ok &= encode_map(&p.tm_ring1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ws + fw.ring_off, d, st, b1,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    ok &= encode_map(&p.tm_ring64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ws + fw.ring_off, d, st, b64,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (T_q > 0) {
    const uint64_t d[3] = {(uint64_t)kDqk, (uint64_t)H, (uint64_t)T_q};
    const uint64_t st[2] = {(uint64_t)kDqk * 2, (uint64_t)H * kDqk * 2};
    const uint32_t b[3] = {64, 1, 128};
    ok &= encode_map(&p.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, d, st, b, CU_TENSOR_MAP_SWIZZLE_128B);
    // out and the partial states as (column, head, row): a consumer stores a
    // full 128-row tile of one head with 128-byte boxes
    const bool ob = out_dtype == MLA_OUT_BF16;
    const uint64_t es = ob ? 2 : 4;
    const uint64_t dout[3] = {(uint64_t)kDv, (uint64_t)H, (uint64_t)T_q};
    const uint64_t sout[2] = {(uint64_t)kDv * es, (uint64_t)H * kDv * es};
    const uint32_t bout[3] = {ob ? 64u : 32u, 1, 128};
    ok &= encode_map(&p.tm_out, ob ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, out, dout,
                     sout, bout, CU_TENSOR_MAP_SWIZZLE_128B);
    if (fp.max_slots > 0) {
      const uint64_t dpart[3] = {(uint64_t)kDv, (uint64_t)H, (uint64_t)fp.max_slots * (uint64_t)T_q};
      const uint64_t spart[2] = {(uint64_t)kDv * 4, (uint64_t)H * kDv * 4};
      const uint32_t bpart[3] = {32, 1, 128};
      ok &= encode_map(&p.tm_part, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ws + fw.out_off, dpart, spart, bpart,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    }
  }
  if (!ok) return MLA_ERR_CUDA;

  uint32_t* err = reinterpret_cast<uint32_t*>(ws + fw.err_off);
  p.err = err;
  p.queue = reinterpret_cast<uint32_t*>(ws + fw.queue_off);
  p.flags = reinterpret_cast<uint32_t*>(ws + fw.flags_off);
  p.ring = reinterpret_cast<uint16_t*>(ws + fw.ring_off);
  p.block_table = block_table;
  p.q_pos = q_pos;
  p.out = out;
  p.lse = lse;
  p.part_out = reinterpret_cast<float*>(ws + fw.out_off);
  p.part_lse = reinterpret_cast<float*>(ws + fw.lse_off);
  p.slot_stride_rows = T_q;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.num_heads = H;
  p.out_bf16 = out_dtype == MLA_OUT_BF16;
  p.out_scale = fp8w ? kv_scale * w_scale : (fp8 ? kv_scale : 1.f);
  p.fp8w = fp8w ? 1 : 0;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  rope_fracs((double)rope_theta, p.rope_frac);

  // The persistent CTA-pair kernel (fused2.cu): every role runs on a cluster
  // of two CTAs with M = 256 MMAs.  MLA_FUSED_GRID caps the persistent grid (a
  // tuning and measurement knob; the role queue is correct for any grid with
  // more CTA pairs than producer pairs per job).
  int grid = 0;
  int st = cuda_status(fused2_grid_size(&grid));
  if (st != MLA_OK) return st;
  grid = std::min(grid, std::max(8, env_int("MLA_FUSED_GRID", grid))) & ~1;
  p.ring_depth = fw.ring_depth;
  p.ring_lanes = fw.ring_lanes;
  // Producers run prod_ahead heads ahead of their consumers in the queue
  // (capped at 8: on a ring shallower than a piece, producers that run ahead
  // wait for their consumers, and fewer than the grid's pairs may wait at
  // once), and fewer than the ring lanes: a producer waits for the lane's
  // previous job, whose consumers must precede it in the queue.
  p.prod_ahead = std::max(1, std::min(producer_lookahead(), fw.ring_lanes - 1));
  // Every wait of the kernel gives up after 2 s (the error word then reads
  // MLA_ERR_TIMEOUT).  Tests shorten it (MLA_WAIT_LIMIT_US, at least 1 ms) and
  // withhold the producers of one job (MLA_TEST_WITHHOLD_JOB) to make a wait
  // run out on purpose.
  p.wait_limit_ns = (uint64_t)std::max(1000, std::min(2000000, env_int("MLA_WAIT_LIMIT_US", 2000000))) * 1000ull;
  p.withhold_job = env_int("MLA_TEST_WITHHOLD_JOB", -1);
  p.l2_hints = env_int("MLA_L2_HINTS", 1) != 0 ? 1 : 0;
  // error word + role queue (keep_err: a caller running several sub-calls keeps the error word)
  st = keep_err ? cuda_status(cudaMemsetAsync(err + 1, 0, 256 - 4, s)) : cuda_status(cudaMemsetAsync(err, 0, 256, s));
  if (st != MLA_OK) return st;
  st = fp8w ? gather_rows_raw(fp, kv_cache, num_blocks, block_table, max_blocks, ws + fw.gath_off, err, s)
            : gather_rows(fp, kv_cache, fp8, num_blocks, block_table, max_blocks, ws + fw.gath_off, err, s);
  if (st != MLA_OK) return st;

  cudaEvent_t ev_b = static_cast<cudaEvent_t>(g_ev_begin.load());
  cudaEvent_t ev_e = static_cast<cudaEvent_t>(g_ev_end.load());
  if (ev_b != nullptr && ev_e != nullptr && (st = cuda_status(cudaEventRecord(ev_b, s))) != MLA_OK) return st;
  const size_t ppl = (size_t)std::max(fw.pieces_per_launch, 1);
  for (size_t b0 = 0; b0 < fp.pieces.size(); b0 += ppl) {
    const size_t n = std::min(fp.pieces.size() - b0, ppl);
    int groups = 0;
    for (size_t i = 0; i < n; ++i) {
      Piece pc = fp.pieces[b0 + i];
      pc.group_begin = groups;
      pc.n_prod = std::max(1, (pc.n_prod + 1) / 2);   // producer roles of a pair: two CTAs each
      groups += H * (pc.n_prod + (pc.n_cons + 1) / 2);
      p.pieces[i] = pc;
    }
    p.n_pieces = (int)n;
    p.n_groups = groups;
    const size_t slots = (size_t)groups * 2;   // trace slot = group * 2 + cluster rank
    void* tr = g_trace.load();
    p.trace = (tr != nullptr && g_trace_bytes.load() >= slots * kTraceWords * 8 && fp.pieces.size() <= ppl)
                  ? static_cast<unsigned long long*>(tr) : nullptr;
    // per-stage detail of one role slot when the buffer has room for 4096 more stages
    p.trace_detail_role = (p.trace && g_trace_bytes.load() >= (slots * kTraceWords + 4096 * 8) * 8)
                              ? env_int("MLA_TRACE_DETAIL_ROLE", -1) : -1;
    if (b0 > 0 && (st = cuda_status(cudaMemsetAsync(p.queue, 0, sizeof(uint32_t), s))) != MLA_OK) return st;
    if ((st = cuda_status(cudaMemsetAsync(p.flags, 0, fw.flags_bytes, s))) != MLA_OK) return st;
    const cudaError_t le = launch_fused2(p, std::min(grid, groups * 2), s);
    if ((st = cuda_status(le)) != MLA_OK) return st;
  }
  if (ev_b != nullptr && ev_e != nullptr && (st = cuda_status(cudaEventRecord(ev_e, s))) != MLA_OK) return st;

  if (!fp.merge.empty()) {
    MergeParams mp;
    std::memset(&mp, 0, sizeof(mp));
    mp.part_out = p.part_out;
    mp.part_lse = p.part_lse;
    mp.slot_stride_rows = T_q;
    mp.out = out;
    mp.lse = lse;
    mp.out_bf16 = p.out_bf16;
    mp.num_heads = H;
    for (size_t b0 = 0; b0 < fp.merge.size(); b0 += kMaxRangesPerLaunch) {
      const size_t n = std::min(fp.merge.size() - b0, (size_t)kMaxRangesPerLaunch);
      int rows = 0;
      for (size_t i = 0; i < n; ++i) {
        RowRange rr = fp.merge[b0 + i];
        rr.prefix = rows;
        rows += rr.row_end - rr.row_begin;
        mp.ranges[i] = rr;
      }
      mp.num_ranges = (int)n;
      mp.total_rows = rows;
      if ((st = cuda_status(launch_merge_slots(mp, s))) != MLA_OK) return st;
    }
  }
  return MLA_OK;
}


// ------------------------------------------------------------------ absorbed path
struct AbsPlan {
  std::vector<AbsPiece> pieces;    // the fused plan's pieces, LPT order
  std::vector<RowRange> ranges;    // every request with queries, with its slot count
  int max_slots = 0;
  bool any_merge = false;
  int64_t items = 0;
};

// Estimated run time, in keys of one work item, of the absorbed path's
// latent attention and merge when every piece's keys are cut into splits of
// at most `split` keys: the items (rows_per_item rows x one split each) are
// placed longest first on the least-loaded of `clusters` resident clusters
// (items of one piece and length go round by round), each item also paying
// `item_keys` of start and epilogue; a request cut into several slots adds the
// merge of its latent states (a pass over the whole GPU), `merge_keys_per_row`
// per (row, slot + 1).
// With `bound` > 0 it stops at a lower bound (the items' work spread evenly,
// plus the merge) when that is already at least `bound`, returns it and sets
// *bounded.
static double abs_split_cost(const std::vector<Piece>& pieces, int H, int64_t rows_per_item, int split,
                             int clusters, double item_keys, double merge_keys_per_row, int num_reqs,
                             double bound = 0.0, bool* bounded = nullptr) {
  std::vector<std::pair<int, int64_t>> groups;   // (item length in keys, item count)
  std::vector<int> slots(num_reqs, 0);
  std::vector<int64_t> rows(num_reqs, 0);
  double work = 0.0;
  for (const Piece& pc : pieces) {
    const int keys = pc.k_end - pc.k_begin;
    const int ns = std::max(1, (keys + split - 1) / split);
    const int64_t r_items = (pc.q_count * (int64_t)H + rows_per_item - 1) / rows_per_item;
    groups.push_back({(keys + ns - 1) / ns, r_items * ns});
    work += (double)r_items * ns * ((keys + ns - 1) / ns + item_keys);
    slots[pc.req] += ns;
    rows[pc.req] = pc.q_count * (int64_t)H;
  }
  double merge = 0.0;
  for (int r = 0; r < num_reqs; ++r)
    if (slots[r] > 1) merge += merge_keys_per_row * (double)rows[r] * (slots[r] + 1);
  const double lower = work / clusters + merge;
  if (bound > 0.0 && lower >= bound) {
    if (bounded) *bounded = true;
    return lower;
  }
  std::sort(groups.begin(), groups.end(), [](const auto& a, const auto& b) { return a.first > b.first; });
  std::vector<double> load(clusters, 0.0);
  for (const auto& g : groups) {
    const double len = g.first + item_keys;
    const int64_t full = g.second / clusters;
    const int rem = (int)(g.second - full * clusters);
    if (full > 0)
      for (double& l : load) l += (double)full * len;
    if (rem > 0) {
      std::partial_sort(load.begin(), load.begin() + rem, load.end());
      for (int i = 0; i < rem; ++i) load[i] += len;
    }
  }
  return *std::max_element(load.begin(), load.end()) + merge;
}

// The absorbed path's pieces: the fused plan's pieces of a request that share
// its query rows and RoPE offset and whose key ranges meet are one piece (the
// chunk bounds the up-projected K/V, which this path does not form), longest
// first.
static std::vector<Piece> abs_pieces(const FusedPlan& fp) {
  std::vector<Piece> v = fp.pieces;
  std::sort(v.begin(), v.end(), [](const Piece& a, const Piece& b) {
    if (a.req != b.req) return a.req < b.req;
    if (a.rope_offset != b.rope_offset) return a.rope_offset < b.rope_offset;
    return a.k_begin < b.k_begin;
  });
  std::vector<Piece> out;
  for (const Piece& pc : v) {
    if (!out.empty()) {
      Piece& l = out.back();
      if (l.req == pc.req && l.rope_offset == pc.rope_offset && l.q_begin == pc.q_begin &&
          l.q_count == pc.q_count && l.q_tok0 == pc.q_tok0 && l.row_block0 == pc.row_block0 &&
          l.k_end == pc.k_begin) {
        l.k_end = pc.k_end;
        continue;
      }
    }
    out.push_back(pc);
  }
  std::stable_sort(out.begin(), out.end(), [](const Piece& a, const Piece& b) {
    return (int64_t)(a.k_end - a.k_begin) * a.q_count > (int64_t)(b.k_end - b.k_begin) * b.q_count;
  });
  return out;
}

// Work items of the absorbed path: each piece's tiles of 256 rows of
// (token, head) pairs, each tile's keys cut into splits of split_keys (a
// multiple of the 128-key tile, at least 512).  The split size is the one
// of the longest piece's keys cut 1 to 64 ways with the least estimated time
// (abs_split_cost, with the kernels' measured costs); MLA_ABS_SPLIT_KEYS
// overrides it (rounded up to a multiple of the key tile).
static void build_abs_plan(const FusedPlan& fp, int H, const int32_t* cu_q, int num_reqs, AbsPlan* ap) {
  ap->pieces.clear();
  ap->ranges.clear();
  ap->max_slots = 0;
  ap->any_merge = false;
  ap->items = 0;
  const int64_t rows_per_item = 256;
  const int key_tile = 128;
  // resident clusters (36 of four CTAs on a GB300), an item's start and epilogue (about 8 us) and the
  // latent merge (2 KB read or written per row and slot at about 3.5 TB/s) in keys of an item (about
  // 1.36 us per 128 keys)
  const int clusters = 36;
  const double ns_per_key = 10.6;
  const double item_keys = 8000.0 / ns_per_key;
  const double merge_keys_per_row = 2048.0 / 3500.0 / ns_per_key;   // bytes / (bytes per ns) / (ns per key)
  const std::vector<Piece> pieces = abs_pieces(fp);
  int k_max = 0;
  for (const Piece& pc : pieces) k_max = std::max(k_max, pc.k_end - pc.k_begin);
  auto round_split = [&](int v) { return std::max(512, (v + key_tile - 1) & ~(key_tile - 1)); };
  int split = round_split(std::max(k_max, 1));
  const int forced = env_int("MLA_ABS_SPLIT_KEYS", 0);
  double best = forced > 0 ? 0.0
                           : abs_split_cost(pieces, H, rows_per_item, split, clusters, item_keys, merge_keys_per_row,
                                            num_reqs);
  int last = split;
  for (int ways = 2; ways <= 64 && k_max > 512 && forced <= 0; ++ways) {
    const int cand = round_split((k_max + ways - 1) / ways);
    if (cand >= last) continue;   // the same cut as a fewer-way one once rounded
    last = cand;
    // finer cuts only add items (each with its start and epilogue) and slots to merge, so once the
    // lower bound of a cut reaches the best estimate the search ends
    bool bounded = false;
    const double c = abs_split_cost(pieces, H, rows_per_item, cand, clusters, item_keys, merge_keys_per_row,
                                    num_reqs, best * 0.99, &bounded);
    if (bounded) break;
    if (c < best * 0.99) {   // a split must buy a clear gain: more items and slots cost workspace
      best = c;
      split = cand;
    }
  }
  if (forced > 0) split = (forced + key_tile - 1) & ~(key_tile - 1);
  std::vector<int> next_slot(num_reqs, 0);
  for (const Piece& pc : pieces) {
    AbsPiece a{};
    a.req = pc.req;
    a.q_begin = pc.q_begin;
    a.q_count = pc.q_count;
    a.q_tok0 = pc.q_tok0;
    a.k_begin = pc.k_begin;
    a.k_end = pc.k_end;
    a.row_block0 = pc.row_block0;
    a.rope_offset = pc.rope_offset;
    a.n_row_tiles = (int)((pc.q_count * (int64_t)H + rows_per_item - 1) / rows_per_item);
    const int keys = pc.k_end - pc.k_begin;
    a.n_splits = std::max(1, (keys + split - 1) / split);
    a.split_keys = ((keys + a.n_splits - 1) / a.n_splits + key_tile - 1) & ~(key_tile - 1);
    a.slot = next_slot[pc.req];
    next_slot[pc.req] += a.n_splits;
    ap->pieces.push_back(a);
  }
  for (int r = 0; r < num_reqs; ++r) {
    if (cu_q[r + 1] == cu_q[r] || (!fp.skip.empty() && fp.skip[r])) continue;
    RowRange rr{};
    rr.row_begin = cu_q[r];
    rr.row_end = cu_q[r + 1];
    rr.nslots = next_slot[r];
    ap->ranges.push_back(rr);
    ap->max_slots = std::max(ap->max_slots, rr.nslots);
    ap->any_merge |= rr.nslots > 1;
  }
}

struct AbsWs {
  size_t gath_off = 0, qlat_off = 0, lat_out_off = 0, lat_lse_off = 0, qlat8_off = 0, qscale_off = 0,
         total = 0;
};

// Workspace of the absorbed path: header (error word), gathered rows, the
// absorbed queries and the latent states of every slot (a request's slots are
// merged into slot 0 before the output projection).
static AbsWs abs_ws_layout(const FusedPlan& fp, const AbsPlan& ap, int H, bool fp8_scores = false) {
  AbsWs w;
  const size_t rows = (size_t)fp.total_q * (size_t)H;
  const size_t slots = (size_t)std::max(ap.max_slots, 1);
  w.gath_off = 256;
  w.qlat_off = up256(w.gath_off + (size_t)fp.gather_blocks * kBlock * kRowBytesBf16);
  w.lat_out_off = up256(w.qlat_off + rows * kDc * sizeof(uint16_t));
  w.lat_lse_off = up256(w.lat_out_off + slots * rows * kDc * sizeof(float));
  w.total = up256(w.lat_lse_off + slots * rows * sizeof(float));
  if (fp8_scores) {   // E4M3 scores: E4M3 qlat and its row scales (the FP8 rows are read in place)
    w.qlat8_off = w.total;
    w.qscale_off = up256(w.qlat8_off + rows * kDc);
    w.total = up256(w.qscale_off + rows * sizeof(float));
  }
  return w;
}

static int prefill_absorbed(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                            int num_blocks, const int32_t* block_table, int max_blocks, int H, const void* kv_b_proj,
                            float softmax_scale, float rope_theta, void* out, int out_dtype, float* lse,
                            void* workspace, const FusedPlan& fp, const AbsPlan& ap, const AbsWs& aw,
                            cudaStream_t s, bool fp8_scores = false, uint32_t* err_word = nullptr,
                            const int32_t* q_tok = nullptr) {
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t T_q = fp.total_q;
  static AbsorbParams p;           // large; built on the host under a lock
  static ProjParams pp;
  static MergeParams mp;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  std::memset(&p, 0, sizeof(p));
  const bool fp8 = kv_dtype == MLA_KV_FP8_E4M3;
  const float vscale = fp8 ? kv_scale : 1.f;
  // err_word: a caller running several sub-calls gives the one word they all report into
  uint32_t* err = err_word ? err_word : reinterpret_cast<uint32_t*>(ws);

  const void* rows_base = static_cast<const void*>(ws + aw.gath_off);
  const uint64_t rows_total = (uint64_t)std::max(fp.gather_blocks, 1) * kBlock;
  bool ok = true;
  {
    // [c | k_rope] of a bf16 row as 9 blocks of 64 columns: three to a box for the scores, the latent
    // blocks two to a box for P c; qlat 128 rows x 64 columns to a box
    const uint64_t d[3] = {64, rows_total, 9};
    const uint64_t st[2] = {(uint64_t)kRowBytesBf16, 128};
    const uint32_t b[3] = {64, 64, 3}, b2[3] = {64, 64, 2};
    ok &= encode_map(&p.tm_c3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, rows_base, d, st, b, CU_TENSOR_MAP_SWIZZLE_128B);
    ok &= encode_map(&p.tm_c2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, rows_base, d, st, b2, CU_TENSOR_MAP_SWIZZLE_128B);
    const uint64_t d3[2] = {(uint64_t)kDc, (uint64_t)T_q * H};
    const uint64_t st3[1] = {(uint64_t)kDc * 2};
    const uint32_t b3[2] = {64, 128};
    ok &= encode_map(&p.tm_qlat, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ws + aw.qlat_off, d3, st3, b3,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    // the latent states of every slot, 32 columns x 128 rows to a box (the epilogue's stores)
    const uint64_t dl[2] = {(uint64_t)kDc, (uint64_t)std::max(ap.max_slots, 1) * (uint64_t)T_q * H};
    const uint64_t sl[1] = {(uint64_t)kDc * sizeof(float)};
    const uint32_t bl[2] = {32, 128};
    ok &= encode_map(&p.tm_lat, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ws + aw.lat_out_off, dl, sl, bl,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  }
  // Rows read in place: a score stage or a P c stage is one whole cache block, so both sides read a BF16
  // cache's blocks where they are (P c takes a request's last block from a copy whose rows past the
  // sequence are zeros), and E4M3 scores read an FP8 cache's rows as stored; an FP8 cache's P c side, and
  // its bf16 scores, read the dequantised rows of the gather pass.
  p.s_in_place = (!fp8 || fp8_scores) ? 1 : 0;
  p.o_in_place = fp8 ? 0 : 1;
  p.block_table = block_table;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  {
    const uint64_t rows_cache = (uint64_t)std::max(num_blocks, 1) * kBlock;
    if (!fp8) {
      const uint64_t d[3] = {64, rows_cache, 9};
      const uint64_t st[2] = {(uint64_t)kRowBytesBf16, 128};
      const uint32_t b[3] = {64, 64, 3}, b2[3] = {64, 64, 2};
      ok &= encode_map(&p.tm_k3, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv_cache, d, st, b, CU_TENSOR_MAP_SWIZZLE_128B);
      ok &= encode_map(&p.tm_k2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, kv_cache, d, st, b2, CU_TENSOR_MAP_SWIZZLE_128B);
    } else if (fp8_scores) {
      // a 640-byte row as stored as 5 blocks of 128 bytes (4 of E4M3 codes, k_rope as bf16), one box a stage
      const uint64_t d[3] = {128, rows_cache, 5};
      const uint64_t st[2] = {(uint64_t)kRowBytesFp8, 128};
      const uint32_t b[3] = {128, 64, 5};
      ok &= encode_map(&p.tm_f5, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, kv_cache, d, st, b, CU_TENSOR_MAP_SWIZZLE_128B);
    }
  }
  if (fp8_scores) {
    // the E4M3 qlat 128 rows x 128 bytes to a box (the FP8 rows themselves are read in place, tm_f5 below)
    const uint64_t d3[2] = {(uint64_t)kDc, (uint64_t)T_q * H};
    const uint64_t st3[1] = {(uint64_t)kDc};
    const uint32_t b3[2] = {128, 128};
    ok &= encode_map(&p.tm_qlat8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ws + aw.qlat8_off, d3, st3, b3,
                     CU_TENSOR_MAP_SWIZZLE_128B);
    p.qscale = reinterpret_cast<const float*>(ws + aw.qscale_off);
    p.kv_scale = kv_scale;
    p.fp8_scores = 1;
  }
  if (!ok) return MLA_ERR_CUDA;

  int st = err_word ? MLA_OK : cuda_status(cudaMemsetAsync(err, 0, 256, s));
  if (st != MLA_OK) return st;
  st = p.o_in_place ? gather_last_blocks(fp, kv_cache, num_blocks, block_table, max_blocks, ws + aw.gath_off, err, s)
                    : gather_rows(fp, kv_cache, fp8, num_blocks, block_table, max_blocks, ws + aw.gath_off, err, s);
  if (st != MLA_OK) return st;
  {
    static QAbsorbParams qp;
    std::memset(&qp, 0, sizeof(qp));
    qp.qscale = fp8_scores ? reinterpret_cast<float*>(ws + aw.qscale_off) : nullptr;
    qp.err = err;
    qp.scale = fp8_scores ? 1.f : vscale;   // E4M3 scores: kv_scale enters through the per-row score factor
    qp.num_heads = H;
    const uint64_t dw[2] = {(uint64_t)H * (kDnope + kDv), (uint64_t)kDc};
    const uint64_t sw[1] = {(uint64_t)H * (kDnope + kDv) * 2};
    const uint32_t bw[2] = {64, 256};
    if (!encode_map(&qp.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_b_proj, dw, sw, bw, CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
    // only the rows of this call's requests, one launch per run of adjacent ones;
    // the maps end at the run's last token so the tile past it reads zeros and
    // stores nothing
    for (size_t i = 0; i < ap.ranges.size();) {
      size_t j = i + 1;
      while (j < ap.ranges.size() && ap.ranges[j].row_begin == ap.ranges[j - 1].row_end) ++j;
      qp.row0 = ap.ranges[i].row_begin;
      qp.tokens = ap.ranges[j - 1].row_end - ap.ranges[i].row_begin;
      const uint64_t row_end = (uint64_t)ap.ranges[j - 1].row_end;
      const uint64_t dq[3] = {(uint64_t)kDqk, (uint64_t)H, row_end};
      const uint64_t sq[2] = {(uint64_t)kDqk * 2, (uint64_t)H * kDqk * 2};
      const uint32_t bq[3] = {64, 1, 128};
      bool ok2 = encode_map(&qp.tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dq, sq, bq, CU_TENSOR_MAP_SWIZZLE_128B);
      const uint64_t dl[3] = {(uint64_t)kDc, (uint64_t)H, row_end};
      if (fp8_scores) {
        const uint64_t sl[2] = {(uint64_t)kDc, (uint64_t)H * kDc};
        const uint32_t bl[3] = {128, 1, 128};
        ok2 &= encode_map(&qp.tm_out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, ws + aw.qlat8_off, dl, sl, bl,
                          CU_TENSOR_MAP_SWIZZLE_128B);
      } else {
        const uint64_t sl[2] = {(uint64_t)kDc * 2, (uint64_t)H * kDc * 2};
        const uint32_t bl[3] = {64, 1, 128};
        ok2 &= encode_map(&qp.tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, ws + aw.qlat_off, dl, sl, bl,
                          CU_TENSOR_MAP_SWIZZLE_128B);
      }
      if (!ok2) return MLA_ERR_CUDA;
      if ((st = cuda_status(launch_qabsorb(qp, s))) != MLA_OK) return st;
      i = j;
    }
  }

  p.q = static_cast<const uint16_t*>(q);
  p.qlat = reinterpret_cast<const uint16_t*>(ws + aw.qlat_off);
  p.q_pos = q_pos;
  p.q_tok = q_tok;
  p.lat_out = reinterpret_cast<float*>(ws + aw.lat_out_off);
  p.lat_lse = reinterpret_cast<float*>(ws + aw.lat_lse_off);
  p.slot_stride_rows = T_q * H;
  p.err = err;
  p.num_heads = H;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  rope_fracs((double)rope_theta, p.rope_frac);
  cudaEvent_t ev_b = static_cast<cudaEvent_t>(g_ev_begin.load());
  cudaEvent_t ev_e = static_cast<cudaEvent_t>(g_ev_end.load());
  if (ev_b != nullptr && ev_e != nullptr && (st = cuda_status(cudaEventRecord(ev_b, s))) != MLA_OK) return st;
  int req_max = 0;
  for (const GatherReq& g : fp.gather) req_max = std::max(req_max, g.req + 1);
  std::vector<int> greq(req_max, 0);   // request -> its place in the gather list
  for (size_t i = 0; i < fp.gather.size(); ++i) greq[fp.gather[i].req] = (int)i;
  for (size_t b0 = 0; b0 < ap.pieces.size(); b0 += kMaxAbsPieces) {
    const size_t n = std::min(ap.pieces.size() - b0, (size_t)kMaxAbsPieces);
    int64_t items = 0;
    for (size_t i = 0; i < n; ++i) {
      AbsPiece a = ap.pieces[b0 + i];
      const int gi = greq[a.req];
      a.last_lb = std::max(0, (fp.gather[gi].seq_len + kBlock - 1) / kBlock - 1);
      if (p.o_in_place) a.row_block0 = gi;   // the copy of the request's last block
      a.item_begin = (int32_t)items;
      items += (int64_t)a.n_row_tiles * a.n_splits;
      p.pieces[i] = a;
    }
    if (items > (int64_t)1 << 30) return MLA_ERR_UNSUPPORTED;
    p.n_pieces = (int)n;
    p.n_items = (int)items;
    if ((st = cuda_status(launch_absorb_attn(p, s))) != MLA_OK) return st;
  }
  if (ev_b != nullptr && ev_e != nullptr && (st = cuda_status(cudaEventRecord(ev_e, s))) != MLA_OK) return st;

  // fold each request's slots into slot 0, in latent space
  if (ap.any_merge) {
    std::memset(&mp, 0, sizeof(mp));
    mp.part_out = p.lat_out;
    mp.part_lse = p.lat_lse;
    mp.slot_stride_rows = T_q;
    mp.out = p.lat_out;
    mp.lse = p.lat_lse;
    mp.out_bf16 = 0;
    mp.num_heads = H;
    std::vector<RowRange> multi;
    for (const RowRange& rr : ap.ranges)
      if (rr.nslots > 1) multi.push_back(rr);
    for (size_t b0 = 0; b0 < multi.size(); b0 += kMaxRangesPerLaunch) {
      const size_t n = std::min(multi.size() - b0, (size_t)kMaxRangesPerLaunch);
      int rows = 0;
      for (size_t i = 0; i < n; ++i) {
        RowRange rr = multi[b0 + i];
        rr.prefix = rows;
        rows += rr.row_end - rr.row_begin;
        mp.ranges[i] = rr;
      }
      mp.num_ranges = (int)n;
      mp.total_rows = rows;
      if ((st = cuda_status(launch_merge_slots_latent(mp, s))) != MLA_OK) return st;
    }
  }
  std::memset(&pp, 0, sizeof(pp));
  {
    const uint64_t dw[2] = {(uint64_t)H * (kDnope + kDv), (uint64_t)kDc};
    const uint64_t sw[1] = {(uint64_t)H * (kDnope + kDv) * 2};
    const uint32_t bw[2] = {64, 128};
    if (!encode_map(&pp.tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv_b_proj, dw, sw, bw, CU_TENSOR_MAP_SWIZZLE_128B))
      return MLA_ERR_CUDA;
  }
  pp.lat_out = p.lat_out;
  pp.lat_lse = p.lat_lse;
  pp.err = err;
  pp.out = out;
  pp.lse = lse;
  pp.out_bf16 = out_dtype == MLA_OUT_BF16;
  pp.scale = vscale;
  pp.num_heads = H;
  for (size_t b0 = 0; b0 < ap.ranges.size(); b0 += kMaxRangesPerLaunch) {
    const size_t n = std::min(ap.ranges.size() - b0, (size_t)kMaxRangesPerLaunch);
    int rows = 0;
    for (size_t i = 0; i < n; ++i) {
      RowRange rr = ap.ranges[b0 + i];
      rr.prefix = rows;
      rows += rr.row_end - rr.row_begin;
      pp.ranges[i] = rr;
    }
    pp.num_ranges = (int)n;
    pp.total_rows = rows;
    if ((st = cuda_status(launch_absorb_proj(pp, s))) != MLA_OK) return st;
  }
  return MLA_OK;
}

// Shared validation of the prefill entry points; fills the plans.
static int prefill_plans(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                         int num_blocks, const int32_t* block_table, int max_blocks_per_req, const int32_t* seq_lens,
                         const int32_t* cu_q, int num_reqs, int num_heads, const mla_segment* segments,
                         int num_segments, int chunk, const void* kv_b_proj, float softmax_scale, float rope_theta,
                         int parts, void* out, int out_dtype, float* lse, Plan* plan, FusedPlan* fplan) {
  int st = build_plan(num_reqs, seq_lens, cu_q, num_heads, segments, num_segments, chunk, parts, plan);
  if (st != MLA_OK) return st;
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (out_dtype != MLA_OUT_FP32 && out_dtype != MLA_OUT_BF16) return MLA_ERR_INVALID_ARG;
  if (!(rope_theta > 1.f) || !std::isfinite(softmax_scale) || !std::isfinite(rope_theta)) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_FP8_E4M3 && !(std::isfinite(kv_scale) && kv_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (plan->total_q == 0) return MLA_OK;
  if (!q || !q_pos || !kv_cache || !block_table || !kv_b_proj || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (num_blocks <= 0 || max_blocks_per_req <= 0) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(kv_b_proj, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  for (int r = 0; r < num_reqs; ++r)
    if ((seq_lens[r] + kBlock - 1) / kBlock > max_blocks_per_req) return MLA_ERR_INVALID_ARG;
  build_fused_plan(*plan, seq_lens, cu_q, num_reqs, chunk, true, fplan);
  return MLA_OK;
}

// ------------------------------------------------------------------ head-split reuse
// A request with at most this many queries goes through the absorbed path,
// the others through the up-projected one.  On GB300 (128 heads, 32K cached
// tokens) the two break even near 230 queries: the absorbed path is 1.85x at
// 128, 1.23x at 192 and 1.02x at 224; on a 128K FP8 cache it is 1.31x at 192
// and 0.97x at 256.  The FLOP counts alone put it near 170: the latent kernel
// runs its MMAs closer to peak than the up-projected one.  208 keeps a margin
// below the crossover and takes v3_8k's 10% protected rows (205) through the
// absorbed path (1.77x against 1.70x for head-split reuse).
constexpr int kAutoAbsorbedMaxQueries = 208;

struct ReusePlan {
  std::vector<int32_t> global, local, prot_rows, prot_tok, gidx, lidx, pidx, cu_p, ctx;
  Plan plan_g, plan_p;
  FusedPlan fp_g, fp_p;
  FusedWs fw_g, fw_p;
  bool prot_absorbed = false;      // the protected part goes through the absorbed path
  AbsPlan ap_p;
  AbsWs aw_p;
  size_t off_maps = 0, off_qg = 0, off_wg = 0, off_og = 0, off_lg = 0, off_qp = 0, off_posp = 0, off_tokp = 0,
         off_wp = 0, off_op = 0, off_lp = 0, off_fused = 0, total = 0;
  size_t map_words = 0;
};

// The two compacted sub-problems and the workspace that holds them, in order:
// one fused workspace shared by the two sub-calls (they run one after the
// other; its header, with the device error word, is the call's header); index
// maps (gidx[H], lidx[H], pidx[T_q], protected rows and their token indices,
// the Global and the Local head lists); Global part (q, kv_b_proj columns,
// out, lse); protected part (q, q_pos, kv_b_proj columns, out, lse).
static int build_reuse_plan(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q, int H,
                            const mla_segment* segs, int nseg, int chunk, int parts, const int32_t* global_heads,
                            int n_global, const uint8_t* row_protected, ReusePlan* rp) {
  if (n_global < 0 || (n_global > 0 && global_heads == nullptr)) return MLA_ERR_INVALID_ARG;
  Plan base;
  int st = build_plan(num_reqs, seq_lens, cu_q, H, segs, nseg, chunk, parts, &base);
  if (st != MLA_OK) return st;
  const int64_t T_q = base.total_q;
  rp->gidx.assign(H, -1);
  rp->lidx.assign(H, -1);
  rp->global.clear();
  rp->local.clear();
  for (int i = 0; i < n_global; ++i) {
    const int h = global_heads[i];
    if (h < 0 || h >= H) return MLA_ERR_INVALID_ARG;
    if (rp->gidx[h] < 0) {
      rp->gidx[h] = (int32_t)rp->global.size();
      rp->global.push_back(h);
    }
  }
  for (int h = 0; h < H; ++h)
    if (rp->gidx[h] < 0) {
      rp->lidx[h] = (int32_t)rp->local.size();
      rp->local.push_back(h);
    }
  rp->pidx.assign((size_t)T_q, -1);
  rp->prot_rows.clear();
  rp->prot_tok.clear();
  rp->cu_p.assign(num_reqs + 1, 0);
  rp->ctx.assign(num_reqs, 0);
  for (int r = 0; r < num_reqs; ++r) {
    const int E = cu_q[r + 1] - cu_q[r];
    rp->ctx[r] = seq_lens[r] - E;
    for (int i = 0; i < E && row_protected != nullptr; ++i)
      if (row_protected[cu_q[r] + i]) {
        rp->pidx[cu_q[r] + i] = (int32_t)rp->prot_rows.size();
        rp->prot_rows.push_back(cu_q[r] + i);
        rp->prot_tok.push_back(rp->ctx[r] + i);
      }
    rp->cu_p[r + 1] = (int32_t)rp->prot_rows.size();
  }
  const int nG = (int)rp->global.size(), nL = (int)rp->local.size(), nP = (int)rp->prot_rows.size();
  size_t fused_bytes = 0;
  if (nG > 0) {
    if ((st = build_plan(num_reqs, seq_lens, cu_q, nG, segs, nseg, chunk, parts, &rp->plan_g)) != MLA_OK) return st;
    build_fused_plan(rp->plan_g, seq_lens, cu_q, num_reqs, chunk, true, &rp->fp_g);
    rp->fw_g = fused_ws_layout(rp->fp_g, nG);
    fused_bytes = std::max(fused_bytes, rp->fw_g.total);
  }
  rp->prot_absorbed = false;
  if (nP > 0 && nL > 0) {
    if ((st = build_plan(num_reqs, seq_lens, rp->cu_p.data(), nL, segs, nseg, chunk, parts, &rp->plan_p,
                         rp->ctx.data())) != MLA_OK)
      return st;
    build_fused_plan(rp->plan_p, seq_lens, rp->cu_p.data(), num_reqs, chunk, true, &rp->fp_p, rp->ctx.data(),
                     rp->prot_tok.data());
    // The protected rows take the absorbed path when it is the faster one for every request (at most
    // kAutoAbsorbedMaxQueries of them) and no row needs exact scores (each sees kExactKeys keys or more,
    // counting its context and causal extend keys).
    bool absorbed = true;
    for (int r = 0; r < num_reqs && absorbed; ++r) {
      const int np_r = rp->cu_p[r + 1] - rp->cu_p[r];
      if (np_r == 0) continue;
      const int64_t first_keys = ((parts & MLA_PART_CONTEXT) ? (int64_t)rp->ctx[r] : 0) +
                                 ((parts & MLA_PART_EXTEND) ? (int64_t)rp->prot_tok[rp->cu_p[r]] - rp->ctx[r] + 1 : 0);
      absorbed = np_r <= kAutoAbsorbedMaxQueries && first_keys >= kExactKeys;
    }
    if (env_int("MLA_REUSE_ABSORBED", 1) == 0) absorbed = false;
    if (absorbed) {
      build_abs_plan(rp->fp_p, nL, rp->cu_p.data(), num_reqs, &rp->ap_p);
      rp->aw_p = abs_ws_layout(rp->fp_p, rp->ap_p, nL);
      fused_bytes = std::max(fused_bytes, rp->aw_p.total);
      rp->prot_absorbed = true;
    } else {
      rp->fw_p = fused_ws_layout(rp->fp_p, nL);
      fused_bytes = std::max(fused_bytes, rp->fw_p.total);
    }
  }
  rp->map_words = 2 * (size_t)H + (size_t)T_q + 2 * (size_t)nP + (size_t)nG + (size_t)nL;
  rp->off_fused = 0;
  rp->off_maps = up256(std::max(fused_bytes, (size_t)256));
  rp->off_qg = up256(rp->off_maps + rp->map_words * 4);
  rp->off_wg = up256(rp->off_qg + (size_t)T_q * nG * kDqk * 2);
  rp->off_og = up256(rp->off_wg + (size_t)kDc * nG * 256 * 2);
  rp->off_lg = up256(rp->off_og + (size_t)T_q * nG * kDv * 4);
  rp->off_qp = up256(rp->off_lg + (size_t)T_q * nG * 4);
  rp->off_posp = up256(rp->off_qp + (size_t)nP * nL * kDqk * 2);
  rp->off_tokp = up256(rp->off_posp + (size_t)nP * 4);
  rp->off_wp = up256(rp->off_tokp + (size_t)nP * 4);
  rp->off_op = up256(rp->off_wp + (size_t)kDc * nL * 256 * 2);
  rp->off_lp = up256(rp->off_op + (size_t)nP * nL * kDv * 4);
  rp->total = up256(rp->off_lp + (size_t)nP * nL * 4);
  return MLA_OK;
}

static int prefill_reuse(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                         int num_blocks, const int32_t* block_table, int max_blocks, int H, const void* kv_b_proj,
                         float softmax_scale, float rope_theta, const float* art_out, const float* art_lse,
                         void* out, int out_dtype, float* lse, uint8_t* ws, const ReusePlan& rp, int64_t T_q,
                         cudaStream_t s) {
  int st = cuda_status(cudaMemsetAsync(ws, 0, 256, s));
  if (st != MLA_OK) return st;
  // index maps: host vectors -> workspace (pageable copies complete their host reads before returning)
  std::vector<int32_t> maps;
  maps.reserve(rp.map_words);
  maps.insert(maps.end(), rp.gidx.begin(), rp.gidx.end());
  maps.insert(maps.end(), rp.lidx.begin(), rp.lidx.end());
  maps.insert(maps.end(), rp.pidx.begin(), rp.pidx.end());
  maps.insert(maps.end(), rp.prot_rows.begin(), rp.prot_rows.end());
  maps.insert(maps.end(), rp.prot_tok.begin(), rp.prot_tok.end());
  maps.insert(maps.end(), rp.global.begin(), rp.global.end());
  maps.insert(maps.end(), rp.local.begin(), rp.local.end());
  int32_t* dmaps = reinterpret_cast<int32_t*>(ws + rp.off_maps);
  if (!maps.empty() && (st = cuda_status(cudaMemcpyAsync(dmaps, maps.data(), maps.size() * 4,
                                                         cudaMemcpyHostToDevice, s))) != MLA_OK)
    return st;
  const int32_t* d_gidx = dmaps;
  const int32_t* d_lidx = dmaps + H;
  const int32_t* d_pidx = dmaps + 2 * H;
  const int32_t* d_prows = dmaps + 2 * H + T_q;
  const int32_t* d_ptok = d_prows + rp.prot_rows.size();
  const int nG = (int)rp.global.size(), nL = (int)rp.local.size(), nP = (int)rp.prot_rows.size();
  const int32_t* d_global = d_ptok + nP;
  const int32_t* d_local = d_global + nG;
  const uint16_t* qb = static_cast<const uint16_t*>(q);
  const uint16_t* wb = static_cast<const uint16_t*>(kv_b_proj);
  uint8_t* fused_ws = ws + rp.off_fused;
  if (nG > 0) {
    uint16_t* qg = reinterpret_cast<uint16_t*>(ws + rp.off_qg);
    uint16_t* wg = reinterpret_cast<uint16_t*>(ws + rp.off_wg);
    if ((st = cuda_status(launch_gather_q(qb, q_pos, nullptr, d_global, (int)T_q, nG, H, qg, nullptr, s))) != MLA_OK)
      return st;
    if ((st = cuda_status(launch_gather_w(wb, d_global, nG, H, wg, s))) != MLA_OK) return st;
    if ((st = prefill_fused(qg, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks, nG, wg,
                            softmax_scale, rope_theta, ws + rp.off_og, MLA_OUT_FP32,
                            reinterpret_cast<float*>(ws + rp.off_lg), fused_ws, rp.fp_g, rp.fw_g, s, nullptr,
                            true)) != MLA_OK)
      return st;
  }
  if (nP > 0 && nL > 0) {
    uint16_t* qp = reinterpret_cast<uint16_t*>(ws + rp.off_qp);
    int32_t* posp = reinterpret_cast<int32_t*>(ws + rp.off_posp);
    uint16_t* wp = reinterpret_cast<uint16_t*>(ws + rp.off_wp);
    if ((st = cuda_status(launch_gather_q(qb, q_pos, d_prows, d_local, nP, nL, H, qp, posp, s))) != MLA_OK)
      return st;
    if ((st = cuda_status(launch_gather_w(wb, d_local, nL, H, wp, s))) != MLA_OK) return st;
    if (rp.prot_absorbed) {
      if ((st = prefill_absorbed(qp, posp, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks, nL, wp,
                                 softmax_scale, rope_theta, ws + rp.off_op, MLA_OUT_FP32,
                                 reinterpret_cast<float*>(ws + rp.off_lp), fused_ws, rp.fp_p, rp.ap_p, rp.aw_p, s,
                                 false, reinterpret_cast<uint32_t*>(ws), d_ptok)) != MLA_OK)
        return st;
    } else if ((st = prefill_fused(qp, posp, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks, nL,
                                   wp, softmax_scale, rope_theta, ws + rp.off_op, MLA_OUT_FP32,
                                   reinterpret_cast<float*>(ws + rp.off_lp), fused_ws, rp.fp_p, rp.fw_p, s, d_ptok,
                                   true)) != MLA_OK) {
      return st;
    }
  }
  ReuseAssemble ra;
  ra.out_g = reinterpret_cast<const float*>(ws + rp.off_og);
  ra.lse_g = reinterpret_cast<const float*>(ws + rp.off_lg);
  ra.out_p = reinterpret_cast<const float*>(ws + rp.off_op);
  ra.lse_p = reinterpret_cast<const float*>(ws + rp.off_lp);
  ra.art_out = art_out;
  ra.art_lse = art_lse;
  ra.gidx = d_gidx;
  ra.lidx = d_lidx;
  ra.pidx = d_pidx;
  ra.out = out;
  ra.lse = lse;
  ra.out_bf16 = out_dtype == MLA_OUT_BF16;
  ra.rows = (int)T_q;
  ra.H = H;
  ra.n_global = nG;
  ra.n_local = nL;
  return cuda_status(launch_reuse_assemble(ra, s));
}

// ------------------------------------------------------------------ per-request dispatch

struct AutoPlan {
  Plan plan_f, plan_a;
  FusedPlan fp_f, fp_a;
  AbsPlan ap;
  FusedWs fw;
  AbsWs aw;
  size_t off_abs = 0, total = 0;
  bool any_f = false, any_a = false;
};

// Keys the first query row of each request sees (its context keys, plus
// itself when the extend stage is attended): the fewest of any of its rows.
static std::vector<int64_t> first_row_keys(const Plan& plan, const int32_t* seq_lens, const int32_t* cu_q,
                                           int num_reqs, int parts) {
  std::vector<int64_t> n(num_reqs, 0);
  for (const Split& sp : plan.splits)
    if (sp.k_begin < sp.q_tok0) n[sp.req] += std::min(sp.k_end, sp.q_tok0) - sp.k_begin;
  for (int r = 0; r < num_reqs; ++r)
    if ((parts & MLA_PART_EXTEND) && cu_q[r + 1] > cu_q[r]) n[r] += 1;
  return n;
}

// The requests of a call split between the up-projected and the absorbed
// paths.  The absorbed path takes a request when all its rows see at least
// kExactKeys keys (it rounds the absorbed query to bf16, which moves each
// score by about 1.4e-3 and a row's lse by as much when it has few keys; the
// up-projected kernel takes such rows with exact scores) and, for the
// per-request dispatch (by_queries), when it has at most
// kAutoAbsorbedMaxQueries queries.
static int build_auto_plan(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q, int H,
                           const mla_segment* segs, int nseg, int chunk, int parts, AutoPlan* au,
                           bool by_queries = true) {
  Plan all;
  int st = build_plan(num_reqs, seq_lens, cu_q, H, segs, nseg, chunk, parts, &all);
  if (st != MLA_OK) return st;
  const std::vector<int64_t> keys = first_row_keys(all, seq_lens, cu_q, num_reqs, parts);
  std::vector<uint8_t> is_short(num_reqs), is_long(num_reqs);
  for (int r = 0; r < num_reqs; ++r) {
    const int E = cu_q[r + 1] - cu_q[r];
    is_short[r] = (!by_queries || E <= kAutoAbsorbedMaxQueries) && keys[r] >= kExactKeys;
    is_long[r] = !is_short[r];
    au->any_a |= E > 0 && is_short[r];
    au->any_f |= E > 0 && is_long[r];
  }
  st = build_plan(num_reqs, seq_lens, cu_q, H, segs, nseg, chunk, parts, &au->plan_f, nullptr, is_short.data());
  if (st != MLA_OK) return st;
  if ((st = build_plan(num_reqs, seq_lens, cu_q, H, segs, nseg, chunk, parts, &au->plan_a, nullptr,
                       is_long.data())) != MLA_OK)
    return st;
  build_fused_plan(au->plan_f, seq_lens, cu_q, num_reqs, chunk, true, &au->fp_f);
  build_fused_plan(au->plan_a, seq_lens, cu_q, num_reqs, chunk, true, &au->fp_a);
  build_abs_plan(au->fp_a, H, cu_q, num_reqs, &au->ap);
  au->fw = fused_ws_layout(au->fp_f, H);
  au->aw = abs_ws_layout(au->fp_a, au->ap, H);
  au->off_abs = up256(std::max(au->fw.total, (size_t)256));
  au->total = up256(au->off_abs + au->aw.total);
  return MLA_OK;
}

extern "C" {

int mla_abi_version(void) { return 1; }

void mla_set_trace(void* device_buffer, size_t bytes) {
  g_trace.store(bytes ? device_buffer : nullptr);
  g_trace_bytes.store(device_buffer ? bytes : 0);
}

void mla_set_kernel_events(void* begin_event, void* end_event) {
  const bool on = begin_event != nullptr && end_event != nullptr;
  g_ev_begin.store(on ? begin_event : nullptr);
  g_ev_end.store(on ? end_event : nullptr);
}

uint64_t mla_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* mla_last_cuda_error(void) { return g_cuda_err; }

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_BAD_BLOCK_ID: return "MLA_ERR_BAD_BLOCK_ID";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_TOO_LARGE: return "MLA_ERR_TOO_LARGE";
    default: return "MLA_ERR_UNKNOWN";
  }
}

size_t mla_prefill_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q, int num_heads,
                                  const mla_segment* segments, int num_segments, int chunk, int parts) {
  Plan plan;
  if (build_plan(num_reqs, seq_lens, cu_q, num_heads, segments, num_segments, chunk, parts, &plan) != MLA_OK)
    return 0;
  FusedPlan fp;
  build_fused_plan(plan, seq_lens, cu_q, num_reqs, chunk, true, &fp);   // room for the gathered rows
  return fused_ws_layout(fp, num_heads).total;
}

size_t mla_prefill_min_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q, int num_heads,
                                      const mla_segment* segments, int num_segments, int chunk, int parts) {
  Plan plan;
  if (build_plan(num_reqs, seq_lens, cu_q, num_heads, segments, num_segments, chunk, parts, &plan) != MLA_OK)
    return 0;
  FusedPlan fp;
  build_fused_plan(plan, seq_lens, cu_q, num_reqs, chunk, true, &fp);
  return fused_ws_layout(fp, num_heads, 1, 4, 2).total;
}

int mla_prefill_ctx(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                    int num_blocks, const int32_t* block_table, int max_blocks_per_req, const int32_t* seq_lens,
                    const int32_t* cu_q, int num_reqs, int num_heads, const mla_segment* segments,
                    int num_segments, int chunk, const void* kv_b_proj, float softmax_scale, float rope_theta,
                    int parts, void* out, int out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                    mla_stream_t stream) {
  Plan plan;
  FusedPlan fplan;
  const int st = prefill_plans(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req,
                               seq_lens, cu_q, num_reqs, num_heads, segments, num_segments, chunk, kv_b_proj,
                               softmax_scale, rope_theta, parts, out, out_dtype, lse, &plan, &fplan);
  if (st != MLA_OK || plan.total_q == 0) return st;
  const FusedWs fw = fused_ws_fitting(fplan, num_heads, workspace_bytes);
  if (workspace == nullptr || !aligned(workspace, 256) || fw.pieces_per_launch < 1) return MLA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return prefill_fused(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req, num_heads,
                         kv_b_proj, softmax_scale, rope_theta, out, out_dtype, lse, workspace, fplan, fw, s);
}

int mla_prefill_ctx_fp8w(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                         int num_blocks, const int32_t* block_table, int max_blocks_per_req, const int32_t* seq_lens,
                         const int32_t* cu_q, int num_reqs, int num_heads, const mla_segment* segments,
                         int num_segments, int chunk, const void* kv_b_proj_e4m3_t, float w_scale,
                         float softmax_scale, float rope_theta, int parts, void* out, int out_dtype, float* lse,
                         void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  if (kv_dtype != MLA_KV_FP8_E4M3) return kv_dtype == MLA_KV_BF16 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (!(std::isfinite(w_scale) && w_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  Plan plan;
  FusedPlan fplan;
  const int st = prefill_plans(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req,
                               seq_lens, cu_q, num_reqs, num_heads, segments, num_segments, chunk, kv_b_proj_e4m3_t,
                               softmax_scale, rope_theta, parts, out, out_dtype, lse, &plan, &fplan);
  if (st != MLA_OK || plan.total_q == 0) return st;
  const FusedWs fw = fused_ws_fitting(fplan, num_heads, workspace_bytes);
  if (workspace == nullptr || !aligned(workspace, 256) || fw.pieces_per_launch < 1) return MLA_ERR_WORKSPACE;
  return prefill_fused(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req, num_heads,
                       nullptr, softmax_scale, rope_theta, out, out_dtype, lse, workspace, fplan, fw,
                       reinterpret_cast<cudaStream_t>(stream), nullptr, false, kv_b_proj_e4m3_t, w_scale);
}

int mla_kv_b_proj_absmax(const void* kv_b_proj, int num_heads, float* absmax, mla_stream_t stream) {
  if (kv_b_proj == nullptr || absmax == nullptr || num_heads < 1 || num_heads > kMaxHeads) return MLA_ERR_INVALID_ARG;
  if (!aligned(kv_b_proj, 16)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_absmax_bf16(static_cast<const uint16_t*>(kv_b_proj),
                                        (int64_t)kDc * num_heads * (kDnope + kDv), absmax,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int mla_kv_b_proj_to_e4m3(const void* kv_b_proj, int num_heads, float w_scale, void* out_e4m3_t,
                          mla_stream_t stream) {
  if (kv_b_proj == nullptr || out_e4m3_t == nullptr || num_heads < 1 || num_heads > kMaxHeads)
    return MLA_ERR_INVALID_ARG;
  if (!(std::isfinite(w_scale) && w_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_t(static_cast<const uint16_t*>(kv_b_proj), num_heads * (kDnope + kDv), w_scale,
                                       static_cast<uint8_t*>(out_e4m3_t), reinterpret_cast<cudaStream_t>(stream)));
}

int mla_prefill_ctx_noalloc(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                            int num_blocks, const int32_t* block_table, int max_blocks_per_req,
                            const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                            const mla_segment* segments, int num_segments, int chunk, const void* kv_b_proj,
                            float softmax_scale, float rope_theta, int parts, void* out, int out_dtype, float* lse,
                            mla_stream_t stream) {
  // the same validation as mla_prefill_ctx first, then one plan for the size
  // check and the launches
  Plan plan;
  FusedPlan fplan;
  int st = prefill_plans(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req, seq_lens,
                         cu_q, num_reqs, num_heads, segments, num_segments, chunk, kv_b_proj, softmax_scale,
                         rope_theta, parts, out, out_dtype, lse, &plan, &fplan);
  if (st != MLA_OK || plan.total_q == 0) return st;
  const FusedWs fw = fused_ws_fitting(fplan, num_heads, MLA_NOALLOC_SCRATCH_BYTES);
  if (fw.pieces_per_launch < 1) return MLA_ERR_TOO_LARGE;
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != MLA_OK) return st;
  return prefill_fused(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req, num_heads,
                       kv_b_proj, softmax_scale, rope_theta, out, out_dtype, lse, scratch, fplan, fw,
                       reinterpret_cast<cudaStream_t>(stream));
}

size_t mla_prefill_absorbed_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q, int num_heads,
                                           const mla_segment* segments, int num_segments, int chunk, int parts) {
  static AutoPlan au;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  au = AutoPlan();
  if (build_auto_plan(num_reqs, seq_lens, cu_q, num_heads, segments, num_segments, chunk, parts, &au, false) != MLA_OK)
    return 0;
  return au.total;
}

// The absorbed and the per-request paths: the requests split by build_auto_plan,
// the up-projected part first (its workspace header holds the call's error word).
static int prefill_split(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                         int num_blocks, const int32_t* block_table, int max_blocks_per_req, const int32_t* seq_lens,
                         const int32_t* cu_q, int num_reqs, int num_heads, const mla_segment* segments,
                         int num_segments, int chunk, const void* kv_b_proj, float softmax_scale, float rope_theta,
                         int parts, void* out, int out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                         mla_stream_t stream, bool by_queries) {
  Plan plan;
  FusedPlan fplan;
  int st = prefill_plans(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req,
                         seq_lens, cu_q, num_reqs, num_heads, segments, num_segments, chunk, kv_b_proj,
                         softmax_scale, rope_theta, parts, out, out_dtype, lse, &plan, &fplan);
  if (st != MLA_OK || plan.total_q == 0) return st;
  static AutoPlan au;              // large; built on the host under a lock
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  au = AutoPlan();
  if ((st = build_auto_plan(num_reqs, seq_lens, cu_q, num_heads, segments, num_segments, chunk, parts, &au,
                            by_queries)) != MLA_OK)
    return st;
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < au.total) return MLA_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* err = reinterpret_cast<uint32_t*>(ws);   // the up-projected part's header is the call's
  if ((st = cuda_status(cudaMemsetAsync(ws, 0, 256, s))) != MLA_OK) return st;
  if (au.any_f &&
      (st = prefill_fused(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req,
                          num_heads, kv_b_proj, softmax_scale, rope_theta, out, out_dtype, lse, ws, au.fp_f, au.fw, s,
                          nullptr, true)) != MLA_OK)
    return st;
  if (au.any_a &&
      (st = prefill_absorbed(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req,
                             num_heads, kv_b_proj, softmax_scale, rope_theta, out, out_dtype, lse, ws + au.off_abs,
                             au.fp_a, au.ap, au.aw, s, false, err)) != MLA_OK)
    return st;
  return MLA_OK;
}

int mla_prefill_ctx_absorbed(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                             int num_blocks, const int32_t* block_table, int max_blocks_per_req,
                             const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                             const mla_segment* segments, int num_segments, int chunk, const void* kv_b_proj,
                             float softmax_scale, float rope_theta, int parts, void* out, int out_dtype, float* lse,
                             void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  return prefill_split(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req, seq_lens,
                       cu_q, num_reqs, num_heads, segments, num_segments, chunk, kv_b_proj, softmax_scale, rope_theta,
                       parts, out, out_dtype, lse, workspace, workspace_bytes, stream, false);
}

size_t mla_prefill_reuse_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q, int num_heads,
                                        const mla_segment* segments, int num_segments, int chunk, int parts,
                                        const int32_t* global_heads, int n_global, const uint8_t* row_protected) {
  ReusePlan rp;
  if (build_reuse_plan(num_reqs, seq_lens, cu_q, num_heads, segments, num_segments, chunk, parts, global_heads,
                       n_global, row_protected, &rp) != MLA_OK)
    return 0;
  return rp.total;
}

int mla_prefill_reuse(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                      int num_blocks, const int32_t* block_table, int max_blocks_per_req, const int32_t* seq_lens,
                      const int32_t* cu_q, int num_reqs, int num_heads, const mla_segment* segments,
                      int num_segments, int chunk, const void* kv_b_proj, float softmax_scale, float rope_theta,
                      int parts, const int32_t* global_heads, int n_global, const uint8_t* row_protected,
                      const float* art_out, const float* art_lse, void* out, int out_dtype, float* lse,
                      void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  Plan plan;
  FusedPlan fplan;
  int st = prefill_plans(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req,
                         seq_lens, cu_q, num_reqs, num_heads, segments, num_segments, chunk, kv_b_proj,
                         softmax_scale, rope_theta, parts, out, out_dtype, lse, &plan, &fplan);
  if (st != MLA_OK || plan.total_q == 0) return st;
  if (!art_out || !art_lse || !aligned(art_out, 16) || !aligned(art_lse, 4)) return MLA_ERR_INVALID_ARG;
  static ReusePlan rp;             // large; built on the host under a lock
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if ((st = build_reuse_plan(num_reqs, seq_lens, cu_q, num_heads, segments, num_segments, chunk, parts, global_heads,
                             n_global, row_protected, &rp)) != MLA_OK)
    return st;
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < rp.total) return MLA_ERR_WORKSPACE;
  return prefill_reuse(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req,
                       num_heads, kv_b_proj, softmax_scale, rope_theta, art_out, art_lse, out, out_dtype, lse,
                       static_cast<uint8_t*>(workspace), rp, plan.total_q, reinterpret_cast<cudaStream_t>(stream));
}

size_t mla_prefill_absorbed_fp8_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q,
                                               int num_heads, const mla_segment* segments, int num_segments,
                                               int chunk, int parts) {
  Plan plan;
  if (build_plan(num_reqs, seq_lens, cu_q, num_heads, segments, num_segments, chunk, parts, &plan) != MLA_OK)
    return 0;
  FusedPlan fp;
  build_fused_plan(plan, seq_lens, cu_q, num_reqs, chunk, true, &fp);
  AbsPlan ap;
  build_abs_plan(fp, num_heads, cu_q, num_reqs, &ap);
  return abs_ws_layout(fp, ap, num_heads, true).total;
}

int mla_prefill_ctx_absorbed_fp8(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype,
                                 float kv_scale, int num_blocks, const int32_t* block_table, int max_blocks_per_req,
                                 const int32_t* seq_lens, const int32_t* cu_q, int num_reqs, int num_heads,
                                 const mla_segment* segments, int num_segments, int chunk, const void* kv_b_proj,
                                 float softmax_scale, float rope_theta, int parts, void* out, int out_dtype,
                                 float* lse, void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  if (kv_dtype != MLA_KV_FP8_E4M3) return kv_dtype == MLA_KV_BF16 ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  Plan plan;
  FusedPlan fplan;
  const int st = prefill_plans(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req,
                               seq_lens, cu_q, num_reqs, num_heads, segments, num_segments, chunk, kv_b_proj,
                               softmax_scale, rope_theta, parts, out, out_dtype, lse, &plan, &fplan);
  if (st != MLA_OK || plan.total_q == 0) return st;
  AbsPlan ap;
  build_abs_plan(fplan, num_heads, cu_q, num_reqs, &ap);
  const AbsWs aw = abs_ws_layout(fplan, ap, num_heads, true);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < aw.total) return MLA_ERR_WORKSPACE;
  return prefill_absorbed(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req,
                          num_heads, kv_b_proj, softmax_scale, rope_theta, out, out_dtype, lse, workspace, fplan, ap,
                          aw, reinterpret_cast<cudaStream_t>(stream), true);
}

size_t mla_prefill_auto_workspace_size(int num_reqs, const int32_t* seq_lens, const int32_t* cu_q, int num_heads,
                                       const mla_segment* segments, int num_segments, int chunk, int parts) {
  static AutoPlan au;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  au = AutoPlan();
  if (build_auto_plan(num_reqs, seq_lens, cu_q, num_heads, segments, num_segments, chunk, parts, &au) != MLA_OK)
    return 0;
  return au.total;
}

int mla_prefill_ctx_auto(const void* q, const int32_t* q_pos, const void* kv_cache, int kv_dtype, float kv_scale,
                         int num_blocks, const int32_t* block_table, int max_blocks_per_req, const int32_t* seq_lens,
                         const int32_t* cu_q, int num_reqs, int num_heads, const mla_segment* segments,
                         int num_segments, int chunk, const void* kv_b_proj, float softmax_scale, float rope_theta,
                         int parts, void* out, int out_dtype, float* lse, void* workspace, size_t workspace_bytes,
                         mla_stream_t stream) {
  return prefill_split(q, q_pos, kv_cache, kv_dtype, kv_scale, num_blocks, block_table, max_blocks_per_req, seq_lens,
                       cu_q, num_reqs, num_heads, segments, num_segments, chunk, kv_b_proj, softmax_scale, rope_theta,
                       parts, out, out_dtype, lse, workspace, workspace_bytes, stream, true);
}

int mla_get_device_error(void* workspace, mla_stream_t stream) {
  if (workspace == nullptr) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  int st = cuda_status(cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s));
  if (st == MLA_OK) st = cuda_status(cudaStreamSynchronize(s));
  if (st != MLA_OK) return st;
  st = cuda_status(cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s));
  if (st != MLA_OK) return st;
  if (word & kErrBadBlock) return MLA_ERR_BAD_BLOCK_ID;
  if (word & kErrTimeout) return MLA_ERR_TIMEOUT;
  return MLA_OK;
}

int mla_merge_states(const float* out_a, const float* lse_a, const float* out_b, const float* lse_b, float* out,
                     float* lse, int64_t rows, int d_v, mla_stream_t stream) {
  if (rows < 0 || d_v <= 0 || d_v % 4 != 0) return MLA_ERR_INVALID_ARG;
  if (rows == 0) return MLA_OK;
  if (!out_a || !lse_a || !out_b || !lse_b || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned(out_a, 16) || !aligned(out_b, 16) || !aligned(out, 16)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_merge2(out_a, lse_a, out_b, lse_b, out, lse, rows, d_v,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

int mla_rope_relocate(const void* x, const int32_t* pos, int64_t offset, float theta, void* y, int tokens,
                      int heads, int row_stride, int rope_col, mla_stream_t stream) {
  if (tokens < 0 || heads < 0) return MLA_ERR_INVALID_ARG;
  if (rope_col < 0 || rope_col % 8 != 0 || row_stride % 8 != 0 || rope_col + kDr > row_stride) return MLA_ERR_INVALID_ARG;
  if (!(theta > 1.f) || !std::isfinite(theta)) return MLA_ERR_INVALID_ARG;
  if (tokens == 0 || heads == 0) return MLA_OK;
  if (!x || !pos || !y || !aligned(x, 16) || !aligned(y, 16)) return MLA_ERR_INVALID_ARG;
  uint64_t frac[kDr / 2];
  rope_fracs((double)theta, frac);
  return cuda_status(launch_rope(static_cast<const uint16_t*>(x), pos, offset, frac, static_cast<uint16_t*>(y),
                                 tokens, heads, row_stride, rope_col, reinterpret_cast<cudaStream_t>(stream)));
}

int mla_gather_latent(const void* kv_cache, int kv_dtype, float kv_scale, int num_blocks,
                      const int32_t* block_table_row, int max_blocks, int start, int len, void* dst,
                      uint32_t* dev_error, mla_stream_t stream) {
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (start < 0 || len < 0 || num_blocks <= 0 || max_blocks <= 0) return MLA_ERR_INVALID_ARG;
  if (((int64_t)start + len + kBlock - 1) / kBlock > max_blocks) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_FP8_E4M3 && !(std::isfinite(kv_scale) && kv_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (len == 0) return MLA_OK;
  if (!kv_cache || !block_table_row || !dst || !aligned(kv_cache, 16) || !aligned(dst, 16)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_gather(static_cast<const uint8_t*>(kv_cache), kv_dtype == MLA_KV_FP8_E4M3, kv_scale,
                                   num_blocks, block_table_row, max_blocks, start, len, static_cast<uint16_t*>(dst),
                                   dev_error, reinterpret_cast<cudaStream_t>(stream)));
}

int mla_block_hash(const void* kv_cache, int kv_dtype, int num_blocks, const int32_t* block_ids, int n,
                   uint64_t* hashes, uint32_t* dev_error, mla_stream_t stream) {
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (n < 0 || num_blocks <= 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (!kv_cache || !block_ids || !hashes || !aligned(kv_cache, 16) || !aligned(hashes, 8)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_block_hash(static_cast<const uint8_t*>(kv_cache), kv_dtype == MLA_KV_FP8_E4M3, num_blocks,
                                       block_ids, n, hashes, dev_error, reinterpret_cast<cudaStream_t>(stream)));
}

int mla_block_compare(const void* kv_cache, int kv_dtype, int num_blocks, const int32_t* block_a,
                      const int32_t* block_b, int n, int32_t* equal, uint32_t* dev_error, mla_stream_t stream) {
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (n < 0 || num_blocks <= 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (!kv_cache || !block_a || !block_b || !equal || !aligned(kv_cache, 16)) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_block_compare(static_cast<const uint8_t*>(kv_cache), kv_dtype == MLA_KV_FP8_E4M3,
                                          num_blocks, block_a, block_b, n, equal, dev_error,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
