// host.cu -- the C ABI: cache creation, argument validation, the per-call
// plan (sub-chunks, decode / chunk rows, split-K schedule) and kernel launches.
//
// The plan uses only host data: n_new and rows arrive in host memory and lens
// is mirrored on the host (tiny_agent/generate.py keeps `lens_cpu` for the same
// reason), so no call reads device memory back.  Every check runs before the
// first enqueue, so a rejected call changes nothing (pycraft-1 `update` guards;
// "KV cache full" is raised before any write in tiny_agent/generate.py
// `append`).
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <unordered_map>
#include <vector>

#include "../../include/kvinc.h"
#include "kvinc_internal.h"

namespace kvinc {
cudaError_t configure_decode();
cudaError_t configure_prefill();
cudaError_t configure_prefill_tc();
cudaError_t launch_prefill_tc(const PrefillParams &p, int D, int tiles, cudaStream_t s,
                              bool pdl);
int prefill_tc_tiles(int D, int n_rho);
}  // namespace kvinc

using namespace kvinc;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D bf16 view [rows][D] with 64-column x kTileKeys-row boxes, 128-byte swizzle.
bool make_tmap(CUtensorMap *m, void *base, int64_t rows, int D, int box_rows = kTileKeys) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
      changed = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

struct ProfRec {
  cudaEvent_t a, b;
  int kind;
  double bytes, flops;
};

constexpr size_t kMaxProfRecs = 1 << 16;
// Chunk rows with at least this many query rows (tokens x GQA group) use the tcgen05
// prefill kernel, the others the mma.sync kernel.  At D = 64 the one-tile tcgen05 kernel
// (two CTAs per SM) takes every row: the continuous-batch mix ran 2.78 M tokens/s that way
// against 2.48 M with rows under 64 query rows on the mma.sync kernel.  At D = 128 (two
// tiles, one CTA per SM) the mma.sync kernel stays faster for those rows: 2-7-token chunks
// against 8k cached keys, 64 rows, Hq = 64, Hk = 8: 38.1 vs 39.4 ms of prefill over 30 steps.
int tc_min_rows(int D) { return D == 64 ? 1 : 64; }
// Key splits of chunked prefill: at most kMaxPrefillSplits per row, and at most one per
// kMinSplitBlocks 128-key blocks (rounded up), so a row of up to that many blocks is never
// split.
constexpr int kMinSplitBlocks = 4;
// Prefill key-split partials: a cache reserves room for this many vectors per SM at
// create (capped by the most its rows can ever need), and the planner lengthens a call's
// splits until its partials fit.  Load balancing alone stays below about 4 waves of split
// CTAs (2560 vectors per SM over the three launch kinds); the mixes measured need under
// 600 per SM (continuous-batch mix at 152 SMs: 78k vectors).
constexpr int64_t kPrefillPartVecsPerSm = 1024;
// Decode splits: at most one per kMinDecodeSplitTiles 64-key tiles of a segment (rounded
// up), so a row of up to that many tiles is one CTA with no split merge, which is what
// small (ring) layers want (4 measured 10% slower on the long-context step: more
// prologues and merges for the same keys).
constexpr int kMinDecodeSplitTiles = 8;

}  // namespace

struct kv_cache {
  int B, max_len, Hq, Hk, D, W, R, n_layers, device, num_sms;
  double theta;
  std::vector<int32_t> kind;
  std::vector<int32_t> lens;  // host mirror
  std::vector<void *> K, V;
  std::vector<int> seg_rows;
  std::vector<CUtensorMap> tmK, tmV;
  std::vector<CUtensorMap> tmK16, tmV16;  // paged layers: 16-row boxes over the pool
  // hybrid layers: K/V above is the group's global storage (owned by the group's full
  // layer, aliased by its local layers); every hybrid layer also owns a ring
  std::vector<int> group;                 // full layer of a hybrid layer's group, else -1
  std::vector<char> owns;                 // K[l] / V[l] allocated for this layer
  std::vector<void *> RK, RV;             // hybrid rings [B][Hk][R+1][D], else nullptr
  std::vector<CUtensorMap> tmRK, tmRV;
  CUtensorMap tmSK, tmSV;
  void *scrK = nullptr, *scrV = nullptr;
  float2 *rope = nullptr;
  int32_t *lpos = nullptr, *err = nullptr, *counters = nullptr;
  float *part_o = nullptr;
  float2 *part_ml = nullptr;
  // prefill key-split partials ([vector][D] fp32 O, [vector] (m, l)), reserved at create
  float *ppart_o = nullptr;
  float2 *ppart_ml = nullptr;
  int64_t ppart_cap = 0;  // vectors
  // host-buffer entry point staging
  void *stage = nullptr;
  size_t stage_bytes = 0;
  // profiling
  bool prof = false;
  std::vector<ProfRec> recs;
  std::vector<cudaEvent_t> free_events;
  // paged global layers: per layer a pool of n_blocks blocks of [Hk][16][D]; one block
  // table for all of them (their rows always have equal lengths)
  int n_blocks = 0;                           // 0: dense cache
  int max_blocks = 0;                         // table entries per row, a multiple of 4
  int32_t *table = nullptr;                   // device [B][max_blocks]
  std::vector<std::vector<int32_t>> rblocks;  // host: pool blocks of each row, in order
  std::vector<int32_t> free_blocks;           // host: free pool blocks
  // host: per pool block, the rows whose tables hold it (0: free).  A block held by
  // several rows (a shared prompt prefix) lies below every holder's length, so no append
  // writes it.
  std::vector<int32_t> refs;
  // hybrid full layers: per row, lens + the tokens of its last append in this step (a
  // local layer of the group may only append the same tokens after it)
  std::vector<std::vector<int32_t>> hy_end;
  // the cache's last kernel launch (stream, kernel kind or -1 for one that may write any
  // storage, layer) and the layer of the call in progress: a decode launch may stream
  // K/V before its grid dependency wait only when the launch before it on the stream
  // wrote none of that layer's storage
  bool pdl = true;  // decode launches use programmatic dependent launch (KVINC_PDL=0: off)
  cudaStream_t last_stream = nullptr;
  int last_kind = -1, last_layer = -1, cur_layer = -1;
};

namespace {

int set_err(cudaError_t e) { return e == cudaSuccess ? KV_OK : KV_ERR_CUDA; }

bool is_hybrid(int kind) { return kind == KV_HYBRID_FULL || kind == KV_HYBRID_LOCAL; }

bool has_hybrid(const kv_cache *c) {
  for (int k : c->kind)
    if (is_hybrid(k)) return true;
  return false;
}

// A layer whose storage (K[l], V[l]) is a full-length cache: global layers and the group
// caches of hybrid layers.
bool cache_layer(const kv_cache *c, int layer) { return c->kind[layer] != KV_SLIDING; }

bool paged_layer(const kv_cache *c, int layer) {
  return c->n_blocks > 0 && cache_layer(c, layer);
}

PageTable page_table(const kv_cache *c, int layer) {
  PageTable pt;
  pt.table = paged_layer(c, layer) ? c->table : nullptr;
  pt.max_blocks = paged_layer(c, layer) ? c->max_blocks : 0;
  pt.n_pool = c->n_blocks;
  return pt;
}

int blocks_for(int len) { return (len + kBlockTokens - 1) / kBlockTokens; }

// A free pool block, now held by one row (the caller has checked that one is free).
int take_block(kv_cache *c) {
  const int blk = c->free_blocks.back();
  c->free_blocks.pop_back();
  c->refs[blk] = 1;
  return blk;
}

// One row lets go of `blk`; the last one returns it to the pool.
void drop_block(kv_cache *c, int blk) {
  if (--c->refs[blk] == 0) c->free_blocks.push_back(blk);
}

// Give each (row, length) of `want` the pool blocks its first `length` positions need, and
// write the new table entries on `s`.  All or nothing: KV_ERR_POOL before any change if the
// pool cannot supply every row.
int ensure_blocks(kv_cache *c, const std::vector<std::pair<int, int>> &want, cudaStream_t s) {
  if (c->n_blocks == 0) return KV_OK;
  int64_t need = 0;
  for (auto &w : want) need += std::max(0, blocks_for(w.second) - (int)c->rblocks[w.first].size());
  if (need > (int64_t)c->free_blocks.size()) return KV_ERR_POOL;
  if (need == 0) return KV_OK;
  static thread_local TableParams tp;
  tp.table = c->table;
  tp.max_blocks = c->max_blocks;
  tp.n = 0;
  for (auto &w : want) {
    auto &rb = c->rblocks[w.first];
    while ((int)rb.size() < blocks_for(w.second)) {
      const int blk = take_block(c);
      tp.row[tp.n] = w.first;
      tp.idx[tp.n] = (int)rb.size();
      tp.blk[tp.n] = blk;
      rb.push_back(blk);
      if (++tp.n == kMaxTableEntries) {
        c->last_stream = s;
        c->last_kind = -1;
        if (launch_table(tp, s) != cudaSuccess) return KV_ERR_CUDA;
        tp.n = 0;
      }
    }
  }
  c->last_stream = s;  // table entries: not to be read before a grid dependency wait
  c->last_kind = -1;
  return launch_table(tp, s) == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

// Let go of the blocks of `row` past its first `len` positions (the pool gets back those
// no other row holds).
void release_blocks(kv_cache *c, int row, int len) {
  if (c->n_blocks == 0) return;
  auto &rb = c->rblocks[row];
  while ((int)rb.size() > blocks_for(len)) {
    drop_block(c, rb.back());
    rb.pop_back();
  }
}

cudaEvent_t take_event(kv_cache *c) {
  if (!c->free_events.empty()) {
    cudaEvent_t e = c->free_events.back();
    c->free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Record a launch of kernel kind `kind` (-1: one that may write any storage of the cache)
// for the layer of the call in progress.
void note_launch(kv_cache *c, cudaStream_t s, int kind) {
  c->last_stream = s;
  c->last_kind = kind;
  c->last_layer = c->cur_layer;
}

// Launch `fn` with an optional event pair around it.
template <class F>
cudaError_t timed(kv_cache *c, int kind, double bytes, double flops, cudaStream_t s, F fn) {
  note_launch(c, s, kind);
  if (!c->prof || c->recs.size() >= kMaxProfRecs) return fn();
  ProfRec r{take_event(c), take_event(c), kind, bytes, flops};
  if (!r.a || !r.b) return fn();
  cudaEventRecord(r.a, s);
  cudaError_t e = fn();
  cudaEventRecord(r.b, s);
  c->recs.push_back(r);
  return e;
}

// Validate (n_new, rows) against the cache; fills the effective cache rows.
int check_rows(const kv_cache *c, const int32_t *n_new, const int32_t *rows, int Bs, int C,
               std::vector<int32_t> &cache_rows) {
  if (Bs < 0 || Bs > c->B) return KV_ERR_ARG;
  if (Bs > 0 && !n_new) return KV_ERR_ARG;
  cache_rows.resize(Bs);
  std::vector<char> seen(c->B, 0);
  for (int i = 0; i < Bs; ++i) {
    const int r = rows ? rows[i] : i;
    if (r < 0 || r >= c->B || seen[r]) return KV_ERR_ARG;
    seen[r] = 1;
    cache_rows[i] = r;
    if (n_new[i] < 0 || n_new[i] > C) return KV_ERR_ARG;
  }
  for (int i = 0; i < Bs; ++i)
    if ((int64_t)c->lens[cache_rows[i]] + n_new[i] > c->max_len) return KV_ERR_FULL;
  return KV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DecodeIn {
  int cache_row, call_row, pos;
};

// What the split planners read of a layer: the device's SM count and the layer's shape
// (R: the ring slots of a sliding or hybrid layer).
struct Geom {
  int num_sms, Hq, Hk, D, R, kind;
};

Geom geom_of(const kv_cache *c, int layer) {
  return {c->num_sms, c->Hq, c->Hk, c->D, c->R, c->kind[layer]};
}

// The storage a layer's decode reads: its own, or for a hybrid layer its group's (the
// group cache, written by the full layer, and the rings of the group's layers).
int storage_id(const kv_cache *c, int layer) {
  return c->group[layer] >= 0 ? c->group[layer] : layer;
}

// Whether a decode launch of `layer` on `s` may stream K/V before its grid dependency
// wait: the cache's previous launch on s wrote nothing it reads -- a decode of another
// storage (new keys, partials, tickets, outputs) or a ring-state update (lpos only).
// Launches of the caller between them write no cache storage; older grids have completed
// by the time a programmatic launch starts.
bool early_kv_ok(const kv_cache *c, int layer, cudaStream_t s) {
  if (!c->pdl || c->last_stream != s) return false;
  if (c->last_kind == KV_KERNEL_STATE) return true;
  return c->last_kind == KV_KERNEL_DECODE && c->last_layer >= 0 &&
         storage_id(c, c->last_layer) != storage_id(c, layer);
}

}  // namespace

int kvinc::plan_decode_splits(int num_sms, int Hk, int n, const int *nk2, DecodeParams &p,
                              int max_parts) {
  const auto tiles_of = [](int keys) { return (keys + kTileKeys - 1) / kTileKeys; };
  int64_t total_tiles = 0;
  int most_tiles = 1;
  for (int i = 0; i < n; ++i) {
    total_tiles += tiles_of(p.rows[i].nk) + tiles_of(nk2[i]);
    most_tiles = std::max(most_tiles, std::max(tiles_of(p.rows[i].nk), tiles_of(nk2[i])));
  }
  // Aim for about four waves of two CTAs per SM: `per` tiles per split, at least
  // kMinDecodeSplitTiles.
  const int64_t target = (int64_t)num_sms * 2 * 4;
  int64_t per = (total_tiles * Hk + target - 1) / target;
  if (per < kMinDecodeSplitTiles) per = kMinDecodeSplitTiles;
  // splits of one segment: at most `cap`, each a whole number of tiles
  const auto splits = [&](int keys, int cap, int &st) {
    const int tiles = tiles_of(keys);
    int ns = (int)std::min<int64_t>(cap, (tiles + per - 1) / per);
    if (ns < 1) ns = 1;
    st = (tiles + ns - 1) / ns;
    return (tiles + st - 1) / st;
  };
  // Partial slots the schedule at `per` needs (one per split of a row of two or more).
  const auto parts_at = [&]() {
    int64_t part = 0;
    for (int i = 0; i < n; ++i) {
      int st = 0, st2 = 0;
      const int ns2 = nk2[i] > 0 ? splits(nk2[i], kMaxSplits / 4, st2) : 0;
      const int ns = splits(p.rows[i].nk, kMaxSplits - ns2, st);
      if (ns + ns2 > 1) part += ns + ns2;
    }
    return part;
  };
  // Fewer, longer splits until the partials fit: at per >= most_tiles every segment is
  // one split, so only hybrid rows (two segments) still need slots, 2 per row.
  while (per < most_tiles && parts_at() > max_parts) per *= 2;
  int item = 0, part = 0;
  for (int i = 0; i < n; ++i) {
    DecodeRow &r = p.rows[i];
    int st = 0, st2 = 0;
    const int ns2 = nk2[i] > 0 ? splits(nk2[i], kMaxSplits / 4, st2) : 0;
    const int ns = splits(r.nk, kMaxSplits - ns2, st);
    r.item0 = (uint16_t)item;
    r.split_tiles = st;
    r.n_splits = (uint8_t)ns;
    r.split_tiles2 = st2;
    r.n_splits2 = (uint8_t)ns2;
    const int total = ns + ns2;
    r.part0 = (uint16_t)(total > 1 ? part : 0);
    if (total > 1) part += total;
    item += total;
  }
  p.n_rows = n;
  p.n_items = item;
  // one wave or less: the deep-pipeline variant (one CTA per SM, twice the stages);
  // KVINC_DEEP=0 in the environment keeps every launch on the shallow one (measurement)
  static const bool deep_ok = [] {
    const char *e = std::getenv("KVINC_DEEP");
    return !(e && e[0] == '0');
  }();
  p.deep_pipeline = deep_ok && (int64_t)item * Hk <= num_sms ? 1 : 0;
  p.uniform_items = n == 0 ? 0 : p.rows[0].n_splits + p.rows[0].n_splits2;
  for (int i = 1; i < n && p.uniform_items; ++i)
    if (p.rows[i].n_splits + p.rows[i].n_splits2 != p.uniform_items) p.uniform_items = 0;
  return part;
}

namespace {

// Split-K schedule for one batch of decode rows (<= kMaxRowsPerLaunch).  Segment 0 holds
// storage slots [0, nk) of the layer storage (the ring of a sliding layer, else a cache);
// a hybrid layer adds segment 1, its own ring, with its own splits.  Merge tickets are
// kept per cache row.
void plan_decode(const Geom &g, const std::vector<DecodeIn> &in, DecodeParams &p,
                 double &kv_bytes, double &flops) {
  const bool sliding = g.kind == KV_SLIDING, hybrid = is_hybrid(g.kind);
  std::vector<int> nk2(in.size(), 0);
  kv_bytes = 0;
  flops = 0;
  for (size_t i = 0; i < in.size(); ++i) {
    DecodeRow &r = p.rows[i];
    r.cache_row = in[i].cache_row;
    r.call_row = (uint16_t)in[i].call_row;
    r.pos = in[i].pos;
    r.nk = sliding ? std::min(in[i].pos + 1, g.R) : in[i].pos + 1;
    r.ctr = in[i].cache_row;
    if (hybrid) nk2[i] = std::min(in[i].pos + 1, g.R);
    kv_bytes += 2.0 * (r.nk + nk2[i]) * g.Hk * g.D * 2.0;
    flops += 4.0 * (r.nk + nk2[i]) * g.Hq * g.D;
  }
  // the cache's partial buffer holds kMaxSplits slots per row of a launch: no bound
  plan_decode_splits(g.num_sms, g.Hk, (int)in.size(), nk2.data(), p, INT32_MAX);
  p.seg0_ring = sliding ? 1 : 0;
  p.ring_R = g.R > 0 ? g.R : 1;
}

// Parameters of one decode launch (fused RoPE + append + split-K attention + merge) for a
// batch of single-token rows; kv_bytes and flops are the algorithmic counts.
// A hybrid layer's segment 0 is its group's cache: its new global key (k, v) is appended
// by the kernel on a full layer only (on a local layer that key is already in the cache);
// segment 1 is its ring, which takes the new local key (k_local, v_local).
void fill_decode(const kv_cache *c, int layer, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                 const __nv_bfloat16 *v, __nv_bfloat16 *out, int64_t q_row, int64_t kv_row,
                 const std::vector<DecodeIn> &batch, DecodeParams &dp, double &bytes,
                 double &flops, const __nv_bfloat16 *k_local = nullptr,
                 const __nv_bfloat16 *v_local = nullptr) {
  const bool hybrid = is_hybrid(c->kind[layer]);
  dp.tmap_k = c->tmK[layer];
  dp.tmap_v = c->tmV[layer];
  dp.q = q;
  dp.q_row_stride = q_row;
  dp.out = out;
  dp.out_row_stride = q_row;
  dp.rope = c->rope;
  dp.part_o = c->part_o;
  dp.part_ml = c->part_ml;
  dp.counters = c->counters;
  dp.err = c->err;
  dp.k_new = k;
  dp.v_new = v;
  dp.kv_row_stride = kv_row;
  dp.cache_k = (__nv_bfloat16 *)c->K[layer];
  dp.cache_v = (__nv_bfloat16 *)c->V[layer];
  dp.fuse_append = c->kind[layer] != KV_HYBRID_LOCAL;
  dp.Hq = c->Hq;
  dp.Hk = c->Hk;
  dp.rep = c->Hq / c->Hk;
  dp.seg_rows = c->seg_rows[layer];
  dp.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c->D));
  dp.pt = page_table(c, layer);
  dp.tmap_k16 = c->tmK16[layer];
  dp.tmap_v16 = c->tmV16[layer];
  dp.fuse_append2 = hybrid ? 1 : 0;
  dp.early_kv = 0;
  dp.tmap_k2 = hybrid ? c->tmRK[layer] : c->tmK[layer];
  dp.tmap_v2 = hybrid ? c->tmRV[layer] : c->tmV[layer];
  dp.k_new2 = k_local;
  dp.v_new2 = v_local;
  dp.cache_k2 = (__nv_bfloat16 *)c->RK[layer];
  dp.cache_v2 = (__nv_bfloat16 *)c->RV[layer];
  dp.seg_rows2 = c->R + 1;
  double kvb = 0;
  plan_decode(geom_of(c, layer), batch, dp, kvb, flops);
  // q, k, v in (and a hybrid layer's local k, v); new K and V and the output out
  bytes = kvb + (double)batch.size() * (c->Hq + (hybrid ? 4 : 2) * c->Hk) * c->D * 2.0 * 2.0;
}

// Entries of one prefill launch kind for the rows `sel`, each with its key-tile range.
// Without splitting every row is one entry over all its keys.  A launch whose longest CTA
// (a row's whole key range) exceeds the average load per SM is rebalanced: rows longer
// than `per` blocks (about two waves' worth of work per CTA) are cut into key splits,
// each an entry that writes partials at part (vectors counted in *part_vecs), merged
// afterwards by the rows appended to `merges`.
std::vector<PrefillRow> split_prefill_rows(const Geom &g, const std::vector<PrefillRow> &sel,
                                           int rows_per_cta, int ctas_per_sm, int64_t min_per,
                                           std::vector<MergeRow> &merges, int64_t *part_vecs) {
  const bool sliding = g.kind == KV_SLIDING, hybrid = is_hybrid(g.kind);
  const int rep = g.Hq / g.Hk;
  const auto tiles = [](int keys) { return (keys + kTileKeys - 1) / kTileKeys; };
  // the kernels' tile count for a row's last token (t_max = n - 1)
  const auto blocks_of = [&](const PrefillRow &r) {
    const int lr = std::min(r.lens, g.R);
    const int t = sliding ? tiles(lr) + tiles(r.n)
                          : hybrid ? tiles(r.lens + r.n) + tiles(lr) + tiles(r.n)
                                   : tiles(r.lens + r.n);
    return (t + 1) / 2;
  };
  int64_t work = 0;
  int max_blocks = 0;
  for (const PrefillRow &r : sel) {
    const int q = (r.n * rep + rows_per_cta - 1) / rows_per_cta;
    work += (int64_t)q * g.Hk * blocks_of(r);
    max_blocks = std::max(max_blocks, blocks_of(r));
  }
  const int64_t cap = (int64_t)g.num_sms * ctas_per_sm;
  const bool split = max_blocks > (work + cap - 1) / cap;
  const int64_t per = std::max<int64_t>(min_per, (work + 2 * cap - 1) / (2 * cap));
  std::vector<PrefillRow> out;
  for (PrefillRow r : sel) {
    const int blocks = blocks_of(r);
    int ns = split ? (int)std::min<int64_t>(kMaxPrefillSplits, (blocks + per - 1) / per) : 1;
    if (ns <= 1) {
      r.tile0 = 0;
      r.tile1 = INT32_MAX;
      r.part = -1;
      out.push_back(r);
      continue;
    }
    const int bs = (blocks + ns - 1) / ns;
    ns = (blocks + bs - 1) / bs;
    const int n_rho = r.n * rep;
    const int64_t base = *part_vecs;
    *part_vecs += (int64_t)ns * g.Hk * n_rho;
    for (int k = 0; k < ns; ++k) {
      r.tile0 = 2 * bs * k;
      r.tile1 = k == ns - 1 ? INT32_MAX : 2 * bs * (k + 1);
      r.part = (int32_t)(base + (int64_t)k * g.Hk * n_rho);
      out.push_back(r);
    }
    merges.push_back({r.call_row, n_rho, ns, (int32_t)base, 0});
  }
  return out;
}

// Prefill launch kinds: 0 the mma.sync kernel (64 query rows per CTA, two CTAs per SM),
// 1 the tcgen05 kernel with two 128-row query tiles per CTA (one CTA per SM), 2 the
// tcgen05 kernel with one tile per CTA (two CTAs per SM).
constexpr int kPrefillKinds = 3;
constexpr int kRowsPerCta[kPrefillKinds] = {64, 256, 128};
constexpr int kCtasPerSm[kPrefillKinds] = {2, 1, 2};

// Rows whose GQA group x chunk gives at least tc_min_rows(D) query rows go to the tcgen05
// kernel, smaller ones to the mma.sync kernel; hybrid layers (three key segments) all go
// to the tcgen05 kernel.
int prefill_kind(const Geom &g, int n) {
  const int n_rho = n * (g.Hq / g.Hk);
  if (!is_hybrid(g.kind) && n_rho < tc_min_rows(g.D)) return 0;
  return prefill_tc_tiles(g.D, n_rho) == 2 ? 1 : 2;
}

// Partial vectors a cache reserves for prefill key splits (the planner keeps every call
// within it): kPrefillPartVecsPerSm per SM, or the most B rows can need (every query
// vector of a 64-token sub-chunk in kMaxPrefillSplits splits), whichever is smaller.
int64_t prefill_part_cap(int num_sms) { return kPrefillPartVecsPerSm * num_sms; }
int64_t prefill_part_reserve(int num_sms, int B, int Hq) {
  return std::min<int64_t>(prefill_part_cap(num_sms),
                           (int64_t)B * Hq * kChunk * kMaxPrefillSplits);
}

// The prefill entries of one sub-chunk, per launch kind, with their key splits; the
// merges of the split rows and the partial vectors they need, at most
// prefill_part_cap(num_sms): when the load-balancing splits would need more, every split
// is made longer (the minimum blocks per split doubles) until they fit -- at a minimum
// of more blocks than any row has, no row is split.
void plan_prefill(const Geom &g, const std::vector<PrefillRow> &prows,
                  std::vector<PrefillRow> ents[kPrefillKinds], std::vector<MergeRow> &merges,
                  int64_t *part_vecs) {
  std::vector<PrefillRow> sel[kPrefillKinds];
  for (const PrefillRow &r : prows) sel[prefill_kind(g, r.n)].push_back(r);
  const int64_t cap = prefill_part_cap(g.num_sms);
  for (int64_t min_per = kMinSplitBlocks;; min_per *= 2) {
    *part_vecs = 0;
    merges.clear();
    for (int kind = 0; kind < kPrefillKinds; ++kind)
      ents[kind] = split_prefill_rows(g, sel[kind], kRowsPerCta[kind], kCtasPerSm[kind], min_per,
                                      merges, part_vecs);
    if (*part_vecs <= cap || merges.empty()) return;
  }
}

// One layer's chunk for rows `cache_rows`.  k, v: the keys and values of the layer
// storage (a hybrid layer: its group's global keys, nullptr on a local layer); kl, vl: a
// hybrid layer's own local keys and values (its ring), else nullptr.
int append_device(kv_cache *c, int layer, const __nv_bfloat16 *q, const __nv_bfloat16 *k,
                  const __nv_bfloat16 *v, int C, const int32_t *n_new,
                  const std::vector<int32_t> &cache_rows, int Bs, __nv_bfloat16 *out,
                  cudaStream_t s, const __nv_bfloat16 *kl = nullptr,
                  const __nv_bfloat16 *vl = nullptr) {
  const bool sliding = c->kind[layer] == KV_SLIDING, hybrid = is_hybrid(c->kind[layer]);
  const bool writes_global = c->kind[layer] != KV_HYBRID_LOCAL;  // appends k, v anywhere
  c->cur_layer = layer;
  const bool ringed = sliding || hybrid;                          // keeps a ring
  const int Hq = c->Hq, Hk = c->Hk, D = c->D, rep = Hq / Hk;
  int max_n = 0;
  for (int i = 0; i < Bs; ++i) max_n = std::max(max_n, (int)n_new[i]);
  if (max_n == 0) return KV_OK;
  // the chunk rows of the sub-chunk at token offset `off`: rows of two or more new tokens
  // with tokens left there
  const auto chunk_rows = [&](int off) {
    std::vector<PrefillRow> rows;
    for (int i = 0; i < Bs; ++i)
      if (n_new[i] >= 2 && n_new[i] > off)
        rows.push_back({cache_rows[i], i, c->lens[cache_rows[i]] + off,
                        std::min(kChunk, n_new[i] - off), 0});
    return rows;
  };
  if (c->n_blocks > 0) {  // pool blocks for the new positions, before anything is enqueued
    std::vector<std::pair<int, int>> want;
    for (int i = 0; i < Bs; ++i)
      if (n_new[i] > 0) want.push_back({cache_rows[i], c->lens[cache_rows[i]] + n_new[i]});
    const int rc = ensure_blocks(c, want, s);
    if (rc != KV_OK) return rc;
  }

  const int64_t q_row = (int64_t)C * Hq * D, kv_row = (int64_t)C * Hk * D;
  static thread_local AppendParams ap;
  static thread_local DecodeParams dp;
  static thread_local PrefillParams pp;
  static thread_local CommitParams mp;
  const float scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));

  for (int off = 0; off < max_n; off += kChunk) {
    std::vector<AppendRow> arows, lrows;  // to the layer storage / a hybrid ring's scratch
    std::vector<DecodeIn> drows;          // single-token rows: appended inside the decode kernel
    const std::vector<PrefillRow> prows = chunk_rows(off);
    if (off == 0)
      for (int i = 0; i < Bs; ++i)
        if (n_new[i] == 1) drows.push_back({cache_rows[i], i, c->lens[cache_rows[i]]});
    for (const PrefillRow &r : prows) {
      if (writes_global)
        arows.push_back({r.cache_row, r.call_row, r.lens, r.n,
                         sliding ? kDestScratch : kDestGlobal, 0});
      if (hybrid) lrows.push_back({r.cache_row, r.call_row, r.lens, r.n, kDestScratch, 0});
    }

    // ---- RoPE + append of the chunk rows of this sub-chunk (a hybrid layer: the global
    // keys to the group's cache, then its local keys to the chunk scratch)
    for (int pass = 0; pass < 2; ++pass) {
    const std::vector<AppendRow> &rows_p = pass == 0 ? arows : lrows;
    const __nv_bfloat16 *kp = pass == 0 ? k : kl, *vp = pass == 0 ? v : vl;
    for (size_t r0 = 0; r0 < rows_p.size(); r0 += kMaxRowsPerLaunch) {
      const size_t r1 = std::min(rows_p.size(), r0 + kMaxRowsPerLaunch);
      ap.k = kp + (int64_t)off * Hk * D;
      ap.v = vp + (int64_t)off * Hk * D;
      ap.kv_row_stride = kv_row;
      ap.cache_k = (__nv_bfloat16 *)c->K[layer];
      ap.cache_v = (__nv_bfloat16 *)c->V[layer];
      ap.scr_k = (__nv_bfloat16 *)c->scrK;
      ap.scr_v = (__nv_bfloat16 *)c->scrV;
      ap.rope = c->rope;
      ap.Hk = Hk;
      ap.D = D;
      ap.seg_rows = c->seg_rows[layer];
      ap.ring_R = c->R;
      ap.max_len = c->max_len;
      ap.c_avail = C - off;
      ap.pt = page_table(c, layer);
      int blk = 0;
      double bytes = 0;
      for (size_t j = r0; j < r1; ++j) {
        AppendRow r = rows_p[j];
        r.blk0 = blk;
        blk += (r.n + 7) / 8;
        ap.rows[j - r0] = r;
        bytes += 4.0 * r.n * Hk * D * 2.0;
      }
      ap.n_rows = (int)(r1 - r0);
      ap.n_blocks = blk;
      cudaError_t e = timed(c, KV_KERNEL_APPEND, bytes, 0, s, [&] { return launch_append(ap, s, c->pdl); });
      if (e != cudaSuccess) return KV_ERR_CUDA;
    }
    }

    // ---- split-K decode for single-token rows (append and split merge fused in)
    for (size_t r0 = 0; r0 < drows.size(); r0 += kMaxRowsPerLaunch) {
      const size_t r1 = std::min(drows.size(), r0 + kMaxRowsPerLaunch);
      std::vector<DecodeIn> batch(drows.begin() + r0, drows.begin() + r1);
      double bytes = 0, fl = 0;
      fill_decode(c, layer, q, k, v, out, q_row, kv_row, batch, dp, bytes, fl, kl, vl);
      const int nt = rep <= 8 ? 1 : 2;
      dp.early_kv = early_kv_ok(c, layer, s) ? 1 : 0;
      // the deep variant pays off with the programmatic overlap of successive launches
      // (long-context step 6058 -> 6201 GB/s), not without it
      if (!c->pdl) dp.deep_pipeline = 0;
      cudaError_t e = timed(c, KV_KERNEL_DECODE, bytes, fl, s,
                            [&] { return launch_decode(dp, D, nt, s, c->pdl); });
      if (e != cudaSuccess) return KV_ERR_CUDA;
    }

    // ---- chunked prefill (+ ring commit on sliding layers), in launches of each kind
    std::vector<PrefillRow> ents[kPrefillKinds];
    std::vector<MergeRow> merges;
    int64_t part_vecs = 0;  // within the reserve made at create (the planner's bound)
    plan_prefill(geom_of(c, layer), prows, ents, merges, &part_vecs);
    for (int kind = 0; kind < kPrefillKinds; ++kind) {
      const std::vector<PrefillRow> &sel = ents[kind];
      for (size_t r0 = 0; r0 < sel.size(); r0 += kMaxRowsPerLaunch) {
        const size_t r1 = std::min(sel.size(), r0 + kMaxRowsPerLaunch);
        pp.tmap_k = c->tmK[layer];
        pp.tmap_v = c->tmV[layer];
        pp.tmap_sk = c->tmSK;
        pp.tmap_sv = c->tmSV;
        pp.q = q + (int64_t)off * Hq * D;
        pp.q_row_stride = q_row;
        pp.out = out + (int64_t)off * Hq * D;
        pp.out_row_stride = q_row;
        pp.rope = c->rope;
        pp.err = c->err;
        pp.Hq = Hq;
        pp.Hk = Hk;
        pp.rep = rep;
        pp.seg_rows = c->seg_rows[layer];
        pp.sliding = sliding ? 1 : 0;
        pp.ring_R = c->R;
        pp.window = c->W;
        pp.scale_log2 = scale_log2;
        pp.pt = page_table(c, layer);
        pp.tmap_k16 = c->tmK16[layer];
        pp.tmap_v16 = c->tmV16[layer];
        pp.hybrid = hybrid ? 1 : 0;
        pp.tmap_k2 = hybrid ? c->tmRK[layer] : c->tmK[layer];
        pp.tmap_v2 = hybrid ? c->tmRV[layer] : c->tmV[layer];
        pp.seg_rows2 = c->R + 1;
        pp.part_o = c->ppart_o;
        pp.part_ml = c->ppart_ml;
        int cta = 0;
        double bytes = 0, fl = 0;
        for (size_t j = r0; j < r1; ++j) {
          PrefillRow r = sel[j];
          r.cta0 = cta;
          cta += (r.n * rep + kRowsPerCta[kind] - 1) / kRowsPerCta[kind];
          pp.rows[j - r0] = r;
          if (r.tile0 != 0) continue;  // a row's work is counted with its first entry
          const int lkeys = std::min(r.lens, c->R) + r.n;
          const int keys = sliding ? lkeys : hybrid ? r.lens + r.n + lkeys : r.lens + r.n;
          bytes += 2.0 * keys * Hk * D * 2.0 + 2.0 * r.n * Hq * D * 2.0;
          for (int t = 0; t < r.n; ++t) {
            const int pz = r.lens + t;
            const int lvis = std::min(pz + 1, c->W);
            const int vis = sliding ? lvis : hybrid ? pz + 1 + lvis : pz + 1;
            fl += 4.0 * vis * Hq * D;
          }
        }
        pp.n_rows = (int)(r1 - r0);
        pp.n_ctas = cta;
        cudaError_t e = timed(c, KV_KERNEL_PREFILL, bytes, fl, s, [&] {
          return kind == 0 ? launch_prefill(pp, D, s, c->pdl)
                           : launch_prefill_tc(pp, D, kind == 1 ? 2 : 1, s, c->pdl);
        });
        if (e != cudaSuccess) return KV_ERR_CUDA;
      }
    }
    // ---- merge of the key-split rows (log-sum-exp over their partials)
    for (size_t r0 = 0; r0 < merges.size(); r0 += kMaxRowsPerLaunch) {
      const size_t r1 = std::min(merges.size(), r0 + kMaxRowsPerLaunch);
      static thread_local MergeParams mg;
      mg.part_o = c->ppart_o;
      mg.part_ml = c->ppart_ml;
      mg.out = out + (int64_t)off * Hq * D;
      mg.out_row_stride = q_row;
      mg.Hq = Hq;
      mg.Hk = Hk;
      mg.rep = rep;
      int vec = 0;
      double mb = 0;
      for (size_t j = r0; j < r1; ++j) {
        MergeRow m = merges[j];
        m.vec0 = vec;
        vec += Hk * m.n_rho;
        mg.rows[j - r0] = m;
        mb += (double)Hk * m.n_rho * (m.n_splits * (D * 4.0 + 8.0) + D * 2.0);
      }
      mg.n_rows = (int)(r1 - r0);
      mg.n_vec = vec;
      cudaError_t e = timed(c, KV_KERNEL_COMBINE, mb, 0, s,
                            [&] { return launch_prefill_merge(mg, D, s, c->pdl); });
      if (e != cudaSuccess) return KV_ERR_CUDA;
    }
    if (ringed) {
      for (size_t r0 = 0; r0 < prows.size(); r0 += kMaxRowsPerLaunch) {
        const size_t r1 = std::min(prows.size(), r0 + kMaxRowsPerLaunch);
        mp.scr_k = (const __nv_bfloat16 *)c->scrK;
        mp.scr_v = (const __nv_bfloat16 *)c->scrV;
        mp.ring_k = (__nv_bfloat16 *)(hybrid ? c->RK[layer] : c->K[layer]);
        mp.ring_v = (__nv_bfloat16 *)(hybrid ? c->RV[layer] : c->V[layer]);
        mp.Hk = Hk;
        mp.D = D;
        mp.ring_R = c->R;
        mp.window = c->W;
        mp.seg_rows = hybrid ? c->R + 1 : c->seg_rows[layer];
        double cb = 0;
        for (size_t j = r0; j < r1; ++j) {
          mp.cache_row[j - r0] = prows[j].cache_row;
          mp.lens[j - r0] = prows[j].lens;
          mp.n[j - r0] = prows[j].n;
          cb += 4.0 * std::min(prows[j].n, c->W) * Hk * D * 2.0;
        }
        mp.n_rows = (int)(r1 - r0);
        cudaError_t e = timed(c, KV_KERNEL_COMMIT, cb, 0, s, [&] { return launch_commit(mp, s, c->pdl); });
        if (e != cudaSuccess) return KV_ERR_CUDA;
      }
    }
  }
  return KV_OK;
}

// lpos update of one advance for rows [r0, r1) of `rows` (rows with n_new = 0 skipped).
void fill_state(const kv_cache *c, const std::vector<int32_t> &rows, const int32_t *n_new,
                bool reset, size_t r0, size_t r1, StateParams &sp) {
  sp.lpos = c->lpos;
  sp.ring_R = c->R;
  sp.window = c->W;
  sp.reset = reset ? 1 : 0;
  int n = 0;
  for (size_t j = r0; j < r1; ++j) {
    if (!reset && n_new[j] == 0) continue;
    sp.cache_row[n] = rows[j];
    sp.lens[n] = c->lens[rows[j]];
    sp.n[n] = reset ? 0 : n_new[j];
    ++n;
  }
  sp.n_rows = n;
}

int state_update(kv_cache *c, const std::vector<int32_t> &rows, const int32_t *n_new, bool reset,
                 cudaStream_t s) {
  if (!c->lpos) return KV_OK;  // lens lives on the host; lpos exists with sliding layers only
  static thread_local StateParams sp;
  for (size_t r0 = 0; r0 < rows.size(); r0 += kMaxRowsPerLaunch) {
    const size_t r1 = std::min(rows.size(), r0 + kMaxRowsPerLaunch);
    fill_state(c, rows, n_new, reset, r0, r1, sp);
    cudaError_t e = timed(c, KV_KERNEL_STATE, 0, 0, s, [&] { return launch_state(sp, s, c->pdl); });
    if (e != cudaSuccess) return KV_ERR_CUDA;
  }
  return KV_OK;
}

void free_all(kv_cache *c) {
  for (size_t l = 0; l < c->K.size(); ++l)
    if (l < c->owns.size() && c->owns[l]) {
      cudaFree(c->K[l]);
      cudaFree(c->V[l]);
    }
  for (void *p : c->RK) cudaFree(p);
  for (void *p : c->RV) cudaFree(p);
  cudaFree(c->scrK);
  cudaFree(c->scrV);
  cudaFree(c->rope);
  cudaFree(c->counters);
  cudaFree(c->lpos);
  cudaFree(c->err);
  cudaFree(c->part_o);
  cudaFree(c->part_ml);
  cudaFree(c->ppart_o);
  cudaFree(c->ppart_ml);
  cudaFree(c->stage);
  cudaFree(c->table);
  for (auto &r : c->recs) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  for (auto e : c->free_events) cudaEventDestroy(e);
}

}  // namespace

static int create_impl(kv_cache **out, int B, int max_len, int Hq, int Hk, int D, int W,
                       int n_layers, const int32_t *layer_kind, double rope_theta, int device,
                       int n_blocks) {
  if (!out) return KV_ERR_ARG;
  *out = nullptr;
  if (n_blocks < 0 || (int64_t)n_blocks * Hk * kBlockTokens >= (1LL << 31)) return KV_ERR_ARG;
  if (B < 1 || max_len < 1 || max_len > (1 << 20) || Hk < 1 || Hq < 1 || Hq % Hk != 0 ||
      Hq / Hk > kMaxRep || (D != 64 && D != 128) || n_layers < 1 || !layer_kind ||
      !(rope_theta > 0.0) || device < 0)
    return KV_ERR_ARG;
  bool any_sliding = false;  // any ring (sliding or hybrid layers)
  int last_full = -1;
  for (int l = 0; l < n_layers; ++l) {
    const int k = layer_kind[l];
    if (k != KV_GLOBAL && k != KV_SLIDING && k != KV_HYBRID_FULL && k != KV_HYBRID_LOCAL)
      return KV_ERR_ARG;
    if (k == KV_HYBRID_FULL) last_full = l;
    if (k == KV_HYBRID_LOCAL && last_full < 0) return KV_ERR_ARG;  // no group to read
    any_sliding |= k != KV_GLOBAL;
  }
  if (any_sliding && W < 1) return KV_ERR_ARG;
  const int R = any_sliding ? (W < max_len ? W : max_len) : 0;
  // TMA row coordinates of the dense caches, the rings and the chunk scratch
  if (n_blocks == 0 && (int64_t)B * Hk * (max_len + 1) >= (1LL << 31)) return KV_ERR_ARG;
  if ((int64_t)B * Hk * (R + 1) >= (1LL << 31) || (int64_t)B * Hk * kChunk >= (1LL << 31))
    return KV_ERR_ARG;

  int n_dev = 0;
  if (cudaGetDeviceCount(&n_dev) != cudaSuccess || device >= n_dev) return KV_ERR_CUDA;
  DeviceGuard guard(device);
  if (!get_encode_fn()) return KV_ERR_CUDA;
  if (configure_decode() != cudaSuccess || configure_prefill() != cudaSuccess ||
      configure_prefill_tc() != cudaSuccess)
    return KV_ERR_CUDA;

  kv_cache *c = new kv_cache();
  c->B = B;
  c->max_len = max_len;
  c->Hq = Hq;
  c->Hk = Hk;
  c->D = D;
  c->W = any_sliding ? W : 0;
  c->R = R;
  c->n_layers = n_layers;
  c->device = device;
  c->theta = rope_theta;
  c->kind.assign(layer_kind, layer_kind + n_layers);
  c->lens.assign(B, 0);
  cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device);
  if (c->num_sms < 1) c->num_sms = 1;

  auto fail = [&](int code) {
    free_all(c);
    delete c;
    return code;
  };
  auto alloc = [&](void **p, size_t bytes) {
    if (cudaMalloc(p, bytes) != cudaSuccess) return false;
    return cudaMemset(*p, 0, bytes) == cudaSuccess;  // stale slots stay finite
  };

  c->n_blocks = n_blocks;
  if (n_blocks > 0) {
    c->max_blocks = (blocks_for(max_len) + 3) / 4 * 4;
    if (!alloc((void **)&c->table, (size_t)B * c->max_blocks * 4)) return fail(KV_ERR_OOM);
    c->rblocks.assign(B, {});
    c->refs.assign(n_blocks, 0);
    for (int b = n_blocks - 1; b >= 0; --b) c->free_blocks.push_back(b);
  }
  int group_full = -1;
  c->hy_end.assign(n_layers, {});
  for (int l = 0; l < n_layers; ++l) {
    if (c->kind[l] == KV_HYBRID_FULL) {
      group_full = l;
      c->hy_end[l].assign(B, 0);
    }
    c->group.push_back(is_hybrid(c->kind[l]) ? group_full : -1);
    // the ring of a hybrid layer
    if (is_hybrid(c->kind[l])) {
      const size_t rbytes = (size_t)B * Hk * (R + 1) * D * 2;
      void *rk = nullptr, *rv = nullptr;
      if (!alloc(&rk, rbytes)) return fail(KV_ERR_OOM);
      c->RK.push_back(rk);
      if (!alloc(&rv, rbytes)) return fail(KV_ERR_OOM);
      c->RV.push_back(rv);
      CUtensorMap rmk, rmv;
      if (!make_tmap(&rmk, rk, (int64_t)B * Hk * (R + 1), D) ||
          !make_tmap(&rmv, rv, (int64_t)B * Hk * (R + 1), D))
        return fail(KV_ERR_CUDA);
      c->tmRK.push_back(rmk);
      c->tmRV.push_back(rmv);
    } else {
      c->RK.push_back(nullptr);
      c->RV.push_back(nullptr);
      c->tmRK.push_back(CUtensorMap{});
      c->tmRV.push_back(CUtensorMap{});
    }
    if (c->kind[l] == KV_HYBRID_LOCAL) {  // the group's cache, owned by its full layer
      const int f = c->group[l];
      c->K.push_back(c->K[f]);
      c->V.push_back(c->V[f]);
      c->owns.push_back(0);
      c->seg_rows.push_back(c->seg_rows[f]);
      c->tmK.push_back(c->tmK[f]);
      c->tmV.push_back(c->tmV[f]);
      c->tmK16.push_back(c->tmK16[f]);
      c->tmV16.push_back(c->tmV16[f]);
      continue;
    }
    // dense: [B][Hk][rows][D]; paged cache layer: pool [Hk][n_blocks][16][D]
    const bool pg = n_blocks > 0 && c->kind[l] != KV_SLIDING;
    const int rows = pg ? kBlockTokens : c->kind[l] == KV_SLIDING ? R + 1 : max_len + 1;
    c->owns.push_back(1);
    const int64_t units = pg ? n_blocks : B;
    const size_t bytes = (size_t)units * Hk * rows * D * 2;
    void *k = nullptr, *v = nullptr;
    if (!alloc(&k, bytes)) return fail(KV_ERR_OOM);
    c->K.push_back(k);
    if (!alloc(&v, bytes)) return fail(KV_ERR_OOM);
    c->V.push_back(v);
    c->seg_rows.push_back(rows);
    CUtensorMap mk, mv, mk16, mv16;
    if (!make_tmap(&mk, k, units * Hk * rows, D) || !make_tmap(&mv, v, units * Hk * rows, D))
      return fail(KV_ERR_CUDA);
    if (pg) {
      if (!make_tmap(&mk16, k, units * Hk * rows, D, kBlockTokens) ||
          !make_tmap(&mv16, v, units * Hk * rows, D, kBlockTokens))
        return fail(KV_ERR_CUDA);
    } else {
      mk16 = mk;
      mv16 = mv;
    }
    c->tmK.push_back(mk);
    c->tmV.push_back(mv);
    c->tmK16.push_back(mk16);
    c->tmV16.push_back(mv16);
  }
  const size_t scr = (size_t)B * Hk * kChunk * D * 2;
  if (!alloc(&c->scrK, scr) || !alloc(&c->scrV, scr)) return fail(KV_ERR_OOM);
  if (!make_tmap(&c->tmSK, c->scrK, (int64_t)B * Hk * kChunk, D) ||
      !make_tmap(&c->tmSV, c->scrV, (int64_t)B * Hk * kChunk, D))
    return fail(KV_ERR_CUDA);

  // RoPE table: theta^(-2i/D) with the exponent as the double quotient (-2i)/D,
  // angle p * theta_i in double, cos/sin rounded once to float.
  {
    const int half = D / 2;
    std::vector<double> inv(half);
    for (int i = 0; i < half; ++i) inv[i] = std::pow(rope_theta, (double)(-2 * i) / (double)D);
    std::vector<float2> tab((size_t)max_len * half);
    for (int p = 0; p < max_len; ++p)
      for (int i = 0; i < half; ++i) {
        const double a = (double)p * inv[i];
        tab[(size_t)p * half + i] = make_float2((float)std::cos(a), (float)std::sin(a));
      }
    if (cudaMalloc((void **)&c->rope, tab.size() * sizeof(float2)) != cudaSuccess)
      return fail(KV_ERR_OOM);
    if (cudaMemcpy(c->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) !=
        cudaSuccess)
      return fail(KV_ERR_CUDA);
  }
  if (!alloc((void **)&c->counters, (size_t)B * Hk * 4) || !alloc((void **)&c->err, 16))
    return fail(KV_ERR_OOM);
  if (R > 0) {
    if (cudaMalloc((void **)&c->lpos, (size_t)B * R * 4) != cudaSuccess) return fail(KV_ERR_OOM);
    if (cudaMemset(c->lpos, 0xFF, (size_t)B * R * 4) != cudaSuccess) return fail(KV_ERR_CUDA);
  }
  // decode partial slots are numbered per launch (at most kMaxRowsPerLaunch rows)
  const size_t parts = (size_t)std::min(B, kMaxRowsPerLaunch) * kMaxSplits * Hq;
  if (!alloc((void **)&c->part_o, parts * D * 4) || !alloc((void **)&c->part_ml, parts * 8))
    return fail(KV_ERR_OOM);
  // prefill key-split partials: every call's plan fits (plan_prefill), so kv_append never
  // allocates
  c->ppart_cap = prefill_part_reserve(c->num_sms, B, Hq);
  if (!alloc((void **)&c->ppart_o, (size_t)c->ppart_cap * D * 4) ||
      !alloc((void **)&c->ppart_ml, (size_t)c->ppart_cap * 8))
    return fail(KV_ERR_OOM);
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(KV_ERR_CUDA);
  if (const char *pdl = std::getenv("KVINC_PDL")) c->pdl = pdl[0] != '0';
  if (const char *log = std::getenv("KVINC_LOG")) {
    if (log[0] == '1')
      std::fprintf(stderr, "[kv] %.1f MiB K/V (%d layers, B=%d, Hk=%d, D=%d, max_len=%d, R=%d)\n",
                   kv_nbytes(c) / 1048576.0, n_layers, B, Hk, D, max_len, R);
  }
  *out = c;
  return KV_OK;
}

extern "C" {

int kv_cache_create(kv_cache **out, int B, int max_len, int Hq, int Hk, int D, int W,
                    int n_layers, const int32_t *layer_kind, double rope_theta, int device) {
  return create_impl(out, B, max_len, Hq, Hk, D, W, n_layers, layer_kind, rope_theta, device, 0);
}

int kv_cache_create_paged(kv_cache **out, int B, int max_len, int Hq, int Hk, int D, int W,
                          int n_layers, const int32_t *layer_kind, double rope_theta, int device,
                          int n_blocks) {
  if (n_blocks < 1) {
    if (out) *out = nullptr;
    return KV_ERR_ARG;
  }
  return create_impl(out, B, max_len, Hq, Hk, D, W, n_layers, layer_kind, rope_theta, device,
                     n_blocks);
}

int kv_get_block_table(const kv_cache *c, int row, int32_t *blocks_out, int capacity,
                       int *n_out) {
  if (!c || row < 0 || row >= c->B || capacity < 0 || (capacity > 0 && !blocks_out))
    return KV_ERR_ARG;
  const int n = c->n_blocks > 0 ? (int)c->rblocks[row].size() : 0;
  if (n_out) *n_out = n;
  for (int i = 0; i < n && i < capacity; ++i) blocks_out[i] = c->rblocks[row][i];
  return KV_OK;
}

int kv_free_blocks(const kv_cache *c) {
  return c ? (int)c->free_blocks.size() : -1;
}

void kv_cache_destroy(kv_cache *c) {
  if (!c) return;
  DeviceGuard guard(c->device);
  cudaDeviceSynchronize();
  free_all(c);
  delete c;
}

int kv_reset(kv_cache *c, const int32_t *rows, int n_rows, void *stream) {
  if (!c || n_rows < 0 || (n_rows > 0 && !rows)) return KV_ERR_ARG;
  std::vector<char> seen(c->B, 0);
  std::vector<int32_t> rv(rows, rows + n_rows);
  for (int r : rv) {
    if (r < 0 || r >= c->B || seen[r]) return KV_ERR_ARG;
    seen[r] = 1;
  }
  if (n_rows == 0) return KV_OK;
  DeviceGuard guard(c->device);
  const int rc = state_update(c, rv, nullptr, true, (cudaStream_t)stream);
  if (rc != KV_OK) return rc;
  for (int r : rv) {
    c->lens[r] = 0;
    release_blocks(c, r, 0);  // later launches on this stream may reuse them
    for (auto &he : c->hy_end)
      if (!he.empty()) he[r] = 0;
  }
  return KV_OK;
}

int kv_append(kv_cache *c, int layer, const void *q, const void *k, const void *v, int Hq, int C,
              const int32_t *n_new, const int32_t *rows, int Bs, void *out, void *stream) {
  if (!c || layer < 0 || layer >= c->n_layers || Hq != c->Hq || C < 1) return KV_ERR_ARG;
  if (is_hybrid(c->kind[layer])) return KV_ERR_ARG;  // kv_append_hybrid
  std::vector<int32_t> cache_rows;
  const int rc = check_rows(c, n_new, rows, Bs, C, cache_rows);
  if (rc != KV_OK) return rc;
  bool any = false;
  for (int i = 0; i < Bs; ++i) any |= n_new[i] > 0;
  if (!any) return KV_OK;
  if (!q || !k || !v || !out || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return KV_ERR_ARG;
  DeviceGuard guard(c->device);
  return append_device(c, layer, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k,
                       (const __nv_bfloat16 *)v, C, n_new, cache_rows, Bs, (__nv_bfloat16 *)out,
                       (cudaStream_t)stream);
}

// Device address of a page-locked host buffer the GPU can reach directly (on GB300
// pinned host memory is coherent over NVLink-C2C), or nullptr.
static const void *mapped_host(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error of a plain pageable pointer
    return nullptr;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer) return a.devicePointer;
  return nullptr;
}

// Host-buffer form of one layer's append: k, v are the layer's keys and values (a hybrid
// layer: the group's global ones, NULL on a local layer), kl, vl a hybrid layer's local ones.
// Page-locked buffers are used in place (the kernels read the inputs and write the outputs in
// host memory; the bytes cross NVLink-C2C inside the kernels); pageable ones are staged
// through device buffers owned by the cache.
static int append_host_impl(kv_cache *c, int layer, const void *q, const void *k, const void *v,
                            const void *kl, const void *vl, int C, const int32_t *n_new,
                            const std::vector<int32_t> &cache_rows, int Bs, void *out,
                            cudaStream_t s) {
  const void *src[5] = {q, k, v, kl, vl};
  const void *mapped[5] = {};
  bool all_mapped = true;
  for (int i = 0; i < 5; ++i) {
    if (!src[i]) continue;
    mapped[i] = mapped_host(src[i]);
    all_mapped = all_mapped && mapped[i] && aligned16(mapped[i]);
  }
  void *mo = const_cast<void *>(mapped_host(out));
  if (all_mapped && mo && aligned16(mo))
    return append_device(c, layer, (const __nv_bfloat16 *)mapped[0],
                         (const __nv_bfloat16 *)mapped[1], (const __nv_bfloat16 *)mapped[2], C,
                         n_new, cache_rows, Bs, (__nv_bfloat16 *)mo, s,
                         (const __nv_bfloat16 *)mapped[3], (const __nv_bfloat16 *)mapped[4]);
  const size_t qb = (size_t)Bs * C * c->Hq * c->D * 2, kb = (size_t)Bs * C * c->Hk * c->D * 2;
  const size_t sizes[5] = {qb, kb, kb, kb, kb};
  auto al = [](size_t x) { return (x + 15) & ~size_t(15); };
  size_t need = al(qb) + 64;  // the output
  for (int i = 0; i < 5; ++i)
    if (src[i]) need += al(sizes[i]);
  if (need > c->stage_bytes) {
    // The old buffer may still be in use by queued work on this stream.
    if (c->stage && cudaStreamSynchronize(s) != cudaSuccess) return KV_ERR_CUDA;
    cudaFree(c->stage);
    c->stage = nullptr;
    c->stage_bytes = 0;
    if (cudaMalloc(&c->stage, need) != cudaSuccess) return KV_ERR_OOM;
    c->stage_bytes = need;
  }
  char *cur = (char *)c->stage;
  const __nv_bfloat16 *dev[5] = {};
  for (int i = 0; i < 5; ++i) {
    if (!src[i]) continue;
    if (cudaMemcpyAsync(cur, src[i], sizes[i], cudaMemcpyHostToDevice, s) != cudaSuccess)
      return KV_ERR_CUDA;
    dev[i] = (const __nv_bfloat16 *)cur;
    cur += al(sizes[i]);
  }
  __nv_bfloat16 *dout = (__nv_bfloat16 *)cur;
  const int r = append_device(c, layer, dev[0], dev[1], dev[2], C, n_new, cache_rows, Bs, dout,
                              s, dev[3], dev[4]);
  if (r != KV_OK) return r;
  return set_err(cudaMemcpyAsync(out, dout, qb, cudaMemcpyDeviceToHost, s));
}

int kv_append_host(kv_cache *c, int layer, const void *q, const void *k, const void *v, int Hq,
                   int C, const int32_t *n_new, const int32_t *rows, int Bs, void *out,
                   void *stream) {
  if (!c || layer < 0 || layer >= c->n_layers || Hq != c->Hq || C < 1) return KV_ERR_ARG;
  if (is_hybrid(c->kind[layer])) return KV_ERR_ARG;
  std::vector<int32_t> cache_rows;
  const int rc = check_rows(c, n_new, rows, Bs, C, cache_rows);
  if (rc != KV_OK) return rc;
  bool any = false;
  for (int i = 0; i < Bs; ++i) any |= n_new[i] > 0;
  if (!any) return KV_OK;
  if (!q || !k || !v || !out) return KV_ERR_ARG;
  DeviceGuard guard(c->device);
  return append_host_impl(c, layer, q, k, v, nullptr, nullptr, C, n_new, cache_rows, Bs, out,
                          (cudaStream_t)stream);
}

// Checks shared by the hybrid entry points; fills cache_rows.  KV_OK with any = false: no
// row has new tokens.
static int check_hybrid(kv_cache *c, int layer, const void *q, const void *k_local,
                        const void *v_local, const void *k_global, const void *v_global, int Hq,
                        int C, const int32_t *n_new, const int32_t *rows, int Bs, const void *out,
                        std::vector<int32_t> &cache_rows, bool &any) {
  if (!c || layer < 0 || layer >= c->n_layers || Hq != c->Hq || C < 1) return KV_ERR_ARG;
  if (!is_hybrid(c->kind[layer])) return KV_ERR_ARG;
  const bool full = c->kind[layer] == KV_HYBRID_FULL;
  const int rc = check_rows(c, n_new, rows, Bs, C, cache_rows);
  if (rc != KV_OK) return rc;
  any = false;
  for (int i = 0; i < Bs; ++i) any |= n_new[i] > 0;
  if (!any) return KV_OK;
  if (!q || !k_local || !v_local || !out) return KV_ERR_ARG;
  if (full ? (!k_global || !v_global) : (k_global || v_global)) return KV_ERR_ARG;
  // a local layer reads the group's global keys of these tokens: its full layer must
  // have appended exactly them
  const std::vector<int32_t> &he = c->hy_end[c->group[layer]];
  if (!full)
    for (int i = 0; i < Bs; ++i)
      if (n_new[i] > 0 && he[cache_rows[i]] != c->lens[cache_rows[i]] + n_new[i])
        return KV_ERR_ARG;
  return KV_OK;
}

static void note_hybrid_append(kv_cache *c, int layer, const int32_t *n_new,
                               const std::vector<int32_t> &cache_rows, int Bs) {
  if (c->kind[layer] != KV_HYBRID_FULL) return;
  for (int i = 0; i < Bs; ++i)
    if (n_new[i] > 0) c->hy_end[layer][cache_rows[i]] = c->lens[cache_rows[i]] + n_new[i];
}

int kv_append_hybrid(kv_cache *c, int layer, const void *q, const void *k_local,
                     const void *v_local, const void *k_global, const void *v_global, int Hq,
                     int C, const int32_t *n_new, const int32_t *rows, int Bs, void *out,
                     void *stream) {
  std::vector<int32_t> cache_rows;
  bool any = false;
  int rc = check_hybrid(c, layer, q, k_local, v_local, k_global, v_global, Hq, C, n_new, rows,
                        Bs, out, cache_rows, any);
  if (rc != KV_OK || !any) return rc;
  for (const void *x : {q, k_local, v_local, (const void *)out})
    if (!aligned16(x)) return KV_ERR_ARG;
  if (k_global && (!aligned16(k_global) || !aligned16(v_global))) return KV_ERR_ARG;
  DeviceGuard guard(c->device);
  rc = append_device(c, layer, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)k_global,
                     (const __nv_bfloat16 *)v_global, C, n_new, cache_rows, Bs,
                     (__nv_bfloat16 *)out, (cudaStream_t)stream,
                     (const __nv_bfloat16 *)k_local, (const __nv_bfloat16 *)v_local);
  if (rc == KV_OK) note_hybrid_append(c, layer, n_new, cache_rows, Bs);
  return rc;
}

int kv_append_hybrid_host(kv_cache *c, int layer, const void *q, const void *k_local,
                          const void *v_local, const void *k_global, const void *v_global, int Hq,
                          int C, const int32_t *n_new, const int32_t *rows, int Bs, void *out,
                          void *stream) {
  std::vector<int32_t> cache_rows;
  bool any = false;
  int rc = check_hybrid(c, layer, q, k_local, v_local, k_global, v_global, Hq, C, n_new, rows,
                        Bs, out, cache_rows, any);
  if (rc != KV_OK || !any) return rc;
  DeviceGuard guard(c->device);
  rc = append_host_impl(c, layer, q, k_global, v_global, k_local, v_local, C, n_new, cache_rows,
                        Bs, out, (cudaStream_t)stream);
  if (rc == KV_OK) note_hybrid_append(c, layer, n_new, cache_rows, Bs);
  return rc;
}

int kv_advance(kv_cache *c, const int32_t *n_new, const int32_t *rows, int Bs, void *stream) {
  if (!c) return KV_ERR_ARG;
  std::vector<int32_t> cache_rows;
  const int rc = check_rows(c, n_new, rows, Bs, c->max_len, cache_rows);
  if (rc != KV_OK) return rc;
  DeviceGuard guard(c->device);
  const int r = state_update(c, cache_rows, n_new, false, (cudaStream_t)stream);
  if (r != KV_OK) return r;
  for (int i = 0; i < Bs; ++i) c->lens[cache_rows[i]] += n_new[i];
  return KV_OK;
}

int64_t kv_nbytes(const kv_cache *c) {
  if (!c) return -1;
  int64_t total = 0;
  for (int l = 0; l < c->n_layers; ++l) {
    if (c->owns[l])
      total += paged_layer(c, l) ? 2LL * c->n_blocks * c->Hk * kBlockTokens * c->D * 2
                                 : 2LL * c->B * c->Hk * c->seg_rows[l] * c->D * 2;
    if (c->RK[l]) total += 2LL * c->B * c->Hk * (c->R + 1) * c->D * 2;  // a hybrid ring
  }
  return total;
}

int kv_get_lens(const kv_cache *c, int32_t *lens_out) {
  if (!c || !lens_out) return KV_ERR_ARG;
  std::memcpy(lens_out, c->lens.data(), sizeof(int32_t) * c->B);
  return KV_OK;
}

int kv_debug_ptrs(const kv_cache *c, int layer, void **K, void **V, int32_t **lpos) {
  if (!c || layer < 0 || layer >= c->n_layers) return KV_ERR_ARG;
  if (K) *K = c->K[layer];
  if (V) *V = c->V[layer];
  if (lpos) *lpos = c->lpos;
  return KV_OK;
}

int kv_debug_ring_ptrs(const kv_cache *c, int layer, void **K, void **V) {
  if (!c || layer < 0 || layer >= c->n_layers || !is_hybrid(c->kind[layer])) return KV_ERR_ARG;
  if (K) *K = c->RK[layer];
  if (V) *V = c->RV[layer];
  return KV_OK;
}

int kv_get_config(const kv_cache *c, int *B, int *max_len, int *Hq, int *Hk, int *D, int *W,
                  int *R, int *n_layers) {
  if (!c) return KV_ERR_ARG;
  if (B) *B = c->B;
  if (max_len) *max_len = c->max_len;
  if (Hq) *Hq = c->Hq;
  if (Hk) *Hk = c->Hk;
  if (D) *D = c->D;
  if (W) *W = c->W;
  if (R) *R = c->R;
  if (n_layers) *n_layers = c->n_layers;
  return KV_OK;
}

int kv_device_error(kv_cache *c, int32_t *code_out) {
  if (!c) return KV_ERR_ARG;
  DeviceGuard guard(c->device);
  int32_t v = 0;
  if (cudaMemcpy(&v, c->err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return KV_ERR_CUDA;
  if (cudaMemset(c->err, 0, 4) != cudaSuccess) return KV_ERR_CUDA;
  if (code_out) *code_out = v;
  return v ? KV_ERR_DEVICE : KV_OK;
}

int kv_debug_wait_timeout(kv_cache *c, uint32_t limit, void *stream) {
  if (!c || limit < 1 || limit > (1u << 20)) return KV_ERR_ARG;
  DeviceGuard guard(c->device);
  return set_err(launch_wait_probe(c->err, limit, (cudaStream_t)stream));
}

// ---- host-only schedules (no cache, no CUDA call)

constexpr int kPlanMaxLen = 1 << 20;  // the largest max_len a cache takes

static bool plan_geom_ok(int num_sms, int Hq, int Hk, int D, int R, int kind) {
  if (num_sms < 1 || num_sms > 4096 || Hk < 1 || Hq < Hk || Hq % Hk || Hq / Hk > kMaxRep)
    return false;
  if (D != 64 && D != 128) return false;
  if (kind < KV_GLOBAL || kind > KV_HYBRID_LOCAL) return false;
  return kind == KV_GLOBAL || (R >= 1 && R <= kPlanMaxLen);
}

int kv_plan_decode(int num_sms, int Hq, int Hk, int D, int R, int kind, int n_rows,
                   const int32_t *pos, int32_t *n_splits, int32_t *split_tiles,
                   int32_t *n_splits2, int32_t *split_tiles2, int32_t *part0, int32_t *n_items) {
  if (!plan_geom_ok(num_sms, Hq, Hk, D, R, kind) || n_rows < 0 ||
      n_rows > kMaxRowsPerLaunch || !n_items)
    return KV_ERR_ARG;
  if (n_rows > 0 && (!pos || !n_splits || !split_tiles || !n_splits2 || !split_tiles2 || !part0))
    return KV_ERR_ARG;
  std::vector<DecodeIn> in(n_rows);
  for (int i = 0; i < n_rows; ++i) {
    if (pos[i] < 0 || pos[i] >= kPlanMaxLen) return KV_ERR_ARG;
    in[i] = {i, i, pos[i]};
  }
  const Geom g{num_sms, Hq, Hk, D, kind == KV_GLOBAL ? 0 : R, kind};
  std::unique_ptr<DecodeParams> p(new DecodeParams());
  double bytes = 0, flops = 0;
  plan_decode(g, in, *p, bytes, flops);
  for (int i = 0; i < n_rows; ++i) {
    const DecodeRow &r = p->rows[i];
    n_splits[i] = r.n_splits;
    split_tiles[i] = r.split_tiles;
    n_splits2[i] = r.n_splits2;
    split_tiles2[i] = r.split_tiles2;
    part0[i] = r.n_splits + r.n_splits2 > 1 ? r.part0 : -1;
  }
  *n_items = p->n_items;
  return KV_OK;
}

int kv_plan_prefill(int num_sms, int Hq, int Hk, int D, int R, int kind, int n_rows,
                    const int32_t *lens, const int32_t *n, int capacity, int32_t *entry_row,
                    int32_t *entry_kind, int32_t *tile0, int32_t *tile1, int32_t *part,
                    int32_t *n_entries, int32_t *n_splits, int64_t *part_vecs) {
  if (!plan_geom_ok(num_sms, Hq, Hk, D, R, kind) || n_rows < 0 || capacity < 0 ||
      !n_entries || !part_vecs)
    return KV_ERR_ARG;
  if (n_rows > 0 && (!lens || !n || !n_splits)) return KV_ERR_ARG;
  if (capacity > 0 && (!entry_row || !entry_kind || !tile0 || !tile1 || !part)) return KV_ERR_ARG;
  std::vector<PrefillRow> prows(n_rows);
  for (int i = 0; i < n_rows; ++i) {
    if (lens[i] < 0 || n[i] < 1 || n[i] > kChunk || lens[i] > kPlanMaxLen - n[i])
      return KV_ERR_ARG;
    prows[i] = {i, i, lens[i], n[i], 0, 0, 0, 0};
  }
  const Geom g{num_sms, Hq, Hk, D, kind == KV_GLOBAL ? 0 : R, kind};
  std::vector<PrefillRow> ents[kPrefillKinds];
  std::vector<MergeRow> merges;
  int64_t vecs = 0;
  plan_prefill(g, prows, ents, merges, &vecs);
  int total = 0;
  for (const auto &e : ents) total += (int)e.size();
  *n_entries = total;
  if (total > capacity) return KV_ERR_ARG;
  int j = 0;
  for (int kd = 0; kd < kPrefillKinds; ++kd)
    for (const PrefillRow &r : ents[kd]) {
      entry_row[j] = r.call_row;
      entry_kind[j] = kd;
      tile0[j] = r.tile0;
      tile1[j] = r.tile1;
      part[j] = r.part;
      ++j;
    }
  for (int i = 0; i < n_rows; ++i) n_splits[i] = 1;
  for (const MergeRow &m : merges) n_splits[m.call_row] = m.n_splits;
  *part_vecs = vecs;
  return KV_OK;
}

int kv_profile_enable(kv_cache *c, int enable) {
  if (!c) return KV_ERR_ARG;
  if (!enable) {
    for (auto &r : c->recs) {
      c->free_events.push_back(r.a);
      c->free_events.push_back(r.b);
    }
    c->recs.clear();
  }
  c->prof = enable != 0;
  return KV_OK;
}

int kv_profile_read(kv_cache *c, int kind, int reset, int64_t *launches, double *total_ms,
                    double *alg_bytes, double *alg_flops) {
  if (!c || kind < 0 || kind >= KV_KERNEL_NKINDS) return KV_ERR_ARG;
  DeviceGuard guard(c->device);
  int64_t n = 0;
  double ms = 0, by = 0, fl = 0;
  for (auto &r : c->recs) {
    if (r.kind != kind) continue;
    if (cudaEventSynchronize(r.b) != cudaSuccess) return KV_ERR_CUDA;
    float t = 0;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return KV_ERR_CUDA;
    ++n;
    ms += t;
    by += r.bytes;
    fl += r.flops;
  }
  if (launches) *launches = n;
  if (total_ms) *total_ms = ms;
  if (alg_bytes) *alg_bytes = by;
  if (alg_flops) *alg_flops = fl;
  if (reset) {
    std::vector<ProfRec> keep;
    for (auto &r : c->recs) {
      if (r.kind == kind) {
        c->free_events.push_back(r.a);
        c->free_events.push_back(r.b);
      } else {
        keep.push_back(r);
      }
    }
    c->recs.swap(keep);
  }
  return KV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- decode-step graph
// One decode step of a fixed row set as a CUDA graph: a chain of one decode kernel node
// per layer and, with sliding layers, the ring-state node.  Every launch re-plans the step
// from the host lengths and rewrites the nodes' parameters (and grid sizes) in the
// instantiated graph, so the kernels see exactly what kv_append / kv_advance would pass.
struct kv_step_graph {
  kv_cache *c = nullptr;
  int Bs = 0;
  std::vector<int32_t> rows;  // cache rows
  std::vector<const __nv_bfloat16 *> q, k, v;
  std::vector<const __nv_bfloat16 *> kg, vg;  // hybrid full layers: the group's new global keys
  std::vector<__nv_bfloat16 *> out;
  std::vector<DecodeParams> dps;  // per layer (each ~20 KB: kept on the heap)
  StateParams sp;
  std::vector<cudaGraphNode_t> dec;
  cudaGraphNode_t state = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  double bytes = 0, flops = 0;
};

namespace {

// Parameters of every node for the current lengths (a full row is planned at max_len - 1;
// launches refuse full rows before they get here).
void plan_step(kv_step_graph *g) {
  kv_cache *c = g->c;
  std::vector<DecodeIn> batch(g->Bs);
  for (int i = 0; i < g->Bs; ++i)
    batch[i] = {g->rows[i], i, std::min(c->lens[g->rows[i]], c->max_len - 1)};
  const int64_t q_row = (int64_t)c->Hq * c->D, kv_row = (int64_t)c->Hk * c->D;
  g->bytes = 0;
  g->flops = 0;
  for (int l = 0; l < c->n_layers; ++l) {
    double by = 0, fl = 0;
    if (is_hybrid(c->kind[l]))  // k, v: the layer's local keys; kg, vg: the group's
      fill_decode(c, l, g->q[l], g->kg[l], g->vg[l], g->out[l], q_row, kv_row, batch,
                  g->dps[l], by, fl, g->k[l], g->v[l]);
    else
      fill_decode(c, l, g->q[l], g->k[l], g->v[l], g->out[l], q_row, kv_row, batch, g->dps[l],
                  by, fl);
    // Graph nodes keep the shallow variant: a node's kernel is fixed at instantiation (the
    // deep variant would change it between replays).  Their edges are programmatic (as
    // stream launches are), so a node may stream K/V early when the node before it decodes
    // another storage.
    g->dps[l].deep_pipeline = 0;
    g->dps[l].early_kv =
        c->pdl && l > 0 && storage_id(c, l - 1) != storage_id(c, l) ? 1 : 0;
    g->bytes += by;
    g->flops += fl;
  }
  if (c->lpos) {
    const std::vector<int32_t> ones(g->Bs, 1);
    fill_state(c, g->rows, ones.data(), false, 0, g->rows.size(), g->sp);
  }
}

// Per-layer buffer arrays valid for the cache's layers: every q, k, v, out set and 16-byte
// aligned; kg, vg (may be NULL on a cache without hybrid full layers) set exactly on
// KV_HYBRID_FULL layers.
bool step_buffers_ok(const kv_cache *c, const void *const *q, const void *const *k,
                     const void *const *v, const void *const *kg, const void *const *vg,
                     void *const *outp) {
  if (!q || !k || !v || !outp) return false;
  for (int l = 0; l < c->n_layers; ++l) {
    if (!q[l] || !k[l] || !v[l] || !outp[l] || !aligned16(q[l]) || !aligned16(k[l]) ||
        !aligned16(v[l]) || !aligned16(outp[l]))
      return false;
    const bool full = c->kind[l] == KV_HYBRID_FULL;
    const void *a = kg ? kg[l] : nullptr, *b = vg ? vg[l] : nullptr;
    if (full ? (!a || !b || !aligned16(a) || !aligned16(b)) : (a || b)) return false;
  }
  return true;
}

void set_step_buffers(kv_step_graph *g, const void *const *q, const void *const *k,
                      const void *const *v, const void *const *kg, const void *const *vg,
                      void *const *outp) {
  const int L = g->c->n_layers;
  g->q.assign(L, nullptr);
  g->k.assign(L, nullptr);
  g->v.assign(L, nullptr);
  g->kg.assign(L, nullptr);
  g->vg.assign(L, nullptr);
  g->out.assign(L, nullptr);
  for (int l = 0; l < L; ++l) {
    g->q[l] = (const __nv_bfloat16 *)q[l];
    g->k[l] = (const __nv_bfloat16 *)k[l];
    g->v[l] = (const __nv_bfloat16 *)v[l];
    g->kg[l] = (const __nv_bfloat16 *)(kg ? kg[l] : nullptr);
    g->vg[l] = (const __nv_bfloat16 *)(vg ? vg[l] : nullptr);
    g->out[l] = (__nv_bfloat16 *)outp[l];
  }
}

// Edge from -> to: programmatic (the downstream kernel may start once every CTA of the
// upstream one has let it, and waits for its completion with griddepcontrol.wait) or full.
bool add_edge(cudaGraph_t graph, cudaGraphNode_t from, cudaGraphNode_t to, bool programmatic) {
  cudaGraphEdgeData e{};
  if (programmatic) {
    e.from_port = cudaGraphKernelNodePortProgrammatic;
    e.type = cudaGraphDependencyTypeProgrammatic;
  }
  return cudaGraphAddDependencies(graph, &from, &to, &e, 1) == cudaSuccess;
}

int step_graph_create(kv_cache *c, kv_step_graph **out, const void *const *q,
                      const void *const *k, const void *const *v, const void *const *kg,
                      const void *const *vg, void *const *outp, int Hq, const int32_t *rows,
                      int Bs) {
  if (out) *out = nullptr;
  if (!c || !out || Hq != c->Hq) return KV_ERR_ARG;
  if (Bs < 1 || Bs > c->B || Bs > kMaxRowsPerLaunch) return KV_ERR_ARG;
  std::vector<int32_t> cache_rows;
  std::vector<char> seen(c->B, 0);
  for (int i = 0; i < Bs; ++i) {
    const int r = rows ? rows[i] : i;
    if (r < 0 || r >= c->B || seen[r]) return KV_ERR_ARG;
    seen[r] = 1;
    cache_rows.push_back(r);
  }
  if (!step_buffers_ok(c, q, k, v, kg, vg, outp)) return KV_ERR_ARG;
  DeviceGuard guard(c->device);
  kv_step_graph *g = new kv_step_graph;
  g->c = c;
  g->Bs = Bs;
  g->rows = cache_rows;
  set_step_buffers(g, q, k, v, kg, vg, outp);
  g->dps.resize(c->n_layers);
  plan_step(g);
  const int nt = c->Hq / c->Hk <= 8 ? 1 : 2;
  bool ok = cudaGraphCreate(&g->graph, 0) == cudaSuccess;
  cudaGraphNode_t prev = nullptr;
  for (int l = 0; ok && l < c->n_layers; ++l) {
    void *args[1];
    cudaKernelNodeParams kp{};
    cudaGraphNode_t node = nullptr;
    ok = decode_node(&g->dps[l], c->D, nt, args, &kp) == cudaSuccess &&
         cudaGraphAddKernelNode(&node, g->graph, nullptr, 0, &kp) == cudaSuccess &&
         (!prev || add_edge(g->graph, prev, node, c->pdl));
    g->dec.push_back(node);
    prev = node;
  }
  if (ok && c->lpos) {
    void *args[1];
    cudaKernelNodeParams kp{};
    ok = state_node(&g->sp, args, &kp) == cudaSuccess &&
         cudaGraphAddKernelNode(&g->state, g->graph, nullptr, 0, &kp) == cudaSuccess &&
         add_edge(g->graph, prev, g->state, c->pdl);
  }
  ok = ok && cudaGraphInstantiate(&g->exec, g->graph, 0) == cudaSuccess;
  if (!ok) {
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    delete g;
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  *out = g;
  return KV_OK;
}

void free_step_graph(kv_step_graph *g) {
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
}

}  // namespace

extern "C" {

int kv_step_graph_create(kv_cache *c, kv_step_graph **out, const void *const *q,
                         const void *const *k, const void *const *v, void *const *outp, int Hq,
                         const int32_t *rows, int Bs) {
  if (!c || has_hybrid(c)) {  // kv_step_graph_create_hybrid
    if (out) *out = nullptr;
    return KV_ERR_ARG;
  }
  return step_graph_create(c, out, q, k, v, nullptr, nullptr, outp, Hq, rows, Bs);
}

int kv_step_graph_create_hybrid(kv_cache *c, kv_step_graph **out, const void *const *q,
                                const void *const *k, const void *const *v,
                                const void *const *k_global, const void *const *v_global,
                                void *const *outp, int Hq, const int32_t *rows, int Bs) {
  return step_graph_create(c, out, q, k, v, k_global, v_global, outp, Hq, rows, Bs);
}

int kv_step_graph_set_buffers(kv_step_graph *g, const void *const *q, const void *const *k,
                              const void *const *v, void *const *outp) {
  if (!g || has_hybrid(g->c) || !step_buffers_ok(g->c, q, k, v, nullptr, nullptr, outp))
    return KV_ERR_ARG;
  set_step_buffers(g, q, k, v, nullptr, nullptr, outp);
  return KV_OK;
}

int kv_step_graph_set_buffers_hybrid(kv_step_graph *g, const void *const *q,
                                     const void *const *k, const void *const *v,
                                     const void *const *k_global, const void *const *v_global,
                                     void *const *outp) {
  if (!g || !step_buffers_ok(g->c, q, k, v, k_global, v_global, outp)) return KV_ERR_ARG;
  set_step_buffers(g, q, k, v, k_global, v_global, outp);
  return KV_OK;
}

int kv_step_graph_launch(kv_step_graph *g, void *stream) {
  if (!g) return KV_ERR_ARG;
  kv_cache *c = g->c;
  for (int r : g->rows)
    if ((int64_t)c->lens[r] + 1 > c->max_len) return KV_ERR_FULL;
  DeviceGuard guard(c->device);
  cudaStream_t s = (cudaStream_t)stream;
  if (c->n_blocks > 0) {  // the new position's block, written to the table before the replay
    std::vector<std::pair<int, int>> want;
    for (int r : g->rows) want.push_back({r, c->lens[r] + 1});
    const int rc = ensure_blocks(c, want, s);
    if (rc != KV_OK) return rc;
  }
  plan_step(g);
  const int nt = c->Hq / c->Hk <= 8 ? 1 : 2;
  for (int l = 0; l < c->n_layers; ++l) {
    void *args[1];
    cudaKernelNodeParams kp{};
    if (decode_node(&g->dps[l], c->D, nt, args, &kp) != cudaSuccess ||
        cudaGraphExecKernelNodeSetParams(g->exec, g->dec[l], &kp) != cudaSuccess)
      return KV_ERR_CUDA;
  }
  if (g->state) {
    void *args[1];
    cudaKernelNodeParams kp{};
    if (state_node(&g->sp, args, &kp) != cudaSuccess ||
        cudaGraphExecKernelNodeSetParams(g->exec, g->state, &kp) != cudaSuccess)
      return KV_ERR_CUDA;
  }
  const cudaError_t e = timed(c, KV_KERNEL_STEP, g->bytes, g->flops, s,
                              [&] { return cudaGraphLaunch(g->exec, s); });
  if (e != cudaSuccess) return KV_ERR_CUDA;
  for (int r : g->rows) {
    c->lens[r] += 1;
    for (auto &he : c->hy_end)
      if (!he.empty()) he[r] = c->lens[r];  // the step's layers ran in order
  }
  return KV_OK;
}

void kv_step_graph_destroy(kv_step_graph *g) {
  if (!g) return;
  DeviceGuard guard(g->c->device);
  free_step_graph(g);
}

}  // extern "C"

// ---------------------------------------------------------------- row copies
namespace {

// A storage unit of a row's state: a layer's own storage (a global cache, a sliding ring,
// a hybrid group's cache held by its full layer; a hybrid local layer has none of its own),
// or a hybrid layer's ring.  Units in order: per layer, its storage, then its ring.
struct Unit {
  int layer;
  bool hring;  // the layer's hybrid ring (else its storage K[layer] / V[layer])
  bool ring;   // positions p live at slot p % R
};

std::vector<Unit> units(const kv_cache *c) {
  std::vector<Unit> u;
  for (int l = 0; l < c->n_layers; ++l) {
    if (c->owns[l]) u.push_back({l, false, c->kind[l] == KV_SLIDING});
    if (is_hybrid(c->kind[l])) u.push_back({l, true, true});
  }
  return u;
}

int first_kept(const kv_cache *c, const Unit &u, int keep) {
  return u.ring ? std::max(0, keep - c->R) : 0;
}

// Storage block of (row, unit): K, V and the element stride between heads.
// A paged global layer returns its pool and the row's block-table row instead.
void row_block(const kv_cache *c, const Unit &u, int row, __nv_bfloat16 *&k,
               __nv_bfloat16 *&v, int64_t &head_stride, const int32_t *&table, int32_t &pool) {
  const int layer = u.layer;
  pool = c->n_blocks;
  table = nullptr;
  if (u.hring) {
    const int64_t off = (int64_t)row * c->Hk * (c->R + 1) * c->D;
    k = (__nv_bfloat16 *)c->RK[layer] + off;
    v = (__nv_bfloat16 *)c->RV[layer] + off;
    head_stride = (int64_t)(c->R + 1) * c->D;
    return;
  }
  if (paged_layer(c, layer)) {
    k = (__nv_bfloat16 *)c->K[layer];
    v = (__nv_bfloat16 *)c->V[layer];
    head_stride = 0;
    table = c->table + (int64_t)row * c->max_blocks;
    return;
  }
  const int64_t off = (int64_t)row * c->Hk * c->seg_rows[layer] * c->D;
  k = (__nv_bfloat16 *)c->K[layer] + off;
  v = (__nv_bfloat16 *)c->V[layer] + off;
  head_stride = (int64_t)c->seg_rows[layer] * c->D;
  table = nullptr;
}

// Can the source row, at length `lens`, supply every position a destination of length `keep`
// keeps?  Ring positions older than lens - R are gone from a sliding layer.
bool positions_present(const kv_cache *src, int lens, int keep, int dst_R) {
  if (keep > lens) return false;
  bool ringed = false;  // any ring: sliding or hybrid layers
  for (int k : src->kind) ringed |= k != KV_GLOBAL;
  if (!ringed) return true;
  const int need_lo = std::max(0, keep - dst_R);
  const int have_lo = std::max(0, lens - src->R);
  return need_lo >= have_lo;
}

int flush_copies(CopyParams &cp, cudaStream_t s) {
  const cudaError_t e = launch_copy(cp, s);
  cp.n_items = 0;
  return e == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

// Copy items span at most this many positions: a long row is cut into pieces that run in
// CTAs of their own (both sides address positions absolutely -- slot p, p % R, p - base or
// a block-table entry -- so the pieces are independent).
constexpr int kCopySpan = 2048;

int add_copy(CopyParams &cp, const CopyItem &it, cudaStream_t s) {
  for (int p = it.p0; p < it.p1; p += kCopySpan) {
    CopyItem piece = it;
    piece.p0 = p;
    piece.p1 = std::min(it.p1, p + kCopySpan);
    cp.items[cp.n_items++] = piece;
    if (cp.n_items == kMaxCopyItems) {
      const int rc = flush_copies(cp, s);
      if (rc != KV_OK) return rc;
    }
  }
  return KV_OK;
}

// lpos of rows that now hold [0, keep): reset, then record the kept positions.
int set_ring_state(kv_cache *c, const std::vector<int32_t> &rows, const std::vector<int32_t> &keep,
                   cudaStream_t s) {
  if (!c->lpos || rows.empty()) return KV_OK;
  const std::vector<int32_t> saved = [&] {
    std::vector<int32_t> v;
    for (int r : rows) v.push_back(c->lens[r]);
    return v;
  }();
  int rc = state_update(c, rows, nullptr, true, s);
  for (int r : rows) c->lens[r] = 0;
  if (rc == KV_OK) rc = state_update(c, rows, keep.data(), false, s);
  for (size_t i = 0; i < rows.size(); ++i) c->lens[rows[i]] = saved[i];
  return rc;
}

bool same_layout(const kv_cache *a, const kv_cache *b) {
  return a->Hk == b->Hk && a->D == b->D && a->W == b->W && a->n_layers == b->n_layers &&
         a->kind == b->kind && a->theta == b->theta && a->device == b->device;
}

// Table entry (row, idx) = blk, written on `s` in batches of kMaxTableEntries.
int put_entry(kv_cache *c, TableParams &tp, int row, int idx, int blk, cudaStream_t s) {
  tp.row[tp.n] = row;
  tp.idx[tp.n] = idx;
  tp.blk[tp.n] = blk;
  if (++tp.n < kMaxTableEntries) return KV_OK;
  c->last_stream = s;
  c->last_kind = -1;
  tp.n = 0;
  return launch_table(tp, s) == cudaSuccess ? KV_OK : KV_ERR_CUDA;
}

// Copy item for positions [p0, p1) of one pool block to another (paged unit u): both
// sides addressed as a dense [Hk][16][D] block inside the head-major pool.
CopyItem block_item(const kv_cache *c, const Unit &u, int from, int to, int p0, int p1) {
  CopyItem it;
  const int64_t blk_elems = (int64_t)kBlockTokens * c->D;
  const int64_t hs = (int64_t)c->n_blocks * blk_elems;
  it.src_k = (const __nv_bfloat16 *)c->K[u.layer] + from * blk_elems;
  it.src_v = (const __nv_bfloat16 *)c->V[u.layer] + from * blk_elems;
  it.dst_k = (__nv_bfloat16 *)c->K[u.layer] + to * blk_elems;
  it.dst_v = (__nv_bfloat16 *)c->V[u.layer] + to * blk_elems;
  it.src_head_stride = it.dst_head_stride = hs;
  it.src_table = it.dst_table = nullptr;
  it.src_pool = it.dst_pool = 0;
  it.p0 = p0;
  it.p1 = p1;
  it.src_ring = it.dst_ring = 0;
  it.src_base = it.dst_base = (p0 / kBlockTokens) * kBlockTokens;
  return it;
}

}  // namespace

extern "C" {

int kv_copy_rows(kv_cache *dst, const int32_t *dst_rows, const kv_cache *src,
                 const int32_t *src_rows, const int32_t *keep, int n, void *stream) {
  if (!dst || !src || n < 0 || (n > 0 && (!dst_rows || !src_rows))) return KV_ERR_ARG;
  if (!same_layout(dst, src)) return KV_ERR_ARG;
  std::vector<int32_t> kp(n);
  std::vector<char> dseen(dst->B, 0);
  for (int i = 0; i < n; ++i) {
    const int d = dst_rows[i], r = src_rows[i];
    if (d < 0 || d >= dst->B || r < 0 || r >= src->B || dseen[d]) return KV_ERR_ARG;
    dseen[d] = 1;
    kp[i] = keep ? keep[i] : src->lens[r];
    if (kp[i] < 0 || kp[i] > dst->max_len || !positions_present(src, src->lens[r], kp[i], dst->R))
      return KV_ERR_ARG;
  }
  if (dst == src)  // a row written by one pair must not be read by another
    for (int i = 0; i < n; ++i)
      for (int j = 0; j < n; ++j)
        if (i != j && dst_rows[i] == src_rows[j]) return KV_ERR_ARG;
  if (n == 0) return KV_OK;
  DeviceGuard guard(dst->device);
  cudaStream_t s = (cudaStream_t)stream;
  const bool paged = dst->n_blocks > 0;
  const bool share = paged && dst == src;  // forks inside one paged cache share blocks
  auto in_place = [&](int i) { return dst == src && dst_rows[i] == src_rows[i]; };
  if (paged) {
    // Blocks this call takes against those it frees, all or nothing before anything is
    // enqueued.  Each destination row lets go of its blocks (past keep, when it is cut in
    // place).  A fork inside the cache then holds the source's full blocks of the prefix
    // and takes one block for a partly filled last one; a row cut in place inside a block
    // that other rows hold takes a copy of it; a copy from another cache takes fresh
    // blocks.  (A block a source row holds is never freed here: no source row is another
    // pair's destination.)
    std::unordered_map<int32_t, int32_t> drops;
    int64_t take = 0;
    for (int i = 0; i < n; ++i) {
      const auto &rb = dst->rblocks[dst_rows[i]];
      const int k = kp[i];
      for (size_t x = in_place(i) ? blocks_for(k) : 0; x < rb.size(); ++x) ++drops[rb[x]];
      if (in_place(i))
        take += k % kBlockTokens != 0 && dst->refs[rb[k / kBlockTokens]] > 1;
      else
        take += share ? (k % kBlockTokens != 0) : blocks_for(k);
    }
    int64_t freed = 0;
    for (const auto &e : drops) freed += dst->refs[e.first] == e.second;
    if (take > (int64_t)dst->free_blocks.size() + freed) return KV_ERR_POOL;
  }
  static thread_local CopyParams cp;
  cp.Hk = dst->Hk;
  cp.D = dst->D;
  cp.n_items = 0;
  const std::vector<Unit> us = units(dst);  // the same for src (same layout)
  auto paged_unit = [&](const Unit &u) {
    return paged && !u.hring && paged_layer(dst, u.layer);
  };
  std::vector<CopyItem> block_copies;  // partly filled blocks a row now holds alone
  if (paged) {
    static thread_local TableParams tp;
    tp.table = dst->table;
    tp.max_blocks = dst->max_blocks;
    tp.n = 0;
    int rc = KV_OK;
    for (int i = 0; i < n; ++i) release_blocks(dst, dst_rows[i], in_place(i) ? kp[i] : 0);
    for (int i = 0; i < n && rc == KV_OK; ++i) {
      const int d = dst_rows[i], k = kp[i], last = k / kBlockTokens;
      auto &rb = dst->rblocks[d];
      if (in_place(i)) {
        if (k % kBlockTokens == 0 || dst->refs[rb[last]] == 1) continue;
        const int old = rb[last], nb = take_block(dst);
        drop_block(dst, old);  // still held by another row
        rb[last] = nb;
        for (const Unit &u : us)
          if (paged_unit(u))
            block_copies.push_back(block_item(dst, u, old, nb, last * kBlockTokens, k));
        rc = put_entry(dst, tp, d, last, nb, s);
      } else if (share) {
        const auto &sb = dst->rblocks[src_rows[i]];
        for (int x = 0; x < last && rc == KV_OK; ++x) {
          ++dst->refs[sb[x]];
          rb.push_back(sb[x]);
          rc = put_entry(dst, tp, d, x, sb[x], s);
        }
        if (k % kBlockTokens == 0 || rc != KV_OK) continue;
        const int nb = take_block(dst);
        rb.push_back(nb);
        for (const Unit &u : us)
          if (paged_unit(u))
            block_copies.push_back(block_item(dst, u, sb[last], nb, last * kBlockTokens, k));
        rc = put_entry(dst, tp, d, last, nb, s);
      }
    }
    if (rc == KV_OK && tp.n > 0) {
      dst->last_stream = s;
      dst->last_kind = -1;
      rc = launch_table(tp, s) == cudaSuccess ? KV_OK : KV_ERR_CUDA;
    }
    if (rc != KV_OK) return rc;
  }
  if (!share) {  // fresh destination blocks for [0, keep) (checked above: cannot run out)
    std::vector<std::pair<int, int>> want;
    for (int i = 0; i < n; ++i) want.push_back({dst_rows[i], kp[i]});
    const int rc = ensure_blocks(dst, want, s);
    if (rc != KV_OK) return rc;
  }
  for (const CopyItem &it : block_copies)
    if (add_copy(cp, it, s) != KV_OK) return KV_ERR_CUDA;
  for (int i = 0; i < n; ++i) {
    if (in_place(i)) continue;  // the row keeps its own slots
    for (const Unit &u : us) {
      if (share && paged_unit(u)) continue;  // held, or copied block by block above
      CopyItem it;
      __nv_bfloat16 *sk, *sv;
      row_block(src, u, src_rows[i], sk, sv, it.src_head_stride, it.src_table, it.src_pool);
      it.src_k = sk;
      it.src_v = sv;
      row_block(dst, u, dst_rows[i], it.dst_k, it.dst_v, it.dst_head_stride, it.dst_table,
                it.dst_pool);
      const bool ring = u.ring;
      it.p0 = first_kept(dst, u, kp[i]);
      it.p1 = kp[i];
      it.src_ring = ring ? src->R : 0;
      it.dst_ring = ring ? dst->R : 0;
      it.src_base = it.dst_base = 0;
      if (add_copy(cp, it, s) != KV_OK) return KV_ERR_CUDA;
    }
  }
  if (cp.n_items && flush_copies(cp, s) != KV_OK) return KV_ERR_CUDA;
  dst->last_stream = s;  // the copies wrote the destination's storage
  dst->last_kind = -1;
  dst->cur_layer = -1;
  std::vector<int32_t> rows(dst_rows, dst_rows + n);
  if (set_ring_state(dst, rows, kp, s) != KV_OK) return KV_ERR_CUDA;
  for (int i = 0; i < n; ++i) {
    dst->lens[dst_rows[i]] = kp[i];
    release_blocks(dst, dst_rows[i], kp[i]);  // a shortened row gives its tail back
    for (auto &he : dst->hy_end)
      if (!he.empty()) he[dst_rows[i]] = kp[i];  // no step in progress
  }
  return KV_OK;
}

int64_t kv_export_bytes(const kv_cache *c, int keep) {
  if (!c || keep < 0 || keep > c->max_len) return -1;
  int64_t b = 0;
  for (const Unit &u : units(c)) b += 2LL * c->Hk * (keep - first_kept(c, u, keep)) * c->D * 2;
  return b;
}

// Flat layout, per storage unit in order (a layer's own storage, then a hybrid layer's
// ring): K [Hk][positions][D] then V [Hk][positions][D], positions ascending over the ones
// the unit keeps at length `keep`.
static int export_import(kv_cache *c, int row, int keep, void *buf, int64_t bytes,
                         cudaStream_t s, bool to_buf) {
  __nv_bfloat16 *b = (__nv_bfloat16 *)buf;
  static thread_local CopyParams cp;
  cp.Hk = c->Hk;
  cp.D = c->D;
  cp.n_items = 0;
  int64_t off = 0;
  for (const Unit &u : units(c)) {
    const int p0 = first_kept(c, u, keep), np = keep - p0;
    const int64_t blk = (int64_t)c->Hk * np * c->D;
    __nv_bfloat16 *rk, *rv;
    int64_t hs;
    const int32_t *tab;
    int32_t pool;
    row_block(c, u, row, rk, rv, hs, tab, pool);
    const int ring = u.ring ? c->R : 0;
    CopyItem it;
    it.p0 = p0;
    it.p1 = keep;
    if (to_buf) {
      it.src_k = rk;
      it.src_v = rv;
      it.src_head_stride = hs;
      it.src_table = tab;
      it.src_pool = pool;
      it.src_ring = ring;
      it.src_base = 0;
      it.dst_k = b + off;
      it.dst_v = b + off + blk;
      it.dst_head_stride = (int64_t)np * c->D;
      it.dst_table = nullptr;
      it.dst_pool = 0;
      it.dst_ring = 0;
      it.dst_base = p0;
    } else {
      it.src_k = b + off;
      it.src_v = b + off + blk;
      it.src_head_stride = (int64_t)np * c->D;
      it.src_table = nullptr;
      it.src_pool = 0;
      it.src_ring = 0;
      it.src_base = p0;
      it.dst_k = rk;
      it.dst_v = rv;
      it.dst_head_stride = hs;
      it.dst_table = tab;
      it.dst_pool = pool;
      it.dst_ring = ring;
      it.dst_base = 0;
    }
    off += 2 * blk;
    if (add_copy(cp, it, s) != KV_OK) return KV_ERR_CUDA;
  }
  if (off * 2 != bytes) return KV_ERR_ARG;  // unreachable: checked by the callers
  if (cp.n_items && flush_copies(cp, s) != KV_OK) return KV_ERR_CUDA;
  if (!to_buf) {  // an import wrote the cache's storage
    c->last_stream = s;
    c->last_kind = -1;
    c->cur_layer = -1;
  }
  return KV_OK;
}

int kv_export_row(const kv_cache *c, int row, int keep, void *dst, int64_t bytes, void *stream) {
  if (!c || row < 0 || row >= c->B || !dst || (reinterpret_cast<uintptr_t>(dst) & 15u)) return KV_ERR_ARG;
  if (keep < 0 || !positions_present(c, c->lens[row], keep, c->R)) return KV_ERR_ARG;
  if (bytes != kv_export_bytes(c, keep)) return KV_ERR_ARG;
  DeviceGuard guard(c->device);
  return export_import(const_cast<kv_cache *>(c), row, keep, dst, bytes, (cudaStream_t)stream,
                       true);
}

int kv_import_row(kv_cache *c, int row, int keep, const void *src, int64_t bytes, void *stream) {
  if (!c || row < 0 || row >= c->B || !src || (reinterpret_cast<uintptr_t>(src) & 15u)) return KV_ERR_ARG;
  if (keep < 0 || keep > c->max_len || bytes != kv_export_bytes(c, keep)) return KV_ERR_ARG;
  DeviceGuard guard(c->device);
  cudaStream_t s = (cudaStream_t)stream;
  if (c->n_blocks > 0) {  // the row lets go of its blocks and writes fresh ones of its own
    int64_t avail = (int64_t)c->free_blocks.size();
    for (int b : c->rblocks[row]) avail += c->refs[b] == 1;
    if (blocks_for(keep) > avail) return KV_ERR_POOL;
    release_blocks(c, row, 0);
  }
  int rc = ensure_blocks(c, {{row, keep}}, s);
  if (rc != KV_OK) return rc;
  rc = export_import(c, row, keep, const_cast<void *>(src), bytes, s, false);
  if (rc != KV_OK) return rc;
  if (set_ring_state(c, {row}, {keep}, s) != KV_OK) return KV_ERR_CUDA;
  c->lens[row] = keep;
  release_blocks(c, row, keep);
  for (auto &he : c->hy_end)
    if (!he.empty()) he[row] = keep;
  return KV_OK;
}

const char *kv_strerror(int code) {
  switch (code) {
    case KV_OK: return "KV_OK";
    case KV_ERR_ARG: return "KV_ERR_ARG: invalid argument";
    case KV_ERR_FULL: return "KV_ERR_FULL: KV cache full (lens + n_new > max_len)";
    case KV_ERR_DTYPE: return "KV_ERR_DTYPE: tensors must be bfloat16";
    case KV_ERR_CUDA: return "KV_ERR_CUDA: CUDA runtime error";
    case KV_ERR_OOM: return "KV_ERR_OOM: device allocation failed";
    case KV_ERR_DEVICE: return "KV_ERR_DEVICE: a kernel reported a timed-out wait";
    case KV_ERR_SCRATCH: return "KV_ERR_SCRATCH: request exceeds the fixed no-allocation scratch";
    case KV_ERR_POOL: return "KV_ERR_POOL: no free block in the paged cache's pool";
    default: return "unknown kv status";
  }
}

}  // extern "C"
