// kvinc_internal.h -- structures shared by the host planner (host.cu) and the
// kernels.  Nothing here is part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace kvinc {

// Sub-chunk width: a row's new tokens are processed 64 at a time
// (tiny_agent/generate.py, CHUNK = 64).
constexpr int kChunk = 64;
// Keys per shared-memory tile (one TMA box height).
constexpr int kTileKeys = 64;
// Upper bound of key splits per (row, kv head) in split-K decode.
constexpr int kMaxSplits = 32;
// Row records carried in kernel parameters per launch.
constexpr int kMaxRowsPerLaunch = 512;
// Largest GQA group (query heads per kv head).
constexpr int kMaxRep = 16;
// Spin limit of every mbarrier wait (each try_wait may also suspend briefly);
// reaching it sets the device error word and abandons the work item.
constexpr uint32_t kWaitLimit = 1u << 24;

// Paged global layers: a row's key slots are grouped in blocks of kBlockTokens, found
// through the row's block table (shared by all global layers of the cache: their rows have
// the same lengths).  A layer's pool is head-major, [Hk][n_pool][kBlockTokens][D], so that
// consecutive pool blocks of one head are contiguous.
constexpr int kBlockTokens = 16;
struct PageTable {
  const int32_t *table;  // [B][max_blocks] pool block of each block of a row
  int max_blocks;        // 0: the layer's storage is dense [B][Hk][seg_rows][D]
  int n_pool;            // blocks in the pool
};

// Row of key slot `slot` of (row, kv head g) in the 2-D [rows][D] view of a layer's storage:
// dense (row * Hk + g) * seg_rows + slot; paged (g * n_pool + table[row][slot / 16]) * 16 +
// slot % 16.  A slot past the table (only masked keys) reads the row's last table entry.
__device__ __forceinline__ int64_t kv_row(const PageTable &pt, int row, int Hk, int g,
                                          int seg_rows, int slot) {
  if (pt.max_blocks == 0) return ((int64_t)row * Hk + g) * seg_rows + slot;
  const int idx = min(slot / kBlockTokens, pt.max_blocks - 1);
  const int64_t blk = pt.table[(int64_t)row * pt.max_blocks + idx];
  return ((int64_t)g * pt.n_pool + blk) * kBlockTokens + slot % kBlockTokens;
}

// Storage rows of the four 16-key blocks of the 64-key tile at `slot0` (a multiple of 64) of
// (row, kv head g) in a paged layer, with one 16-byte table load (the table's rows are padded
// to a multiple of 4 entries and every entry holds a valid pool block).
__device__ __forceinline__ int4 kv_rows4(const PageTable &pt, int row, int g, int slot0) {
  const int4 b = *reinterpret_cast<const int4 *>(pt.table + (int64_t)row * pt.max_blocks +
                                                 slot0 / kBlockTokens);
  const int h0 = g * pt.n_pool;
  return make_int4((h0 + b.x) * kBlockTokens, (h0 + b.y) * kBlockTokens,
                   (h0 + b.z) * kBlockTokens, (h0 + b.w) * kBlockTokens);
}
// The tile's four blocks are consecutive in the pool: one 64-row box covers them.
__device__ __forceinline__ bool rows4_contiguous(const int4 &y) {
  return y.y == y.x + kBlockTokens && y.z == y.x + 2 * kBlockTokens &&
         y.w == y.x + 3 * kBlockTokens;
}

enum DestMode : int32_t {
  kDestGlobal = 0,   // cache slot lens + t (pads: scratch slot max_len)
  kDestRing = 1,     // ring slot (lens + t) % R (pads: scratch slot R)
  kDestScratch = 2,  // chunk scratch row t of [B][Hk][64][D]
};

// ---------------------------------------------------------------- append
struct AppendRow {
  int32_t cache_row;
  int32_t call_row;
  int32_t lens;   // position of token t = 0 of this sub-chunk
  int32_t n;      // real tokens in this sub-chunk
  int32_t mode;   // DestMode
  int32_t blk0;   // first token block (8 tokens each) of this row in the grid
};

struct AppendParams {
  const __nv_bfloat16 *k;  // call tensor [Bs][C][Hk][D], already offset to the sub-chunk
  const __nv_bfloat16 *v;
  int64_t kv_row_stride;   // elements between call rows (C*Hk*D)
  __nv_bfloat16 *cache_k;  // layer storage [B][Hk][seg_rows][D]
  __nv_bfloat16 *cache_v;
  __nv_bfloat16 *scr_k;    // chunk scratch [B][Hk][64][D]
  __nv_bfloat16 *scr_v;
  const float2 *rope;      // [max_len][D/2] (cos, sin)
  int Hk, D;
  int seg_rows;            // rows per (row, kv head) of the layer storage
  int ring_R;              // ring slots (sliding) -- scratch slot index R
  int max_len;             // global scratch slot index
  int c_avail;             // tokens per call row present in the tensors from the sub-chunk on
  int n_rows;
  int n_blocks;            // token blocks in the grid
  PageTable pt;            // paged global layer: pads are not written
  AppendRow rows[kMaxRowsPerLaunch];
};

// ---------------------------------------------------------------- decode
// Keys of a decode row: segment 0 (storage slots [0, nk) of the layer storage) and, for a
// hybrid layer, segment 1 (its ring, slots [0, nk2)); each segment has its own splits, and
// the items of segment 1 follow those of segment 0.  All splits merge into one output.
// One decode row, 32 bytes: the parameter block (all rows of a launch) is fetched on every
// launch, so the fields that follow from others (the new key's slots, a ring's length) are
// derived in the kernel and the small ones are 16 or 8 bits wide.
struct DecodeRow {
  int32_t cache_row;
  int32_t pos;          // absolute position of the new token
  int32_t nk;           // segment 0: storage slots [0, nk)
  int32_t ctr;          // row index of this row's merge tickets
  int32_t split_tiles;  // segment 0 tiles (kTileKeys keys) per split
  int32_t split_tiles2; // segment 1 (hybrid ring; keys min(pos + 1, ring_R)) tiles per split
  uint16_t call_row;    // < kMaxRowsPerLaunch
  uint16_t item0;       // first work item of this row (< kMaxRowsPerLaunch * kMaxSplits)
  uint16_t part0;       // first partial slot of this row (items of multi-split rows)
  uint8_t n_splits;     // segment 0 splits
  uint8_t n_splits2;    // segment 1 splits; 0 unless the layer is hybrid
};
static_assert(sizeof(DecodeRow) == 32, "decode row layout");
static_assert(kMaxRowsPerLaunch * kMaxSplits <= 65535, "item and partial indices in 16 bits");

struct DecodeParams {  // 64-byte aligned through its CUtensorMap members
  CUtensorMap tmap_k;       // layer K storage as 2-D [rows][D], box 64 x kTileKeys
  CUtensorMap tmap_v;
  CUtensorMap tmap_k16;     // paged layer: the pool with box 64 x kBlockTokens
  CUtensorMap tmap_v16;
  const __nv_bfloat16 *q;   // [Bs][C][Hq][D] (token 0 of each row is the decode token)
  int64_t q_row_stride;
  __nv_bfloat16 *out;       // [Bs][C][Hq][D]
  int64_t out_row_stride;
  const float2 *rope;
  float *part_o;            // [part][Hq][D] unnormalised partial outputs
  float2 *part_ml;          // [part][Hq] (running max in log2 units, sum of weights)
  int32_t *counters;        // [ctr][Hk] merge tickets, zero between launches
  int32_t *err;
  // fused append of the decode token (fuse_append = 1): its pre-RoPE k and v
  const __nv_bfloat16 *k_new;  // [Bs][C][Hk][D], token 0
  const __nv_bfloat16 *v_new;
  int64_t kv_row_stride;
  __nv_bfloat16 *cache_k;      // layer storage [B][Hk][seg_rows][D]
  __nv_bfloat16 *cache_v;
  int fuse_append;          // the new key goes to segment 0 at slot pos (global) or
  int seg0_ring;            // pos % ring_R (seg0_ring = 1: a sliding layer's ring)
  int ring_R;
  int Hq, Hk, rep, seg_rows;
  int n_rows, n_items;
  int uniform_items;        // > 0: every row has exactly this many items (row = item / it)
  float scale_log2;         // log2(e) / sqrt(D)
  PageTable pt;             // paged global layer (tmap_k16 / tmap_v16 valid)
  // segment 1 of a hybrid layer: the layer's own ring and its new local key
  CUtensorMap tmap_k2;
  CUtensorMap tmap_v2;
  const __nv_bfloat16 *k_new2, *v_new2;
  __nv_bfloat16 *cache_k2, *cache_v2;  // ring storage [B][Hk][seg_rows2][D]
  int seg_rows2;
  int fuse_append2;
  // Programmatic dependent launch: 1 lets the producer stream K/V tiles before the grid
  // dependency wait (the host sets it only when the launch before it on the stream wrote
  // none of the storage this launch reads); every other read and every write of the
  // kernel follows the wait.
  int early_kv;
  // Host only: the launch fits one wave (n_items x Hk <= the SM count), so it runs the
  // variant with twice the K/V stages and one CTA per SM.
  int deep_pipeline;
  DecodeRow rows[kMaxRowsPerLaunch];
};

// ---------------------------------------------------------------- prefill
// One row of a prefill launch, or one key split of it: the CTAs of the entry read the
// 64-key tiles [tile0, tile1) of the row's key space (tile0 even: 128-key blocks; tile1
// beyond the last tile means "to the end").  part < 0: the entry covers all keys and
// writes the output; else it writes unnormalised partials -- vector (kv head g, query row
// rho) at part + g * n * rep + rho of PrefillParams::part_o / part_ml -- for the merge.
struct PrefillRow {
  int32_t cache_row;
  int32_t call_row;
  int32_t lens;   // position of token 0 of the sub-chunk
  int32_t n;      // tokens of the sub-chunk
  int32_t cta0;   // first CTA (query tile) of this entry
  int32_t tile0, tile1;
  int32_t part;
};

struct PrefillParams {  // 64-byte aligned through its CUtensorMap members
  CUtensorMap tmap_k;       // layer storage (global cache or ring), box 64 x kTileKeys
  CUtensorMap tmap_v;
  CUtensorMap tmap_k16;     // paged layer: the pool with box 64 x kBlockTokens
  CUtensorMap tmap_v16;
  CUtensorMap tmap_sk;      // chunk scratch [B*Hk*64][D] (sliding only)
  CUtensorMap tmap_sv;
  const __nv_bfloat16 *q;   // [Bs][C][Hq][D], offset to the sub-chunk
  int64_t q_row_stride;
  __nv_bfloat16 *out;       // offset to the sub-chunk
  int64_t out_row_stride;
  const float2 *rope;
  int32_t *err;
  int Hq, Hk, rep, seg_rows;
  int sliding;              // 0: keys from the global cache; 1: ring + chunk scratch
  int ring_R, window;
  int n_rows, n_ctas;
  float scale_log2;
  PageTable pt;             // paged global layer (tmap_k16 / tmap_v16 valid)
  // hybrid layer: keys = the group's cache (tmap_k/v) + the layer's ring (tmap_k2/v2,
  // seg_rows2 rows per (row, kv head)) + the chunk scratch
  int hybrid;
  CUtensorMap tmap_k2;
  CUtensorMap tmap_v2;
  int seg_rows2;
  // key splits: [vector][D] fp32 O (relative to m), [vector] (m in log2 units, l)
  float *part_o;
  float2 *part_ml;
  PrefillRow rows[kMaxRowsPerLaunch];
};

// Merge of a prefill row's key splits: out = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s
// (M = max_s m_s) for every (kv head, query row) vector; split s of the row starts at
// part + s * Hk * n_rho.
// At most this many key splits per prefill row (the merge holds all of a row's partials of
// one vector in registers).
constexpr int kMaxPrefillSplits = 16;

struct MergeRow {
  int32_t call_row;
  int32_t n_rho;     // query rows per kv head (tokens x GQA group)
  int32_t n_splits;
  int32_t part;
  int32_t vec0;      // first vector of this row in the launch
};

struct MergeParams {
  const float *part_o;
  const float2 *part_ml;
  __nv_bfloat16 *out;       // offset to the sub-chunk
  int64_t out_row_stride;
  int Hq, Hk, rep;
  int n_rows, n_vec;
  MergeRow rows[kMaxRowsPerLaunch];
};

// ---------------------------------------------------------------- ring commit / state
struct CommitParams {
  const __nv_bfloat16 *scr_k, *scr_v;
  __nv_bfloat16 *ring_k, *ring_v;
  int Hk, D, ring_R, window, seg_rows;
  int n_rows;
  int32_t cache_row[kMaxRowsPerLaunch];
  int32_t lens[kMaxRowsPerLaunch];
  int32_t n[kMaxRowsPerLaunch];
};

struct StateParams {
  int32_t *lpos;       // [B][R]
  int ring_R, window;
  int reset;           // 1: lpos = -1; 0: record the kept positions of the advance
  int n_rows;
  int32_t cache_row[kMaxRowsPerLaunch];
  int32_t lens[kMaxRowsPerLaunch];   // lens before the advance
  int32_t n[kMaxRowsPerLaunch];
};

// ---------------------------------------------------------------- position copies
// One (row, layer) block of K/V positions [p0, p1) copied from one storage to another.
// A storage is [Hk][slots][D] per (row, layer) at `k`/`v` with `head_stride` elements
// between heads; position p sits at slot p % ring (ring > 0) or p - base (ring == 0).
// A paged side (table != nullptr: the row's block-table row) has `k`/`v` at its pool's
// start and position p of head h at pool row (h * n_pool + table[p / 16]) * 16 + p % 16.
struct CopyItem {
  const __nv_bfloat16 *src_k, *src_v;
  __nv_bfloat16 *dst_k, *dst_v;
  int64_t src_head_stride, dst_head_stride;
  const int32_t *src_table, *dst_table;
  int32_t src_pool, dst_pool;  // pool blocks of a paged side
  int32_t p0, p1;
  int32_t src_ring, src_base, dst_ring, dst_base;
};
constexpr int kMaxCopyItems = 256;
struct CopyParams {
  int Hk, D;
  int n_items;
  CopyItem items[kMaxCopyItems];
};

// ---------------------------------------------------------------- block tables
constexpr int kMaxTableEntries = 2048;
struct TableParams {
  int32_t *table;  // [B][max_blocks]
  int max_blocks;
  int n;
  int32_t row[kMaxTableEntries], idx[kMaxTableEntries], blk[kMaxTableEntries];
};

// ---------------------------------------------------------------- launchers
// Launch kernel(p) on s.  With pdl, as a programmatic dependent launch: the grid may start
// while the previous kernel on the stream finishes, and waits for it (griddepcontrol.wait)
// before it touches global memory; every kernel of the library does so at its start and
// only then lets its own successor start, so that when a grid starts, every grid before
// its predecessor has completed.
template <typename P>
cudaError_t launch_k(void (*kernel)(P), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     const P &p, bool pdl) {
  if (!pdl) {
    kernel<<<grid, block, smem, s>>>(p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_copy(const CopyParams &p, cudaStream_t s);
cudaError_t launch_table(const TableParams &p, cudaStream_t s);
// Split-K schedule of one decode launch over p.rows[0, n) (n <= kMaxRowsPerLaunch), whose
// cache_row, call_row, pos, nk and ctr the caller has set: row i reads nk slots of segment
// 0 and nk2[i] slots of segment 1 (0: none).  Sets each row's splits, tiles per split,
// first item and first partial slot, and p.n_rows, p.n_items, p.uniform_items, aiming at
// about four waves of two CTAs per SM over Hk kv heads; returns the partial slots used.
// When that schedule would use more than max_parts partial slots the splits are made
// longer (down to one per segment) until it does not; only rows with two segments (a
// hybrid layer) then still use slots, two each.
int plan_decode_splits(int num_sms, int Hk, int n, const int *nk2, DecodeParams &p,
                       int max_parts);
cudaError_t launch_append(const AppendParams &p, cudaStream_t s, bool pdl = false);
// pdl: launch with programmatic stream serialisation, so that the kernel may start while
// the previous kernel on the stream finishes (see DecodeParams::early_kv).
cudaError_t launch_decode(const DecodeParams &p, int D, int n_tiles_heads, cudaStream_t s,
                          bool pdl = false);
// Graph kernel-node descriptions of the decode and state launches (args: one-slot storage
// that must outlive the call that consumes *kp).
cudaError_t decode_node(const DecodeParams *p, int D, int n_tiles_heads, void **args,
                        cudaKernelNodeParams *kp);
cudaError_t state_node(const StateParams *p, void **args, cudaKernelNodeParams *kp);
cudaError_t launch_prefill(const PrefillParams &p, int D, cudaStream_t s, bool pdl = false);
cudaError_t launch_prefill_merge(const MergeParams &p, int D, cudaStream_t s, bool pdl = false);
cudaError_t launch_commit(const CommitParams &p, cudaStream_t s, bool pdl = false);
cudaError_t launch_state(const StateParams &p, cudaStream_t s, bool pdl = false);
cudaError_t launch_wait_probe(int32_t *err, uint32_t limit, cudaStream_t s);
// Opt kernels into their dynamic shared memory sizes (once per process and device).
cudaError_t configure_kernels();

// Kernel parameters are passed by value: at most 32764 bytes per launch.
constexpr size_t kMaxParamBytes = 32764;
static_assert(sizeof(DecodeParams) <= kMaxParamBytes, "decode parameters too large");
static_assert(sizeof(PrefillParams) <= kMaxParamBytes, "prefill parameters too large");
static_assert(sizeof(AppendParams) <= kMaxParamBytes, "append parameters too large");
static_assert(sizeof(CommitParams) <= kMaxParamBytes, "commit parameters too large");
static_assert(sizeof(CopyParams) <= kMaxParamBytes, "copy parameters too large");
static_assert(sizeof(TableParams) <= kMaxParamBytes, "table parameters too large");
static_assert(sizeof(StateParams) <= kMaxParamBytes, "state parameters too large");
static_assert(sizeof(MergeParams) <= kMaxParamBytes, "merge parameters too large");

}  // namespace kvinc
