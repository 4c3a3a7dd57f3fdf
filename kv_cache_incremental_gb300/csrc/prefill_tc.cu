// prefill_tc.cu -- chunked prefill on the 5th-generation tensor cores (tcgen05, TMEM).
//
// What is computed is the same as prefill.cu: query row rho of a (row, kv head) is
// token t = rho / rep, head h = rho % rep of the GQA group at absolute position
// p = lens + t; it attends to the visible keys of the layer storage (global: slots
// [0, lens + t], sliding: the ring's occupied slots, whose positions follow from
// lens) and of the chunk scratch (sliding layers), reading the ring before this
// chunk is committed to it ("inkling: ring-buffer KV cache for sliding-window
// layers", How it works; Lab 07 section 3; tiny_agent/generate.py `_append_chunk`).
// A hybrid layer's keys are three segments in one softmax: its group's global cache,
// its own ring, the chunk's local keys.  A launch entry may cover a range of the key
// tiles only (a key split): it then writes its unnormalised partials for the merge
// instead of the output.
//
// One CTA owns one or two 128-row query tiles (the MMA's M) of one (row, kv head): two
// at D = 128, sharing every K/V block the CTA streams; one at D = 64, two CTAs per SM.
// A block is 128 keys: two 64-key tiles, each a TMA box, a unit of the masking logic and
// one half of the softmax pass.
// Warp roles (with two tiles; with one, warps 0-3, 4 and 5):
//   warps 0-7  softmax, four per query tile: thread i of a tile owns query row i =
//              TMEM lane i of that tile's accumulators.  They rotate the queries into
//              shared memory (while the producer already streams K/V), read S from TMEM,
//              mask it through a 64-bit visibility mask per 64-key tile, run the online
//              softmax (lazy rescaling: O in TMEM is rescaled only when a row's maximum
//              grows by more than 2^8), write P as bf16 high and low parts back into the
//              TMEM columns that held S (with one tile, the second 64-key tile's P into
//              the spare columns), and finally read O from TMEM and normalise.  With one
//              tile, a warp none of whose rows is a query row only keeps the barriers.
//   warp 8     TMA producer of the K and V blocks (128-byte swizzle).
//   warps 9-10 MMA issuers, one thread per query tile (warp 9 also owns TMEM).  Per
//              block: S = Q K^T (M=128, N=128) into the tile's S buffer, then, once the
//              softmax wrote P of each 64-key tile, O += P_hi V + P_lo V (M=128, N=D)
//              with P read from TMEM and V read in place as an MN-major operand (keys are
//              its K).  tcgen05.mma operations are ordered only among those with the same
//              accumulator and shape, so QK(b+1), which overwrites the P that PV(b) reads,
//              waits for that PV to finish: for all of it with two tiles, for PV of the
//              first 64-key tile with one (the second tile's P sits in the spare columns),
//              once the softmax has read S of the second tile.  The two query tiles'
//              chains run independently.  A two-tile CTA with a single query tile in use
//              double-buffers S in the other tile's columns, so QK(b+1) (after PV(b - 1))
//              runs during the softmax of block b.
// Every mbarrier wait is bounded; on a timeout the CTA records the error, lets its
// own TMA loads and MMAs finish (bounded), frees its TMEM and returns.
#include "kvinc_internal.h"
#include "ptx.cuh"

namespace kvinc {
namespace {

constexpr int kRows = 128;        // query rows per tile (MMA M)
constexpr int kKeys = kTileKeys;  // keys per tile (one TMA box, one softmax half)
constexpr int kBlockKeys = 2 * kKeys;  // keys per K/V block (MMA N of S, K of PV)
constexpr int kSoftmaxWarps = 4;  // per query tile
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (log2 units)

// Warp roles of a CTA with TQ query tiles: softmax warps, then the producer, then one
// MMA-issuing warp per tile.
template <int TQ>
struct Roles {
  static constexpr int kProducerWarp = TQ * kSoftmaxWarps, kMmaWarp = kProducerWarp + 1;
  static constexpr int kThreads = (kMmaWarp + TQ) * 32;
};

// TQ = 2 (D = 128): two query tiles share every K/V block (one CTA per SM).  TQ = 1
// (D = 64): one tile in 256 TMEM columns and two K/V stages, so that two CTAs fit on an SM.
template <int D, int TQ>
struct TcCfg {
  static constexpr int kTilesQ = TQ;
  static constexpr int kPanels = D / 64;
  static constexpr int kStages = D == 128 ? 2 : TQ == 2 ? 4 : 2;
  static constexpr int kQBytes = kPanels * kRows * 128;        // one Q tile, K-major, 128B swizzle
  static constexpr int kPanelBytes = kBlockKeys * 128;         // 64 dims of one K or V block
  static constexpr int kHalfBytes = kKeys * 128;               // one 64-key TMA box of a panel
  static constexpr int kKVBlock = kPanels * kPanelBytes;       // one K or V block
  static constexpr int kStageBytes = 2 * kKVBlock;             // [K panels][V panels]
  // TMEM: per query tile one 128-column S buffer (S fp32 of the block's two 64-key tiles;
  // then per tile P as 32 columns of bf16 pairs for the high part and 32 for the low
  // part, in the columns that held that tile's S) and one D-column O accumulator.
  static constexpr int kTmemCols = TQ == 2 ? 512 : 256;        // [S0 S1] [O0] [O1] or [S0] [O0]
  // With one query tile the columns left after [S0][O0] (64 at D = 64) hold P of the
  // block's second 64-key tile, so that QK of the next block, which overwrites S0, waits
  // only for the PV of the first tile's P and for the softmax to have read the second
  // tile's S.
  static constexpr bool kSpareP1 = TQ == 1 && kBlockKeys + D + kKeys <= kTmemCols;
  static constexpr int kColP1 = kBlockKeys + D;
  static constexpr int kOff_Q = 0;
  static constexpr int kOff_KV = kOff_Q + kTilesQ * kQBytes;
  static constexpr int kOff_Bar = kOff_KV + kStages * kStageBytes;
  static constexpr int kBars = 3 * kStages + kTilesQ * 7 + 1;
  static constexpr int kSmem = 1024 + kOff_Bar + kBars * 8 + 32;
  static_assert(kSmem <= 232448, "shared memory per CTA");
  static_assert(kTilesQ * kBlockKeys + kTilesQ * D <= kTmemCols, "TMEM columns");
};

__device__ __forceinline__ int find_cta_row(const PrefillParams &p, int b) {
  int lo = 0, hi = p.n_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.rows[mid].cta0 <= b) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Visible key indices of one query row within a key segment, as two inclusive ranges
// (an empty range has lo > hi).  mode 0, a global cache (which holds this chunk too): slots
// 0..p.  mode 1, a ring: slot s holds position s + base (s <= rem) or s + base - R
// (s > rem), or just s while lens <= R; it is visible iff that position is >= p - W + 1.
// mode 2, the chunk scratch: token j sits at lens + j and is visible iff
// p - W + 1 <= lens + j <= p.
enum SegMode { kSegGlobal = 0, kSegRing = 1, kSegScratch = 2 };
__device__ __forceinline__ void row_ranges(int mode, bool qvalid, int qpos, int lens,
                                           const PrefillParams &p, int (&rg)[4]) {
  rg[0] = 1; rg[1] = 0; rg[2] = 1; rg[3] = 0;
  if (!qvalid) return;
  if (mode == kSegGlobal) {
    rg[0] = 0;
    rg[1] = qpos;
    return;
  }
  const int thr = qpos - p.window + 1;  // first visible position
  if (mode == kSegScratch) {
    rg[0] = max(0, thr - lens);
    rg[1] = qpos - lens;
    return;
  }
  const int R = p.ring_R;
  if (lens <= R) {
    rg[0] = max(0, thr);
    rg[1] = lens - 1;
    return;
  }
  const int base = ((lens - 1) / R) * R, rem = (lens - 1) % R;
  rg[0] = max(0, thr - base);
  rg[1] = rem;
  rg[2] = max(rem + 1, thr - base + R);
  rg[3] = R - 1;
}

// 2^x with the hardware approximation (relative error ~2^-22), denormals flushed.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Maximum of 64 values: eight running three-input maxima, then a short tree (36
// instructions, eight temporaries).
__device__ __forceinline__ float max64(const float (&v)[64]) {
  float a[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = fmax3(v[k], v[8 + k], v[16 + k]);
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = fmax3(a[k], v[24 + k], v[32 + k]);
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = fmax3(a[k], v[40 + k], v[48 + k]);
#pragma unroll
  for (int k = 0; k < 8; ++k) a[k] = fmaxf(a[k], v[56 + k]);
  return fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

template <int D, int TQ>
__global__ void __launch_bounds__(Roles<TQ>::kThreads, TQ == 1 ? 2 : 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using Cfg = TcCfg<D, TQ>;
  constexpr int kTilesQ = TQ;
  constexpr int kProducerWarp = Roles<TQ>::kProducerWarp, kMmaWarp = Roles<TQ>::kMmaWarp;
  constexpr int kStages = Cfg::kStages;
  constexpr int kHalf = D / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *qsm = smem + Cfg::kOff_Q;     // Q tile qt at qt * kQBytes
  uint8_t *kv = smem + Cfg::kOff_KV;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Cfg::kOff_Bar);
  uint64_t *kv_full = bars;                       // [kStages] TMA -> MMA and softmax
  uint64_t *kv_empty = kv_full + kStages;         // [kStages] every MMA of the stage done
  // Per query tile, one phase per K/V block.  Every barrier's phases are waited for in
  // block order, and no phase can complete before its predecessor has been waited for,
  // so no parity wait is ever two phases ahead or behind (the argument is given at each
  // wait whose predecessor is not waited for by the same thread).
  // With one query tile, S buffer i (i = block parity) uses s_full[i] and p_full[2i + h].
  uint64_t *s_full = kv_empty + kStages;          // [tile] QK done -> softmax
  uint64_t *p_full = s_full + kTilesQ;            // [tile][half] softmax wrote P -> MMA
  uint64_t *pv0_done = p_full + 2 * kTilesQ;      // [tile] PV of half 0 done -> softmax
  uint64_t *pv_done = pv0_done + kTilesQ;         // [tile] PV done -> MMA, softmax
  uint64_t *v_ready = pv_done + kTilesQ;          // [stage] tile 0 zeroed V -> MMA of tile 1
  uint64_t *drain = v_ready + kStages;            // [1] every MMA done (teardown)
  uint64_t *s1_read = drain + 1;                  // [tile] softmax read S of tile 1 -> MMA
  uint64_t *q_ready = s1_read + kTilesQ;          // [tile] rotated Q tile stored -> MMA
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::kBars);
  volatile int *fail = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *issued = fail + 1;

  ptx::grid_dep_wait();  // the previous grid on the stream has completed
  ptx::grid_dep_launch();
  const PrefillRow &row = p.rows[find_cta_row(p, blockIdx.x)];
  const int g = blockIdx.y;
  const int rho0 = (blockIdx.x - row.cta0) * kRows * kTilesQ;
  const int n_rho = row.n * p.rep;
  const int n_qt = min(kTilesQ, (n_rho - rho0 + kRows - 1) / kRows);  // query tiles in use
  const int rho_last = min(n_rho, rho0 + kRows * kTilesQ) - 1;
  // one query tile in use in a two-tile CTA: S double-buffered in the other tile's columns
  const bool dbl = kTilesQ == 2 && n_qt == 1;
  const int t_max = rho_last / p.rep;
  const int lens = row.lens;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Key segments: 0 the layer storage (a global cache: slots [0, lens + t_max]; a sliding
  // layer: its ring), 1 a hybrid layer's own ring (after its group's cache), 2 the chunk
  // scratch (sliding and hybrid layers).  Tiles of segment s start at tile seg_t0[s].
  // (scalars, not arrays: a runtime index would put them in local memory)
  const int sl0 = p.sliding && !p.hybrid ? min(lens, p.ring_R) : lens + t_max + 1;
  const int sl1 = p.hybrid ? min(lens, p.ring_R) : 0;
  const int sl2 = p.sliding || p.hybrid ? t_max + 1 : 0;
  const int st1 = (sl0 + kKeys - 1) / kKeys, st2 = st1 + (sl1 + kKeys - 1) / kKeys;
  const int n_tiles = st2 + (sl2 + kKeys - 1) / kKeys;  // 64-key tiles
  const int seg0_mode = p.sliding && !p.hybrid ? kSegRing : kSegGlobal;
  auto seg_of = [&](int j) { return j < st1 ? 0 : j < st2 ? 1 : 2; };
  auto seg_len = [&](int sg) { return sg == 0 ? sl0 : sg == 1 ? sl1 : sl2; };
  auto seg_t0 = [&](int sg) { return sg == 0 ? 0 : sg == 1 ? st1 : st2; };
  // This entry's tiles [j_begin, j_end) (a key split, or all of them): blocks
  // b_begin .. b_begin + n_blocks - 1 of 128 keys; loop indices below count from b_begin.
  const int j_begin = row.tile0, j_end = min(row.tile1, n_tiles);
  const int b_begin = j_begin / 2;
  const int n_blocks = j_end > j_begin ? (j_end - j_begin + 1) / 2 : 0;
  const int64_t rh = (int64_t)row.cache_row * p.Hk + g;
  auto seg_base = [&](int sg) {
    return rh * (sg == 0 ? p.seg_rows : sg == 1 ? p.seg_rows2 : kChunk);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&kv_full[s], 1);
      ptx::mbar_init(&kv_empty[s], n_qt);  // one commit per query tile's MMA warp
    }
    for (int qt = 0; qt < kTilesQ; ++qt) {
      ptx::mbar_init(&s_full[qt], 1);
      ptx::mbar_init(&p_full[2 * qt], kSoftmaxWarps);
      ptx::mbar_init(&p_full[2 * qt + 1], kSoftmaxWarps);
      ptx::mbar_init(&pv0_done[qt], 1);
      ptx::mbar_init(&pv_done[qt], 1);
      ptx::mbar_init(&s1_read[qt], kSoftmaxWarps);
      ptx::mbar_init(&q_ready[qt], kSoftmaxWarps);
    }
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(&v_ready[s], kSoftmaxWarps);
    ptx::mbar_init(drain, n_qt);
    *fail = 0;
    *issued = 0;
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) tc::alloc(tmem_slot, Cfg::kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;
  const int qt_me = warp / kSoftmaxWarps;  // query tile of a softmax warp

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&p.tmap_k);
      ptx::prefetch_tmap(&p.tmap_v);
      for (int it = 0; it < n_blocks && !*fail; ++it) {
        const int s = it % kStages;
        if (it >= kStages &&
            !ptx::mbar_wait(&kv_empty[s], ((it / kStages) - 1) & 1, kWaitLimit)) {
          atomicExch(p.err, 1);
          *fail = 1;
          break;
        }
        uint8_t *kt = kv + s * Cfg::kStageBytes;
        uint8_t *vt = kt + Cfg::kKVBlock;
        const int halves = min(2, j_end - 2 * (b_begin + it));  // a last block may hold one tile
        ptx::mbar_arrive_expect_tx(&kv_full[s], halves * 2 * Cfg::kPanels * Cfg::kHalfBytes);
        for (int h = 0; h < halves; ++h) {
          const int j = 2 * (b_begin + it) + h;
          const int sg = seg_of(j);
          const CUtensorMap *mk = sg == 0 ? &p.tmap_k : sg == 1 ? &p.tmap_k2 : &p.tmap_sk;
          const CUtensorMap *mv = sg == 0 ? &p.tmap_v : sg == 1 ? &p.tmap_v2 : &p.tmap_sv;
          const bool in_a = sg == 0;
          const int y = static_cast<int>(seg_base(sg) + (int64_t)(j - seg_t0(sg)) * kKeys);
          int4 y4 = make_int4(y, y + kBlockTokens, y + 2 * kBlockTokens, y + 3 * kBlockTokens);
          if (in_a && p.pt.max_blocks) y4 = kv_rows4(p.pt, row.cache_row, g, j * kKeys);
          if (rows4_contiguous(y4)) {  // dense, or a paged tile of consecutive blocks
#pragma unroll
            for (int pn = 0; pn < Cfg::kPanels; ++pn) {
              const int off = pn * Cfg::kPanelBytes + h * Cfg::kHalfBytes;
              ptx::tma_load_2d(kt + off, mk, pn * 64, y4.x, &kv_full[s]);
              ptx::tma_load_2d(vt + off, mv, pn * 64, y4.x, &kv_full[s]);
            }
          } else {  // paged: four 16-key blocks, 16-row boxes
            const int ys[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
            for (int q4 = 0; q4 < kKeys / kBlockTokens; ++q4)
#pragma unroll
              for (int pn = 0; pn < Cfg::kPanels; ++pn) {
                const int off =
                    pn * Cfg::kPanelBytes + h * Cfg::kHalfBytes + q4 * kBlockTokens * 128;
                ptx::tma_load_2d(kt + off, &p.tmap_k16, pn * 64, ys[q4], &kv_full[s]);
                ptx::tma_load_2d(vt + off, &p.tmap_v16, pn * 64, ys[q4], &kv_full[s]);
              }
          }
        }
        *issued = it + 1;
      }
    }
  } else if (warp >= kMmaWarp) {
    // ------------------------------------------------------------ MMA issuers
    // One warp per query tile, so each tile's chain QK -> softmax -> PV -> QK runs at its
    // own pace and the tensor pipe interleaves the two.  A K/V stage is released when
    // both have committed their PV of it.
    const int qt = warp - kMmaWarp;
    if (lane == 0 && qt < n_qt) {
      constexpr uint32_t kIdQK = tc::idesc_bf16_f32(kRows, kBlockKeys);
      constexpr uint32_t kIdPV = tc::idesc_bf16_f32(kRows, D, /*b_mn_major=*/true);
      const uint32_t q_addr = ptx::smem_u32(qsm + qt * Cfg::kQBytes);
      const uint32_t tO = tmem + kTilesQ * kBlockKeys + qt * D;
      // S buffer of block b, its barriers' index and phase: this tile's own, or with one
      // query tile, buffer b & 1 (phase b >> 1).
      auto sbuf = [&](int b) { return dbl ? (b & 1) : qt; };
      auto sphase = [&](int b) -> uint32_t { return dbl ? (b >> 1) & 1 : b & 1; };
      // QK(b): S of block b into its S buffer, once the K/V stage has landed.  The caller
      // has waited for the PV that last read P out of that buffer: tcgen05.mma operations
      // are ordered only among those with the same accumulator and shape, so a QK issued
      // behind a PV could overwrite P before the PV has read it.  A block with one tile
      // still multiplies all 128 rows of its K stage; the softmax masks the absent half.
      auto issue_qk = [&](int b) -> bool {
        if (!ptx::mbar_wait(&kv_full[b % kStages], (b / kStages) & 1, kWaitLimit)) return false;
        tc::fence_after();
        const uint32_t tS = tmem + sbuf(b) * kBlockKeys;
        const uint32_t k_addr = ptx::smem_u32(kv + (b % kStages) * Cfg::kStageBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off_q = (kk / 4) * (kRows * 128) + 32 * (kk % 4);
          const uint32_t off_k = (kk / 4) * Cfg::kPanelBytes + 32 * (kk % 4);
          tc::mma(tS, tc::desc_sw128(q_addr + off_q), tc::desc_sw128(k_addr + off_k), kIdQK,
                  kk > 0);
        }
        tc::commit(&s_full[sbuf(b)]);
        return true;
      };
      // A tile of the block is partial when a segment ends inside it.
      auto partial = [&](int j) {
        if (j >= j_end) return false;
        const int sg = seg_of(j);
        const int next = sg == 0 ? st1 : sg == 1 ? st2 : n_tiles;
        return j == next - 1 && seg_len(sg) % kKeys != 0;
      };
      // PV(b): O += P V over the block's tiles.  B = V as stored by TMA: rows = keys (K),
      // 64-dim panels (MN) kPanelBytes apart; A = P of tile h in S-buffer columns
      // 64h + [0, 32) (high part) and 64h + [32, 64) (low part), 16 keys = 8 columns (tile
      // 1 in the spare columns kColP1 + [0, 64) when there are any).
      // The softmax publishes P per tile, so PV of tile 0 runs while it computes tile 1.
      // With the spare columns, QK(b + 1) is issued between the block's two PVs, once the
      // softmax has read tile 1's S and PV of tile 0 has finished, so that it runs while
      // the softmax computes tile 1.
      // Query tile 1 reads V of a partial block only after tile 0's softmax zeroed the
      // rows past the segment's end (v_ready, one barrier per stage: tile 0 cannot get
      // kStages blocks ahead of this PV, whose stage it would need, so it cannot lap it).
      auto issue_pv = [&](int b) -> bool {
        const int jb = 2 * (b_begin + b);
        if (qt == 1 && (partial(jb) || partial(jb + 1)) &&
            !ptx::mbar_wait(&v_ready[b % kStages], (b / kStages) & 1, kWaitLimit))
          return false;
        const uint32_t v_addr =
            ptx::smem_u32(kv + (b % kStages) * Cfg::kStageBytes + Cfg::kKVBlock);
        const int halves = min(2, j_end - jb);
        const uint32_t tS = tmem + sbuf(b) * kBlockKeys;
        for (int h = 0; h < halves; ++h) {
          if (!ptx::mbar_wait(&p_full[2 * sbuf(b) + h], sphase(b), kWaitLimit)) return false;
          tc::fence_after();
          const uint32_t tP = Cfg::kSpareP1 && h == 1 ? tmem + Cfg::kColP1 : tS + kKeys * h;
#pragma unroll
          for (int ks = 0; ks < kKeys / 16; ++ks) {
            const uint64_t bd = tc::desc_sw128_mn(v_addr + h * Cfg::kHalfBytes + ks * 16 * 128,
                                                  Cfg::kPanelBytes, 1024);
            tc::mma_ts(tO, tP + 8 * ks, bd, kIdPV, b > 0 || h > 0 || ks > 0);
            tc::mma_ts(tO, tP + kKeys / 2 + 8 * ks, bd, kIdPV, true);
          }
          if (h == 0) {
            tc::commit(&pv0_done[qt]);
            // (s1_read and pv0_done: this thread waited for phase b - 1 of each in block
            // b - 1, which had two tiles since block b follows it)
            if (Cfg::kSpareP1 && halves == 2 && b + 1 < n_blocks &&
                !(ptx::mbar_wait(&s1_read[qt], b & 1, kWaitLimit) &&
                  ptx::mbar_wait(&pv0_done[qt], b & 1, kWaitLimit) && issue_qk(b + 1)))
              return false;
          }
        }
        tc::commit(&pv_done[qt]);
        tc::commit(&kv_empty[b % kStages]);  // this tile's MMAs of the stage issued
        return true;
      };
      if (n_blocks > 0) {  // (a key split past this CTA's last tile has no work)
        // Double-buffered, QK(b + 1) goes into the buffer PV(b - 1) read, once that has
        // finished, and is issued before PV(b) waits for the softmax of block b, so it
        // overlaps that.  Otherwise QK(b + 1) waits for PV(b), or, with the spare columns,
        // is issued inside PV(b).
        bool ok = ptx::mbar_wait(&q_ready[qt], 0, kWaitLimit) && issue_qk(0);
        for (int b = 0; ok && b < n_blocks; ++b) {
          if (*fail) {
            ok = false;
            break;
          }
          if (dbl)
            ok = (b + 1 >= n_blocks ||
                  ((b < 1 || ptx::mbar_wait(&pv_done[qt], (b - 1) & 1, kWaitLimit)) &&
                   issue_qk(b + 1))) &&
                 issue_pv(b);
          else if (Cfg::kSpareP1)
            ok = issue_pv(b);
          else
            ok = issue_pv(b) &&
                 (b + 1 >= n_blocks ||
                  (ptx::mbar_wait(&pv_done[qt], b & 1, kWaitLimit) && issue_qk(b + 1)));
        }
        if (!ok) {
          atomicExch(p.err, 1);
          *fail = 1;
        }
        // Every MMA issued by either warp has completed before TMEM can be released.
        tc::commit(drain);
        ptx::mbar_wait(drain, 0, kWaitLimit);
      }
    }
  } else if (qt_me < n_qt) {
    // ------------------------------------------------------------ softmax warps
    {  // Rotated query of this thread's row into its tile's 128-byte-swizzled Q tile,
       // while the producer already streams K/V (the query may sit in host memory).
      const int r = threadIdx.x % kRows;
      const int rho = rho0 + qt_me * kRows + r;
      const bool valid = rho < n_rho;
      const int t = valid ? rho / p.rep : 0, h = valid ? rho % p.rep : 0;
      const __nv_bfloat16 *q = p.q + (int64_t)row.call_row * p.q_row_stride +
                               ((int64_t)t * p.Hq + g * p.rep + h) * D;
      const float2 *cs = p.rope + (int64_t)(lens + t) * kHalf;
      uint8_t *qtile = qsm + qt_me * Cfg::kQBytes;
#pragma unroll 2
      for (int c = 0; c < kHalf / 8; ++c) {
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (valid) {
          const uint4 x1v = *reinterpret_cast<const uint4 *>(q + 8 * c);
          const uint4 x2v = *reinterpret_cast<const uint4 *>(q + kHalf + 8 * c);
          const __nv_bfloat16 *x1 = reinterpret_cast<const __nv_bfloat16 *>(&x1v);
          const __nv_bfloat16 *x2 = reinterpret_cast<const __nv_bfloat16 *>(&x2v);
          __nv_bfloat16 *o1 = reinterpret_cast<__nv_bfloat16 *>(&lo);
          __nv_bfloat16 *o2 = reinterpret_cast<__nv_bfloat16 *>(&hi);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float a = __bfloat162float(x1[j]), b = __bfloat162float(x2[j]);
            const float2 e = cs[8 * c + j];
            o1[j] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(a, e.x), __fmul_rn(b, e.y)));
            o2[j] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(a, e.y), __fmul_rn(b, e.x)));
          }
        }
        const int c_lo = c, c_hi = kHalf / 8 + c;  // 16-byte chunk index along D
        *reinterpret_cast<uint4 *>(qtile + (c_lo / 8) * kRows * 128 +
                                   ptx::swz128(r, c_lo % 8)) = lo;
        *reinterpret_cast<uint4 *>(qtile + (c_hi / 8) * kRows * 128 +
                                   ptx::swz128(r, c_hi % 8)) = hi;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q -> tensor core
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&q_ready[qt_me]);
    }
    const int qt = qt_me;
    const int r = threadIdx.x % kRows;  // query row of this thread = TMEM lane
    const int rho = rho0 + qt * kRows + r;
    const bool qvalid = rho < n_rho;
    const int qpos = lens + (qvalid ? rho / p.rep : 0);
    const uint32_t lane_off = (uint32_t)(32 * (warp % 4)) << 16;
    const uint32_t tO = tmem + kTilesQ * kBlockKeys + qt * D + lane_off;
    uint32_t tS = tmem + qt * kBlockKeys + lane_off;  // S buffer of the current block
    float m_used = -INFINITY;
    // visible key-index ranges of this row in the two segments
    int rg3[3][4];
    row_ranges(seg0_mode, qvalid, qpos, lens, p, rg3[0]);
    row_ranges(kSegRing, qvalid, qpos, lens, p, rg3[1]);
    row_ranges(kSegScratch, qvalid, qpos, lens, p, rg3[2]);
    // Mask and scale (log2 units) of 64-key tile j: returns its key base within the
    // segment and the two ranges, or all_vis when the whole tile is visible.
    struct TileMask {
      int kb, r0, r1, r2, r3;
      bool all_vis;
    };
    auto tile_mask = [&](int j) {
      TileMask m;
      const int sg = seg_of(j);
      m.kb = (j - seg_t0(sg)) * kKeys;
      m.r0 = sg == 0 ? rg3[0][0] : sg == 1 ? rg3[1][0] : rg3[2][0];
      m.r1 = sg == 0 ? rg3[0][1] : sg == 1 ? rg3[1][1] : rg3[2][1];
      m.r2 = sg == 0 ? rg3[0][2] : sg == 1 ? rg3[1][2] : rg3[2][2];
      m.r3 = sg == 0 ? rg3[0][3] : sg == 1 ? rg3[1][3] : rg3[2][3];
      m.all_vis = (m.kb >= m.r0 && m.kb + kKeys - 1 <= m.r1) ||
                  (m.kb >= m.r2 && m.kb + kKeys - 1 <= m.r3);
      return m;
    };
    const float scale = p.scale_log2;
    // Bits lo..hi of a 64-key tile (clamped to the tile; none when lo > hi).
    auto range_bits = [](int lo, int hi) -> uint64_t {
      lo = max(lo, 0);
      hi = min(hi, kKeys - 1);
      if (lo > hi) return 0ull;
      const uint64_t upto = hi == 63 ? ~0ull : (2ull << hi) - 1ull;
      return upto & ~((1ull << lo) - 1ull);
    };
    // S of tile h of the block (64 columns) into v, unscaled (the scale goes into the
    // exponent's FMA), keys the row does not see set to -inf through the tile's visibility
    // bits (one bit test and one select per key); returns its maximum in log2 units
    // (scaling by a positive number commutes with max).
    auto load_tile = [&](int j, int h, float (&v)[kKeys]) {
      const TileMask m = tile_mask(j);
#pragma unroll
      for (int c = 0; c < kKeys / 16; ++c) {
        float t16[16];
        tc::ld16(tS + kKeys * h + 16 * c, t16);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * c + i] = t16[i];
      }
      tc::wait_ld();
      if (!m.all_vis) {
        const uint64_t bits =
            range_bits(m.r0 - m.kb, m.r1 - m.kb) | range_bits(m.r2 - m.kb, m.r3 - m.kb);
        const uint32_t b0 = (uint32_t)bits, b1 = (uint32_t)(bits >> 32);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v[i] = (b0 >> i) & 1u ? v[i] : -INFINITY;
          v[32 + i] = (b1 >> i) & 1u ? v[32 + i] : -INFINITY;
        }
      }
      return max64(v) * scale;
    };
    // P = 2^(s - m) of tile h as bf16 high + low parts over its S columns (tile 1: the
    // spare columns, when there are any): keys 2i, 2i+1 of the high part in column
    // 64h + i, of the low part in column 64h + 32 + i.  The row sum is kept in two packed
    // lanes.
    uint64_t l2 = ptx::f2_pack(0.f, 0.f);
    auto store_p = [&](int h, const float (&v)[kKeys]) {
      const float base = m_used == -INFINITY ? 0.f : m_used;
      const uint64_t nb = ptx::f2_pack(-base, -base);
      // x = s * scale - m (one packed FMA per pair)
      const uint64_t sc2 = ptx::f2_pack(scale, scale);
      const uint32_t tP = Cfg::kSpareP1 && h == 1 ? tmem + Cfg::kColP1 + lane_off : tS + kKeys * h;
#pragma unroll
      for (int c = 0; c < kKeys / 32; ++c) {
        uint32_t hv[16], lv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float x0, x1;
          ptx::f2_unpack(
              ptx::f2_fma(ptx::f2_pack(v[32 * c + 2 * i], v[32 * c + 2 * i + 1]), sc2, nb), x0,
              x1);
          const uint64_t e = ptx::f2_pack(fast_exp2(x0), fast_exp2(x1));
          l2 = ptx::f2_add(l2, e);
          ptx::split_bf16x2(e, hv[i], lv[i]);
        }
        tc::st16(tP + 16 * c, hv);
        tc::st16(tP + kKeys / 2 + 16 * c, lv);
      }
    };
    // Lazy rescale to the tile maximum mt (log2 units): O and l are multiplied by
    // 2^(m_used - mt) only when mt exceeds m_used by more than 2^8.  `stable` waits until
    // every PV issued so far for this query tile has finished writing O.
    auto rescale_to = [&](float mt, auto stable) -> bool {
      float alpha = 1.f;
      bool rescale = false;
      if (m_used == -INFINITY) {
        m_used = mt;  // O and l of this row are still zero
      } else if (mt > m_used + kRescaleLog2) {
        alpha = exp2f(m_used - mt);
        m_used = mt;
        rescale = true;
      }
      if (__any_sync(0xffffffffu, rescale)) {
        if (!__all_sync(0xffffffffu, stable())) return false;
        tc::fence_after();
#pragma unroll 1  // one 16-column chunk of code (instruction fetch)
        for (int c = 0; c < D / 16; ++c) {
          float o16[16];
          tc::ld16(tO + 16 * c, o16);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] *= alpha;
          tc::st16(tO + 16 * c, o16);
        }
        tc::wait_st();
        l2 = ptx::f2_mul(l2, ptx::f2_pack(alpha, alpha));
      }
      return true;
    };
    // Keys past a segment's end may hold anything: query tile 0 zeroes their V rows in
    // tile h of block b so that 0 * V stays 0 in the PV product (its own PV waits for
    // its P, query tile 1's PV of the block for v_ready; the stage cannot be refilled
    // before both PVs are issued).  Returns -1 on a timeout, 1 if rows were zeroed.
    auto zero_v = [&](int b, int h) -> int {
      const int j = 2 * (b_begin + b) + h;
      const int sg = seg_of(j);
      const int kb = (j - seg_t0(sg)) * kKeys;
      const int seg_len_j = seg_len(sg);
      if (seg_len_j - kb >= kKeys) return 0;
      if (!__all_sync(0xffffffffu,
                      ptx::mbar_wait(&kv_full[b % kStages], (b / kStages) & 1, kWaitLimit)))
        return -1;
      uint8_t *vtile =
          kv + (b % kStages) * Cfg::kStageBytes + Cfg::kKVBlock + h * Cfg::kHalfBytes;
      const int first = seg_len_j - kb > 0 ? seg_len_j - kb : 0;
      for (int u = r; u < (kKeys - first) * (D / 8); u += kRows) {
        const int vr = first + u / (D / 8), ch = u % (D / 8);
        *reinterpret_cast<uint4 *>(vtile + (ch / 8) * Cfg::kPanelBytes + ptx::swz128(vr, ch % 8)) =
            make_uint4(0, 0, 0, 0);
      }
      return 1;
    };
    int buf = qt;  // S buffer (and barrier index) of the current block
    // A warp whose 32 rows are all past the CTA's last query row (a part-filled tile) computes
    // nothing: PV reads its lanes' P (stale or zero), which only reach O rows that are never
    // stored, and its sub-partition's issue slots and exponent unit go to the other warps on
    // it.  It still waits for S before each arrival, so it never arrives for a later phase.
    // Only in the one-tile kernel, whose short chunk rows leave tiles part-filled: the
    // two-tile kernel's fills have none, and the branch costs them 1-2%.
    const bool warp_idle = kTilesQ == 1 && rho0 + qt * kRows + 32 * (warp % 4) >= n_rho;
    auto publish = [&](int h) {
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&p_full[2 * buf + h]);
    };
    bool ok = true;
    for (int b = 0; b < n_blocks && ok; ++b) {
      buf = dbl ? (b & 1) : qt;
      tS = tmem + buf * kBlockKeys + lane_off;
      const uint32_t sph = dbl ? (b >> 1) & 1 : b & 1;
      // warp-uniform decisions: tcgen05.ld / st are warp-collective
      const bool good = !*fail && ptx::mbar_wait(&s_full[buf], sph, kWaitLimit);
      if (!__all_sync(0xffffffffu, good)) {
        ok = false;
        break;
      }
      tc::fence_after();
      const int j0 = 2 * (b_begin + b);
      const int halves = j0 + 1 < j_end ? 2 : 1;  // a last block may hold one tile
      // The block's two 64-key tiles run through one copy of the code (a loop that is not
      // unrolled): short CTAs, as in continuous batching, otherwise spend much of their time
      // fetching instructions.
      if (qt == 0) {
        int z = 0;
#pragma unroll 1
        for (int h = 0; h < halves && z >= 0; ++h) {
          const int zh = zero_v(b, h);
          z = zh < 0 ? -1 : max(z, zh);
        }
        if (z < 0) {
          ok = false;
          break;
        }
        if (z > 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&v_ready[b % kStages]);
      }
      if (warp_idle) {  // its rows' P reaches no output: only the barriers' arrivals
#pragma unroll 1
        for (int h = 0; h < halves && ok; ++h) {
          if (Cfg::kSpareP1 && h == 1) {
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s1_read[qt]);
            // With the spare columns S of this block can land before the other warps have
            // published tile 1's P of block b - 1; arriving now could complete that phase.
            // PV(b - 1) having finished shows it is complete (the wait the other warps make
            // before writing P into the spare columns).
            ok = b < 1 || __all_sync(0xffffffffu,
                                     ptx::mbar_wait(&pv_done[qt], (b - 1) & 1, kWaitLimit));
            if (!ok) break;
          }
          publish(h);
        }
        continue;
      }
      float sv[kKeys];
#pragma unroll 1
      for (int h = 0; h < halves; ++h) {
        // A new maximum rescales O once every PV issued so far has finished: PV(b - 1),
        // which may still run when S is double-buffered or the spare columns are used, and
        // for tile 1 PV of tile 0.  Its phases are waited for in order, so a parity wait is
        // never two phases ahead.
        const float mt = load_tile(j0 + h, h, sv);
        if (Cfg::kSpareP1 && h == 1) {  // S of this block may now be overwritten
          tc::fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&s1_read[qt]);
        }
        if (!rescale_to(mt, [&] {
              return (b < 1 || ptx::mbar_wait(&pv_done[qt], (b - 1) & 1, kWaitLimit)) &&
                     (h == 0 || ptx::mbar_wait(&pv0_done[qt], b & 1, kWaitLimit));
            })) {
          ok = false;
          break;
        }
        // The spare columns still hold P of block b - 1 until its PV has finished (QK of
        // this block was issued before that PV).  Phase b - 2 was waited for here in block
        // b - 1, so this wait is not two phases ahead.
        if (Cfg::kSpareP1 && h == 1 && b > 0) {
          if (!__all_sync(0xffffffffu,
                          ptx::mbar_wait(&pv_done[qt], (b - 1) & 1, kWaitLimit))) {
            ok = false;
            break;
          }
          tc::fence_after();
        }
        store_p(h, sv);
        publish(h);
      }
    }
    if (warp_idle) {
      if (!ok) {
        atomicExch(p.err, 1);
        *fail = 1;
      }
    } else {
      float l0, l1;
      ptx::f2_unpack(l2, l0, l1);
      const float l_run = l0 + l1;
      // The last PV's completion implies every earlier MMA of the issuing thread is done.
      // Double-buffered or with the spare columns, PV(n_blocks - 2) may still run here, so
      // pv_done may be two phases behind, or already done with both: wait on the one-phase
      // drain barrier instead.
      const bool last_done =
          ok && n_blocks > 0 &&
          (dbl || Cfg::kSpareP1 ? ptx::mbar_wait(drain, 0, kWaitLimit)
                                : ptx::mbar_wait(&pv_done[qt], (n_blocks - 1) & 1, kWaitLimit));
      if (!ok) {
        atomicExch(p.err, 1);
        *fail = 1;
      } else if (row.part >= 0 && (n_blocks == 0 || __all_sync(0xffffffffu, last_done))) {
        // A key split: this row's unnormalised O, its maximum (log2 units) and sum.
        if (n_blocks > 0) tc::fence_after();
        const int64_t vec = (int64_t)row.part + (int64_t)g * n_rho + rho;
        float4 *po = reinterpret_cast<float4 *>(p.part_o + vec * D);
#pragma unroll 1  // one 16-column chunk of code (instruction fetch)
        for (int c = 0; c < D / 16; ++c) {
          float o16[16];
          if (n_blocks > 0) {
            tc::ld16(tO + 16 * c, o16);
            tc::wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) o16[i] = 0.f;
          }
          if (qvalid) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              po[4 * c + i] =
                  make_float4(o16[4 * i], o16[4 * i + 1], o16[4 * i + 2], o16[4 * i + 3]);
          }
        }
        if (qvalid) p.part_ml[vec] = make_float2(m_used, l_run);
      } else if (__all_sync(0xffffffffu, last_done)) {
        tc::fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const int t = qvalid ? rho / p.rep : 0, h = qvalid ? rho % p.rep : 0;
        __nv_bfloat16 *dst = p.out + (int64_t)row.call_row * p.out_row_stride +
                             ((int64_t)t * p.Hq + g * p.rep + h) * D;
#pragma unroll 1  // one 16-column chunk of code (instruction fetch)
        for (int c = 0; c < D / 16; ++c) {
          float o16[16];
          tc::ld16(tO + 16 * c, o16);
          tc::wait_ld();
          uint4 w0, w1;
          w0.x = ptx::pack_bf16(o16[0] * inv, o16[1] * inv);
          w0.y = ptx::pack_bf16(o16[2] * inv, o16[3] * inv);
          w0.z = ptx::pack_bf16(o16[4] * inv, o16[5] * inv);
          w0.w = ptx::pack_bf16(o16[6] * inv, o16[7] * inv);
          w1.x = ptx::pack_bf16(o16[8] * inv, o16[9] * inv);
          w1.y = ptx::pack_bf16(o16[10] * inv, o16[11] * inv);
          w1.z = ptx::pack_bf16(o16[12] * inv, o16[13] * inv);
          w1.w = ptx::pack_bf16(o16[14] * inv, o16[15] * inv);
          if (qvalid) {
            *reinterpret_cast<uint4 *>(dst + 16 * c) = w0;
            *reinterpret_cast<uint4 *>(dst + 16 * c + 8) = w1;
          }
        }
      } else if (n_blocks > 0) {
        atomicExch(p.err, 1);
        *fail = 1;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc::fence_before();
  __syncthreads();
  if (*fail && threadIdx.x == 0) {
    // Let every TMA load this CTA issued land before its shared memory is released.
    const int n_issued = *issued;
    for (int s = 0; s < kStages && s < n_issued; ++s) {
      const int lst = s + ((n_issued - 1 - s) / kStages) * kStages;
      ptx::mbar_wait(&kv_full[s], (lst / kStages) & 1, kWaitLimit);
    }
  }
  if (warp == kMmaWarp) {
    tc::fence_after();
    tc::dealloc(tmem, Cfg::kTmemCols);
  }
}

}  // namespace

// Query tiles per CTA of the tcgen05 prefill for head dimension D.  D = 128: two tiles
// share every K/V block (a CTA whose row fills one tile double-buffers S instead).  D = 64:
// one tile per CTA, two CTAs per SM (two independent chains per SM; each K/V block is
// streamed once per tile).  Measured on the continuous-batch mix (D = 64): 2.49 M tokens/s
// with one tile per CTA, 2.39 M with two; rows of one tile alone on the one-tile kernel,
// 2.24 M.
int prefill_tc_tiles(int D, int) { return D == 64 ? 1 : 2; }

template <int D, int TQ>
static cudaError_t launch_tc(const PrefillParams &p, cudaStream_t s, bool pdl) {
  return launch_k(prefill_tc_kernel<D, TQ>, dim3(p.n_ctas, p.Hk), dim3(Roles<TQ>::kThreads),
                  TcCfg<D, TQ>::kSmem, s, p, pdl);
}

cudaError_t launch_prefill_tc(const PrefillParams &p, int D, int tiles, cudaStream_t s,
                              bool pdl) {
  if (p.n_ctas <= 0) return cudaSuccess;
  if (D == 128 && tiles == 2) return launch_tc<128, 2>(p, s, pdl);
  if (D == 64 && tiles == 1) return launch_tc<64, 1>(p, s, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t configure_prefill_tc() {
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<128, 2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcCfg<128, 2>::kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(prefill_tc_kernel<64, 1>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<64, 1>::kSmem);
  return e;
}

}  // namespace kvinc
