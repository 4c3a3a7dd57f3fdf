// prefill_tc.cu -- chunked prefill on the 5th-generation tensor cores (tcgen05, TMEM).
//
// What is computed is the same as prefill.cu: query row rho of a (row, kv head) is
// token t = rho / rep, head h = rho % rep of the GQA group at absolute position
// p = lens + t; it attends to the visible keys of the layer storage (global: slots
// [0, lens + t], sliding: the ring's occupied slots, whose positions follow from
// lens) and of the chunk scratch (sliding layers), reading the ring before this
// chunk is committed to it ("inkling: ring-buffer KV cache for sliding-window
// layers", How it works; Lab 07 section 3; tiny_agent/generate.py `_append_chunk`).
//
// One CTA owns up to two 128-row query tiles (the MMA's M) of one (row, kv head);
// both tiles share every K/V tile the CTA streams.  Warp roles:
//   warps 0-7  softmax, four per query tile: thread i of a tile owns query row i =
//              TMEM lane i of that tile's accumulators.  They rotate the queries into
//              shared memory, read S from TMEM, mask, run the online softmax (lazy
//              rescaling: O in TMEM is rescaled only when a row's maximum grows by
//              more than 2^8), write P as bf16 high and low parts back into the TMEM
//              columns that held S, and finally read O from TMEM and normalise.  Two warps of different
//              tiles share each SM sub-partition and hide each other's latency.
//   warp 8     TMA producer of 64-key K and V tiles (128-byte swizzle).
//   warp 9     TMEM owner and MMA issuer (one thread).  For each query tile it keeps
//              two cursors: S = Q K^T (M=128, N=64) of K/V tile j into one of the
//              tile's two TMEM S buffers once the K/V stage has landed and the PV that
//              last read that buffer is done, and O += P_hi V + P_lo V (M=128, N=D)
//              once the softmax warps have written P of tile j, with P read from TMEM
//              and V read in place as an MN-major operand (keys are its K).  It polls both query tiles and issues whichever step
//              is ready, so one tile's slow softmax does not stall the other's MMAs; a
//              K/V stage is released when both tiles' PV of it has been issued.
// Every mbarrier wait is bounded; on a timeout the CTA records the error, lets its
// own TMA loads and MMAs finish (bounded), frees its TMEM and returns.
#include "kvinc_internal.h"
#include "ptx.cuh"

namespace kvinc {
namespace {

constexpr int kRows = 128;        // query rows per tile (MMA M)
constexpr int kTilesQ = 2;        // query tiles per CTA
constexpr int kKeys = kTileKeys;  // keys per tile (MMA N of S, K of PV)
constexpr int kSoftmaxWarps = 4;  // per query tile
constexpr int kProducerWarp = kTilesQ * kSoftmaxWarps, kMmaWarp = kProducerWarp + 1;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (log2 units)

template <int D>
struct TcCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kStages = D == 128 ? 5 : 8;
  static constexpr int kQBytes = kPanels * kRows * 128;   // one Q tile, K-major, 128B swizzle
  static constexpr int kKVTile = kPanels * kKeys * 128;    // one K or V tile (TMA layout)
  static constexpr int kStageBytes = 2 * kKVTile;
  // TMEM: per query tile two 64-column S buffers (S fp32; then P as 32 columns of bf16
  // pairs for the high part and 32 for the low part) and one D-column O accumulator.
  static constexpr int kTmemCols = 512;                    // [S0 S0' S1 S1'] [O0] [O1]
  static constexpr int kOff_Q = 0;
  static constexpr int kOff_KV = kOff_Q + kTilesQ * kQBytes;
  static constexpr int kOff_Bar = kOff_KV + kStages * kStageBytes;
  static constexpr int kBars = 2 * kStages + kTilesQ * 6 + 1;
  static constexpr int kSmem = 1024 + kOff_Bar + kBars * 8 + 32;
  static_assert(kSmem <= 232448, "shared memory per CTA");
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
// (an empty range has lo > hi).  Global layer: cache slots 0..p.  Sliding layer, ring
// segment: slot s holds position s + base (s <= rem) or s + base - R (s > rem), or just s
// while lens <= R; it is visible iff that position is >= p - W + 1.  Sliding layer, chunk
// scratch: token j sits at lens + j and is visible iff p - W + 1 <= lens + j <= p.
__device__ __forceinline__ void row_ranges(bool ring_or_cache, bool qvalid, int qpos, int lens,
                                           const PrefillParams &p, int (&rg)[4]) {
  rg[0] = 1; rg[1] = 0; rg[2] = 1; rg[3] = 0;
  if (!qvalid) return;
  if (!p.sliding) {  // the global cache holds this chunk too: slots 0..qpos
    rg[0] = 0;
    rg[1] = qpos;
    return;
  }
  const int thr = qpos - p.window + 1;  // first visible position
  if (!ring_or_cache) {                 // chunk scratch
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ PrefillParams p) {
  using Cfg = TcCfg<D>;
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
  // Per query tile and S buffer b (tile j uses b = j & 1); each barrier completes one
  // phase per use of its buffer, and a buffer is reused only after its previous PV is
  // done, so no waiter can fall two phases behind.
  uint64_t *s_full = kv_empty + kStages;          // [tile][b] QK done -> softmax
  uint64_t *p_full = s_full + 2 * kTilesQ;        // [tile][b] softmax wrote P -> MMA
  uint64_t *pv_done = p_full + 2 * kTilesQ;       // [tile][b] PV done -> MMA, softmax
  uint64_t *drain = pv_done + 2 * kTilesQ;        // [1] every MMA done (teardown)
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + Cfg::kBars);
  volatile int *fail = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *issued = fail + 1;

  const PrefillRow &row = p.rows[find_cta_row(p, blockIdx.x)];
  const int g = blockIdx.y;
  const int rho0 = (blockIdx.x - row.cta0) * kRows * kTilesQ;
  const int n_rho = row.n * p.rep;
  const int n_qt = min(kTilesQ, (n_rho - rho0 + kRows - 1) / kRows);  // query tiles in use
  const int rho_last = min(n_rho, rho0 + kRows * kTilesQ) - 1;
  const int t_max = rho_last / p.rep;
  const int lens = row.lens;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int len_a = p.sliding ? min(lens, p.ring_R) : lens + t_max + 1;
  const int len_b = p.sliding ? t_max + 1 : 0;
  const int tiles_a = (len_a + kKeys - 1) / kKeys;
  const int n_tiles = tiles_a + (len_b + kKeys - 1) / kKeys;
  const int64_t base_a = ((int64_t)row.cache_row * p.Hk + g) * p.seg_rows;
  const int64_t base_b = ((int64_t)row.cache_row * p.Hk + g) * kChunk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&kv_full[s], 1);
      ptx::mbar_init(&kv_empty[s], 1);
    }
    for (int qt = 0; qt < kTilesQ; ++qt) {
      for (int b = 0; b < 2; ++b) {
        ptx::mbar_init(&s_full[2 * qt + b], 1);
        ptx::mbar_init(&p_full[2 * qt + b], kSoftmaxWarps);
        ptx::mbar_init(&pv_done[2 * qt + b], 1);
      }
    }
    ptx::mbar_init(drain, 1);
    *fail = 0;
    *issued = 0;
    ptx::fence_barrier_init();
  }
  if (warp == kMmaWarp) tc::alloc(tmem_slot, Cfg::kTmemCols);
  const int qt_me = warp / kSoftmaxWarps;  // query tile of a softmax warp
  if (warp < kProducerWarp) {
    // Rotated query of this thread's row into its tile's 128-byte-swizzled Q tile.
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
      *reinterpret_cast<uint4 *>(qtile + (c_lo / 8) * kRows * 128 + ptx::swz128(r, c_lo % 8)) = lo;
      *reinterpret_cast<uint4 *>(qtile + (c_hi / 8) * kRows * 128 + ptx::swz128(r, c_hi % 8)) = hi;
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // Q -> tensor core
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      ptx::prefetch_tmap(&p.tmap_k);
      ptx::prefetch_tmap(&p.tmap_v);
      for (int it = 0; it < n_tiles && !*fail; ++it) {
        const int s = it % kStages;
        if (it >= kStages &&
            !ptx::mbar_wait(&kv_empty[s], ((it / kStages) - 1) & 1, kWaitLimit)) {
          atomicExch(p.err, 1);
          *fail = 1;
          break;
        }
        uint8_t *kt = kv + s * Cfg::kStageBytes;
        uint8_t *vtile = kt + Cfg::kKVTile;
        const bool in_a = it < tiles_a;
        const CUtensorMap *mk = in_a ? &p.tmap_k : &p.tmap_sk;
        const CUtensorMap *mv = in_a ? &p.tmap_v : &p.tmap_sv;
        const int y = static_cast<int>(in_a ? base_a + (int64_t)it * kKeys
                                            : base_b + (int64_t)(it - tiles_a) * kKeys);
        ptx::mbar_arrive_expect_tx(&kv_full[s], Cfg::kStageBytes);
#pragma unroll
        for (int pn = 0; pn < Cfg::kPanels; ++pn) {
          ptx::tma_load_2d(kt + pn * kKeys * 128, mk, pn * 64, y, &kv_full[s]);
          ptx::tma_load_2d(vtile + pn * kKeys * 128, mv, pn * 64, y, &kv_full[s]);
        }
        *issued = it + 1;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdQK = tc::idesc_bf16_f32(kRows, kKeys);
      constexpr uint32_t kIdPV = tc::idesc_bf16_f32(kRows, D, /*b_mn_major=*/true);
      // Fixed issue order.  Prologue QK(0, q0), QK(0, q1), QK(1, q0); then per K/V tile r:
      //   PV(r, q0), QK(r + 1, q1), PV(r, q1), QK(r + 2, q0).
      // QK(j, q) reuses the S buffer of PV(j - 2, q), which was issued three groups
      // earlier, so the tensor pipe is not left waiting on its own work; each PV waits
      // for its softmax, which runs while the three groups before it execute.  PV(r, q1)
      // follows PV(r, q0), i.e. query tile 0's P of tile r, which is published after its
      // softmax warps zeroed the V rows past a segment's end.
      auto issue_qk = [&](int qt, int j) -> bool {
        if (qt >= n_qt || j >= n_tiles) return true;
        if (!ptx::mbar_wait(&kv_full[j % kStages], (j / kStages) & 1, kWaitLimit)) return false;
        if (j >= 2 && !ptx::mbar_wait(&pv_done[2 * qt + (j & 1)], ((j - 2) >> 1) & 1, kWaitLimit))
          return false;
        tc::fence_after();
        const uint32_t k_addr = ptx::smem_u32(kv + (j % kStages) * Cfg::kStageBytes);
        const uint32_t q_addr = ptx::smem_u32(qsm + qt * Cfg::kQBytes);
        const uint32_t tS = tmem + (2 * qt + (j & 1)) * kKeys;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off_q = (kk / 4) * (kRows * 128) + 32 * (kk % 4);
          const uint32_t off_k = (kk / 4) * (kKeys * 128) + 32 * (kk % 4);
          tc::mma(tS, tc::desc_sw128(q_addr + off_q), tc::desc_sw128(k_addr + off_k), kIdQK,
                  kk > 0);
        }
        tc::commit(&s_full[2 * qt + (j & 1)]);
        return true;
      };
      auto issue_pv = [&](int qt, int j) -> bool {
        if (qt >= n_qt) return true;
        if (!ptx::mbar_wait(&p_full[2 * qt + (j & 1)], (j >> 1) & 1, kWaitLimit)) return false;
        tc::fence_after();
        // B = V as stored by TMA: rows = keys (K), 64-dim panels (MN) kKeys*128 apart;
        // A = P in the S buffer: high part in columns 0-31, low part in 32-63, one
        // 16-key step = 8 columns.
        const uint32_t v_addr =
            ptx::smem_u32(kv + (j % kStages) * Cfg::kStageBytes + Cfg::kKVTile);
        const uint32_t tP = tmem + (2 * qt + (j & 1)) * kKeys;
        const uint32_t tO = tmem + 4 * kKeys + qt * D;
#pragma unroll
        for (int ks = 0; ks < kKeys / 16; ++ks) {
          const uint64_t bd = tc::desc_sw128_mn(v_addr + ks * 16 * 128, kKeys * 128, 1024);
          tc::mma_ts(tO, tP + 8 * ks, bd, kIdPV, j > 0 || ks > 0);
          tc::mma_ts(tO, tP + kKeys / 2 + 8 * ks, bd, kIdPV, true);
        }
        tc::commit(&pv_done[2 * qt + (j & 1)]);
        return true;
      };
      bool ok = issue_qk(0, 0) && issue_qk(1, 0) && issue_qk(0, 1);
      for (int r = 0; ok && r < n_tiles; ++r) {
        if (*fail) {
          ok = false;
          break;
        }
        ok = issue_pv(0, r) && issue_qk(1, r + 1) && issue_pv(1, r);
        if (ok) tc::commit(&kv_empty[r % kStages]);  // every PV of the stage issued
        ok = ok && issue_qk(0, r + 2);
      }
      if (!ok) {
        atomicExch(p.err, 1);
        *fail = 1;
      }
      // Every MMA issued has completed before TMEM can be released.
      tc::commit(drain);
      ptx::mbar_wait(drain, 0, kWaitLimit);
    }
  } else if (qt_me < n_qt) {
    // ------------------------------------------------------------ softmax warps
    const int qt = qt_me;
    const int r = threadIdx.x % kRows;  // query row of this thread = TMEM lane
    const int rho = rho0 + qt * kRows + r;
    const bool qvalid = rho < n_rho;
    const int qpos = lens + (qvalid ? rho / p.rep : 0);
    const uint32_t lane_off = (uint32_t)(32 * (warp % 4)) << 16;
    const uint32_t tO = tmem + 4 * kKeys + qt * D + lane_off;
    float m_used = -INFINITY, l_run = 0.f;
    int rg[4];  // visible key-index ranges [rg0, rg1] and [rg2, rg3] of the current segment
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int sb = j & 1;
      // warp-uniform decisions: tcgen05.ld / st are warp-collective
      const bool good = !*fail && ptx::mbar_wait(&s_full[2 * qt + sb], (j >> 1) & 1, kWaitLimit);
      if (!__all_sync(0xffffffffu, good)) {
        ok = false;
        break;
      }
      tc::fence_after();
      float sv[kKeys];
      const uint32_t tS = tmem + (2 * qt + sb) * kKeys + lane_off;
#pragma unroll
      for (int c = 0; c < kKeys / 16; ++c) {
        float t16[16];
        tc::ld16(tS + 16 * c, t16);
#pragma unroll
        for (int i = 0; i < 16; ++i) sv[16 * c + i] = t16[i];
      }
      tc::wait_ld();

      // mask and scale (log2 units): the visible keys of a segment are at most two
      // index ranges per row (computed when the segment starts)
      const bool in_a = j < tiles_a;
      const int kb = (in_a ? j : j - tiles_a) * kKeys;
      const int seg_len = in_a ? len_a : len_b;
      if (j == 0 || j == tiles_a) row_ranges(in_a, qvalid, qpos, lens, p, rg);
      float mt = -INFINITY;
      const bool all_vis = (kb >= rg[0] && kb + kKeys - 1 <= rg[1]) ||
                           (kb >= rg[2] && kb + kKeys - 1 <= rg[3]);
      if (all_vis) {
#pragma unroll
        for (int i = 0; i < kKeys; ++i) {
          sv[i] *= p.scale_log2;
          mt = fmaxf(mt, sv[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < kKeys; ++i) {
          const int kidx = kb + i;
          const bool vis = (kidx >= rg[0] && kidx <= rg[1]) || (kidx >= rg[2] && kidx <= rg[3]);
          sv[i] = vis ? sv[i] * p.scale_log2 : -INFINITY;
          mt = fmaxf(mt, sv[i]);
        }
      }
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
        // O must be stable: PV(j-1) of this tile is done (PV(j) waits for this P).
        const bool prev = j < 1 || ptx::mbar_wait(&pv_done[2 * qt + ((j - 1) & 1)],
                                                  ((j - 1) >> 1) & 1, kWaitLimit);
        if (!__all_sync(0xffffffffu, prev)) {
          ok = false;
          break;
        }
        tc::fence_after();
#pragma unroll
        for (int c = 0; c < D / 16; ++c) {
          float o16[16];
          tc::ld16(tO + 16 * c, o16);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] *= alpha;
          tc::st16(tO + 16 * c, o16);
        }
        tc::wait_st();
      }
      l_run *= alpha;
      if (qt == 0 && seg_len - kb < kKeys) {
        // Keys past the segment may hold anything: zero their V rows so that 0 * V
        // stays 0 in the PV product (every PV of this tile is issued after query tile
        // 0 publishes its P).  The stage cannot be refilled before that either.
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&kv_full[j % kStages], (j / kStages) & 1,
                                                    kWaitLimit))) {
          ok = false;
          break;
        }
        uint8_t *vtile = kv + (j % kStages) * Cfg::kStageBytes + Cfg::kKVTile;
        const int first = seg_len - kb > 0 ? seg_len - kb : 0;
        for (int u = r; u < (kKeys - first) * (D / 8); u += kRows) {
          const int vr = first + u / (D / 8), ch = u % (D / 8);
          *reinterpret_cast<uint4 *>(vtile + (ch / 8) * (kKeys * 128) + ptx::swz128(vr, ch % 8)) =
              make_uint4(0, 0, 0, 0);
        }
      }
      const float base = m_used == -INFINITY ? 0.f : m_used;
      // P = 2^(s - m) as bf16 high + low parts over S in TMEM: keys 2i, 2i+1 of the high
      // part in column i, of the low part in column 32 + i.
#pragma unroll
      for (int c = 0; c < kKeys / 32; ++c) {
        uint32_t hv[16], lv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float e0 = fast_exp2(sv[32 * c + 2 * i] - base);
          const float e1 = fast_exp2(sv[32 * c + 2 * i + 1] - base);
          l_run += e0 + e1;
          ptx::split_bf16(e0, e1, hv[i], lv[i]);
        }
        tc::st16(tS + 16 * c, hv);
        tc::st16(tS + kKeys / 2 + 16 * c, lv);
      }
      tc::wait_st();
      if (qt == 0 && seg_len - kb < kKeys)
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // zeroed V -> MMA
      tc::fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&p_full[2 * qt + sb]);
    }
    // The last PV's completion implies every earlier MMA of the issuing thread is done.
    const bool last_done =
        ok && n_tiles > 0 &&
        ptx::mbar_wait(&pv_done[2 * qt + ((n_tiles - 1) & 1)], ((n_tiles - 1) >> 1) & 1,
                       kWaitLimit);
    if (!ok) {
      atomicExch(p.err, 1);
      *fail = 1;
    } else if (__all_sync(0xffffffffu, last_done)) {
      tc::fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const int t = qvalid ? rho / p.rep : 0, h = qvalid ? rho % p.rep : 0;
      __nv_bfloat16 *dst = p.out + (int64_t)row.call_row * p.out_row_stride +
                           ((int64_t)t * p.Hq + g * p.rep + h) * D;
#pragma unroll
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
    } else if (n_tiles > 0) {
      atomicExch(p.err, 1);
      *fail = 1;
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

// Query rows one CTA of the tcgen05 prefill covers.
int prefill_tc_rows_per_cta() { return kRows * kTilesQ; }

cudaError_t launch_prefill_tc(const PrefillParams &p, int D, cudaStream_t s) {
  if (p.n_ctas <= 0) return cudaSuccess;
  if (D == 128) {
    prefill_tc_kernel<128><<<dim3(p.n_ctas, p.Hk), kThreads, TcCfg<128>::kSmem, s>>>(p);
  } else if (D == 64) {
    prefill_tc_kernel<64><<<dim3(p.n_ctas, p.Hk), kThreads, TcCfg<64>::kSmem, s>>>(p);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t configure_prefill_tc() {
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<128>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcCfg<128>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TcCfg<64>::kSmem);
}

}  // namespace kvinc
