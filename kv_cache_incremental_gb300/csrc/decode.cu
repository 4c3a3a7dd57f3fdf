// decode.cu -- split-K grouped-query decode attention against the cache, with the
// decode token's append and the split merge fused in.
//
// One CTA owns one (row, kv head, key split).  A producer warp streams the
// split's K and V rows through a multi-stage shared-memory ring with TMA 2-D
// tile loads (128-byte swizzle, one mbarrier pair per stage); four consumer
// warps each take 16 keys of every 64-key tile.  For the whole GQA group at
// once a warp computes S^T = K Q^T on the tensor cores (keys on the MMA's M
// side, the group's query heads on N), keeps a per-warp online softmax in
// float, and accumulates O^T = V^T P^T with P split into a bf16 high and low
// part so that the probabilities keep ~16 significant bits.
//
// Append fused in (kv_append's decode rows): the CTA whose key range holds the
// new token's storage slot rotates the new key itself (tiny_agent/generate.py
// `_rope_pos`), masks the slot's stale content in its tiles, scores the new key
// from a 16-row shared-memory mini-tile after its main loop, and stores the
// rotated key and the value to the cache once all of its loads have landed.  No
// other CTA reads that slot, and later launches see the stored key.
//
// Split merge fused in: a split writes its float partial (m, l, O); the last
// CTA of a (row, kv head) to finish -- found with an atomic ticket -- merges
// all splits (log-sum-exp) and writes the bf16 output, then re-arms the ticket.
// A row with a single split writes its output directly.
//
// Programmatic dependent launch: the kernel may be launched so that it starts while
// the previous kernel on the stream finishes.  The consumers wait for the previous grid
// (griddepcontrol.wait) before any other read or write, then let the next launch start;
// the producer waits too unless the host allowed early K/V loads (early_kv: the launch
// before it wrote none of this layer's storage -- with every PDL launch letting its
// successor start only after its own wait, all older grids have completed by then).
//
// What is computed follows tiny_agent/generate.py `_append_chunk` (grouped
// queries straight against the cache, scale 1/sqrt(D), float softmax) and the
// inkling ring-buffer pull request (the sliding scan covers the last W
// positions): for a decode token at position p the visible keys are storage
// slots [0, nk) with nk = p + 1 (global) or min(p + 1, R) (sliding ring, which
// holds exactly positions max(0, p - W + 1) .. p once the new key is in).  A
// softmax does not depend on the order of its keys, so slots are read in
// storage order.
#include "kvinc_internal.h"
#include "ptx.cuh"

namespace kvinc {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMiniRows = 16;  // rows of the new-key mini-tile

// Stages of the K/V ring: 96 KB at D = 128 (two CTAs per SM) and 64 KB at D = 64 (three CTAs
// per SM: more warps to hide the shorter tiles' latency; the continuous-batch mix's decode
// launches 5.45 -> 5.04 ms over 50 steps against six stages at two CTAs per SM), or with
// DEEP twice that (one CTA per SM) for launches of at most one wave, whose CTAs each need
// twice the bytes in flight to keep HBM busy.
template <int D, bool DEEP>
struct DecodeCfg {
  static constexpr int kPanels = D / 64;                        // 128-byte swizzle panels
  static constexpr int kTileBytes = kPanels * kTileKeys * 128;  // one K or V tile
  static constexpr int kStages = (D == 128 ? 3 : 4) * (DEEP ? 2 : 1);
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kMiniBytes = kPanels * kMiniRows * 128;  // one K or V mini-tile
};

template <int D, int NT, bool DEEP>
constexpr int decode_smem_bytes() {
  using C = DecodeCfg<D, DEEP>;
  return 1024 /*alignment slack*/ + C::kStages * C::kStageBytes + 2 * C::kMiniBytes +
         NT * 8 * D * 2 /*Q*/ + 2 * D * 2 /*new K, V*/ + 2 * C::kStages * 8 /*barriers*/ +
         16 /*flags*/;
}

// Row of work item `item`: a division when every row of the launch has the same number of
// items (each probe of the search below is a dependent parameter load, slow at kernel
// start), else a binary search over the rows' first items.
__device__ __forceinline__ int find_item_row(const DecodeParams &p, int item) {
  if (p.uniform_items > 0) return item / p.uniform_items;
  int lo = 0, hi = p.n_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.rows[mid].item0 <= item) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

template <int D, int NT>
struct WarpAcc {
  float o[D / 16][NT][4];  // O^T fragments: (head dim, head)
  float m[NT][2];          // running max (log2 units) of the lane's two heads
  float l[NT][2];          // lane-partial sum of weights
};

// One warp, 16 keys at smem rows [row0, row0 + 16) of a K tile `kt` and V tile `vt`
// whose 128-byte panels are `pstride` bytes apart.  Keys r < n_valid, r != skip are
// visible; the V rows of the others must already be zero.
template <int D, int NT>
__device__ __forceinline__ void attend16(WarpAcc<D, NT> &acc, const uint32_t (&qb)[NT][D / 16][2],
                                         const uint8_t *kt, const uint8_t *vt, int pstride,
                                         int row0, int n_valid, int skip, float scale_log2,
                                         int lane) {
  const int gq = lane >> 2;
  float sacc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
  {
    const int mrow = row0 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int ch = 2 * (kk % 4) + (lane >> 4);
      uint32_t a0, a1, a2, a3;
      ptx::ldsm_x4(ptx::smem_u32(kt + (kk / 4) * pstride) + ptx::swz128(mrow, ch), a0, a1, a2,
                   a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        ptx::mma_bf16(sacc[nt], a0, a1, a2, a3, qb[nt][kk][0], qb[nt][kk][1]);
    }
  }
  const bool va = gq < n_valid && gq != skip;
  const bool vb = gq + 8 < n_valid && gq + 8 != skip;
  uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float t0 = va ? sacc[nt][0] * scale_log2 : -INFINITY;
    const float t1 = va ? sacc[nt][1] * scale_log2 : -INFINITY;
    const float t2 = vb ? sacc[nt][2] * scale_log2 : -INFINITY;
    const float t3 = vb ? sacc[nt][3] * scale_log2 : -INFINITY;
    float mx0 = fmaxf(t0, t2), mx1 = fmaxf(t1, t3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(acc.m[nt][0], mx0), mn1 = fmaxf(acc.m[nt][1], mx1);
    const float b0 = mn0 == -INFINITY ? 0.f : mn0;
    const float b1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2f(acc.m[nt][0] - b0), al1 = exp2f(acc.m[nt][1] - b1);
    const float p0 = exp2f(t0 - b0), p1 = exp2f(t1 - b1);
    const float p2 = exp2f(t2 - b0), p3 = exp2f(t3 - b1);
    acc.m[nt][0] = mn0;
    acc.m[nt][1] = mn1;
    acc.l[nt][0] = acc.l[nt][0] * al0 + (p0 + p2);
    acc.l[nt][1] = acc.l[nt][1] * al1 + (p1 + p3);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      acc.o[mt][nt][0] *= al0;
      acc.o[mt][nt][1] *= al1;
      acc.o[mt][nt][2] *= al0;
      acc.o[mt][nt][3] *= al1;
    }
    uint32_t h01, l01, h23, l23;
    ptx::split_bf16(p0, p1, h01, l01);
    ptx::split_bf16(p2, p3, h23, l23);
    // (key, head) fragments -> (head, key) fragments: the B operand of O^T = V^T P^T
    bh[nt][0] = ptx::movm_t(h01);
    bh[nt][1] = ptx::movm_t(h23);
    bl[nt][0] = ptx::movm_t(l01);
    bl[nt][1] = ptx::movm_t(l23);
  }
  {
    const int mi = lane >> 3;
    const int vrow = row0 + (lane & 7) + (mi >> 1) * 8;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      const int ch = 2 * (mt % 4) + (mi & 1);
      uint32_t a0, a1, a2, a3;
      ptx::ldsm_x4_t(ptx::smem_u32(vt + (mt / 4) * pstride) + ptx::swz128(vrow, ch), a0, a1, a2,
                     a3);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        ptx::mma_bf16(acc.o[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
        ptx::mma_bf16(acc.o[mt][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
      }
    }
  }
}

// RoPE of 8 half-split pairs (x1[j], x2[j]) at one position, (cos, sin) pairs in
// registers two per float4: f32 products and sums without contraction, then RNE to bf16
// (tiny_agent/generate.py `_rope_pos`).
__device__ __forceinline__ void rope8r(const uint4 &x1v, const uint4 &x2v, const float4 (&cs)[4],
                                       uint4 &lo, uint4 &hi) {
  const __nv_bfloat16 *x1 = reinterpret_cast<const __nv_bfloat16 *>(&x1v);
  const __nv_bfloat16 *x2 = reinterpret_cast<const __nv_bfloat16 *>(&x2v);
  __nv_bfloat16 *o1 = reinterpret_cast<__nv_bfloat16 *>(&lo);
  __nv_bfloat16 *o2 = reinterpret_cast<__nv_bfloat16 *>(&hi);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float a = __bfloat162float(x1[j]), b = __bfloat162float(x2[j]);
    const float cc = (j & 1) ? cs[j / 2].z : cs[j / 2].x, sn = (j & 1) ? cs[j / 2].w : cs[j / 2].y;
    o1[j] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(a, cc), __fmul_rn(b, sn)));
    o2[j] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, cc)));
  }
}

// Zero one 16-byte chunk of V row `r` of a swizzled tile.
__device__ __forceinline__ void zero_v_chunk(uint8_t *vt, int pstride, int r, int ch) {
  *reinterpret_cast<uint4 *>(vt + (ch / 8) * pstride + ptx::swz128(r, ch % 8)) =
      make_uint4(0, 0, 0, 0);
}

// Occupancy is set by shared memory (two CTAs per SM at D = 128, three at D = 64, one with
// DEEP); the bound tells the register allocator so (left alone it chose 64 registers and
// spilled at D = 64).
template <int D, int NT, bool DEEP>
__global__ void __launch_bounds__(kThreads, DEEP ? 1 : D == 64 ? 3 : 2)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  using Cfg = DecodeCfg<D, DEEP>;
  constexpr int kStages = Cfg::kStages;
  constexpr int kHalf = D / 2;
  static_assert(kHalf % 8 == 0, "head dim must be a multiple of 16");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *tiles = smem;                                     // [stage][K tile | V tile]
  uint8_t *mini_k = smem + kStages * Cfg::kStageBytes;       // new-key mini-tiles
  uint8_t *mini_v = mini_k + Cfg::kMiniBytes;
  __nv_bfloat16 *qs = reinterpret_cast<__nv_bfloat16 *>(mini_v + Cfg::kMiniBytes);
  __nv_bfloat16 *knew = qs + NT * 8 * D;                     // rotated new key, then value
  __nv_bfloat16 *vnew = knew + D;
  uint64_t *full = reinterpret_cast<uint64_t *>(vnew + D);
  uint64_t *empty = full + kStages;
  volatile int *fail = reinterpret_cast<volatile int *>(empty + kStages);  // a wait gave up
  volatile int *issued = fail + 1;                                          // tiles loaded
  volatile int *last = fail + 2;                                            // merging CTA

  const int item = blockIdx.x;
  const int g = blockIdx.y;
  const DecodeRow &row = p.rows[find_item_row(p, item)];
  // The item's key segment: 0 = the layer storage (a global cache, a sliding ring, or a
  // hybrid layer's group cache), 1 = a hybrid layer's own ring.
  const int split = item - row.item0;          // over all the row's splits (merge slot)
  const bool seg1 = split >= row.n_splits;
  const int n_total = row.n_splits + row.n_splits2;
  const int ssplit = seg1 ? split - row.n_splits : split;
  const int split_len = (seg1 ? row.split_tiles2 : row.split_tiles) * kTileKeys;
  const int k0 = ssplit * split_len;
  const int k1 = min(seg1 ? min(row.pos + 1, p.ring_R) : row.nk, k0 + split_len);
  const int n_tiles = (k1 - k0 + kTileKeys - 1) / kTileKeys;
  const int new_slot = seg1 || p.seg0_ring ? row.pos % p.ring_R : row.pos;
  const bool owner = (seg1 ? p.fuse_append2 : p.fuse_append) && new_slot >= k0 && new_slot < k1;
  const int seg_rows = seg1 ? p.seg_rows2 : p.seg_rows;
  PageTable pt = p.pt;
  if (seg1) pt.max_blocks = 0;                 // rings are dense
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], kConsumerWarps);
    }
    *fail = 0;
    *issued = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();  // barriers ready: the producer streams while consumers set up
  const int64_t row0 = ((int64_t)row.cache_row * p.Hk + g) * seg_rows + k0;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // One copy of the loop per segment, so that each names its tensor maps by their
    // fixed parameter addresses.
    auto produce = [&](const CUtensorMap *map_k, const CUtensorMap *map_v) {
      ptx::prefetch_tmap(map_k);
      ptx::prefetch_tmap(map_v);
      for (int it = 0; it < n_tiles; ++it) {
        const int s = it % kStages;
        if (it >= kStages) {
          if (!ptx::mbar_wait(&empty[s], ((it / kStages) - 1) & 1, kWaitLimit)) {
            atomicExch(p.err, 1);  // consumers then give up on the tiles never loaded
            break;
          }
        }
        uint8_t *kt = tiles + s * Cfg::kStageBytes;
        uint8_t *vt = kt + Cfg::kTileBytes;
        ptx::mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
        if (pt.max_blocks == 0) {
          const int y = static_cast<int>(row0 + (int64_t)it * kTileKeys);
#pragma unroll
          for (int pn = 0; pn < Cfg::kPanels; ++pn) {
            ptx::tma_load_2d(kt + pn * kTileKeys * 128, map_k, pn * 64, y, &full[s]);
            ptx::tma_load_2d(vt + pn * kTileKeys * 128, map_v, pn * 64, y, &full[s]);
          }
        } else {  // paged: the tile's four 16-key blocks, one box when consecutive
          const int4 y4 = kv_rows4(pt, row.cache_row, g, k0 + it * kTileKeys);
          if (rows4_contiguous(y4)) {
#pragma unroll
            for (int pn = 0; pn < Cfg::kPanels; ++pn) {
              ptx::tma_load_2d(kt + pn * kTileKeys * 128, &p.tmap_k, pn * 64, y4.x, &full[s]);
              ptx::tma_load_2d(vt + pn * kTileKeys * 128, &p.tmap_v, pn * 64, y4.x, &full[s]);
            }
          } else {
            const int ys[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
            for (int j = 0; j < kTileKeys / kBlockTokens; ++j) {
#pragma unroll
              for (int pn = 0; pn < Cfg::kPanels; ++pn) {
                const int off = pn * kTileKeys * 128 + j * kBlockTokens * 128;
                ptx::tma_load_2d(kt + off, &p.tmap_k16, pn * 64, ys[j], &full[s]);
                ptx::tma_load_2d(vt + off, &p.tmap_v16, pn * 64, ys[j], &full[s]);
              }
            }
          }
        }
        *issued = it + 1;
      }
    };
    if (lane == 0) {
      if (!p.early_kv) ptx::grid_dep_wait();
      if (seg1)
        produce(&p.tmap_k2, &p.tmap_v2);
      else
        produce(&p.tmap_k, &p.tmap_v);
    }
    return;
  }

  // Inputs, partials, tickets and the cache are read or written only after the previous
  // grid on the stream has completed; the next launch may then start.
  ptx::grid_dep_wait();
  ptx::grid_dep_launch();

  // -------------------------------------------------------------- consumers
  {
    // Rotate the decode query for the group's heads into shared memory
    // (tiny_agent/generate.py `_rope_pos`; float ops without contraction), and, in the
    // split that holds the new key, rotate it and keep it and the value plainly for the
    // store to the cache and as row 0 of the mini-tiles.  Work units: 8-pair chunks of
    // the query heads, then of the new key, then 16-byte chunks of the value; every
    // thread issues all loads of its units (and their cos/sin) before using any, so
    // the prologue costs one memory round trip.
    const __nv_bfloat16 *q = p.q + (int64_t)row.call_row * p.q_row_stride +
                             (int64_t)g * p.rep * D;
    const __nv_bfloat16 *k = (seg1 ? p.k_new2 : p.k_new) + (int64_t)row.call_row * p.kv_row_stride +
                             (int64_t)g * D;
    const __nv_bfloat16 *v = (seg1 ? p.v_new2 : p.v_new) + (int64_t)row.call_row * p.kv_row_stride +
                             (int64_t)g * D;
    const float2 *cs = p.rope + (int64_t)row.pos * kHalf;
    constexpr int kVec = kHalf / 8;                 // 8-pair chunks per head
    constexpr int kQUnits = NT * 8 * kVec;
    constexpr int kUnits = kQUnits + kVec + D / 8;  // with the new key and value
    constexpr int kPasses = (kUnits + kConsumerWarps * 32 - 1) / (kConsumerWarps * 32);
    const int n_units = owner ? kUnits : kQUnits;
    uint4 x1[kPasses], x2[kPasses];
    float4 cv[kPasses][4];
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      const int u = threadIdx.x + i * kConsumerWarps * 32;
      x1[i] = x2[i] = make_uint4(0, 0, 0, 0);
      if (u < kQUnits) {
        const int h = u / kVec, c = u % kVec;
        if (h < p.rep) {
          x1[i] = *reinterpret_cast<const uint4 *>(q + h * D + 8 * c);
          x2[i] = *reinterpret_cast<const uint4 *>(q + h * D + kHalf + 8 * c);
#pragma unroll
          for (int j = 0; j < 4; ++j) cv[i][j] = reinterpret_cast<const float4 *>(cs + 8 * c)[j];
        }
      } else if (u < kQUnits + kVec && u < n_units) {
        const int c = u - kQUnits;
        x1[i] = *reinterpret_cast<const uint4 *>(k + 8 * c);
        x2[i] = *reinterpret_cast<const uint4 *>(k + kHalf + 8 * c);
#pragma unroll
        for (int j = 0; j < 4; ++j) cv[i][j] = reinterpret_cast<const float4 *>(cs + 8 * c)[j];
      } else if (u < n_units) {
        x1[i] = *reinterpret_cast<const uint4 *>(v + 8 * (u - kQUnits - kVec));
      }
    }
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      const int u = threadIdx.x + i * kConsumerWarps * 32;
      if (u < kQUnits) {
        const int h = u / kVec, c = u % kVec;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
        if (h < p.rep) rope8r(x1[i], x2[i], cv[i], lo, hi);
        *reinterpret_cast<uint4 *>(qs + h * D + 8 * c) = lo;
        *reinterpret_cast<uint4 *>(qs + h * D + kHalf + 8 * c) = hi;
      } else if (u < kQUnits + kVec && u < n_units) {
        const int c = u - kQUnits;
        uint4 lo, hi;
        rope8r(x1[i], x2[i], cv[i], lo, hi);
        *reinterpret_cast<uint4 *>(knew + 8 * c) = lo;
        *reinterpret_cast<uint4 *>(knew + kHalf + 8 * c) = hi;
      } else if (u < n_units) {
        *reinterpret_cast<uint4 *>(vnew + 8 * (u - kQUnits - kVec)) = x1[i];
      }
    }
    consumer_sync();
    if (owner) {
      for (int u = threadIdx.x; u < kMiniRows * (D / 8); u += kConsumerWarps * 32) {
        const int r = u / (D / 8), ch = u % (D / 8);
        uint4 kv = make_uint4(0, 0, 0, 0), vv = kv;
        if (r == 0) {
          kv = *reinterpret_cast<const uint4 *>(knew + 8 * ch);
          vv = *reinterpret_cast<const uint4 *>(vnew + 8 * ch);
        }
        const uint32_t off = (ch / 8) * (kMiniRows * 128) + ptx::swz128(r, ch % 8);
        *reinterpret_cast<uint4 *>(mini_k + off) = kv;
        *reinterpret_cast<uint4 *>(mini_v + off) = vv;
      }
      consumer_sync();  // the mini-tiles are complete before warp 0 reads them
    }
  }
  const int gq = lane >> 2;  // fragment row group
  const int qq = lane & 3;   // fragment column pair

  // Q^T as the B operand (k = head dim, n = query head), fixed for the CTA.
  uint32_t qb[NT][D / 16][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const __nv_bfloat16 *qr = qs + (nt * 8 + gq) * D + 16 * kk + 2 * qq;
      qb[nt][kk][0] = *reinterpret_cast<const uint32_t *>(qr);
      qb[nt][kk][1] = *reinterpret_cast<const uint32_t *>(qr + 8);
    }

  WarpAcc<D, NT> acc;
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc.o[mt][nt][j] = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    acc.m[nt][0] = acc.m[nt][1] = -INFINITY;
    acc.l[nt][0] = acc.l[nt][1] = 0.f;
  }

  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % kStages;
    if (*fail || !ptx::mbar_wait(&full[s], (it / kStages) & 1, kWaitLimit)) {
      atomicExch(p.err, 1);
      *fail = 1;
      break;
    }
    uint8_t *kt = tiles + s * Cfg::kStageBytes;
    uint8_t *vt = kt + Cfg::kTileBytes;
    const int key_base = k0 + it * kTileKeys + 16 * warp;  // first key of this warp
    const int n_valid = k1 - key_base;                      // may be <= 0 or >= 16
    const int skip = owner ? new_slot - key_base : -1;      // stale slot of the new key
    const bool skip_here = skip >= 0 && skip < 16;

    if (n_valid < 16 || skip_here) {
      // Masked keys may hold anything (stale rows, another row's data, padding):
      // zero their V rows so that 0 * V stays 0 in the PV product.
      const int first = n_valid > 0 ? (n_valid < 16 ? n_valid : 16) : 0;
      for (int u = lane; u < (16 - first) * (D / 8); u += 32)
        zero_v_chunk(vt, kTileKeys * 128, 16 * warp + first + u / (D / 8), u % (D / 8));
      if (skip_here && skip < first)
        for (int ch = lane; ch < D / 8; ch += 32)
          zero_v_chunk(vt, kTileKeys * 128, 16 * warp + skip, ch);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }
    attend16<D, NT>(acc, qb, kt, vt, kTileKeys * 128, 16 * warp, n_valid, skip_here ? skip : -1,
                    p.scale_log2, lane);
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&empty[s]);
  }
  if (owner && warp == 0 && !*fail)  // the new key, from the mini-tile (row 0 only)
    attend16<D, NT>(acc, qb, mini_k, mini_v, kMiniRows * 128, 0, 1, -1, p.scale_log2, lane);

  // ---------------------------------------------------------------- merge warps
  // All consumers are past their last tile before the stage memory is reused.
  consumer_sync();
  if (*fail) {
    // A wait gave up: let every load this CTA issued land (bounded) before the CTA
    // retires, so no copy writes into shared memory that is no longer ours.
    if (threadIdx.x == 0) {
      const int n_issued = *issued;
      for (int s = 0; s < kStages && s < n_issued; ++s) {
        const int lst = s + ((n_issued - 1 - s) / kStages) * kStages;
        ptx::mbar_wait(&full[s], (lst / kStages) & 1, kWaitLimit);
      }
    }
    return;
  }
  if (owner) {
    // Every load of this CTA has landed: store the new key and value in the cache.
    const int64_t dst = kv_row(pt, row.cache_row, p.Hk, g, seg_rows, new_slot) * D;
    __nv_bfloat16 *ck = seg1 ? p.cache_k2 : p.cache_k, *cv = seg1 ? p.cache_v2 : p.cache_v;
    for (int ch = threadIdx.x; ch < D / 8; ch += kConsumerWarps * 32) {
      *reinterpret_cast<uint4 *>(ck + dst + 8 * ch) =
          *reinterpret_cast<const uint4 *>(knew + 8 * ch);
      *reinterpret_cast<uint4 *>(cv + dst + 8 * ch) =
          *reinterpret_cast<const uint4 *>(vnew + 8 * ch);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
        acc.l[nt][j] += __shfl_xor_sync(0xffffffffu, acc.l[nt][j], off);

  constexpr int kH = NT * 8;
  float *mw = reinterpret_cast<float *>(tiles);  // [warp][kH]
  float *lw = mw + kConsumerWarps * kH;          // [warp][kH]
  float *ow = lw + kConsumerWarps * kH;          // [warp][kH][D]
  if (gq == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mw[warp * kH + nt * 8 + 2 * qq] = acc.m[nt][0];
      mw[warp * kH + nt * 8 + 2 * qq + 1] = acc.m[nt][1];
      lw[warp * kH + nt * 8 + 2 * qq] = acc.l[nt][0];
      lw[warp * kH + nt * 8 + 2 * qq + 1] = acc.l[nt][1];
    }
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h0 = nt * 8 + 2 * qq;
      float *base = ow + (int64_t)warp * kH * D;
      base[h0 * D + 16 * mt + gq] = acc.o[mt][nt][0];
      base[(h0 + 1) * D + 16 * mt + gq] = acc.o[mt][nt][1];
      base[h0 * D + 16 * mt + gq + 8] = acc.o[mt][nt][2];
      base[(h0 + 1) * D + 16 * mt + gq + 8] = acc.o[mt][nt][3];
    }
  consumer_sync();

  const bool single = n_total == 1;
  const int64_t part = (int64_t)row.part0 + split;
  // Per head: the warps' merge weights 2^(m_w - m) (divided by l for a finished output)
  // and this split's (m, l); then 8 consecutive dims per thread, vectorised.
  float *wsm = ow + kConsumerWarps * kH * D;  // [warp][kH]
  if (threadIdx.x < p.rep) {
    const int h = threadIdx.x;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) m = fmaxf(m, mw[w * kH + h]);
    float f[kConsumerWarps], l = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      f[w] = exp2f(mw[w * kH + h] - m);  // warps without keys: exp2(-inf) = 0
      l += f[w] * lw[w * kH + h];
    }
    const float sc = single ? 1.f / l : 1.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) wsm[w * kH + h] = f[w] * sc;
    if (!single) p.part_ml[part * p.Hq + g * p.rep + h] = make_float2(m, l);
  }
  consumer_sync();
  for (int u = threadIdx.x; u < p.rep * (D / 8); u += kConsumerWarps * 32) {
    const int h = u / (D / 8), d = 8 * (u % (D / 8));
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float f = wsm[w * kH + h];
      const float4 o0 = *reinterpret_cast<const float4 *>(ow + ((int64_t)w * kH + h) * D + d);
      const float4 o1 = *reinterpret_cast<const float4 *>(ow + ((int64_t)w * kH + h) * D + d + 4);
      a[0] += f * o0.x; a[1] += f * o0.y; a[2] += f * o0.z; a[3] += f * o0.w;
      a[4] += f * o1.x; a[5] += f * o1.y; a[6] += f * o1.z; a[7] += f * o1.w;
    }
    const int hq = g * p.rep + h;
    if (single) {
      uint4 w8;
      w8.x = ptx::pack_bf16(a[0], a[1]);
      w8.y = ptx::pack_bf16(a[2], a[3]);
      w8.z = ptx::pack_bf16(a[4], a[5]);
      w8.w = ptx::pack_bf16(a[6], a[7]);
      *reinterpret_cast<uint4 *>(p.out + (int64_t)row.call_row * p.out_row_stride +
                                 (int64_t)hq * D + d) = w8;
    } else {
      float *dst = p.part_o + (part * p.Hq + hq) * D + d;
      *reinterpret_cast<float4 *>(dst) = make_float4(a[0], a[1], a[2], a[3]);
      *reinterpret_cast<float4 *>(dst + 4) = make_float4(a[4], a[5], a[6], a[7]);
    }
  }
  if (single) return;

  // ---------------------------------------------------------------- split merge
  // Publish this split's partial and take a ticket; the last split of the (row, kv
  // head) to arrive merges all of them: weights 2^(m_s - max m),
  // out = sum_s w_s O_s / sum_s w_s l_s (log-sum-exp merge of partial softmaxes).
  __threadfence();
  consumer_sync();
  int32_t *ticket = p.counters + (int64_t)row.ctr * p.Hk + g;
  if (threadIdx.x == 0) *last = atomicAdd(ticket, 1) == n_total - 1;
  consumer_sync();
  if (!*last) return;
  __threadfence();
  // Stage every split's (m, l) of the group's heads, turn them into merge weights
  // 2^(m_s - max m) / sum_s 2^(m_s - max m) l_s, then sum the weighted partials with
  // all loads of an element in flight at once.
  const int ns = n_total;
  const int64_t base = row.part0;
  float2 *wml = reinterpret_cast<float2 *>(tiles);            // [split][rep] (m, l) -> weight
  for (int u = threadIdx.x; u < ns * p.rep; u += kConsumerWarps * 32) {
    const int sp = u / p.rep, h = u % p.rep;
    wml[u] = __ldcg(&p.part_ml[(base + sp) * p.Hq + g * p.rep + h]);
  }
  consumer_sync();
  if (threadIdx.x < p.rep) {
    const int h = threadIdx.x;
    float m = -INFINITY;
    for (int sp = 0; sp < ns; ++sp) m = fmaxf(m, wml[sp * p.rep + h].x);
    float l = 0.f;
    for (int sp = 0; sp < ns; ++sp) l += exp2f(wml[sp * p.rep + h].x - m) * wml[sp * p.rep + h].y;
    const float inv = 1.f / l;
    for (int sp = 0; sp < ns; ++sp)
      wml[sp * p.rep + h].x = exp2f(wml[sp * p.rep + h].x - m) * inv;
  }
  consumer_sync();
  for (int u = threadIdx.x; u < p.rep * D; u += kConsumerWarps * 32) {
    const int h = u / D, d = u % D;
    const int hq = g * p.rep + h;
    const float *src = p.part_o + (base * p.Hq + hq) * D + d;
    const int64_t stride = (int64_t)p.Hq * D;
    float a = 0.f;
    int sp = 0;
    for (; sp + 4 <= ns; sp += 4) {
      const float x0 = __ldcg(src + (sp + 0) * stride), x1 = __ldcg(src + (sp + 1) * stride);
      const float x2 = __ldcg(src + (sp + 2) * stride), x3 = __ldcg(src + (sp + 3) * stride);
      a += wml[(sp + 0) * p.rep + h].x * x0 + wml[(sp + 1) * p.rep + h].x * x1 +
           wml[(sp + 2) * p.rep + h].x * x2 + wml[(sp + 3) * p.rep + h].x * x3;
    }
    for (; sp < ns; ++sp) a += wml[sp * p.rep + h].x * __ldcg(src + sp * stride);
    p.out[(int64_t)row.call_row * p.out_row_stride + (int64_t)hq * D + d] = __float2bfloat16_rn(a);
  }
  if (threadIdx.x == 0) *ticket = 0;  // re-armed for the next launch on the stream
}

template <int D, int NT, bool DEEP>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t s, bool pdl) {
  return launch_k(decode_kernel<D, NT, DEEP>, dim3(p.n_items, p.Hk), dim3(kThreads),
                  decode_smem_bytes<D, NT, DEEP>(), s, p, pdl);
}

template <int D, int NT, bool DEEP>
cudaError_t configure_decode_t() {
  constexpr int smem = decode_smem_bytes<D, NT, DEEP>();
  return cudaFuncSetAttribute(decode_kernel<D, NT, DEEP>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

// Function and shared memory of the variant for (D, tiles of heads, deep pipeline).
template <int D, int NT>
bool pick_t(bool deep, void **fn, int *smem) {
  if (deep) {
    *fn = reinterpret_cast<void *>(decode_kernel<D, NT, true>);
    *smem = decode_smem_bytes<D, NT, true>();
  } else {
    *fn = reinterpret_cast<void *>(decode_kernel<D, NT, false>);
    *smem = decode_smem_bytes<D, NT, false>();
  }
  return true;
}

bool pick(int D, int n_tiles_heads, bool deep, void **fn, int *smem) {
  if (D == 128) return n_tiles_heads == 1 ? pick_t<128, 1>(deep, fn, smem)
                                          : pick_t<128, 2>(deep, fn, smem);
  if (D == 64) return n_tiles_heads == 1 ? pick_t<64, 1>(deep, fn, smem)
                                         : pick_t<64, 2>(deep, fn, smem);
  return false;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, int D, int n_tiles_heads, cudaStream_t s,
                          bool pdl) {
  if (p.n_items <= 0) return cudaSuccess;
  const bool deep = p.deep_pipeline != 0;
  if (D == 128) {
    if (n_tiles_heads == 1)
      return deep ? launch_decode_t<128, 1, true>(p, s, pdl) : launch_decode_t<128, 1, false>(p, s, pdl);
    return deep ? launch_decode_t<128, 2, true>(p, s, pdl) : launch_decode_t<128, 2, false>(p, s, pdl);
  }
  if (D == 64) {
    if (n_tiles_heads == 1)
      return deep ? launch_decode_t<64, 1, true>(p, s, pdl) : launch_decode_t<64, 1, false>(p, s, pdl);
    return deep ? launch_decode_t<64, 2, true>(p, s, pdl) : launch_decode_t<64, 2, false>(p, s, pdl);
  }
  return cudaErrorInvalidValue;
}

// The same launch as a graph kernel node: function, grid, block, shared memory and the one
// argument (the node copies *p when it is added or its parameters are set).
cudaError_t decode_node(const DecodeParams *p, int D, int n_tiles_heads, void **args,
                        cudaKernelNodeParams *kp) {
  if (p->n_items <= 0) return cudaErrorInvalidValue;
  args[0] = const_cast<DecodeParams *>(p);
  kp->gridDim = dim3(p->n_items, p->Hk);
  kp->blockDim = dim3(kThreads);
  kp->kernelParams = args;
  kp->extra = nullptr;
  int smem = 0;
  if (!pick(D, n_tiles_heads, p->deep_pipeline != 0, &kp->func, &smem))
    return cudaErrorInvalidValue;
  kp->sharedMemBytes = smem;
  return cudaSuccess;
}

cudaError_t configure_decode() {
  cudaError_t e;
  if ((e = configure_decode_t<128, 1, false>()) != cudaSuccess) return e;
  if ((e = configure_decode_t<128, 2, false>()) != cudaSuccess) return e;
  if ((e = configure_decode_t<64, 1, false>()) != cudaSuccess) return e;
  if ((e = configure_decode_t<64, 2, false>()) != cudaSuccess) return e;
  if ((e = configure_decode_t<128, 1, true>()) != cudaSuccess) return e;
  if ((e = configure_decode_t<128, 2, true>()) != cudaSuccess) return e;
  if ((e = configure_decode_t<64, 1, true>()) != cudaSuccess) return e;
  return configure_decode_t<64, 2, true>();
}

}  // namespace kvinc
