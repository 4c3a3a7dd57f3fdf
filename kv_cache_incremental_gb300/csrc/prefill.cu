// prefill.cu -- chunked prefill: attention of a chunk's queries against the
// cache plus the chunk's own keys, on the tensor cores.
//
// Query row rho of a (row, kv head) is token t = rho / rep, head h = rho % rep
// of the GQA group, at absolute position p = lens + t.  One CTA owns 64 query
// rows (4 consumer warps x 16); a producer warp streams key tiles with TMA.
// Per warp: S = Q K^T (16 rows x 64 keys), float online softmax per row,
// O += P V with P split into bf16 high and low parts.
//
// Key sources ("inkling: ring-buffer KV cache for sliding-window layers", How
// it works; Lab 07 section 3; pycraft-1 `build_attn_mask`):
//  - global layer: cache slots [0, lens + t_max] -- the append kernel already
//    stored this chunk's keys at their positions; key j is visible iff j <= p.
//  - sliding layer: the ring's occupied slots [0, min(lens, R)), slot s holding
//    position P(s) = largest t < lens with t % R == s, then the chunk scratch
//    (rows 0..t_max, position lens + j).  The ring is read before this chunk is
//    committed to it, so a chunk longer than the window cannot overwrite
//    history its own earlier queries still need.  Key position j is visible
//    iff j <= p and p - j < W.
#include "kvinc_internal.h"
#include "ptx.cuh"

namespace kvinc {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kRowsPerCta = 16 * kConsumerWarps;

template <int D>
struct PrefillCfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kTileBytes = kPanels * kTileKeys * 128;
  static constexpr int kStages = D == 128 ? 3 : 5;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kQBytes = kPanels * kRowsPerCta * 128;  // swizzled like the key tiles
};

template <int D>
constexpr int prefill_smem_bytes() {
  using C = PrefillCfg<D>;
  return 1024 + C::kStages * C::kStageBytes + C::kQBytes + 2 * C::kStages * 8 + 16;
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ int find_cta_row(const PrefillParams &p, int b) {
  int lo = 0, hi = p.n_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.rows[mid].cta0 <= b) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <int D>
__global__ void __launch_bounds__(kThreads) prefill_kernel(const __grid_constant__ PrefillParams p) {
  ptx::grid_dep_wait();  // the previous grid on the stream has completed
  ptx::grid_dep_launch();
  using Cfg = PrefillCfg<D>;
  constexpr int kStages = Cfg::kStages;
  constexpr int kHalf = D / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *tiles = smem;
  uint8_t *qsm = smem + kStages * Cfg::kStageBytes;
  uint64_t *full = reinterpret_cast<uint64_t *>(qsm + Cfg::kQBytes);
  uint64_t *empty = full + kStages;
  volatile int *fail = reinterpret_cast<volatile int *>(empty + kStages);
  volatile int *issued = fail + 1;

  const PrefillRow &row = p.rows[find_cta_row(p, blockIdx.x)];
  const int g = blockIdx.y;
  const int rho0 = (blockIdx.x - row.cta0) * kRowsPerCta;  // first query row of the CTA
  const int n_rho = row.n * p.rep;
  const int rho_last = min(n_rho, rho0 + kRowsPerCta) - 1;
  const int t_max = rho_last / p.rep;  // last token any row of this CTA needs
  const int lens = row.lens;
  // Ring slot s holds position s + ring_base, less R when s > ring_rem: the largest
  // position below lens congruent to s modulo R (every slot is occupied once lens >= R).
  const int ring_base = (lens > p.ring_R && p.ring_R > 0) ? ((lens - 1) / p.ring_R) * p.ring_R : 0;
  const int ring_rem = (lens > p.ring_R && p.ring_R > 0) ? (lens - 1) % p.ring_R : 0x7fffffff;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Key segments: A = layer storage, B = chunk scratch (sliding layers only).
  const int len_a = p.sliding ? min(lens, p.ring_R) : lens + t_max + 1;
  const int len_b = p.sliding ? t_max + 1 : 0;
  const int tiles_a = (len_a + kTileKeys - 1) / kTileKeys;
  const int n_tiles = tiles_a + (len_b + kTileKeys - 1) / kTileKeys;
  // This entry's tiles [j_begin, j_end): a key split, or all of them.
  const int j_begin = row.tile0, j_end = min(row.tile1, n_tiles);
  const int n_local = max(0, j_end - j_begin);
  const int64_t base_a = ((int64_t)row.cache_row * p.Hk + g) * p.seg_rows;
  const int64_t base_b = ((int64_t)row.cache_row * p.Hk + g) * kChunk;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], kConsumerWarps);
    }
    *fail = 0;
    *issued = 0;
    ptx::fence_barrier_init();
  }
  if (warp < kConsumerWarps) {
    // Rotated queries of the CTA's 64 rows, stored in 128-byte swizzled panels.
    for (int u = threadIdx.x; u < kRowsPerCta * (kHalf / 8); u += kConsumerWarps * 32) {
      const int r = u / (kHalf / 8), c = u % (kHalf / 8);
      const int rho = rho0 + r;
      uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
      if (rho < n_rho) {
        const int t = rho / p.rep, h = rho % p.rep;
        const __nv_bfloat16 *q = p.q + (int64_t)row.call_row * p.q_row_stride +
                                 ((int64_t)t * p.Hq + g * p.rep + h) * D;
        const uint4 x1v = *reinterpret_cast<const uint4 *>(q + 8 * c);
        const uint4 x2v = *reinterpret_cast<const uint4 *>(q + kHalf + 8 * c);
        const __nv_bfloat16 *x1 = reinterpret_cast<const __nv_bfloat16 *>(&x1v);
        const __nv_bfloat16 *x2 = reinterpret_cast<const __nv_bfloat16 *>(&x2v);
        __nv_bfloat16 *o1 = reinterpret_cast<__nv_bfloat16 *>(&lo);
        __nv_bfloat16 *o2 = reinterpret_cast<__nv_bfloat16 *>(&hi);
        const float2 *cs = p.rope + (int64_t)(lens + t) * kHalf + 8 * c;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float a = __bfloat162float(x1[j]), b = __bfloat162float(x2[j]);
          const float2 e = cs[j];
          o1[j] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(a, e.x), __fmul_rn(b, e.y)));
          o2[j] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(a, e.y), __fmul_rn(b, e.x)));
        }
      }
      const int c_lo = c, c_hi = kHalf / 8 + c;  // 16-byte chunk index along D
      *reinterpret_cast<uint4 *>(qsm + (c_lo / 8) * kRowsPerCta * 128 + ptx::swz128(r, c_lo % 8)) = lo;
      *reinterpret_cast<uint4 *>(qsm + (c_hi / 8) * kRowsPerCta * 128 + ptx::swz128(r, c_hi % 8)) = hi;
    }
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      ptx::prefetch_tmap(&p.tmap_k);
      ptx::prefetch_tmap(&p.tmap_v);
      for (int it = 0; it < n_local; ++it) {
        const int s = it % kStages;
        if (it >= kStages &&
            !ptx::mbar_wait(&empty[s], ((it / kStages) - 1) & 1, kWaitLimit)) {
          atomicExch(p.err, 1);  // consumers then give up on the tiles never loaded
          break;
        }
        uint8_t *kt = tiles + s * Cfg::kStageBytes;
        uint8_t *vt = kt + Cfg::kTileBytes;
        const int jt = j_begin + it;  // tile of the row's key space
        const bool in_a = jt < tiles_a;
        const CUtensorMap *mk = in_a ? &p.tmap_k : &p.tmap_sk;
        const CUtensorMap *mv = in_a ? &p.tmap_v : &p.tmap_sv;
        const int y = static_cast<int>(in_a ? base_a + (int64_t)jt * kTileKeys
                                            : base_b + (int64_t)(jt - tiles_a) * kTileKeys);
        ptx::mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
        int4 y4 = make_int4(y, y + kBlockTokens, y + 2 * kBlockTokens, y + 3 * kBlockTokens);
        if (in_a && p.pt.max_blocks) y4 = kv_rows4(p.pt, row.cache_row, g, jt * kTileKeys);
        if (rows4_contiguous(y4)) {  // dense, or a paged tile of consecutive blocks
#pragma unroll
          for (int pn = 0; pn < Cfg::kPanels; ++pn) {
            ptx::tma_load_2d(kt + pn * kTileKeys * 128, mk, pn * 64, y4.x, &full[s]);
            ptx::tma_load_2d(vt + pn * kTileKeys * 128, mv, pn * 64, y4.x, &full[s]);
          }
        } else {  // paged: four 16-key blocks, 16-row boxes
          const int ys[4] = {y4.x, y4.y, y4.z, y4.w};
#pragma unroll
          for (int j = 0; j < kTileKeys / kBlockTokens; ++j)
#pragma unroll
            for (int pn = 0; pn < Cfg::kPanels; ++pn) {
              const int off = pn * kTileKeys * 128 + j * kBlockTokens * 128;
              ptx::tma_load_2d(kt + off, &p.tmap_k16, pn * 64, ys[j], &full[s]);
              ptx::tma_load_2d(vt + off, &p.tmap_v16, pn * 64, ys[j], &full[s]);
            }
        }
        *issued = it + 1;
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int gq = lane >> 2, qq = lane & 3;
  // A fragments of the warp's 16 query rows (k = head dim).
  uint32_t qa[D / 16][4];
  {
    const int mrow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int ch = 2 * (kk % 4) + (lane >> 4);
      ptx::ldsm_x4(ptx::smem_u32(qsm + (kk / 4) * kRowsPerCta * 128) + ptx::swz128(mrow, ch),
                   qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
    }
  }
  // Positions of the lane's two query rows (gq and gq + 8 of the warp's 16).
  int qpos[2];
  bool qvalid[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int rho = rho0 + 16 * warp + gq + 8 * j;
    qvalid[j] = rho < n_rho;
    qpos[j] = lens + (qvalid[j] ? rho / p.rep : 0);
  }

  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  for (int it = 0; it < n_local; ++it) {
    const int s = it % kStages;
    // After a give-up the loop keeps running without waiting or computing, so that
    // every consumer warp passes the same named barriers in the same order.
    const bool have = !*fail && ptx::mbar_wait(&full[s], (it / kStages) & 1, kWaitLimit);
    if (!have && !*fail) {
      atomicExch(p.err, 1);
      *fail = 1;
    }
    uint8_t *kt = tiles + s * Cfg::kStageBytes;
    uint8_t *vt = kt + Cfg::kTileBytes;
    const int jt = j_begin + it;
    const bool in_a = jt < tiles_a;
    const int kb = (in_a ? jt : jt - tiles_a) * kTileKeys;  // first key index of the tile
    const int seg_len = in_a ? len_a : len_b;
    const int n_valid = seg_len - kb;

    if (n_valid < kTileKeys) {
      // Keys past the segment may hold anything: zero their V rows (all warps read
      // every key of the tile, so the consumers do it together and then sync).
      if (have)
        for (int u = threadIdx.x; u < (kTileKeys - n_valid) * (D / 8); u += kConsumerWarps * 32) {
          const int r = n_valid + u / (D / 8), ch = u % (D / 8);
          *reinterpret_cast<uint4 *>(vt + (ch / 8) * kTileKeys * 128 + ptx::swz128(r, ch % 8)) =
              make_uint4(0, 0, 0, 0);
        }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      consumer_sync();
    }
    if (!have) continue;

    // S = Q K^T : 16 rows x 64 keys (8 n-tiles of 8 keys)
    float sc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
    {
      const int mi = lane >> 3;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {  // pairs of n-tiles
          const int key = 16 * jp + 8 * (mi >> 1) + (lane & 7);
          const int ch = 2 * (kk % 4) + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ptx::ldsm_x4(ptx::smem_u32(kt + (kk / 4) * kTileKeys * 128) + ptx::swz128(key, ch), b0,
                       b1, b2, b3);
          ptx::mma_bf16(sc[2 * jp], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          ptx::mma_bf16(sc[2 * jp + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
      }
    }

    // Mask, scale and the online softmax of the lane's two rows.
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rj = e >> 1;                      // 0: row gq, 1: row gq + 8
        const int kidx = kb + 8 * j + 2 * qq + (e & 1);
        bool vis = qvalid[rj] && kidx < seg_len;
        if (vis) {
          int kpos;
          if (!p.sliding) kpos = kidx;
          else if (!in_a) kpos = lens + kidx;
          else kpos = kidx + ring_base - (kidx > ring_rem ? p.ring_R : 0);
          vis = kpos <= qpos[rj] && (!p.sliding || qpos[rj] - kpos < p.window);
        }
        sc[j][e] = vis ? sc[j][e] * p.scale_log2 : -INFINITY;
        mx[rj] = fmaxf(mx[rj], sc[j][e]);
      }
    }
    float al[2], bs[2];
#pragma unroll
    for (int rj = 0; rj < 2; ++rj) {
      mx[rj] = fmaxf(mx[rj], __shfl_xor_sync(0xffffffffu, mx[rj], 1));
      mx[rj] = fmaxf(mx[rj], __shfl_xor_sync(0xffffffffu, mx[rj], 2));
      const float mn = fmaxf(m_run[rj], mx[rj]);
      bs[rj] = mn == -INFINITY ? 0.f : mn;
      al[rj] = exp2f(m_run[rj] - bs[rj]);
      m_run[rj] = mn;
      l_run[rj] *= al[rj];
    }
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      o[nd][0] *= al[0];
      o[nd][1] *= al[0];
      o[nd][2] *= al[1];
      o[nd][3] *= al[1];
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        sc[j][e] = exp2f(sc[j][e] - bs[e >> 1]);
        l_run[e >> 1] += sc[j][e];
      }
    }

    // O += P V over 4 key steps of 16; P as the A operand (high + low bf16 parts).
    {
      const int mi = lane >> 3;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t ah[4], alo[4];
        ptx::split_bf16(sc[2 * ks][0], sc[2 * ks][1], ah[0], alo[0]);
        ptx::split_bf16(sc[2 * ks][2], sc[2 * ks][3], ah[1], alo[1]);
        ptx::split_bf16(sc[2 * ks + 1][0], sc[2 * ks + 1][1], ah[2], alo[2]);
        ptx::split_bf16(sc[2 * ks + 1][2], sc[2 * ks + 1][3], ah[3], alo[3]);
        const int key = 16 * ks + (lane & 7) + (mi & 1) * 8;
#pragma unroll
        for (int ndp = 0; ndp < D / 16; ++ndp) {  // pairs of 8-wide dim tiles
          const int ch = 2 * ndp + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ptx::ldsm_x4_t(ptx::smem_u32(vt + (ch / 8) * kTileKeys * 128) + ptx::swz128(key, ch % 8),
                         b0, b1, b2, b3);
          ptx::mma_bf16(o[2 * ndp], ah[0], ah[1], ah[2], ah[3], b0, b1);
          ptx::mma_bf16(o[2 * ndp], alo[0], alo[1], alo[2], alo[3], b0, b1);
          ptx::mma_bf16(o[2 * ndp + 1], ah[0], ah[1], ah[2], ah[3], b2, b3);
          ptx::mma_bf16(o[2 * ndp + 1], alo[0], alo[1], alo[2], alo[3], b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&empty[s]);
  }

  consumer_sync();
  if (*fail) {
    if (threadIdx.x == 0) {
      const int n_issued = *issued;
      for (int s = 0; s < kStages && s < n_issued; ++s) {
        const int last = s + ((n_issued - 1 - s) / kStages) * kStages;
        ptx::mbar_wait(&full[s], (last / kStages) & 1, kWaitLimit);
      }
    }
    return;
  }

#pragma unroll
  for (int rj = 0; rj < 2; ++rj) {
    l_run[rj] += __shfl_xor_sync(0xffffffffu, l_run[rj], 1);
    l_run[rj] += __shfl_xor_sync(0xffffffffu, l_run[rj], 2);
  }
  if (row.part >= 0) {
    // A key split: unnormalised O of the lane's dims, the row's maximum (log2 units), sum.
#pragma unroll
    for (int rj = 0; rj < 2; ++rj) {
      const int rho = rho0 + 16 * warp + gq + 8 * rj;
      if (rho >= n_rho) continue;
      const int64_t vec = (int64_t)row.part + (int64_t)g * n_rho + rho;
      float *po = p.part_o + vec * D;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd)
        *reinterpret_cast<float2 *>(po + 8 * nd + 2 * qq) =
            make_float2(o[nd][2 * rj], o[nd][2 * rj + 1]);
      if (qq == 0) p.part_ml[vec] = make_float2(m_run[rj], l_run[rj]);
    }
    return;
  }
#pragma unroll
  for (int rj = 0; rj < 2; ++rj) {
    const int rho = rho0 + 16 * warp + gq + 8 * rj;
    if (rho >= n_rho) continue;
    const int t = rho / p.rep, h = rho % p.rep;
    __nv_bfloat16 *dst = p.out + (int64_t)row.call_row * p.out_row_stride +
                         ((int64_t)t * p.Hq + g * p.rep + h) * D;
    const float inv = 1.f / l_run[rj];
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      const float x0 = o[nd][2 * rj] * inv, x1 = o[nd][2 * rj + 1] * inv;
      *reinterpret_cast<__nv_bfloat162 *>(dst + 8 * nd + 2 * qq) = __floats2bfloat162_rn(x0, x1);
    }
  }
}

__device__ __forceinline__ int find_merge_row(const MergeParams &p, int v) {
  int lo = 0, hi = p.n_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.rows[mid].vec0 <= v) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

constexpr int kMergeWarps = 8;

// One warp per (row, kv head, query row) vector: the log-sum-exp merge of the row's key
// splits (a split in which the query row sees no key has m = -inf and weighs nothing).
// Every split's (m, l) and then every split's slice of O are loaded before any is used, so
// a vector costs two memory round trips whatever its split count.
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32)
    prefill_merge_kernel(const __grid_constant__ MergeParams p) {
  ptx::grid_dep_wait();  // the previous grid on the stream has completed
  ptx::grid_dep_launch();
  constexpr int kPer = D / 32;  // dims per lane
  const int v = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (v >= p.n_vec) return;
  const MergeRow &row = p.rows[find_merge_row(p, v)];
  const int local = v - row.vec0;  // g * n_rho + rho
  const int g = local / row.n_rho, rho = local % row.n_rho;
  const int64_t stride = (int64_t)p.Hk * row.n_rho;
  const int ns = row.n_splits;
  float2 ml[kMaxPrefillSplits];
#pragma unroll
  for (int sp = 0; sp < kMaxPrefillSplits; ++sp)
    ml[sp] = sp < ns ? p.part_ml[row.part + sp * stride + local] : make_float2(-INFINITY, 0.f);
  float o[kMaxPrefillSplits][kPer];
#pragma unroll
  for (int sp = 0; sp < kMaxPrefillSplits; ++sp) {
#pragma unroll
    for (int i = 0; i < kPer; ++i) o[sp][i] = 0.f;
    if (sp < ns) {
      const float *po = p.part_o + (row.part + sp * stride + local) * D + kPer * lane;
      if (kPer == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(po);
        o[sp][0] = x.x;
        o[sp][1] = x.y;
        o[sp][2 % kPer] = x.z;
        o[sp][3 % kPer] = x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2 *>(po);
        o[sp][0] = x.x;
        o[sp][1] = x.y;
      }
    }
  }
  float m_max = -INFINITY;
#pragma unroll
  for (int sp = 0; sp < kMaxPrefillSplits; ++sp) m_max = fmaxf(m_max, ml[sp].x);
  float acc[kPer] = {};
  float l = 0.f;
#pragma unroll
  for (int sp = 0; sp < kMaxPrefillSplits; ++sp) {
    const float w = ml[sp].x == -INFINITY ? 0.f : exp2f(ml[sp].x - m_max);
    l += w * ml[sp].y;
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] += w * o[sp][i];
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int t = rho / p.rep, h = rho % p.rep;
  __nv_bfloat16 *dst = p.out + (int64_t)row.call_row * p.out_row_stride +
                       ((int64_t)t * p.Hq + g * p.rep + h) * D + kPer * lane;
  if (kPer == 4) {
    uint2 w;
    w.x = ptx::pack_bf16(acc[0] * inv, acc[1] * inv);
    w.y = ptx::pack_bf16(acc[2 % kPer] * inv, acc[3 % kPer] * inv);
    *reinterpret_cast<uint2 *>(dst) = w;
  } else {
    *reinterpret_cast<uint32_t *>(dst) = ptx::pack_bf16(acc[0] * inv, acc[1] * inv);
  }
}

template <int D>
cudaError_t launch_prefill_t(const PrefillParams &p, cudaStream_t s, bool pdl) {
  return launch_k(prefill_kernel<D>, dim3(p.n_ctas, p.Hk), dim3(kThreads),
                  prefill_smem_bytes<D>(), s, p, pdl);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams &p, int D, cudaStream_t s, bool pdl) {
  if (p.n_ctas <= 0) return cudaSuccess;
  if (D == 128) return launch_prefill_t<128>(p, s, pdl);
  if (D == 64) return launch_prefill_t<64>(p, s, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_merge(const MergeParams &p, int D, cudaStream_t s, bool pdl) {
  if (p.n_vec <= 0) return cudaSuccess;
  const dim3 blocks((p.n_vec + kMergeWarps - 1) / kMergeWarps), threads(kMergeWarps * 32);
  if (D == 128) return launch_k(prefill_merge_kernel<128>, blocks, threads, 0, s, p, pdl);
  if (D == 64) return launch_k(prefill_merge_kernel<64>, blocks, threads, 0, s, p, pdl);
  return cudaErrorInvalidValue;
}

cudaError_t configure_prefill() {
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<128>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       prefill_smem_bytes<128>());
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(prefill_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              prefill_smem_bytes<64>());
}

}  // namespace kvinc
