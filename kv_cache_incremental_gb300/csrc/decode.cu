// decode.cu -- split-K grouped-query decode attention against the cache.
//
// One CTA owns one (row, kv head, key split).  A producer warp streams the
// split's K and V rows through a multi-stage shared-memory ring with TMA 2-D
// tile loads (128-byte swizzle, one mbarrier per stage); four consumer warps
// each take 16 keys of every 64-key tile.  For the whole GQA group at once a
// warp computes S^T = K Q^T on the tensor cores (keys on the MMA's M side,
// the group's query heads on N), keeps a per-warp online softmax in float,
// and accumulates O^T = V^T P^T with P split into a bf16 high and low part so
// that the probabilities keep ~16 significant bits.  Warps merge at the end;
// a split either writes the normalised bf16 output (single split) or a float
// partial (m, l, O) for the combine pass.
//
// What is computed follows tiny_agent/generate.py `_append_chunk` (grouped
// queries straight against the cache, scale 1/sqrt(D), float softmax) and the
// inkling ring-buffer pull request (the sliding scan covers the last W
// positions): for a decode token at position p the visible keys are storage
// slots [0, nk) with nk = p + 1 (global) or min(p + 1, R) (sliding ring, where
// the ring holds exactly positions max(0, p - W + 1) .. p once the new key is
// written).  The order of keys does not change a softmax, so slots are read in
// storage order.
#include "kvinc_internal.h"
#include "ptx.cuh"

namespace kvinc {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <int D>
struct DecodeCfg {
  static constexpr int kPanels = D / 64;                        // 128-byte swizzle panels
  static constexpr int kTileBytes = kPanels * kTileKeys * 128;  // one K or V tile
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kStageBytes = 2 * kTileBytes;
};

template <int D, int NT>
constexpr int decode_smem_bytes() {
  using C = DecodeCfg<D>;
  return 1024 /*alignment slack*/ + C::kStages * C::kStageBytes + NT * 8 * D * 2 /*Q*/ +
         2 * C::kStages * 8 /*barriers*/ + 16 /*flags*/;
}

__device__ __forceinline__ int find_item_row(const DecodeParams &p, int item) {
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
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ DecodeParams p) {
  using Cfg = DecodeCfg<D>;
  constexpr int kStages = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *tiles = smem;                                       // [stage][K tile | V tile]
  __nv_bfloat16 *qs = reinterpret_cast<__nv_bfloat16 *>(smem + kStages * Cfg::kStageBytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * Cfg::kStageBytes + NT * 8 * D * 2);
  uint64_t *empty = full + kStages;
  volatile int *fail = reinterpret_cast<volatile int *>(empty + kStages);  // any wait gave up
  volatile int *issued = fail + 1;                                          // tiles loaded

  const int item = blockIdx.x;
  const int g = blockIdx.y;
  const DecodeRow &row = p.rows[find_item_row(p, item)];
  const int split = item - row.item0;
  const int k0 = split * row.split_len;
  const int k1 = min(row.nk, k0 + row.split_len);
  const int n_tiles = (k1 - k0 + kTileKeys - 1) / kTileKeys;
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
  if (warp < kConsumerWarps) {
    // Rotate this row's decode query for the group's heads into shared memory
    // (tiny_agent/generate.py `_rope_pos`; float ops without contraction).
    constexpr int kHalf = D / 2;
    const __nv_bfloat16 *q = p.q + (int64_t)row.call_row * p.q_row_stride +
                             (int64_t)g * p.rep * D;
    const float2 *cs = p.rope + (int64_t)row.pos * kHalf;
    for (int u = threadIdx.x; u < NT * 8 * kHalf; u += kConsumerWarps * 32) {
      const int h = u / kHalf, i = u % kHalf;
      __nv_bfloat16 lo = __float2bfloat16_rn(0.f), hi = lo;
      if (h < p.rep) {
        const float a = __bfloat162float(q[h * D + i]);
        const float b = __bfloat162float(q[h * D + i + kHalf]);
        const float2 c = cs[i];
        lo = __float2bfloat16_rn(__fsub_rn(__fmul_rn(a, c.x), __fmul_rn(b, c.y)));
        hi = __float2bfloat16_rn(__fadd_rn(__fmul_rn(a, c.y), __fmul_rn(b, c.x)));
      }
      qs[h * D + i] = lo;
      qs[h * D + i + kHalf] = hi;
    }
  }
  __syncthreads();

  const int64_t row0 = ((int64_t)row.cache_row * p.Hk + g) * p.seg_rows + k0;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      ptx::prefetch_tmap(&p.tmap_k);
      ptx::prefetch_tmap(&p.tmap_v);
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
        const int y = static_cast<int>(row0 + (int64_t)it * kTileKeys);
#pragma unroll
        for (int pn = 0; pn < Cfg::kPanels; ++pn) {
          ptx::tma_load_2d(kt + pn * kTileKeys * 128, &p.tmap_k, pn * 64, y, &full[s]);
          ptx::tma_load_2d(vt + pn * kTileKeys * 128, &p.tmap_v, pn * 64, y, &full[s]);
        }
        *issued = it + 1;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
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

  float o[D / 16][NT][4];
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) o[mt][nt][j] = 0.f;
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
  }

  bool ok = true;
  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % kStages;
    if (*fail || !ptx::mbar_wait(&full[s], (it / kStages) & 1, kWaitLimit)) {
      atomicExch(p.err, 1);
      *fail = 1;
      ok = false;
      break;
    }
    uint8_t *kt = tiles + s * Cfg::kStageBytes;
    uint8_t *vt = kt + Cfg::kTileBytes;
    const int key_base = k0 + it * kTileKeys + 16 * warp;  // first key of this warp
    const int n_valid = k1 - key_base;                      // may be <= 0 or >= 16

    if (n_valid < 16) {
      // Masked keys may hold anything (stale rows, another row's data, padding):
      // zero their V rows so that 0 * V stays 0 in the PV product.
      const int first = n_valid > 0 ? n_valid : 0;
      for (int u = lane; u < (16 - first) * (D / 8); u += 32) {
        const int r = 16 * warp + first + u / (D / 8);
        const int ch = u % (D / 8);
        *reinterpret_cast<uint4 *>(vt + (ch / 8) * kTileKeys * 128 + ptx::swz128(r, ch % 8)) =
            make_uint4(0, 0, 0, 0);
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }

    // S^T (16 keys x 8 heads per n-tile) = K Q^T
    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
    {
      const int mrow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int ch = 2 * (kk % 4) + (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ptx::ldsm_x4(ptx::smem_u32(kt + (kk / 4) * kTileKeys * 128) + ptx::swz128(mrow, ch), a0,
                     a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          ptx::mma_bf16(sacc[nt], a0, a1, a2, a3, qb[nt][kk][0], qb[nt][kk][1]);
      }
    }

    // Online softmax for the lane's two heads (columns 2qq, 2qq+1 of each n-tile).
    const bool va = gq < n_valid, vb = gq + 8 < n_valid;
    uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float t0 = va ? sacc[nt][0] * p.scale_log2 : -INFINITY;
      float t1 = va ? sacc[nt][1] * p.scale_log2 : -INFINITY;
      float t2 = vb ? sacc[nt][2] * p.scale_log2 : -INFINITY;
      float t3 = vb ? sacc[nt][3] * p.scale_log2 : -INFINITY;
      float mx0 = fmaxf(t0, t2), mx1 = fmaxf(t1, t3);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
      const float b0 = mn0 == -INFINITY ? 0.f : mn0;
      const float b1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m_run[nt][0] - b0), al1 = exp2f(m_run[nt][1] - b1);
      const float p0 = exp2f(t0 - b0), p1 = exp2f(t1 - b1);
      const float p2 = exp2f(t2 - b0), p3 = exp2f(t3 - b1);
      m_run[nt][0] = mn0;
      m_run[nt][1] = mn1;
      l_run[nt][0] = l_run[nt][0] * al0 + (p0 + p2);
      l_run[nt][1] = l_run[nt][1] * al1 + (p1 + p3);
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        o[mt][nt][0] *= al0;
        o[mt][nt][1] *= al1;
        o[mt][nt][2] *= al0;
        o[mt][nt][3] *= al1;
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

    // O^T (head dim x heads) += V^T P^T
    {
      const int mi = lane >> 3;
      const int vrow = 16 * warp + (lane & 7) + (mi >> 1) * 8;
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        const int ch = 2 * (mt % 4) + (mi & 1);
        uint32_t a0, a1, a2, a3;
        ptx::ldsm_x4_t(ptx::smem_u32(vt + (mt / 4) * kTileKeys * 128) + ptx::swz128(vrow, ch),
                       a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          ptx::mma_bf16(o[mt][nt], a0, a1, a2, a3, bh[nt][0], bh[nt][1]);
          ptx::mma_bf16(o[mt][nt], a0, a1, a2, a3, bl[nt][0], bl[nt][1]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(&empty[s]);
  }

  // ---------------------------------------------------------------- merge warps
  // All consumers are past their last tile before the stage memory is reused.
  consumer_sync();
  if (*fail) {
    // A wait gave up: let every load this CTA issued land (bounded) before the CTA
    // retires, so no copy writes into shared memory that is no longer ours.
    if (threadIdx.x == 0) {
      const int n_issued = *issued;
      for (int s = 0; s < kStages && s < n_issued; ++s) {
        const int last = s + ((n_issued - 1 - s) / kStages) * kStages;
        ptx::mbar_wait(&full[s], (last / kStages) & 1, kWaitLimit);
      }
    }
    return;
  }
  (void)ok;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
        l_run[nt][j] += __shfl_xor_sync(0xffffffffu, l_run[nt][j], off);

  constexpr int kH = NT * 8;
  float *mw = reinterpret_cast<float *>(tiles);  // [warp][kH]
  float *lw = mw + kConsumerWarps * kH;          // [warp][kH]
  float *ow = lw + kConsumerWarps * kH;          // [warp][kH][D]
  if (gq == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      mw[warp * kH + nt * 8 + 2 * qq] = m_run[nt][0];
      mw[warp * kH + nt * 8 + 2 * qq + 1] = m_run[nt][1];
      lw[warp * kH + nt * 8 + 2 * qq] = l_run[nt][0];
      lw[warp * kH + nt * 8 + 2 * qq + 1] = l_run[nt][1];
    }
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h0 = nt * 8 + 2 * qq;
      float *base = ow + (int64_t)warp * kH * D;
      base[h0 * D + 16 * mt + gq] = o[mt][nt][0];
      base[(h0 + 1) * D + 16 * mt + gq] = o[mt][nt][1];
      base[h0 * D + 16 * mt + gq + 8] = o[mt][nt][2];
      base[(h0 + 1) * D + 16 * mt + gq + 8] = o[mt][nt][3];
    }
  consumer_sync();

  const bool single = row.n_splits == 1;
  for (int u = threadIdx.x; u < p.rep * D; u += kConsumerWarps * 32) {
    const int h = u / D, d = u % D;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) m = fmaxf(m, mw[w * kH + h]);
    float l = 0.f, acc = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float f = exp2f(mw[w * kH + h] - m);  // warps without keys: exp2(-inf) = 0
      l += f * lw[w * kH + h];
      acc += f * ow[((int64_t)w * kH + h) * D + d];
    }
    const int hq = g * p.rep + h;
    if (single) {
      p.out[(int64_t)row.call_row * p.out_row_stride + (int64_t)hq * D + d] =
          __float2bfloat16_rn(acc / l);
    } else {
      const int64_t part = (int64_t)row.part0 + split;
      p.part_o[(part * p.Hq + hq) * D + d] = acc;
      if (d == 0) p.part_ml[part * p.Hq + hq] = make_float2(m, l);
    }
  }
}

// Merge the splits of each multi-split row: weights 2^(m_s - max m), output
// sum_s w_s O_s / sum_s w_s l_s (the log-sum-exp merge of partial softmaxes).
__global__ void __launch_bounds__(128) combine_kernel(const __grid_constant__ CombineParams p) {
  const int r = blockIdx.x, h = blockIdx.y;
  const int n = p.n_splits[r];
  const int64_t base = p.part0[r];
  float m = -INFINITY;
  for (int s = 0; s < n; ++s) m = fmaxf(m, p.part_ml[(base + s) * p.Hq + h].x);
  for (int d = threadIdx.x; d < p.D; d += blockDim.x) {
    float l = 0.f, acc = 0.f;
    for (int s = 0; s < n; ++s) {
      const float2 ml = p.part_ml[(base + s) * p.Hq + h];
      const float f = exp2f(ml.x - m);
      l += f * ml.y;
      acc += f * p.part_o[((base + s) * p.Hq + h) * p.D + d];
    }
    p.out[(int64_t)p.call_row[r] * p.out_row_stride + (int64_t)h * p.D + d] =
        __float2bfloat16_rn(acc / l);
  }
}

template <int D, int NT>
cudaError_t launch_decode_t(const DecodeParams &p, cudaStream_t s) {
  constexpr int smem = decode_smem_bytes<D, NT>();
  decode_kernel<D, NT><<<dim3(p.n_items, p.Hk), kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int D, int NT>
cudaError_t configure_decode_t() {
  constexpr int smem = decode_smem_bytes<D, NT>();
  return cudaFuncSetAttribute(decode_kernel<D, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams &p, int D, int n_tiles_heads, cudaStream_t s) {
  if (p.n_items <= 0) return cudaSuccess;
  if (D == 128) return n_tiles_heads == 1 ? launch_decode_t<128, 1>(p, s) : launch_decode_t<128, 2>(p, s);
  if (D == 64) return n_tiles_heads == 1 ? launch_decode_t<64, 1>(p, s) : launch_decode_t<64, 2>(p, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_combine(const CombineParams &p, cudaStream_t s) {
  if (p.n_rows <= 0) return cudaSuccess;
  combine_kernel<<<dim3(p.n_rows, p.Hq), 128, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t configure_decode() {
  cudaError_t e;
  if ((e = configure_decode_t<128, 1>()) != cudaSuccess) return e;
  if ((e = configure_decode_t<128, 2>()) != cudaSuccess) return e;
  if ((e = configure_decode_t<64, 1>()) != cudaSuccess) return e;
  return configure_decode_t<64, 2>();
}

}  // namespace kvinc
