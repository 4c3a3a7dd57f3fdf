// rowcopy.cu -- K/V position copies between storages: whole-row prefix reuse and
// export / import of a row's live positions.
//
// A global layer holds position p at slot p; a sliding layer holds it at ring slot
// p % R.  Copying a prefix therefore copies global slots linearly and moves ring entries
// position by position (slot p % R_src to slot p % R_dst), never a block of ring slots as
// if they were positions ("inkling: ring-buffer KV cache for sliding-window layers",
// review: grow-with-copy keeps `t % win` valid only when the ring is copied by position).
#include "kvinc_internal.h"

namespace kvinc {
namespace {

// Element offset of position p, head h of one side of a copy.
__device__ __forceinline__ int64_t elem_of(int p, int h, int D, const int32_t *table, int pool,
                                           int64_t head_stride, int ring, int base) {
  if (table)
    return (((int64_t)h * pool + table[p / kBlockTokens]) * kBlockTokens + p % kBlockTokens) * D;
  return h * head_stride + (int64_t)(ring > 0 ? p % ring : p - base) * D;
}

// grid (items, Hk): one CTA per (item, kv head), the host cutting long rows into items of at
// most 2048 positions; 16-byte chunks of K and V, every load of a pass issued before the
// first store.
__global__ void __launch_bounds__(256) copy_kernel(const __grid_constant__ CopyParams p) {
  const CopyItem &it = p.items[blockIdx.x];
  const int h = blockIdx.y;
  const int vec = p.D / 8;
  const int units = (it.p1 - it.p0) * vec;
  const __nv_bfloat16 *sk = it.src_k, *sv = it.src_v;
  __nv_bfloat16 *dk = it.dst_k, *dv = it.dst_v;
  constexpr int kPer = 4;
  for (int u0 = threadIdx.x; u0 < units; u0 += kPer * blockDim.x) {
    uint4 kk[kPer], vv[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int u = u0 + i * blockDim.x;
      if (u >= units) continue;
      const int pos = it.p0 + u / vec, c = u % vec;
      const int64_t s =
          elem_of(pos, h, p.D, it.src_table, it.src_pool, it.src_head_stride, it.src_ring,
                  it.src_base) +
          8 * c;
      kk[i] = *reinterpret_cast<const uint4 *>(sk + s);
      vv[i] = *reinterpret_cast<const uint4 *>(sv + s);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int u = u0 + i * blockDim.x;
      if (u >= units) continue;
      const int pos = it.p0 + u / vec, c = u % vec;
      const int64_t d =
          elem_of(pos, h, p.D, it.dst_table, it.dst_pool, it.dst_head_stride, it.dst_ring,
                  it.dst_base) +
          8 * c;
      *reinterpret_cast<uint4 *>(dk + d) = kk[i];
      *reinterpret_cast<uint4 *>(dv + d) = vv[i];
    }
  }
}

}  // namespace

cudaError_t launch_copy(const CopyParams &p, cudaStream_t s) {
  if (p.n_items <= 0) return cudaSuccess;
  copy_kernel<<<dim3(p.n_items, p.Hk), 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvinc
