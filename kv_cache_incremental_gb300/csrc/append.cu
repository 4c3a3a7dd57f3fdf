// append.cu -- RoPE-and-append (chunk rows), ring commit and lpos state kernels.
//
// RoPE follows tiny_agent/generate.py `_rope_pos` (half-split pairing,
// (x1 c - x2 s, x1 s + x2 c)) at each row's absolute position; the cos/sin
// table is computed on the host in double and rounded once to float.  The
// arithmetic is float multiply / subtract / add with no contraction, and one
// round-to-nearest-even to bfloat16.
//
// Destinations follow tiny_agent/generate.py `_append_chunk`: a real token t
// of a row goes to position lens + t of the global cache, or to ring slot
// (lens + t) % R; a padding token of a launched token block goes to the
// scratch slot (max_len, or R) instead of being branched around.  For a
// chunk of a sliding layer the rotated keys go to the chunk scratch first
// ("inkling: ring-buffer KV cache for sliding-window layers", How it works:
// the batch is read from scratch and appended after scoring).
#include "kvinc_internal.h"
#include "ptx.cuh"

namespace kvinc {
namespace {

constexpr int kTokBlock = 8;  // tokens per CTA of the append grid

__device__ __forceinline__ int find_row_blk(const AppendParams &p, int b) {
  int lo = 0, hi = p.n_rows - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.rows[mid].blk0 <= b) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void rope8(const uint4 &x1v, const uint4 &x2v, const float2 *cs,
                                      uint4 &lo, uint4 &hi) {
  const __nv_bfloat16 *x1 = reinterpret_cast<const __nv_bfloat16 *>(&x1v);
  const __nv_bfloat16 *x2 = reinterpret_cast<const __nv_bfloat16 *>(&x2v);
  __nv_bfloat16 *o1 = reinterpret_cast<__nv_bfloat16 *>(&lo);
  __nv_bfloat16 *o2 = reinterpret_cast<__nv_bfloat16 *>(&hi);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float a = __bfloat162float(x1[j]);
    const float b = __bfloat162float(x2[j]);
    const float c = cs[j].x, s = cs[j].y;
    o1[j] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s)));
    o2[j] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(a, s), __fmul_rn(b, c)));
  }
}

__global__ void __launch_bounds__(256) append_kernel(const __grid_constant__ AppendParams p) {
  ptx::grid_dep_wait();  // the previous grid on the stream has completed
  ptx::grid_dep_launch();
  const int c_avail = p.c_avail < kChunk ? p.c_avail : kChunk;
  const int r = find_row_blk(p, blockIdx.x);
  const AppendRow &row = p.rows[r];
  const int t0 = (blockIdx.x - row.blk0) * kTokBlock;
  const int half = p.D / 2;
  const int chunks = half / 8;  // 8-pair chunks per head
  const int units = kTokBlock * p.Hk * chunks;
  // Two units per thread and pass, both units' loads issued before either is used.
  constexpr int kPer = 2;
  for (int u0 = threadIdx.x; u0 < units; u0 += kPer * blockDim.x) {
    uint4 in[kPer][4];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int u = u0 + i * blockDim.x;
      const int t = t0 + u / (p.Hk * chunks);
      if (u >= units || t >= c_avail) continue;
      const int g = (u / chunks) % p.Hk, c = u % chunks;
      const int64_t src =
          (int64_t)row.call_row * p.kv_row_stride + ((int64_t)t * p.Hk + g) * p.D + 8 * c;
      in[i][0] = *reinterpret_cast<const uint4 *>(p.k + src);
      in[i][1] = *reinterpret_cast<const uint4 *>(p.k + src + half);
      in[i][2] = *reinterpret_cast<const uint4 *>(p.v + src);
      in[i][3] = *reinterpret_cast<const uint4 *>(p.v + src + half);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int u = u0 + i * blockDim.x;
      const int tl = u / (p.Hk * chunks);
      const int g = (u / chunks) % p.Hk;
      const int c = u % chunks;
      const int t = t0 + tl;
      if (u >= units || t >= c_avail) continue;  // beyond the caller's tensor: nothing to route
      const bool real = t < row.n;
      const int pos = row.lens + t;
      const uint4 k1 = in[i][0], k2 = in[i][1], v1 = in[i][2], v2 = in[i][3];
      uint4 o1 = k1, o2 = k2;  // padding keys are routed unrotated
      if (real) rope8(k1, k2, p.rope + (int64_t)pos * half + 8 * c, o1, o2);

      __nv_bfloat16 *dk, *dv;
      int64_t dst;
      if (row.mode == kDestGlobal && p.pt.max_blocks) {  // paged: pads are not stored
        if (!real) continue;
        dst = kv_row(p.pt, row.cache_row, p.Hk, g, 0, pos) * p.D;
        dk = p.cache_k;
        dv = p.cache_v;
      } else if (row.mode == kDestScratch) {
        dst = (((int64_t)row.cache_row * p.Hk + g) * kChunk + t) * p.D;
        dk = p.scr_k;
        dv = p.scr_v;
      } else {
        int slot;
        if (row.mode == kDestGlobal) slot = real ? pos : p.max_len;
        else slot = real ? pos % p.ring_R : p.ring_R;
        dst = (((int64_t)row.cache_row * p.Hk + g) * p.seg_rows + slot) * p.D;
        dk = p.cache_k;
        dv = p.cache_v;
      }
      *reinterpret_cast<uint4 *>(dk + dst + 8 * c) = o1;
      *reinterpret_cast<uint4 *>(dk + dst + half + 8 * c) = o2;
      *reinterpret_cast<uint4 *>(dv + dst + 8 * c) = v1;
      *reinterpret_cast<uint4 *>(dv + dst + half + 8 * c) = v2;
    }
  }
}

// Copy the kept tokens of a sliding chunk from the chunk scratch into the ring:
// token t is kept iff t >= n - W (the last min(n, W) real tokens; tiny_agent
// keep rule, inkling skip rule s0 = max(0, S - win)).
__global__ void __launch_bounds__(256) commit_kernel(const __grid_constant__ CommitParams p) {
  ptx::grid_dep_wait();  // the previous grid on the stream has completed
  ptx::grid_dep_launch();
  const int r = blockIdx.x, g = blockIdx.y;
  const int n = p.n[r];
  const int first = n - p.window > 0 ? n - p.window : 0;
  const int vec = p.D / 8;
  const int units = (n - first) * vec;
  const int64_t srow = ((int64_t)p.cache_row[r] * p.Hk + g) * kChunk;
  const int64_t rrow = ((int64_t)p.cache_row[r] * p.Hk + g) * p.seg_rows;
  // Four units per thread and pass, every load issued before the first store.
  constexpr int kPer = 4;
  for (int u0 = threadIdx.x; u0 < units; u0 += kPer * blockDim.x) {
    uint4 kk[kPer], vv[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int u = u0 + i * blockDim.x;
      if (u >= units) continue;
      const int64_t s = (srow + first + u / vec) * p.D + 8 * (u % vec);
      kk[i] = *reinterpret_cast<const uint4 *>(p.scr_k + s);
      vv[i] = *reinterpret_cast<const uint4 *>(p.scr_v + s);
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int u = u0 + i * blockDim.x;
      if (u >= units) continue;
      const int t = first + u / vec;
      const int slot = (p.lens[r] + t) % p.ring_R;
      const int64_t d = (rrow + slot) * p.D + 8 * (u % vec);
      *reinterpret_cast<uint4 *>(p.ring_k + d) = kk[i];
      *reinterpret_cast<uint4 *>(p.ring_v + d) = vv[i];
    }
  }
}

// lpos (tiny_agent/generate.py keeps the position held by every ring slot): -1 on
// reset; on advance, the kept tokens' positions at their slots.
__global__ void __launch_bounds__(128) state_kernel(const __grid_constant__ StateParams p) {
  ptx::grid_dep_wait();  // the previous grid on the stream has completed
  ptx::grid_dep_launch();
  const int r = blockIdx.x;
  const int b = p.cache_row[r];
  if (p.reset) {
    for (int s = threadIdx.x; s < p.ring_R; s += blockDim.x) p.lpos[(int64_t)b * p.ring_R + s] = -1;
    return;
  }
  const int lens = p.lens[r], n = p.n[r];
  const int first = n - p.window > 0 ? n - p.window : 0;
  for (int t = first + threadIdx.x; t < n; t += blockDim.x)
    p.lpos[(int64_t)b * p.ring_R + (lens + t) % p.ring_R] = lens + t;
}

}  // namespace

cudaError_t launch_append(const AppendParams &p, cudaStream_t s, bool pdl) {
  if (p.n_blocks <= 0) return cudaSuccess;
  return launch_k(append_kernel, dim3(p.n_blocks), dim3(256), 0, s, p, pdl);
}

cudaError_t launch_commit(const CommitParams &p, cudaStream_t s, bool pdl) {
  if (p.n_rows <= 0) return cudaSuccess;
  return launch_k(commit_kernel, dim3(p.n_rows, p.Hk), dim3(256), 0, s, p, pdl);
}

// Block-table entries of newly allocated blocks (the values travel in the parameters, so a
// later change of the host's tables cannot race with this launch).
__global__ void __launch_bounds__(256) table_kernel(const __grid_constant__ TableParams p) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < p.n; i += gridDim.x * blockDim.x)
    p.table[(int64_t)p.row[i] * p.max_blocks + p.idx[i]] = p.blk[i];
}

cudaError_t launch_table(const TableParams &p, cudaStream_t s) {
  if (p.n <= 0) return cudaSuccess;
  table_kernel<<<(p.n + 255) / 256, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t state_node(const StateParams *p, void **args, cudaKernelNodeParams *kp) {
  if (p->n_rows <= 0) return cudaErrorInvalidValue;
  args[0] = const_cast<StateParams *>(p);
  kp->func = reinterpret_cast<void *>(state_kernel);
  kp->gridDim = dim3(p->n_rows);
  kp->blockDim = dim3(128);
  kp->sharedMemBytes = 0;
  kp->kernelParams = args;
  kp->extra = nullptr;
  return cudaSuccess;
}

cudaError_t launch_state(const StateParams &p, cudaStream_t s, bool pdl) {
  if (p.n_rows <= 0) return cudaSuccess;
  return launch_k(state_kernel, dim3(p.n_rows), dim3(128), 0, s, p, pdl);
}

namespace {

// The kernels' failure path with nothing else around it: a bounded wait on an mbarrier
// that no thread or copy ever completes gives up after `limit` polls and records the
// error in the cache's error word, as every kernel of the library does on a timed-out wait.
__global__ void __launch_bounds__(32) wait_probe_kernel(int32_t *err, uint32_t limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bar, 1);
    ptx::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !ptx::mbar_wait(&bar, 0, limit)) atomicExch(err, 1);
}

}  // namespace

cudaError_t launch_wait_probe(int32_t *err, uint32_t limit, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(err, limit);
  return cudaGetLastError();
}

}  // namespace kvinc
