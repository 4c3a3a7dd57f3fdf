// synth_device.cu -- device twin of synth/__init__.py's counter-based generator.
//
// Test and benchmark input generation only; it is not part of the KV-cache
// library.  The definition (SplitMix64 as a counter-based generator, the
// per-stream key chain, twelve 16-bit lanes summed and centred, one rounding
// to bfloat16) is stated in synth/__init__.py; integer arithmetic only, so the
// CPU and GPU produce identical bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ inline int lanes_sum(uint64_t u) {
  return (int)(u & 0xFFFF) + (int)((u >> 16) & 0xFFFF) + (int)((u >> 32) & 0xFFFF) +
         (int)((u >> 48) & 0xFFFF);
}

__host__ __device__ inline uint64_t stream_key(uint64_t seed, int tensor, int layer, int row,
                                               int seq) {
  uint64_t k = mix64(seed + kGamma);
  k = mix64(k + (uint64_t)(tensor + 1) * kGamma);
  k = mix64(k + (uint64_t)(layer + 1) * kGamma);
  k = mix64(k + (uint64_t)(row + 1) * kGamma);
  k = mix64(k + (uint64_t)(seq + 1) * kGamma);
  return k;
}

__global__ void fill_kernel(__nv_bfloat16 *__restrict__ dst, uint64_t seed, int tensor,
                            int layer, const int32_t *__restrict__ rows,
                            const int32_t *__restrict__ seqs, const int32_t *__restrict__ pos0,
                            int C, int H, int D) {
  const int i = blockIdx.y;  // row of the batch
  const int64_t per_row = (int64_t)C * H * D;
  const uint64_t key = stream_key(seed, tensor, layer, rows[i], seqs[i]);
  const int64_t p0 = pos0[i];
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < per_row;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = idx / ((int64_t)H * D);
    const int64_t rem = idx - t * H * D;  // head * D + d
    const uint64_t e = (uint64_t)((p0 + t) * H * D + rem);
    int s = 0;
#pragma unroll
    for (int j = 0; j < 3; ++j) s += lanes_sum(mix64(key + (3 * e + j + 1) * kGamma));
    const float x = (float)(s - 393210) * (1.0f / 65536.0f);  // exact: power-of-two scale
    dst[(int64_t)i * per_row + idx] = __float2bfloat16_rn(x);
  }
}

}  // namespace

extern "C" int kvsynth_fill_bf16(void *dst, uint64_t seed, int tensor, int layer,
                                 const int32_t *rows, const int32_t *seqs, const int32_t *pos0,
                                 int n_rows, int C, int H, int D, void *stream) {
  if (n_rows <= 0 || C <= 0) return 0;
  const int64_t per_row = (int64_t)C * H * D;
  int bx = (int)((per_row + 255) / 256);
  if (bx > 1024) bx = 1024;
  dim3 grid(bx, n_rows);
  fill_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>((__nv_bfloat16 *)dst, seed, tensor, layer,
                                                       rows, seqs, pos0, C, H, D);
  return (int)cudaGetLastError();
}
