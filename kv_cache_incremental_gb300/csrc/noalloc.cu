// noalloc.cu -- kv_decode_noalloc: split-K decode attention that allocates nothing.
//
// Some callers cannot call cudaMalloc at all: processes whose device memory is
// owned by another allocator (a framework's caching pool or a fixed arena that
// forbids allocations from outside it), or latency-critical loops that must not
// allocate.  Such a caller owns the K/V storage, the queries, the RoPE table, the
// output and an error word; this entry point runs the same split-K decode kernel
// as kv_append, with its split partials and merge tickets in the file-scope device
// array below instead of memory from kv_cache_create.
//
// The array is fixed at kNoallocScratchBytes; every GPU that loads the library
// holds it until the process exits.  All calls share it and it keeps the last
// call's contents, so calls whose work overlaps on the GPU (two streams, or two
// host threads) race on it.  The merge tickets must start at zero: each call
// clears the ones it uses on its stream before the kernel runs.  The split
// schedule is kv_append's, with splits made longer when the partials of a call
// would not fit the array, so every call within the row and head limits fits.
#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/kvinc.h"
#include "kvinc_internal.h"

namespace kvinc {
cudaError_t configure_decode();
}  // namespace kvinc

using namespace kvinc;

namespace {

constexpr int kNoallocMaxHk = 64;                  // kv heads per call
constexpr size_t kPartOBytes = size_t(16) << 20;   // float partial outputs: 4 Mi floats
constexpr size_t kPartMLBytes = size_t(2) << 20;   // float2 (m, l): 256 Ki entries
constexpr size_t kTicketBytes = size_t(kMaxRowsPerLaunch) * kNoallocMaxHk * 4;  // 128 KiB
constexpr size_t kNoallocScratchBytes = kPartOBytes + kPartMLBytes + kTicketBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// segment-1 keys of every row: none (the caller's storage is one segment)
const int kNoRing[kMaxRowsPerLaunch] = {};

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
unsigned char *g_scratch_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Per-device set-up on the first call with that device current: the device
// address of the scratch array (host code only sees a host-side stand-in for
// the symbol), the SM count, and the decode kernels' shared-memory opt-in.
int setup_device(int dev, unsigned char **scratch, int *num_sms) {
  if (dev < 0 || dev >= kMaxDevices) return KV_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KV_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return KV_ERR_CUDA;
    if (configure_decode() != cudaSuccess) return KV_ERR_CUDA;
    g_num_sms[dev] = sms > 0 ? sms : 1;
    g_scratch_ptr[dev] = static_cast<unsigned char *>(p);
  }
  *scratch = g_scratch_ptr[dev];
  *num_sms = g_num_sms[dev];
  return KV_OK;
}

EncodeTiledFn g_encode_fn = nullptr;
std::once_flag g_encode_once;

bool encode(CUtensorMap *m, const void *base, int64_t rows, int D) {
  std::call_once(g_encode_once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode_fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  const EncodeTiledFn fn = g_encode_fn;
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTileKeys};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int kv_decode_noalloc(const void *K, const void *V, int n_cache_rows, int seg_rows,
                                 int Hq, int Hk, int D, const void *q, const void *rope,
                                 int rope_positions, const int32_t *cache_rows,
                                 const int32_t *pos, const int32_t *n_keys, int Bs, void *out,
                                 int32_t *err, void *stream) {
  if (!K || !V || !q || !rope || !out || !err || !cache_rows || !pos || !n_keys)
    return KV_ERR_ARG;
  if (n_cache_rows < 1 || seg_rows < 1 || Hk < 1 || Hq < 1 || Hq % Hk != 0 ||
      Hq / Hk > kMaxRep || (D != 64 && D != 128) || rope_positions < 1 || Bs < 1)
    return KV_ERR_ARG;
  if (Hk > kNoallocMaxHk) return KV_ERR_SCRATCH;
  if ((int64_t)n_cache_rows * Hk * seg_rows >= (1LL << 31)) return KV_ERR_ARG;
  if (!aligned16(K) || !aligned16(V) || !aligned16(q) || !aligned16(out) || !aligned16(rope) ||
      (reinterpret_cast<uintptr_t>(err) & 3u) != 0)
    return KV_ERR_ARG;
  if (Bs > kMaxRowsPerLaunch) return KV_ERR_SCRATCH;
  for (int i = 0; i < Bs; ++i) {
    if (cache_rows[i] < 0 || cache_rows[i] >= n_cache_rows || pos[i] < 0 ||
        pos[i] >= rope_positions || n_keys[i] < 1 || n_keys[i] > seg_rows)
      return KV_ERR_ARG;
  }

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return KV_ERR_CUDA;
  unsigned char *scratch = nullptr;
  int num_sms = 1;
  const int rc = setup_device(dev, &scratch, &num_sms);
  if (rc != KV_OK) return rc;

  static thread_local DecodeParams dp;
  if (!encode(&dp.tmap_k, K, (int64_t)n_cache_rows * Hk * seg_rows, D) ||
      !encode(&dp.tmap_v, V, (int64_t)n_cache_rows * Hk * seg_rows, D))
    return KV_ERR_CUDA;

  // The split schedule of kv_append over one key segment; merge tickets per call row (the
  // caller's rows may lie beyond the ticket array).
  for (int i = 0; i < Bs; ++i) {
    DecodeRow &r = dp.rows[i];
    r.cache_row = cache_rows[i];
    r.call_row = (uint16_t)i;
    r.pos = pos[i];
    r.nk = n_keys[i];
    r.ctr = i;
  }
  // The partials of a call must fit the fixed scratch: the planner lengthens the splits
  // until they do (one split per row needs no partial slot at all).
  const int max_parts = (int)std::min(kPartOBytes / ((size_t)Hq * D * sizeof(float)),
                                      kPartMLBytes / ((size_t)Hq * sizeof(float2)));
  plan_decode_splits(num_sms, Hk, Bs, kNoRing, dp, max_parts);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t *tickets = reinterpret_cast<int32_t *>(scratch + kPartOBytes + kPartMLBytes);
  if (cudaMemsetAsync(tickets, 0, (size_t)Bs * Hk * sizeof(int32_t), s) != cudaSuccess)
    return KV_ERR_CUDA;

  dp.q = static_cast<const __nv_bfloat16 *>(q);
  dp.q_row_stride = (int64_t)Hq * D;
  dp.out = static_cast<__nv_bfloat16 *>(out);
  dp.out_row_stride = (int64_t)Hq * D;
  dp.rope = static_cast<const float2 *>(rope);
  dp.part_o = reinterpret_cast<float *>(scratch);
  dp.part_ml = reinterpret_cast<float2 *>(scratch + kPartOBytes);
  dp.counters = tickets;
  dp.err = err;  // the caller's word: set to 1 by a timed-out wait, never cleared here
  dp.k_new = nullptr;
  dp.v_new = nullptr;
  dp.kv_row_stride = 0;
  dp.cache_k = nullptr;
  dp.cache_v = nullptr;
  dp.fuse_append = 0;  // the caller has stored the new key already
  dp.fuse_append2 = 0;
  dp.early_kv = 0;  // a plain launch: nothing runs before the previous kernel completes
  dp.seg0_ring = 0;
  dp.ring_R = 1;
  dp.pt = PageTable{nullptr, 0, 0};  // the caller's storage is dense
  dp.tmap_k16 = dp.tmap_k;
  dp.tmap_v16 = dp.tmap_v;
  dp.Hq = Hq;
  dp.Hk = Hk;
  dp.rep = Hq / Hk;
  dp.seg_rows = seg_rows;
  dp.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
  if (launch_decode(dp, D, dp.rep <= 8 ? 1 : 2, s) != cudaSuccess) return KV_ERR_CUDA;
  return KV_OK;
}
