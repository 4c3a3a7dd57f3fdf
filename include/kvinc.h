/*
 * kvinc.h -- C ABI of a GB300 (sm_103a) library for incremental decoding
 * against a preallocated per-row KV cache.
 *
 * The caller owns a model; per layer and step it hands the library the new
 * tokens' pre-RoPE queries, keys and values.  The library rotates them (RoPE
 * at each row's absolute positions), appends keys and values to the layer's
 * cache, and returns the attention output of every new token.
 *
 * Sources (web pages, by title and section):
 *  [G]  tiny_agent/generate.py -- `KVCache` (global cache with a scratch
 *       slot, per-layer W-slot ring with a scratch slot, lens mirrored on the
 *       host), `reset`, `append` (right-padded chunk, n_new per row, optional
 *       rows, "KV cache full" raised before any write, sub-chunks of CHUNK=64),
 *       `_append_chunk` (pos = lens + i, pads to the scratch slot, keep the
 *       last W real tokens, ring slot pos % W, grouped queries read the cache
 *       directly), `_rope_pos` (half-split RoPE).
 *  [T]  tinyllm/kv_cache.py -- `SlotKVCache` (per-slot lengths; the device
 *       half of end_step adds the active mask; begin/update/end protocol).
 *  [P]  pycraft-1 model/kv_cache.py -- `KVCache.update` (does NOT advance;
 *       overflow, batch and dtype guards), `advance`, `reset` (no memset),
 *       `memory_bytes`; pre-expansion (n_kv_heads) post-RoPE storage.
 *  [I]  "inkling: ring-buffer KV cache for sliding-window layers" -- "How it
 *       works": ring rows = window when 0 < window < max_t else max_t; the
 *       current batch is read from scratch before the ring append; the append
 *       skips rows the batch would overwrite; a fail-fast bound check.
 *  [L]  Lab 07 -- KV cache and sampling -- section 2 (query i sees key
 *       j <= pos + i), section 3 (chunked prefill equals one pass), the note
 *       that the model advances the cache once after all layers updated.
 *
 * Conventions for every entry point:
 *  - Return value: KV_OK or a kv_status code; kv_strerror() names it.
 *  - Every argument is validated on the host before any work is enqueued; a
 *    call that returns an error has changed no state (host or device).
 *  - Device work runs asynchronously on the caller's CUDA stream (`stream`,
 *    a cudaStream_t passed as void*, NULL = legacy default stream).  No entry
 *    point synchronises the device unless its comment says so.
 *  - The library's kernels are programmatic dependent launches: one may be
 *    scheduled while the kernel before it on the stream finishes, and waits for
 *    that kernel to complete before it reads or writes memory.  Stream order is
 *    kept for every caller kernel launched the ordinary way; a caller kernel
 *    that is itself launched programmatically after a library call must wait
 *    for its predecessor (griddepcontrol.wait) before reading the call's output,
 *    as with any programmatic launch.
 *  - Not thread-safe: one cache is driven from one host thread and one
 *    stream at a time.
 *  - Tensors are bfloat16, row-major, contiguous, 16-byte aligned.
 */
#ifndef KVINC_H
#define KVINC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kv_cache kv_cache; /* opaque; the library owns all cache memory */

/* Layer kinds of the layer layout. */
enum kv_layer_kind {
    KV_GLOBAL = 0,        /* full-length cache, every past key visible ([G] global K/V) */
    KV_SLIDING = 1,       /* ring of W slots, keys p-W+1..p visible ([I], [G] local K/V) */
    /* [G]'s hybrid layers (tiny_agent/generate.py, module docstring and `_append_chunk`):
     * a group of layers shares one global K/V, written by the group's first layer, and
     * every layer of the group also keeps its own local ring of W slots; a layer attends
     * to the group's global keys at every position <= p and to its own local keys at
     * p-W+1..p, in ONE softmax.  Use kv_append_hybrid on these layers. */
    KV_HYBRID_FULL = 2,   /* opens a group: owns the group's global K/V, and its ring */
    KV_HYBRID_LOCAL = 3   /* reads the global K/V of the nearest preceding KV_HYBRID_FULL
                             layer; owns its ring */
};

enum kv_status {
    KV_OK = 0,
    KV_ERR_ARG = 1,    /* invalid argument: sizes, layer, rows, n_new, pointers */
    KV_ERR_FULL = 2,   /* lens[row] + n_new > max_len for some row ([G] append, [P] update) */
    KV_ERR_DTYPE = 3,  /* tensor dtype is not bfloat16 (raised by language bindings; [P]) */
    KV_ERR_CUDA = 4,   /* a CUDA runtime call failed */
    KV_ERR_OOM = 5,    /* device memory allocation failed at create */
    KV_ERR_DEVICE = 6, /* a kernel reported a timed-out wait (see kv_device_error) */
    KV_ERR_SCRATCH = 7, /* request too large for kv_decode_noalloc's fixed scratch */
    KV_ERR_POOL = 8     /* a paged cache has no free block for the new positions */
};

/*
 * Create a cache for B rows on CUDA device `device`.  [G] KVCache, [P] KVCache,
 * [I] kv_ring_rows.
 *
 *  max_len     positions per row (>= 1, <= 2^20)
 *  Hq, Hk      query heads and key/value heads; Hq % Hk == 0, Hq/Hk <= 16
 *  D           head dimension: 64 or 128
 *  W           sliding window in tokens (>= 1) when any layer is KV_SLIDING,
 *              else ignored.  A sliding layer stores R = W < max_len ? W :
 *              max_len ring slots per (row, kv head) plus one scratch slot.
 *  layer_kind  host array [n_layers] of kv_layer_kind
 *  rope_theta  RoPE base (e.g. 10000); frequencies theta^(-2i/D), i < D/2
 *
 * Device memory, allocated here with cudaMalloc and freed by
 * kv_cache_destroy (per layer, K and V):
 *    global layer   [B][Hk][max_len + 1][D] bf16   (slot max_len = scratch)
 *    sliding layer  [B][Hk][R + 1][D] bf16         (slot R = scratch)
 * plus lens [B] and lpos [B][R] (int32), a chunk scratch [B][Hk][64][D] for K
 * and V, the RoPE table [max_len][D/2] of (cos, sin) float pairs computed on
 * the host in double, decode split-K partials (min(B, 512) x 32 x Hq vectors of
 * D floats) and chunked-prefill key-split partials (min(1024 x SMs,
 * B x Hq x 64 x 16) vectors of D floats).  Every later call works within this
 * memory: none allocates device memory except kv_append_host / kv_append_hybrid_host
 * with pageable buffers (their staging) and kv_step_graph_create (the graph's own
 * resources, at instantiation).  All lens start at 0.
 * On success *out holds the cache; on failure *out is NULL.
 */
int kv_cache_create(kv_cache **out, int B, int max_len, int Hq, int Hk, int D, int W,
                    int n_layers, const int32_t *layer_kind, double rope_theta, int device);

/*
 * Paged cache: as kv_cache_create, but every global layer keeps its K/V in a pool of
 * n_blocks blocks of 16 positions (bf16 [Hk][n_blocks][16][D]: head-major, so that a
 * row's consecutive blocks are contiguous per head) and each row a table of the
 * blocks that hold its positions 16i..16i+15, shared by all global layers (a row has
 * the same length on all of them) ("Lab 07 -- KV cache and sampling", Stretch:
 * fixed 16-token blocks plus a per-sequence block table; "tinyllm/kv_cache.py": a
 * dense cache reserves max_len slots per row whatever its length).  Blocks are taken
 * from the pool when a call appends positions past a row's last block (kv_append,
 * kv_append_host, kv_step_graph_launch, kv_copy_rows, kv_import_row) and let go of on
 * kv_reset or when a copy shortens or replaces a row.  Blocks are reference-counted
 * (same page, Stretch: prefix sharing): kv_copy_rows inside one paged cache gives the
 * destination row the source row's full blocks of the kept prefix instead of copies,
 * and a block returns to the pool when the last row holding it lets go.  A block held
 * by several rows lies below each holder's length, so no append writes it; a row cut in
 * place inside such a block first takes a copy of it, and kv_import_row and copies from
 * another cache give the row blocks of its own.  kv_get_block_table shows the sharing
 * (equal block ids) and kv_free_blocks the memory it saves.  A call whose rows need
 * more blocks than are free returns KV_ERR_POOL before anything is enqueued.  Sliding
 * layers keep their dense rings.  Results are those of the dense cache, bit for bit.
 * 1 <= n_blocks, n_blocks * Hk * 16 < 2^31; with n_blocks >= B * ceil(max_len / 16)
 * no call runs out of blocks.  The pool is reused on the caller's stream order: one
 * stream per cache.
 */
int kv_cache_create_paged(kv_cache **out, int B, int max_len, int Hq, int Hk, int D, int W,
                          int n_layers, const int32_t *layer_kind, double rope_theta, int device,
                          int n_blocks);
/* Pool blocks of a row, in position order (host mirror): writes min(count, capacity)
 * entries and the count to *n_out (0 for a dense cache).  Free blocks of the pool, or
 * -1 for NULL. */
int kv_get_block_table(const kv_cache *c, int row, int32_t *blocks_out, int capacity,
                       int *n_out);
int kv_free_blocks(const kv_cache *c);

/* Free all device and host memory of the cache (NULL is a no-op).  Waits for
 * the device to finish work that uses the cache. */
void kv_cache_destroy(kv_cache *c);

/*
 * Empty rows so new sequences can start there.  [G] reset, [P] reset.
 *  rows  host int32 [n_rows], distinct, in [0, B)
 * Sets lens[row] = 0 (host mirror and device) and lpos[row][*] = -1.  Cached
 * K/V are not cleared: stale slots are never read, because every key a
 * query can see was written after the reset.
 */
int kv_reset(kv_cache *c, const int32_t *rows, int n_rows, void *stream);

/*
 * Append one layer's new tokens and return their attention outputs.
 * [G] append / _append_chunk, [P] update, [I], [L] sections 2-3.
 *
 *  layer   0 <= layer < n_layers
 *  q       device bf16 [Bs][C][Hq][D]   pre-RoPE queries
 *  k, v    device bf16 [Bs][C][Hk][D]   pre-RoPE keys, values
 *  Hq      must equal the cache's Hq (checked)
 *  C       chunk width (>= 1); row i carries n_new[i] real tokens at
 *          t = 0..n_new[i]-1, the rest of the row is padding
 *  n_new   host int32 [Bs], each in [0, C]; 0 leaves the row untouched
 *  rows    host int32 [Bs] cache rows (distinct, in [0, B)), or NULL for
 *          rows 0..Bs-1
 *  out     device bf16 [Bs][C][Hq][D]; for every real token t of row i,
 *          out[i][t][h] = softmax over the visible keys of
 *          (rope(q,p) . K_j) / sqrt(D), times V_j, at p = lens[row] + t,
 *          with head h reading kv head h / (Hq/Hk).  Visible keys: j <= p
 *          (global) or p-W < j <= p (sliding), the chunk's own earlier
 *          tokens included.  Padding positions of `out` are not written.
 *
 * Effects on layer `layer`: rope(k, p) and v are stored at position p of
 * every real token (global: cache slot p; sliding: ring slot p % R for the
 * last min(n_new, W) tokens of the row only -- [G] keep rule, [I] skip
 * rule).  lens is NOT advanced: every layer of a step sees the same
 * positions, and the caller ends the step with kv_advance ([P] update/
 * advance, [L]).  Tokens are processed in sub-chunks of 64 per row.
 * The call allocates nothing and never synchronises: it plans on the host
 * (lens is mirrored there) and enqueues kernels that use only the memory
 * reserved by kv_cache_create -- the chunked-prefill key splits are planned to
 * fit the reserved partials (longer splits when a call would need more).
 * Errors: KV_ERR_FULL if lens[row] + n_new[i] > max_len for any row,
 * KV_ERR_ARG for bad sizes, rows, counts or pointers, KV_ERR_POOL (paged cache)
 * when the pool has too few free blocks, KV_ERR_CUDA if a launch fails.
 */
int kv_append(kv_cache *c, int layer, const void *q, const void *k, const void *v, int Hq,
              int C, const int32_t *n_new, const int32_t *rows, int Bs, void *out,
              void *stream);

/*
 * kv_append for a hybrid layer.  k_local, v_local: device bf16 [Bs][C][Hk][D], the
 * layer's own pre-RoPE local keys and values (stored in its ring by the keep rule, as on
 * a sliding layer).  k_global, v_global: the group's pre-RoPE global keys and values
 * (same shape), required on a KV_HYBRID_FULL layer (stored in the group's cache, as on a
 * global layer) and NULL on a KV_HYBRID_LOCAL layer, whose group's full layer must
 * already have been appended in this step (stream order).  out: for every real token t
 * at p = lens[row] + t, softmax over the group's global keys j <= p and the layer's local
 * keys p-W < j <= p together, of (rope(q, p) . K_j) / sqrt(D), times the matching V_j.
 * Same rules and errors as kv_append; KV_ERR_ARG on a layer that is not hybrid (and
 * kv_append returns KV_ERR_ARG on a hybrid layer).
 */
int kv_append_hybrid(kv_cache *c, int layer, const void *q, const void *k_local,
                     const void *v_local, const void *k_global, const void *v_global, int Hq,
                     int C, const int32_t *n_new, const int32_t *rows, int Bs, void *out,
                     void *stream);
/* kv_append_hybrid with HOST buffers, as kv_append_host (page-locked ones used in place,
 * pageable ones staged; `out` is written when the stream reaches this call). */
int kv_append_hybrid_host(kv_cache *c, int layer, const void *q, const void *k_local,
                          const void *v_local, const void *k_global, const void *v_global, int Hq,
                          int C, const int32_t *n_new, const int32_t *rows, int Bs, void *out,
                          void *stream);

/*
 * Same as kv_append, but q, k, v and out are HOST buffers.  Page-locked buffers
 * (cudaHostAlloc / cudaHostRegister, e.g. torch pin_memory) are read and written
 * by the kernels directly through their device addresses: on GB300 host memory
 * is coherent over NVLink-C2C, so the inputs and outputs cross the link inside
 * the kernels with no copy-engine operation; the work is queued on `stream` and
 * the call returns before it finishes (synchronise the stream before reading
 * `out`) and, like kv_append, allocates nothing and never synchronises.
 * Pageable buffers are staged with cudaMemcpyAsync through a device buffer the
 * cache owns, allocated on the first such call and grown when a larger call
 * arrives: growing synchronises `stream` (the old buffer may still be in use),
 * frees it and allocates the new one (KV_ERR_OOM if that fails; the cache is
 * unchanged), and the copies from and to pageable memory make the call return
 * only after `stream` has finished it.  Padding positions of `out` are not
 * written with page-locked buffers and are unspecified with pageable ones.
 */
int kv_append_host(kv_cache *c, int layer, const void *q, const void *k, const void *v,
                   int Hq, int C, const int32_t *n_new, const int32_t *rows, int Bs,
                   void *out, void *stream);

/*
 * End a step: lens[row] += n_new[i] (host mirror and device) and record the
 * ring-slot positions lpos[row][p % R] = p of the kept tokens.  Call once per
 * step, after every layer has been appended with the same n_new and rows.
 * [P] advance, [T] end_step, [L] "who advances the cache".
 * Errors: as kv_append (KV_ERR_FULL, KV_ERR_ARG); nothing changes on error.
 */
int kv_advance(kv_cache *c, const int32_t *n_new, const int32_t *rows, int Bs, void *stream);

/* Bytes of K and V storage of all layers, scratch slots included ([G] nbytes,
 * [P] memory_bytes); a paged cache counts its global layers' whole pools.  -1 for
 * a NULL cache. */
int64_t kv_nbytes(const kv_cache *c);

/* Copy the host mirror of lens into lens_out (host int32 [B]).  No device sync. */
int kv_get_lens(const kv_cache *c, int32_t *lens_out);

/* Device pointers of a layer's K and V storage and of lpos ([B][R] int32, or
 * NULL without sliding or hybrid layers), for inspection and tests.  For a hybrid
 * layer: its group's global storage; kv_debug_ring_ptrs gives its ring ([B][Hk][R+1][D]).  Layouts as in
 * kv_cache_create; a paged cache's global layers point at their block pools
 * ([Hk][n_blocks][16][D], see kv_get_block_table).  The pointers stay owned by the
 * cache. */
int kv_debug_ptrs(const kv_cache *c, int layer, void **K, void **V, int32_t **lpos);
int kv_debug_ring_ptrs(const kv_cache *c, int layer, void **K, void **V);

/* Shape query: fills any non-NULL output with the cache's parameters. */
int kv_get_config(const kv_cache *c, int *B, int *max_len, int *Hq, int *Hk, int *D, int *W,
                  int *R, int *n_layers);

/* Read and clear the device error word (0 = no kernel reported a timed-out
 * wait).  SYNCHRONISES the device.  Returns KV_ERR_DEVICE when the word was
 * non-zero, else KV_OK. */
int kv_device_error(kv_cache *c, int32_t *code_out);

/* Failure-path check: enqueues, on `stream`, a kernel whose bounded wait on a barrier
 * that nothing completes gives up after `limit` polls (1 <= limit <= 2^20; every kernel
 * of the library bounds its waits the same way, with a larger limit) and records the
 * timeout in the cache's device error word, which kv_device_error then reports.  Touches
 * nothing else.  KV_ERR_ARG for a bad limit. */
int kv_debug_wait_timeout(kv_cache *c, uint32_t limit, void *stream);

/*
 * Host-only schedules, for inspection and tests: the work split that kv_append plans for
 * one call on a layer, computed from the shapes alone -- no cache, no CUDA call, no
 * device work, so they run without a GPU.  Shape arguments as at kv_cache_create, plus
 * num_sms (the device's SM count, 1..4096, which a cache reads from its device), R (the ring
 * slots of a sliding or hybrid layer, min(W, max_len); ignored when kind = KV_GLOBAL)
 * and kind (the layer's kv_layer_kind).  Both write nothing and return KV_ERR_ARG for
 * a shape kv_cache_create refuses, a NULL array that is needed, or inputs out of range.
 *
 * kv_plan_decode: the split-K schedule of one decode launch, n_rows <= 512 single-token
 * rows at positions pos[] (host, each < 2^20; a row's pos is its lens).  A row's keys
 * are one or two segments: segment 0 the layer storage -- keys 0..pos of a global
 * layer's cache or of a hybrid layer's group cache, or the min(pos + 1, R) ring slots of
 * a sliding layer -- and, on a hybrid layer, segment 1 its own ring (min(pos + 1, R)
 * slots).  Each segment is cut into splits of whole 64-key tiles.  Per row (host arrays
 * of n_rows): n_splits / split_tiles -- segment 0's splits and the tiles of each (the
 * last split takes the rest); n_splits2 / split_tiles2 -- the same for segment 1 (0 off
 * hybrid layers); part0 -- the first of the row's n_splits + n_splits2 partial slots,
 * -1 for a row with one split in all (no merge).  *n_items: the launch's CTAs per kv
 * head, the sum of every row's splits.
 *
 * kv_plan_prefill: the prefill launches of one sub-chunk of n_rows chunk rows, row i
 * with n[i] (1..64) new tokens after lens[i] cached ones (host arrays; lens + n <= 2^20).
 * Entries (host arrays of `capacity`, in launch order): entry_row -- the input row;
 * entry_kind -- 0 the mma.sync kernel (64 query rows per CTA), 1 the tcgen05 kernel
 * with two 128-row query tiles per CTA, 2 the tcgen05 kernel with one; tile0, tile1 --
 * the 64-key tiles [tile0, tile1) of the row's key space the entry reads (INT32_MAX:
 * to the end); part -- the first partial vector a key split writes, -1 for a row in one
 * entry.  A row's key space runs over its storage segments in order (a global layer:
 * cache keys 0..lens+n-1; a sliding layer: its ring keys, then the chunk; a hybrid
 * layer: the group cache, its ring, then the chunk).  *n_entries: the entries; if that
 * is above capacity the call returns KV_ERR_ARG and writes nothing else.  n_splits[i]:
 * the entries of row i; *part_vecs: the partial vectors of the sub-chunk
 * (Hk * n * Hq / Hk per split of a split row), never above 1024 * num_sms -- the
 * reserve a cache makes at create -- because splits are lengthened until they fit.
 */
int kv_plan_decode(int num_sms, int Hq, int Hk, int D, int R, int kind, int n_rows,
                   const int32_t *pos, int32_t *n_splits, int32_t *split_tiles,
                   int32_t *n_splits2, int32_t *split_tiles2, int32_t *part0, int32_t *n_items);
int kv_plan_prefill(int num_sms, int Hq, int Hk, int D, int R, int kind, int n_rows,
                    const int32_t *lens, const int32_t *n, int capacity, int32_t *entry_row,
                    int32_t *entry_kind, int32_t *tile0, int32_t *tile1, int32_t *part,
                    int32_t *n_entries, int32_t *n_splits, int64_t *part_vecs);

/*
 * Kernel timing for measurement.  kv_profile_enable(c, 1) makes the library
 * record a CUDA event pair around each kernel launch it makes, on the stream
 * of the launch; kv_profile_read sums, per kernel kind, the launches, the
 * event-timed milliseconds (it SYNCHRONISES the device) and the algorithmic
 * bytes the host counted for those launches; kv_profile_enable(c, 0) or a read
 * with reset=1 clears the record.  Kinds: KV_KERNEL_APPEND, KV_KERNEL_DECODE,
 * KV_KERNEL_COMBINE, KV_KERNEL_PREFILL, KV_KERNEL_COMMIT, KV_KERNEL_STATE, and
 * KV_KERNEL_STEP: one replay of a decode-step graph (kv_step_graph_launch), all
 * its layers' decode kernels and the state update, with their algorithmic bytes.
 */
enum kv_kernel_kind {
    KV_KERNEL_APPEND = 0,
    KV_KERNEL_DECODE = 1,
    KV_KERNEL_COMBINE = 2,
    KV_KERNEL_PREFILL = 3,
    KV_KERNEL_COMMIT = 4,
    KV_KERNEL_STATE = 5,
    KV_KERNEL_STEP = 6,
    KV_KERNEL_NKINDS = 7
};
int kv_profile_enable(kv_cache *c, int enable);
int kv_profile_read(kv_cache *c, int kind, int reset, int64_t *launches, double *total_ms,
                    double *alg_bytes, double *alg_flops);

/*
 * Static-shape decode step as a CUDA graph.  One decode step of a fixed set of rows
 * -- for every layer, kv_append with one new token per row, then kv_advance -- is
 * built once into a graph (one decode kernel node per layer, then the ring-state
 * node when the cache has sliding layers) and replayed per step.  The pages keep
 * the step's shapes fixed so that a captured graph can be replayed, and advance
 * the host's lengths after each replay ("tinyllm/kv_cache.py" (tiny-llm):
 * end_step / advance_host; "Lab 07 -- KV cache and sampling", Stretch:
 * static shapes for CUDA graphs).  Here positions live in each kernel's
 * parameters, so every launch re-plans the step from the host lengths, updates the
 * nodes' parameters and grid sizes in the instantiated graph, replays it on the
 * stream, and then advances the host lengths: the result is bit-identical to the
 * kv_append / kv_advance sequence, with one graph launch instead of one launch per
 * layer.
 *
 *  q, k, v, out  host arrays of n_layers device pointers: layer l's bf16 query
 *                [Bs][1][Hq][D], key and value [Bs][1][Hk][D] and output
 *                [Bs][1][Hq][D] buffers, 16-byte aligned, read and written by the
 *                launches that follow (the caller writes each step's inputs, in
 *                stream order, before the launch, or points the graph at new
 *                buffers with kv_step_graph_set_buffers)
 *  rows          host int32 [Bs] distinct cache rows, or NULL for 0..Bs-1;
 *                1 <= Bs <= min(B, 512)
 *  Hq            must equal the cache's Hq
 *
 * kv_step_graph_create plans for the current lengths and enqueues nothing;
 * KV_ERR_ARG for bad arguments, KV_ERR_CUDA if graph construction fails, and on
 * any failure *out is NULL (when out is not).
 * kv_step_graph_launch returns KV_ERR_FULL (and changes no state) if a row is at
 * max_len, KV_ERR_CUDA if a CUDA call fails; it never synchronises.  Rows of the
 * cache that are not in `rows` are untouched.  A reset of one of the rows between
 * launches is allowed (the next launch plans from the new length).
 * kv_step_graph_set_buffers replaces the four pointer arrays for the following
 * launches (same rules as at create; KV_ERR_ARG leaves the old ones in place); it
 * enqueues nothing, since every launch rewrites the nodes' parameters anyway.
 * kv_step_graph_destroy frees the graph (not the caller's buffers); destroy graphs
 * before their cache.
 */
typedef struct kv_step_graph kv_step_graph;
int kv_step_graph_create(kv_cache *c, kv_step_graph **out, const void *const *q,
                         const void *const *k, const void *const *v, void *const *outp, int Hq,
                         const int32_t *rows, int Bs);
int kv_step_graph_set_buffers(kv_step_graph *g, const void *const *q, const void *const *k,
                              const void *const *v, void *const *outp);
/* The step graph of a cache with hybrid layers (kv_step_graph_create returns KV_ERR_ARG
 * for one): k[l], v[l] of a hybrid layer are its local keys and values, k_global[l],
 * v_global[l] the group's global ones -- device bf16 [Bs][1][Hk][D], 16-byte aligned,
 * given exactly for the KV_HYBRID_FULL layers and NULL for every other layer (the arrays
 * themselves may be NULL on a cache without full hybrid layers).  A launch is then
 * kv_append_hybrid / kv_append on every layer in order, then kv_advance.  Works on any
 * cache. */
int kv_step_graph_create_hybrid(kv_cache *c, kv_step_graph **out, const void *const *q,
                                const void *const *k, const void *const *v,
                                const void *const *k_global, const void *const *v_global,
                                void *const *outp, int Hq, const int32_t *rows, int Bs);
int kv_step_graph_set_buffers_hybrid(kv_step_graph *g, const void *const *q,
                                     const void *const *k, const void *const *v,
                                     const void *const *k_global, const void *const *v_global,
                                     void *const *outp);
int kv_step_graph_launch(kv_step_graph *g, void *stream);
void kv_step_graph_destroy(kv_step_graph *g);

/*
 * Prefix reuse and row export / import.  A row's state is its length and, per storage
 * unit, the K/V of the positions it keeps: all of [0, lens) in a full-length cache (a
 * global layer's, a hybrid group's), the last R of them in a ring (a sliding layer's, a
 * hybrid layer's own; slot p % R).  Units in order: per layer, the storage it owns (a
 * hybrid local layer owns none), then its hybrid ring.  Copies move positions, so a
 * ring is copied position by position and a global prefix linearly ("inkling:
 * ring-buffer KV cache for sliding-window layers", review of the change: prefix reuse
 * by grow-with-copy must copy the ring whole, keeping t % win valid, and global rows
 * linearly; "Lab 07 -- KV cache and sampling", Stretch: prefix sharing).
 *
 * kv_copy_rows: for i < n, destination row dst_rows[i] of `dst` becomes the first
 *   keep[i] tokens of source row src_rows[i] of `src` (keep == NULL: the source's
 *   whole length): its K/V, ring state (lpos) and length.  Inside one paged cache the
 *   global layers' full blocks of the prefix are shared with the source row, not
 *   copied (see kv_cache_create_paged); only a partly filled last block is copied.  Uses: forking a sequence
 *   into another row, reusing a shared prompt prefix, truncating a row (src == dst,
 *   same row), and moving rows into a cache with another max_len or B (grow-with-
 *   copy).  dst and src may be the same cache.  Both caches must have the same Hk, D,
 *   W, layer layout, rope_theta and device.  Rows: host int32 [n]; destination rows
 *   distinct; in one cache no destination row may be another pair's source row.
 *   keep[i] <= the source length and <= dst's max_len, and every position the
 *   destination keeps must still be in the source: on caches with rings,
 *   max(0, keep - R_dst) >= max(0, src_len - R_src) (a ring that has wrapped holds
 *   only its last R positions, so such a row can be copied whole but not truncated).
 *   Violations return KV_ERR_ARG before anything is enqueued.  Asynchronous on
 *   `stream`; the source rows must not be written until the copy has run.
 *
 * kv_export_bytes: size of a row's state at length keep (-1 for a bad keep).
 * kv_export_row: writes the first `keep` tokens of `row` (keep <= its length, same
 *   presence rule) to the device buffer `dst` of exactly kv_export_bytes(c, keep)
 *   bytes, 16-byte aligned: per storage unit in order, K [Hk][n_u][D] then V [Hk][n_u][D]
 *   bf16, n_u = the unit's kept positions in ascending order.
 * kv_import_row: row `row` becomes that state (its length keep <= max_len); K/V of
 *   positions the row does not keep are left as they are.  The buffer is read on
 *   `stream`.  KV_ERR_ARG for bad arguments or a byte count that does not match.
 */
int kv_copy_rows(kv_cache *dst, const int32_t *dst_rows, const kv_cache *src,
                 const int32_t *src_rows, const int32_t *keep, int n, void *stream);
int64_t kv_export_bytes(const kv_cache *c, int keep);
int kv_export_row(const kv_cache *c, int row, int keep, void *dst, int64_t bytes, void *stream);
int kv_import_row(kv_cache *c, int row, int keep, const void *src, int64_t bytes, void *stream);

/*
 * Decode attention that allocates nothing.  The pages have no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc -- for example a
 * process whose device memory is owned by another allocator (a framework's
 * caching pool or a fixed arena that forbids allocations from outside it), or a
 * latency-critical loop that must never allocate.  Such a caller cannot create a
 * kv_cache, so it passes its own memory: the cache storage, the queries, the
 * RoPE table, the output and an error word.  The call runs the same split-K
 * decode kernel as kv_append, with kv_append's split schedule (kv_plan_decode with
 * kind KV_GLOBAL and pos = n_keys - 1 gives it) except that splits are made longer
 * when their partials would not fit the scratch; its split partials and merge
 * tickets live in one file-scope device array of 18 MiB + 128 KiB that every GPU
 * which loads the library holds until the process exits.
 *
 *  K, V        device bf16 [n_cache_rows][Hk][seg_rows][D] (one layer's storage in
 *              the kv_cache layout, e.g. from kv_debug_ptrs, or the caller's own)
 *  q           device bf16 [Bs][Hq][D], pre-RoPE query of each row's decode token
 *  rope        device float2 [rope_positions][D/2]: (cos, sin) of position p,
 *              pair i, as kv_cache_create computes them
 *  cache_rows  host int32 [Bs], row of K/V for each query, in [0, n_cache_rows)
 *  pos         host int32 [Bs], the query's absolute position (for RoPE),
 *              in [0, rope_positions)
 *  n_keys      host int32 [Bs], keys in storage slots [0, n_keys) are visible
 *              (1 <= n_keys <= seg_rows); the new token's key must already be
 *              stored (global layer: n_keys = pos + 1; ring: min(pos + 1, R))
 *  out         device bf16 [Bs][Hq][D]
 *  err         device int32, 4-byte aligned, owned by the caller: a kernel whose
 *              bounded wait timed out sets it to 1 (that call's output is then
 *              incomplete); the call never clears it, so the caller zeroes it once
 *              and reads it whenever it synchronises
 *  D is 64 or 128, Hq % Hk == 0, Hq / Hk <= 16.
 *
 * Limits: Bs <= 512 and Hk <= 64; a request beyond them returns KV_ERR_SCRATCH
 * before any work is enqueued.  Within them every call fits the scratch (16 MiB of
 * float partial outputs, 2 MiB of (max, sum) pairs, merge tickets for 512 x 64
 * (row, kv head) pairs).
 * Set-up: the first call on each device (made with that device current)
 * resolves the scratch array's device address with cudaGetSymbolAddress and
 * opts the kernels into their shared-memory size, so make that first call
 * before any stream capture.  All calls share the scratch and it keeps the
 * last call's contents: calls whose work overlaps on the GPU (different
 * streams or host threads) race on it and must be ordered by the caller.
 * Each call clears the merge tickets it uses on `stream` before its kernel.
 */
int kv_decode_noalloc(const void *K, const void *V, int n_cache_rows, int seg_rows, int Hq,
                      int Hk, int D, const void *q, const void *rope, int rope_positions,
                      const int32_t *cache_rows, const int32_t *pos, const int32_t *n_keys,
                      int Bs, void *out, int32_t *err, void *stream);

/* Static name of a status code. */
const char *kv_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* KVINC_H */
