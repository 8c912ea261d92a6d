/*
 * iqkv.h — C ABI of libiqkv: a rotated, asymmetric K4/V3 bit-packed KV cache
 * and GQA decode / short-query verify attention over it, for one sm_103a GPU.
 *
 * Source of the method: the page "sparkle mlx_streaming/core/cache/quant_kv.py"
 * (sections "SO(4) block rotation", "AsymmetricQuantizedKVCache",
 * "asym_quantized_sdpa") and the page "sparkle mlx_streaming/mtp/kv_cache.py"
 * (`commit_verified_prefix`, `_snapshot` / `_restore`, `tile_caches`,
 * `commit_tree_row`).
 *
 * Conventions shared by every entry point:
 *  - Every device buffer is allocated and owned by the caller; the library
 *    never allocates, frees or keeps a pointer after a call returns.
 *  - Work is enqueued asynchronously on the caller's stream (`iq_stream_t` is a
 *    `cudaStream_t`; NULL is the legacy default stream).  No entry point
 *    synchronises the device, except `iq_read_status`, which says so.
 *  - A cache has an element dtype, bfloat16 (IQ_DTYPE_BF16) or float32
 *    (IQ_DTYPE_F32): the dtype of the keys, values and queries it is fed, of
 *    its scales and biases (the page's `_init_quant(..., dt)` takes `dt` from
 *    the keys), and of the rotation blocks it is given (the page's
 *    `rotate_last` casts M to the input's dtype: M_b for bfloat16, M itself
 *    for float32).  Data arguments are `const void*` of that dtype; bfloat16
 *    values are 16-bit patterns.
 *  - Functions return an `iq_status`; nothing is thrown across the ABI.  On an
 *    error nothing is enqueued and nothing the caller owns is modified, and
 *    `iq_last_error()` holds a one-line explanation (per host thread).
 *  - Supported shapes: head_dim 256; k_bits and v_bits 2, 3, 4, 5, 6 or 8 (the
 *    widths the page's `_packed_words` lists); group_size 32, 64 or 128;
 *    1 <= batch <= IQ_MAX_BATCH, kv heads >= 1, query heads a multiple of kv
 *    heads with at most 8 query heads per kv head and 8 % rep == 0.  Anything
 *    else returns IQ_ERR_UNSUPPORTED.  k_bits 4, v_bits 3, group 64 runs the
 *    tuned kernels when the dtype is bfloat16; every other format, and every
 *    float32 cache, runs a generic path (same arithmetic, float32 attention
 *    over shared-memory tiles) that serves at most 64 query rows (query heads
 *    per kv head x n_queries) per call and never fuses the append into the
 *    attention.
 */
#ifndef IQKV_H
#define IQKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IQ_MAX_BATCH 256
#define IQ_STEP 256 /* capacity granule, the page's `AsymmetricQuantizedKVCache.step` */

typedef void* iq_stream_t; /* a cudaStream_t */

#define IQ_DTYPE_BF16 0 /* bfloat16 data, scales and biases (the tuned kernels) */
#define IQ_DTYPE_F32 1  /* float32 data, scales and biases (generic path) */

typedef enum {
  IQ_OK = 0,
  IQ_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned buffer, bad mask */
  IQ_ERR_CAPACITY = 2,    /* an append would write past the cache capacity */
  IQ_ERR_WORKSPACE = 3,   /* workspace missing or smaller than iq_attend_workspace() */
  IQ_ERR_UNSUPPORTED = 4, /* valid but not built: other dims / bits / group sizes */
  IQ_ERR_CUDA = 5,        /* a CUDA runtime call failed (launch, copy, attribute) */
  IQ_ERR_DEVICE = 6       /* a kernel reported a failure in its status word */
} iq_status;

/* Static, NUL-terminated name of a status code ("IQ_OK", ...). */
const char* iq_status_string(int status);

/* Last error message of the calling host thread ("" if none). */
const char* iq_last_error(void);

/*
 * iq_build_rotation — the seed-fixed block-diagonal rotation
 * (quant_kv.py, `build_block_so4`, `_quat_left`, `_quat_right_conj`).
 *
 * draws_host: host float32 [head_dim/4][2][4], the raw standard-normal draws of
 *   each block's left then right quaternion, in generator order (the caller
 *   draws them; the library normalises them in float32 and forms
 *   L(qL) . R(qR) with float64 accumulation, rounded once to float32).
 * rot_f32: device float32 [head_dim/4][4][4] out (the blocks of M, what
 *   float32 caches use).
 * rot_bf16: device bf16 [head_dim/4][4][4] out (M_b = bf16(M), what bfloat16
 *   caches use).
 * The draws are copied to the device before the call returns, so the host
 * buffer may be reused at once.  Errors: INVALID_ARG (null, head_dim not a
 * positive multiple of 4), UNSUPPORTED (head_dim != 256), CUDA.
 */
int iq_build_rotation(int head_dim, const float* draws_host, float* rot_f32,
                      uint16_t* rot_bf16, iq_stream_t stream);

/*
 * iq_cache — plain descriptor of one quantised cache
 * (quant_kv.py, `AsymmetricQuantizedKVCache`: keys and values each stored as a
 * (wq, scales, biases) triple).  The caller owns every pointer.
 *
 *   dtype    IQ_DTYPE_BF16 or IQ_DTYPE_F32: the element type of the scales and
 *            biases and of every data argument the cache is used with
 *   k_codes  uint32 [B][Hkv][capacity][head_dim*k_bits/32]  (LSB-first stream)
 *   k_scales dtype  [B][Hkv][capacity][head_dim/group_size]
 *   k_biases dtype  [B][Hkv][capacity][head_dim/group_size]
 *   v_codes  uint32 [B][Hkv][capacity][head_dim*v_bits/32]
 *   v_scales, v_biases dtype as above
 *   lens     HOST int32 [B]: tokens held by each sequence.  This host array is
 *            the authoritative length; the library reads it to size launches
 *            and passes lengths to kernels by value, and updates it in
 *            iq_cache_append / iq_cache_trim / iq_cache_gather.
 * Device buffers must be 16-byte aligned; capacity must be a positive multiple
 * of IQ_STEP.  Rows at or past lens[b] are stale and are never read.
 */
typedef struct {
  int32_t batch, kv_heads, head_dim, group_size, k_bits, v_bits, capacity, dtype;
  uint32_t* k_codes;
  void* k_scales;
  void* k_biases;
  uint32_t* v_codes;
  void* v_scales;
  void* v_biases;
  int32_t* lens;
} iq_cache;

/*
 * iq_cache_bytes — byte sizes of the six device buffers of a cache
 * (quant_kv.py, `_init_quant`, `_packed_words`), in descriptor order
 * (k_codes, k_scales, k_biases, v_codes, v_scales, v_biases); scales and
 * biases take 2 bytes each for IQ_DTYPE_BF16 and 4 for IQ_DTYPE_F32.
 * Errors: INVALID_ARG (bad sizes, unknown dtype), UNSUPPORTED.
 */
int iq_cache_bytes(int batch, int kv_heads, int head_dim, int group_size, int k_bits,
                   int v_bits, int capacity, int dtype, size_t out_bytes[6]);

/*
 * iq_cache_alloc — bind the caller's six buffers and host lengths array into a
 * descriptor of an empty cache (quant_kv.py, `AsymmetricQuantizedKVCache`
 * construction: offset 0, buffers sized by `_init_quant` / `_packed_words`).
 * buffers: device pointers in descriptor order (k_codes, k_scales, k_biases,
 * v_codes, v_scales, v_biases), each at least the size iq_cache_bytes gives
 * and 16-byte aligned; lens_host: host int32 [batch], set to 0.  Nothing is
 * copied or launched.  Errors: INVALID_ARG, UNSUPPORTED (as iq_cache_check).
 */
int iq_cache_alloc(iq_cache* cache, int batch, int kv_heads, int head_dim, int group_size, int k_bits,
                   int v_bits, int capacity, int dtype, void* const buffers[6], int32_t* lens_host);

/*
 * iq_cache_check — validate a descriptor (quant_kv.py, the buffer layout of
 * `AsymmetricQuantizedKVCache`: shapes of a supported format, 16-byte aligned
 * buffers, lens in [0, capacity]).
 */
int iq_cache_check(const iq_cache* cache);

/*
 * iq_cache_grow — copy rows [0, lens[b]) of every sequence of `src` into the
 * larger `dst` and set dst.lens = src.lens (quant_kv.py, `update_and_fetch`'s
 * growth branch: a buffer ceil(n/256)*256 tokens larger, the old rows copied).
 * dst: the same batch, kv heads and format, capacity >= every src length,
 * buffers disjoint from src.  The same copy as iq_cache_gather with the
 * identity map.  Errors: as iq_cache_gather.
 */
int iq_cache_grow(const iq_cache* src, iq_cache* dst, iq_stream_t stream);

/* iq_cache_nbytes — total bytes of the six buffers (quant_kv.py, `nbytes`). */
size_t iq_cache_nbytes(const iq_cache* cache);

/*
 * iq_cache_append — rotate, group-quantise, bit-pack and store n new tokens per
 * sequence at rows [lens[b], lens[b] + n) (quant_kv.py, `rotate_last` +
 * `update_and_fetch`; quantiser scale = (max-min)/(2^b-1), bias = min,
 * code = clamp(round-half-even((x - bias)/scale))).
 *
 * keys, values: device [B][Hkv][n][head_dim] of the cache's dtype,
 *   contiguous, unrotated.
 * rot: device rotation blocks from iq_build_rotation in the cache's dtype
 *   (rot_bf16 for a bfloat16 cache, rot_f32 for a float32 one).
 * bfloat16: each rotated element is the float32 sum, in block-row order, of
 * exact bf16 x bf16 products, rounded once to bf16; the scale is rounded to
 * bf16 before the codes are formed from it.  float32: products and sums
 * rounded to float32 one by one in block-row order; scale and bias stored as
 * computed.  Either way codes come from the stored scale and bias.
 * On success lens[b] += n for every b.  n == 0 is a no-op.
 * Errors: INVALID_ARG, CAPACITY (some lens[b] + n > capacity; grow first —
 * see iq_cache_gather), UNSUPPORTED, CUDA.
 */
int iq_cache_append(iq_cache* cache, const void* keys, const void* values, int n, const void* rot,
                    iq_stream_t stream);

/*
 * iq_cache_trim — drop the last tokens of each sequence
 * (quant_kv.py, `trim`: n = min(offset, n); offset -= n; return n).
 * Host-only bookkeeping: no device work, no stream.
 * n_host: host int32 [B], non-negative counts.  trimmed_host: host int32 [B]
 * out (may be NULL).  Errors: INVALID_ARG (null, negative count).
 */
int iq_cache_trim(iq_cache* cache, const int32_t* n_host, int32_t* trimmed_host);

/*
 * iq_cache_gather — dst sequence i becomes a copy of src sequence src_of[i]:
 * rows [0, src.lens[src_of[i]]) of every kv head and all six buffers are
 * copied device to device and dst.lens[i] is set to that length.
 * This one copy serves capacity growth (identity map into a larger cache,
 * quant_kv.py `update_and_fetch` growth), snapshot and restore
 * (kv_cache.py `_snapshot` / `_restore`: the copy never aliases),
 * tiling a batch-1 cache to P paths (kv_cache.py `tile_caches`: all zeros) and
 * keeping the winning path (kv_cache.py `commit_tree_row`: one index).
 * src_of: host int32 [dst.batch].  src and dst must share kv_heads, head_dim,
 * group_size, bits and dtype, and must not overlap in memory.
 * Errors: INVALID_ARG, CAPACITY (dst capacity too small), UNSUPPORTED, CUDA.
 */
int iq_cache_gather(const iq_cache* src, iq_cache* dst, const int32_t* src_of,
                    iq_stream_t stream);

/*
 * iq_attend_workspace — device scratch bytes iq_attend needs for this batch
 * and these shapes (status word and the split-KV partial results); the size
 * does not depend on the lengths.
 */
#define IQ_WORKSPACE_HEAD_BYTES 8448u
int iq_attend_workspace(const iq_cache* cache, int q_heads, int n_queries, size_t* bytes);

/*
 * iq_attend — GQA attention of n_queries new queries per sequence over the
 * cache (quant_kv.py, `asym_quantized_sdpa`, followed by the inverse rotation
 * the page leaves to its caller).
 *
 * q: device [B][Hq][n_queries][head_dim] of the cache's dtype, unrotated.
 *    The library rotates it with the blocks `rot` (the cache's dtype, as in
 *    iq_cache_append; result rounded to that dtype), multiplies by `scale`
 *    (result rounded likewise; 1/sqrt(head_dim) is the usual value), and lets
 *    query head h read kv head h / (Hq/Hkv).
 * causal: 0 = every query sees all lens[b] tokens; 1 = query i sees tokens
 *    t <= lens[b] - n_queries + i (its own token already appended).
 * out: device [B][Hq][n_queries][head_dim], bf16 (out_f32 == 0) or float32
 *    (out_f32 == 1), in unrotated space: out = o @ rot^T rounded to the
 *    output type.
 * workspace: device buffer of at least iq_attend_workspace() bytes,
 *    256-byte aligned.  Its first IQ_WORKSPACE_HEAD_BYTES (the status word
 *    and per-unit partial counters) must be zero before the first call (e.g.
 *    a zero-filled allocation); the kernels return the counters to zero and
 *    only ever set bits in the status word, which iq_read_status clears.  The
 *    rest needs no initialisation.  Two kernels run per 1024 query tiles: the
 *    attention grid and, as its programmatic dependent, the split combine,
 *    which merges each split unit as soon as its partials are stored and
 *    completes after the attention grid.
 * Scores, softmax and P.V accumulate in float32; for bfloat16 caches of the
 * tuned format they run on tensor cores.  Key and
 * value codes enter the products exactly (as bare fp16 bit fields), queries as
 * q'' times a per-row power of two that keeps them inside fp16 (any bf16
 * query), P times the value scale as fp16 with the softmax reference raised
 * when a value scale reaches 2^9 (value groups of any bf16 range).  Calls with
 * 128 or more query rows per kv head take the tensor-memory prefill kernel,
 * whose dequantised values are fp16: a value at or above 2^15 in magnitude
 * sets status bit 16 there.
 * Errors: INVALID_ARG (null, bad causal flag, empty sequence, lens[b] <
 * n_queries when causal), WORKSPACE, UNSUPPORTED, CUDA.  A kernel-side failure
 * (a pipeline wait that timed out, an empty softmax row, a value outside the
 * prefill kernel's range) sets a bit in the workspace status word, reported by
 * iq_read_status.
 */
int iq_attend(const iq_cache* cache, const void* q, int q_heads, int n_queries,
              float scale, int causal, const void* rot, void* out, int out_f32,
              void* workspace, size_t workspace_bytes, iq_stream_t stream);

/*
 * iq_attend_mask — iq_attend with the page's general masks (quant_kv.py,
 * `asym_quantized_sdpa`: a bool mask keeps a score where true and replaces it
 * by the dtype's most negative value elsewhere; a float mask is added to the
 * scores).
 * mask_kind: IQ_MASK_NONE, IQ_MASK_CAUSAL (as iq_attend's causal flag),
 *    IQ_MASK_ADD_F32 (device float32, may hold -inf) or IQ_MASK_BOOL_U8
 *    (device uint8, 0 = masked).
 * mask: [B][n_queries][mask_stride] elements, row (b, i) covering keys
 *    0 .. lens[b]-1 (mask_stride >= every lens[b], a multiple of 128; the base
 *    16-byte aligned); shared by every query head.  The attention streams the
 *    rows in 128-key pieces with the cache tiles.
 * A row whose keys are all masked by a bool mask averages the values
 * uniformly, as the page's softmax does; a float-mask row that is -inf
 * everywhere has no softmax (NaN output, status bit 4).  Scores are float32:
 * a float mask should use -inf (not huge finite values) to exclude keys, and
 * scaled scores are taken to stay above -1e5 (bool-masked keys score -1e6).
 * Other arguments as iq_attend.  Errors: as iq_attend, plus INVALID_ARG for a
 * bad kind, a null or misaligned mask, or a mask row shorter than a sequence.
 */
#define IQ_MASK_NONE 0
#define IQ_MASK_CAUSAL 1
#define IQ_MASK_ADD_F32 2
#define IQ_MASK_BOOL_U8 3
int iq_attend_mask(const iq_cache* cache, const void* q, int q_heads, int n_queries, float scale,
                   int mask_kind, const void* mask, long long mask_stride, const void* rot,
                   void* out, int out_f32, void* workspace, size_t workspace_bytes, iq_stream_t stream);

/*
 * iq_cache_append_attend — iq_cache_append(keys, values, n) followed by
 * iq_attend(q, ...), the page's decode step (quant_kv.py: `update_and_fetch`,
 * then `asym_quantized_sdpa` over the updated cache), with the same results
 * as the two calls.  For a bfloat16 cache of the tuned format it is one
 * launch in two cases:
 *  - every (sequence, kv head) holds at most 8 query rows (q_heads / kv_heads
 *    * n_queries <= 8) and each sequence's n new rows fall in one 128-token
 *    tile: the split-KV attention, whose CTAs encode the new rows themselves
 *    before streaming the tiles that hold them;
 *  - 128 or more query rows per kv head and at most 2046 (sequence, kv head)
 *    pairs: the tensor-memory prefill kernel, whose CTAs take the new rows in
 *    chunks from a counter in the workspace head, encode them, and stream a
 *    sequence's tiles holding new rows only once all of that sequence's new
 *    rows are stored (a wait that runs out sets status bit 0x20000).
 * Otherwise it is the append launch followed by the attention.
 * Arguments, layouts and workspace as iq_cache_append and iq_attend; lens[b]
 * grows by n on success (the causal mask and the scanned length use the
 * grown lengths).  Errors: as both (nothing is launched on an error).
 * Overlap: an attention grid starts streaming cache tiles while the previous
 * call's grids finish (only its stores wait for them).  The library remembers,
 * per key-code buffer, the rows the latest attention on it reads; when a trim
 * since then puts the new rows below that mark, the fused encode also waits.
 * Writing the cache by other means (outside this library's calls) while a call
 * on the same stream is in flight is not supported.
 */
int iq_cache_append_attend(iq_cache* cache, const void* keys, const void* values, int n,
                           const void* q, int q_heads, int n_queries, float scale, int causal,
                           const void* rot, void* out, int out_f32, void* workspace,
                           size_t workspace_bytes, iq_stream_t stream);

/*
 * iq_attend_noalloc — iq_attend for callers that cannot allocate device
 * memory.  (The source pages have no counterpart: this is a library service.)
 *
 * Some callers cannot call cudaMalloc for a workspace: a serving process whose
 * allocator already owns all of HBM (weights and KV pool), a plugin that only
 * receives the buffers its host hands it, or a decode loop where an allocation
 * (which can synchronise the device) would break the latency budget.  This
 * entry point computes exactly what iq_attend computes, with its scratch in a
 * library-owned device array of IQ_NOALLOC_SCRATCH_BYTES (16 MiB) that every
 * GPU using this entry point keeps until the process exits.  It allocates
 * nothing and calls no allocating routine; the caller still passes q and out.
 *
 * Set-up: the first call on a device (this one or iq_noalloc_read_status)
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current.  With CUDA's lazy module loading that is also when the array's
 * memory is reserved on the device, so make the first call at start-up:
 * before the caller's own allocator takes the rest of device memory, and
 * before any stream capture (iq_noalloc_read_status does the set-up and
 * nothing else when nothing has run).
 * Sharing: every call uses the same array and it keeps the last call's
 * contents (the partials are written before they are read; the head, zero at
 * load, returns its unit counters to zero after every call, also one whose
 * wait ran out, and its status word only gains bits until
 * iq_noalloc_read_status clears it).  Calls that can run at the same time on
 * the GPU (different streams without ordering) race on the array: serialise
 * them.
 * Errors: as iq_attend, plus WORKSPACE when the call needs more scratch than
 * IQ_NOALLOC_SCRATCH_BYTES (use iq_attend with a caller workspace then); calls
 * that take the tensor-memory prefill kernel need only the IQ_WORKSPACE_HEAD_BYTES head.
 * Kernel-side failures land in the shared status word: read it with
 * iq_noalloc_read_status.
 */
#define IQ_NOALLOC_SCRATCH_BYTES (16u << 20)
int iq_attend_noalloc(const iq_cache* cache, const void* q, int q_heads, int n_queries,
                      float scale, int causal, const void* rot, void* out, int out_f32,
                      iq_stream_t stream);

/*
 * iq_noalloc_read_status — iq_read_status for the library-owned scratch of
 * iq_attend_noalloc on the current device (no counterpart on the pages):
 * synchronise `stream`, read the status word the noalloc calls left, and clear
 * it (after a failure, the whole head).  Allocates nothing.  Blocks the
 * calling thread.  *device_status is 0 when every kernel completed normally.
 */
int iq_noalloc_read_status(iq_stream_t stream, int* device_status);

/*
 * iq_debug_inject — a fault-injection hook for tests (no counterpart on the
 * pages).  The next split-KV attention call made from this host thread (the
 * decode / verify kernels; not the prefill kernel or the generic formats)
 * uses `spin_limit` mbarrier tests per pipeline wait (0: the default, seconds)
 * and a combine wait of `combine_wait_ns` (0: the default, 4 s), and injects
 * the failures in `flags`:
 *   IQ_INJECT_COMBINE_WAIT: the combine waits for one partial more than will
 *     ever be stored, so its wait runs out (status bit 8);
 *   IQ_INJECT_STAGE_NEVER_FILLED: the consumers wait, in place of their first
 *     stage, on a barrier that nothing completes in a call without new rows
 *     (iq_attend), so their wait runs out (status bit 2, and bit 1 when the
 *     producer's own wait for the stage to be released runs out).
 * Every wait still ends within its limit and the kernels return normally (no
 * fault, trap or unbounded wait); outputs of that call are not meaningful.
 * The setting then resets.  Errors: INVALID_ARG (unknown flag).
 */
#define IQ_INJECT_COMBINE_WAIT 1
#define IQ_INJECT_STAGE_NEVER_FILLED 2
int iq_debug_inject(int flags, unsigned spin_limit, unsigned long long combine_wait_ns);

/*
 * iq_read_status — synchronise `stream`, read the status word that the
 * iq_attend calls on this workspace since the last read left, and clear it
 * (after a failure, the whole workspace head).  *device_status is 0 when
 * every kernel completed normally.  Blocks the calling thread.
 */
int iq_read_status(void* workspace, iq_stream_t stream, int* device_status);

#ifdef __cplusplus
}
#endif
#endif /* IQKV_H */
