/*
 * pkv.h -- C ABI of libpkv.so: a paged KV cache for single-token decode
 * attention on one GB300 (sm_103a).
 *
 * Sources the operations restate (web pages, by title and section):
 *   [A] "无 vLLM 环境下的 Paged-KV 与连续批处理调度" (mixtureofinsights.com)
 *   [B] "vLLM核心概念：PagedAttention、Continuous Batching、KV Cache等原理" (5688vip.com, ch. 3)
 *   [C] "离开 N 卡后的真实世界：Ultra x7 358h 平台上的 TTS 推理框架重构" (mixtureofinsights.com)
 *   [D] "连续批处理与KV缓存" (5688vip.com, course ch. 4)
 *   [E] "轻量级推理引擎实战：KV Cache 量化与连续批处理的底层优化" (lpnh.cn)
 *
 * Conventions
 *   - Every function returns an int status (PKV_OK or a negative PKV_ERR_*),
 *     except the two size queries and the allocator constructor.
 *   - Host functions (allocator, tables) touch only host memory and are not
 *     thread-safe: callers serialise access to one allocator.
 *   - Device functions enqueue kernels on the given CUDA stream (a
 *     cudaStream_t passed as void*; NULL = legacy default stream) and return
 *     without synchronising. They validate their scalar arguments and pointer
 *     alignment on the host and return PKV_ERR_INVALID / PKV_ERR_UNSUPPORTED
 *     without launching anything; PKV_ERR_CUDA reports a launch failure.
 *     Values that live in device memory (block ids, slots, context lengths)
 *     are checked inside the kernels: an out-of-range value is skipped (no
 *     memory access is made with it) and, if the descriptor carries an error
 *     word, a PKV_DEVERR_* bit is OR-ed into it.
 *   - All device buffers are owned by the caller. No device function
 *     allocates memory. bf16 data is passed as raw 16-bit words.
 *
 * Layout (all row-major, per layer):
 *   k_pool, v_pool  [num_blocks][Hkv][block_size][head_dim]  bf16 or int8
 *   scales          [num_blocks][Hkv][2] fp32 (INT8 only; [..][0] = K, [..][1] = V)
 *   k_tail, v_tail  [max_slots][Hkv][block_size][head_dim] bf16 (INT8 only)
 *   block tables    [B][max_blocks] int32, logical block -> physical block, -1 pad
 *   q, out          [B][Hq][head_dim] bf16
 *   query head h reads kv head h / (Hq / Hkv).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------- */
#define PKV_OK                 0
#define PKV_ERR_INVALID       -1  /* null pointer, bad size or alignment */
#define PKV_ERR_OOM           -2  /* not enough free blocks; nothing changed */
#define PKV_ERR_NOT_FOUND     -3  /* request id is not live */
#define PKV_ERR_EXISTS        -4  /* request id is already live */
#define PKV_ERR_UNSUPPORTED   -5  /* shape outside the compiled set (see below) */
#define PKV_ERR_CUDA          -6  /* a CUDA runtime call failed */
#define PKV_ERR_DEVICE_TIMEOUT -7 /* a kernel's bounded wait expired (pkv_sync_status) */
#define PKV_ERR_TOO_LARGE     -8  /* the request needs more than the library's fixed scratch array */

/* bits a kernel ORs into the descriptor's error word */
#define PKV_DEVERR_BLOCK_ID    1  /* block id < 0 or >= num_blocks */
#define PKV_DEVERR_SLOT        2  /* slot < 0 or >= max_slots */
#define PKV_DEVERR_CTX_LEN     4  /* context length < 0 or > max_blocks * block_size */
#define PKV_DEVERR_OFFSET      8  /* in-block offset < 0 or >= block_size */
#define PKV_DEVERR_TIMEOUT    16  /* a bounded wait on an asynchronous copy expired */

#define PKV_DTYPE_BF16 0
#define PKV_DTYPE_INT8 1

/* Compiled shapes: head_dim in {64, 128}; block_size in {16, 64};
 * Hq / Hkv in {1, 2, 4, 8}. */

/* ======================================================================== */
/* Host block allocator ([D] §4.2; [A] §1.2; [B] §3.2; [E] §2.1)            */
/* ======================================================================== */

/* A FIFO pool of block ids: allocations take ids from the front, frees
 * return them to the back, each in O(1) per block ([D] §4.2's free-block pool).
 * Each live request owns an ordered list of private blocks, optionally
 * preceded by shared blocks (a common prompt prefix, [B] §3.2) that it
 * references but does not own. */
typedef struct pkv_allocator pkv_allocator;

/* Creates a pool of num_blocks ids. initial_order (nullable, num_blocks
 * entries, a permutation of 0..num_blocks-1) sets the initial free-list
 * order, e.g. a shuffled pool; NULL means 0, 1, 2, ... block_size is
 * recorded for the caller's arithmetic. Returns NULL on invalid arguments or
 * host allocation failure. The handle owns only host memory. */
pkv_allocator* pkv_allocator_create(int32_t num_blocks, int32_t block_size,
                                    const int32_t* initial_order);
void pkv_allocator_destroy(pkv_allocator* a);

/* All-or-nothing allocation of n_blocks >= 0 private blocks for a new
 * request ([D] §4.2 "allocate"): writes the ids, in order, to out_ids
 * (n_blocks entries; may be NULL when n_blocks == 0).
 * PKV_ERR_OOM if fewer are free (pool unchanged); PKV_ERR_EXISTS if req_id is
 * live (the page's sketch would silently overwrite it and leak its blocks). */
int pkv_alloc(pkv_allocator* a, int64_t req_id, int32_t n_blocks, int32_t* out_ids);

/* One more block at the end of a live request's list ([D] §4.2
 * "append_block"; [E] §2.1 on-demand allocation). PKV_ERR_OOM when the pool
 * is empty ("wait"), PKV_ERR_NOT_FOUND for an unknown request. */
int pkv_append_block(pkv_allocator* a, int64_t req_id, int32_t* out_id);

/* Drops the request's hold on its blocks and forgets the request ([D] §4.2
 * "free"): each block no other live request holds (see pkv_fork) goes to the
 * back of the free list, in the order the request held them.
 * PKV_ERR_NOT_FOUND (no change) for an unknown request. */
int pkv_free(pkv_allocator* a, int64_t req_id);

/* Copy-on-write forking ([B] §3.2: requests sharing a prefix point at the
 * same physical blocks, and a block is copied only when one of them needs to
 * write into it -- parallel sampling, beam search). A block's reference count
 * is the number of live requests holding it (1 after pkv_alloc or
 * pkv_append_block).
 *
 * pkv_fork: new request `child` holds every block of live request `parent`
 * (same table, pinned prefix included); each held block's count goes up by
 * one. PKV_ERR_NOT_FOUND (parent), PKV_ERR_EXISTS (child); no change then. */
int pkv_fork(pkv_allocator* a, int64_t parent, int64_t child);

/* Before request req_id writes into its logical block `index`: if that block
 * is also held by another request, a block from the front of the free list
 * takes its place in req_id's table (the old block's count drops by one)
 * and *out_src / *out_dst receive the old and new ids -- the caller copies
 * the old block's contents into the new one (pkv_copy_blocks) before
 * writing. A block held by req_id alone needs nothing: *out_src = *out_dst
 * = -1. PKV_ERR_OOM if a copy is needed and the pool is empty (no change);
 * PKV_ERR_INVALID for an index past the table or inside the pinned prefix
 * (pkv_attach_shared blocks are read-only); PKV_ERR_NOT_FOUND for an unknown
 * request. */
int pkv_cow_block(pkv_allocator* a, int64_t req_id, int32_t index, int32_t* out_src, int32_t* out_dst);

/* Reference count of a block (0 = free, or pinned-only); PKV_ERR_INVALID for
 * an id outside the pool. */
int pkv_block_refs(const pkv_allocator* a, int32_t block);

/* Puts n shared block ids in front of a live request's table. They are
 * never returned by pkv_free; their owner (the request that allocated them)
 * frees them. No check is made that the ids are live. */
int pkv_attach_shared(pkv_allocator* a, int64_t req_id, const int32_t* ids, int32_t n);

/* Number of free blocks; -1 for a NULL handle. */
int pkv_num_free(const pkv_allocator* a);

/* Writes up to cap ids of the request's table (shared then private) to out
 * (nullable when cap == 0) and returns the table length, or a negative
 * status. */
int pkv_request_table(const pkv_allocator* a, int64_t req_id, int32_t* out, int32_t cap);

/* Writes up to cap ids of the free list, front first, and returns its length. */
int pkv_free_list(const pkv_allocator* a, int32_t* out, int32_t cap);

/* Block tables for B requests: out_table[B][max_blocks] (host memory), each
 * row the request's table padded with -1 ([B] §3.2, [E] §2.1 "Block Table").
 * PKV_ERR_NOT_FOUND for an unknown request, PKV_ERR_INVALID if a table is
 * longer than max_blocks; out_table is then unspecified. */
int pkv_build_block_tables(const pkv_allocator* a, const int64_t* req_ids, int32_t B,
                           int32_t max_blocks, int32_t* out_table);

/* ======================================================================== */
/* Device side                                                             */
/* ======================================================================== */

/* One layer's cache. Pools and tails must be 16-byte aligned. In BF16 mode
 * scales, k_tail and v_tail are unused (may be NULL) and max_slots may be 0.
 * err_word (nullable) is a device int32 the kernels OR PKV_DEVERR_* bits into. */
typedef struct pkv_cache_desc {
    void*    k_pool;
    void*    v_pool;
    float*   scales;
    void*    k_tail;
    void*    v_tail;
    int32_t  num_blocks;
    int32_t  num_q_heads;
    int32_t  num_kv_heads;
    int32_t  head_dim;
    int32_t  block_size;
    int32_t  max_slots;
    int32_t  dtype;          /* PKV_DTYPE_BF16 or PKV_DTYPE_INT8 */
    int32_t* err_word;
} pkv_cache_desc;

/* Per-step append ([D] §4.2 "expand: a request that generates a new token
 * appends to its cache"; [E] §2.1). Writes the T new rows k[T][Hkv][d],
 * v[T][Hkv][d] (device, bf16) of token t at in-block offset offsets[t]:
 *   BF16 mode: into pool block block_ids[t];
 *   INT8 mode: into the bf16 tail of sequence slot slots[t] (the block is
 *              quantized into the pool once it fills, see below).
 * block_ids (BF16) / slots (INT8) and offsets are device int32 [T]; the
 * unused one may be NULL. T == 0 is a no-op. */
int pkv_append_kv(const pkv_cache_desc* c, const void* k, const void* v,
                  const int32_t* block_ids, const int32_t* offsets, const int32_t* slots,
                  int32_t T, void* stream);

/* Quantize-on-fill ([E] §3 quantize_block, granularity per
 * (block, kv_head, K|V)): for each m < M, quantizes the full bf16 tail of
 * slot slots[m] into pool block block_ids[m] and writes its scales:
 *   s = max|x| / 127 (fp32 IEEE division), or 1.0 if max|x| < 1e-6;
 *   q = clamp(round_half_even(x / s), -127, 127) (fp32 IEEE division).
 * The bytes and scales are a deterministic function of the tail's bf16
 * values. INT8 mode only. block_ids, slots: device int32 [M]; an entry whose
 * block id is -1 is skipped, so a fixed-size list may be padded (e.g. one
 * entry per running sequence, -1 where no block filled this step). */
int pkv_quantize_full_blocks(const pkv_cache_desc* c, const int32_t* block_ids,
                             const int32_t* slots, int32_t M, void* stream);

/* Same quantization with a caller-given source instead of a tail: block m
 * takes rows m*block_size .. m*block_size+block_size-1 of k_src / v_src
 * ([M*block_size][Hkv][d] bf16, device) -- e.g. the full blocks of a prompt.
 * INT8 mode only. */
int pkv_quantize_blocks_from(const pkv_cache_desc* c, const void* k_src, const void* v_src,
                             const int32_t* block_ids, int32_t M, void* stream);

/* Copies whole pool blocks, src_ids[i] -> dst_ids[i] for i < n (device int32
 * arrays): the K and V rows of every kv head and, INT8, the block's scales
 * -- the copy half of copy-on-write ([B] §3.2; the ids come from
 * pkv_cow_block). src_ids[i] < 0 or == dst_ids[i] is an entry with nothing
 * to copy; another id outside [0, num_blocks) is skipped and reported
 * (PKV_DEVERR_BLOCK_ID). Destinations must not overlap sources in flight.
 * In INT8 mode a block that has not filled yet holds no pool data (its rows
 * are in the slot's tail), so a write into a shared partial block needs the
 * tail copied (pkv_copy_slots, at fork time) but no pool copy. */
int pkv_copy_blocks(const pkv_cache_desc* c, const int32_t* src_ids, const int32_t* dst_ids, int32_t n,
                    void* stream);

/* INT8 mode: copies the bf16 tails of slots src_slots[i] -> dst_slots[i]
 * (device int32, n entries; negative src = nothing to copy; other indices
 * outside [0, max_slots) skipped and reported as PKV_DEVERR_SLOT) -- a
 * forked request starts from its parent's partly filled block.
 * PKV_ERR_INVALID in BF16 mode. */
int pkv_copy_slots(const pkv_cache_desc* c, const int32_t* src_slots, const int32_t* dst_slots, int32_t n,
                   void* stream);

/* Decode attention ([B] §3.1 one new query against all cached K, V;
 * [E] §1 each decode step reads the whole cache; [A] §2 GQA; [C] §2 tiled
 * softmax in on-chip memory). For each sequence b < B and query head h:
 *   out[b][h] = sum_t softmax_t(sm_scale * q[b][h] . k_t) v_t
 * over the ctx_lens[b] tokens t of sequence b, where token t lives in block
 * block_tables[b][t / bs] at offset t % bs, dequantized as q * scale in INT8
 * mode -- except that in INT8 mode the last ctx_lens[b] % bs tokens (the
 * partly filled block) are read from the bf16 tail of slot slots[b].
 * Accumulation is fp32; out is bf16. ctx_lens[b] == 0 gives a zero row.
 *
 * split_tokens == 0: one pass per (b, kv_head); the workspace is unused (NULL ok).
 * split_tokens > 0 (a multiple of block_size and of 16): the context is cut
 *   into chunks of split_tokens tokens, computed independently into the
 *   caller's workspace and then merged. Needs
 *   max_splits * split_tokens >= max_blocks * block_size and
 *   ws_o  >= pkv_splitk_ws_o_bytes(B, Hq, d, max_splits),
 *   ws_ml >= pkv_splitk_ws_ml_bytes(B, Hq, max_splits), 16-byte aligned.
 *   ws_count NULL: the merge is a second kernel (pkv_splitk_reduce) on the
 *   same stream. ws_count non-NULL: device int32 [B][Hkv], all zero before
 *   the first call; the last split of each (b, kv_head) to finish merges in
 *   the same kernel and sets its counter back to zero, so the array stays
 *   ready for the next call (a sequence whose context fits one split writes
 *   its output directly, leaving workspace and counter untouched). Calls
 *   sharing a workspace must not overlap.
 * slots may be NULL in BF16 mode. With rows of 128 or 256 bytes (INT8 or bf16
 * at head_dim 128, bf16 at head_dim 64) the kernel reads the pools through
 * tensor maps that the call encodes on the host (cached per thread);
 * PKV_ERR_CUDA if the driver's encoder is unavailable or refuses the pool. */
int pkv_decode_attention(const pkv_cache_desc* c, const void* q, const int32_t* block_tables,
                         int32_t max_blocks, const int32_t* ctx_lens, const int32_t* slots,
                         int32_t B, float sm_scale, int32_t split_tokens, int32_t max_splits,
                         float* ws_o, float* ws_ml, int32_t* ws_count, void* out, void* stream);

/* One layer's whole decode step in one kernel: for each sequence b, append
 * the new rows k_new[b], v_new[b] ([B][Hkv][d] bf16, device, 16-byte
 * aligned; PKV_ERR_INVALID otherwise) as token
 * ctx_lens[b] - 1 (BF16: into block block_tables[b][(ctx_lens[b]-1)/bs],
 * which must already be allocated; INT8: into the tail of slots[b]); in INT8
 * mode, if that token fills its block, quantize the block into the pool
 * exactly as pkv_quantize_full_blocks does; then attend over ctx_lens[b]
 * tokens exactly as pkv_decode_attention does. The result equals
 * pkv_append_kv + pkv_quantize_full_blocks + pkv_decode_attention; the
 * row is written (and the block quantized) by the CTA that reads it, so no
 * separate kernel sits between the layer's inputs and its attention. All
 * other arguments are those of pkv_decode_attention. */
int pkv_decode_step(const pkv_cache_desc* c, const void* q, const void* k_new, const void* v_new,
                    const int32_t* block_tables, int32_t max_blocks, const int32_t* ctx_lens,
                    const int32_t* slots, int32_t B, float sm_scale, int32_t split_tokens,
                    int32_t max_splits, float* ws_o, float* ws_ml, int32_t* ws_count, void* out,
                    void* stream);

/* A whole decode step over num_layers layers in one call, layer l after
 * layer l-1 on the stream: layer l runs pkv_decode_step on descs[l] with
 * q + l*q_layer_stride, k_new/v_new + l*kv_layer_stride and
 * out + l*out_layer_stride (strides in bytes, multiples of 16; k_new and
 * v_new 16-byte aligned), or pkv_decode_attention when k_new and v_new are
 * both NULL (one NULL without the other: PKV_ERR_INVALID). The block tables,
 * context lengths, slots, split settings and workspace are shared by all
 * layers (the layers of a model allocate the same blocks). Stops at, and
 * returns, the first error. */
int pkv_decode_layers(const pkv_cache_desc* descs, int32_t num_layers, const void* q,
                      int64_t q_layer_stride, const void* k_new, const void* v_new,
                      int64_t kv_layer_stride, void* out, int64_t out_layer_stride,
                      const int32_t* block_tables, int32_t max_blocks, const int32_t* ctx_lens,
                      const int32_t* slots, int32_t B, float sm_scale, int32_t split_tokens,
                      int32_t max_splits, float* ws_o, float* ws_ml, int32_t* ws_count, void* stream);

/* CTAs of the decode kernel for this cache shape that fit on one SM at once
 * (registers and shared memory), for a given split_tokens (0 = none) and
 * max_blocks; a caller sizes its splits so that B * Hkv * splits fills
 * SMs x this number. Returns a negative status on invalid arguments. */
int pkv_decode_ctas_per_sm(const pkv_cache_desc* c, int32_t split_tokens, int32_t max_blocks);

/* Split-K merge of partial softmax states (the combination rule of a
 * softmax over a partition of the context; the pages' tiled softmax, [C] §2).
 * ws_o [B][Hq][max_splits][d] and ws_ml [B][Hq][max_splits][2] fp32 hold,
 * for split j < ceil(ctx_lens[b] / split_tokens): m_j, l_j and
 * o_j = sum_t 2^(x_t - m_j) v_t with x_t = log2(e) * sm_scale * q . k_t
 * (so m is in log2 units) and l_j = sum_t 2^(x_t - m_j). Writes
 *   out[b][h] = sum_j 2^(m_j - M) o_j / sum_j 2^(m_j - M) l_j,  M = max_j m_j
 * as bf16 (a zero row when ctx_lens[b] == 0). */
int pkv_splitk_reduce(const float* ws_o, const float* ws_ml, const int32_t* ctx_lens,
                      int32_t B, int32_t Hq, int32_t head_dim, int32_t split_tokens,
                      int32_t max_splits, void* out, void* stream);

size_t pkv_splitk_ws_o_bytes(int32_t B, int32_t Hq, int32_t head_dim, int32_t max_splits);
size_t pkv_splitk_ws_ml_bytes(int32_t B, int32_t Hq, int32_t max_splits);

/* Reads, clears and reports the error words of n descriptors once the work
 * queued on `stream` has finished: synchronises the stream, copies each
 * descriptor's err_word to the host (descriptors with a NULL err_word are
 * skipped; descriptors may share one word), resets every nonzero word to 0
 * on the stream, and writes the OR of the words to *out_bits (nullable).
 * Returns PKV_ERR_DEVICE_TIMEOUT if PKV_DEVERR_TIMEOUT was set (a bounded
 * wait of a kernel expired: its outputs are meaningless, later launches are
 * unaffected), else PKV_ERR_INVALID if any other PKV_DEVERR_* bit was set (a
 * block id, slot, context length or offset in device memory was out of range
 * and skipped), else PKV_OK; PKV_ERR_CUDA if a CUDA call failed. Host-side,
 * blocking; not for use inside stream capture. */
int pkv_sync_status(const pkv_cache_desc* descs, int32_t n, void* stream, int32_t* out_bits);

/* Process-wide switch (default off) for programmatic dependent launch: with
 * it on, every kernel of this library is launched so that it may start while
 * the previous kernel on the stream is still running, and each waits for that
 * kernel to complete before it reads anything the kernel could have written.
 * The one exception is the early start of pkv_decode_attention: before its
 * wait it already reads ctx_lens, block_tables, slots, and the cache blocks
 * (and scales) below the block holding each sequence's last token. With the
 * switch on, those must therefore not be written by the kernel launched just
 * before on the same stream (this library's append and quantize kernels
 * write only the last block). Lets a decode step's per-layer kernels overlap
 * each other's launch and drain. */
int pkv_set_programmatic_launch(int enable);

/* Test hook for the bounded waits (no counterpart on the pages): with tile
 * >= 0, decode launches issued afterwards run a separately compiled test
 * build of the decode kernel (head_dim 64 only; other shapes then return
 * PKV_ERR_UNSUPPORTED) that leaves the K/V copies of that tile of warp 0 of
 * its first CTA unissued, so that warp's wait on it runs out (about a
 * second), PKV_DEVERR_TIMEOUT is OR-ed into the error word, and the kernel
 * drains its other copies (each wait again bounded) and returns -- the GPU
 * stays usable and later launches are unaffected. The outputs of the
 * affected (sequence, kv head) are then meaningless. -1 (the default) turns
 * it off and selects the regular kernels, which carry no such check.
 * PKV_ERR_INVALID for tile < -1. Process-wide. */
int pkv_debug_skip_copy(int32_t tile);

/* Bytes of the library-owned split-K scratch array used by
 * pkv_decode_attention_static_ws (8 MiB, held on every GPU that loads the
 * library for the life of the process). */
#define PKV_STATIC_WS_BYTES (8u << 20)

/* pkv_decode_attention without a caller-provided workspace: the pages have
 * no counterpart; this exists for callers that cannot allocate device memory
 * when they decode -- an engine that gives all free HBM to its cache pool at
 * start-up and forbids later allocations, code running inside such an
 * engine, or a latency-critical loop that must not pay for cudaMalloc's
 * implicit synchronisation. The split-K partials and the merge's arrival
 * counters live in a fixed array inside the library; this function allocates
 * nothing and calls no allocating routine.
 *
 * Arguments and results are those of pkv_decode_attention with split_tokens
 * and max_splits as given (split_tokens == 0 uses no scratch at all). The
 * scratch needed is B*Hkv*4 bytes of counters plus
 * pkv_splitk_ws_ml_bytes(B, Hq, max_splits) and
 * pkv_splitk_ws_o_bytes(B, Hq, d, max_splits), each part rounded up to
 * 256 bytes; if that exceeds PKV_STATIC_WS_BYTES the call returns
 * PKV_ERR_TOO_LARGE and launches nothing.
 *
 * The array is part of the library's device code: it takes device memory when
 * that code is loaded on a device -- with CUDA's lazy module loading, at the
 * library's first kernel launch or first call of this function there. The
 * first call on a device also looks up the array's device address on that
 * device (the current one). Make that first call (or any launch of this
 * library) on each device before the caller hands the device's free memory to
 * a pool, and before any stream capture; after cudaDeviceReset the cached
 * address is stale and the process must not call this function again.
 * split_tokens < 0 returns PKV_ERR_INVALID.
 * Every call on a device shares the one array and it keeps the last call's
 * contents: each call first clears its counters (an asynchronous memset on
 * the stream), then writes its partials before reading them. Calls whose
 * executions overlap on the GPU -- on different streams, or from different
 * host threads -- race on the array and give wrong results; serialise them. */
int pkv_decode_attention_static_ws(const pkv_cache_desc* c, const void* q, const int32_t* block_tables,
                                   int32_t max_blocks, const int32_t* ctx_lens, const int32_t* slots,
                                   int32_t B, float sm_scale, int32_t split_tokens, int32_t max_splits,
                                   void* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
