// C ABI of libpkv.so: argument validation and kernel launches for the
// append, quantize-on-fill, decode-attention and split-K-merge entry points
// declared in include/pkv.h. Every entry point launches on the caller's
// stream and never allocates device memory.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

#include <nvtx3/nvToolsExt.h>

#include "../../include/pkv.h"
#include "decode_registry.h"

namespace pkv {

// ---------------------------------------------------------------------------
// Append: one 16-byte chunk of one (token, K|V, kv head) row per thread.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) append_kernel(const uint16_t* __restrict__ k,
                                                     const uint16_t* __restrict__ v,
                                                     const int32_t* __restrict__ block_ids,
                                                     const int32_t* __restrict__ offsets,
                                                     const int32_t* __restrict__ slots, int32_t T,
                                                     int32_t Hkv, int32_t bs, int32_t num_blocks,
                                                     int32_t max_slots, int int8_mode, void* k_dst,
                                                     void* v_dst, int32_t* err) {
    constexpr int CH = D / 8;  // 16-byte chunks per row
    pdl_launch_dependents();
    pdl_wait();
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t rows = int64_t(T) * 2 * Hkv;
    if (e >= rows * CH) return;
    const int64_t r = e / CH;
    const int c = int(e % CH);
    const int t = int(r / (2 * Hkv));
    const int kv = int((r / Hkv) % 2);
    const int h = int(r % Hkv);
    const int off = offsets[t];
    if (off < 0 || off >= bs) {
        if (c == 0) report(err, kErrOffset);
        return;
    }
    int64_t row;
    if (int8_mode) {
        const int s = slots[t];
        if (s < 0 || s >= max_slots) {
            if (c == 0) report(err, kErrSlot);
            return;
        }
        row = (int64_t(s) * Hkv + h) * bs + off;
    } else {
        const int blk = block_ids[t];
        if (blk < 0 || blk >= num_blocks) {
            if (c == 0) report(err, kErrBlockId);
            return;
        }
        row = (int64_t(blk) * Hkv + h) * bs + off;
    }
    const uint16_t* src = (kv ? v : k) + (int64_t(t) * Hkv + h) * D + c * 8;
    uint16_t* dst = static_cast<uint16_t*>(kv ? v_dst : k_dst) + row * D + c * 8;
    *reinterpret_cast<uint4*>(dst) = ldg128(src);
}

// ---------------------------------------------------------------------------
// Quantize: one warp per (block m, kv head, K|V) slab of bs x D bf16 values.
//   scale = max|x| / 127 (IEEE fp32 division), 1.0 if max|x| < 1e-6;
//   q = clamp(rint(x / scale), -127, 127), IEEE fp32 division, ties to even.
// The source slab is rows [bs] with a row stride (elements) and a base.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(128) quantize_kernel(const uint16_t* __restrict__ k_src,
                                                       const uint16_t* __restrict__ v_src,
                                                       int from_tail, const int32_t* __restrict__ block_ids,
                                                       const int32_t* __restrict__ slots, int32_t M,
                                                       int32_t Hkv, int32_t bs, int32_t num_blocks,
                                                       int32_t max_slots, int8_t* k_pool, int8_t* v_pool,
                                                       float* scales, int32_t* err) {
    pdl_launch_dependents();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t slab = int64_t(blockIdx.x) * 4 + warp;
    if (slab >= int64_t(M) * 2 * Hkv) return;
    const int m = int(slab / (2 * Hkv));
    const int kv = int((slab / Hkv) % 2);
    const int h = int(slab % Hkv);
    const int blk = block_ids[m];
    if (blk == -1) return;  // padding entry of a fixed-size list
    if (blk < 0 || blk >= num_blocks) {
        if (lane == 0) report(err, kErrBlockId);
        return;
    }
    const uint16_t* base;
    int64_t row_stride;
    if (from_tail) {
        const int s = slots[m];
        if (s < 0 || s >= max_slots) {
            if (lane == 0) report(err, kErrSlot);
            return;
        }
        base = (kv ? v_src : k_src) + (int64_t(s) * Hkv + h) * bs * D;
        row_stride = D;
    } else {
        base = (kv ? v_src : k_src) + (int64_t(m) * bs * Hkv + h) * D;
        row_stride = int64_t(Hkv) * D;
    }
    int8_t* dst = (kv ? v_pool : k_pool) + (int64_t(blk) * Hkv + h) * bs * D;
    quantize_slab<D, false>(lane, base, row_stride, bs, dst, scales + (int64_t(blk) * Hkv + h) * 2 + kv);
}

// ---------------------------------------------------------------------------
// Host helpers
// ---------------------------------------------------------------------------
static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static int check_desc(const pkv_cache_desc* c) {
    if (!c || !c->k_pool || !c->v_pool) return PKV_ERR_INVALID;
    if (!aligned16(c->k_pool) || !aligned16(c->v_pool)) return PKV_ERR_INVALID;
    if (c->num_blocks <= 0 || c->num_q_heads <= 0 || c->num_kv_heads <= 0) return PKV_ERR_INVALID;
    if (c->dtype != PKV_DTYPE_BF16 && c->dtype != PKV_DTYPE_INT8) return PKV_ERR_INVALID;
    if (c->head_dim != 64 && c->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (c->block_size != 16 && c->block_size != 64) return PKV_ERR_UNSUPPORTED;
    if (c->num_q_heads % c->num_kv_heads) return PKV_ERR_UNSUPPORTED;
    const int g = c->num_q_heads / c->num_kv_heads;
    const bool g_ok = g == 1 || g == 2 || g == 4 || g == 8;
    if (!g_ok) return PKV_ERR_UNSUPPORTED;
    if (c->dtype == PKV_DTYPE_INT8) {
        if (!c->scales || !c->k_tail || !c->v_tail || c->max_slots <= 0) return PKV_ERR_INVALID;
        if (!aligned16(c->k_tail) || !aligned16(c->v_tail) ||
            (reinterpret_cast<uintptr_t>(c->scales) & 7u))
            return PKV_ERR_INVALID;
    }
    return PKV_OK;
}

static inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

static std::atomic<int> g_pdl{0};
static std::atomic<int> g_skip_copy{-1};

// Copies whole slabs src[i] -> dst[i] for up to three arrays at once (slab
// index * slab bytes = offset; arrays may be NULL): a0 and a1 with slabs of
// bytes01 (a multiple of 16) -- the K and V pools, or the K and V tails --
// and a2 with slabs of bytes2 (a multiple of 8) -- the INT8 scales. One CTA
// per pair; a negative src is a "nothing to copy" entry; an index outside
// [0, limit) is skipped and reported.
__global__ void __launch_bounds__(256) copy_slabs_kernel(const int32_t* __restrict__ src,
                                                         const int32_t* __restrict__ dst, int32_t limit,
                                                         uint8_t* a0, uint8_t* a1, size_t bytes01, uint8_t* a2,
                                                         size_t bytes2, int32_t* err, int err_bit) {
    pdl_launch_dependents();
    pdl_wait();
    const int i = blockIdx.x;
    const int s = src[i], d = dst[i];
    if (s < 0 || s == d) return;
    if (s >= limit || d < 0 || d >= limit) {
        if (threadIdx.x == 0) report(err, err_bit);
        return;
    }
    uint8_t* arr[2] = {a0, a1};
    for (int k = 0; k < 2; ++k) {
        if (!arr[k]) continue;
        const uint4* from = reinterpret_cast<const uint4*>(arr[k] + size_t(s) * bytes01);
        uint4* to = reinterpret_cast<uint4*>(arr[k] + size_t(d) * bytes01);
        for (size_t c = threadIdx.x; c < bytes01 / 16; c += blockDim.x) to[c] = from[c];
    }
    if (a2) {
        const uint2* from = reinterpret_cast<const uint2*>(a2 + size_t(s) * bytes2);
        uint2* to = reinterpret_cast<uint2*>(a2 + size_t(d) * bytes2);
        for (size_t c = threadIdx.x; c < bytes2 / 8; c += blockDim.x) to[c] = from[c];
    }
}

// Launches with the programmatic-stream-serialization attribute when enabled
// (pkv_set_programmatic_launch), plainly otherwise.
template <typename... Params, typename... Args>
static int launch(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    if (g_pdl.load(std::memory_order_relaxed)) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cuda_status(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

// The decode instantiation for a shape, and a small index for per-kernel state.
static DecodeFn pick_decode(int d, int g, bool int8, bool split, bool hook, int* index) {
    const int lg = g == 1 ? 0 : g == 2 ? 1 : g == 4 ? 2 : 3;
    *index = ((((d == 128) * 4 + lg) * 2 + int8) * 2 + split) * 2 + hook;
    if (d == 128) return int8 ? decode_fn_d128_int8(g, split, hook) : decode_fn_d128_bf16(g, split, hook);
    return int8 ? decode_fn_d64_int8(g, split, hook) : decode_fn_d64_bf16(g, split, hook);
}

// Raises the kernel's dynamic shared-memory limit (once per kernel, device
// and size) so that it can be launched or sized with `smem` bytes. Safe from
// several host threads: the limit is only ever raised, under a lock, and the
// record of the largest size set is read without one.
static int allow_smem(DecodeFn fn, int index, size_t smem) {
    static std::atomic<int> configured[64][64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
    if (int(smem) <= configured[index][dev].load(std::memory_order_acquire)) return PKV_OK;
    std::lock_guard<std::mutex> lock(mu);
    if (int(smem) <= configured[index][dev].load(std::memory_order_relaxed)) return PKV_OK;
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(smem)) != cudaSuccess)
        return PKV_ERR_CUDA;
    // all of the unified L1 as shared memory: the kernel streams through
    // shared memory and gains nothing from L1, and a smaller carveout would
    // cap the CTAs per SM below what registers allow
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn), cudaFuncAttributePreferredSharedMemoryCarveout,
                             int(cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
        return PKV_ERR_CUDA;
    configured[index][dev].store(int(smem), std::memory_order_release);
    return PKV_OK;
}

// cuTensorMapEncodeTiled, looked up once through the runtime's driver entry
// point (no link against the driver library); nullptr if unavailable.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return PFN_cuTensorMapEncodeTiled_v12000(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// The decode kernel's tensor map of a pool: the pool as bytes
// [num_blocks][rows = Hkv * bs][row_bytes], boxes of 16 rows x 128 bytes,
// 128-byte swizzle. Encoding is host-only work; the last map of each pool is
// kept per thread (a small direct-mapped cache keyed by the pool's shape).
static int pool_tensor_map(const void* pool, int32_t num_blocks, int32_t rows, int32_t row_bytes, CUtensorMap* out) {
    struct Entry {
        CUtensorMap map;
        const void* pool;
        int32_t num_blocks, rows, row_bytes;
    };
    thread_local Entry cache[128] = {};
    const uint64_t h = (uint64_t(reinterpret_cast<uintptr_t>(pool)) >> 8) * 0x9E3779B97F4A7C15ull;
    Entry& e = cache[h >> 57];
    if (e.pool != pool || e.num_blocks != num_blocks || e.rows != rows || e.row_bytes != row_bytes) {
        const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
        if (!enc) return PKV_ERR_CUDA;
        const cuuint64_t dims[3] = {cuuint64_t(row_bytes), cuuint64_t(rows), cuuint64_t(num_blocks)};
        const cuuint64_t strides[2] = {cuuint64_t(row_bytes), cuuint64_t(rows) * cuuint64_t(row_bytes)};
        const cuuint32_t box[3] = {128, 16, 1};
        const cuuint32_t elem[3] = {1, 1, 1};
        e.pool = nullptr;
        if (enc(&e.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(pool), dims, strides, box, elem,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return PKV_ERR_CUDA;
        e.pool = pool;
        e.num_blocks = num_blocks;
        e.rows = rows;
        e.row_bytes = row_bytes;
    }
    *out = e.map;
    return PKV_OK;
}

// Dynamic shared memory of a decode CTA: rings and mbarriers, the block table
// (tab_cap entries) and, INT8, the block scales.
static size_t decode_smem(int d, bool int8, int tab_cap) {
    size_t fixed = 0;
    if (d == 64) fixed = int8 ? decode_smem_fixed<64, true>() : decode_smem_fixed<64, false>();
    else fixed = int8 ? decode_smem_fixed<128, true>() : decode_smem_fixed<128, false>();
    return fixed + size_t(tab_cap) * (int8 ? 12 : 4);
}

}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_set_programmatic_launch(int enable) {
    g_pdl.store(enable ? 1 : 0);
    return PKV_OK;
}

int pkv_debug_skip_copy(int32_t tile) {
    if (tile < -1) return PKV_ERR_INVALID;
    g_skip_copy.store(tile);
    return PKV_OK;
}

size_t pkv_splitk_ws_o_bytes(int32_t B, int32_t Hq, int32_t head_dim, int32_t max_splits) {
    if (B < 0 || Hq < 0 || head_dim < 0 || max_splits < 0) return 0;
    return size_t(B) * size_t(Hq) * size_t(max_splits) * size_t(head_dim) * sizeof(float);
}

size_t pkv_splitk_ws_ml_bytes(int32_t B, int32_t Hq, int32_t max_splits) {
    if (B < 0 || Hq < 0 || max_splits < 0) return 0;
    return size_t(B) * size_t(Hq) * size_t(max_splits) * 2 * sizeof(float);
}

int pkv_append_kv(const pkv_cache_desc* c, const void* k, const void* v, const int32_t* block_ids,
                  const int32_t* offsets, const int32_t* slots, int32_t T, void* stream) {
    int st = check_desc(c);
    if (st != PKV_OK) return st;
    if (T < 0) return PKV_ERR_INVALID;
    if (T == 0) return PKV_OK;
    if (!k || !v || !offsets || !aligned16(k) || !aligned16(v)) return PKV_ERR_INVALID;
    const bool int8 = c->dtype == PKV_DTYPE_INT8;
    if (int8 ? !slots : !block_ids) return PKV_ERR_INVALID;
    const int64_t total = int64_t(T) * 2 * c->num_kv_heads * (c->head_dim / 8);
    const int64_t grid = (total + 255) / 256;
    if (grid > 0x7FFFFFFF) return PKV_ERR_INVALID;
    void* kd = int8 ? c->k_tail : c->k_pool;
    void* vd = int8 ? c->v_tail : c->v_pool;
    auto s = static_cast<cudaStream_t>(stream);
    const auto* kk = static_cast<const uint16_t*>(k);
    const auto* vv = static_cast<const uint16_t*>(v);
    const int i8 = int8 ? 1 : 0;
    if (c->head_dim == 128)
        return launch(append_kernel<128>, dim3(unsigned(grid)), dim3(256), 0, s, kk, vv, block_ids, offsets, slots, T,
                      c->num_kv_heads, c->block_size, c->num_blocks, c->max_slots, i8, kd, vd, c->err_word);
    return launch(append_kernel<64>, dim3(unsigned(grid)), dim3(256), 0, s, kk, vv, block_ids, offsets, slots, T,
                  c->num_kv_heads, c->block_size, c->num_blocks, c->max_slots, i8, kd, vd, c->err_word);
}

static int quantize_common(const pkv_cache_desc* c, const void* k_src, const void* v_src, int from_tail,
                           const int32_t* block_ids, const int32_t* slots, int32_t M, void* stream) {
    int st = check_desc(c);
    if (st != PKV_OK) return st;
    if (c->dtype != PKV_DTYPE_INT8 || M < 0) return PKV_ERR_INVALID;
    if (M == 0) return PKV_OK;
    if (!block_ids || (from_tail && !slots) || !k_src || !v_src || !aligned16(k_src) || !aligned16(v_src))
        return PKV_ERR_INVALID;
    const int64_t slabs = int64_t(M) * 2 * c->num_kv_heads;
    const int64_t grid = (slabs + 3) / 4;
    if (grid > 0x7FFFFFFF) return PKV_ERR_INVALID;
    auto s = static_cast<cudaStream_t>(stream);
    const auto* ks = static_cast<const uint16_t*>(k_src);
    const auto* vs = static_cast<const uint16_t*>(v_src);
    auto* kp = static_cast<int8_t*>(c->k_pool);
    auto* vp = static_cast<int8_t*>(c->v_pool);
    if (c->head_dim == 128)
        return launch(quantize_kernel<128>, dim3(unsigned(grid)), dim3(128), 0, s, ks, vs, from_tail, block_ids, slots,
                      M, c->num_kv_heads, c->block_size, c->num_blocks, c->max_slots, kp, vp, c->scales,
                      c->err_word);
    return launch(quantize_kernel<64>, dim3(unsigned(grid)), dim3(128), 0, s, ks, vs, from_tail, block_ids, slots, M,
                  c->num_kv_heads, c->block_size, c->num_blocks, c->max_slots, kp, vp, c->scales, c->err_word);
}

int pkv_quantize_full_blocks(const pkv_cache_desc* c, const int32_t* block_ids, const int32_t* slots,
                             int32_t M, void* stream) {
    if (!c) return PKV_ERR_INVALID;
    return quantize_common(c, c->k_tail, c->v_tail, 1, block_ids, slots, M, stream);
}

int pkv_quantize_blocks_from(const pkv_cache_desc* c, const void* k_src, const void* v_src,
                             const int32_t* block_ids, int32_t M, void* stream) {
    return quantize_common(c, k_src, v_src, 0, block_ids, nullptr, M, stream);
}

static int copy_slabs(const pkv_cache_desc* c, bool slots, const int32_t* src, const int32_t* dst, int32_t n,
                      void* stream) {
    int st = check_desc(c);
    if (st != PKV_OK) return st;
    if (n < 0) return PKV_ERR_INVALID;
    if (n == 0) return PKV_OK;
    if (!src || !dst) return PKV_ERR_INVALID;
    const bool int8 = c->dtype == PKV_DTYPE_INT8;
    if (slots && !int8) return PKV_ERR_INVALID;
    const size_t rows = size_t(c->num_kv_heads) * size_t(c->block_size) * size_t(c->head_dim);
    auto s = static_cast<cudaStream_t>(stream);
    if (slots)  // bf16 tails [slot][Hkv][bs][d]
        return launch(copy_slabs_kernel, dim3(unsigned(n)), dim3(256), 0, s, src, dst, c->max_slots,
                      static_cast<uint8_t*>(c->k_tail), static_cast<uint8_t*>(c->v_tail), rows * 2,
                      static_cast<uint8_t*>(nullptr), size_t(0), c->err_word, int(kErrSlot));
    // pool blocks [block][Hkv][bs][d] (+ INT8 scales [block][Hkv][2] fp32)
    const size_t sc_bytes = int8 ? size_t(c->num_kv_heads) * 8 : 0;
    return launch(copy_slabs_kernel, dim3(unsigned(n)), dim3(256), 0, s, src, dst, c->num_blocks,
                  static_cast<uint8_t*>(c->k_pool), static_cast<uint8_t*>(c->v_pool), rows * (int8 ? 1 : 2),
                  reinterpret_cast<uint8_t*>(int8 ? c->scales : nullptr), sc_bytes, c->err_word, int(kErrBlockId));
}

int pkv_copy_blocks(const pkv_cache_desc* c, const int32_t* src_ids, const int32_t* dst_ids, int32_t n,
                    void* stream) {
    return copy_slabs(c, false, src_ids, dst_ids, n, stream);
}

int pkv_copy_slots(const pkv_cache_desc* c, const int32_t* src_slots, const int32_t* dst_slots, int32_t n,
                   void* stream) {
    return copy_slabs(c, true, src_slots, dst_slots, n, stream);
}

static int launch_reduce(const float* ws_o, const float* ws_ml, const int32_t* ctx_lens, int32_t B, int32_t Hq,
                         int32_t head_dim, int32_t split_tokens, int32_t max_splits, void* out, int32_t* err,
                         void* stream) {
    if (B < 0 || Hq <= 0 || split_tokens <= 0 || max_splits <= 0) return PKV_ERR_INVALID;
    if (head_dim != 64 && head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (B == 0) return PKV_OK;
    if (!ws_o || !ws_ml || !ctx_lens || !out || B > 65535) return PKV_ERR_INVALID;
    const size_t smem = size_t(max_splits) * sizeof(float);
    if (smem > 48 * 1024) return PKV_ERR_UNSUPPORTED;
    auto s = static_cast<cudaStream_t>(stream);
    const dim3 grid{unsigned(Hq), unsigned(B), 1u};
    auto* o = static_cast<uint16_t*>(out);
    if (head_dim == 128)
        return launch(splitk_reduce_kernel<128>, grid, dim3(128), smem, s, ws_o, ws_ml, ctx_lens, Hq, split_tokens,
                      max_splits, o, err);
    return launch(splitk_reduce_kernel<64>, grid, dim3(128), smem, s, ws_o, ws_ml, ctx_lens, Hq, split_tokens,
                  max_splits, o, err);
}

int pkv_splitk_reduce(const float* ws_o, const float* ws_ml, const int32_t* ctx_lens, int32_t B, int32_t Hq,
                      int32_t head_dim, int32_t split_tokens, int32_t max_splits, void* out, void* stream) {
    return launch_reduce(ws_o, ws_ml, ctx_lens, B, Hq, head_dim, split_tokens, max_splits, out, nullptr, stream);
}

static int decode_tab_cap(const pkv_cache_desc* c, int32_t split_tokens, int32_t max_blocks) {
    int tab_cap = split_tokens > 0 ? split_tokens / c->block_size : max_blocks;
    return tab_cap + (tab_cap & 1);
}

int pkv_decode_ctas_per_sm(const pkv_cache_desc* c, int32_t split_tokens, int32_t max_blocks) {
    int st = check_desc(c);
    if (st != PKV_OK) return st;
    if (split_tokens < 0 || max_blocks <= 0) return PKV_ERR_INVALID;
    if (split_tokens > 0 && (split_tokens % c->block_size || split_tokens % kTile)) return PKV_ERR_INVALID;
    const bool int8 = c->dtype == PKV_DTYPE_INT8;
    const int g = c->num_q_heads / c->num_kv_heads;
    const size_t smem = decode_smem(c->head_dim, int8, decode_tab_cap(c, split_tokens, max_blocks));
    if (smem > 227 * 1024) return PKV_ERR_UNSUPPORTED;
    int index = 0;
    DecodeFn fn = pick_decode(c->head_dim, g, int8, split_tokens > 0, false, &index);
    if (!fn) return PKV_ERR_UNSUPPORTED;
    if ((st = allow_smem(fn, index, smem)) != PKV_OK) return st;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kThreads, smem) != cudaSuccess) return PKV_ERR_CUDA;
    return n;
}

static int decode_impl(const pkv_cache_desc* c, const void* q, const void* k_new, const void* v_new,
                       const int32_t* block_tables, int32_t max_blocks, const int32_t* ctx_lens, const int32_t* slots,
                       int32_t B, float sm_scale, int32_t split_tokens, int32_t max_splits, float* ws_o, float* ws_ml,
                       int32_t* ws_count, void* out, void* stream) {
    int st = check_desc(c);
    if (st != PKV_OK) return st;
    if (B < 0 || max_blocks <= 0 || split_tokens < 0 || !(sm_scale == sm_scale)) return PKV_ERR_INVALID;
    if (B == 0) return PKV_OK;
    if (!q || !block_tables || !ctx_lens || !out || B > 65535 || c->num_kv_heads > 65535) return PKV_ERR_INVALID;
    if (!aligned16(q) || (reinterpret_cast<uintptr_t>(out) & 3u)) return PKV_ERR_INVALID;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID;  // 16-byte row loads
    const bool int8 = c->dtype == PKV_DTYPE_INT8;
    if (int8 && !slots) return PKV_ERR_INVALID;
    const int64_t max_ctx = int64_t(max_blocks) * c->block_size;
    if (max_ctx > 0x7FFFFFFF) return PKV_ERR_INVALID;
    const bool split = split_tokens > 0;
    if (split) {
        if (split_tokens % c->block_size || split_tokens % kTile) return PKV_ERR_INVALID;
        if (int64_t(max_splits) * split_tokens < max_ctx || max_splits > 65535) return PKV_ERR_INVALID;
        if (!ws_o || !ws_ml || !aligned16(ws_o) || !aligned16(ws_ml)) return PKV_ERR_INVALID;
        if (ws_count && (reinterpret_cast<uintptr_t>(ws_count) & 3u)) return PKV_ERR_INVALID;
    }
    const int g = c->num_q_heads / c->num_kv_heads;
    const int tab_cap = decode_tab_cap(c, split_tokens, max_blocks);
    const size_t smem = decode_smem(c->head_dim, int8, tab_cap);
    if (smem > 227 * 1024) return PKV_ERR_UNSUPPORTED;  // too many blocks per CTA: use a split

    DecodeParams p;
    const int32_t row_bytes = c->head_dim * (int8 ? 1 : 2);
    if (row_bytes >= 128) {  // tiles staged by tensor copies
        const int32_t rows = c->num_kv_heads * c->block_size;
        if ((st = pool_tensor_map(c->k_pool, c->num_blocks, rows, row_bytes, &p.tm_k)) != PKV_OK) return st;
        if ((st = pool_tensor_map(c->v_pool, c->num_blocks, rows, row_bytes, &p.tm_v)) != PKV_OK) return st;
    } else {
        std::memset(&p.tm_k, 0, sizeof(p.tm_k));
        std::memset(&p.tm_v, 0, sizeof(p.tm_v));
    }
    p.k_pool = c->k_pool;
    p.v_pool = c->v_pool;
    p.scales = c->scales;
    p.k_tail = c->k_tail;
    p.v_tail = c->v_tail;
    p.q = static_cast<const uint16_t*>(q);
    p.k_new = static_cast<const uint16_t*>(k_new);
    p.v_new = static_cast<const uint16_t*>(v_new);
    p.block_tables = block_tables;
    p.ctx_lens = ctx_lens;
    p.slots = slots;
    p.out = static_cast<uint16_t*>(out);
    p.ws_o = ws_o;
    p.ws_ml = ws_ml;
    const bool fuse = split && ws_count;
    p.ws_count = fuse ? ws_count : nullptr;
    p.err = c->err_word;
    p.Hq = c->num_q_heads;
    p.Hkv = c->num_kv_heads;
    p.bs = c->block_size;
    p.max_blocks = max_blocks;
    p.num_blocks = c->num_blocks;
    p.max_slots = c->max_slots;
    p.split_tokens = split_tokens;
    p.max_splits = split ? max_splits : 1;
    p.tab_cap = tab_cap;
    p.qscale = sm_scale * 1.4426950408889634f;
    p.skip_copy = g_skip_copy.load(std::memory_order_relaxed);

    const dim3 grid(split ? unsigned(max_splits) : 1u, unsigned(c->num_kv_heads), unsigned(B));
    auto s = static_cast<cudaStream_t>(stream);
    int index = 0;
    DecodeFn fn = pick_decode(c->head_dim, g, int8, split, p.skip_copy >= 0, &index);
    if (!fn) return PKV_ERR_UNSUPPORTED;
    if ((st = allow_smem(fn, index, smem)) != PKV_OK) return st;
    if ((st = launch(fn, grid, dim3(kThreads), smem, s, p)) != PKV_OK) return st;
    if (!split || fuse) return PKV_OK;
    return launch_reduce(ws_o, ws_ml, ctx_lens, B, c->num_q_heads, c->head_dim, split_tokens, max_splits, out,
                         c->err_word, stream);
}

int pkv_decode_attention(const pkv_cache_desc* c, const void* q, const int32_t* block_tables, int32_t max_blocks,
                         const int32_t* ctx_lens, const int32_t* slots, int32_t B, float sm_scale,
                         int32_t split_tokens, int32_t max_splits, float* ws_o, float* ws_ml, int32_t* ws_count,
                         void* out, void* stream) {
    return decode_impl(c, q, nullptr, nullptr, block_tables, max_blocks, ctx_lens, slots, B, sm_scale, split_tokens,
                       max_splits, ws_o, ws_ml, ws_count, out, stream);
}

int pkv_decode_layers(const pkv_cache_desc* descs, int32_t num_layers, const void* q, int64_t q_layer_stride,
                      const void* k_new, const void* v_new, int64_t kv_layer_stride, void* out,
                      int64_t out_layer_stride, const int32_t* block_tables, int32_t max_blocks,
                      const int32_t* ctx_lens, const int32_t* slots, int32_t B, float sm_scale,
                      int32_t split_tokens, int32_t max_splits, float* ws_o, float* ws_ml, int32_t* ws_count,
                      void* stream) {
    if (!descs || num_layers < 0 || !q || !out) return PKV_ERR_INVALID;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID;
    if ((q_layer_stride | out_layer_stride | (k_new ? kv_layer_stride : 0)) & 15) return PKV_ERR_INVALID;
    const auto* qb = static_cast<const uint8_t*>(q);
    const auto* kb = static_cast<const uint8_t*>(k_new);
    const auto* vb = static_cast<const uint8_t*>(v_new);
    auto* ob = static_cast<uint8_t*>(out);
    for (int32_t l = 0; l < num_layers; ++l) {
        // one NVTX range per layer (visible to a profiler attached to the process)
        char name[32];
        snprintf(name, sizeof(name), "pkv layer %d", int(l));
        nvtxRangePushA(name);
        const int rc = decode_impl(descs + l, qb + l * q_layer_stride, kb ? kb + l * kv_layer_stride : nullptr,
                                   vb ? vb + l * kv_layer_stride : nullptr, block_tables, max_blocks, ctx_lens, slots,
                                   B, sm_scale, split_tokens, max_splits, ws_o, ws_ml, ws_count,
                                   ob + l * out_layer_stride, stream);
        nvtxRangePop();
        if (rc != PKV_OK) return rc;
    }
    return PKV_OK;
}

int pkv_sync_status(const pkv_cache_desc* descs, int32_t n, void* stream, int32_t* out_bits) {
    if (out_bits) *out_bits = 0;
    if (n < 0 || (n > 0 && !descs)) return PKV_ERR_INVALID;
    auto s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    int32_t bits = 0;
    for (int32_t i = 0; i < n; ++i) {
        int32_t* w = descs[i].err_word;
        if (!w) continue;
        int32_t v = 0;
        if (cudaMemcpyAsync(&v, w, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return PKV_ERR_CUDA;
        if (v && cudaMemsetAsync(w, 0, sizeof(v), s) != cudaSuccess) return PKV_ERR_CUDA;
        bits |= v;
    }
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    if (out_bits) *out_bits = bits;
    if (bits & PKV_DEVERR_TIMEOUT) return PKV_ERR_DEVICE_TIMEOUT;
    return bits ? PKV_ERR_INVALID : PKV_OK;
}

int pkv_decode_step(const pkv_cache_desc* c, const void* q, const void* k_new, const void* v_new,
                    const int32_t* block_tables, int32_t max_blocks, const int32_t* ctx_lens, const int32_t* slots,
                    int32_t B, float sm_scale, int32_t split_tokens, int32_t max_splits, float* ws_o, float* ws_ml,
                    int32_t* ws_count, void* out, void* stream) {
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID;
    return decode_impl(c, q, k_new, v_new, block_tables, max_blocks, ctx_lens, slots, B, sm_scale, split_tokens,
                       max_splits, ws_o, ws_ml, ws_count, out, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode attention with library-owned split-K scratch (no allocation).
//
// Some callers cannot allocate device memory at decode time: an engine that
// hands all free HBM to its KV-cache pool at start-up and forbids later
// allocations (a cudaMalloc would fail or evict cache), a plugin living
// inside such an engine, or a latency-critical loop that must not pay for
// cudaMalloc's implicit synchronisation. This entry point takes no workspace
// argument: the split-K partials and arrival counters live in the fixed
// array below, which every GPU that loads the library holds until the
// process exits.
// ---------------------------------------------------------------------------
namespace pkv {
static __device__ __align__(256) unsigned char g_static_ws[PKV_STATIC_WS_BYTES];
}  // namespace pkv

// Device address of g_static_ws on the current device, looked up once per
// device (in host code the array's name is only a host-side stand-in).
static int static_ws_address(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, pkv::g_static_ws) != cudaSuccess || !p) return PKV_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return PKV_OK;
}

extern "C" int pkv_decode_attention_static_ws(const pkv_cache_desc* c, const void* q, const int32_t* block_tables,
                                              int32_t max_blocks, const int32_t* ctx_lens, const int32_t* slots,
                                              int32_t B, float sm_scale, int32_t split_tokens, int32_t max_splits,
                                              void* out, void* stream) {
    if (split_tokens < 0) return PKV_ERR_INVALID;
    if (split_tokens == 0)  // no split: no scratch is used at all
        return pkv_decode_attention(c, q, block_tables, max_blocks, ctx_lens, slots, B, sm_scale, 0, 0, nullptr,
                                    nullptr, nullptr, out, stream);
    int st = check_desc(c);
    if (st != PKV_OK) return st;
    if (B < 0 || max_splits <= 0) return PKV_ERR_INVALID;
    // layout: [counters B*Hkv int32 | pad to 256 B][m,l: B*Hq*S*2 f32][o: B*Hq*S*d f32]
    const size_t cnt_bytes = (size_t(B) * size_t(c->num_kv_heads) * 4 + 255) / 256 * 256;
    const size_t ml_bytes = (pkv_splitk_ws_ml_bytes(B, c->num_q_heads, max_splits) + 255) / 256 * 256;
    const size_t o_bytes = pkv_splitk_ws_o_bytes(B, c->num_q_heads, c->head_dim, max_splits);
    if (cnt_bytes + ml_bytes + o_bytes > size_t(PKV_STATIC_WS_BYTES)) return PKV_ERR_TOO_LARGE;
    void* base = nullptr;
    if ((st = static_ws_address(&base)) != PKV_OK) return st;
    auto* bytes = static_cast<unsigned char*>(base);
    auto* counters = reinterpret_cast<int32_t*>(bytes);
    auto* ws_ml = reinterpret_cast<float*>(bytes + cnt_bytes);
    auto* ws_o = reinterpret_cast<float*>(bytes + cnt_bytes + ml_bytes);
    // The array keeps the previous call's contents: the arrival counters must
    // start at zero, the partials are always written before they are read.
    if (B > 0 && cudaMemsetAsync(counters, 0, size_t(B) * size_t(c->num_kv_heads) * 4,
                                 static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKV_ERR_CUDA;
    return pkv_decode_attention(c, q, block_tables, max_blocks, ctx_lens, slots, B, sm_scale, split_tokens, max_splits,
                                ws_o, ws_ml, counters, out, stream);
}
