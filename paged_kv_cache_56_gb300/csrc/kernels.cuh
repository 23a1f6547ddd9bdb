// Device kernels of the paged KV cache: append, quantize-on-fill, decode
// attention (whole context or one split of it) and the split-K merge.
//
// Decode-attention design (sm_103a):
//   * one CTA per (split j, kv head, sequence b); it loads the query rows of
//     the whole GQA group of that kv head, so every KV byte crosses HBM once
//     per step;
//   * four warps; each owns a ring of STAGES shared-memory stages and pulls
//     16-token K and V tiles into them with bulk asynchronous copies (the TMA
//     engine, one elected lane, completion on an mbarrier), gathering tiles
//     through the block table. A (block, kv head) tile is contiguous in the
//     [num_blocks][Hkv][bs][d] pools, so every copy is one linear transfer;
//   * a token is spread over d/16 lanes, each holding 16 of its dims; QK and
//     PV run on packed fp32 FMAs (f32x2); INT8 values are converted exactly
//     in registers and the per-block scales are applied to the scores and to
//     the softmax weights, not per element;
//   * fp32 online softmax in base 2 (scores pre-multiplied by log2 e), one
//     state per group of lanes, merged across lanes with shuffles and across
//     warps through shared memory at the end.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace pkv {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 16;  // tokens per staged tile
constexpr unsigned kFull = 0xFFFFFFFFu;

constexpr int kErrBlockId = 1;
constexpr int kErrSlot = 2;
constexpr int kErrCtxLen = 4;
constexpr int kErrOffset = 8;
constexpr int kErrTimeout = 16;

__device__ __forceinline__ void report(int32_t* err, int bits) {
    if (err) atomicOr(err, bits);
}

struct DecodeParams {
    const void* k_pool;
    const void* v_pool;
    const float* scales;
    const void* k_tail;
    const void* v_tail;
    const uint16_t* q;
    const int32_t* block_tables;
    const int32_t* ctx_lens;
    const int32_t* slots;
    uint16_t* out;
    float* ws_o;
    float* ws_ml;
    int32_t* err;
    int32_t Hq, Hkv, bs, max_blocks, num_blocks, max_slots, split_tokens, max_splits;
    int32_t tab_cap;  // block-table entries the shared table holds (even)
    float qscale;     // sm_scale * log2(e)
};

template <int D, bool INT8>
struct DecodeTraits {
    static constexpr int kElemBytes = INT8 ? 1 : 2;
    static constexpr int kRowBytes = D * kElemBytes;
    static constexpr int kTileBytes = kTile * kRowBytes;  // K or V of one tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = INT8 ? 6 : 4;
    static constexpr int kLPT = D / 16;         // lanes per token
    static constexpr int kTPW = 32 / kLPT;      // tokens per warp pass
    static constexpr int kIters = kTile / kTPW; // passes per tile
};

// Shared-memory bytes one decode CTA needs.
template <int D, int G, bool INT8>
constexpr size_t decode_smem_fixed() {
    using T = DecodeTraits<D, INT8>;
    return size_t(kWarps) * T::kStages * T::kStageBytes   // stages
         + size_t(kWarps) * T::kStages * 8                // mbarriers
         + size_t(kWarps) * G * D * 4                     // merge: o
         + size_t(kWarps) * G * 2 * 4;                    // merge: m, l
}

// Lane-to-dimension map. Lane `sub` of a token holds 16 dims:
//   INT8 kernels: dims sub*16 .. sub*16+15 (one 16-byte int8 chunk);
//   BF16 kernels: dims sub*8 .. sub*8+7 and D/2 + sub*8 .. +7 (two 16-byte
//   chunks, so that eight consecutive lanes read 128 contiguous bytes).
template <int D, bool INT8>
__device__ __forceinline__ int lane_dim(int sub, int i) {
    if (INT8) return sub * 16 + i;
    return i < 8 ? sub * 8 + i : D / 2 + sub * 8 + (i - 8);
}

// 16 bf16 values of a global row at this lane's dims -> fp32 pairs.
template <int D, bool INT8>
__device__ __forceinline__ void load_bf16_dims_global(const uint16_t* row, int sub, float2 (&x)[8]) {
    uint4 a, b;
    if (INT8) {
        a = ldg128(row + sub * 16);
        b = ldg128(row + sub * 16 + 8);
    } else {
        a = ldg128(row + sub * 8);
        b = ldg128(row + D / 2 + sub * 8);
    }
    x[0] = bf16x2_to_f2(a.x); x[1] = bf16x2_to_f2(a.y); x[2] = bf16x2_to_f2(a.z); x[3] = bf16x2_to_f2(a.w);
    x[4] = bf16x2_to_f2(b.x); x[5] = bf16x2_to_f2(b.y); x[6] = bf16x2_to_f2(b.z); x[7] = bf16x2_to_f2(b.w);
}

// Row loader for a staged tile in shared memory.
template <int D, bool INT8>
struct SmemTile {
    uint32_t base;
    __device__ __forceinline__ void load(int r, int sub, float2 (&x)[8]) const {
        using T = DecodeTraits<D, INT8>;
        const uint32_t row = base + uint32_t(r) * T::kRowBytes;
        if (INT8) {
            uint4 w = lds128(row + sub * 16);
            s8x4_to_f4(w.x, x[0], x[1]);
            s8x4_to_f4(w.y, x[2], x[3]);
            s8x4_to_f4(w.z, x[4], x[5]);
            s8x4_to_f4(w.w, x[6], x[7]);
        } else {
            uint4 a = lds128(row + sub * 16);
            uint4 b = lds128(row + D + sub * 16);
            x[0] = bf16x2_to_f2(a.x); x[1] = bf16x2_to_f2(a.y); x[2] = bf16x2_to_f2(a.z); x[3] = bf16x2_to_f2(a.w);
            x[4] = bf16x2_to_f2(b.x); x[5] = bf16x2_to_f2(b.y); x[6] = bf16x2_to_f2(b.z); x[7] = bf16x2_to_f2(b.w);
        }
    }
};

// Row loader for bf16 rows in global memory (the INT8 cache's tail block).
template <int D, bool INT8>
struct GlobalBf16Rows {
    const uint16_t* base;  // row 0
    __device__ __forceinline__ void load(int r, int sub, float2 (&x)[8]) const {
        load_bf16_dims_global<D, INT8>(base + size_t(r) * D, sub, x);
    }
};

// One 16-token tile: scores, online-softmax update, weighted V accumulation.
// nvalid < 16 masks the tile's last rows (their scores become -inf and their
// V rows are zeroed, so stale or uninitialised rows cannot leak NaNs in).
template <int D, int G, class Loader>
__device__ __forceinline__ void tile_step(const Loader& kl, const Loader& vl, int nvalid, float ksc,
                                          float vsc, int tk, int sub, const float2 (&q2)[G][8],
                                          float (&m)[G], float (&l)[G], float2 (&o2)[G][8]) {
    constexpr int LPT = D / 16, TPW = 32 / LPT, ITERS = kTile / TPW;
    float s[ITERS][G];
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
        float2 x[8];
        kl.load(it * TPW + tk, sub, x);
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float2 a = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) a = __ffma2_rn(q2[g][i], x[i], a);
            s[it][g] = a.x + a.y;
        }
    }
#pragma unroll
    for (int off = 1; off < LPT; off <<= 1)
#pragma unroll
        for (int it = 0; it < ITERS; ++it)
#pragma unroll
            for (int g = 0; g < G; ++g) s[it][g] += __shfl_xor_sync(kFull, s[it][g], off);

    const bool full = nvalid >= kTile;
#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
        const bool ok = full || (it * TPW + tk) < nvalid;
#pragma unroll
        for (int g = 0; g < G; ++g) s[it][g] = ok ? s[it][g] * ksc : -INFINITY;
    }

    float mnew[G];
    bool up = false;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float mx = m[g];
#pragma unroll
        for (int it = 0; it < ITERS; ++it) mx = fmaxf(mx, s[it][g]);
        mnew[g] = mx;
        up |= mx > m[g];
    }
    if (__any_sync(kFull, up)) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float c = fast_exp2(m[g] - mnew[g]);
            m[g] = mnew[g];
            l[g] *= c;
            const float2 c2 = make_float2(c, c);
#pragma unroll
            for (int i = 0; i < 8; ++i) o2[g][i] = __fmul2_rn(o2[g][i], c2);
        }
    }
#pragma unroll
    for (int it = 0; it < ITERS; ++it)
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float pr = fast_exp2(s[it][g] - m[g]);
            l[g] += pr;
            s[it][g] = pr * vsc;
        }

#pragma unroll
    for (int it = 0; it < ITERS; ++it) {
        float2 x[8];
        vl.load(it * TPW + tk, sub, x);
        if (!full && (it * TPW + tk) >= nvalid) {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float2 p2 = make_float2(s[it][g], s[it][g]);
#pragma unroll
            for (int i = 0; i < 8; ++i) o2[g][i] = __ffma2_rn(p2, x[i], o2[g][i]);
        }
    }
}

// Waits for an mbarrier phase for at most ~1 s of GPU time.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < 64; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > 1000000000ull) return false;
    }
}

template <int D, int G, bool INT8, bool SPLIT>
__global__ void __launch_bounds__(kThreads) decode_kernel(const DecodeParams p) {
    using T = DecodeTraits<D, INT8>;
    constexpr int LPT = T::kLPT, STAGES = T::kStages;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(kWarps) * STAGES * T::kStageBytes);
    float* mo = reinterpret_cast<float*>(bars + kWarps * STAGES);
    float* mml = mo + kWarps * G * D;
    int32_t* tab = reinterpret_cast<int32_t*>(mml + kWarps * G * 2);
    float2* bsc = reinterpret_cast<float2*>(tab + p.tab_cap);

    const int j = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sub = lane % LPT, tk = lane / LPT;

    int ctx = p.ctx_lens[b];
    if (ctx < 0 || ctx > p.max_blocks * p.bs) {
        if (tid == 0 && j == 0) report(p.err, kErrCtxLen);
        ctx = 0;
    }
    const int t0 = SPLIT ? j * p.split_tokens : 0;
    const int t1 = SPLIT ? min(ctx, t0 + p.split_tokens) : ctx;
    if (t0 >= t1 && j > 0) return;  // this split lies past the context

    const int nfull = INT8 ? (ctx / p.bs) * p.bs : ctx;
    const int pool_end = min(t1, nfull);
    const int npool = max(0, pool_end - t0);
    const int nt = (npool + kTile - 1) / kTile;
    const int blk0 = t0 / p.bs;
    const int nblk = npool > 0 ? min((pool_end - 1) / p.bs - blk0 + 1, p.tab_cap) : 0;

    const uint32_t bar0 = smem_addr(bars);
    const uint32_t stage0 = smem_addr(stages);
    auto bar_of = [&](int s) { return bar0 + uint32_t(warp * STAGES + s) * 8u; };
    auto stage_of = [&](int s) { return stage0 + uint32_t(warp * STAGES + s) * T::kStageBytes; };

    if (lane == 0)
        for (int s = 0; s < STAGES; ++s) mbar_init(bar_of(s), 1);
    const int32_t* trow = p.block_tables + size_t(b) * p.max_blocks + blk0;
    for (int i = tid; i < nblk; i += kThreads) {
        int id = trow[i];
        if (id < 0 || id >= p.num_blocks) {
            report(p.err, kErrBlockId);
            id = -1;
        }
        tab[i] = id;
    }
    fence_mbar_init();
    __syncthreads();

    const uint64_t pol = l2_policy_evict_first();
    auto issue = [&](int tile, int s) {
        const int tok = t0 + tile * kTile;
        const int id = tab[tok / p.bs - blk0];
        const uint32_t bar = bar_of(s);
        if (id < 0) {
            mbar_arrive(bar);
            return;
        }
        const size_t row = (size_t(id) * p.Hkv + kvh) * p.bs + (tok % p.bs);
        const uint8_t* ks = static_cast<const uint8_t*>(p.k_pool) + row * T::kRowBytes;
        const uint8_t* vs = static_cast<const uint8_t*>(p.v_pool) + row * T::kRowBytes;
        mbar_arrive_expect_tx(bar, T::kStageBytes);
        bulk_g2s(stage_of(s), ks, T::kTileBytes, bar, pol);
        bulk_g2s(stage_of(s) + T::kTileBytes, vs, T::kTileBytes, bar, pol);
    };
    if (lane == 0)
        for (int s = 0; s < STAGES; ++s) {
            const int tile = warp + s * kWarps;
            if (tile < nt) issue(tile, s);
        }

    if (INT8) {
        for (int i = tid; i < nblk; i += kThreads) {
            const int id = tab[i];
            float2 sc = make_float2(0.f, 0.f);
            if (id >= 0) sc = *reinterpret_cast<const float2*>(p.scales + (size_t(id) * p.Hkv + kvh) * 2);
            bsc[i] = sc;
        }
    }

    float2 q2[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        load_bf16_dims_global<D, INT8>(p.q + (size_t(b) * p.Hq + kvh * G + g) * D, sub, q2[g]);
        const float2 qs = make_float2(p.qscale, p.qscale);
#pragma unroll
        for (int i = 0; i < 8; ++i) q2[g][i] = __fmul2_rn(q2[g][i], qs);
    }
    float m[G], l[G];
    float2 o2[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -1e30f;
        l[g] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o2[g][i] = make_float2(0.f, 0.f);
    }
    __syncthreads();

    // ---- main loop over this warp's pool tiles ----------------------------------
    int k = 0;
    bool timed_out = false;
    for (int tile = warp; tile < nt; tile += kWarps, ++k) {
        const int s = k % STAGES;
        if (!wait_phase(bar_of(s), uint32_t(k / STAGES) & 1u)) {
            timed_out = true;
            break;
        }
        const int tok = t0 + tile * kTile;
        const int bl = tok / p.bs - blk0;
        int nvalid = min(kTile, pool_end - tok);
        if (tab[bl] < 0) nvalid = 0;
        float ksc = 1.f, vsc = 1.f;
        if (INT8) {
            const float2 sc = bsc[bl];
            ksc = sc.x;
            vsc = sc.y;
        }
        const SmemTile<D, INT8> kt{stage_of(s)}, vt{stage_of(s) + T::kTileBytes};
        tile_step<D, G>(kt, vt, nvalid, ksc, vsc, tk, sub, q2, m, l, o2);
        __syncwarp();
        const int nxt = tile + STAGES * kWarps;
        if (lane == 0 && nxt < nt) {
            fence_proxy_async_smem();
            issue(nxt, s);
        }
    }
    if (timed_out) {
        // Drain this warp's copies still in flight (each wait again bounded)
        // so that no copy lands in shared memory after the CTA has exited.
        if (lane == 0) report(p.err, kErrTimeout);
        for (int kk = k; kk < k + STAGES && warp + kk * kWarps < nt; ++kk)
            (void)wait_phase(bar_of(kk % STAGES), uint32_t(kk / STAGES) & 1u);
    }

    // ---- INT8: the partly filled last block is read from the bf16 tail -------
    if (INT8) {
        const int tail_lo = max(t0, nfull);
        const int ntail = t1 - tail_lo;
        if (ntail > 0) {
            const int slot = p.slots ? p.slots[b] : -1;
            if (slot < 0 || slot >= p.max_slots) {
                if (tid == 0) report(p.err, kErrSlot);
            } else {
                const size_t rbase = (size_t(slot) * p.Hkv + kvh) * p.bs + (tail_lo - nfull);
                const uint16_t* kt = static_cast<const uint16_t*>(p.k_tail) + rbase * D;
                const uint16_t* vt = static_cast<const uint16_t*>(p.v_tail) + rbase * D;
                for (int tt = warp; tt * kTile < ntail; tt += kWarps) {
                    const GlobalBf16Rows<D, INT8> kr{kt + size_t(tt) * kTile * D};
                    const GlobalBf16Rows<D, INT8> vr{vt + size_t(tt) * kTile * D};
                    tile_step<D, G>(kr, vr, min(kTile, ntail - tt * kTile), 1.f, 1.f, tk, sub, q2, m, l, o2);
                }
            }
        }
    }

    // ---- merge the lane groups of this warp ---------------------------------
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float mb = __shfl_xor_sync(kFull, m[g], off);
            const float lb = __shfl_xor_sync(kFull, l[g], off);
            const float mm = fmaxf(m[g], mb);
            const float ca = fast_exp2(m[g] - mm), cb = fast_exp2(mb - mm);
            m[g] = mm;
            l[g] = l[g] * ca + lb * cb;
            const float2 ca2 = make_float2(ca, ca), cb2 = make_float2(cb, cb);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float2 ob;
                ob.x = __shfl_xor_sync(kFull, o2[g][i].x, off);
                ob.y = __shfl_xor_sync(kFull, o2[g][i].y, off);
                o2[g][i] = __ffma2_rn(o2[g][i], ca2, __fmul2_rn(ob, cb2));
            }
        }
    }
    if (tk == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float* dst = mo + (warp * G + g) * D;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                dst[lane_dim<D, INT8>(sub, 2 * i)] = o2[g][i].x;
                dst[lane_dim<D, INT8>(sub, 2 * i + 1)] = o2[g][i].y;
            }
            if (sub == 0) {
                mml[(warp * G + g) * 2] = m[g];
                mml[(warp * G + g) * 2 + 1] = l[g];
            }
        }
    }
    __syncthreads();

    // ---- merge the warps and write ---------------------------------------------
    for (int e = tid; e < G * D; e += kThreads) {
        const int g = e / D, dim = e % D;
        float mm = -1e30f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, mml[(w * G + g) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float c = fast_exp2(mml[(w * G + g) * 2] - mm);
            L += mml[(w * G + g) * 2 + 1] * c;
            O += mo[(w * G + g) * D + dim] * c;
        }
        const size_t hrow = size_t(b) * p.Hq + kvh * G + g;
        if (SPLIT) {
            const size_t w = hrow * p.max_splits + j;
            p.ws_o[w * D + dim] = O;
            if (dim == 0) {
                p.ws_ml[w * 2] = mm;
                p.ws_ml[w * 2 + 1] = L;
            }
        } else {
            const float r = L > 0.f ? O / L : 0.f;
            reinterpret_cast<__nv_bfloat16*>(p.out)[hrow * D + dim] = __float2bfloat16_rn(r);
        }
    }
}

// Split-K merge: one CTA per (query head, sequence).
template <int D>
__global__ void __launch_bounds__(128) splitk_reduce_kernel(const float* __restrict__ ws_o,
                                                            const float* __restrict__ ws_ml,
                                                            const int32_t* __restrict__ ctx_lens,
                                                            int32_t Hq, int32_t split_tokens,
                                                            int32_t max_splits, uint16_t* out,
                                                            int32_t* err) {
    extern __shared__ float cw[];  // [max_splits] weights
    __shared__ float red[32];
    const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    int ctx = ctx_lens[b];
    if (ctx < 0) ctx = 0;
    int ns = (ctx + split_tokens - 1) / split_tokens;
    if (ns > max_splits) {
        if (tid == 0) report(err, kErrCtxLen);
        ns = 0;
    }
    const size_t hrow = size_t(b) * Hq + h;
    const float* ml = ws_ml + hrow * max_splits * 2;
    float mm = -1e30f;
    for (int s = tid; s < ns; s += 128) mm = fmaxf(mm, ml[2 * s]);
    for (int off = 16; off > 0; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFull, mm, off));
    if ((tid & 31) == 0) red[tid >> 5] = mm;
    __syncthreads();
    mm = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    float L = 0.f;
    for (int s = tid; s < ns; s += 128) {
        const float c = fast_exp2(ml[2 * s] - mm);
        cw[s] = c;
        L += c * ml[2 * s + 1];
    }
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
    if ((tid & 31) == 0) red[tid >> 5] = L;
    __syncthreads();
    L = red[0] + red[1] + red[2] + red[3];
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const float* o = ws_o + hrow * max_splits * D;
    for (int dim = tid; dim < D; dim += 128) {
        float acc = 0.f;
        for (int s = 0; s < ns; ++s) acc += cw[s] * o[size_t(s) * D + dim];
        reinterpret_cast<__nv_bfloat16*>(out)[hrow * D + dim] = __float2bfloat16_rn(acc * inv);
    }
}

}  // namespace pkv
