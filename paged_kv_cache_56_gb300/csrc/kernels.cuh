// Device kernels of the paged KV cache: append, quantize-on-fill, decode
// attention (whole context or one split of it) and the split-K merge.
//
// Decode-attention design (sm_103a):
//   * one CTA per (split j, kv head, sequence b); it loads the query rows of
//     the whole GQA group of that kv head, so every KV byte crosses HBM once
//     per step;
//   * four warps; each owns a ring of STAGES shared-memory stages and pulls
//     16-token K and V tiles into them with asynchronous copies of the TMA
//     engine (one elected lane, completion on an mbarrier), gathering tiles
//     through the block table. A (block, kv head) tile is contiguous in the
//     [num_blocks][Hkv][bs][d] pools; rows of 128 or 256 bytes arrive by
//     tensor copies with the 128-byte swizzle (conflict-free shared-memory
//     reads), 64-byte rows by one linear copy per tile;
//   * QK and PV of each 16-token tile run on tensor cores (mma.m16n8k16,
//     fp32 accumulate) straight from registers: INT8 codes are converted
//     exactly to f16 in registers, and the per-block scales are applied to
//     the scores and to the softmax weights, not per element; the weights of
//     an INT8 block are kept inside f16's range by a per-warp power-of-two
//     unit of the accumulator that follows the blocks' V scales;
//   * fp32 online softmax in base 2 (scores pre-multiplied by log2 e); each
//     warp keeps its own state, merged across warps through shared memory;
//     with a bf16 cache the weights enter the PV product as two bf16 terms
//     (rounded weight + residual);
//   * the split holding token ctx-1 first appends that token's row and, when
//     it fills a block, quantizes the block (the decode step fused into one
//     kernel); the last split of a (sequence, kv head) to finish merges the
//     splits' partial states (arrival counter), or a second kernel does;
//   * under programmatic dependent launch the prologue (context length,
//     block table, the first tiles below the block this step may write) runs
//     before waiting for the previous kernel.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

#ifndef PKV_STAGES_INT8
#define PKV_STAGES_INT8 2  // TMA-copy stages per warp, INT8 cache (4 KB each at d = 128)
#endif
#ifndef PKV_STAGES_BF16
#define PKV_STAGES_BF16 2  // TMA-copy stages per warp, bf16 cache (8 KB each at d = 128)
#endif

namespace pkv {

#ifndef PKV_WARPS
#define PKV_WARPS 4  // warps per decode CTA
#endif
constexpr int kWarps = PKV_WARPS;
constexpr int kThreads = kWarps * 32;
// decode CTAs kept resident per SM: 16 warps (the register file at 128 registers a thread)
constexpr int kMinCtas = kWarps >= 16 ? 1 : 16 / kWarps;
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
    // tensor maps of the K and V pools seen as bytes [num_blocks][Hkv*bs][row],
    // 128-byte x 16-row boxes with the 128-byte swizzle (used when a token row
    // is 128 or 256 bytes; unused for 64-byte rows)
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    const void* k_pool;
    const void* v_pool;
    const float* scales;
    const void* k_tail;
    const void* v_tail;
    const uint16_t* q;
    const uint16_t* k_new;  // [B][Hkv][D] rows appended this step (nullable: cache already written)
    const uint16_t* v_new;
    const int32_t* block_tables;
    const int32_t* ctx_lens;
    const int32_t* slots;
    uint16_t* out;
    float* ws_o;
    float* ws_ml;
    int32_t* ws_count;  // split-K arrival counters [B][Hkv] (nullable: merge in a separate kernel)
    int32_t* err;
    int32_t Hq, Hkv, bs, max_blocks, num_blocks, max_slots, split_tokens, max_splits;
    int32_t tab_cap;  // block-table entries the shared table holds (even)
    int32_t skip_copy;  // test build only: the first CTA's warp 0 never issues its tile of this index
    float qscale;     // sm_scale * log2(e)
};

template <int D, bool INT8>
struct DecodeTraits {
    static constexpr int kElemBytes = INT8 ? 1 : 2;
    static constexpr int kRowBytes = D * kElemBytes;
    static constexpr int kTileBytes = kTile * kRowBytes;  // K or V of one tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = INT8 ? PKV_STAGES_INT8 : PKV_STAGES_BF16;
    // Rows of 128 or 256 bytes are staged by tensor copies with the 128-byte
    // swizzle: each 128-byte half of a row goes to its own 2048-byte slab
    // (16 rows x 128 bytes), whose 16-byte chunk c of row r sits at chunk
    // position c ^ (r % 8) -- the eight rows a quarter-warp reads then hit
    // eight different bank groups. 64-byte rows (INT8, d = 64) are copied
    // linearly.
    static constexpr bool kSwz = kRowBytes >= 128;
    // bf16 at d = 128 (256-byte rows, two slabs): the lanes' dims are
    // interleaved over the two halves of a row (see the tile math below).
    static constexpr bool kHalves = !INT8 && D == 128;
    // slack to align the stages to 1024 bytes (the swizzle pattern's period)
    static constexpr int kAlignSlack = kSwz ? 1024 : 0;
};

// Shared-memory bytes of a decode CTA before its block table.
template <int D, bool INT8>
constexpr size_t decode_smem_fixed() {
    using T = DecodeTraits<D, INT8>;
    return size_t(T::kAlignSlack)                         // alignment of the stages
         + size_t(kWarps) * T::kStages * T::kStageBytes   // stages (and, after the loop, the merge)
         + size_t(kWarps) * T::kStages * 8;               // mbarriers
}

// ---- tensor-core tile math ---------------------------------------------------
// One warp computes a 16-token tile with mma.m16n8k16 (fp32 accumulate):
//   S   [16 tok x 8 heads] = K [16 tok x D] . Q^T [D x 8 heads]
//   O^T [D x 8 heads]     += V^T [D x 16 tok] . P^T [16 tok x 8 heads]
// Lane (g = lane / 4, t = lane % 4). The GQA group (G <= 8 query heads) is the
// 8-wide N dimension; heads >= G are zero columns.
// K operand: lane holds tokens g and g+8; the MMA's k index is permuted so
// that lane t's dims for all k-steps are the contiguous run [t*D/4, t*D/4 +
// D/4) (k-step ks uses dims t*D/4 + 4ks + 0..3), the same permutation on Q.
// V operand: m-tile m's rows are dims g*D/8 + 2m (row g) and g*D/8 + 2m + 1
// (row g+8), so lane g reads the contiguous run [g*D/8, g*D/8 + D/8) of
// tokens 2t, 2t+1, 2t+8, 2t+9; the output row of a lane is that run too.
// HALVES (bf16, d = 128: 256-byte rows staged as two 128-byte slabs): the
// runs are split over the two halves of the row instead -- lane t's K dims
// are [16t, 16t+16) and [64+16t, 64+16t+16), lane g's V dims [8g, 8g+8) and
// [64+8g, 64+8g+8) -- so that with the swizzle the 16-byte loads of a
// quarter-warp (g in {2i, 2i+1}, t in 0..3) fall in eight different chunk
// positions, for K (chunk 2t + c ^ g) and for V (chunk g ^ row) alike.
// P^T comes from S by an in-register 8x8 transpose (movmatrix).
// INT8 codes are exact in f16 (x + 1152 = f16 bits 0x6400 | (x ^ 0x80), then
// subtract 1152); bf16 caches multiply in bf16.

template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    if (F16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
            "{%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if (F16) asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t hsub1152(uint32_t x) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x64806480u));  // 1152 = f16 0x6480
    return r;
}

// int8 dims (d, d+1, d+2, d+3) of one word -> f16x2 (d, d+1), (d+2, d+3).
__device__ __forceinline__ void s8_pairs(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    lo = hsub1152(__byte_perm(u, 0x64646464u, 0x4140));
    hi = hsub1152(__byte_perm(u, 0x64646464u, 0x4342));
}

// int8 words of two tokens (same dims d..d+3) -> f16x2 (t0[d+i], t1[d+i]), i = 0..3.
__device__ __forceinline__ void s8_interleave(uint32_t w0, uint32_t w1, uint32_t (&r)[4]) {
    const uint32_t x = __byte_perm(w0, w1, 0x5140) ^ 0x80808080u;
    const uint32_t y = __byte_perm(w0, w1, 0x7362) ^ 0x80808080u;
    r[0] = hsub1152(__byte_perm(x, 0x64646464u, 0x4140));
    r[1] = hsub1152(__byte_perm(x, 0x64646464u, 0x4342));
    r[2] = hsub1152(__byte_perm(y, 0x64646464u, 0x4140));
    r[3] = hsub1152(__byte_perm(y, 0x64646464u, 0x4342));
}

template <int D, bool I8>
struct Geom {
    static constexpr int kE = I8 ? 1 : 2;    // bytes per element
    static constexpr int kRow = D * kE;      // bytes per token row
    static constexpr int kKB = D / 4 * kE;   // K bytes a lane reads per token
    static constexpr int kKW = kKB / 4;      // ... as words
    static constexpr int kVB = D / 8 * kE;   // V bytes a lane reads per token
    static constexpr int kVW = kVB / 4;
    static constexpr int kSteps = D / 16;    // QK k-steps = PV m-tiles
};

// 16-byte / 8-byte row loads from a staged tile (shared) or from global rows.
struct SmemRows {
    uint32_t base;
    int row;  // bytes
    __device__ __forceinline__ uint4 ld16(int r, int off) const { return lds128(base + uint32_t(r * row + off)); }
    __device__ __forceinline__ uint2 ld8(int r, int off) const {
        uint2 v;
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(base + uint32_t(r * row + off)));
        return v;
    }
};
// A tile staged by tensor copies with the 128-byte swizzle (1024-byte
// aligned): byte `off` of row r lies in slab off / 128, at chunk position
// ((off % 128) / 16) ^ (r % 8) of that row.
struct SwzRows {
    uint32_t base;
    __device__ __forceinline__ uint4 ld16(int r, int off) const {
        return lds128(base + uint32_t((off >> 7) * 2048 + r * 128 + ((((off >> 4) & 7) ^ (r & 7)) << 4)));
    }
};
struct GmemRows {  // rows this kernel may itself have written: read through L2
    const uint8_t* base;
    int row;
    __device__ __forceinline__ uint4 ld16(int r, int off) const { return ldcg128(base + size_t(r) * row + off); }
    __device__ __forceinline__ uint2 ld8(int r, int off) const {
        return __ldcg(reinterpret_cast<const uint2*>(base + size_t(r) * row + off));
    }
};

// Byte offset in a row of the c-th 16-byte chunk of a lane's K run (lane t)
// or V run (lane g), NB bytes long; HALVES splits the run over the two
// 128-byte halves of the row (see the tile math above).
template <int NB, bool HALVES>
__device__ __forceinline__ int k_chunk(int t, int c) {
    return HALVES ? (c >> 1) * 128 + t * (NB / 2) + (c & 1) * 16 : t * NB + c * 16;
}
template <int NB, bool HALVES>
__device__ __forceinline__ int v_chunk(int g, int c) {
    return HALVES ? c * 128 + g * (NB / 2) : g * NB + c * 16;
}

// The NB bytes of a lane's run in row r: 16-byte chunks at chunk(c), or one
// 8-byte piece at chunk(0).
template <int NB, class Rows, class Chunk>
__device__ __forceinline__ void load_run(const Rows& R, int r, Chunk chunk, uint32_t* w) {
    if constexpr (NB % 16 == 0) {
#pragma unroll
        for (int c = 0; c < NB / 16; ++c) {
            const uint4 v = R.ld16(r, chunk(c));
            w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
        }
    } else {
        static_assert(NB == 8, "8- or 16k-byte runs");
        const uint2 v = R.ld8(r, chunk(0));
        w[0] = v.x; w[1] = v.y;
    }
}

// Per-warp online-softmax state: heads 2t and 2t+1 (replicated over g);
// l is this lane's partial sum over its tokens; acc holds O^T fragments.
// INT8 caches (SHIFT): the weights are taken against md = m - delta, i.e.
// scaled by 2^delta, so that acc and l are kept in units of 2^-delta (see
// kExpNone) and the weights times a block's V scale fit f16 whatever the
// scale; otherwise md is unused and delta = 0.
template <int D>
struct WarpState {
    float m[2], md[2], l[2];
    float acc[D / 16][4];
};

// 2^n as a float for -126 <= n <= 127.
__device__ __forceinline__ float exp2i(int n) { return __int_as_float((n + 127) << 23); }

// One 16-token tile. nvalid < 16 masks the last rows: their scores become
// -inf and their V values 0, so stale or uninitialised rows cannot leak NaNs.
// hs[j]: log2-domain logit factor of head 2t+j; ksc: the block's K scale;
// vmul: factor on the softmax weights before the PV product (the block's V
// scale for INT8 tiles). SHIFT: weights against st.md (see WarpState), with
// md kept at m - delta. HALVES: the lanes' dims split over the row's halves.
template <int D, bool I8, bool SHIFT, bool HALVES, class Rows>
__device__ __forceinline__ void mma_tile(const Rows& K, const Rows& V, int nvalid, float ksc, float vmul,
                                         float delta, const uint32_t (&qf)[D / 16][2], const float (&hs)[2],
                                         int g, int t, WarpState<D>& st) {
    using Gm = Geom<D, I8>;
    constexpr bool F16 = I8;
    // ---- S = K . Q^T (two independent accumulator chains, summed)
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    {
        float s2[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t k0[Gm::kKW], k1[Gm::kKW];
        const auto kc = [t](int c) { return k_chunk<Gm::kKB, HALVES>(t, c); };
        load_run<Gm::kKB>(K, g, kc, k0);
        load_run<Gm::kKB>(K, g + 8, kc, k1);
#pragma unroll
        for (int ks = 0; ks < Gm::kSteps; ++ks) {
            uint32_t a0, a1, a2, a3;
            if (I8) {
                s8_pairs(k0[ks], a0, a2);
                s8_pairs(k1[ks], a1, a3);
            } else {
                a0 = k0[2 * ks]; a2 = k0[2 * ks + 1];
                a1 = k1[2 * ks]; a3 = k1[2 * ks + 1];
            }
            if (ks & 1) mma16816<F16>(s2, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            else mma16816<F16>(s, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] += s2[i];
    }
    const float f0 = ksc * hs[0], f1 = ksc * hs[1];
    s[0] *= f0; s[1] *= f1; s[2] *= f0; s[3] *= f1;
    const bool full = nvalid >= kTile;
    if (!full) {
        if (g >= nvalid) s[0] = s[1] = -INFINITY;
        if (g + 8 >= nvalid) s[2] = s[3] = -INFINITY;
    }
    // ---- online softmax over the 16 tokens of each head
    float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, off));
    }
    mx0 = fmaxf(mx0, st.m[0]);
    mx1 = fmaxf(mx1, st.m[1]);
    if (__any_sync(kFull, (mx0 > st.m[0]) | (mx1 > st.m[1]))) {
        const float c0 = fast_exp2(st.m[0] - mx0), c1 = fast_exp2(st.m[1] - mx1);
        st.m[0] = mx0;
        st.m[1] = mx1;
        if (SHIFT) {
            st.md[0] = mx0 - delta;
            st.md[1] = mx1 - delta;
        }
        st.l[0] *= c0;
        st.l[1] *= c1;
#pragma unroll
        for (int m = 0; m < Gm::kSteps; ++m) {
            st.acc[m][0] *= c0; st.acc[m][1] *= c1; st.acc[m][2] *= c0; st.acc[m][3] *= c1;
        }
    }
    const float r0 = SHIFT ? st.md[0] : st.m[0], r1 = SHIFT ? st.md[1] : st.m[1];
    const float p0 = fast_exp2(s[0] - r0), p1 = fast_exp2(s[1] - r1);
    const float p2 = fast_exp2(s[2] - r0), p3 = fast_exp2(s[3] - r1);
    st.l[0] += p0 + p2;
    st.l[1] += p1 + p3;
    const float x0 = p0 * vmul, x1 = p1 * vmul, x2 = p2 * vmul, x3 = p3 * vmul;
    const uint32_t w01 = pack2<F16>(x0, x1), w23 = pack2<F16>(x2, x3);
    const uint32_t b0 = movmatrix_t(w01), b1 = movmatrix_t(w23);
    // bf16 keeps 8 bits of a weight (a relative error up to 2^-9, visible when
    // a few tokens dominate); the rounding residual goes in as a second bf16
    // term, so that P enters the sum to ~2^-17 like the fp32 l beside it
    uint32_t b0l = 0u, b1l = 0u;
    if (!F16) {
        const float2 h01 = bf16x2_to_f2(w01), h23 = bf16x2_to_f2(w23);
        b0l = movmatrix_t(pack2<false>(x0 - h01.x, x1 - h01.y));
        b1l = movmatrix_t(pack2<false>(x2 - h23.x, x3 - h23.y));
    }
    // ---- O^T += V^T . P^T
    uint32_t v0[Gm::kVW], v1[Gm::kVW], v2[Gm::kVW], v3[Gm::kVW];
    const auto vc = [g](int c) { return v_chunk<Gm::kVB, HALVES>(g, c); };
    load_run<Gm::kVB>(V, 2 * t, vc, v0);
    load_run<Gm::kVB>(V, 2 * t + 1, vc, v1);
    load_run<Gm::kVB>(V, 2 * t + 8, vc, v2);
    load_run<Gm::kVB>(V, 2 * t + 9, vc, v3);
    if (!full) {
#pragma unroll
        for (int i = 0; i < Gm::kVW; ++i) {
            if (2 * t >= nvalid) v0[i] = 0u;
            if (2 * t + 1 >= nvalid) v1[i] = 0u;
            if (2 * t + 8 >= nvalid) v2[i] = 0u;
            if (2 * t + 9 >= nvalid) v3[i] = 0u;
        }
    }
    if (I8) {
#pragma unroll
        for (int j = 0; j < Gm::kVW; ++j) {
            uint32_t r01[4], r23[4];
            s8_interleave(v0[j], v1[j], r01);
            s8_interleave(v2[j], v3[j], r23);
            mma16816<true>(st.acc[2 * j], r01[0], r01[1], r23[0], r23[1], b0, b1);
            mma16816<true>(st.acc[2 * j + 1], r01[2], r01[3], r23[2], r23[3], b0, b1);
        }
    } else {
#pragma unroll
        for (int j = 0; j < Gm::kVW; ++j) {
            const uint32_t a0 = __byte_perm(v0[j], v1[j], 0x5410), a1 = __byte_perm(v0[j], v1[j], 0x7632);
            const uint32_t a2 = __byte_perm(v2[j], v3[j], 0x5410), a3 = __byte_perm(v2[j], v3[j], 0x7632);
            mma16816<false>(st.acc[j], a0, a1, a2, a3, b0, b1);
            mma16816<false>(st.acc[j], a0, a1, a2, a3, b0l, b1l);
        }
    }
}

// The query words behind a lane's Q^T fragments (head g, zero for g >= G):
// dims t*D/4 .. t*D/4 + D/4 - 1 of the query row (HALVES: the split run of
// the K operand), read through L2 (the row is written by the kernel this one
// waits for).
template <int D, int G, bool HALVES>
__device__ __forceinline__ void load_q_words(const uint16_t* qrow, int g, int t, uint32_t (&w)[D / 8]) {
    constexpr int NW = D / 8;  // bf16 words in a lane's D/4 dims
    if (g < G) {
#pragma unroll
        for (int c = 0; c < NW / 4; ++c) {
            const uint4 v = ldcg128(qrow + k_chunk<D / 2, HALVES>(t, c) / 2);
            w[4 * c] = v.x; w[4 * c + 1] = v.y; w[4 * c + 2] = v.z; w[4 * c + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < NW; ++i) w[i] = 0u;
    }
}

// Q^T fragments from the words of load_q_words: dims t*D/4 + 4ks + {0,1} and
// {2,3} of the query row. F16: the row is scaled by 2^e (e per head, chosen so
// that max|q| * 2^e lies in [2^14, 2^15) -- exact, and safe from f16
// overflow); returns e. BF16: the raw row, e = 0.
template <int D, bool F16>
__device__ __forceinline__ int q_frags(const uint32_t (&w)[D / 8], uint32_t (&qf)[D / 16][2]) {
    constexpr int NW = D / 8;
    if (!F16) {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            qf[ks][0] = w[2 * ks];
            qf[ks][1] = w[2 * ks + 1];
        }
        return 0;
    }
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        const float2 f = bf16x2_to_f2(w[i]);
        mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
    int e = 0;
    if (mx > 0.f) e = 15 - (int((__float_as_uint(mx) >> 23) & 0xFF) - 126);
    e = max(-100, min(100, e));
    const float sc = ldexpf(1.0f, e);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const float2 a = bf16x2_to_f2(w[2 * ks]), b = bf16x2_to_f2(w[2 * ks + 1]);
        qf[ks][0] = pack2<true>(a.x * sc, a.y * sc);
        qf[ks][1] = pack2<true>(b.x * sc, b.y * sc);
    }
    return e;
}

// Quantizes one (block, kv head, K|V) slab of bs x D bf16 values with one
// warp, the definition of the INT8 cache ("轻量级推理引擎实战" §3 under this
// build's readings): scale = max|x| / 127 by IEEE fp32 division, or 1.0 when
// max|x| < 1e-6; code = clamp(round-half-even(x / scale), -127, 127) with
// IEEE fp32 division. Source rows are `row_stride` elements apart; the codes
// are written to `dst` as bs x D bytes and the scale to *scale_out.
// COHERENT: read the source through L2 (it was written earlier in this kernel).
template <int D, bool COHERENT>
__device__ __forceinline__ void quantize_slab(int lane, const uint16_t* base, int64_t row_stride, int bs,
                                              int8_t* dst, float* scale_out) {
    constexpr int CH = D / 8;
    const int nch = bs * CH;
    auto load = [&](int c) {
        const uint16_t* ptr = base + int64_t(c / CH) * row_stride + (c % CH) * 8;
        return COHERENT ? ldcg128(ptr) : ldg128(ptr);
    };
    float mx = 0.f;
    for (int c = lane; c < nch; c += 32) {
        const uint4 w = load(c);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = bf16x2_to_f2(ws[i]);
            mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    const float scale = mx < 1e-6f ? 1.0f : __fdiv_rn(mx, 127.0f);
    for (int c = lane; c < nch; c += 32) {
        const uint4 w = load(c);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        uint32_t packed[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = bf16x2_to_f2(ws[i]);
            int q0 = __float2int_rn(__fdiv_rn(f.x, scale));
            int q1 = __float2int_rn(__fdiv_rn(f.y, scale));
            q0 = min(127, max(-127, q0));
            q1 = min(127, max(-127, q1));
            const uint32_t pair = (uint32_t(q0) & 0xFFu) | ((uint32_t(q1) & 0xFFu) << 8);
            packed[i >> 1] |= pair << (16 * (i & 1));
        }
        *reinterpret_cast<uint2*>(dst + int64_t(c) * 8) = make_uint2(packed[0], packed[1]);
    }
    if (lane == 0) *scale_out = scale;
}

// Waits for an mbarrier phase for at most ~1 s of GPU time. A waiting warp
// sleeps in try_wait (up to 2 us per poll) rather than spinning, so it does
// not take issue slots from warps that have data.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 2000u)) return true;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > 1000000000ull) return false;
    }
}

// Quantize-on-fill inside the decode kernel: the K and V slabs of block `id`
// (bs rows of D bf16 each) from the slot's bf16 tail rows, except row `off`
// -- the row this step appends -- which is taken from the new row itself
// (nrow_k / nrow_v), so the quantizer need not wait for that row's store.
// Half of the CTA's threads take each slab, 16 rows at a time: a thread
// holds its chunks of those rows in registers, with all their loads in flight
// at once. A 16-row block is read once; a larger one is read a second time
// (from L2) for the codes. The arithmetic is quantize_slab's (absmax, IEEE
// scale = max/127, round-half-even, clamp to +-127): the same bits.
template <int D>
__device__ __forceinline__ void fill_quantize(const DecodeParams& p, const uint16_t* tail_k, const uint16_t* tail_v,
                                              const uint16_t* nrow_k, const uint16_t* nrow_v, int off, int id,
                                              int kvh) {
    constexpr int CH = D / 8;              // 16-byte chunks per row
    constexpr int TPS = kThreads / 2;      // threads per slab
    static_assert((kTile * CH) % TPS == 0, "16 rows' chunks split evenly over a slab's threads");
    constexpr int NB = kTile * CH / TPS;   // chunks a thread holds per 16 rows
    __shared__ float s_mx[kWarps];
    const int tid = threadIdx.x, kv = tid / TPS, t = tid % TPS, warp = tid >> 5, lane = tid & 31;
    const int npass = p.bs / kTile;
    const uint16_t* tail = kv ? tail_v : tail_k;
    const uint16_t* nrow = kv ? nrow_v : nrow_k;
    uint4 w[NB];
    auto load = [&](int pass) {
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int c = pass * kTile * CH + t + i * TPS, r = c / CH, ch = c % CH;
            w[i] = r == off ? ldg128(nrow + ch * 8) : ldcg128(tail + size_t(r) * D + ch * 8);
        }
    };
    float mx = 0.f;
    for (int pass = 0; pass < npass; ++pass) {
        load(pass);
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = bf16x2_to_f2(ws[k]);
                mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    if (lane == 0) s_mx[warp] = mx;
    __syncthreads();
    constexpr int WPS = TPS / 32;  // warps per slab
    mx = 0.f;
#pragma unroll
    for (int k = 0; k < WPS; ++k) mx = fmaxf(mx, s_mx[kv * WPS + k]);
    const float scale = mx < 1e-6f ? 1.0f : __fdiv_rn(mx, 127.0f);
    int8_t* dst = static_cast<int8_t*>(const_cast<void*>(kv ? p.v_pool : p.k_pool)) +
                  (size_t(id) * p.Hkv + kvh) * p.bs * D;
    for (int pass = 0; pass < npass; ++pass) {
        if (npass > 1) load(pass);  // one pass: still held from the maximum
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int c = pass * kTile * CH + t + i * TPS;
            const uint32_t ws[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
            uint32_t packed[2] = {0u, 0u};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = bf16x2_to_f2(ws[k]);
                int q0 = __float2int_rn(__fdiv_rn(f.x, scale));
                int q1 = __float2int_rn(__fdiv_rn(f.y, scale));
                q0 = min(127, max(-127, q0));
                q1 = min(127, max(-127, q1));
                const uint32_t pair = (uint32_t(q0) & 0xFFu) | ((uint32_t(q1) & 0xFFu) << 8);
                packed[k >> 1] |= pair << (16 * (k & 1));
            }
            *reinterpret_cast<uint2*>(dst + size_t(c) * 8) = make_uint2(packed[0], packed[1]);
        }
    }
    if (t == 0) const_cast<float*>(p.scales)[(size_t(id) * p.Hkv + kvh) * 2 + kv] = scale;
}

// The step update of (sequence b, kv head kvh) whose context now ends at
// token ctx-1: writes that token's K/V row (k_new / v_new) into the cache --
// the slot's bf16 tail (INT8) or pool block `id` (bf16) -- and, in INT8 mode,
// quantizes block `id` if the row filled it ("轻量级推理引擎实战" §3,
// quantize-on-fill). Called by every thread of the CTA; ends with a barrier.
template <int D, bool INT8>
__device__ __forceinline__ void step_update(const DecodeParams& p, const int b, const int kvh, const int ctx,
                                            const int id) {
    const int tid = threadIdx.x;
    const int pos = ctx - 1, off = pos % p.bs;
    const int slot = (INT8 && p.slots) ? p.slots[b] : -1;
    const bool ok = INT8 ? (slot >= 0 && slot < p.max_slots) : (id >= 0);
    if (ok) {
        const size_t row = INT8 ? (size_t(slot) * p.Hkv + kvh) * p.bs + off : (size_t(id) * p.Hkv + kvh) * p.bs + off;
        uint16_t* dk = static_cast<uint16_t*>(const_cast<void*>(INT8 ? p.k_tail : p.k_pool)) + row * D;
        uint16_t* dv = static_cast<uint16_t*>(const_cast<void*>(INT8 ? p.v_tail : p.v_pool)) + row * D;
        const uint16_t* sk = p.k_new + (size_t(b) * p.Hkv + kvh) * D;
        const uint16_t* sv = p.v_new + (size_t(b) * p.Hkv + kvh) * D;
        for (int c = tid; c < 2 * (D / 8); c += kThreads) {
            const int kv = c / (D / 8), ch = c % (D / 8);
            *reinterpret_cast<uint4*>((kv ? dv : dk) + ch * 8) = ldg128((kv ? sv : sk) + ch * 8);
        }
        if (!INT8) fence_proxy_async_global();  // the pool row is read by a TMA copy later
    } else if (tid == 0) {
        report(p.err, INT8 ? kErrSlot : kErrBlockId);
    }
    if (INT8 && ok && (pos + 1) % p.bs == 0) {  // the row filled block id
        if (id >= 0) {
            const size_t t0 = (size_t(slot) * p.Hkv + kvh) * p.bs * D;
            const uint16_t* tk = static_cast<const uint16_t*>(p.k_tail) + t0;
            const uint16_t* tv = static_cast<const uint16_t*>(p.v_tail) + t0;
            const uint16_t* nk = p.k_new + (size_t(b) * p.Hkv + kvh) * D;
            const uint16_t* nv = p.v_new + (size_t(b) * p.Hkv + kvh) * D;
            fill_quantize<D>(p, tk, tv, nk, nv, off, id, kvh);
            fence_proxy_async_global();  // the codes are read by a TMA copy later
        } else if (tid == 0) {
            report(p.err, kErrBlockId);
        }
    }
    __syncthreads();
}

// INT8 caches keep the PV accumulators (and l) of a CTA in units of
// 2^(ew - 14), where ew is the largest exponent among the V scales of the
// CTA's blocks: a block's softmax weights enter the f16 product as
// p * 2^(14 - ew) * vscale < 2^15, finite whatever the scales (the factor
// 2^delta, delta = 14 - ew, is taken into the softmax's reference maximum, so
// no tile pays a multiply for it). A block whose V scale is 2^k below the
// largest keeps f16's normal range for weights p >= 2^(k - 28); smaller
// weights of such a block lose relative precision (below 2^-24 of that
// block's largest contribution, they flush to zero).
constexpr int kExpNone = -1000;

// Decode attention, one CTA per (split j = blockIdx.x, kv head = blockIdx.y,
// sequence b = blockIdx.z). HOOK: the test build of pkv_debug_skip_copy, which
// can leave one tile's copies unissued.
template <int D, int G, bool INT8, bool SPLIT, bool HOOK>
__global__ void __launch_bounds__(kThreads, kMinCtas) decode_kernel(const __grid_constant__ DecodeParams p) {
    static_assert(G >= 1 && G <= 8, "the GQA group is the MMA's 8-wide N dimension");
    using T = DecodeTraits<D, INT8>;
    using Gm = Geom<D, INT8>;
    constexpr int STAGES = T::kStages;
    constexpr bool HALVES = T::kHalves;
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_launch_dependents();
    const int j = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    uint8_t* stages = smem + (T::kSwz ? (1024u - (smem_addr(smem) & 1023u)) & 1023u : 0u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(stages + size_t(kWarps) * STAGES * T::kStageBytes);
    int32_t* tab = reinterpret_cast<int32_t*>(bars + kWarps * STAGES);
    float2* bsc = reinterpret_cast<float2*>(tab + p.tab_cap);
    // Cross-warp merge space: warp w's o [G][D] and (m, l) [G][2], in its own
    // ring (free once its last tile has been consumed).
    static_assert(G * D * 4 + G * 8 <= STAGES * T::kStageBytes, "merge space fits one warp's ring");
    auto mo_of = [&](int w) { return reinterpret_cast<float*>(stages + size_t(w) * STAGES * T::kStageBytes); };
    auto mml_of = [&](int w) { return mo_of(w) + G * D; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;

    // Before pdl_wait() this kernel reads only what no preceding kernel of the
    // step writes: context lengths, block tables, slots, and the blocks (and
    // scales) below the one holding token ctx-1 -- the only block this step's
    // append / quantize-on-fill may have written.
    const int t0 = SPLIT ? j * p.split_tokens : 0;
    // the first table entry of each thread is loaded together with the
    // context length (the table row starts at t0, known without it), so the
    // two reads cost one round trip instead of two
    const int32_t* trow = p.block_tables + size_t(b) * p.max_blocks + t0 / p.bs;
    const int id_first = (t0 / p.bs + tid < p.max_blocks && tid < p.tab_cap) ? trow[tid] : -1;
    const int slot = (INT8 && p.slots) ? p.slots[b] : -1;
    int ctx = p.ctx_lens[b];
    if (ctx < 0 || ctx > p.max_blocks * p.bs) {
        if (tid == 0 && j == 0) report(p.err, kErrCtxLen);
        ctx = 0;
    }
    const int t1 = SPLIT ? min(ctx, t0 + p.split_tokens) : ctx;
    if (t0 >= t1 && j > 0) return;  // past the context

    const int nfull = INT8 ? (ctx / p.bs) * p.bs : ctx;
    const int pool_end = min(t1, nfull);
    const int npool = max(0, pool_end - t0);
    const int nt = (npool + kTile - 1) / kTile;
    const int blk0 = t0 / p.bs;
    const int nblk = npool > 0 ? min((pool_end - 1) / p.bs - blk0 + 1, p.tab_cap) : 0;
    // the block holding token ctx-1 may change this step
    const int last_blk = ctx > 0 ? (ctx - 1) / p.bs : 0;
    const int nt_stable = max(0, min(nt, (last_blk * p.bs - t0) / kTile));  // tiles below it
    const int nblk_stable = max(0, min(nblk, last_blk - blk0));

    // INT8: the largest V-scale exponent of the CTA's blocks, one slot per warp
    __shared__ int s_ev[kWarps];
    // exponent of a V scale (a positive normal float for every block the
    // quantizer wrote; 0 marks a block id the table check dropped), clamped so
    // that the powers of two built from it stay finite
    auto v_exp = [](float v) {
        const uint32_t u = __float_as_uint(v);
        return u ? min(121, max(-40, int((u >> 23) & 0xFFu) - 127)) : kExpNone;
    };

    const uint32_t bar0 = smem_addr(bars);
    const uint32_t stage0 = smem_addr(stages);
    // this warp's k-th tile uses ring stage k % STAGES and waits for
    // completion number k / STAGES of that stage's mbarrier
    auto bar_of = [&](int s) { return bar0 + uint32_t(warp * STAGES + s) * 8u; };
    auto stage_of = [&](int s) { return stage0 + uint32_t(warp * STAGES + s) * T::kStageBytes; };

    if (lane == 0)
        for (int s = 0; s < STAGES; ++s) mbar_init(bar_of(s), 1);
    for (int i = tid; i < nblk; i += kThreads) {
        int id = i == tid ? id_first : trow[i];
        if (id < 0 || id >= p.num_blocks) {
            report(p.err, kErrBlockId);
            id = -1;
        }
        tab[i] = id;
    }
    fence_mbar_init();
    __syncthreads();

    const uint64_t pol = l2_policy_evict_first();
    if (T::kSwz && tid == 0) {
        prefetch_tensormap(&p.tm_k);
        prefetch_tensormap(&p.tm_v);
    }
    auto issue = [&](int tile, int s) {
        const int tok = t0 + tile * kTile;
        const int id = tab[tok / p.bs - blk0];
        const uint32_t bar = bar_of(s);
        if (HOOK && tile == p.skip_copy && warp == 0 && blockIdx.x + blockIdx.y + blockIdx.z == 0) return;
        if (id < 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, T::kStageBytes);
        if constexpr (T::kSwz) {
            // boxes of 16 rows x 128 bytes at x = 0 (and 128): rows kvh*bs +
            // tok % bs .. + 15 of block id, inside the block as bs % 16 == 0
            const int y = kvh * p.bs + tok % p.bs;
#pragma unroll
            for (int h = 0; h < T::kRowBytes / 128; ++h) {
                tma_load_3d(stage_of(s) + h * 2048, &p.tm_k, h * 128, y, id, bar, pol);
                tma_load_3d(stage_of(s) + T::kTileBytes + h * 2048, &p.tm_v, h * 128, y, id, bar, pol);
            }
        } else {
            const size_t row = (size_t(id) * p.Hkv + kvh) * p.bs + (tok % p.bs);
            const uint8_t* ks = static_cast<const uint8_t*>(p.k_pool) + row * T::kRowBytes;
            const uint8_t* vs = static_cast<const uint8_t*>(p.v_pool) + row * T::kRowBytes;
            bulk_g2s(stage_of(s), ks, T::kTileBytes, bar, pol);
            bulk_g2s(stage_of(s) + T::kTileBytes, vs, T::kTileBytes, bar, pol);
        }
    };
    // block scales, copied asynchronously (waited for before the main loop)
    auto load_scales = [&](int lo, int hi) {
        for (int i = lo + tid; i < hi; i += kThreads) {
            const int id = tab[i];
            if (id >= 0)
                cp_async8(smem_addr(bsc + i), p.scales + (size_t(id) * p.Hkv + kvh) * 2);
            else
                bsc[i] = make_float2(0.f, 0.f);
        }
    };
    if (lane == 0)
        for (int s = 0; s < STAGES; ++s) {
            const int tile = warp + s * kWarps;
            if (tile < nt_stable) issue(tile, s);
        }
    int ev_max = kExpNone;  // this thread's blocks; loads complete while the previous kernel drains
    if (INT8) {
        load_scales(0, nblk_stable);
        for (int i = tid; i < nblk_stable; i += kThreads) {
            const int id = tab[i];
            if (id >= 0) ev_max = max(ev_max, v_exp(__ldg(p.scales + (size_t(id) * p.Hkv + kvh) * 2 + 1)));
        }
    }

    pdl_wait();  // the previous kernel (and so the previous layer) has completed

    // the query: loaded first, so that its latency overlaps the update below
    const uint16_t* qbase = p.q + (size_t(b) * p.Hq + size_t(kvh) * G) * D;
    uint32_t qw[D / 8];
    load_q_words<D, G, HALVES>(qbase + size_t(g) * D, g, t, qw);

    // ---- fused step update: the split holding token ctx-1 writes that token's
    // K/V row (given in k_new / v_new) and, in INT8 mode, quantizes its block if
    // the row filled it -- before any read of that block.
    if (p.k_new != nullptr && ctx > 0 && t0 <= ctx - 1 && ctx - 1 < t1) {
        const int bl = (ctx - 1) / p.bs - blk0;
        step_update<D, INT8>(p, b, kvh, ctx, (bl >= 0 && bl < nblk) ? tab[bl] : -1);
    }

    if (lane == 0)
        for (int s = 0; s < STAGES; ++s) {
            const int tile = warp + s * kWarps;
            if (tile >= nt_stable && tile < nt) issue(tile, s);
        }
    if (INT8) {
        load_scales(nblk_stable, nblk);
        // the block this step may have filled: its scale was written above
        for (int i = nblk_stable + tid; i < nblk; i += kThreads) {
            const int id = tab[i];
            if (id >= 0) ev_max = max(ev_max, v_exp(__ldcg(p.scales + (size_t(id) * p.Hkv + kvh) * 2 + 1)));
        }
    }

    // a warp's state -> o [G][D] and (m, l) [G][2] in shared memory, in plain
    // units (acc and l times `units`); l is summed over the lanes of a head first
    auto store_state = [&](WarpState<D>& w, float* o, float* ml, float units) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            w.l[0] += __shfl_xor_sync(kFull, w.l[0], off);
            w.l[1] += __shfl_xor_sync(kFull, w.l[1], off);
        }
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int h = 2 * t + jj;
            if (h < G) {
                float* dst = o + h * D;
#pragma unroll
                for (int m = 0; m < D / 16; ++m) {
                    // dims of m-tile m's rows g and g+8 (see the tile math)
                    const int d0 = HALVES ? (m >> 2) * (D / 2) + g * 8 + 2 * (m & 3) : g * (D / 8) + 2 * m;
                    dst[d0] = w.acc[m][jj] * units;
                    dst[d0 + 1] = w.acc[m][2 + jj] * units;
                }
                if (g == 0) {
                    ml[h * 2] = w.m[jj];
                    ml[h * 2 + 1] = w.l[jj] * units;
                }
            }
        }
    };
    auto init_state = [&](WarpState<D>& w) {
        w.m[0] = w.m[1] = w.md[0] = w.md[1] = -1e30f;
        w.l[0] = w.l[1] = 0.f;
#pragma unroll
        for (int m = 0; m < D / 16; ++m) w.acc[m][0] = w.acc[m][1] = w.acc[m][2] = w.acc[m][3] = 0.f;
    };

    // ---- INT8: the partly filled last block, read from the slot's bf16 tail.
    // Done before the pool tiles, so that its global loads overlap the ring's
    // first copies; tail tile tt goes to warp kWarps-1-tt (the warps with
    // the fewest pool tiles), accumulated in plain units (converted to the
    // CTA's units once those are known).
    const int tail_lo = INT8 ? max(t0, nfull) : 0;
    const int ntail = INT8 ? t1 - tail_lo : 0;
    const bool tail_ok = ntail > 0 && slot >= 0 && slot < p.max_slots;
    if (INT8 && ntail > 0 && !tail_ok && tid == 0) report(p.err, kErrSlot);
    const int ntt = tail_ok ? (ntail + kTile - 1) / kTile : 0;  // tail tiles (<= bs / 16 <= kWarps)
    WarpState<D> st;
    init_state(st);
    const bool tail_warp = INT8 && kWarps - 1 - warp < ntt;
    if (tail_warp) {
        const int tt = kWarps - 1 - warp;
        uint32_t qb[D / 16][2];
        (void)q_frags<D, false>(qw, qb);
        const float hb[2] = {p.qscale, p.qscale};
        const size_t rbase = (size_t(slot) * p.Hkv + kvh) * p.bs + (tail_lo - nfull) + tt * kTile;
        const GmemRows kr{static_cast<const uint8_t*>(p.k_tail) + rbase * D * 2, D * 2};
        const GmemRows vr{static_cast<const uint8_t*>(p.v_tail) + rbase * D * 2, D * 2};
        mma_tile<D, false, INT8, false>(kr, vr, min(kTile, ntail - tt * kTile), 1.f, 1.f, 0.f, qb, hb, g, t, st);
    }

    uint32_t qf[D / 16][2];
    const int qe = q_frags<D, INT8>(qw, qf);
    float hs[2];
#pragma unroll
    for (int jj = 0; jj < 2; ++jj) {
        const int eh = __shfl_sync(kFull, qe, ((2 * t + jj) & 7) * 4);
        hs[jj] = p.qscale * ldexpf(1.0f, -eh);
    }
    if (INT8) {
        cp_async_wait_all();  // this thread's scale copies
        // reduced after the tail, whose loads overlap the scales' latency
        ev_max = __reduce_max_sync(kFull, ev_max);
        if (lane == 0) s_ev[warp] = ev_max;
    }
    __syncthreads();

    // INT8: the CTA's accumulator units (see kExpNone)
    int ew = 14;
    if (INT8) {
        int e = kExpNone;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) e = max(e, s_ev[w]);
        if (e != kExpNone) ew = e;  // else: no pool block
    }
    const float delta = float(14 - ew);
    if (INT8) {
        st.md[0] = st.m[0] - delta;
        st.md[1] = st.m[1] - delta;
        if (tail_warp && ew != 14) {  // the tail's plain units -> the CTA's
            const float f = exp2i(14 - ew);
            st.l[0] *= f;
            st.l[1] *= f;
#pragma unroll
            for (int m = 0; m < D / 16; ++m)
#pragma unroll
                for (int i = 0; i < 4; ++i) st.acc[m][i] *= f;
        }
    }

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
        float ksc = 1.f, vmul = 1.f;
        if (INT8) {
            const float2 sc = bsc[bl];
            ksc = sc.x;
            vmul = sc.y;
        }
        if constexpr (T::kSwz) {
            const SwzRows kr{stage_of(s)}, vr{stage_of(s) + T::kTileBytes};
            mma_tile<D, INT8, INT8, HALVES>(kr, vr, nvalid, ksc, vmul, delta, qf, hs, g, t, st);
        } else {
            const SmemRows kr{stage_of(s), Gm::kRow}, vr{stage_of(s) + T::kTileBytes, Gm::kRow};
            mma_tile<D, INT8, INT8, false>(kr, vr, nvalid, ksc, vmul, delta, qf, hs, g, t, st);
        }
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

    store_state(st, mo_of(warp), mml_of(warp), INT8 ? exp2i(ew - 14) : 1.f);
    __syncthreads();

    // ---- merge the warps and write ---------------------------------------------
    if (SPLIT && ctx == 0) {
        // no tokens: a zero row (no partials, no counter)
        for (int e = tid; e < G * D; e += kThreads)
            reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t(b) * p.Hq + kvh * G) * D + e] = __float2bfloat16_rn(0.f);
        return;
    }
    // With the fused merge, a sequence whose context fits one split has
    // nothing to merge: its only split writes the output itself.
    const int ns = SPLIT ? (ctx + p.split_tokens - 1) / p.split_tokens : 1;
    const bool partial = SPLIT && !(p.ws_count && ns == 1);
    for (int e = tid; e < G * D; e += kThreads) {
        const int h = e / D, dim = e % D;
        float mm = -1e30f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, mml_of(w)[h * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float c = fast_exp2(mml_of(w)[h * 2] - mm);
            L += mml_of(w)[h * 2 + 1] * c;
            O += mo_of(w)[h * D + dim] * c;
        }
        const size_t hrow = size_t(b) * p.Hq + kvh * G + h;
        if (partial) {
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
    if (partial && p.ws_count) {
        // Fused split-K merge: the last split of (b, kv head) to arrive merges
        // all of them. Partials are read through L2 (past this SM's L1).
        __shared__ int s_last;
        int32_t* cnt = p.ws_count + size_t(b) * p.Hkv + kvh;
        __syncthreads();
        if (tid == 0) s_last = atom_add_acq_rel_gpu(cnt, 1) == ns - 1;
        __syncthreads();
        if (!s_last) return;
        constexpr int EPT = (G * D + kThreads - 1) / kThreads;  // output elements per thread
        constexpr int QB = EPT >= 48 ? 1 : 48 / EPT;   // splits per batch of loads
        // [G][ns] weights, then [G] sums, in the rings
        float* wsm = reinterpret_cast<float*>(stages);
        const bool staged = size_t(G) * ns + G <= size_t(kWarps) * STAGES * T::kStageBytes / 4;
        // first batch of partial outputs: issued before the weights are known
        float ov[QB][EPT];
        auto load_o = [&](int q0) {
#pragma unroll
            for (int u = 0; u < QB; ++u)
#pragma unroll
                for (int i = 0; i < EPT; ++i) {
                    const int e = tid + i * kThreads, h = e / D, dim = e % D;
                    const size_t hrow = size_t(b) * p.Hq + kvh * G + h;
                    ov[u][i] = (q0 + u < ns && e < G * D)
                                   ? __ldcg(p.ws_o + (hrow * p.max_splits + q0 + u) * D + dim) : 0.f;
                }
        };
        load_o(0);
        if (staged) {
            for (int h = warp; h < G; h += kWarps) {
                const size_t hrow = size_t(b) * p.Hq + kvh * G + h;
                const float2* ml = reinterpret_cast<const float2*>(p.ws_ml + hrow * p.max_splits * 2);
                float mm = -1e30f;
                for (int q = lane; q < ns; q += 32) mm = fmaxf(mm, __ldcg(ml + q).x);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) mm = fmaxf(mm, __shfl_xor_sync(kFull, mm, off));
                float L = 0.f;
                for (int q = lane; q < ns; q += 32) {
                    const float2 v = __ldcg(ml + q);
                    const float c = fast_exp2(v.x - mm);
                    wsm[h * ns + q] = c;
                    L += c * v.y;
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
                if (lane == 0) wsm[G * ns + h] = L;
            }
            __syncthreads();
            float acc[EPT];
#pragma unroll
            for (int i = 0; i < EPT; ++i) acc[i] = 0.f;
            for (int q0 = 0; q0 < ns; q0 += QB) {
                if (q0 > 0) load_o(q0);
#pragma unroll
                for (int u = 0; u < QB; ++u)
#pragma unroll
                    for (int i = 0; i < EPT; ++i) {
                        const int e = tid + i * kThreads, h = e / D;
                        if (q0 + u < ns && e < G * D) acc[i] += wsm[h * ns + q0 + u] * ov[u][i];
                    }
            }
#pragma unroll
            for (int i = 0; i < EPT; ++i) {
                const int e = tid + i * kThreads, h = e / D, dim = e % D;
                if (e >= G * D) continue;
                const float L = wsm[G * ns + h];
                reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t(b) * p.Hq + kvh * G + h) * D + dim] =
                    __float2bfloat16_rn(L > 0.f ? acc[i] / L : 0.f);
            }
        } else {
            // very many splits: one online pass per element
            for (int e = tid; e < G * D; e += kThreads) {
                const int h = e / D, dim = e % D;
                const size_t hrow = size_t(b) * p.Hq + kvh * G + h;
                const float2* ml = reinterpret_cast<const float2*>(p.ws_ml + hrow * p.max_splits * 2);
                const float* o = p.ws_o + hrow * p.max_splits * D + dim;
                float mm = -1e30f, L = 0.f, O = 0.f;
                for (int q = 0; q < ns; ++q) {
                    const float2 v = __ldcg(ml + q);
                    const float nm = fmaxf(mm, v.x);
                    const float c = fast_exp2(mm - nm), w = fast_exp2(v.x - nm);
                    L = L * c + w * v.y;
                    O = O * c + w * __ldcg(o + size_t(q) * D);
                    mm = nm;
                }
                reinterpret_cast<__nv_bfloat16*>(p.out)[hrow * D + dim] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
            }
        }
        if (tid == 0) *cnt = 0;  // ready for the next call
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
    pdl_launch_dependents();
    pdl_wait();
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
#pragma unroll 8
        for (int s = 0; s < ns; ++s) acc += cw[s] * o[size_t(s) * D + dim];
        reinterpret_cast<__nv_bfloat16*>(out)[hrow * D + dim] = __float2bfloat16_rn(acc * inv);
    }
}

}  // namespace pkv
