// Single-token paged decode attention over the quantized KV cache.
//
// "Accelerating Inference with FP8 KV Cache" (intro): the KV cache is stored in
// FP8 and computation runs in FP16; here every product is fp16 x fp16 and every
// sum fp32.  The FP8 per-tensor scale ("FP8 Formats: E4M3 and E5M2") and the
// INT8 / INT4 row scales ("[Feature] TurboMind support W8A8 or FP8 KV Cache",
// online INT8 and the INT4 named beside it) are folded out of the dot products:
// logits take s_K, outputs take s_V.  INT4 rows are head_dim / 2 bytes (two
// codes per byte) and use the tensor-core consumer only.
//
// Work decomposition.  Every (sequence, kv-head) pair owns ceil(ctx / 32)
// tiles of 32 tokens; all pairs' tiles, in (sequence, kv-head, tile) order,
// form one flat list.  A persistent grid (two CTAs per SM of six independent
// warps, eight for INT4) splits that list into equal contiguous ranges, one
// per warp, so every warp streams the same number of bytes whatever the context lengths.
// All q-heads of a kv-head's group are served by the warp that reads its tile,
// so each cached byte is read from HBM once.  Contexts are cut into chunks of
// C tiles; a warp range is never shorter than C, so a chunk is streamed by at
// most two warps and owns two partial slots (max, sum, unnormalised acc) that
// decode_reduce_kernel merges into the fp16 output.
//
// Every warp owns a ring of kSpw stages (a stage is a 32-token tile: two
// 16-row boxes of K and of V from paged blocks, 128-byte swizzled for head_dim
// 128, plus INT8 / INT4 scales), each with an mbarrier, and refills a stage
// with 2-D TMA tile loads (cp.async.bulk.tensor, issued by lane 0) right after
// consuming it, so its loads run the ring's length ahead across pair
// boundaries.  (More stages for the half-size INT4 tiles measured no faster:
// INT4 decode is not bound by the bytes in flight.)  Block ids of the 32
// boxes of the next 16 tiles are held one per lane (loaded one window ahead);
// the first tile of each (sequence, kv-head) pair also carries a bulk copy of
// the pair's query rows into the warp's query buffer.
//
// Two consumer families:
//   * kKindSimt: CUDA cores; 16 head-dim values per lane, mixed-precision
//     fma.rn.f32.f16 dot products and warp-shuffle reductions, group <= 4;
//   * kKindMma: tensor cores via mma.sync m16n8k16 (f16 in, fp32 accumulate).
//     QK^T is computed transposed (S^T = Q K^T with the q-group padded to 16
//     rows, 8 tokens per n8 tile) so that its accumulator fragment is already
//     the B operand of PV (out^T = V^T P^T, head_dim as M).  The contraction
//     index (head_dim for QK, tokens for PV) is permuted so that every thread
//     loads contiguous 16-byte runs; Q is permuted the same way.
// Every wait is bounded (2 s); on timeout a warp records the error, waits for
// its copies in flight and stops.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kvq_device.cuh"
#include "kvq_launch.h"

#ifndef KVQ_SPW
#define KVQ_SPW 2
#endif
#ifndef KVQ_MIN_BLOCKS
#define KVQ_MIN_BLOCKS 2
#endif
#ifndef KVQ_GA_WARPS
#define KVQ_GA_WARPS 4
#endif
#ifndef KVQ_GA4_WARPS
#define KVQ_GA4_WARPS 16
#endif
#ifndef KVQ_GA4_CTAS
#define KVQ_GA4_CTAS 1
#endif
#ifndef KVQ_INT4_WARPS
#define KVQ_INT4_WARPS 16
#endif
#ifndef KVQ_MMA_WARPS
#define KVQ_MMA_WARPS 6
#endif
#ifndef KVQ_R16_WARPS
#define KVQ_R16_WARPS 4
#endif

namespace kvq {
namespace {

constexpr int kTile = kDecodeTileTokens;       // tokens per stage: two boxes
constexpr int kBox = 16;                       // rows per TMA box (a 16-token slice of one paged block)
constexpr int kSpw = KVQ_SPW;                  // stages per warp
constexpr int kMinBlocks = KVQ_MIN_BLOCKS;     // CTAs per SM the registers are sized for
constexpr float kLog2e = 1.4426950408889634f;

enum { kKindSimt = 1, kKindMma = 2 };

// Shared-memory layout of one CTA (bytes from a 1024-aligned base).  Tiles
// first (1024-aligned for the 128-byte swizzle), then per warp its INT8 row
// scales, its stage barriers and (consumers that stage them: G > 0) the
// query rows of the (sequence, kv-head) pair it is on; when the launch
// appends the newest tokens, per warp the fp16
// K and V rows of the token that ends the pending pair and the block id its
// row goes to; then the scan of tiles per sequence and the clamped context
// lengths.
struct Layout {
    int tile_bytes, q_bytes, scales, full, qbuf, newkv, patch, scan, total;
    // rb: bytes of one cached row (head_dim, or head_dim / 2 for INT4); int8:
    // the format carries row scales (INT8 or INT4), ng of them per row
    // W: warps of the CTA
    __host__ __device__ Layout(int W, int rb, int D, int G, int B, bool int8, bool append, int ng) {
        tile_bytes = kTile * rb;
        q_bytes = (G * D * 2 + 127) / 128 * 128;
        scales = W * kSpw * 2 * tile_bytes;            // [warp][stage][K,V][tile] before this
        // INT8 / INT4: f32 [warp][stage][K,V][32 tokens][ng]
        full = scales + (int8 ? W * kSpw * 2 * kTile * 4 * ng : 0);
        qbuf = (full + W * kSpw * 8 + 127) / 128 * 128;  // u64 [warp][stage], then f16 [warp][G][D]
        newkv = qbuf + W * q_bytes;                    // f16 [warp][K,V][D]
        patch = newkv + (append ? W * 2 * D * 2 : 0);  // int [warp]
        scan = patch + (append ? W * 4 : 0);           // int S[B + 1], ctx[B]
        total = scan + (2 * B + 1) * 4;
    }
};

template <int D>
__device__ __forceinline__ int tile_off(int row, int chunk) {
    if (D == 128) return row * 128 + ((chunk ^ (row & 7)) << 4);
    return row * D + (chunk << 4);
}

// Position in the flat tile list: sequence b, kv-head kvh, tile t of n.
struct Walk {
    int b, kvh, t, n;
};

// S[b] = tiles of sequences 0..b-1 (S[B] = all); pair (b, kvh) covers flat
// tiles [Hkv*S[b] + kvh*n_b, ... + n_b).  f must be below Hkv * S[B]; the
// largest b with Hkv * S[b] <= f then has n_b > 0.
__device__ __forceinline__ Walk locate(const int* S, int B, int Hkv, int f) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (Hkv * S[mid] <= f) lo = mid; else hi = mid - 1;
    }
    Walk w;
    w.b = lo;
    w.n = S[lo + 1] - S[lo];
    const int r = f - Hkv * S[lo];
    w.kvh = r / w.n;
    w.t = r - w.kvh * w.n;
    return w;
}

__device__ __forceinline__ void advance(Walk& w, const int* S, int B, int Hkv) {
    if (++w.t < w.n) return;
    w.t = 0;
    if (++w.kvh < Hkv) return;
    w.kvh = 0;
    do {
        ++w.b;
    } while (w.b < B && S[w.b + 1] == S[w.b]);
    w.n = w.b < B ? S[w.b + 1] - S[w.b] : 0;
}

// One staged tile, by 32-bit shared-memory address: K codes, V codes, and
// (INT8) 16 K row scales followed by 16 V row scales.
struct Tile {
    uint32_t k, v, s;
    int valid;
};

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 r;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "r"(a));
    return r;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t r;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(r) : "r"(a));
    return r;
}
// Four 8x8 matrices of 16-bit elements: lane t gives the row address of row
// t % 8 of matrix t / 8; register m of lane t receives elements 2 (t % 4),
// 2 (t % 4) + 1 of row t / 4 of matrix m (here: bytes 4 (t % 4) .. + 3 of a
// 16-byte row segment).
__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ void ldsm_x2(uint32_t a, uint32_t (&r)[2]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(a));
}
// transposed: lane (g, c) gets 16-bit element g of rows 2c (low half) and 2c + 1 (high half)
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ float2 __uint_as_float2(uint2 v) { return make_float2(__uint_as_float(v.x), __uint_as_float(v.y)); }
__device__ __forceinline__ float ldsf(uint32_t a) {
    float r;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(r) : "r"(a));
    return r;
}

// Where a finished segment's state goes: partial slot (chunk, half) of the
// q-heads hq0 .. hq0 + G - 1; values are multiplied by s_out.
struct Flush {
    float* acc;
    float2* ml;
    int64_t hq0;
    int ch, half, nch;
    float s_out;
};

__device__ __forceinline__ int64_t slot_index(int64_t hq, int nch, int ch, int half) {
    return (hq * nch + ch) * 2 + half;
}

// ---------------------------------------------------------------- SIMT --

template <int FMT, int D, int GM>
struct SimtConsumer {
    static constexpr int LPT = D / 16;     // lanes per token
    static constexpr int TPP = 32 / LPT;   // tokens per pass
    static constexpr int PASSES = kBox / TPP;
    static constexpr int kMinCtas = GM == 4 ? 3 : kMinBlocks;  // 4 query rows need more registers
    static constexpr int kWarps = 6;
    static constexpr bool kQGlobal = false;   // query rows staged in shared memory
    uint32_t qh[GM][8];
    float m[GM], l[GM], acc[GM][16];
    int lane, j, grp, G, ng, gi;   // INT8: ng scales per row; this lane's 16 dims lie in group gi
    float qk_scale;

    __device__ void init(int G_, float qks, int ng_) {
        lane = threadIdx.x & 31;
        j = lane % LPT;
        grp = lane / LPT;
        G = G_;
        ng = ng_;
        gi = (16 * j) / (D / ng_);
        qk_scale = qks;
    }
    // q: the group's G query rows (shared-memory copy)
    __device__ void set_q(const uint16_t* q) {
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            if (h < G) {
                const uint4* src = reinterpret_cast<const uint4*>(q + h * D + 16 * j);
                const uint4 x0 = src[0], x1 = src[1];
                qh[h][0] = x0.x; qh[h][1] = x0.y; qh[h][2] = x0.z; qh[h][3] = x0.w;
                qh[h][4] = x1.x; qh[h][5] = x1.y; qh[h][6] = x1.z; qh[h][7] = x1.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) qh[h][e] = 0u;
            }
        }
    }
    __device__ void reset() {
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[h][e] = 0.f;
        }
    }

    // One 16-row half of a tile: K rows at k, V rows at v, INT8 scales at sk / sv
    // ([token][ng]: a lane's partial dot product and its weights take the
    // scale of the group its 16 dims lie in).
    __device__ void half(uint32_t k, uint32_t v, uint32_t sk, uint32_t sv, int valid) {
        float z[PASSES][GM];
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const int t = ps * TPP + grp;
            const uint4 kw = lds128(k + tile_off<D>(t, j));
            const uint32_t w[4] = {kw.x, kw.y, kw.z, kw.w};
            uint32_t kh[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kh[2 * e] = dec_x2<FMT>((uint16_t)(w[e] & 0xFFFFu));
                kh[2 * e + 1] = dec_x2<FMT>((uint16_t)(w[e] >> 16));
            }
            const float ks = FMT == INT8 ? ldsf(sk + 4 * (t * ng + gi)) : 1.0f;
#pragma unroll
            for (int h = 0; h < GM; ++h) {
                float d0 = 0.f, d1 = 0.f;
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    d0 = fma_f16x2_f32(qh[h][e], kh[e], d0);
                    d1 = fma_f16x2_f32(qh[h][e + 1], kh[e + 1], d1);
                }
                float d = (d0 + d1) * ks;
#pragma unroll
                for (int off = LPT / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, off);
                z[ps][h] = t < valid ? d * qk_scale : -INFINITY;
            }
        }
        float p[PASSES][GM];
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            float mx = z[0][h];
#pragma unroll
            for (int ps = 1; ps < PASSES; ++ps) mx = fmaxf(mx, z[ps][h]);
#pragma unroll
            for (int off = LPT; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
            const float mn = fmaxf(m[h], mx);
            float alpha = 1.f;
            if (mn == -INFINITY) {
#pragma unroll
                for (int ps = 0; ps < PASSES; ++ps) p[ps][h] = 0.f;
            } else {
                alpha = fast_exp2(m[h] - mn);
#pragma unroll
                for (int ps = 0; ps < PASSES; ++ps) p[ps][h] = fast_exp2(z[ps][h] - mn);
            }
            m[h] = mn;
            float ps_sum = 0.f;
#pragma unroll
            for (int ps = 0; ps < PASSES; ++ps) ps_sum += p[ps][h];
            l[h] = l[h] * alpha + ps_sum;
            if (alpha != 1.f) {
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[h][e] *= alpha;
            }
        }
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const int t = ps * TPP + grp;
            uint4 vw = lds128(v + tile_off<D>(t, j));
            // rows past the context may hold any bytes (NaN codes too): zero them
            if (t >= valid) vw = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[4] = {vw.x, vw.y, vw.z, vw.w};
            const float vs = (FMT == INT8 && t < valid) ? ldsf(sv + 4 * (t * ng + gi)) : 1.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 lo = f16x2_to_f32x2(dec_x2<FMT>((uint16_t)(w[e] & 0xFFFFu)));
                const float2 hi = f16x2_to_f32x2(dec_x2<FMT>((uint16_t)(w[e] >> 16)));
#pragma unroll
                for (int h = 0; h < GM; ++h) {
                    const float pp = p[ps][h] * vs;
                    acc[h][4 * e] = fmaf(pp, lo.x, acc[h][4 * e]);
                    acc[h][4 * e + 1] = fmaf(pp, lo.y, acc[h][4 * e + 1]);
                    acc[h][4 * e + 2] = fmaf(pp, hi.x, acc[h][4 * e + 2]);
                    acc[h][4 * e + 3] = fmaf(pp, hi.y, acc[h][4 * e + 3]);
                }
            }
        }
    }

    __device__ void tile(const Tile& c) {
        const uint32_t sv = c.s + 4 * kTile * ng;
        half(c.k, c.v, c.s, sv, c.valid);
        if (c.valid > kBox)
            half(c.k + kBox * D, c.v + kBox * D, c.s + 4 * kBox * ng, sv + 4 * kBox * ng, c.valid - kBox);
    }

    // Sum the per-group partials and write this segment's partial slot.
    __device__ void flush(const Flush& f) {
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            float lh = l[h];
            float a[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) a[e] = acc[h][e];
#pragma unroll
            for (int off = LPT; off < 32; off <<= 1) {
                lh += __shfl_xor_sync(0xFFFFFFFFu, lh, off);
#pragma unroll
                for (int e = 0; e < 16; ++e) a[e] += __shfl_xor_sync(0xFFFFFFFFu, a[e], off);
            }
            if (h < G && grp == 0) {
                const int64_t si = slot_index(f.hq0 + h, f.nch, f.ch, f.half);
                float* dst = f.acc + si * D + 16 * j;
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4*>(dst + e) =
                        make_float4(a[e] * f.s_out, a[e + 1] * f.s_out, a[e + 2] * f.s_out, a[e + 3] * f.s_out);
                if (j == 0) f.ml[si] = make_float2(m[h], lh);
            }
        }
    }
    __device__ void flush_empty(const Flush& f) {
        if (lane < G) f.ml[slot_index(f.hq0 + lane, f.nch, f.ch, f.half)] = make_float2(-INFINITY, 0.f);
    }
};

// ----------------------------------------------------------------- MMA --

template <int FMT, int D, bool R16 = false, bool WIDE = false>
struct MmaConsumer {
    static constexpr bool I4 = FMT == INT4;
    static constexpr bool kRowScaled = FMT == INT8 || FMT == INT4;
    static constexpr int RB = row_bytes(FMT, D);  // bytes of one cached row
    static constexpr int KS = D / 16;   // k-steps of QK^T
    static constexpr int DC = D / 4;    // K codes per thread per token row
    static constexpr int KW = I4 ? DC / 8 : DC / 4;   // ... as 32-bit words (== KS for 8-bit codes)
    static constexpr int DV = D / 8;    // V codes per thread per token row
    static constexpr int VW = DV / 4;   // ... as 32-bit words (8-bit codes; INT4 V is read by ldmatrix.trans)
    static constexpr int MT = D / 16;   // m-tiles of PV (head_dim / 16)
    // Operand rows (q-head, scale group pairs) per pass: 8, or 16 with R16.
    // QK^T's m16 tile has 16 rows; the 8-row consumer fills rows 0-7 (this
    // thread's row g) and leaves rows 8-15 zero, the 16-row one also fills
    // rows 8-15 (row g + 8) and takes a second n8 tile of PV columns.  The
    // 16-row consumer serves INT4 caches with 16-channel groups (head_dim 64)
    // whose q-heads x groups per kv-head exceed 8, so that one pass over the
    // cache serves twice the pairs (the grouped consumer below takes the other
    // grouped caches); it holds twice the accumulators, so it runs 4 warps per
    // CTA with up to 255 registers.
    static constexpr int NR = R16 ? 2 : 1;
    static constexpr int kRows = 8 * NR;
    // Warps per CTA, each streaming its own range.  INT4 tiles are half the
    // bytes of the others, and the kernel is bound by the latency of the
    // per-warp register work rather than by HBM: 16 warps per SM (registers
    // capped at 128) are 11% faster than 12, and as one CTA of 16 warps 2%
    // faster than as two of 8 (the warp schedulers favour the older of two
    // CTAs, whose warps then finish their equal ranges ~10% earlier and leave
    // the SM half occupied).  The 8-bit formats stay at two CTAs of 6: their
    // stages fill shared memory, and at 12 warps per CTA a large batch of
    // 8-head groups would not fit.
    static constexpr int kMinCtas = ((I4 && !R16) || WIDE) ? 1 : kMinBlocks;
    // WIDE: the 8-bit formats' 12 warps as one CTA per SM (8-head groups, when
    // the stages fit: +0.7% on the Llama-3-70B batch; neutral to -0.3% for
    // the smaller groups, which keep two CTAs)
    static constexpr int kWarps = R16 ? KVQ_R16_WARPS : (I4 ? KVQ_INT4_WARPS : (WIDE ? 2 * KVQ_MMA_WARPS : KVQ_MMA_WARPS));
    // INT8 / INT4 read a pair's query rows from global memory when it starts
    // (set_q), FP8 has them staged in shared memory with the pair's first
    // tile: the global reads measured +2% on the Llama-2-13B INT8 and INT4
    // shapes and -0.4% on FP8's (same box)
    static constexpr bool kQGlobal = kRowScaled;
    // INT8 codes enter the tensor cores as fp16 subnormals, code * 2^-24, and
    // INT4 codes the same, or 16x that where the nibble is left in mantissa
    // bits 4..7 -- the high nibble of a byte is masked in place, which saves
    // the shifts and byte moves of a full expansion.  The matching query
    // values are fed divided by 16 (QK), and the output rows of such head dims
    // are divided by 16 at the flush (PV); results are multiplied back by 2^24.
    //   K (QK): the offset code + 128 (INT8) or code + 8 (INT4) is the
    //   mantissa as loaded, and bias * sum(q) is taken out of each logit.  A
    //   logit depends only on its own token, so this rounding does not depend
    //   on how a context is split.
    //   V (PV): one exact fp16 subtraction per operand register removes the
    //   offset before the product, so the accumulators hold unbiased sums.  An
    //   offset left in them, drained by bias * sum(P') later, made their fp32
    //   rounding relative to the biased sums: INT8 rows holding a x20 outlier
    //   channel (row scales ~19x the Gaussian rows') reached 6.6e-3 relative
    //   error over 4096-token chunks with 1152 + code operands, and even with
    //   a small offset drained every four tiles the result still moved by 4e-5
    //   with the context split (INT4 outlier rows: scales ~8.6).
    static constexpr bool kBiased = kRowScaled;
    static constexpr float kUnit = 5.9604644775390625e-08f;           // operand value of one code step (2^-24)
    static constexpr float kBias = (I4 ? 8.f : 128.f) * kUnit;        // K operand - code * kUnit
    // INT8 / INT4 weights enter PV as P' times the token's V scale, in fp16
    // (hi + residual).  INT8 row scales of Gaussian rows are ~0.025, which
    // would put most weights below fp16's normal range (6.1e-5), where hi and
    // residual keep only an absolute 2^-25: 2e-5 relative error over 4096
    // tokens.  The weights are therefore computed as 2^kLogF * 2^(z - m): the
    // running sum l and the accumulators carry the same factor, which cancels
    // when the partials are merged (out = acc / l).
    // 2^6 (INT8) and 2^2 (INT4) keep every weight of any fp16 row (scale at most
    // 65504 / 127, or / 7) below fp16's largest value.
    static constexpr float kLogF = FMT == INT8 ? 6.f : (I4 ? 2.f : 0.f);
    // Operand row / column r (QK rows, PV columns) is (q-head r / ng, scale
    // group r % ng): with ng groups per row, a row of QK sees only its group's
    // head dims, its partial logits are scaled by that group's K scales and
    // summed over the ng rows of the head, and the PV column carries P times
    // the group's V scales; output dims are taken from the column of their own
    // group.  ng = 1 is the per-row (or per-tensor) format.  A thread holds
    // rows g and (R16) g + 8, which share their scale group (ng divides 8).
    uint32_t qa[NR][2 * KS];
    float acc[NR][MT][4];
    float m[NR], l[NR];
    float qsum[NR];  // INT8 / INT4: sum of this operand row's query values (rows g, g + 8)
    int lane, g, c, G, ng, kg;  // kg = g % ng: this lane's scale group
    // INT8 / INT4 with at most 4 operand rows (q-head, group pairs): PV
    // columns 0-3 carry the weights' fp16 high parts and columns 4-7 their
    // residuals, so one MMA does both products; the flush adds column n + 4 to
    // column n (1.4-1.8% faster).  With more rows every column is a row's own
    // and PV takes two MMAs per m-tile.  FP8 keeps the two MMAs: the extra
    // shuffles on the way to PV cost its HBM-bound stream 2%.
    bool lo_cols;
    float qk_scale;
    // this lane's byte offsets inside a stage tile (the 128-byte swizzle folded
    // in): K row g at chunks 2c, 2c+1 (row 8+g is 8 rows further), V rows 2c
    // and 2c+1 at chunk g (rows 8+2c, 9+2c are 8 rows further).  INT4 rows
    // hold the codes at half the bytes (64-byte swizzle at head_dim 128): K row
    // g at chunk c, and v_off0 / v_off1 are this lane's row addresses for the
    // two ldmatrix.trans of a box's V
    uint32_t k_off0, k_off1, v_off0, v_off1;

    __device__ void init(int G_, float qks, int ng_) {
        lane = threadIdx.x & 31;
        g = lane >> 2;
        c = lane & 3;
        G = G_;
        ng = ng_;
        kg = g % ng_;
        lo_cols = !R16 && kRowScaled && G_ * ng_ <= 4;
        qk_scale = qks;
        if (I4) {
            // 64-byte rows (head_dim 128): 64-byte swizzle, 16-byte chunk ^= (row / 2) % 4;
            // 32-byte rows plain.  V: row addresses of ldmatrix.trans x (v_off0, v_off1):
            // lane t gives row 8 ((t >> 3) & 1) + t % 8 of chunk 2x + t / 16
            const int vr = 8 * ((lane >> 3) & 1) + (lane & 7), vc = lane >> 4;
            if (D == 128) {
                k_off0 = g * RB + ((c ^ ((g >> 1) & 3)) << 4);
                v_off0 = vr * RB + ((vc ^ ((vr >> 1) & 3)) << 4);
                v_off1 = vr * RB + (((2 + vc) ^ ((vr >> 1) & 3)) << 4);
            } else {
                k_off0 = g * RB + c * (DC / 2);
                v_off0 = vr * RB + 16 * vc;
                v_off1 = 0;
            }
            k_off1 = 0;
        } else if (D == 128) {
            k_off0 = g * 128 + (((2 * c) ^ g) << 4);
            k_off1 = g * 128 + (((2 * c + 1) ^ g) << 4);
            v_off0 = (2 * c) * 128 + ((g ^ (2 * c)) << 4);
            v_off1 = (2 * c + 1) * 128 + ((g ^ (2 * c + 1)) << 4);
        } else {
            k_off0 = g * D + c * 16;
            k_off1 = 0;
            v_off0 = (2 * c) * D + DV * g;
            v_off1 = (2 * c + 1) * D + DV * g;
        }
    }
    // qa[r][2j] = Q[h][DC*c + 4j + {0,1}], qa[r][2j+1] = Q[h][DC*c + 4j + {2,3}]:
    // the DC halves Q[h][DC*c ...] in order, for operand row g (r = 0) or g + 8
    // (r = 1) with h = row / ng, where this thread's DC dims lie in the row's
    // scale group (the DC dims of a thread are within one group: groups are
    // D / ng >= DC wide); else zero.  q: the kv-head's G query rows
    // (shared-memory copy).
    __device__ void set_q(const uint16_t* q) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const int row = g + 8 * r;
            if (row < G * ng && ((c * ng) >> 2) == kg) {
                const uint4* src = reinterpret_cast<const uint4*>(q + (row / ng) * D + DC * c);
#pragma unroll
                for (int i = 0; i < (2 * KS) / 4; ++i) {
                    const uint4 x = src[i];
                    qa[r][4 * i] = x.x; qa[r][4 * i + 1] = x.y; qa[r][4 * i + 2] = x.z; qa[r][4 * i + 3] = x.w;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 2 * KS; ++i) qa[r][i] = 0u;
            }
            if (I4) {  // per 8 dims: [q0, q5/16] [q1/16, q4] [q2, q7/16] [q3/16, q6], the K operand order
#pragma unroll
                for (int w = 0; w < KW; ++w) {
                    const float2 q01 = f16x2_to_f32x2(qa[r][4 * w]), q23 = f16x2_to_f32x2(qa[r][4 * w + 1]);
                    const float2 q45 = f16x2_to_f32x2(qa[r][4 * w + 2]), q67 = f16x2_to_f32x2(qa[r][4 * w + 3]);
                    qa[r][4 * w] = pack_f16x2(q01.x, q45.y * 0.0625f);
                    qa[r][4 * w + 1] = pack_f16x2(q01.y * 0.0625f, q45.x);
                    qa[r][4 * w + 2] = pack_f16x2(q23.x, q67.y * 0.0625f);
                    qa[r][4 * w + 3] = pack_f16x2(q23.y * 0.0625f, q67.x);
                }
            }
            if (kBiased) {  // sum of q as fed times each operand's step (16 for the divided values)
                float sq = 0.f;
#pragma unroll
                for (int i = 0; i < 2 * KS; ++i) {
                    const float2 v = f16x2_to_f32x2(qa[r][i]);
                    sq += I4 ? ((i & 1) ? 16.f * v.x + v.y : v.x + 16.f * v.y) : v.x + v.y;
                }
                sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 1);
                sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 2);
                qsum[r] = sq;
            }
        }
    }
    // INT8 word (4 codes) -> the two f16x2 operands (code + 128) * 2^-24 of bytes (0,1) and (2,3)
    __device__ __forceinline__ static void int8_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
        const uint32_t x = w ^ 0x80808080u;  // code + 128 as an unsigned byte
        lo = prmt(x, 0u, 0x4140u);
        hi = prmt(x, 0u, 0x4342u);
    }
    __device__ void reset() {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
#pragma unroll
            for (int i = 0; i < MT; ++i) acc[r][i][0] = acc[r][i][1] = acc[r][i][2] = acc[r][i][3] = 0.f;
        }
    }

    // K words of rows g (half 0) or 8 + g (half 1): the DC contiguous codes at DC*c.
    __device__ __forceinline__ void load_k(uint32_t kt, int half, uint32_t (&w)[KW]) {
        const uint32_t rb = kt + half * 8 * RB;
        if (I4) {
            if (D == 128) {
                const uint4 x0 = lds128(rb + k_off0);
                w[0] = x0.x; w[1] = x0.y; w[KW > 2 ? 2 : 0] = x0.z; w[KW > 3 ? 3 : 1] = x0.w;
            } else {
                const uint2 x0 = lds64(rb + k_off0);
                w[0] = x0.x; w[KW > 1 ? 1 : 0] = x0.y;
            }
        } else if (D == 128) {
            const uint4 x0 = lds128(rb + k_off0), x1 = lds128(rb + k_off1);
            w[0] = x0.x; w[1] = x0.y; w[2] = x0.z; w[3] = x0.w;
            w[4] = x1.x; w[5] = x1.y; w[6] = x1.z; w[7] = x1.w;
        } else {
            const uint4 x0 = lds128(rb + k_off0);
            w[0] = x0.x; w[1] = x0.y; w[2] = x0.z; w[3] = x0.w;
        }
    }

    // V words of a row: the thread's DV contiguous codes at DV*g.
    __device__ __forceinline__ void load_v(uint32_t a, uint32_t (&w)[VW]) {
        if (D == 128) {
            const uint4 x = lds128(a);
            w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        } else {
            const uint2 x = lds64(a);
            w[0] = x.x; w[1] = x.y;
        }
    }

    // One QK^T product of the 16-row operand: rows g (and g + 8 with R16).
    __device__ __forceinline__ void qk_mma(float (&s)[4], int i0, int i1, uint32_t b0, uint32_t b1) {
        if (R16) mma_16816(s, qa[0][i0], qa[NR - 1][i0], qa[0][i1], qa[NR - 1][i1], b0, b1);
        else mma_16816(s, qa[0][i0], 0u, qa[0][i1], 0u, b0, b1);
    }

    // QK^T of one 16-row box: this thread's logits of operand rows g (z[0]) and
    // g + 8 (z[1], R16), box tokens 2c, 2c+1, 8+2c, 9+2c (already scaled,
    // masked past `valid`).
    __device__ __forceinline__ void qk_box(uint32_t kt, uint32_t sk, int valid, float (&z)[NR][4]) {
        // S^T: rows = operand rows (g, g + 8), columns = tokens; half A = box
        // tokens 0..7 (this thread's B operand row is token g), half B = tokens 8..15.
        float sA[4] = {0.f, 0.f, 0.f, 0.f}, sB[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t kw[KW];
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            load_k(kt, hb, kw);
            if (I4) {  // word w: codes 8w .. 8w+7 = k-steps 2w and 2w+1
#pragma unroll
                for (int w = 0; w < KW; ++w) {
                    // byte i holds dims 2i (low nibble) and 2i+1 (high); bit 3 of every
                    // nibble flipped (code + 8), then masked in place:
                    // h0 = [d0, 16 d5], h1 = [16 d1, d4], h2 = [d2, 16 d7], h3 = [16 d3, d6].
                    // (One flip per word and single-constant masks: a mask and a flip per
                    // operand, two constants each, ran 12% more instructions per tile.)
                    const uint32_t x = kw[w] ^ 0x88888888u, y = x >> 8;
                    const uint32_t h0 = x & 0x00F0000Fu, h1 = x & 0x000F00F0u;
                    const uint32_t h2 = y & 0x00F0000Fu, h3 = y & 0x000F00F0u;
                    if (hb == 0) {
                        qk_mma(sA, 4 * w, 4 * w + 1, h0, h1);
                        qk_mma(sA, 4 * w + 2, 4 * w + 3, h2, h3);
                    } else {
                        qk_mma(sB, 4 * w, 4 * w + 1, h0, h1);
                        qk_mma(sB, 4 * w + 2, 4 * w + 3, h2, h3);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < KS; ++j) {
                    uint32_t b0, b1;
                    if (FMT == INT8) int8_biased(kw[j < KW ? j : 0], b0, b1);
                    else dec_fp8x4<FMT>(kw[j < KW ? j : 0], b0, b1);
                    if (hb == 0) qk_mma(sA, 2 * j, 2 * j + 1, b0, b1);
                    else qk_mma(sB, 2 * j, 2 * j + 1, b0, b1);
                }
            }
        }
        if (kRowScaled) {  // remove the operand bias, then apply the K row (group) scales
            const float ks = qk_scale / kUnit;
            float2 k01, k23;
            if (ng == 1) {
                k01 = __uint_as_float2(lds64(sk + 8 * c));
                k23 = __uint_as_float2(lds64(sk + 32 + 8 * c));
            } else {  // scales [token][ng]: tokens 2c, 2c+1, 8+2c, 9+2c of group kg
                const uint32_t a0 = sk + 4 * (2 * c * ng + kg);
                k01 = make_float2(ldsf(a0), ldsf(a0 + 4 * ng));
                k23 = make_float2(ldsf(a0 + 32 * ng), ldsf(a0 + 36 * ng));
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float corr = kBias * qsum[r];
                z[r][0] = (sA[2 * r] - corr) * (ks * k01.x);
                z[r][1] = (sA[2 * r + 1] - corr) * (ks * k01.y);
                z[r][2] = (sB[2 * r] - corr) * (ks * k23.x);
                z[r][3] = (sB[2 * r + 1] - corr) * (ks * k23.y);
                // the head's logits: sum of its ng group rows (lanes 4 apart per row)
                for (int off = 1; off < ng; off <<= 1) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) z[r][e] += __shfl_xor_sync(0xFFFFFFFFu, z[r][e], 4 * off);
                }
            }
        } else {
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                z[r][0] = sA[2 * r] * qk_scale; z[r][1] = sA[2 * r + 1] * qk_scale;
                z[r][2] = sB[2 * r] * qk_scale; z[r][3] = sB[2 * r + 1] * qk_scale;
            }
        }
        if (valid < kBox) {
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (2 * c >= valid) z[r][0] = -INFINITY;
                if (2 * c + 1 >= valid) z[r][1] = -INFINITY;
                if (8 + 2 * c >= valid) z[r][2] = -INFINITY;
                if (9 + 2 * c >= valid) z[r][3] = -INFINITY;
            }
        }
    }

    // out^T += V^T P^T for one box.  A operand rows = head_dim DV*g + 2i (+1
    // for rows g+8), columns = box tokens 2c, 2c+1 | 8+2c, 9+2c.
    // LO: the residual weights ride in columns 4-7 of pb[0]; else they are
    // pl[0], a second MMA per m-tile.  R16: pb[1] / pl[1] are the weights of
    // operand columns 8-15 (the second accumulator).
    template <bool LO>
    __device__ __forceinline__ void pv_box(uint32_t vt, int valid, const uint32_t (&pb)[NR][2],
                                           const uint32_t (&pl)[NR][2]) {
        if constexpr (I4) {
            // ldmatrix.trans: r[x][0] / r[x][2] = bytes 2g, 2g + 1 of 16-byte chunk 2x / 2x + 1 of
            // tokens 2c (bits 0-15) and 2c + 1 (bits 16-31); r[x][1] / r[x][3] tokens 8 + 2c, 9 + 2c
            constexpr int NCH = RB / 16;
            uint32_t r[NCH / 2][4];
            ldsm_x4_t(vt + v_off0, r[0]);
            if constexpr (NCH == 4) ldsm_x4_t(vt + v_off1, r[NCH / 2 - 1]);
            if (valid < kBox) {  // rows past the context may hold NaN codes: zero them
                const uint32_t mlo = (2 * c < valid ? 0x0000FFFFu : 0u) | (2 * c + 1 < valid ? 0xFFFF0000u : 0u);
                const uint32_t mhi = (8 + 2 * c < valid ? 0x0000FFFFu : 0u) | (9 + 2 * c < valid ? 0xFFFF0000u : 0u);
#pragma unroll
                for (int x = 0; x < NCH / 2; ++x) {
                    r[x][0] &= mlo; r[x][1] &= mhi; r[x][2] &= mlo; r[x][3] &= mhi;
                }
            }
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) {
                // code + 8 in every nibble (a zeroed token becomes 8 - 8 = 0)
                const uint32_t lo = r[ch >> 1][2 * (ch & 1)] ^ 0x88888888u, hi = r[ch >> 1][2 * (ch & 1) + 1] ^ 0x88888888u;
#pragma unroll
                for (int bb = 0; bb < 2; ++bb) {
                    // m-tile 2 ch + bb: dim 32 ch + 4g + 2bb (low nibble, rows g) and + 1 (the high
                    // nibble in place: 16x, rows g + 8), less the offsets (8 and 16 * 8 steps, exact)
                    const uint32_t u = bb ? lo >> 8 : lo, w = bb ? hi >> 8 : hi;
                    const uint32_t a0 = hsub2_exact(u & 0x000F000Fu, 0x00080008u);
                    const uint32_t a1 = hsub2_exact(u & 0x00F000F0u, 0x00800080u);
                    const uint32_t a2 = hsub2_exact(w & 0x000F000Fu, 0x00080008u);
                    const uint32_t a3 = hsub2_exact(w & 0x00F000F0u, 0x00800080u);
#pragma unroll
                    for (int rr = 0; rr < NR; ++rr) {
                        mma_16816(acc[rr][2 * ch + bb], a0, a1, a2, a3, pb[rr][0], pb[rr][1]);
                        if (!LO) mma_16816(acc[rr][2 * ch + bb], a0, a1, a2, a3, pl[rr][0], pl[rr][1]);
                    }
                }
            }
            return;
        }
        uint32_t v0[VW], v1[VW], v2[VW], v3[VW];
        load_v(vt + v_off0, v0);
        load_v(vt + v_off1, v1);
        load_v(vt + v_off0 + 8 * RB, v2);
        load_v(vt + v_off1 + 8 * RB, v3);
        if (valid < kBox) {  // rows past the context may hold NaN codes: zero them
#pragma unroll
            for (int e = 0; e < VW; ++e) {
                if (2 * c >= valid) v0[e] = 0u;
                if (2 * c + 1 >= valid) v1[e] = 0u;
                if (8 + 2 * c >= valid) v2[e] = 0u;
                if (9 + 2 * c >= valid) v3[e] = 0u;
            }
        }
        if (FMT == INT8) {  // code + 128 as unsigned bytes, once per word
#pragma unroll
            for (int e = 0; e < VW; ++e) {
                v0[e] ^= 0x80808080u; v1[e] ^= 0x80808080u; v2[e] ^= 0x80808080u; v3[e] ^= 0x80808080u;
            }
        }
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
            const uint32_t x01 = prmt(v0[i >> 1], v1[i >> 1], sel);
            const uint32_t x23 = prmt(v2[i >> 1], v3[i >> 1], sel);
            uint32_t a0, a1, a2, a3;
            if (FMT == INT8) {  // fp16 subnormals (code + 128) * 2^-24, less 128 * 2^-24 (exact)
                a0 = hsub2_exact(prmt(x01, 0u, 0x4140u), 0x00800080u);
                a1 = hsub2_exact(prmt(x01, 0u, 0x4342u), 0x00800080u);
                a2 = hsub2_exact(prmt(x23, 0u, 0x4140u), 0x00800080u);
                a3 = hsub2_exact(prmt(x23, 0u, 0x4342u), 0x00800080u);
            } else {
                dec_fp8x4<FMT>(x01, a0, a1);
                dec_fp8x4<FMT>(x23, a2, a3);
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                mma_16816(acc[r][i], a0, a1, a2, a3, pb[r][0], pb[r][1]);
                if (!LO) mma_16816(acc[r][i], a0, a1, a2, a3, pl[r][0], pl[r][1]);
            }
        }
    }

    // P of one box as the B operand of PV (k = token, n = operand row g), as
    // an fp16 pair hi + lo (lo = the fp16 residual of p - hi): the PV product
    // keeps about 22 bits of each weight instead of 11.  With outlier channels
    // the weighted mean of large V values can cancel, and a single fp16
    // rounding of P would then show in the output.
    __device__ __forceinline__ void p_frags(const float (&p)[4], uint32_t& pb0, uint32_t& pb1, uint32_t& pl0,
                                            uint32_t& pl1) {
        pb0 = pack_f16x2(p[0], p[1]);
        pb1 = pack_f16x2(p[2], p[3]);
        const float2 h01 = f16x2_to_f32x2(pb0), h23 = f16x2_to_f32x2(pb1);
        pl0 = pack_f16x2(p[0] - h01.x, p[1] - h01.y);
        pl1 = pack_f16x2(p[2] - h23.x, p[3] - h23.y);
    }

    __device__ void tile(const Tile& cx) {
        // The second box is always computed, also when it lies past the context
        // (its logits masked, its V codes zeroed and its weights 0, whatever the
        // stage holds), so that the two boxes' products can overlap: 1-3% faster
        // than skipping it on the last tile of a pair.
        float z0[NR][4], z1[NR][4];
        qk_box(cx.k, cx.s, cx.valid, z0);
        qk_box(cx.k + kBox * RB, cx.s + 4 * kBox * ng, cx.valid - kBox, z1);
        float alpha[NR], p0[NR][4], p1[NR][4];
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            float mx = fmaxf(fmaxf(fmaxf(z0[r][0], z0[r][1]), fmaxf(z0[r][2], z0[r][3])),
                             fmaxf(fmaxf(z1[r][0], z1[r][1]), fmaxf(z1[r][2], z1[r][3])));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
            const float mn = fmaxf(m[r], mx);
            alpha[r] = 1.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) p0[r][e] = p1[r][e] = 0.f;
            if (mn != -INFINITY) {
                alpha[r] = fast_exp2(m[r] - mn);
                const float mb = mn - kLogF;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    p0[r][e] = fast_exp2(z0[r][e] - mb);
                    p1[r][e] = fast_exp2(z1[r][e] - mb);
                }
            }
            m[r] = mn;
            l[r] = l[r] * alpha[r] + (((p0[r][0] + p0[r][1]) + (p0[r][2] + p0[r][3])) +
                                      ((p1[r][0] + p1[r][1]) + (p1[r][2] + p1[r][3])));
        }
        if (kRowScaled) {  // fold the V row (column group) scales into P; rows g and g + 8 share a group
            const uint32_t sv = cx.s + 4 * kTile * ng;
            float a[4], b[4];
            if (ng == 1) {
                const float2 a01 = __uint_as_float2(lds64(sv + 8 * c)), a23 = __uint_as_float2(lds64(sv + 32 + 8 * c));
                const float2 b01 = __uint_as_float2(lds64(sv + 64 + 8 * c)), b23 = __uint_as_float2(lds64(sv + 96 + 8 * c));
                a[0] = a01.x; a[1] = a01.y; a[2] = a23.x; a[3] = a23.y;
                b[0] = b01.x; b[1] = b01.y; b[2] = b23.x; b[3] = b23.y;
            } else {  // scales [token][ng]: tokens 2c, 2c+1, 8+2c, 9+2c (+16) of group kg
                const uint32_t a0 = sv + 4 * (2 * c * ng + kg), b0 = a0 + 64 * ng;
                a[0] = ldsf(a0); a[1] = ldsf(a0 + 4 * ng); a[2] = ldsf(a0 + 32 * ng); a[3] = ldsf(a0 + 36 * ng);
                b[0] = ldsf(b0); b[1] = ldsf(b0 + 4 * ng); b[2] = ldsf(b0 + 32 * ng); b[3] = ldsf(b0 + 36 * ng);
            }
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                if (cx.valid >= kTile) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        p0[r][e] *= a[e];
                        p1[r][e] *= b[e];
                    }
                } else {  // a masked token keeps p = 0 whatever its (never written) scale slot holds
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        p0[r][e] = p0[r][e] != 0.f ? p0[r][e] * a[e] : 0.f;
                        p1[r][e] = p1[r][e] != 0.f ? p1[r][e] * b[e] : 0.f;
                    }
                }
            }
        }
        // rescale the accumulators: columns 2c and 2c+1 are operand rows 2c and
        // 2c+1 (rows (2c and 2c+1) mod 4 when the residuals use columns 4-7);
        // the second accumulator's columns are rows 8 + 2c and 9 + 2c
        bool any = alpha[0] != 1.f;
        if (R16) any = any || alpha[NR - 1] != 1.f;
        if (__any_sync(0xFFFFFFFFu, any)) {
            const int src = 8 * ((kRowScaled && lo_cols) ? (c & 1) : c);
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float a0 = __shfl_sync(0xFFFFFFFFu, alpha[r], src);
                const float a1 = __shfl_sync(0xFFFFFFFFu, alpha[r], src + 4);
#pragma unroll
                for (int i = 0; i < MT; ++i) {
                    acc[r][i][0] *= a0; acc[r][i][1] *= a1; acc[r][i][2] *= a0; acc[r][i][3] *= a1;
                }
            }
        }
        uint32_t pb[NR][2], pl[NR][2];
        if (kRowScaled && lo_cols) {  // lanes of rows 4-7 feed the residuals of rows 0-3 (16 lanes below)
            p_frags(p0[0], pb[0][0], pb[0][1], pl[0][0], pl[0][1]);
            pl[0][0] = __shfl_xor_sync(0xFFFFFFFFu, pl[0][0], 16);
            pl[0][1] = __shfl_xor_sync(0xFFFFFFFFu, pl[0][1], 16);
            if (g >= 4) { pb[0][0] = pl[0][0]; pb[0][1] = pl[0][1]; }
            pv_box<true>(cx.v, cx.valid, pb, pl);
            p_frags(p1[0], pb[0][0], pb[0][1], pl[0][0], pl[0][1]);
            pl[0][0] = __shfl_xor_sync(0xFFFFFFFFu, pl[0][0], 16);
            pl[0][1] = __shfl_xor_sync(0xFFFFFFFFu, pl[0][1], 16);
            if (g >= 4) { pb[0][0] = pl[0][0]; pb[0][1] = pl[0][1]; }
            pv_box<true>(cx.v + kBox * RB, cx.valid - kBox, pb, pl);
        } else {
#pragma unroll
            for (int r = 0; r < NR; ++r) p_frags(p0[r], pb[r][0], pb[r][1], pl[r][0], pl[r][1]);
            pv_box<false>(cx.v, cx.valid, pb, pl);
#pragma unroll
            for (int r = 0; r < NR; ++r) p_frags(p1[r], pb[r][0], pb[r][1], pl[r][0], pl[r][1]);
            pv_box<false>(cx.v + kBox * RB, cx.valid - kBox, pb, pl);
        }
    }

    __device__ void flush(const Flush& f) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            float lq = l[r];
            lq += __shfl_xor_sync(0xFFFFFFFFu, lq, 1);
            lq += __shfl_xor_sync(0xFFFFFFFFu, lq, 2);
            const int row = g + 8 * r;
            if (c == 0 && kg == 0 && row < G * ng)
                f.ml[slot_index(f.hq0 + row / ng, f.nch, f.ch, f.half)] = make_float2(m[r], lq);
        }
        if (kRowScaled && lo_cols) {  // column n += column n + 4 (lanes c and c + 2)
#pragma unroll
            for (int i = 0; i < MT; ++i)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[0][i][e] += __shfl_xor_sync(0xFFFFFFFFu, acc[0][i][e], 2);
        }
        if constexpr (I4) {
            // acc[r][2 ch + bb][e | 2 + e] = out[column 8r + 2c + e][d = 32 ch + 4g + 2bb | + 1];
            // column n is head n / ng with the V scales of group n % ng, which must
            // be the group of the chunk's dims 32 ch + 4g .. + 3; the odd dims were
            // fed as 16x operands
            constexpr int NCH = RB / 16;
            const float so = f.s_out / kUnit, so1 = so * 0.0625f;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int n = 8 * r + 2 * c + e, h = n / ng;
                    if (h >= G) continue;
                    float* dst = f.acc + slot_index(f.hq0 + h, f.nch, f.ch, f.half) * D + 4 * g;
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch) {
                        if (n % ng != ((32 * ch + 4 * g) * ng) / D) continue;
                        *reinterpret_cast<float4*>(dst + 32 * ch) =
                            make_float4(acc[r][2 * ch][e] * so, acc[r][2 * ch][2 + e] * so1,
                                        acc[r][2 * ch + 1][e] * so, acc[r][2 * ch + 1][2 + e] * so1);
                    }
                }
            }
            return;
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            // acc[r][i][0..3] = out[column 8r + 2c | 8r + 2c+1][d = DV*g + 2i | DV*g + 2i + 1];
            // column n is head n / ng with the V scales of group n % ng, which must
            // be the group of this thread's DV dims, (g * ng) / 8
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int n = 8 * r + 2 * c + e, h = n / ng;
                if (h >= G || n % ng != ((g * ng) >> 3)) continue;
                float* dst = f.acc + slot_index(f.hq0 + h, f.nch, f.ch, f.half) * D + DV * g;
                // INT8 operands are 2^-24 per code step
                const float so = kRowScaled ? f.s_out / kUnit : f.s_out;
#pragma unroll
                for (int i = 0; i < MT; i += 2)
                    *reinterpret_cast<float4*>(dst + 2 * i) =
                        make_float4(acc[r][i][e] * so, acc[r][i][2 + e] * so,
                                    acc[r][i + 1][e] * so, acc[r][i + 1][2 + e] * so);
            }
        }
    }
    __device__ void flush_empty(const Flush& f) {
        if (lane < G) f.ml[slot_index(f.hq0 + lane, f.nch, f.ch, f.half)] = make_float2(-INFINITY, 0.f);
    }
};

// ------------------------------------------- MMA, grouped INT8 / INT4 --

// INT8 or INT4 with one scale per group of GS = D / NG channels, for kv-heads
// whose q-heads x groups exceed 8: one pass over the cache serves all G <= 8
// q-heads.  The operand rows are the q-heads (as in the per-row consumer) and
// the group scales are applied per contraction slice (QK) and per output
// m-tile (PV) instead of per operand row.  Both products read the stage tile
// in 16-byte row segments ("chunks": 16 INT8 or 32 INT4 channels) through
// ldmatrix, so that each tensor-core instruction sees the channels of one
// chunk, which lies inside one group (groups are whole chunks):
//   QK: ldmatrix gives lane (g, c) bytes 4c .. 4c + 3 of row g's chunk: one
//   k16 slice of S^T = Q K^T (INT8), or two (INT4, through the per-row
//   consumer's in-place nibble masks, the query permuted to match).  Each
//   group's slices accumulate separately; a logit is
//   sum_g (S_g - bias * sum_g(q)) * s_K[t][g] (the per-row consumer's offset
//   and unit, per group).  (8-byte loads of a lane's group chunk met 2-way
//   bank conflicts: rows g and g ^ 1 share banks under the 128-byte swizzle.)
//   PV: ldmatrix.trans gives lane (g, c) bytes 2g and 2g + 1 of rows 2c and
//   2c + 1 (tokens) of a chunk in one register: A-operand values of
//   out^T = V^T P^T with the token pair already along k.  The m16 tile of INT8
//   chunk q is dims 16q + 2g (rows g) and 16q + 2g + 1 (rows g + 8); INT4
//   chunk q holds two m-tiles, dims 32q + 4g + 2bb (rows g) and + 1 (rows
//   g + 8, fed as 16x operands), bb = 0, 1 -- masked straight out of the
//   loaded register, with no byte permutes.  The m-tiles of group gi take the
//   weights P * s_V[t][gi] (fp16 hi and residual, two MMAs per m-tile).
// The 16-row multi-pass alternative read the cache once per 16 (q-head, group)
// pairs: twice for Llama-3-70B's G = 8 with 32-channel groups.
template <int FMT, int D, int NG, bool NARROW = false>
struct MmaGroupConsumer {
    static constexpr bool I4 = FMT == INT4;
    static constexpr int RB = row_bytes(FMT, D);  // bytes of one cached row
    static constexpr int GS = D / NG;             // channels per scale group
    static constexpr int NCH = RB / 16;           // 16-byte chunks per row
    static constexpr int CPG = GS / (I4 ? 32 : 16);  // chunks per group
    static constexpr int KS = D / 16;             // k-slices of QK^T
    static constexpr int MT = D / 16;             // m-tiles of PV
    static constexpr int NLK = I4 ? 1 : NCH / 4;  // K: ldmatrix per half box (.x4; INT4 at head_dim 64: .x2)
    static constexpr int NLV = NCH / 2;           // V: ldmatrix.x4.trans per box (two chunks each)
    static_assert(CPG >= 1 && GS % (I4 ? 32 : 16) == 0, "groups of whole 16-byte chunks");
    // INT8: 4 warps per CTA, two CTAs per SM (the stages and group scales take
    // ~17 KB per warp; 206 registers).  INT4 stages are
    // half the bytes and the consumer is bound by instruction issue: one CTA of
    // 16 warps per SM with registers capped at 128 (a few spilled) is 3% faster
    // than two CTAs of 8 and 7% faster than three of 4 at 168 registers.
    // NARROW: INT4 in INT8's 4-warp CTAs, for batches whose context-length
    // scan leaves no room for 16 warps' stages in one CTA
    static constexpr bool kWide4 = I4 && !NARROW;
    static constexpr int kMinCtas = kWide4 ? KVQ_GA4_CTAS : kMinBlocks;
    static constexpr int kWarps = kWide4 ? KVQ_GA4_WARPS : KVQ_GA_WARPS;
    // The query rows are read from global memory when a pair starts (set_q)
    // instead of being staged in shared memory with its first tile, so a new
    // pair's first tile need not wait for the previous pair's to be consumed
    // (+1% on the Llama-3-70B shapes for both formats; the 2 KB per warp this
    // frees at G = 8 would let three INT8 CTAs fit an SM, which measured 6%
    // slower than two)
    static constexpr bool kQGlobal = true;
    static constexpr float kUnit = 5.9604644775390625e-08f;      // operand value of one code step (2^-24)
    static constexpr float kBias = (I4 ? 8.f : 128.f) * kUnit;   // K operand - code * kUnit
    static constexpr float kLogF = I4 ? 2.f : 6.f;               // weights carry 2^kLogF (cancels in acc / l)
    // INT8 slice j: {q[16j + 4c], q[16j + 4c + 1] | q[16j + 4c + 2], q[16j + 4c + 3]};
    // INT4 chunk q, dims b = 32q + 8c ..: [q_b0, q_b5/16] [q_b1/16, q_b4] [q_b2, q_b7/16] [q_b3/16, q_b6]
    uint32_t qa[2 * KS];
    float acc[MT][4];
    float m, l;
    float qsum[NG];        // per group: sum of this lane's row's query values over the group
    int lane, g, c, G;
    float qk_scale;
    uint32_t k_off[NLK];   // this lane's row address for K ldmatrix x (chunks 4x .. 4x + 3), swizzle folded in
    uint32_t v_off[NLV];   // ... for V ldmatrix.trans x: chunks 2x, 2x + 1, rows 0-7 and 8-15 each

    // byte offset of byte o of row r inside a stage tile
    __device__ __forceinline__ static uint32_t off(int r, int o) {
        if (I4 && D == 128) return r * 64 + (o ^ (((r >> 1) & 3) << 4));   // 64-byte swizzle
        if (!I4 && D == 128) return r * 128 + (o ^ ((r & 7) << 4));       // 128-byte swizzle
        return r * RB + o;
    }

    __device__ void init(int G_, float qks, int) {
        lane = threadIdx.x & 31;
        g = lane >> 2;
        c = lane & 3;
        G = G_;
        qk_scale = qks;
        // ldmatrix: lane t gives row t % 8 of matrix t / 8 (chunk 4x + t / 8; .x2 reads lanes 0-15)
#pragma unroll
        for (int x = 0; x < NLK; ++x) k_off[x] = off(lane & 7, 16 * ((4 * x + (lane >> 3)) % NCH));
        // matrices of V load x: (chunk 2x, rows 0-7), (2x, 8-15), (2x + 1, 0-7), (2x + 1, 8-15)
#pragma unroll
        for (int x = 0; x < NLV; ++x) v_off[x] = off(8 * ((lane >> 3) & 1) + (lane & 7), 16 * (2 * x + (lane >> 4)));
    }
    // q: the kv-head's G query rows (shared-memory copy)
    __device__ void set_q(const uint16_t* q) {
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            float sq = 0.f;
            if constexpr (I4) {
#pragma unroll
                for (int cc = 0; cc < CPG; ++cc) {
                    const int ch = CPG * gi + cc;
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (g < G) w = *reinterpret_cast<const uint4*>(q + g * D + 32 * ch + 8 * c);
                    const float2 q01 = f16x2_to_f32x2(w.x), q23 = f16x2_to_f32x2(w.y);
                    const float2 q45 = f16x2_to_f32x2(w.z), q67 = f16x2_to_f32x2(w.w);
                    qa[4 * ch] = pack_f16x2(q01.x, q45.y * 0.0625f);
                    qa[4 * ch + 1] = pack_f16x2(q01.y * 0.0625f, q45.x);
                    qa[4 * ch + 2] = pack_f16x2(q23.x, q67.y * 0.0625f);
                    qa[4 * ch + 3] = pack_f16x2(q23.y * 0.0625f, q67.x);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {  // q as fed times each operand's step (16 for the divided values)
                        const float2 v = f16x2_to_f32x2(qa[4 * ch + i]);
                        sq += (i & 1) ? 16.f * v.x + v.y : v.x + 16.f * v.y;
                    }
                }
            } else {
#pragma unroll
                for (int s = 0; s < CPG; ++s) {
                    const int j = CPG * gi + s;
                    uint2 w = make_uint2(0u, 0u);
                    if (g < G) w = *reinterpret_cast<const uint2*>(q + g * D + 16 * j + 4 * c);
                    qa[2 * j] = w.x;
                    qa[2 * j + 1] = w.y;
                    const float2 v0 = f16x2_to_f32x2(w.x), v1 = f16x2_to_f32x2(w.y);
                    sq += (v0.x + v0.y) + (v1.x + v1.y);
                }
            }
            sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 1);
            sq += __shfl_xor_sync(0xFFFFFFFFu, sq, 2);
            qsum[gi] = sq;
        }
    }
    __device__ void reset() {
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int i = 0; i < MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    }

    // One QK^T product of a k16 slice into the accumulator rows g (odd = 0)
    // or g + 8 (odd = 1): the query operand qa[i], qa[i + 1] in that row half
    __device__ __forceinline__ void qk_mma(float (&s)[4], int odd, int i, uint32_t b0, uint32_t b1) {
        if (odd) mma_16816(s, 0u, qa[i], 0u, qa[i + 1], b0, b1);
        else mma_16816(s, qa[i], 0u, qa[i + 1], 0u, b0, b1);
    }

    // QK^T of one 16-row box: this thread's logits of q-head g, box tokens 2c,
    // 2c+1, 8+2c, 9+2c (already scaled, masked past `valid`).
    __device__ __forceinline__ void qk_box(uint32_t kt, uint32_t sk, int valid, float (&z)[4]) {
        const float ks = qk_scale / kUnit;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
            // group 2p accumulates in rows 0-7 of sacc[p] (the A operand's rows g),
            // group 2p + 1 in rows 8-15 (rows g + 8): half the accumulators
            float sacc[NG / 2][4];
#pragma unroll
            for (int gp = 0; gp < NG / 2; ++gp) sacc[gp][0] = sacc[gp][1] = sacc[gp][2] = sacc[gp][3] = 0.f;
            if constexpr (I4) {
                uint32_t kw[NCH];   // chunk ch: row g's codes 32 ch + 8c .. + 7 (byte i: dims 2i, 2i + 1)
                if constexpr (NCH == 4) ldsm_x4(kt + hb * 8 * RB + k_off[0], kw);
                else ldsm_x2(kt + hb * 8 * RB + k_off[0], kw);
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    // bit 3 of every nibble flipped (code + 8), masked in place:
                    // [d0, 16 d5] [16 d1, d4] and [d2, 16 d7] [16 d3, d6]
                    const uint32_t x = kw[ch] ^ 0x88888888u, y = x >> 8;
                    qk_mma(sacc[ch / CPG / 2], (ch / CPG) & 1, 4 * ch, x & 0x00F0000Fu, x & 0x000F00F0u);
                    qk_mma(sacc[ch / CPG / 2], (ch / CPG) & 1, 4 * ch + 2, y & 0x00F0000Fu, y & 0x000F00F0u);
                }
            } else {
#pragma unroll
                for (int x = 0; x < NLK; ++x) {
                    uint32_t kw[4];   // slices 4x .. 4x + 3: row g's bytes 16 j + 4c .. + 3
                    ldsm_x4(kt + hb * 8 * RB + k_off[x], kw);
#pragma unroll
                    for (int m4 = 0; m4 < 4; ++m4) {
                        const int j = 4 * x + m4;
                        const uint32_t w = kw[m4] ^ 0x80808080u;   // code + 128 as an unsigned byte
                        const uint32_t b0 = prmt(w, 0u, 0x4140u), b1 = prmt(w, 0u, 0x4342u);
                        qk_mma(sacc[j / CPG / 2], (j / CPG) & 1, 2 * j, b0, b1);
                    }
                }
            }
            // tokens 8 hb + 2c, 8 hb + 2c + 1: scales [token][NG]
            const uint32_t s0 = sk + 4 * NG * (8 * hb + 2 * c);
            float k0[NG], k1[NG];
            if (NG == 4) {
                const uint4 x0 = lds128(s0), x1 = lds128(s0 + 16);
                k0[0] = __uint_as_float(x0.x); k0[1 % NG] = __uint_as_float(x0.y);
                k0[2 % NG] = __uint_as_float(x0.z); k0[3 % NG] = __uint_as_float(x0.w);
                k1[0] = __uint_as_float(x1.x); k1[1 % NG] = __uint_as_float(x1.y);
                k1[2 % NG] = __uint_as_float(x1.z); k1[3 % NG] = __uint_as_float(x1.w);
            } else {
                const uint4 x = lds128(s0);
                k0[0] = __uint_as_float(x.x); k0[1 % NG] = __uint_as_float(x.y);
                k1[0] = __uint_as_float(x.z); k1[1 % NG] = __uint_as_float(x.w);
            }
            float z0 = 0.f, z1 = 0.f;
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
                const float corr = kBias * qsum[gi];
                z0 = fmaf(sacc[gi / 2][2 * (gi & 1)] - corr, k0[gi], z0);
                z1 = fmaf(sacc[gi / 2][2 * (gi & 1) + 1] - corr, k1[gi], z1);
            }
            z[2 * hb] = z0 * ks;
            z[2 * hb + 1] = z1 * ks;
        }
        if (valid < kBox) {
            if (2 * c >= valid) z[0] = -INFINITY;
            if (2 * c + 1 >= valid) z[1] = -INFINITY;
            if (8 + 2 * c >= valid) z[2] = -INFINITY;
            if (9 + 2 * c >= valid) z[3] = -INFINITY;
        }
    }

    // P (fp16 hi + residual) of one box as the B operand of PV, k = token,
    // n = q-head g
    __device__ __forceinline__ static void p_frags(const float (&p)[4], uint32_t& pb0, uint32_t& pb1, uint32_t& pl0,
                                                   uint32_t& pl1) {
        pb0 = pack_f16x2(p[0], p[1]);
        pb1 = pack_f16x2(p[2], p[3]);
        const float2 h01 = f16x2_to_f32x2(pb0), h23 = f16x2_to_f32x2(pb1);
        pl0 = pack_f16x2(p[0] - h01.x, p[1] - h01.y);
        pl1 = pack_f16x2(p[2] - h23.x, p[3] - h23.y);
    }

    // out^T += V^T P_g^T for one box: p = weights of box tokens 2c, 2c+1, 8+2c,
    // 9+2c; sv = their V scales per group
    __device__ __forceinline__ void pv_box(uint32_t vt, int valid, const float (&p)[4], const float (&sv)[4][NG]) {
        // r[x][0] / r[x][2]: chunk 2x / 2x + 1, tokens 2c (bits 0-15) and 2c + 1 (bits 16-31);
        // r[x][1] / r[x][3]: the same for tokens 8 + 2c and 9 + 2c
        uint32_t r[NLV][4];
#pragma unroll
        for (int x = 0; x < NLV; ++x) ldsm_x4_t(vt + v_off[x], r[x]);
        if (valid < kBox) {  // rows past the context may hold NaN codes: zero them
            const uint32_t mlo = (2 * c < valid ? 0x0000FFFFu : 0u) | (2 * c + 1 < valid ? 0xFFFF0000u : 0u);
            const uint32_t mhi = (8 + 2 * c < valid ? 0x0000FFFFu : 0u) | (9 + 2 * c < valid ? 0xFFFF0000u : 0u);
#pragma unroll
            for (int x = 0; x < NLV; ++x) {
                r[x][0] &= mlo; r[x][1] &= mhi; r[x][2] &= mlo; r[x][3] &= mhi;
            }
        }
#pragma unroll
        for (int x = 0; x < NLV; ++x)   // code + 8 in every nibble, or code + 128 in every byte (zeroed rows give 0 below)
#pragma unroll
            for (int e = 0; e < 4; ++e) r[x][e] ^= I4 ? 0x88888888u : 0x80808080u;
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
            float pg[4];
            if (valid >= kBox) {
#pragma unroll
                for (int e = 0; e < 4; ++e) pg[e] = p[e] * sv[e][gi];
            } else {  // a masked token keeps p = 0 whatever its (never written) scale slot holds
#pragma unroll
                for (int e = 0; e < 4; ++e) pg[e] = p[e] != 0.f ? p[e] * sv[e][gi] : 0.f;
            }
            uint32_t pb0, pb1, pl0, pl1;
            p_frags(pg, pb0, pb1, pl0, pl1);
#pragma unroll
            for (int cc = 0; cc < CPG; ++cc) {
                const int ch = CPG * gi + cc;
                const uint32_t lo = r[ch >> 1][2 * (ch & 1)], hi = r[ch >> 1][2 * (ch & 1) + 1];
                if constexpr (I4) {
#pragma unroll
                    for (int bb = 0; bb < 2; ++bb) {
                        // byte bb of each token's pair: dim 32 ch + 4g + 2bb (low nibble, rows g) and
                        // + 1 (high nibble in place: 16x, rows g + 8), less the offsets (exact)
                        const uint32_t u = bb ? lo >> 8 : lo, w = bb ? hi >> 8 : hi;
                        const uint32_t a0 = hsub2_exact(u & 0x000F000Fu, 0x00080008u);
                        const uint32_t a1 = hsub2_exact(u & 0x00F000F0u, 0x00800080u);
                        const uint32_t a2 = hsub2_exact(w & 0x000F000Fu, 0x00080008u);
                        const uint32_t a3 = hsub2_exact(w & 0x00F000F0u, 0x00800080u);
                        mma_16816(acc[2 * ch + bb], a0, a1, a2, a3, pb0, pb1);
                        mma_16816(acc[2 * ch + bb], a0, a1, a2, a3, pl0, pl1);
                    }
                } else {
                    // bytes 0 | 2: dim 16 ch + 2g (rows g); bytes 1 | 3: dim 16 ch + 2g + 1 (rows g + 8),
                    // as fp16 subnormals (code + 128) * 2^-24, less 128 * 2^-24 (exact)
                    const uint32_t a0 = hsub2_exact(prmt(lo, 0u, 0x4240u), 0x00800080u);
                    const uint32_t a1 = hsub2_exact(prmt(lo, 0u, 0x4341u), 0x00800080u);
                    const uint32_t a2 = hsub2_exact(prmt(hi, 0u, 0x4240u), 0x00800080u);
                    const uint32_t a3 = hsub2_exact(prmt(hi, 0u, 0x4341u), 0x00800080u);
                    mma_16816(acc[ch], a0, a1, a2, a3, pb0, pb1);
                    mma_16816(acc[ch], a0, a1, a2, a3, pl0, pl1);
                }
            }
        }
    }

    __device__ __forceinline__ void v_scales(uint32_t sv0, float (&sv)[4][NG]) {
        // tokens 2c, 2c+1, 8+2c, 9+2c of the box: scales [token][NG]
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t a = sv0 + 4 * NG * (2 * c + (e & 1) + 8 * (e >> 1));
            if (NG == 4) {
                const uint4 x = lds128(a);
                sv[e][0] = __uint_as_float(x.x); sv[e][1 % NG] = __uint_as_float(x.y);
                sv[e][2 % NG] = __uint_as_float(x.z); sv[e][3 % NG] = __uint_as_float(x.w);
            } else {
                const uint2 x = lds64(a);
                sv[e][0] = __uint_as_float(x.x); sv[e][1 % NG] = __uint_as_float(x.y);
            }
        }
    }

    __device__ void tile(const Tile& cx) {
        float z0[4], z1[4];
        qk_box(cx.k, cx.s, cx.valid, z0);
        qk_box(cx.k + kBox * RB, cx.s + 4 * kBox * NG, cx.valid - kBox, z1);
        float mx = fmaxf(fmaxf(fmaxf(z0[0], z0[1]), fmaxf(z0[2], z0[3])), fmaxf(fmaxf(z1[0], z1[1]), fmaxf(z1[2], z1[3])));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const float mn = fmaxf(m, mx);
        float alpha = 1.f, p0[4], p1[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) p0[e] = p1[e] = 0.f;
        if (mn != -INFINITY) {
            alpha = fast_exp2(m - mn);
            const float mb = mn - kLogF;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                p0[e] = fast_exp2(z0[e] - mb);
                p1[e] = fast_exp2(z1[e] - mb);
            }
        }
        m = mn;
        l = l * alpha + (((p0[0] + p0[1]) + (p0[2] + p0[3])) + ((p1[0] + p1[1]) + (p1[2] + p1[3])));
        // rescale the accumulators: columns 2c and 2c+1 are q-heads 2c and 2c+1
        if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
            const float a0 = __shfl_sync(0xFFFFFFFFu, alpha, 8 * c);
            const float a1 = __shfl_sync(0xFFFFFFFFu, alpha, 8 * c + 4);
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                acc[i][0] *= a0; acc[i][1] *= a1; acc[i][2] *= a0; acc[i][3] *= a1;
            }
        }
        const uint32_t sv = cx.s + 4 * kTile * NG;
        float s0[4][NG];
        v_scales(sv, s0);
        pv_box(cx.v, cx.valid, p0, s0);
        v_scales(sv + 4 * kBox * NG, s0);
        pv_box(cx.v + kBox * RB, cx.valid - kBox, p1, s0);
    }

    __device__ void flush(const Flush& f) {
        float lq = l;
        lq += __shfl_xor_sync(0xFFFFFFFFu, lq, 1);
        lq += __shfl_xor_sync(0xFFFFFFFFu, lq, 2);
        if (c == 0 && g < G) f.ml[slot_index(f.hq0 + g, f.nch, f.ch, f.half)] = make_float2(m, lq);
        // acc[i][e] (acc[i][2 + e]) = out[q-head 2c + e][m-tile i's dim of rows g (g + 8)]
        const float so = f.s_out / kUnit;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int h = 2 * c + e;
            if (h >= G) continue;
            float* dst = f.acc + slot_index(f.hq0 + h, f.nch, f.ch, f.half) * D;
            if constexpr (I4) {  // chunk ch: dims 32 ch + 4g .. + 3; the odd ones were fed as 16x operands
                const float so1 = so * 0.0625f;
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch)
                    *reinterpret_cast<float4*>(dst + 32 * ch + 4 * g) =
                        make_float4(acc[2 * ch][e] * so, acc[2 * ch][2 + e] * so1, acc[2 * ch + 1][e] * so,
                                    acc[2 * ch + 1][2 + e] * so1);
            } else {  // chunk ch: dims 16 ch + 2g, + 1
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch)
                    *reinterpret_cast<float2*>(dst + 16 * ch + 2 * g) = make_float2(acc[ch][e] * so, acc[ch][2 + e] * so);
            }
        }
    }
    __device__ void flush_empty(const Flush& f) {
        if (lane < G) f.ml[slot_index(f.hq0 + lane, f.nch, f.ch, f.half)] = make_float2(-INFINITY, 0.f);
    }
};

// ------------------------------------------------------ append in decode --

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void sts8(uint32_t addr, uint8_t v) {
    asm volatile("st.shared.u8 [%0], %1;" ::"r"(addr), "h"((uint16_t)v) : "memory");
}
__device__ __forceinline__ void stsf(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// One warp quantizes the newest token's K and V rows (fp16, in shared memory
// at nkv) exactly as the append kernels do, writes the codes (and INT8 / INT4
// row scales) to the cache row of position `pos`, and patches them into the
// landed stage tile (first token tok0) so this tile's attention sees them.
// blk < 0: the block id was outside the cache (already recorded); nothing is
// written.  Lane l handles values D/32 * l ...
template <int FMT, int D>
__device__ __noinline__ void append_newest(const uint16_t* nkv, int blk, int pos, int tok0, int kvh,
                                           const DecodeArgs& a, float s_fp8, uint32_t kt, int tile_bytes,
                                           uint32_t st, int lane) {
    constexpr int VPL = D / 32;  // values per lane: 4 or 2
    float x[2][VPL];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const uint16_t* src = nkv + w * D + VPL * lane;
        if (VPL == 4) {
            const uint2 r = *reinterpret_cast<const uint2*>(src);
            const float2 f0 = f16x2_to_f32x2(r.x), f1 = f16x2_to_f32x2(r.y);
            x[w][0] = f0.x; x[w][1] = f0.y; x[w][VPL > 2 ? 2 : 0] = f1.x; x[w][VPL > 3 ? 3 : 1] = f1.y;
        } else {
            const float2 f0 = f16x2_to_f32x2(*reinterpret_cast<const uint32_t*>(src));
            x[w][0] = f0.x; x[w][1] = f0.y;
        }
    }
    uint32_t code[2];
    float rs[2] = {0.f, 0.f};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        uint32_t c = 0;
        if (FMT == INT8 || FMT == INT4) {
            constexpr float kQmax = FMT == INT4 ? 7.0f : 127.0f;
            constexpr int kQi = FMT == INT4 ? 7 : 127, kBits = FMT == INT4 ? 4 : 8;
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < VPL; ++i) amax = fmaxf(amax, fabsf(x[w][i]));
            // over the 32 / ng lanes of this lane's scale group (all 32 for one per row)
            const int lpg = 32 / a.cache.ngroups;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                if (off < lpg) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
            const float s = __fdiv_rn(amax, kQmax);
            rs[w] = s;
#pragma unroll
            for (int i = 0; i < VPL; ++i) {
                int q = 0;
                if (s != 0.f) q = max(-kQi, min(kQi, __float2int_rn(__fdiv_rn(x[w][i], s))));
                c |= (uint32_t)(q & ((1 << kBits) - 1)) << (kBits * i);
            }
        } else {
            float y[VPL];
#pragma unroll
            for (int i = 0; i < VPL; ++i) y[i] = s_fp8 != 1.0f ? __fdiv_rn(x[w][i], s_fp8) : x[w][i];
#pragma unroll
            for (int i = 0; i < VPL; i += 2) c |= (uint32_t)enc_fp8x2<FMT>(y[i], y[i + 1]) << (8 * i);
        }
        code[w] = c;
    }
    if (blk >= 0 && FMT == INT4) {  // VPL codes = VPL / 2 bytes per lane
        constexpr int RB = D / 2;
        const int r = pos - tok0;
        const uint32_t kb = kt + (r / kBox) * kBox * RB + (r % kBox) * RB;
        const int BS = a.cache.block_size;
        const int64_t row = ((int64_t)blk * a.cache.num_kv_heads + kvh) * BS + (pos & (BS - 1));
        if (D == 128) {  // the stage's 64-byte rows are 64-byte swizzled
            const uint32_t off = ((((lane >> 3) ^ (r >> 1)) & 3) << 4) | ((2 * lane) & 15);
            sts16(kb + off, (uint16_t)code[0]);
            sts16(kb + tile_bytes + off, (uint16_t)code[1]);
            reinterpret_cast<uint16_t*>(a.cache.k_codes + row * RB)[lane] = (uint16_t)code[0];
            reinterpret_cast<uint16_t*>(a.cache.v_codes + row * RB)[lane] = (uint16_t)code[1];
        } else {
            sts8(kb + lane, (uint8_t)code[0]);
            sts8(kb + tile_bytes + lane, (uint8_t)code[1]);
            a.cache.k_codes[row * RB + lane] = (uint8_t)code[0];
            a.cache.v_codes[row * RB + lane] = (uint8_t)code[1];
        }
        const int ng = a.cache.ngroups, lpg = 32 / ng;
        if (lane % lpg == 0) {  // scales [token][ng]: this lane's group lane / lpg
            const int j = r * ng + lane / lpg;
            stsf(st + 4 * j, rs[0]);
            stsf(st + 4 * kTile * ng + 4 * j, rs[1]);
            a.cache.k_scales[row * ng + lane / lpg] = rs[0];
            a.cache.v_scales[row * ng + lane / lpg] = rs[1];
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    } else if (blk >= 0) {
        const int r = pos - tok0;  // row in the tile: box r / 16, row r % 16
        const uint32_t kb = kt + (r / kBox) * kBox * D;
        if (D == 128) {
            const uint32_t off = tile_off<128>(r % kBox, lane >> 2) + 4 * (lane & 3);
            sts32(kb + off, code[0]);
            sts32(kb + tile_bytes + off, code[1]);
        } else {
            const uint32_t off = (r % kBox) * D + 2 * lane;
            sts16(kb + off, (uint16_t)code[0]);
            sts16(kb + tile_bytes + off, (uint16_t)code[1]);
        }
        const int BS = a.cache.block_size;
        const int64_t row = ((int64_t)blk * a.cache.num_kv_heads + kvh) * BS + (pos & (BS - 1));
        if (D == 128) {
            reinterpret_cast<uint32_t*>(a.cache.k_codes + row * D)[lane] = code[0];
            reinterpret_cast<uint32_t*>(a.cache.v_codes + row * D)[lane] = code[1];
        } else {
            reinterpret_cast<uint16_t*>(a.cache.k_codes + row * D)[lane] = (uint16_t)code[0];
            reinterpret_cast<uint16_t*>(a.cache.v_codes + row * D)[lane] = (uint16_t)code[1];
        }
        const int ng = a.cache.ngroups, lpg = 32 / ng;
        if (FMT == INT8 && lane % lpg == 0) {  // scales [token][ng]: this lane's group lane / lpg
            const int j = r * ng + lane / lpg;
            stsf(st + 4 * j, rs[0]);
            stsf(st + 4 * kTile * ng + 4 * j, rs[1]);
            a.cache.k_scales[row * ng + lane / lpg] = rs[0];
            a.cache.v_scales[row * ng + lane / lpg] = rs[1];
        }
        // the stage is refilled by TMA later: order these generic writes first
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncwarp();
}

// -------------------------------------------------------------- kernel --

template <int FMT, int D, class Consumer>
__global__ void __launch_bounds__(Consumer::kWarps * 32, Consumer::kMinCtas)
    decode_stream_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                         const DecodeArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = a.batch, Hkv = a.cache.num_kv_heads, BS = a.cache.block_size;
    const int Gall = a.num_q_heads / Hkv;   // q-heads per kv-head
    const int G = a.heads, h0 = a.head_off;   // the ones this launch serves
    const bool append = a.k_new != nullptr;
    constexpr bool kRowScaled = FMT == INT8 || FMT == INT4;
    constexpr int RB = row_bytes(FMT, D);
    const int ng = a.cache.ngroups;
    constexpr int kConsumers = Consumer::kWarps, kThreads = kConsumers * 32;
    constexpr bool kQGlobal = Consumer::kQGlobal;
    const Layout L(kConsumers, RB, D, kQGlobal ? 0 : G, B, kRowScaled, append, ng);
    const uint32_t sc_stage = 2 * kTile * 4 * ng;  // bytes of a stage's K and V scales
    int* S = reinterpret_cast<int*>(smem + L.scan);
    int* ctx_s = S + B + 1;
    griddep_wait();    // inputs may come from the previous kernel (an append)
    griddep_launch();  // the reduce kernel may be scheduled as CTAs finish

    // ---- tiles per sequence, scanned (every CTA does this once) -------------
    {
        __shared__ int wsum[kConsumers];
        const int cap = min(a.max_context_len, a.max_blocks_per_seq * BS);
        const int per = (B + kThreads - 1) / kThreads;
        const int b0 = threadIdx.x * per, b1 = min(B, b0 + per);
        int local = 0;
        for (int b = b0; b < b1; ++b) {
            int ctx = a.context_lens[b];
            if (ctx < 0 || ctx > cap) {
                if (blockIdx.x == 0) record_error(a.err, DEV_ERR_RANGE, ctx);
                ctx = ctx < 0 ? 0 : cap;
            }
            ctx_s[b] = ctx;
            local += (ctx + kTile - 1) / kTile;
        }
        int x = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        if (threadIdx.x < kConsumers * kSpw) mbar_init(reinterpret_cast<uint64_t*>(smem + L.full) + threadIdx.x, 1);
        fence_barrier_init();
        __syncthreads();
        int run = x - local;
        for (int w = 0; w < warp; ++w) run += wsum[w];
        for (int b = b0; b < b1; ++b) {
            S[b] = run;
            run += (ctx_s[b] + kTile - 1) / kTile;
        }
        if (threadIdx.x == kThreads - 1) S[B] = run;
        __syncthreads();
    }
    // ---- this warp's range of the flat tile list -----------------------------
    const int T = Hkv * S[B];  // total tiles
    const int C = a.chunk_tiles;
    const int nw = max(1, min((int)gridDim.x * kConsumers, T / C));  // a range is never shorter than a chunk
    const int gw = blockIdx.x * kConsumers + warp;
    if (T == 0 || gw >= nw) return;
    const int base_len = T / nw, extra = T % nw;
    const int lo = gw * base_len + min(gw, extra);
    const int hi = lo + base_len + (gw < extra ? 1 : 0);

    uint8_t* tiles = smem + warp * kSpw * 2 * L.tile_bytes;
    float* scales = reinterpret_cast<float*>(smem + L.scales) + warp * kSpw * 2 * kTile * ng;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full) + warp * kSpw;
    uint8_t* qbuf = smem + L.qbuf + warp * L.q_bytes;
    uint16_t* nkv = reinterpret_cast<uint16_t*>(smem + L.newkv) + warp * 2 * D;  // appending launches only
    int* patch_blk = reinterpret_cast<int*>(smem + L.patch) + warp;
    const uint32_t tiles_u32 = smem_u32(tiles), scales_u32 = smem_u32(scales);

    // Block-table entries of the 32 boxes of flat tiles [first, first + 16):
    // lane j holds box j % 2 of tile first + j / 2 (0 for boxes past the
    // context, which are never loaded).  Read back with a shuffle.
    auto load_id = [&](int first) -> int {
        const int ff = first + (lane >> 1);
        if (ff >= hi) return 0;
        const Walk w = locate(S, B, Hkv, ff);
        const int tok = w.t * kTile + (lane & 1) * kBox;
        if (tok >= ctx_s[w.b]) return 0;
        return __ldg(a.block_tables + (int64_t)w.b * a.max_blocks_per_seq + tok / BS);
    };
    int idc = load_id(lo);       // tiles [window, window + 16)
    int idn = load_id(lo + 16);  // the next window, loaded one window ahead
    if (lane == 0) {
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
    }
    const uint64_t pol = policy_evict_first();
    const uint32_t box_tx = 2 * kBox * RB + (kRowScaled ? 2 * kBox * 4 * ng : 0);
    const bool big_box = BS >= kTile;  // a tile lies in one block: one 32-row box per tensor
    const uint32_t q_tx = kQGlobal ? 0u : (uint32_t)(G * D * 2);

    const float s_fp8 = (!kRowScaled && a.scale) ? __ldg(a.scale) : 1.0f;
    const float s_out = kRowScaled ? 1.0f : s_fp8;
    float* ws_acc = a.ws;
    float2* ws_ml = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(a.ws) +
                                              ws_acc_bytes(B, a.num_q_heads, a.num_chunks, D));
    Consumer cons;
    cons.init(G, a.sm_scale * s_fp8 * kLog2e, ng);

    // issue side: next flat tile fi, its stage ist, its position iw, the
    // first tile of the last pair whose queries were copied (pend) and the
    // last tile of the last pair whose newest K/V row was copied (lpend)
    Walk iw = locate(S, B, Hkv, lo);
    int fi = lo, ist = 0, pend = -1, lpend = -1;
    // consume side: next flat tile fc, its stage cst and barrier parity cph, its
    // position cw, tile ctc within chunk cch, and the slot half of the segment
    // in progress
    Walk cw = iw;
    int fc = lo, cst = 0;
    uint32_t cph = 0;
    int ctc = cw.t % C, cch = cw.t / C;
    int seg_half = ctc == 0 ? 0 : 1;
    cons.reset();

    // Issue tiles while a stage is free.  The first tile of a pair also copies
    // the pair's queries into this warp's query buffer, which must not happen
    // before the previous pair's first tile has been consumed.  In an
    // appending launch the last tile of a pair also copies the fp16 K and V
    // rows of the pair's newest token into the warp's new-row buffer, under
    // the same rule.
    auto issue_ready = [&]() {
        while (fi < hi && fi - fc < kSpw) {
            const int rel = fi - lo;
            const bool new_pair = iw.t == 0 || rel == 0;
            if (!kQGlobal && new_pair && pend >= fc) break;
            const bool ends = append && iw.t == iw.n - 1;
            if (ends && lpend >= fc) break;
            const int id0 = __shfl_sync(0xFFFFFFFFu, idc, (2 * rel) & 31);
            const int id1 = __shfl_sync(0xFFFFFFFFu, idc, (2 * rel + 1) & 31);
            const int tok0 = iw.t * kTile;
            // a 16-row box past the context is not loaded; a 32-row box (blocks
            // of 32 or more tokens) always is (the rows past the context are
            // masked like those of an unwritten second box)
            const int nbox = big_box ? 2 : (ctx_s[iw.b] - tok0 > kBox ? 2 : 1);
            uint64_t* fb = &full[ist];
            if (lane == 0) {
                if (ends) {  // block of the newest row; -1 (not written) if outside the cache
                    const int nb = ctx_s[iw.b] - 1 - tok0 >= kBox ? id1 : id0;
                    *patch_blk = nb < 0 || nb >= a.cache.num_blocks ? -1 : nb;
                }
                mbar_arrive_expect_tx(fb, nbox * box_tx + (new_pair ? q_tx : 0u) + (ends ? 4u * D : 0u));
            }
            // The copies of a tile are issued by lanes 0-7 at once: lane j moves
            // box j & 1 of K (j = 0, 1) or V (2, 3) codes, or of their row
            // scales (4-7); one 32-row copy per tensor (lanes 0, 2, 4, 6) when
            // the tile lies in one block of 32 or more tokens.  (Lane 0's
            // expect-tx may land after some of their bytes; the phase cannot
            // complete before that arrival.)
            const int bx = lane & 1, which = (lane >> 1) & 1;
            if (lane < (kRowScaled ? 8 : 4) && bx < (big_box ? 1 : nbox)) {
                int blk = bx ? id1 : id0;
                if (blk < 0 || blk >= a.cache.num_blocks) {
                    record_error(a.err, DEV_ERR_RANGE, blk);
                    blk = 0;  // keep the pipeline going on a block that exists
                }
                const int row = (blk * Hkv + iw.kvh) * BS + ((tok0 + bx * kBox) & (BS - 1));
                if (lane < 4) {
                    const uint32_t dst = tiles_u32 + ist * (2 * L.tile_bytes) + which * L.tile_bytes + bx * kBox * RB;
                    tma_load_2d_u32(dst, which ? &tmv : &tmk, 0, row, fb, pol);
                } else {
                    const uint32_t sb = (big_box ? kTile : kBox) * 4 * ng;  // the copy's rows of ng scales
                    const uint32_t dst = scales_u32 + ist * sc_stage + which * (kTile * 4 * ng) + bx * (kBox * 4 * ng);
                    bulk_load_u32(dst, (which ? a.cache.v_scales : a.cache.k_scales) + (int64_t)row * ng, sb, fb, pol);
                }
            }
            if (!kQGlobal && new_pair && lane == 8)
                bulk_load(qbuf, a.q + ((int64_t)iw.b * a.num_q_heads + (int64_t)iw.kvh * Gall + h0) * D, q_tx, fb, pol);
            if (ends && (lane == 9 || lane == 10)) {
                const int64_t row = ((int64_t)iw.b * Hkv + iw.kvh) * D;
                if (lane == 9) bulk_load(nkv, a.k_new + row, 2 * D, fb, pol);
                else bulk_load(nkv + D, a.v_new + row, 2 * D, fb, pol);
            }
            if (new_pair) pend = fi;
            if (ends) lpend = fi;
            advance(iw, S, B, Hkv);
            ++fi;
            ist = ist + 1 == kSpw ? 0 : ist + 1;
            if (((rel + 1) & 15) == 0) {  // next 16-tile window
                idc = idn;
                idn = load_id(fi + 16);
            }
        }
    };
    issue_ready();

    bool failed = false;
    while (fc < hi) {
        if (!mbar_wait(&full[cst], cph, nullptr)) {
            if (lane == 0) record_error(a.err, DEV_ERR_TIMEOUT, fc);
            failed = true;
            break;
        }
        if (cw.t == 0 || fc == lo) {  // staged with this tile, or read from global memory
            if (kQGlobal)
                cons.set_q(a.q + ((int64_t)cw.b * a.num_q_heads + (int64_t)cw.kvh * Gall + h0) * D);
            else
                cons.set_q(reinterpret_cast<const uint16_t*>(qbuf));
        }
        if (append && cw.t == cw.n - 1)
            append_newest<FMT, D>(nkv, *patch_blk, ctx_s[cw.b] - 1, cw.t * kTile, cw.kvh, a, s_fp8,
                                  tiles_u32 + cst * (2 * L.tile_bytes), L.tile_bytes,
                                  scales_u32 + cst * sc_stage, lane);
        const uint32_t kt = tiles_u32 + cst * (2 * L.tile_bytes);
        const Tile tl{kt, kt + L.tile_bytes, scales_u32 + cst * sc_stage, min(kTile, ctx_s[cw.b] - cw.t * kTile)};
        cons.tile(tl);
        __syncwarp();
        const bool pair_end = cw.t == cw.n - 1;
        const bool chunk_end = ctc == C - 1 || pair_end;
        if (chunk_end || fc == hi - 1) {
            Flush fl{ws_acc, ws_ml, (int64_t)cw.b * a.num_q_heads + (int64_t)cw.kvh * Gall + h0, cch, seg_half,
                     a.num_chunks, s_out};
            cons.flush(fl);
            if (seg_half == 0 && chunk_end) {  // the whole chunk was this warp's: its second slot is empty
                fl.half = 1;
                cons.flush_empty(fl);
            }
            cons.reset();
            seg_half = 0;
        }
        ++fc;
        cst = cst + 1 == kSpw ? 0 : cst + 1;
        cph ^= cst == 0 ? 1u : 0u;
        if (pair_end) {
            cw.t = 0;
            ctc = 0;
            cch = 0;
            if (++cw.kvh == Hkv) {
                cw.kvh = 0;
                do {
                    ++cw.b;
                } while (cw.b < B && S[cw.b + 1] == S[cw.b]);
                cw.n = cw.b < B ? S[cw.b + 1] - S[cw.b] : 0;
            }
        } else {
            ++cw.t;
            if (++ctc == C) {
                ctc = 0;
                ++cch;
            }
        }
        issue_ready();
    }
    if (failed) {  // let the copies this warp started land before it exits
        for (int f = fc; f < fi; ++f) {
            mbar_wait(&full[cst], cph, nullptr);
            cst = cst + 1 == kSpw ? 0 : cst + 1;
            cph ^= cst == 0 ? 1u : 0u;
        }
    }
}

// Combine the chunk partials of one (sequence, q-head), one warp each:
// out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.  Lanes read the slots'
// (m, l) in parallel; every lane then sums D/32 consecutive outputs over the
// slots with independent vector loads.
constexpr int kReduceWarps = 4;

// One CTA per (sequence, q-head): every thread takes part in the maximum over
// the partial slots, warp w merges slots w, w + 4, ... (four loads in flight
// per lane), and the four warps' partial sums are combined in shared memory.
// A single warp per head walking its slots one at a time was latency-bound at
// small batches with long contexts (hundreds of slots per head).
template <int D>
__global__ void __launch_bounds__(kReduceWarps * 32) decode_reduce_kernel(const DecodeArgs a) {
    constexpr int V = D / 32;  // outputs per lane: 4 (D = 128) or 2 (D = 64)
    __shared__ float red_m[kReduceWarps], red_l[kReduceWarps];
    __shared__ __align__(16) float red_o[kReduceWarps][D];
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t hq = blockIdx.x;
    const int b = (int)(hq / a.num_q_heads);
    int ctx = a.context_lens[b];
    const int cap = min(a.max_context_len, a.max_blocks_per_seq * a.cache.block_size);
    ctx = ctx < 0 ? 0 : min(ctx, cap);
    const int tiles = (ctx + kTile - 1) / kTile;
    const int nslots = 2 * min(a.num_chunks, (tiles + a.chunk_tiles - 1) / a.chunk_tiles);
    const float2* ml = reinterpret_cast<const float2*>(reinterpret_cast<const uint8_t*>(a.ws) +
                                                       ws_acc_bytes(a.batch, a.num_q_heads, a.num_chunks, D));
    const int64_t s0 = hq * a.num_chunks * 2;
    float M = -INFINITY;
    for (int i = threadIdx.x; i < nslots; i += kReduceWarps * 32) M = fmaxf(M, ml[s0 + i].x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
    if (lane == 0) red_m[warp] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kReduceWarps; ++w) M = fmaxf(M, red_m[w]);
    float Lsum = 0.f, O[V];
#pragma unroll
    for (int k = 0; k < V; ++k) O[k] = 0.f;
    if (M != -INFINITY) {
#pragma unroll 4
        for (int i = warp; i < nslots; i += kReduceWarps) {
            const float2 v = ml[s0 + i];
            if (v.x == -INFINITY) continue;  // empty slot: its accumulator was never written
            const float e = fast_exp2(v.x - M);
            Lsum += e * v.y;
            const float* src = a.ws + (s0 + i) * D + V * lane;
            if (V == 4) {
                const float4 x = *reinterpret_cast<const float4*>(src);
                O[0] += e * x.x; O[1] += e * x.y; O[2] += e * x.z; O[3] += e * x.w;
            } else {
                const float2 x = *reinterpret_cast<const float2*>(src);
                O[0] += e * x.x; O[1] += e * x.y;
            }
        }
    }
    if (lane == 0) red_l[warp] = Lsum;
#pragma unroll
    for (int k = 0; k < V; ++k) red_o[warp][V * lane + k] = O[k];
    __syncthreads();
    if (warp != 0) return;
#pragma unroll
    for (int k = 0; k < V; ++k) O[k] = 0.f;
    Lsum = 0.f;
#pragma unroll
    for (int w = 0; w < kReduceWarps; ++w) {
        Lsum += red_l[w];
#pragma unroll
        for (int k = 0; k < V; ++k) O[k] += red_o[w][V * lane + k];
    }
    const float inv = Lsum > 0.f ? 1.0f / Lsum : 0.f;
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + hq * D + V * lane);
    if (V == 4)
        *reinterpret_cast<uint2*>(dst) = make_uint2(pack_f16x2(O[0] * inv, O[1] * inv), pack_f16x2(O[2] * inv, O[3] * inv));
    else
        *dst = pack_f16x2(O[0] * inv, O[1] * inv);
}

// ---------------------------------------------------------------- host --

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view [rows = blocks * kv-heads * block][head_dim] of one code array;
// box = 16 rows (one 16-token slice of a paged block), or 32 rows (a whole
// 32-token tile) when blocks hold 32 or more tokens.
// rb: bytes per row (head_dim, or head_dim / 2 for INT4); 128-byte rows are
// loaded with the 128-byte swizzle, INT4 rows of head_dim 128 (64 bytes) with
// the 64-byte swizzle (16-byte chunk index XOR (row / 2) % 4, so the V rows
// 2c of the four lane groups no longer share their banks), other rows plain
// (the 8-bit formats at head_dim 64 also have 64-byte rows, read unswizzled).
bool make_tmap(CUtensorMap* m, void* base, int64_t rows, int rb, int box_rows, bool int4) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)rb, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)rb};
    cuuint32_t box[2] = {(cuuint32_t)rb, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                               : (int4 && rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE),
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int FMT, int D, class Consumer>
cudaError_t launch_stream(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, cudaStream_t s) {
    auto kern = decode_stream_kernel<FMT, D, Consumer>;
    constexpr int kConsumers = Consumer::kWarps, kThreads = kConsumers * 32;
    const int smem = Layout(kConsumers, row_bytes(FMT, D), D, Consumer::kQGlobal ? 0 : a.heads, a.batch,
                            FMT == INT8 || FMT == INT4, a.k_new != nullptr, a.cache.ngroups).total + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem)) != cudaSuccess) return e;
    per_sm = per_sm < 1 ? 1 : per_sm;
    // no more warps than chunks at the largest context: a range spans a chunk
    const int64_t max_tiles = (int64_t)a.batch * a.cache.num_kv_heads * ((a.max_context_len + kTile - 1) / kTile);
    int64_t want = max_tiles / a.chunk_tiles;
    want = want < 1 ? 1 : want;
    int64_t grid = (want + kConsumers - 1) / kConsumers;
    if (grid > (int64_t)sms * per_sm) grid = (int64_t)sms * per_sm;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), smem, s, tk, tv, a);
}

template <int FMT, int D>
cudaError_t launch_fmt_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, cudaStream_t s) {
    const int G = a.num_q_heads / a.cache.num_kv_heads;
    cudaError_t e;
    if (a.ev_begin && (e = cudaEventRecord(a.ev_begin, s)) != cudaSuccess) return e;
    bool simt = false;
    DecodeArgs p = a;
    p.head_off = 0;
    p.heads = G;
    if constexpr (FMT != INT4) {  // INT4 has the tensor-core consumer only
        if (a.kernel == kKindSimt) {
            simt = true;
            if (G == 1) e = launch_stream<FMT, D, SimtConsumer<FMT, D, 1>>(tk, tv, p, s);
            else if (G == 2) e = launch_stream<FMT, D, SimtConsumer<FMT, D, 2>>(tk, tv, p, s);
            else e = launch_stream<FMT, D, SimtConsumer<FMT, D, 4>>(tk, tv, p, s);
        }
    }
    if (!simt) {
        // The per-row tensor-core consumer's operand rows are (q-head, scale
        // group) pairs, eight per pass.  Kv-heads with more pairs take the
        // grouped consumer (one pass for all G q-heads), except INT4 with
        // 16-channel groups (head_dim 64): the 16-row consumer serves sixteen
        // pairs per pass, and a group of G q-heads with ng scale groups per
        // row takes ceil(G * ng / 16) launches over the same tiles, each
        // serving 16 / ng of the heads; only the first appends the newest rows
        // (the later ones read them from the cache).
        const int ng = a.cache.ngroups;
        if (G * ng <= 8) {
            if constexpr (FMT != INT4) {
                // one CTA of 12 warps per SM for 8-head groups when its shared memory fits
                const int wide_smem = Layout(2 * KVQ_MMA_WARPS, row_bytes(FMT, D), D,
                                             MmaConsumer<FMT, D, false, true>::kQGlobal ? 0 : G, a.batch, FMT == INT8,
                                             a.k_new != nullptr, ng).total + 1024;
                if (G == 8 && wide_smem <= 227 * 1024)
                    e = launch_stream<FMT, D, MmaConsumer<FMT, D, false, true>>(tk, tv, p, s);
                else
                    e = launch_stream<FMT, D, MmaConsumer<FMT, D>>(tk, tv, p, s);
            } else {
                e = launch_stream<FMT, D, MmaConsumer<FMT, D>>(tk, tv, p, s);
            }
        } else if (FMT == INT8 || (FMT == INT4 && D / ng >= 32)) {
            // one pass, a scale group per contraction slice and output m-tile
            // (groups are whole 16-byte chunks of a row: 16 INT8 or 32 INT4 channels)
            e = cudaErrorInvalidValue;
            if constexpr (FMT == INT8) {
                if (ng == 2) e = launch_stream<FMT, D, MmaGroupConsumer<FMT, D, 2>>(tk, tv, p, s);
                else e = launch_stream<FMT, D, MmaGroupConsumer<FMT, D, 4>>(tk, tv, p, s);
            } else if constexpr (FMT == INT4) {
                // 16-warp CTAs while their shared memory fits (it grows with the
                // batch: a fused call with four groups over more than ~3300
                // sequences does not fit), else 4-warp ones
                const bool narrow = Layout(KVQ_GA4_WARPS, row_bytes(FMT, D), D, 0, a.batch, true, a.k_new != nullptr,
                                           ng).total + 1024 > 227 * 1024;
                if (ng == 2) {
                    e = narrow ? launch_stream<FMT, D, MmaGroupConsumer<FMT, D, 2, true>>(tk, tv, p, s)
                               : launch_stream<FMT, D, MmaGroupConsumer<FMT, D, 2>>(tk, tv, p, s);
                } else if constexpr (D >= 128) {
                    e = narrow ? launch_stream<FMT, D, MmaGroupConsumer<FMT, D, 4, true>>(tk, tv, p, s)
                               : launch_stream<FMT, D, MmaGroupConsumer<FMT, D, 4>>(tk, tv, p, s);
                }
            }
        } else if constexpr (FMT == INT4 && D == 64) {
            const int per = 16 / ng;
            for (int h = 0; h < G && e == cudaSuccess; h += per) {
                p.head_off = h;
                p.heads = G - h < per ? G - h : per;
                if (h > 0) p.k_new = p.v_new = nullptr;
                e = launch_stream<FMT, D, MmaConsumer<FMT, D, true>>(tk, tv, p, s);
            }
        } else {
            e = cudaErrorInvalidValue;  // FP8 has no groups and at most 8 q-heads per kv-head
        }
    }
    if (e != cudaSuccess) return e;
    if (a.ev_end && (e = cudaEventRecord(a.ev_end, s)) != cudaSuccess) return e;
    const int64_t heads = (int64_t)a.batch * a.num_q_heads;
    return launch_pdl(decode_reduce_kernel<D>, dim3((unsigned)heads), dim3(kReduceWarps * 32), 0, s, a);
}

template <int FMT>
cudaError_t launch_fmt(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, cudaStream_t s) {
    return a.cache.head_dim == 64 ? launch_fmt_d<FMT, 64>(tk, tv, a, s) : launch_fmt_d<FMT, 128>(tk, tv, a, s);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    const int64_t rows = (int64_t)a.cache.num_blocks * a.cache.num_kv_heads * a.cache.block_size;
    CUtensorMap tk, tv;
    const int rb = row_bytes(a.cache.fmt, a.cache.head_dim);
    const int box_rows = a.cache.block_size >= kTile ? kTile : kBox;
    const bool int4 = a.cache.fmt == INT4;
    if (!make_tmap(&tk, a.cache.k_codes, rows, rb, box_rows, int4) ||
        !make_tmap(&tv, a.cache.v_codes, rows, rb, box_rows, int4))
        return cudaErrorInvalidValue;
    switch (a.cache.fmt) {
        case E4M3: return launch_fmt<E4M3>(tk, tv, a, s);
        case E5M2: return launch_fmt<E5M2>(tk, tv, a, s);
        case INT4: return launch_fmt<INT4>(tk, tv, a, s);
        default: return launch_fmt<INT8>(tk, tv, a, s);
    }
}

}  // namespace kvq
