// Single-token paged decode attention over the quantized KV cache.
//
// "Accelerating Inference with FP8 KV Cache" (intro): the KV cache is stored in
// FP8 and computation runs in FP16; here every product is fp16 x fp16 and every
// sum fp32.  The FP8 per-tensor scale ("FP8 Formats: E4M3 and E5M2") and the
// INT8 row scales ("[Feature] TurboMind support W8A8 or FP8 KV Cache", online
// INT8) are folded out of the dot products: logits take s_K, outputs take s_V.
//
// Work decomposition: one CTA per (context partition, kv-head, sequence).  All
// q-heads of a kv-head's group are processed by that CTA, so each cached byte
// is read from HBM once.  Inside a CTA:
//   * warp 4 (producer) copies 16-token tiles of one paged block -- K rows and
//     V rows of one kv-head -- into an 8-stage shared-memory ring with 2-D TMA
//     tile loads (cp.async.bulk.tensor, 128-byte swizzle for head_dim 128),
//     completion tracked by mbarriers; INT8 row scales ride along as 1-D bulk
//     copies;
//   * warps 0-3 (consumers) take tiles round-robin, dequantize in registers and
//     run QK^T, an online softmax (base-2) and PV, each warp with its own
//     running (max, sum, accumulator);
//   * at the end the four warp states are merged in shared memory and written
//     either as the final fp16 output (one partition) or as a partial
//     (max, sum, unnormalised accumulator) that decode_reduce_kernel combines.
// Two consumer families:
//   * kKindSimt: CUDA cores; 16 head-dim values per lane, warp-shuffle dot
//     reductions, group size <= 4;
//   * kKindMma: tensor cores via mma.sync m16n8k16 (f16 in, fp32 accumulate).
//     QK^T is computed transposed (S^T = Q K^T with the q-group padded to 16
//     rows, 8 tokens per n8 tile) so that its accumulator fragment is already
//     the B operand of PV (out^T = V^T P^T, head_dim as M).  The contraction
//     index (head_dim for QK, tokens for PV) is permuted so that every thread
//     loads contiguous 16-byte runs; Q is permuted the same way.
// Every wait is bounded (2 s); on timeout a kernel records the error and
// drains its copies in flight.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kTile = 16;        // tokens per stage
constexpr int kStages = 8;       // ring depth
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxPartition = 8192;
constexpr int kMaxBlkIds = kMaxPartition / 16;
constexpr int kMergeHeads = 8;   // heads per kv-head the merge area holds
constexpr float kLog2e = 1.4426950408889634f;

enum { kKindSimt = 1, kKindMma = 2 };

template <int D>
struct Smem {
    static constexpr int kTileBytes = kTile * D;                       // one K (or V) tile
    static constexpr int kStageRegion = kStages * 2 * kTileBytes;      // K tiles then V tiles
    static constexpr int kScaleOff = kStageRegion;                     // fp32 [stages][2][16]
    static constexpr int kBarOff = kScaleOff + kStages * 2 * kTile * 4;
    static constexpr int kBlkOff = kBarOff + 2 * kStages * 8;
    static constexpr int kAbortOff = kBlkOff + kMaxBlkIds * 4;
    static constexpr int kBytes = kAbortOff + 16;
    static constexpr int kAlloc = kBytes + 1024;                       // alignment slack
    // merge area (aliases the stage region once the ring has drained)
    static constexpr int kMergeAcc = 0;                                // fp32 [warps][heads][D]
    static constexpr int kMergeM = kConsumerWarps * kMergeHeads * D * 4;
    static constexpr int kMergeL = kMergeM + kConsumerWarps * kMergeHeads * 4;
    static_assert(kMergeL + kConsumerWarps * kMergeHeads * 4 <= kStageRegion, "merge area too large");
};

// Byte offset of the 16-byte chunk `chunk` of tile row `row` inside a stage
// tile as the TMA wrote it: 128-byte swizzle (chunk ^ row % 8) for 128-byte
// rows, plain row-major for 64-byte rows.
template <int D>
__device__ __forceinline__ int tile_off(int row, int chunk) {
    if (D == 128) return row * 128 + ((chunk ^ (row & 7)) << 4);
    return row * D + (chunk << 4);
}

struct Ctx {
    uint8_t* k_tiles;
    uint8_t* v_tiles;
    float* scales;
    int valid;   // valid tokens in the current tile
    int stage;
};

// ---------------------------------------------------------------- SIMT --

template <int FMT, int D, int GM>
struct SimtConsumer {
    static constexpr int LPT = D / 16;     // lanes per token
    static constexpr int TPP = 32 / LPT;   // tokens per pass
    static constexpr int PASSES = kTile / TPP;
    uint32_t qh[GM][8];
    float m[GM], l[GM], acc[GM][16];
    int lane, j, grp, G;
    float qk_scale;

    __device__ void init(const DecodeArgs& a, int b, int kvh, int G_, float qks) {
        lane = threadIdx.x & 31;
        j = lane % LPT;
        grp = lane / LPT;
        G = G_;
        qk_scale = qks;
#pragma unroll
        for (int h = 0; h < GM; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[h][e] = 0.f;
            if (h < G) {
                const uint4* src = reinterpret_cast<const uint4*>(
                    a.q + ((int64_t)b * a.num_q_heads + (int64_t)kvh * G + h) * D + 16 * j);
                uint4 x0 = __ldg(src), x1 = __ldg(src + 1);
                qh[h][0] = x0.x; qh[h][1] = x0.y; qh[h][2] = x0.z; qh[h][3] = x0.w;
                qh[h][4] = x1.x; qh[h][5] = x1.y; qh[h][6] = x1.z; qh[h][7] = x1.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) qh[h][e] = 0u;
            }
        }
    }

    __device__ void tile(const Ctx& c) {
        const uint8_t* kt = c.k_tiles + c.stage * Smem<D>::kTileBytes;
        const uint8_t* vt = c.v_tiles + c.stage * Smem<D>::kTileBytes;
        const float* sk = c.scales + c.stage * 2 * kTile;
        const float* sv = sk + kTile;
        float z[PASSES][GM];
#pragma unroll
        for (int ps = 0; ps < PASSES; ++ps) {
            const int t = ps * TPP + grp;
            const uint4 kw = *reinterpret_cast<const uint4*>(kt + tile_off<D>(t, j));
            const uint32_t w[4] = {kw.x, kw.y, kw.z, kw.w};
            uint32_t kh[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                kh[2 * e] = dec_x2<FMT>((uint16_t)(w[e] & 0xFFFFu));
                kh[2 * e + 1] = dec_x2<FMT>((uint16_t)(w[e] >> 16));
            }
            const float ts = (FMT == INT8 ? sk[t] : 1.0f) * qk_scale;
#pragma unroll
            for (int h = 0; h < GM; ++h) {
                float d0 = 0.f, d1 = 0.f;
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    d0 = fma_f16x2_f32(qh[h][e], kh[e], d0);
                    d1 = fma_f16x2_f32(qh[h][e + 1], kh[e + 1], d1);
                }
                float d = d0 + d1;
#pragma unroll
                for (int off = LPT / 2; off > 0; off >>= 1) d += __shfl_xor_sync(0xFFFFFFFFu, d, off);
                z[ps][h] = t < c.valid ? d * ts : -INFINITY;
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
            uint4 vw = *reinterpret_cast<const uint4*>(vt + tile_off<D>(t, j));
            // rows past the context may hold any bytes (NaN codes too): zero them
            if (t >= c.valid) vw = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t w[4] = {vw.x, vw.y, vw.z, vw.w};
            const float vs = (FMT == INT8 && t < c.valid) ? sv[t] : 1.0f;
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

    // Sum the per-group partials and store this warp's state for the merge.
    __device__ void finish(float* macc, float* mm, float* ml, int warp) {
#pragma unroll
        for (int h = 0; h < GM; ++h) {
#pragma unroll
            for (int off = LPT; off < 32; off <<= 1) {
                l[h] += __shfl_xor_sync(0xFFFFFFFFu, l[h], off);
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[h][e] += __shfl_xor_sync(0xFFFFFFFFu, acc[h][e], off);
            }
            if (h < G && grp == 0) {
                float* dst = macc + ((warp * kMergeHeads) + h) * D + 16 * j;
#pragma unroll
                for (int e = 0; e < 16; e += 4)
                    *reinterpret_cast<float4*>(dst + e) = make_float4(acc[h][e], acc[h][e + 1], acc[h][e + 2], acc[h][e + 3]);
                if (j == 0) {
                    mm[warp * kMergeHeads + h] = m[h];
                    ml[warp * kMergeHeads + h] = l[h];
                }
            }
        }
    }
};

// ----------------------------------------------------------------- MMA --

template <int FMT, int D>
struct MmaConsumer {
    static constexpr int KS = D / 16;   // k-steps of QK^T
    static constexpr int DC = D / 4;    // K bytes per thread per token row
    static constexpr int KW = DC / 4;   // ... as 32-bit words (== KS)
    static constexpr int DV = D / 8;    // V bytes per thread per token row
    static constexpr int VW = DV / 4;
    static constexpr int MT = D / 16;   // m-tiles of PV (head_dim / 16)
    uint32_t qa[2 * KS];
    float acc[MT][4];
    float m, l;
    int lane, g, c, G;
    float qk_scale;

    __device__ void init(const DecodeArgs& a, int b, int kvh, int G_, float qks) {
        lane = threadIdx.x & 31;
        g = lane >> 2;
        c = lane & 3;
        G = G_;
        qk_scale = qks;
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int i = 0; i < MT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        // qa[2j] = Q[g][DC*c + 4j + {0,1}], qa[2j+1] = Q[g][DC*c + 4j + {2,3}]:
        // the DC halves Q[g][DC*c ...] in order.
        if (g < G) {
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + ((int64_t)b * a.num_q_heads + (int64_t)kvh * G + g) * D + DC * c);
#pragma unroll
            for (int i = 0; i < (2 * KS) / 4; ++i) {
                uint4 x = __ldg(src + i);
                qa[4 * i] = x.x; qa[4 * i + 1] = x.y; qa[4 * i + 2] = x.z; qa[4 * i + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 2 * KS; ++i) qa[i] = 0u;
        }
    }

    // K words of tile row `row`: the thread's DC contiguous bytes at DC*c.
    __device__ __forceinline__ void load_k(const uint8_t* kt, int row, uint32_t (&w)[KW]) {
        if (D == 128) {
            const uint4 x0 = *reinterpret_cast<const uint4*>(kt + tile_off<D>(row, 2 * c));
            const uint4 x1 = *reinterpret_cast<const uint4*>(kt + tile_off<D>(row, 2 * c + 1));
            w[0] = x0.x; w[1] = x0.y; w[2] = x0.z; w[3] = x0.w;
            w[4] = x1.x; w[5] = x1.y; w[6] = x1.z; w[7] = x1.w;
        } else {
            const uint4 x0 = *reinterpret_cast<const uint4*>(kt + tile_off<D>(row, c));
            w[0] = x0.x; w[1] = x0.y; w[2] = x0.z; w[3] = x0.w;
        }
    }

    // V words of tile row `row`: the thread's DV contiguous bytes at DV*g.
    __device__ __forceinline__ void load_v(const uint8_t* vt, int row, uint32_t (&w)[VW]) {
        if (D == 128) {
            const uint4 x = *reinterpret_cast<const uint4*>(vt + tile_off<D>(row, g));
            w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        } else {
            const uint2 x = *reinterpret_cast<const uint2*>(vt + row * D + DV * g);
            w[0] = x.x; w[1] = x.y;
        }
    }

    __device__ void tile(const Ctx& cx) {
        const uint8_t* kt = cx.k_tiles + cx.stage * Smem<D>::kTileBytes;
        const uint8_t* vt = cx.v_tiles + cx.stage * Smem<D>::kTileBytes;
        const float* sk = cx.scales + cx.stage * 2 * kTile;
        const float* sv = sk + kTile;
        // S^T: rows = q-heads (g), columns = tokens; half A = tokens 0..7 (this
        // thread's B operand row is token g), half B = tokens 8..15.
        float sA[4] = {0.f, 0.f, 0.f, 0.f}, sB[4] = {0.f, 0.f, 0.f, 0.f};
        {
            uint32_t kA[KW], kB[KW];
            load_k(kt, g, kA);
            load_k(kt, 8 + g, kB);
#pragma unroll
            for (int j = 0; j < KS; ++j) {
                mma_16816(sA, qa[2 * j], 0u, qa[2 * j + 1], 0u, dec_x2<FMT>((uint16_t)(kA[j] & 0xFFFFu)),
                          dec_x2<FMT>((uint16_t)(kA[j] >> 16)));
                mma_16816(sB, qa[2 * j], 0u, qa[2 * j + 1], 0u, dec_x2<FMT>((uint16_t)(kB[j] & 0xFFFFu)),
                          dec_x2<FMT>((uint16_t)(kB[j] >> 16)));
            }
        }
        // this thread's logits: head g, tokens 2c, 2c+1, 8+2c, 9+2c
        const int t0 = 2 * c, t1 = 2 * c + 1, t2 = 8 + 2 * c, t3 = 9 + 2 * c;
        float z0 = sA[0] * qk_scale, z1 = sA[1] * qk_scale, z2 = sB[0] * qk_scale, z3 = sB[1] * qk_scale;
        if (FMT == INT8) {
            z0 *= sk[t0]; z1 *= sk[t1]; z2 *= sk[t2]; z3 *= sk[t3];
        }
        if (cx.valid < kTile) {
            if (t0 >= cx.valid) z0 = -INFINITY;
            if (t1 >= cx.valid) z1 = -INFINITY;
            if (t2 >= cx.valid) z2 = -INFINITY;
            if (t3 >= cx.valid) z3 = -INFINITY;
        }
        float mx = fmaxf(fmaxf(z0, z1), fmaxf(z2, z3));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const float mn = fmaxf(m, mx);
        float alpha = 1.f, p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
        if (mn != -INFINITY) {
            alpha = fast_exp2(m - mn);
            p0 = fast_exp2(z0 - mn);
            p1 = fast_exp2(z1 - mn);
            p2 = fast_exp2(z2 - mn);
            p3 = fast_exp2(z3 - mn);
        }
        m = mn;
        l = l * alpha + ((p0 + p1) + (p2 + p3));
        if (FMT == INT8) {  // fold the V row scales into P (masked tokens keep p = 0)
            if (t0 < cx.valid) p0 *= sv[t0];
            if (t1 < cx.valid) p1 *= sv[t1];
            if (t2 < cx.valid) p2 *= sv[t2];
            if (t3 < cx.valid) p3 *= sv[t3];
        }
        // P^T as the B operand of PV: k = token, n = head g.  P is carried as
        // an fp16 pair hi + lo (lo = the fp16 residual of p - hi), so the PV
        // product keeps about 22 bits of each weight instead of 11: with
        // outlier channels the weighted mean of large V values can cancel, and a
        // single fp16 rounding of P would then show in the output.
        const uint32_t pb0 = pack_f16x2(p0, p1), pb1 = pack_f16x2(p2, p3);
        const float2 h01 = f16x2_to_f32x2(pb0), h23 = f16x2_to_f32x2(pb1);
        const uint32_t pl0 = pack_f16x2(p0 - h01.x, p1 - h01.y), pl1 = pack_f16x2(p2 - h23.x, p3 - h23.y);
        // rescale the accumulators: columns are heads 2c and 2c+1
        if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
            const float a0 = __shfl_sync(0xFFFFFFFFu, alpha, 8 * c);
            const float a1 = __shfl_sync(0xFFFFFFFFu, alpha, 8 * c + 4);
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                acc[i][0] *= a0; acc[i][1] *= a1; acc[i][2] *= a0; acc[i][3] *= a1;
            }
        }
        // out^T += V^T P^T.  A operand rows = head_dim DV*g + 2i (+1 for rows
        // g+8), columns = tokens 2c, 2c+1 | 8+2c, 9+2c.
        uint32_t v0[VW], v1[VW], v2[VW], v3[VW];
        load_v(vt, t0, v0);
        load_v(vt, t1, v1);
        load_v(vt, t2, v2);
        load_v(vt, t3, v3);
        if (cx.valid < kTile) {  // rows past the context may hold NaN codes: zero them
#pragma unroll
            for (int e = 0; e < VW; ++e) {
                if (t0 >= cx.valid) v0[e] = 0u;
                if (t1 >= cx.valid) v1[e] = 0u;
                if (t2 >= cx.valid) v2[e] = 0u;
                if (t3 >= cx.valid) v3[e] = 0u;
            }
        }
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
            const uint32_t x01 = prmt(v0[i >> 1], v1[i >> 1], sel);
            const uint32_t x23 = prmt(v2[i >> 1], v3[i >> 1], sel);
            const uint32_t a0 = dec_x2<FMT>((uint16_t)(x01 & 0xFFFFu)), a1 = dec_x2<FMT>((uint16_t)(x01 >> 16));
            const uint32_t a2 = dec_x2<FMT>((uint16_t)(x23 & 0xFFFFu)), a3 = dec_x2<FMT>((uint16_t)(x23 >> 16));
            mma_16816(acc[i], a0, a1, a2, a3, pb0, pb1);
            mma_16816(acc[i], a0, a1, a2, a3, pl0, pl1);
        }
    }

    __device__ void finish(float* macc, float* mm, float* ml, int warp) {
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);
        if (c == 0 && g < G) {
            mm[warp * kMergeHeads + g] = m;
            ml[warp * kMergeHeads + g] = l;
        }
        // acc[i][0..3] = out[head 2c | 2c+1][d = DV*g + 2i | DV*g + 2i + 1]
        const int h0 = 2 * c, h1 = 2 * c + 1;
#pragma unroll
        for (int i = 0; i < MT; ++i) {
            const int d = DV * g + 2 * i;
            if (h0 < G) *reinterpret_cast<float2*>(macc + (warp * kMergeHeads + h0) * D + d) = make_float2(acc[i][0], acc[i][2]);
            if (h1 < G) *reinterpret_cast<float2*>(macc + (warp * kMergeHeads + h1) * D + d) = make_float2(acc[i][1], acc[i][3]);
        }
    }
};

// -------------------------------------------------------------- kernel --

template <int FMT, int D, class Consumer>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                const __grid_constant__ CUtensorMap tmv,
                                                                const DecodeArgs a) {
    using S = Smem<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint8_t* k_tiles = smem;
    uint8_t* v_tiles = smem + kStages * S::kTileBytes;
    float* scales = reinterpret_cast<float*>(smem + S::kScaleOff);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
    uint64_t* empty = full + kStages;
    int* blk_ids = reinterpret_cast<int*>(smem + S::kBlkOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kAbortOff);

    const int p = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = a.cache.num_kv_heads, BS = a.cache.block_size;
    const int G = a.num_q_heads / Hkv;
    int ctx = a.context_lens[b];
    const int cap = min(a.max_context_len, a.max_blocks_per_seq * BS);
    if (ctx < 0 || ctx > cap) {
        if (threadIdx.x == 0 && p == 0 && kvh == 0) record_error(a.err, DEV_ERR_RANGE, ctx);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int P = a.partition_size;
    const int tok0 = p * P;
    if (a.num_parts > 1 && tok0 >= ctx) return;  // the reduce reads no partial here
    const int tok1 = min(tok0 + P, ctx);
    const int ntiles = tok1 > tok0 ? (tok1 - tok0 + kTile - 1) / kTile : 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer
        const int blk0 = tok0 / BS;
        const int nblk = ntiles ? (tok1 - 1) / BS - blk0 + 1 : 0;
        const int* bt = a.block_tables + (int64_t)b * a.max_blocks_per_seq + blk0;
        for (int i = lane; i < nblk; i += 32) {
            int id = bt[i];
            if (id < 0 || id >= a.cache.num_blocks) {
                record_error(a.err, DEV_ERR_RANGE, id);
                id = 0;  // keep the pipeline going on a block that exists
            }
            blk_ids[i] = id;
        }
        __syncwarp();
        if (lane == 0 && ntiles > 0) {
            prefetch_tmap(&tmk);
            prefetch_tmap(&tmv);
            const uint64_t pol = policy_evict_first();
            const uint32_t bytes = 2 * S::kTileBytes + (FMT == INT8 ? 2 * kTile * 4 : 0);
            int issued = 0;
            for (int i = 0; i < ntiles; ++i) {
                const int st = i % kStages;
                if (!mbar_wait(&empty[st], ((i / kStages) & 1) ^ 1, abort_flag)) {
                    record_error(a.err, DEV_ERR_TIMEOUT, 1);
                    *abort_flag = 1;
                    break;
                }
                const int tok = tok0 + i * kTile;
                const int blk = blk_ids[tok / BS - blk0];
                const int64_t row = ((int64_t)blk * Hkv + kvh) * BS + tok % BS;
                mbar_arrive_expect_tx(&full[st], bytes);
                tma_load_2d(k_tiles + st * S::kTileBytes, &tmk, 0, (int)row, &full[st], pol);
                tma_load_2d(v_tiles + st * S::kTileBytes, &tmv, 0, (int)row, &full[st], pol);
                if (FMT == INT8) {
                    bulk_load(scales + st * 2 * kTile, a.cache.k_scales + row, kTile * 4, &full[st], pol);
                    bulk_load(scales + st * 2 * kTile + kTile, a.cache.v_scales + row, kTile * 4, &full[st], pol);
                }
                issued = i + 1;
            }
            // let every copy this CTA started land before the CTA can exit
            for (int i = max(0, issued - kStages); i < issued; ++i)
                mbar_wait(&full[i % kStages], (i / kStages) & 1, nullptr);
        }
        return;
    }

    // --------------------------------------------------------- consumers
    const float s_fp8 = (FMT != INT8 && a.scale) ? __ldg(a.scale) : 1.0f;
    const float qk_scale = a.sm_scale * s_fp8 * kLog2e;
    Consumer cons;
    cons.init(a, b, kvh, G, qk_scale);
    Ctx cx{k_tiles, v_tiles, scales, 0, 0};
    for (int i = warp; i < ntiles; i += kConsumerWarps) {
        const int st = i % kStages;
        if (!mbar_wait(&full[st], (i / kStages) & 1, abort_flag)) {
            if (lane == 0) record_error(a.err, DEV_ERR_TIMEOUT, 2);
            *abort_flag = 1;
            break;
        }
        cx.stage = st;
        cx.valid = min(kTile, tok1 - (tok0 + i * kTile));
        cons.tile(cx);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    named_barrier_sync(1, kConsumerWarps * 32);  // every tile consumed: the ring is free
    float* macc = reinterpret_cast<float*>(smem + S::kMergeAcc);
    float* mm = reinterpret_cast<float*>(smem + S::kMergeM);
    float* ml = reinterpret_cast<float*>(smem + S::kMergeL);
    cons.finish(macc, mm, ml, warp);
    named_barrier_sync(1, kConsumerWarps * 32);

    const float s_out = FMT == INT8 ? 1.0f : s_fp8;
    for (int idx = threadIdx.x; idx < G * D; idx += kConsumerWarps * 32) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, (w < ntiles) ? mm[w * kMergeHeads + h] : -INFINITY);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                if (w >= ntiles) continue;
                const float mw = mm[w * kMergeHeads + h];
                if (mw == -INFINITY) continue;
                const float e = fast_exp2(mw - M);
                L += e * ml[w * kMergeHeads + h];
                O += e * macc[(w * kMergeHeads + h) * D + d];
            }
        }
        const int64_t hq = (int64_t)b * a.num_q_heads + (int64_t)kvh * G + h;
        if (a.num_parts == 1) {
            const float o = L > 0.f ? O * s_out / L : 0.f;
            a.out[hq * D + d] = __half_as_ushort(__float2half_rn(o));
        } else {
            a.ws[(hq * a.num_parts + p) * D + d] = O * s_out;
            if (d == 0) {
                float2* ml2 = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(a.ws) +
                                                        ws_acc_bytes(a.batch, a.num_q_heads, a.num_parts, D));
                ml2[hq * a.num_parts + p] = make_float2(M, L);
            }
        }
    }
}

// Combine the partials of every context partition of one (sequence, q-head):
// out = sum_i 2^(m_i - M) acc_i / sum_i 2^(m_i - M) l_i.
template <int D>
__global__ void __launch_bounds__(D) decode_reduce_kernel(const DecodeArgs a) {
    const int hq_local = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
    const int64_t hq = (int64_t)b * a.num_q_heads + hq_local;
    int ctx = a.context_lens[b];
    const int cap = min(a.max_context_len, a.max_blocks_per_seq * a.cache.block_size);
    ctx = ctx < 0 ? 0 : min(ctx, cap);
    const int np = min(a.num_parts, (ctx + a.partition_size - 1) / a.partition_size);
    const float2* ml2 = reinterpret_cast<const float2*>(reinterpret_cast<const uint8_t*>(a.ws) +
                                                        ws_acc_bytes(a.batch, a.num_q_heads, a.num_parts, D));
    float M = -INFINITY;
    for (int i = 0; i < np; ++i) M = fmaxf(M, ml2[hq * a.num_parts + i].x);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
        for (int i = 0; i < np; ++i) {
            const float2 v = ml2[hq * a.num_parts + i];
            if (v.x == -INFINITY) continue;
            const float e = fast_exp2(v.x - M);
            L += e * v.y;
            O += e * a.ws[(hq * a.num_parts + i) * D + d];
        }
    }
    const float o = L > 0.f ? O / L : 0.f;
    a.out[hq * D + d] = __half_as_ushort(__float2half_rn(o));
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
// box = one 16-token tile.
bool make_tmap(CUtensorMap* m, void* base, int64_t rows, int D) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)D};
    cuuint32_t box[2] = {(cuuint32_t)D, (cuuint32_t)kTile};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int FMT, int D, class Consumer>
cudaError_t launch_split(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, cudaStream_t s) {
    auto kern = decode_split_kernel<FMT, D, Consumer>;
    const int smem = Smem<D>::kAlloc;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.num_parts, a.cache.num_kv_heads, a.batch);
    kern<<<grid, kThreads, smem, s>>>(tk, tv, a);
    return cudaGetLastError();
}

template <int FMT, int D>
cudaError_t launch_fmt_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, cudaStream_t s) {
    const int G = a.num_q_heads / a.cache.num_kv_heads;
    cudaError_t e;
    if (a.kernel == kKindSimt) {
        if (G == 1) e = launch_split<FMT, D, SimtConsumer<FMT, D, 1>>(tk, tv, a, s);
        else if (G == 2) e = launch_split<FMT, D, SimtConsumer<FMT, D, 2>>(tk, tv, a, s);
        else e = launch_split<FMT, D, SimtConsumer<FMT, D, 4>>(tk, tv, a, s);
    } else {
        e = launch_split<FMT, D, MmaConsumer<FMT, D>>(tk, tv, a, s);
    }
    if (e != cudaSuccess || a.num_parts == 1) return e;
    decode_reduce_kernel<D><<<dim3(a.num_q_heads, a.batch), D, 0, s>>>(a);
    return cudaGetLastError();
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
    if (!make_tmap(&tk, a.cache.k_codes, rows, a.cache.head_dim) ||
        !make_tmap(&tv, a.cache.v_codes, rows, a.cache.head_dim))
        return cudaErrorInvalidValue;
    switch (a.cache.fmt) {
        case E4M3: return launch_fmt<E4M3>(tk, tv, a, s);
        case E5M2: return launch_fmt<E5M2>(tk, tv, a, s);
        default: return launch_fmt<INT8>(tk, tv, a, s);
    }
}

}  // namespace kvq
