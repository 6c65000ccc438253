// Quantize-on-write of fp16 K/V into the paged cache.
//
// "Accelerating Inference with FP8 KV Cache" (intro; "FP8 Formats: E4M3 and
// E5M2"; "FP8 E4M3 KV Cache"): the cache holds FP8 codes of x / scale with one
// fp32 per-tensor scale (1.0 when none is given).  "[Feature] TurboMind support
// W8A8 or FP8 KV Cache" (lmdeploy issue 1463): online INT8, here symmetric with
// one fp32 scale amax / 127 per (token, kv-head) row; INT4 (named beside it)
// the same with amax / 7, codes in [-7, 7] packed two per byte (channel 2i in
// the low nibble).  Group quantization ("[QST] Scale factors and benchmarks",
// the QQQ page) cuts a row into 2 or 4 groups of channels with a scale each.
//
// HBM-bound: per element 2 bytes read, 1 byte written.  One thread handles 16
// consecutive elements of one (token, kv-head) row: two 16-byte loads of fp16,
// one 16-byte store of codes.  The D/16 threads of a row are adjacent lanes, so
// the INT8 / INT4 row (or group) maximum is a shuffle reduction among them.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

// Maximum of v over the cpg adjacent lanes of this lane's scale group (cpg a
// power of two dividing CPR; the CPR lanes of a row are aligned and all active).
template <int CPR>
__device__ __forceinline__ float group_max(float v, int cpg) {
    const unsigned lane = threadIdx.x & 31u;
    const unsigned rmask = (CPR == 32 ? 0xFFFFFFFFu : ((1u << CPR) - 1u) << (lane & ~(unsigned)(CPR - 1)));
#pragma unroll
    for (int off = CPR / 2; off > 0; off >>= 1)
        if (off < cpg) v = fmaxf(v, __shfl_xor_sync(rmask, v, off));
    return v;
}

template <int FMT, int D>
__global__ void __launch_bounds__(kThreads) append_kernel(AppendArgs a) {
    constexpr int CPR = D / 16;  // threads per row
    griddep_wait();
    griddep_launch();
    const int64_t per_tensor = a.num_tokens * a.cache.num_kv_heads * CPR;
    const int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int which = blockIdx.y;  // 0 = K, 1 = V
    if (idx >= per_tensor) return;
    const int c = (int)(idx % CPR);
    const int64_t row = idx / CPR;  // token * Hkv + head
    const int Hkv = a.cache.num_kv_heads;
    const int64_t t = row / Hkv;
    const int h = (int)(row % Hkv);
    const int64_t slot = a.slot_mapping[t];
    if (slot == -1) return;
    const int64_t BS = a.cache.block_size;
    if (slot < 0 || slot >= (int64_t)a.cache.num_blocks * BS) {
        if (c == 0 && which == 0 && h == 0) record_error(a.err, DEV_ERR_RANGE, slot);
        return;
    }
    const uint16_t* src = (which ? a.v : a.k) + row * D + c * 16;
    const uint4 r0 = __ldg(reinterpret_cast<const uint4*>(src));
    const uint4 r1 = __ldg(reinterpret_cast<const uint4*>(src) + 1);
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    float x[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float2 f = f16x2_to_f32x2(w[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
    }
    const int64_t dst_row = ((slot / BS) * Hkv + h) * BS + slot % BS;
    const int ng = a.cache.ngroups, cpg = CPR / ng;  // groups per row, threads per group
    if (FMT == INT4) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
        amax = group_max<CPR>(amax, cpg);
        const float s = __fdiv_rn(amax, 7.0f);
        uint32_t o4[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            int v = 0;
            if (s != 0.f) {
                v = __float2int_rn(__fdiv_rn(x[i], s));
                v = max(-7, min(7, v));
            }
            o4[i >> 3] |= (uint32_t)(v & 0xF) << (4 * (i & 7));   // channel 2j low nibble of byte j
        }
        uint8_t* dst4 = (which ? a.cache.v_codes : a.cache.k_codes) + dst_row * (D / 2) + c * 8;
        *reinterpret_cast<uint2*>(dst4) = make_uint2(o4[0], o4[1]);
        if (c % cpg == 0) (which ? a.cache.v_scales : a.cache.k_scales)[dst_row * ng + c / cpg] = s;
        return;
    }
    uint8_t* dst = (which ? a.cache.v_codes : a.cache.k_codes) + dst_row * D + c * 16;
    uint32_t o[4];
    if (FMT == INT8) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
        amax = group_max<CPR>(amax, cpg);
        const float s = __fdiv_rn(amax, 127.0f);
        int q[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            int v = 0;
            if (s != 0.f) {
                v = __float2int_rn(__fdiv_rn(x[i], s));
                v = max(-127, min(127, v));
            }
            q[i] = v & 0xFF;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = (uint32_t)q[4 * i] | ((uint32_t)q[4 * i + 1] << 8) | ((uint32_t)q[4 * i + 2] << 16) |
                   ((uint32_t)q[4 * i + 3] << 24);
        if (c % cpg == 0) (which ? a.cache.v_scales : a.cache.k_scales)[dst_row * ng + c / cpg] = s;
    } else {
        const float s = a.scale ? __ldg(a.scale) : 1.0f;
        if (s != 1.0f) {
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = __fdiv_rn(x[i], s);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t lo = enc_fp8x2<FMT>(x[4 * i], x[4 * i + 1]);
            uint32_t hi = enc_fp8x2<FMT>(x[4 * i + 2], x[4 * i + 3]);
            o[i] = lo | (hi << 16);
        }
    }
    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
}

// Division of 0 <= n < 2^31 by a divisor d fixed at launch, as a multiply-high
// and a shift (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, round-up multiplier with N = 31): with
// l = ceil(log2 d) and m = ceil(2^(31+l) / d) < 2^32, n / d = (n * m) >> (31 + l).
struct FastDiv {
    uint32_t d = 1, m = 0;
    int shift = 0;  // l - 1
    FastDiv() = default;
    explicit FastDiv(uint32_t d_) : d(d_) {
        int l = 0;
        while ((1ull << l) < d) ++l;
        if (d > 1) {
            m = (uint32_t)(((1ull << (31 + l)) + d - 1) / d);
            shift = l - 1;
        }
    }
    __device__ __forceinline__ uint32_t div(uint32_t n) const { return d == 1 ? n : __umulhi(n, m) >> shift; }
};

// FP8 append of large batches.  The code of x is RNE-satfinite(fl32(x /
// scale)); negating x negates the quotient and flips only the code's sign
// bit, so every CTA first tabulates the codes of the 32768 non-negative fp16
// patterns for this call's scale -- the same division and conversion as
// append_kernel, so the result is bit-identical -- in shared memory, then
// encodes each value with one byte lookup of its magnitude and an XOR of its
// sign into bit 7.  The CTA then streams its share of (token, kv-head,
// 16-value chunk) units, K and V together, two units per iteration with all
// four 32-byte loads issued before the first lookup.  (Quantizing from the
// reciprocal instead -- the IEEE division only for values within 2 fp32 ulps
// of a midpoint between codes -- with one satfinite conversion per two values
// was bit-identical but 2.3x slower on the Llama-3-70B chunk: the FP8
// conversion runs on a slow pipe.  The lookups are bound by the shared-memory
// pipe: 5.75 TB/s there.)
constexpr int kLutThreads = 512;
constexpr int kLutEntries = 32768;

// 16 fp16 values (8 words) -> 16 codes by table lookup
__device__ __forceinline__ uint4 lut_encode16(const uint4& r0, const uint4& r1, const uint8_t* lut) {
    const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = w[2 * i], b = w[2 * i + 1];
        const uint32_t codes = (uint32_t)lut[a & 0x7FFFu] | ((uint32_t)lut[(a >> 16) & 0x7FFFu] << 8) |
                               ((uint32_t)lut[b & 0x7FFFu] << 16) | ((uint32_t)lut[(b >> 16) & 0x7FFFu] << 24);
        const uint32_t signs = prmt(a, b, 0x7531u) & 0x80808080u;  // bit 15 of each half -> bit 7 of its byte
        o[i] = codes ^ signs;
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int FMT, int D>
__global__ void __launch_bounds__(kLutThreads, 2) append_lut_kernel(AppendArgs a, FastDiv by_heads) {
    extern __shared__ __align__(16) uint8_t lut[];
    constexpr int CPR = D / 16;  // units per row
    constexpr int LOG_CPR = D == 128 ? 3 : 2;
    griddep_wait();
    griddep_launch();
    const float s = a.scale ? __ldg(a.scale) : 1.0f;
    for (int w = threadIdx.x; w < kLutEntries / 4; w += kLutThreads) {
        uint32_t word = 0;
#pragma unroll
        for (int k = 0; k < 4; k += 2) {
            float x0 = __half2float(__ushort_as_half((uint16_t)(4 * w + k)));
            float x1 = __half2float(__ushort_as_half((uint16_t)(4 * w + k + 1)));
            if (s != 1.0f) {
                x0 = __fdiv_rn(x0, s);
                x1 = __fdiv_rn(x1, s);
            }
            word |= (uint32_t)enc_fp8x2<FMT>(x0, x1) << (8 * k);
        }
        reinterpret_cast<uint32_t*>(lut)[w] = word;
    }
    __syncthreads();
    const int Hkv = a.cache.num_kv_heads;
    const int BS = a.cache.block_size;  // 16, 32 or 64
    const int lbs = __ffs(BS) - 1;
    const int64_t nslots = (int64_t)a.cache.num_blocks * BS;
    const uint32_t units = (uint32_t)(a.num_tokens * Hkv * CPR);  // < 2^31 (checked by the launcher)
    const uint32_t stride = gridDim.x * kLutThreads;

    // one unit = chunk c of row (token t, head h): its K and V values and slot
    struct Unit {
        uint4 r[4];
        int64_t slot;
        uint32_t row;
    };
    auto load = [&](uint32_t u, Unit& x) {
        const uint4* k = reinterpret_cast<const uint4*>(a.k) + 2 * (int64_t)u;  // 16 fp16 = two uint4
        const uint4* v = reinterpret_cast<const uint4*>(a.v) + 2 * (int64_t)u;
        x.r[0] = __ldg(k);
        x.r[1] = __ldg(k + 1);
        x.r[2] = __ldg(v);
        x.r[3] = __ldg(v + 1);
        x.row = u >> LOG_CPR;
        x.slot = __ldg(a.slot_mapping + by_heads.div(x.row));
    };
    auto store = [&](uint32_t u, const Unit& x) {
        const int c = (int)(u & (CPR - 1));
        const int h = (int)(x.row - by_heads.div(x.row) * (uint32_t)Hkv);
        if (x.slot == -1) return;
        if (x.slot < 0 || x.slot >= nslots) {
            if (c == 0 && h == 0) record_error(a.err, DEV_ERR_RANGE, x.slot);
            return;
        }
        const int64_t dst = ((((x.slot >> lbs) * Hkv + h) << lbs) + (x.slot & (BS - 1))) * D + c * 16;
        *reinterpret_cast<uint4*>(a.cache.k_codes + dst) = lut_encode16(x.r[0], x.r[1], lut);
        *reinterpret_cast<uint4*>(a.cache.v_codes + dst) = lut_encode16(x.r[2], x.r[3], lut);
    };
    for (uint32_t u0 = blockIdx.x * kLutThreads + threadIdx.x; u0 < units; u0 += 2 * stride) {
        const uint32_t u1 = u0 + stride;
        Unit x0, x1;
        load(u0, x0);
        if (u1 < units) load(u1, x1);
        store(u0, x0);
        if (u1 < units) store(u1, x1);
    }
}

// rint(fl32(x / s)) for |x| <= amax and s = fl32(amax / qmax) (so |x / s|
// is at most qmax plus a few ulps), from the quotient by the reciprocal:
// y = fl32(x * r), r = fl32(1 / s), is within |x / s| * 2^-23 <= 1.6e-5 of
// x / s, and fl32(x / s) within half an ulp (<= 2^-18) of it, so y and
// fl32(x / s) round to the same integer unless a half-integer lies between
// them -- only possible when y is within 1.9e-5 of one.  Those rare values
// (y within 2^-14 of a half-integer) take the IEEE division instead, so the
// result is exactly the division's.
//
// The rounding itself is one fp32 addition: t = y + 1.5 * 2^23 lands in the
// binade where the ulp is 1, so it rounds y to the nearest integer, ties to
// even, and for |y| < 2^22 the bit pattern of t is 0x4B400000 + rint(y): its
// low byte is the INT8 code and its low nibble the INT4 code, in two's
// complement.  (This keeps the conversions off the slow transcendental /
// conversion pipe, which bounded the append at about half of HBM speed.)
// quant_t returns that bit pattern and flags a near half-integer.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kNearHalf = 0.5f - 6.103515625e-05f;

__device__ __forceinline__ uint32_t quant_t(float x, float r, bool& near) {
    const float y = x * r;
    const float t = y + kRoundMagic;
    near |= !(fabsf(y - (t - kRoundMagic)) <= kNearHalf);   // NaN (an Inf or NaN input) too
    return __float_as_uint(t);
}

// The same code by the IEEE division (the rare near-tie values, and
// non-finite inputs, as the division treats them).
__device__ __forceinline__ uint32_t quant_div(float x, float s, int qmax) {
    return (uint32_t)max(-qmax, min(qmax, __float2int_rn(__fdiv_rn(x, s))));
}

// INT8 / INT4 append of any batch: a persistent grid streams (token, kv-head,
// 16-value chunk) units, K and V together, two units per iteration with all
// eight 16-byte loads issued before the first row maximum.  The D/16 lanes of
// a row are adjacent (a unit's lane is its index mod 32, and D/16 divides 32),
// so the row (or group) maximum is a shuffle reduction among them, as in
// append_kernel; each value is quantized as quant_rint above (bit-identical to
// the division).
template <int FMT, int D>
__global__ void __launch_bounds__(kLutThreads, 2) append_rows_kernel(AppendArgs a, FastDiv by_heads) {
    constexpr int CPR = D / 16;  // units per row
    constexpr int LOG_CPR = D == 128 ? 3 : 2;
    constexpr float kQmax = FMT == INT4 ? 7.0f : 127.0f;
    constexpr int kQi = FMT == INT4 ? 7 : 127;
    griddep_wait();
    griddep_launch();
    const int Hkv = a.cache.num_kv_heads;
    const int BS = a.cache.block_size;  // 16, 32 or 64
    const int lbs = __ffs(BS) - 1;
    const int64_t nslots = (int64_t)a.cache.num_blocks * BS;
    const uint32_t units = (uint32_t)(a.num_tokens * Hkv * CPR);  // < 2^31 (checked by the launcher)
    const uint32_t stride = gridDim.x * kLutThreads;               // a multiple of 32: lanes keep their rows
    const int ng = a.cache.ngroups, cpg = CPR / ng;                // groups per row, units per group

    struct Unit {
        uint4 r[4];
        int64_t slot;
        uint32_t row;
    };
    auto load = [&](uint32_t u, Unit& x) {
        const uint4* k = reinterpret_cast<const uint4*>(a.k) + 2 * (int64_t)u;  // 16 fp16 = two uint4
        const uint4* v = reinterpret_cast<const uint4*>(a.v) + 2 * (int64_t)u;
        x.r[0] = __ldg(k);
        x.r[1] = __ldg(k + 1);
        x.r[2] = __ldg(v);
        x.r[3] = __ldg(v + 1);
        x.row = u >> LOG_CPR;
        x.slot = __ldg(a.slot_mapping + by_heads.div(x.row));
    };
    // quantize 16 values (two uint4 of fp16) with the row / group maximum of
    // their lanes; returns the scale; codes into o (INT8: 4 words, INT4: 2).
    // The maximum is taken on the fp16 pairs (|x| and max are exact in fp16),
    // and each output word is quantized and packed straight from its fp16
    // source words, so that few values are live at once.
    auto quant16 = [&](const uint4& r0, const uint4& r1, uint32_t (&o)[4]) -> float {
        const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
        __half2 m2 = __habs2(*reinterpret_cast<const __half2*>(&w[0]));
#pragma unroll
        for (int i = 1; i < 8; ++i) m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __half2*>(&w[i])));
        float amax = fmaxf(__low2float(m2), __high2float(m2));
        amax = group_max<CPR>(amax, cpg);
        const float s = __fdiv_rn(amax, kQmax);
        const float rs = s != 0.f ? __frcp_rn(s) : 0.f;   // s == 0: every t is the zero code
        constexpr int VPW = FMT == INT4 ? 8 : 4;            // values per output word
        constexpr int NW = 16 / VPW;
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            uint32_t t[VPW];
            bool near = false;
#pragma unroll
            for (int j = 0; j < VPW / 2; ++j) {
                const float2 f = f16x2_to_f32x2(w[k * (VPW / 2) + j]);
                t[2 * j] = quant_t(f.x, rs, near);
                t[2 * j + 1] = quant_t(f.y, rs, near);
            }
            if (near && s != 0.f) {  // rare: the values within 2^-14 of a half-integer, by division
#pragma unroll
                for (int j = 0; j < VPW / 2; ++j) {
                    const float2 f = f16x2_to_f32x2(w[k * (VPW / 2) + j]);
                    const float v2[2] = {f.x, f.y};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float y = v2[e] * rs;
                        if (!(fabsf(y - (__uint_as_float(t[2 * j + e]) - kRoundMagic)) <= kNearHalf))
                            t[2 * j + e] = quant_div(v2[e], s, kQi);
                    }
                }
            }
            if (FMT == INT4) {  // channel 2j: low nibble of byte j
                uint32_t b[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = (t[2 * j] & 0xFu) | ((t[2 * j + 1] & 0xFu) << 4);
                o[k] = prmt(prmt(b[0], b[1], 0x0040u), prmt(b[2], b[3], 0x0040u), 0x5410u);
            } else {  // byte j: the low byte of t
                o[k] = prmt(prmt(t[0], t[1], 0x0040u), prmt(t[2], t[3], 0x0040u), 0x5410u);
            }
        }
        if (FMT == INT4) o[2] = o[3] = 0u;
        return s;
    };
    auto store = [&](uint32_t u, const Unit& x) {
        const int c = (int)(u & (CPR - 1));
        uint32_t ok[4], ov[4];
        // every lane of the row quantizes (the maxima are shuffles among them),
        // also where the slot is skipped or out of range
        const float sk = quant16(x.r[0], x.r[1], ok);
        const float sv = quant16(x.r[2], x.r[3], ov);
        const int h = (int)(x.row - by_heads.div(x.row) * (uint32_t)Hkv);
        if (x.slot == -1) return;
        if (x.slot < 0 || x.slot >= nslots) {
            if (c == 0 && h == 0) record_error(a.err, DEV_ERR_RANGE, x.slot);
            return;
        }
        const int64_t dst_row = (((x.slot >> lbs) * Hkv + h) << lbs) + (x.slot & (BS - 1));
        if (FMT == INT4) {
            *reinterpret_cast<uint2*>(a.cache.k_codes + dst_row * (D / 2) + c * 8) = make_uint2(ok[0], ok[1]);
            *reinterpret_cast<uint2*>(a.cache.v_codes + dst_row * (D / 2) + c * 8) = make_uint2(ov[0], ov[1]);
        } else {
            *reinterpret_cast<uint4*>(a.cache.k_codes + dst_row * D + c * 16) = make_uint4(ok[0], ok[1], ok[2], ok[3]);
            *reinterpret_cast<uint4*>(a.cache.v_codes + dst_row * D + c * 16) = make_uint4(ov[0], ov[1], ov[2], ov[3]);
        }
        if (c % cpg == 0) {
            a.cache.k_scales[dst_row * ng + c / cpg] = sk;
            a.cache.v_scales[dst_row * ng + c / cpg] = sv;
        }
    };
    // All lanes of a warp run the same number of iterations of both halves:
    // the shuffles of the row maxima need every lane of a row, so a unit past
    // the end is loaded as zeros (never stored) instead of skipped.
    const uint32_t lane0 = blockIdx.x * kLutThreads + (threadIdx.x & ~31u);
    for (uint32_t base = lane0; base < units; base += 2 * stride) {
        const uint32_t u0 = base + (threadIdx.x & 31u), u1 = u0 + stride;
        Unit x0, x1;
        const bool v0 = u0 < units, v1 = u1 < units;
        if (v0) load(u0, x0); else x0 = Unit{{}, -1, 0};
        if (v1) load(u1, x1); else x1 = Unit{{}, -1, 0};
        store(u0, x0);
        if (base + stride < units) store(u1, x1);
    }
}

// Values per call from which the tabulating kernel pays off (its table costs
// 32768 divisions per CTA).
constexpr int64_t kLutMinValues = (int64_t)1 << 22;

template <int FMT>
cudaError_t launch_fmt(const AppendArgs& a, cudaStream_t s) {
    const int D = a.cache.head_dim;
    const int64_t per = a.num_tokens * a.cache.num_kv_heads * (D / 16);
    if constexpr (FMT == E4M3 || FMT == E5M2) {
        if (per * 32 >= kLutMinValues && per < ((int64_t)1 << 31)) {
            int dev = 0, sms = 0;
            cudaError_t e;
            if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
            if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
            auto kern = D == 64 ? append_lut_kernel<FMT, 64> : append_lut_kernel<FMT, 128>;
            if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLutEntries)) !=
                cudaSuccess)
                return e;
            const int64_t want = (per + kLutThreads - 1) / kLutThreads;
            const int64_t grid = want < (int64_t)sms * 2 ? want : (int64_t)sms * 2;
            return launch_pdl(kern, dim3((unsigned)grid), dim3(kLutThreads), kLutEntries, s, a,
                              FastDiv((uint32_t)a.cache.num_kv_heads));
        }
    }
    if constexpr (FMT == INT8 || FMT == INT4) {
        if (per < ((int64_t)1 << 31)) {
            int dev = 0, sms = 0;
            cudaError_t e;
            if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
            if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
            const int64_t want = (per + kLutThreads - 1) / kLutThreads;
            const int64_t grid = want < (int64_t)sms * 2 ? want : (int64_t)sms * 2;
            if (D == 64)
                return launch_pdl(append_rows_kernel<FMT, 64>, dim3((unsigned)grid), dim3(kLutThreads), 0, s, a,
                                  FastDiv((uint32_t)a.cache.num_kv_heads));
            return launch_pdl(append_rows_kernel<FMT, 128>, dim3((unsigned)grid), dim3(kLutThreads), 0, s, a,
                              FastDiv((uint32_t)a.cache.num_kv_heads));
        }
    }
    dim3 grid((unsigned)((per + kThreads - 1) / kThreads), 2);
    if (D == 64) return launch_pdl(append_kernel<FMT, 64>, grid, dim3(kThreads), 0, s, a);
    return launch_pdl(append_kernel<FMT, 128>, grid, dim3(kThreads), 0, s, a);
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
    if (a.num_tokens == 0) return cudaSuccess;
    switch (a.cache.fmt) {
        case E4M3: return launch_fmt<E4M3>(a, s);
        case E5M2: return launch_fmt<E5M2>(a, s);
        case INT4: return launch_fmt<INT4>(a, s);
        default: return launch_fmt<INT8>(a, s);
    }
}

}  // namespace kvq
