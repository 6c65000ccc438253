// Debug gather + dequantize-on-read: the fp32 values the decode kernels see.
// FP8: fl32(decode(code) * scale) with the per-tensor scale ("Accelerating
// Inference with FP8 KV Cache", "FP8 Formats: E4M3 and E5M2"); INT8 and INT4:
// fl32(code * scale) with the row's scale, or its group's.  One thread per 16
// values of one (slot, kv-head) row.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

template <int FMT, int D>
__global__ void __launch_bounds__(kThreads) dequant_kernel(DequantArgs a) {
    constexpr int CPR = D / 16;
    const int Hkv = a.cache.num_kv_heads;
    const int64_t per = a.num_slots * Hkv * CPR;
    const int64_t idx = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int which = blockIdx.y;
    if (idx >= per) return;
    const int c = (int)(idx % CPR);
    const int64_t row = idx / CPR;  // slot index * Hkv + head
    const int64_t i = row / Hkv;
    const int h = (int)(row % Hkv);
    const int64_t slot = a.slots[i];
    const int64_t BS = a.cache.block_size;
    float* out = (which ? a.out_v : a.out_k) + row * D + c * 16;
    if (slot < 0 || slot >= (int64_t)a.cache.num_blocks * BS) {
        if (c == 0 && which == 0 && h == 0) record_error(a.err, DEV_ERR_RANGE, slot);
        return;
    }
    const int64_t src_row = ((slot / BS) * Hkv + h) * BS + slot % BS;
    const int ng = a.cache.ngroups;  // the chunk's 16 values lie in group c / (CPR / ng)
    const float s = (FMT == INT8 || FMT == INT4)
                        ? (which ? a.cache.v_scales : a.cache.k_scales)[src_row * ng + c / (CPR / ng)]
                        : (a.scale ? __ldg(a.scale) : 1.0f);
    if (FMT == INT4) {
        const uint2 r4 = *reinterpret_cast<const uint2*>((which ? a.cache.v_codes : a.cache.k_codes) +
                                                         src_row * (D / 2) + c * 8);
        uint32_t h[8];
        int4x8_to_f16(r4.x, *reinterpret_cast<uint32_t(*)[4]>(&h[0]));
        int4x8_to_f16(r4.y, *reinterpret_cast<uint32_t(*)[4]>(&h[4]));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 p0 = f16x2_to_f32x2(h[2 * j]), p1 = f16x2_to_f32x2(h[2 * j + 1]);
            reinterpret_cast<float4*>(out)[j] = make_float4(p0.x * s, p0.y * s, p1.x * s, p1.y * s);
        }
        return;
    }
    const uint4 r = *reinterpret_cast<const uint4*>((which ? a.cache.v_codes : a.cache.k_codes) +
                                                    src_row * D + c * 16);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
    float y[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float2 lo = f16x2_to_f32x2(dec_x2<FMT>((uint16_t)(w[j] & 0xFFFF)));
        float2 hi = f16x2_to_f32x2(dec_x2<FMT>((uint16_t)(w[j] >> 16)));
        y[4 * j] = lo.x * s;
        y[4 * j + 1] = lo.y * s;
        y[4 * j + 2] = hi.x * s;
        y[4 * j + 3] = hi.y * s;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        reinterpret_cast<float4*>(out)[j] = make_float4(y[4 * j], y[4 * j + 1], y[4 * j + 2], y[4 * j + 3]);
}

template <int FMT>
cudaError_t launch_fmt(const DequantArgs& a, cudaStream_t s) {
    const int D = a.cache.head_dim;
    const int64_t per = a.num_slots * a.cache.num_kv_heads * (D / 16);
    dim3 grid((unsigned)((per + kThreads - 1) / kThreads), 2);
    if (D == 64)
        dequant_kernel<FMT, 64><<<grid, kThreads, 0, s>>>(a);
    else
        dequant_kernel<FMT, 128><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

// Debug: the FP8 encoder of the append kernels (enc_fp8x2, the hardware
// cvt.rn.satfinite conversion) on raw fp32 values, so that it can be checked
// on every fp32 input.  One thread per 16 values (four 16-byte loads, one
// 16-byte store), grid-stride; the last n % 16 values one by one.
template <int FMT>
__global__ void __launch_bounds__(kThreads) encode_kernel(const float* x, uint8_t* codes, int64_t n) {
    const int64_t groups = n / 16;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    for (int64_t gi = (int64_t)blockIdx.x * kThreads + threadIdx.x; gi < groups; gi += stride) {
        const float4* src = reinterpret_cast<const float4*>(x) + 4 * gi;
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 v = src[j];
            o[j] = (uint32_t)enc_fp8x2<FMT>(v.x, v.y) | ((uint32_t)enc_fp8x2<FMT>(v.z, v.w) << 16);
        }
        reinterpret_cast<uint4*>(codes)[gi] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    const int64_t t = 16 * groups + (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (t < n) codes[t] = (uint8_t)(enc_fp8x2<FMT>(x[t], 0.f) & 0xFFu);
}

}  // namespace

cudaError_t launch_encode_fp8(const float* x, uint8_t* codes, int64_t n, int fmt, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int64_t want = (n / 16 + kThreads - 1) / kThreads;
    int64_t grid = want < (int64_t)sms * 8 ? want : (int64_t)sms * 8;
    if (grid < 1) grid = 1;
    if (fmt == E4M3)
        encode_kernel<E4M3><<<(unsigned)grid, kThreads, 0, s>>>(x, codes, n);
    else
        encode_kernel<E5M2><<<(unsigned)grid, kThreads, 0, s>>>(x, codes, n);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t s) {
    if (a.num_slots == 0) return cudaSuccess;
    switch (a.cache.fmt) {
        case E4M3: return launch_fmt<E4M3>(a, s);
        case E5M2: return launch_fmt<E5M2>(a, s);
        case INT4: return launch_fmt<INT4>(a, s);
        default: return launch_fmt<INT8>(a, s);
    }
}

}  // namespace kvq
