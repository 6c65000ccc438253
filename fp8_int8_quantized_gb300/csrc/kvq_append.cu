// Quantize-on-write of fp16 K/V into the paged cache.
//
// "Accelerating Inference with FP8 KV Cache" (intro; "FP8 Formats: E4M3 and
// E5M2"; "FP8 E4M3 KV Cache"): the cache holds FP8 codes of x / scale with one
// fp32 per-tensor scale (1.0 when none is given).  "[Feature] TurboMind support
// W8A8 or FP8 KV Cache" (lmdeploy issue 1463): online INT8, here symmetric with
// one fp32 scale amax / 127 per (token, kv-head) row.
//
// HBM-bound: per element 2 bytes read, 1 byte written.  One thread handles 16
// consecutive elements of one (token, kv-head) row: two 16-byte loads of fp16,
// one 16-byte store of codes.  The D/16 threads of a row are adjacent lanes, so
// the INT8 row maximum is a shuffle reduction among them.
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;

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
    uint8_t* dst = (which ? a.cache.v_codes : a.cache.k_codes) + dst_row * D + c * 16;
    uint32_t o[4];
    if (FMT == INT8) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
        const unsigned lane = threadIdx.x & 31u;
        const unsigned gmask = (CPR == 32 ? 0xFFFFFFFFu : ((1u << CPR) - 1u) << (lane & ~(unsigned)(CPR - 1)));
#pragma unroll
        for (int off = CPR / 2; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(gmask, amax, off));
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
        if (c == 0) (which ? a.cache.v_scales : a.cache.k_scales)[dst_row] = s;
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

// FP8 append of large batches: every CTA first tabulates the code of all
// 65536 fp16 inputs for this call's scale -- RNE-satfinite(fl32(x / scale)),
// the same division and conversion as append_kernel, so the result is
// bit-identical -- into shared memory, then streams its share of (token,
// kv-head, 16-value chunk) units, K and V together, encoding every value with
// one shared-memory lookup instead of an IEEE division.
constexpr int kLutThreads = 512;
constexpr int kLutBytes = 65536;

template <int FMT, int D>
__global__ void __launch_bounds__(kLutThreads, 2) append_lut_kernel(AppendArgs a) {
    extern __shared__ __align__(16) uint8_t lut[];
    constexpr int CPR = D / 16;
    griddep_wait();
    griddep_launch();
    const float s = a.scale ? __ldg(a.scale) : 1.0f;
    for (int w = threadIdx.x; w < kLutBytes / 4; w += kLutThreads) {
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
    const uint32_t lut_base = smem_u32(lut);
    const int Hkv = a.cache.num_kv_heads;
    const int64_t BS = a.cache.block_size;
    const int64_t units = a.num_tokens * Hkv * CPR;
    for (int64_t idx = (int64_t)blockIdx.x * kLutThreads + threadIdx.x; idx < units;
         idx += (int64_t)gridDim.x * kLutThreads) {
        const int c = (int)(idx % CPR);
        const int64_t row = idx / CPR;  // token * Hkv + head
        const int64_t t = row / Hkv;
        const int h = (int)(row % Hkv);
        const int64_t slot = a.slot_mapping[t];
        if (slot == -1) continue;
        if (slot < 0 || slot >= (int64_t)a.cache.num_blocks * BS) {
            if (c == 0 && h == 0) record_error(a.err, DEV_ERR_RANGE, slot);
            continue;
        }
        const int64_t dst_row = ((slot / BS) * Hkv + h) * BS + slot % BS;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const uint4* src = reinterpret_cast<const uint4*>((which ? a.v : a.k) + row * D + c * 16);
            const uint4 r0 = __ldg(src), r1 = __ldg(src + 1);
            const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t b0, b1, b2, b3;
                asm volatile("ld.shared.u8 %0, [%1];" : "=r"(b0) : "r"(lut_base + (w[2 * i] & 0xFFFFu)));
                asm volatile("ld.shared.u8 %0, [%1];" : "=r"(b1) : "r"(lut_base + (w[2 * i] >> 16)));
                asm volatile("ld.shared.u8 %0, [%1];" : "=r"(b2) : "r"(lut_base + (w[2 * i + 1] & 0xFFFFu)));
                asm volatile("ld.shared.u8 %0, [%1];" : "=r"(b3) : "r"(lut_base + (w[2 * i + 1] >> 16)));
                o[i] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
            }
            uint8_t* dst = (which ? a.cache.v_codes : a.cache.k_codes) + dst_row * D + c * 16;
            *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// Values per call from which the tabulating kernel pays off (its table costs
// 65536 divisions per CTA).
constexpr int64_t kLutMinValues = (int64_t)1 << 22;

template <int FMT>
cudaError_t launch_fmt(const AppendArgs& a, cudaStream_t s) {
    const int D = a.cache.head_dim;
    const int64_t per = a.num_tokens * a.cache.num_kv_heads * (D / 16);
    if (FMT != INT8 && per * 32 >= kLutMinValues) {
        int dev = 0, sms = 0;
        cudaError_t e;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        auto kern = D == 64 ? append_lut_kernel<FMT, 64> : append_lut_kernel<FMT, 128>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kLutBytes)) != cudaSuccess)
            return e;
        const int64_t want = (per + kLutThreads - 1) / kLutThreads;
        const int64_t grid = want < (int64_t)sms * 2 ? want : (int64_t)sms * 2;
        return launch_pdl(kern, dim3((unsigned)grid), dim3(kLutThreads), kLutBytes, s, a);
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
        default: return launch_fmt<INT8>(a, s);
    }
}

}  // namespace kvq
