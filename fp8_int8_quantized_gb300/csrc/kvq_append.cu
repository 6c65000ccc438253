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

template <int FMT>
cudaError_t launch_fmt(const AppendArgs& a, cudaStream_t s) {
    const int D = a.cache.head_dim;
    const int64_t per = a.num_tokens * a.cache.num_kv_heads * (D / 16);
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
