// Device-side building blocks of the kvq library (sm_103a): FP8 / INT8 codecs,
// mbarrier + TMA (cp.async.bulk) staging, bounded waits and the error word.
//
// Formats ("Accelerating Inference with FP8 KV Cache", section "FP8 Formats:
// E4M3 and E5M2"; OCP E4M3FN and E5M2):  quantize = round-to-nearest-even with
// saturation to the largest finite value, done by the hardware conversion
// cvt.rn.satfinite.{e4m3x2,e5m2x2}.f32; dequantize = the exact conversion
// cvt.rn.f16x2.{e4m3x2,e5m2x2} (every FP8 value is an fp16 value).
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace kvq {

enum Fmt : int { E4M3 = 1, E5M2 = 2, INT8 = 3, INT4 = 4 };

// Bytes of one cached (token, kv-head) row of head_dim values.
__host__ __device__ constexpr int row_bytes(int fmt, int D) { return fmt == INT4 ? D / 2 : D; }

// Error word codes (top byte of the 64-bit device error word).
enum DevErr : unsigned long long { DEV_ERR_RANGE = 1, DEV_ERR_TIMEOUT = 2 };

__device__ __forceinline__ void record_error(unsigned long long* err, unsigned long long code,
                                             long long detail) {
    unsigned long long v = (code << 56) | ((unsigned long long)detail & 0x00FFFFFFFFFFFFFFull);
    atomicCAS(err, 0ull, v);
}

// ------------------------------------------------------------------ codecs --

// Two fp32 values -> two FP8 codes (lo in bits 0..7, hi in bits 8..15).
template <int FMT>
__device__ __forceinline__ uint16_t enc_fp8x2(float lo, float hi) {
    uint16_t r;
    if (FMT == E4M3)
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two FP8 codes (lo byte, hi byte) -> f16x2 (lo half, hi half), exact.
template <int FMT>
__device__ __forceinline__ uint32_t dec_fp8x2(uint16_t two) {
    uint32_t r;
    if (FMT == E4M3)
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
    else
        asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(r) : "h"(two));
    return r;
}

// Four FP8 codes in a 32-bit word -> two f16x2 (bytes 0,1 -> lo; bytes 2,3 -> hi),
// both halves taken straight from the 32-bit register.
template <int FMT>
__device__ __forceinline__ void dec_fp8x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    if (FMT == E4M3)
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
    else
        asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
            "cvt.rn.f16x2.e5m2x2 %0, l;\n\tcvt.rn.f16x2.e5m2x2 %1, h;\n\t}"
            : "=r"(lo), "=r"(hi)
            : "r"(w));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Two signed INT8 codes sitting in bytes 0 and 2 of `biased_pair` (bytes 1 and
// 3 zero), each already XOR 0x80 (= code + 128) -> f16x2 of the exact integer
// values.  The byte becomes the low mantissa byte of 1024 + (code + 128), and
// subtracting 1152 is exact because every integer below 2048 is an fp16 value.
__device__ __forceinline__ uint32_t int8_biased_pair_to_f16x2(uint32_t biased_pair) {
    const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    uint32_t h = biased_pair | 0x64006400u;
    __half2 v = *reinterpret_cast<__half2*>(&h);
    v = __hsub2(v, off);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Eight packed INT4 codes (one 32-bit word; byte i holds channel 2i in its low
// nibble and 2i+1 in its high nibble, 4-bit two's complement) -> four f16x2
// words of 1032 + code (exact: XOR 0x8 turns each nibble into code + 8, which
// becomes the low mantissa bits of 1024).  Word i holds channels 2i, 2i+1.
__device__ __forceinline__ void int4x8_biased(uint32_t w, uint32_t (&h)[4]) {
    const uint32_t x = w ^ 0x88888888u;
    const uint32_t lo = x & 0x0F0F0F0Fu;          // channels 0, 2, 4, 6 (bytes 0..3)
    const uint32_t hi = (x >> 4) & 0x0F0F0F0Fu;   // channels 1, 3, 5, 7
    const uint32_t a = prmt(lo, hi, 0x5410u);     // [c0, c2, c1, c3]
    const uint32_t b = prmt(lo, hi, 0x7632u);     // [c4, c6, c5, c7]
    h[0] = prmt(a, 0x64646464u, 0x4240u);         // fp16 0x64.. | c0, 0x64.. | c1
    h[1] = prmt(a, 0x64646464u, 0x4341u);         // c2, c3
    h[2] = prmt(b, 0x64646464u, 0x4240u);         // c4, c5
    h[3] = prmt(b, 0x64646464u, 0x4341u);         // c6, c7
}

// The same with the bias removed: four f16x2 words of the exact codes.
__device__ __forceinline__ void int4x8_to_f16(uint32_t w, uint32_t (&h)[4]) {
    int4x8_biased(w, h);
    const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));  // 1032
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 v = *reinterpret_cast<__half2*>(&h[i]);
        v = __hsub2(v, off);
        h[i] = *reinterpret_cast<uint32_t*>(&v);
    }
}

// Codes in bytes (lo, hi) of a 16-bit value -> f16x2, for any format.
template <int FMT>
__device__ __forceinline__ uint32_t dec_x2(uint16_t two) {
    if (FMT == INT8) {
        uint32_t w = (uint32_t)two ^ 0x8080u;
        return int8_biased_pair_to_f16x2(prmt(w, 0u, 0x4140u));
    } else {
        return dec_fp8x2<FMT>(two);
    }
}

// a - b on two f16x2 words, round to nearest with subnormals kept (no flush
// to zero): exact wherever a, b and the difference are all multiples of 2^-24
// inside fp16's range, as for small integers times 2^-24.
__device__ __forceinline__ uint32_t hsub2_exact(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// d = c + a.lo * b.lo + a.hi * b.hi with f16 inputs and fp32 accumulation
// (a product of two fp16 values is exact in fp32).
__device__ __forceinline__ float fma_f16x2_f32(uint32_t a, uint32_t b, float c) {
    float d;
    asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t.reg .f32 t;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 t, al, bl, %3;\n\tfma.rn.f32.f16 %0, ah, bh, t;\n\t}"
        : "=f"(d)
        : "r"(a), "r"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
    __half2 v = *reinterpret_cast<__half2*>(&h);
    return __half22float2(v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// -------------------------------------------------------- mbarrier / TMA --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            smem_u32(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase (for a thread that polls several barriers).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: gives up after kWaitLimitNs (or as soon as *abort is set, when
// abort is not null) and returns false.  Every spin in this library goes
// through here.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort && *abort) return false;
            if (globaltimer_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

// 2-D tiled TMA load (box from the tensor map) into shared memory, completing
// its bytes on `bar`.  c0 = innermost coordinate (0 here), c1 = row.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int c0, int c1, uint64_t* bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// The same with the destination given as a 32-bit shared-memory address.
__device__ __forceinline__ void tma_load_2d_u32(uint32_t dst, const void* tmap, int c0, int c1, uint64_t* bar,
                                                uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void bulk_load_u32(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 2^x through the hardware approximation (relative error a few ulp of fp32).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel on the stream is still
// running; griddep_wait() blocks until that kernel has completed and its
// memory is visible, so it must precede every global read of data a previous
// kernel may have written.  griddep_launch() lets the next kernel start early.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// mma.sync m16n8k16, f16 inputs, fp32 accumulate (D = A * B + D).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace kvq
