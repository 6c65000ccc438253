// Causal attention of a chunk of new queries over the paged quantized cache
// (chunked prefill), on the fifth-generation tensor cores (tcgen05).
//
// "Accelerating Inference with FP8 KV Cache" (intro): the cache is stored in
// FP8 and computation runs in FP16.  Here the cached codes are dequantized
// exactly to fp16 operands (every FP8 value and every INT8 code is an fp16
// value), products are fp16 x fp16 and sums fp32.  The FP8 per-tensor scale
// ("FP8 Formats: E4M3 and E5M2") and the INT8 row scales ("[Feature]
// TurboMind support W8A8 or FP8 KV Cache", online INT8) are folded out of the
// contractions: logits take s_K (per token for INT8), the softmax weights take
// the INT8 s_V of their token, the output takes the FP8 s.
//
// Query i of an n-query chunk of a sequence with ctx cached tokens (the
// chunk's own K/V included) sits at position ctx - n + i and attends to every
// token t <= that position.
//
// Work decomposition.  A CTA owns one M tile of 128 rows: 128 / G consecutive
// queries of one (sequence, kv-head) times the G q-heads of that kv-head's
// group, so every K/V tile a CTA dequantizes serves all G heads.  It walks the
// cache in KV tiles of 128 tokens up to the tile's last position.  Roles:
//   * warps 4-7 (dequant): plain 16-byte loads of the tile's K and V codes
//     through the block table (L2 serves the other M tiles of the same
//     sequence), exact conversion to fp16, stores into the 128-byte-swizzled
//     K-major layout the tensor core reads; positions past the tile's last
//     query are written as zeros.  They also stage the query tile and the INT8
//     row scales;
//   * thread 0 (also a softmax thread) issues S = Q K^T (M 128, N 128, K
//     head_dim) into tensor memory and O += P V (M 128, N head_dim, K 128)
//     with P read from tensor memory, V from shared memory as an MN-major
//     operand, and commits each group of MMAs to an mbarrier.  With one S
//     buffer, S of the next tile can only be computed after O += P V of this
//     one, so a dedicated issuing warp would wait at the same points;
//   * warps 0-3 (softmax): thread r owns row r (tensor-memory lane r): it reads
//     its 128 logits with tcgen05.ld, keeps a running maximum (raised only when
//     the tile's maximum exceeds it by more than 2^8, FA4's lazy rescaling, so
//     weights stay below 256), rescales its O row in tensor memory when the
//     maximum moves, and writes the weights back over its logits as fp16 hi +
//     fp16 residual (two PV MMAs, ~22 bits per weight).  At the end it
//     normalises its O row and stores it as fp16.
// Tensor memory per CTA: 128 columns of S / P and 128 of O (256 allocated), so
// two CTAs share an SM and one's softmax overlaps the other's MMAs.
// Every wait is bounded (2 s); on timeout the CTA records the error, drains
// the MMAs it issued and exits.
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kRows = 128;        // M tile: (query, q-head) rows
constexpr int kKvTile = 128;      // tokens per KV tile
constexpr int kThreads = 256;     // 4 softmax warps (thread 0 issues the MMAs), 4 dequant warps
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 128;   // O accumulator columns start here
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (weights < 2^8)

// ------------------------------------------------------------- tcgen05 ----

// Byte offset of (row, 16-byte chunk) in a [rows][128 B] tile with the 128-byte
// swizzle (rows grouped by 8 into 1024-byte atoms, chunk index XOR row % 8).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (>> 4), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, f16 A and B, A
// K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), N and M.
__host__ __device__ constexpr uint32_t idesc_f16(uint32_t m, uint32_t n, uint32_t b_mn) {
    return (1u << 4) | (b_mn << 16) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// Four INT8 codes (one 32-bit word) -> two f16x2 words, exact.
__device__ __forceinline__ void dec_int8x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t b = w ^ 0x80808080u;
    lo = int8_biased_pair_to_f16x2(prmt(b, 0u, 0x4140u));
    hi = int8_biased_pair_to_f16x2(prmt(b, 0u, 0x4342u));
}

// 16 codes (a uint4) -> 16 fp16 values (two uint4), exact.
template <int FMT>
__device__ __forceinline__ void dec16(const uint4& c, uint4& h0, uint4& h1) {
    if (FMT == INT8) {
        dec_int8x4(c.x, h0.x, h0.y);
        dec_int8x4(c.y, h0.z, h0.w);
        dec_int8x4(c.z, h1.x, h1.y);
        dec_int8x4(c.w, h1.z, h1.w);
    } else {
        dec_fp8x4<FMT>(c.x, h0.x, h0.y);
        dec_fp8x4<FMT>(c.y, h0.z, h0.w);
        dec_fp8x4<FMT>(c.z, h1.x, h1.y);
        dec_fp8x4<FMT>(c.w, h1.z, h1.w);
    }
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ------------------------------------------------------------- layout -----

enum Bar : int { B_KFULL, B_VFULL, B_SFULL, B_PFULL, B_KFREE, B_VFREE, B_OFINAL, B_SC0, B_SC1, kNumBars };

// Shared memory of one CTA (base 1024-byte aligned).  Operand tiles are
// [rows][D] fp16 stored as D / 64 column blocks of [rows][128 B], each with the
// 128-byte swizzle: the query tile (A of S = Q K^T, K-major), the K tile (B of
// S, K-major) and the V tile (B of O = P V, MN-major) share one layout.
template <int D>
struct SmemLayout {
    static constexpr uint32_t kBlk = kRows * 128;          // one 64-column block of 128 rows
    static constexpr uint32_t kTile = kBlk * (D / 64);     // a [128][D] fp16 tile
    static constexpr uint32_t kQ = 0;
    static constexpr uint32_t kK = kQ + kTile;
    static constexpr uint32_t kV = kK + kTile;
    static constexpr uint32_t kKsc = kV + kTile;           // fp32 [2][128] INT8 K row scales
    static constexpr uint32_t kVsc = kKsc + 2 * kKvTile * 4;
    static constexpr uint32_t kBar = kVsc + 2 * kKvTile * 4;
    static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kBytes = kAbort + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;      // slack for the 1024-byte alignment
};

// Byte offset, within an operand tile, of the 8 fp16 values at columns
// 8c .. 8c+7 of row r.
template <int D>
__device__ __forceinline__ uint32_t tile_off(uint32_t r, uint32_t c) {
    return (c >> 3) * SmemLayout<D>::kBlk + sw128(r, c & 7u);
}

struct PrefillParams {
    const uint16_t* q;
    const uint8_t* k_codes;
    const uint8_t* v_codes;
    const float* k_scales;
    const float* v_scales;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start;
    const float* scale;
    uint16_t* out;
    unsigned long long* err;
    int32_t num_blocks, block_size, num_kv_heads, max_blocks_per_seq;
    int32_t num_q_heads, max_query_len;
    int64_t num_q_tokens;
    float sm_scale;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              unsigned long long* err) {
    if (mbar_wait(bar, parity, abort)) return true;
    if (atomicExch((int*)abort, 1) == 0) record_error(err, DEV_ERR_TIMEOUT, 0);
    return false;
}

// ------------------------------------------------------------- kernel -----

template <int FMT, int D>
__global__ void __launch_bounds__(kThreads, 2) prefill_kernel(const PrefillParams a) {
    using L = SmemLayout<D>;
    constexpr int kChunks = D / 8;       // 16-byte fp16 chunks per row
    constexpr int kCodeVecs = D / 16;    // 16-byte code vectors per token row
    constexpr uint32_t kIdescQK = idesc_f16(kRows, kKvTile, 0);
    constexpr uint32_t kIdescPV = idesc_f16(kRows, D, 1);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(sm);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + L::kBar);
    float* ksc = reinterpret_cast<float*>(sm + L::kKsc);
    float* vsc = reinterpret_cast<float*>(sm + L::kVsc);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + L::kTmemSlot);
    volatile int* abort = reinterpret_cast<volatile int*>(sm + L::kAbort);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.z, kvh = blockIdx.y;
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads, G = Hq / Hkv;
    const int TQ = kRows / G;                       // queries per M tile
    const int qt = (int)gridDim.x - 1 - (int)blockIdx.x;  // longest tiles first

    griddep_wait();
    const int q0 = a.query_start[b];
    const int n = a.query_start[b + 1] - q0;
    const int ctx = a.context_lens[b];
    if (qt * TQ >= n) return;                       // uniform: this sequence has fewer queries
    if (n > ctx || n > a.max_query_len || q0 < 0 || (int64_t)q0 + n > a.num_q_tokens ||
        (int64_t)ctx > (int64_t)a.max_blocks_per_seq * a.block_size) {
        if (tid == 0) record_error(a.err, DEV_ERR_RANGE, b);
        return;
    }
    const int nq = min(TQ, n - qt * TQ);            // valid queries in this tile
    const int p_first = ctx - n + qt * TQ;          // position of its first query
    const int p_last = p_first + nq - 1;
    const int nkv = p_last / kKvTile + 1;           // KV tiles to walk
    const float s_fp8 = (FMT != INT8 && a.scale) ? *a.scale : 1.0f;

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const uint32_t cnt = (i == B_KFULL || i == B_VFULL || i == B_PFULL || i == B_SC0 || i == B_SC1) ? 128u : 1u;
            mbar_init(&bars[i], cnt);
        }
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 4) {
        // ------------------------------------------------------ dequant ----
        const int dt = tid - 128;
        const size_t head_stride = (size_t)a.block_size * D;
        const int32_t* bt = a.block_tables + (size_t)b * a.max_blocks_per_seq;
        // query tile: row r = (query qt*TQ + r / G, head kvh*G + r % G)
        for (int e = dt; e < kRows * kChunks; e += 128) {
            const int r = e / kChunks, c = e % kChunks;
            const int qi = r / G;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (r < TQ * G && qi < nq) {
                const size_t row = (size_t)(q0 + qt * TQ + qi) * Hq + kvh * G + r % G;
                v = *reinterpret_cast<const uint4*>(a.q + row * D + c * 8);
            }
            st_shared_v4(sbase + L::kQ + tile_off<D>(r, c), v);
        }
        // codes of K (which = 0) or V (which = 1) of KV tile j -> registers
        auto load_codes = [&](int j, int which, uint4 (&cv)[kCodeVecs]) {
            const uint8_t* codes = which ? a.v_codes : a.k_codes;
#pragma unroll
            for (int it = 0; it < kCodeVecs; ++it) {
                const int e = it * 128 + dt;
                const int u = e / kCodeVecs, c16 = e % kCodeVecs;
                const int t = j * kKvTile + u;
                cv[it] = make_uint4(0, 0, 0, 0);
                if (t <= p_last) {
                    const int blk = bt[t / a.block_size];
                    if (blk >= 0 && blk < a.num_blocks) {
                        cv[it] = ld_global_nc_v4(codes + ((size_t)blk * Hkv + kvh) * head_stride +
                                                 (size_t)(t % a.block_size) * D + c16 * 16);
                    } else if (c16 == 0 && which == 0) {
                        record_error(a.err, DEV_ERR_RANGE, blk);
                    }
                }
            }
        };
        auto store_tile = [&](uint32_t tile, const uint4 (&cv)[kCodeVecs]) {
#pragma unroll
            for (int it = 0; it < kCodeVecs; ++it) {
                const int e = it * 128 + dt;
                const int u = e / kCodeVecs, c16 = e % kCodeVecs;
                uint4 h0, h1;
                dec16<FMT>(cv[it], h0, h1);
                st_shared_v4(tile + tile_off<D>(u, 2 * c16), h0);
                st_shared_v4(tile + tile_off<D>(u, 2 * c16 + 1), h1);
            }
        };
        for (int j = 0; j < nkv; ++j) {
            uint4 cv[kCodeVecs];
            load_codes(j, 0, cv);
            float ks = 0.f, vs = 0.f;
            if (FMT == INT8) {
                const int t = j * kKvTile + dt;
                if (t <= p_last) {
                    const int blk = bt[t / a.block_size];
                    if (blk >= 0 && blk < a.num_blocks) {
                        const size_t srow = ((size_t)blk * Hkv + kvh) * a.block_size + t % a.block_size;
                        ks = a.k_scales[srow];
                        vs = a.v_scales[srow];
                    }
                }
            }
            if (j > 0 && !wait_or_abort(&bars[B_KFREE], (j - 1) & 1, abort, a.err)) break;
            store_tile(sbase + L::kK, cv);
            if (FMT == INT8) {
                ksc[(j & 1) * kKvTile + dt] = ks;
                vsc[(j & 1) * kKvTile + dt] = vs;
            }
            fence_proxy_async();
            mbar_arrive(&bars[B_KFULL]);
            if (FMT == INT8) mbar_arrive(&bars[B_SC0 + (j & 1)]);
            load_codes(j, 1, cv);
            if (j > 0 && !wait_or_abort(&bars[B_VFREE], (j - 1) & 1, abort, a.err)) break;
            store_tile(sbase + L::kV, cv);
            fence_proxy_async();
            mbar_arrive(&bars[B_VFULL]);
        }
    } else {
        // ------------------------------------------------------ softmax ----
        const int r = tid;
        const bool rv = r < TQ * G && r / G < nq;
        const int pos = rv ? p_first + r / G : p_last;
        const float c_k = a.sm_scale * kLog2e * s_fp8;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv && ok; ++j) {
            if (tid == 0 && wait_or_abort(&bars[B_KFULL], j & 1, abort, a.err)) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::kBlk + (kk & 3) * 32;
                    mma_ss(tmem, smem_desc(sbase + L::kQ + off, 16, 1024), smem_desc(sbase + L::kK + off, 16, 1024),
                           kIdescQK, kk > 0);
                }
                mma_commit(&bars[B_SFULL]);
                mma_commit(&bars[B_KFREE]);
            }
            __syncwarp();
            if (!wait_or_abort(&bars[B_SFULL], j & 1, abort, a.err)) { ok = false; break; }
            tc_fence_after();
            if (FMT == INT8 && !wait_or_abort(&bars[B_SC0 + (j & 1)], (j >> 1) & 1, abort, a.err)) {
                ok = false;
                break;
            }
            const float* ks = ksc + (j & 1) * kKvTile;
            const float* vs = vsc + (j & 1) * kKvTile;
            const int lim = pos - j * kKvTile;      // columns u <= lim attend
            uint32_t s[16];
            float mx = -INFINITY;
#pragma unroll 1
            for (int ch = 0; ch < kKvTile / 16; ++ch) {
                tmem_ld16(trow + ch * 16, s);
                tc_wait_ld();
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int u = ch * 16 + q;
                    const float x = __uint_as_float(s[q]) * (FMT == INT8 ? c_k * ks[u] : c_k);
                    if (u <= lim) mx = fmaxf(mx, x);
                }
            }
            const float m_new = fmaxf(m_used, mx);
            float alpha = 1.f;
            bool resc = false;
            if (m_new > m_used + kRescaleLog2) {
                alpha = fast_exp2(m_used - m_new);
                m_used = m_new;
                resc = true;
            }
            if (j > 0 && __any_sync(0xFFFFFFFFu, resc)) {
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(trow + kColO + ch * 32, o);
                    tc_wait_ld();
#pragma unroll
                    for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
                    tmem_st32(trow + kColO + ch * 32, o);
                }
            }
            l *= alpha;
#pragma unroll 1
            for (int ch = 0; ch < kKvTile / 16; ++ch) {
                tmem_ld16(trow + ch * 16, s);
                tc_wait_ld();
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float pv[2];
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const int u = ch * 16 + 2 * q + z;
                        const float x = __uint_as_float(s[2 * q + z]) * (FMT == INT8 ? c_k * ks[u] : c_k);
                        const float p = u <= lim ? fast_exp2(x - m_used) : 0.f;
                        l += p;
                        pv[z] = FMT == INT8 ? p * vs[u] : p;
                    }
                    const __half2 h = __floats2half2_rn(pv[0], pv[1]);
                    const float2 hf = __half22float2(h);
                    const __half2 rl = __floats2half2_rn(pv[0] - hf.x, pv[1] - hf.y);
                    hi[q] = *reinterpret_cast<const uint32_t*>(&h);
                    lo[q] = *reinterpret_cast<const uint32_t*>(&rl);
                }
                // tokens 16c .. 16c+15 (read from columns 16c .. 16c+15) -> hi in
                // columns 16c .. 16c+7, lo in 16c+8 .. 16c+15
                tmem_st8(trow + ch * 16, hi);
                tmem_st8(trow + ch * 16 + 8, lo);
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(&bars[B_PFULL]);
            if (tid == 0 && wait_or_abort(&bars[B_PFULL], j & 1, abort, a.err) &&
                wait_or_abort(&bars[B_VFULL], j & 1, abort, a.err)) {
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kKvTile / 16; ++kk) {
                    const uint32_t a_hi = tmem + 16 * kk;   // P of tokens 16kk .. 16kk+15
                    const uint64_t vd = smem_desc(sbase + L::kV + kk * 2048, L::kBlk, 1024);
                    mma_ts(tmem + kColO, a_hi, vd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_ts(tmem + kColO, a_hi + 8, vd, kIdescPV, 1u);
                }
                mma_commit(&bars[B_VFREE]);
            }
            __syncwarp();
        }
        if (tid == 0) mma_commit(&bars[B_OFINAL]);   // after every MMA this CTA issued
        __syncwarp();
        if (ok && wait_or_abort(&bars[B_OFINAL], 0, abort, a.err)) {
            tc_fence_after();
            const float inv = s_fp8 / l;
            const int qi = r / G;
            uint16_t* orow = a.out + ((size_t)(q0 + qt * TQ + (rv ? qi : 0)) * Hq + kvh * G + r % G) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t o[32];
                tmem_ld32(trow + kColO + ch * 32, o);
                tc_wait_ld();
                uint32_t h[16];
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    h[q] = pack_f16x2(__uint_as_float(o[2 * q]) * inv, __uint_as_float(o[2 * q + 1]) * inv);
                if (rv) {
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        *reinterpret_cast<uint4*>(orow + ch * 32 + w * 8) =
                            make_uint4(h[4 * w], h[4 * w + 1], h[4 * w + 2], h[4 * w + 3]);
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 0) {
        if (lane == 0) mbar_wait(&bars[B_OFINAL], 0, nullptr);   // every issued MMA has completed
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

template <int FMT, int D>
cudaError_t launch_t(const PrefillArgs& x, cudaStream_t s) {
    constexpr uint32_t smem = SmemLayout<D>::kAlloc;
    static_assert(smem <= 113 * 1024, "two CTAs per SM");
    auto kern = prefill_kernel<FMT, D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    PrefillParams p;
    p.q = x.q;
    p.k_codes = x.cache.k_codes;
    p.v_codes = x.cache.v_codes;
    p.k_scales = x.cache.k_scales;
    p.v_scales = x.cache.v_scales;
    p.block_tables = x.block_tables;
    p.context_lens = x.context_lens;
    p.query_start = x.query_start;
    p.scale = x.scale;
    p.out = x.out;
    p.err = x.err;
    p.num_blocks = x.cache.num_blocks;
    p.block_size = x.cache.block_size;
    p.num_kv_heads = x.cache.num_kv_heads;
    p.max_blocks_per_seq = x.max_blocks_per_seq;
    p.num_q_heads = x.num_q_heads;
    p.max_query_len = x.max_query_len;
    p.num_q_tokens = x.num_q_tokens;
    p.sm_scale = x.sm_scale;
    const int G = x.num_q_heads / x.cache.num_kv_heads;
    const int TQ = kRows / G;
    const dim3 grid((unsigned)((x.max_query_len + TQ - 1) / TQ), (unsigned)x.cache.num_kv_heads, (unsigned)x.batch);
    return launch_pdl(kern, grid, dim3(kThreads), smem, s, p);
}

}  // namespace

int prefill_rows_per_tile() { return kRows; }

cudaError_t launch_prefill(const PrefillArgs& x, cudaStream_t s) {
    const int D = x.cache.head_dim;
    switch (x.cache.fmt) {
        case E4M3: return D == 64 ? launch_t<E4M3, 64>(x, s) : launch_t<E4M3, 128>(x, s);
        case E5M2: return D == 64 ? launch_t<E5M2, 64>(x, s) : launch_t<E5M2, 128>(x, s);
        default: return D == 64 ? launch_t<INT8, 64>(x, s) : launch_t<INT8, 128>(x, s);
    }
}

}  // namespace kvq
