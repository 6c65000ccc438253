// Causal attention of a chunk of new queries over the paged quantized cache
// (chunked prefill), on the fifth-generation tensor cores (tcgen05).
//
// "Accelerating Inference with FP8 KV Cache" (intro): the cache is stored in
// FP8 and computation runs in FP16.  Here the cached codes are dequantized
// exactly to fp16 operands (every FP8 value and every INT8 / INT4 code is an
// fp16 value), products are fp16 x fp16 and sums fp32.  The FP8 per-tensor
// scale ("FP8 Formats: E4M3 and E5M2") and the INT8 / INT4 row scales
// ("[Feature] TurboMind support W8A8 or FP8 KV Cache", online INT8 and the INT4
// named beside it) are folded out of the contractions: logits take s_K (per
// token for INT8 / INT4), the softmax weights take the s_V of their token, the
// output takes the FP8 s.
//
// Query i of an n-query chunk of a sequence with ctx cached tokens (the
// chunk's own K/V included) sits at position ctx - n + i and attends to every
// token t <= that position.
//
// Work decomposition.  A query tile is 128 rows: 128 / G consecutive queries
// of one (sequence, kv-head) times the G q-heads of that kv-head's group, so
// every K/V tile dequantized serves all G heads.  A CTA owns two consecutive
// query tiles of the same (sequence, kv-head) and walks the cache in KV tiles
// of 64 tokens up to the later tile's last position; both query tiles use each
// dequantized K/V tile, which halves the dequantization per product.  Roles
// (one CTA per SM: 480 threads, 512 tensor-memory columns, ~131 KB of shared
// memory):
//   * warps 9-14 (dequant): plain 16-byte loads of the tile's K and V codes
//     through the block table (L2 serves the other CTAs of the same
//     sequence), exact conversion to fp16, stores into the 128-byte-swizzled
//     layout the tensor core reads; positions past the last query are written
//     as zeros.  K runs one tile ahead of V, and the codes of the next tiles
//     are held in registers.  They also stage the two query tiles and the
//     INT8 / INT4 row scales;
//   * warp 8 (MMA): one elected lane issues, per KV tile j, S = Q K^T for each
//     query tile (M 128, N 64, K head_dim, into one of two S buffers of that
//     tile in tensor memory), then O += P V of tile j-1 for each query tile
//     (M 128, N head_dim, K 64, P read from tensor memory, V an MN-major
//     shared-memory operand), and commits each group to an mbarrier.  With
//     group scales (2.5x the MMAs) warps 8 and 15 issue for one query tile
//     each: the issue cost of tcgen05.mma is then the critical path, and two
//     issuing warps overlap it (+28% on the grouped INT4 shape);
//   * warps 0-3 and 4-7 (softmax of query tiles 0 and 1): thread r owns row r
//     (tensor-memory lane r): it reads its 64 logits with tcgen05.ld, keeps a
//     running maximum (raised only when the tile's maximum exceeds it by more
//     than 2^8, FA4's lazy rescaling, so weights stay below 256), rescales its
//     O row in tensor memory when the maximum moves, and writes the weights
//     back over its logits as fp16 hi + fp16 residual (two PV MMAs, ~22 bits
//     per weight).  At the end it normalises its O row and stores it as fp16.
// Tensor memory per query tile: two S / P buffers of 64 columns and 128 of O.
// Every wait is bounded (2 s); on timeout the CTA records the error, drains
// the MMAs it issued and exits.
#include <cuda_fp16.h>

#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
namespace {

constexpr int kRows = 128;        // query tile: (query, q-head) rows; a CTA holds two
constexpr int kKvTile = 64;       // tokens per KV tile
constexpr int kMmaWarp = 8;       // warps 0-7 softmax (4 per query tile), 8 MMA, 9-14 dequant
constexpr int kDqThreads = 192;   // dequantizing threads (warps 9-14)
constexpr int kMmaWarp2 = kMmaWarp + 1 + kDqThreads / 32;   // with group scales: query tile 1's MMA warp (15)
constexpr int kThreads = 32 * (kMmaWarp2 + 1);   // launched with one warp fewer without group scales
__host__ __device__ constexpr int threads_for(bool grp) { return grp ? kThreads : kThreads - 32; }
constexpr uint32_t kColsPerTile = 256;   // tensor-memory columns of one query tile
constexpr uint32_t kTmemCols = 2 * kColsPerTile;
constexpr uint32_t kColO = 128;   // a tile's O accumulator columns start here (two S buffers of 64 before)
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

// tcgen05.mma kind::f16, A and B from shared memory (mma_ss_warp) or A from
// tensor memory (mma_ts_warp), executed by a whole converged warp: elect.sync
// picks one lane (the lowest, the same every time) to issue, so the operands
// can stay warp-uniform.
__device__ __forceinline__ void mma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` (by the elected lane) when every tcgen05 operation that
// lane issued so far has completed.
__device__ __forceinline__ void mma_commit_warp(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
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

// After tcgen05.wait::ld: ties the loaded registers to this point so that no
// use of them is scheduled before the wait.
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]));
}

__device__ __forceinline__ void reg_fence32(uint32_t (&r)[32]) {
    uint32_t(&a)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[0]);
    uint32_t(&b)[16] = *reinterpret_cast<uint32_t(*)[16]>(&r[16]);
    reg_fence16(a);
    reg_fence16(b);
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

// fp16 pair (lo, hi) holding RN(p0), RN(p1) -> fp16 pair of the residuals
// RN(p0 - h0), RN(p1 - h1); each difference is one mixed-precision FMA (exact
// product h * -1, one rounding).
__device__ __forceinline__ uint32_t residual_f16x2(uint32_t h, float p0, float p1) {
    uint32_t r;
    asm("{\n\t.reg .f16 a, b, m1;\n\t.reg .f32 r0, r1;\n\t"
        "mov.b32 {a, b}, %1;\n\tmov.b16 m1, 0xBC00;\n\t"
        "fma.rn.f32.f16 r0, a, m1, %2;\n\tfma.rn.f32.f16 r1, b, m1, %3;\n\t"
        "cvt.rn.f16x2.f32 %0, r1, r0;\n\t}"
        : "=r"(r)
        : "r"(h), "f"(p0), "f"(p1));
    return r;
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
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

// Barriers.  Per-slot barriers serve tiles j with j % slots == slot; their
// phase for tile j is (j / slots) % 2.  S and P barriers exist per query tile.
enum Bar : int {
    B_KFULL0, B_KFULL1,    // dequant -> MMA: K tile in its buffer (kDqThreads arrivals)
    B_VFULL0, B_VFULL1,    // dequant -> MMA: V tile (kDqThreads)
    B_KFREE0, B_KFREE1,    // MMA -> dequant: both S = Q K^T done reading the K buffer (commit)
    B_VFREE0, B_VFREE1,    // MMA -> dequant, softmax: both O += P V done (commit)
    B_SFULL00, B_SFULL01,  // MMA -> softmax of query tile 0: S in its buffer 0 / 1 (commit)
    B_SFULL10, B_SFULL11,  // ... of query tile 1
    B_PFULL00, B_PFULL01,  // softmax of query tile 0 -> MMA: P written over S (128)
    B_PFULL10, B_PFULL11,  // ... of query tile 1
    B_SC0, B_SC1, B_SC2, B_SC3,  // dequant -> softmax: INT8 / INT4 row scales of the tile
    B_QREADY,              // softmax -> MMA: both query tiles in shared memory (256)
    B_OFINAL,              // every MMA done (commit)
    kNumBars
};

// Shared memory of one CTA (base 1024-byte aligned).  Operand tiles are
// [rows][D] fp16 stored as D / 64 column blocks of [rows][128 B], each with the
// 128-byte swizzle: the two query tiles (128 rows each; A of S = Q K^T,
// K-major), and two buffers each of K (64 rows; B of S, K-major) and V (64
// rows; B of O = P V, MN-major); with group scales (GRP) also two buffers each
// of the K and V residuals.
template <int D, bool GRP>
struct SmemLayout {
    static constexpr uint32_t kBlkQ = kRows * 128;         // one 64-column block of a query tile
    static constexpr uint32_t kBlkKV = kKvTile * 128;      // one 64-column block of a K / V tile
    static constexpr uint32_t kTileQ = kBlkQ * (D / 64);
    static constexpr uint32_t kTileKV = kBlkKV * (D / 64);
    static constexpr uint32_t kQ = 0;                      // two query tiles
    static constexpr uint32_t kK = kQ + 2 * kTileQ;        // two K buffers
    static constexpr uint32_t kV = kK + 2 * kTileKV;       // two V buffers
    static constexpr uint32_t kKlo = kV + 2 * kTileKV;     // GRP: two K residual buffers
    static constexpr uint32_t kVlo = kKlo + (GRP ? 2 * kTileKV : 0);   // GRP: two V residual buffers
    static constexpr uint32_t kKsc = kVlo + (GRP ? 2 * kTileKV : 0);   // fp32 [4][64] INT8 / INT4 logit multipliers
    static constexpr uint32_t kVsc = kKsc + 4 * kKvTile * 4;  // fp32 [4][64] INT8 / INT4 V row scales
    static constexpr uint32_t kBar = kVsc + 4 * kKvTile * 4;
    static constexpr uint32_t kTmemSlot = kBar + kNumBars * 8;
    static constexpr uint32_t kAbort = kTmemSlot + 4;
    static constexpr uint32_t kBytes = kAbort + 4;
    static constexpr uint32_t kAlloc = kBytes + 1024;      // slack for the 1024-byte alignment
};

// Byte offset, within an operand tile whose 64-column blocks are `blk` bytes
// apart, of the 8 fp16 values at columns 8c .. 8c+7 of row r.
__device__ __forceinline__ uint32_t tile_off(uint32_t blk, uint32_t r, uint32_t c) {
    return (c >> 3) * blk + sw128(r, c & 7u);
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
    int32_t ngroups;   // scales per cached row (INT8 / INT4 group quantization), else 1
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

// GRP: INT8 / INT4 with a scale per group of channels.  The group scale varies
// along the contraction of S = Q K^T (and along the output of P V), so it
// cannot be taken out per token as a row scale is: the dequantizers store each
// K and V value x = code * s_group as fp16 hi + fp16 residual (x exactly to
// ~22 bits), S takes two MMA passes (K hi, K residual) and O three (P hi V hi,
// P residual V hi, P hi V residual).
template <int FMT, int D, bool GRP>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const PrefillParams a) {
    using L = SmemLayout<D, GRP>;
    constexpr int kChunks = D / 8;       // 16-byte fp16 chunks per row
    // one scale per (token, kv-head) row, taken out of the contractions
    constexpr bool kRowScaled = (FMT == INT8 || FMT == INT4) && !GRP;
    constexpr int kRowBytes = row_bytes(FMT, D);
    constexpr int kCodeVecs = kRowBytes / 16;              // 16-byte code vectors per token row
    constexpr int kChunksPerVec = FMT == INT4 ? 4 : 2;     // 8-value fp16 chunks per code vector
    constexpr int kTileVecs = kKvTile * kCodeVecs;         // code vectors per K or V tile
    constexpr int kVecsPerThread = (kTileVecs + kDqThreads - 1) / kDqThreads;
    constexpr uint32_t kIdescQK = idesc_f16(kRows, kKvTile, 0);
    constexpr uint32_t kIdescPV = idesc_f16(kRows, D, 1);
    constexpr int kMmaWarps = GRP ? 2 : 1;

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
    const int TQ = kRows / G;                       // queries per query tile
    const int pair = (int)gridDim.x - 1 - (int)blockIdx.x;  // longest pairs first

    griddep_wait();
    const int q0 = a.query_start[b];
    const int n = a.query_start[b + 1] - q0;
    const int ctx = a.context_lens[b];
    if (2 * pair * TQ >= n) return;                 // uniform: this sequence has fewer queries
    if (n > ctx || n > a.max_query_len || q0 < 0 || (int64_t)q0 + n > a.num_q_tokens ||
        (int64_t)ctx > (int64_t)a.max_blocks_per_seq * a.block_size) {
        if (tid == 0) record_error(a.err, DEV_ERR_RANGE, b);
        return;
    }
    // Query tiles 2 * pair and 2 * pair + 1 (the second may hold no query).
    // Tile g covers queries qt_g * TQ .. + nq_g - 1, at positions p_first_g ..
    // p_last_g, and attends to KV tiles 0 .. nkv_g - 1; the K / V stream walks
    // the longer range, nkv.
    int nq[2], p_first[2], p_last[2], nkv_g[2];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const int qt = 2 * pair + g;
        nq[g] = max(0, min(TQ, n - qt * TQ));
        p_first[g] = ctx - n + qt * TQ;
        p_last[g] = p_first[g] + nq[g] - 1;
        nkv_g[g] = nq[g] > 0 ? p_last[g] / kKvTile + 1 : 0;
    }
    const int nkv = max(nkv_g[0], nkv_g[1]);
    const int p_max = nq[1] > 0 ? p_last[1] : p_last[0];   // last position any query attends to
    const float s_fp8 = ((FMT == E4M3 || FMT == E5M2) && a.scale) ? *a.scale : 1.0f;
    // logits in log2 units: S * c_k (FP8; K carries the scale's sign) or S * c_k * s_K[t] (INT8 / INT4)
    const float c_k = a.sm_scale * kLog2e * fabsf(s_fp8);

    if (tid == 0) {
        for (int i = 0; i < kNumBars; ++i) {
            const bool by_dq = (i >= B_KFULL0 && i <= B_VFULL1) || (i >= B_SC0 && i <= B_SC3);
            const bool by_sm = i >= B_PFULL00 && i <= B_PFULL11;
            const bool by_mma = (i >= B_KFREE0 && i <= B_VFREE1) || i == B_OFINAL;   // every MMA warp commits
            mbar_init(&bars[i], by_dq ? (uint32_t)kDqThreads : by_sm ? 128u : by_mma ? (uint32_t)kMmaWarps
                                 : i == B_QREADY ? 256u : 1u);
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

    if (warp == kMmaWarp || (kMmaWarps == 2 && warp == kMmaWarp2)) {
        // query tiles g0 .. g1 - 1: both, or with group scales (2.5x the MMAs;
        // their issue is then the critical path) one per MMA warp
        const int g0 = kMmaWarps == 2 && warp == kMmaWarp2 ? 1 : 0, g1 = kMmaWarps == 2 ? g0 + 1 : 2;
        // ---------------------------------------------------------- MMA ----
        // One elected lane issues every MMA, per KV tile j: S_0,j and S_1,j
        // (both query tiles against K_j, into S buffer j % 2 of each tile's
        // tensor-memory columns), then O_0 += P_0,j-1 V_j-1 and O_1 += P_1,j-1
        // V_j-1: S of tile j runs while the softmax of tile j-1 works on the
        // other buffers.  S_j overwrites the buffer that held P_j-2, which
        // O += P_j-2 V_j-2 (issued just before, by this thread) reads: the
        // tensor cores run one thread's products in issue order, so that read
        // precedes the write (a wait for its completion here would stall the
        // issue by a commit-to-waiter round trip, ~300-450 cycles, every tile).
        // A query tile takes no MMA for KV tiles past its last position.  The whole warp runs this code; elect.sync picks the issuing
        // lane, so descriptors stay warp-uniform.  Descriptors of the first
        // K-step of each operand tile; every other K-step adds a constant to the
        // 14-bit start-address field (addresses stay below 2^18 bytes, so the
        // field never carries).
        const uint64_t dk0 = smem_desc(sbase + L::kK, 16, 1024);
        const uint64_t dv0 = smem_desc(sbase + L::kV, L::kBlkKV, 1024);
        auto issue_qk = [&](int j) {
            const int sl = j & 1;
            if (j == 0 && !wait_or_abort(&bars[B_QREADY], 0, abort, a.err)) return false;
            if (!wait_or_abort(&bars[B_KFULL0 + sl], (j >> 1) & 1, abort, a.err)) return false;
            tc_fence_after();
            const uint64_t dk = dk0 + ((sl * L::kTileKV) >> 4);
            for (int g = g0; g < g1; ++g) {
                if (j >= (g ? nkv_g[1] : nkv_g[0])) continue;
                const uint64_t dq0 = smem_desc(sbase + L::kQ + g * L::kTileQ, 16, 1024);
                const uint32_t d_tmem = tmem + g * kColsPerTile + sl * kKvTile;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk & 3) * 32;
                    mma_ss_warp(d_tmem, dq0 + (((kk >> 2) * L::kBlkQ + off) >> 4),
                                dk + (((kk >> 2) * L::kBlkKV + off) >> 4), kIdescQK, kk > 0);
                }
                if (GRP) {   // + Q K_residual^T
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk & 3) * 32;
                        mma_ss_warp(d_tmem, dq0 + (((kk >> 2) * L::kBlkQ + off) >> 4),
                                    dk + (((L::kKlo - L::kK) + (kk >> 2) * L::kBlkKV + off) >> 4), kIdescQK, 1u);
                    }
                }
                mma_commit_warp(&bars[B_SFULL00 + 2 * g + sl]);
            }
            mma_commit_warp(&bars[B_KFREE0 + sl]);
            return true;
        };
        auto issue_pv = [&](int j) {
            const int sl = j & 1;
            if (!wait_or_abort(&bars[B_VFULL0 + sl], (j >> 1) & 1, abort, a.err)) return false;
            const uint64_t dv = dv0 + ((sl * L::kTileKV) >> 4);
            for (int g = g0; g < g1; ++g) {
                if (j >= (g ? nkv_g[1] : nkv_g[0])) continue;
                if (!wait_or_abort(&bars[B_PFULL00 + 2 * g + sl], (j >> 1) & 1, abort, a.err)) return false;
                tc_fence_after();
                const uint32_t o_tmem = tmem + g * kColsPerTile + kColO;
                const uint32_t p_tmem = tmem + g * kColsPerTile + sl * kKvTile;
#pragma unroll
                for (int kk = 0; kk < kKvTile / 16; ++kk) {
                    const uint32_t a_hi = p_tmem + 16 * kk;   // P of tokens 16kk .. 16kk+15
                    const uint64_t vd = dv + ((kk * 2048) >> 4);
                    mma_ts_warp(o_tmem, a_hi, vd, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
                    mma_ts_warp(o_tmem, a_hi + 8, vd, kIdescPV, 1u);
                    if (GRP) mma_ts_warp(o_tmem, a_hi, vd + ((L::kVlo - L::kV) >> 4), kIdescPV, 1u);
                }
            }
            mma_commit_warp(&bars[B_VFREE0 + sl]);
            return true;
        };
        bool mma_ok = true;
        for (int j = 0; j < nkv && mma_ok; ++j) {
            mma_ok = issue_qk(j);
            if (mma_ok && j >= 1) mma_ok = issue_pv(j - 1);
        }
        if (mma_ok && !*abort) issue_pv(nkv - 1);
        mma_commit_warp(&bars[B_OFINAL]);   // after every MMA this CTA issued
    } else if (warp > kMmaWarp) {
        // ------------------------------------------------------ dequant ----
        const int dt = tid - 32 * (kMmaWarp + 1);   // 0 .. kDqThreads - 1
        const int32_t* bt = a.block_tables + (size_t)b * a.max_blocks_per_seq;
        // Thread dt handles vectors e = it * kDqThreads + dt (e below
        // kTileVecs): the 16 codes c16 of token row u, with rows varying
        // fastest across groups of 8 lanes: each 8-lane group stores one 16-byte
        // column chunk of 8 consecutive rows, which the 128-byte swizzle spreads
        // over all 32 banks, and each warp load reads whole 32-byte sectors of 8
        // rows.
        auto has = [&](int it) { return it * kDqThreads + dt < kTileVecs; };
        auto row_of = [&](int it) {
            const int e = it * kDqThreads + dt;
            return ((e >> 3) / kCodeVecs) * 8 + (e & 7);
        };
        auto vec_of = [&](int it) { const int e = it * kDqThreads + dt; return (e >> 3) % kCodeVecs; };
        const int lbs = 31 - __clz(a.block_size);   // block sizes are powers of two
        int blk_k[kVecsPerThread];                  // physical block of each row of the tile whose K codes
                                                    // are loaded next, -1 = zeros
        int blk_v[kVecsPerThread];                  // the same for the tile whose V codes are loaded next
        // Block ids are loaded one iteration before they are used (fetch_raw),
        // and checked at that use (check_ids): the loads of a tile's codes then
        // wait on one global latency, not on the id load and the code load in
        // series.  kNoRow marks a row past the tile's last position.
        constexpr int kNoRow = (int)0x80000000;
        auto fetch_raw = [&](int j, int (&raw)[kVecsPerThread]) {
#pragma unroll
            for (int it = 0; it < kVecsPerThread; ++it) {
                const int t = j * kKvTile + row_of(it);
                raw[it] = (has(it) && j < nkv && t <= p_max) ? __ldg(bt + (t >> lbs)) : kNoRow;
            }
        };
        auto check_ids = [&](int (&blk)[kVecsPerThread]) {
#pragma unroll
            for (int it = 0; it < kVecsPerThread; ++it) {
                int id = blk[it];
                if (id == kNoRow) {
                    id = -1;
                } else if (id < 0 || id >= a.num_blocks) {
                    record_error(a.err, DEV_ERR_RANGE, id);
                    id = -1;
                }
                blk[it] = id;
            }
        };
        auto fetch_ids = [&](int j, int (&blk)[kVecsPerThread]) {
            fetch_raw(j, blk);
            check_ids(blk);
        };
        // GRP: a code vector's two 16-value halves (one for INT8) each lie in one
        // scale group (groups are at least 16 channels wide and 16-aligned)
        constexpr int kSubs = FMT == INT4 ? 2 : 1;
        constexpr int kVecDims = FMT == INT4 ? 32 : 16;   // head dims of one code vector
        const int ng = a.ngroups, gdims = D / ng;
        auto load_codes = [&](const uint8_t* codes, const float* scales, int j, uint4 (&cv)[kVecsPerThread],
                              float (&gs)[kVecsPerThread][kSubs], const int (&blk)[kVecsPerThread]) {
#pragma unroll
            for (int it = 0; it < kVecsPerThread; ++it) {
                const int t = j * kKvTile + row_of(it);
                cv[it] = make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int z = 0; z < kSubs; ++z) gs[it][z] = 0.f;
                if (blk[it] >= 0) {
                    const size_t row = ((size_t)blk[it] * Hkv + kvh) * a.block_size + (t & (a.block_size - 1));
                    cv[it] = ld_global_nc_v4(codes + row * kRowBytes + vec_of(it) * 16);
                    if (GRP) {
#pragma unroll
                        for (int z = 0; z < kSubs; ++z)
                            gs[it][z] = __ldg(scales + row * ng + (vec_of(it) * kVecDims + 16 * z) / gdims);
                    }
                }
            }
        };
        auto load_scales = [&](int j, float& ks, float& vs) {
            ks = vs = 0.f;
            const int t = j * kKvTile + dt;
            if (dt < kKvTile && t <= p_max) {
                const int id = bt[t >> lbs];
                if (id >= 0 && id < a.num_blocks) {
                    const size_t srow = ((size_t)id * Hkv + kvh) * a.block_size + (t & (a.block_size - 1));
                    ks = a.k_scales[srow];
                    vs = a.v_scales[srow];
                }
            }
        };
        // A negative FP8 scale is folded into K's fp16 signs, so the logit
        // multiplier is never negative.
        const uint32_t kflip = (!kRowScaled && s_fp8 < 0.f) ? 0x80008000u : 0u;
        // GRP: each fp16 code value c becomes x = c * s_group, stored as fp16 hi in
        // `tile` and the fp16 residual RN(x - hi) in `tile_lo`
        auto store_scaled = [&](uint32_t tile, uint32_t tile_lo, uint32_t off, const uint32_t (&hw)[4], float sc) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float2 c = f16x2_to_f32x2(hw[w]);
                const float x0 = c.x * sc, x1 = c.y * sc;
                hi[w] = pack_f16x2(x0, x1);
                lo[w] = residual_f16x2(hi[w], x0, x1);
            }
            st_shared_v4(tile + off, make_uint4(hi[0], hi[1], hi[2], hi[3]));
            st_shared_v4(tile_lo + off, make_uint4(lo[0], lo[1], lo[2], lo[3]));
        };
        auto store_tile = [&](uint32_t tile, uint32_t tile_lo, const uint4 (&cv)[kVecsPerThread],
                              const float (&gs)[kVecsPerThread][kSubs], uint32_t flip) {
#pragma unroll
            for (int it = 0; it < kVecsPerThread; ++it) {
                if (!has(it)) continue;
                const int u = row_of(it), c16 = vec_of(it);
                if (GRP) {
                    const uint32_t cw[4] = {cv[it].x, cv[it].y, cv[it].z, cv[it].w};
                    if (FMT == INT4) {   // 32 codes -> four 8-value chunks, two per scale half
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            uint32_t hw[4];
                            int4x8_to_f16(cw[w], hw);
                            store_scaled(tile, tile_lo, tile_off(L::kBlkKV, u, kChunksPerVec * c16 + w), hw,
                                         gs[it][w >> 1]);
                        }
                    } else {             // 16 INT8 codes -> two 8-value chunks
                        uint4 h0, h1;
                        dec16<FMT>(cv[it], h0, h1);
                        const uint32_t a0[4] = {h0.x, h0.y, h0.z, h0.w}, a1[4] = {h1.x, h1.y, h1.z, h1.w};
                        store_scaled(tile, tile_lo, tile_off(L::kBlkKV, u, 2 * c16), a0, gs[it][0]);
                        store_scaled(tile, tile_lo, tile_off(L::kBlkKV, u, 2 * c16 + 1), a1, gs[it][0]);
                    }
                    continue;
                }
                if (FMT == INT4) {   // 32 codes -> four 8-value chunks
                    uint32_t hw[4];
                    const uint32_t cw[4] = {cv[it].x, cv[it].y, cv[it].z, cv[it].w};
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        int4x8_to_f16(cw[w], hw);
                        st_shared_v4(tile + tile_off(L::kBlkKV, u, kChunksPerVec * c16 + w),
                                     make_uint4(hw[0], hw[1], hw[2], hw[3]));
                    }
                    continue;
                }
                uint4 h0, h1;
                dec16<FMT>(cv[it], h0, h1);
                if (flip) {
                    h0.x ^= flip; h0.y ^= flip; h0.z ^= flip; h0.w ^= flip;
                    h1.x ^= flip; h1.y ^= flip; h1.z ^= flip; h1.w ^= flip;
                }
                st_shared_v4(tile + tile_off(L::kBlkKV, u, 2 * c16), h0);
                st_shared_v4(tile + tile_off(L::kBlkKV, u, 2 * c16 + 1), h1);
            }
        };
        // Tile t goes to buffer t % 2 once the MMAs of tile t - 2 have read it.
        // K runs one tile ahead of V (K_{j+1} is stored before V_j), so the next
        // S never waits on the V side of the pipeline; the codes of the next K
        // and V tiles are loaded into registers meanwhile.
        uint4 kc[kVecsPerThread], vc[kVecsPerThread];
        float kg[kVecsPerThread][kSubs], vg[kVecsPerThread][kSubs];   // GRP: group scales of the codes
        float ks = 0.f, vs = 0.f;
        auto put_k = [&](int t) {
            const int sl = t & 1;
            if (t >= 2 && !wait_or_abort(&bars[B_KFREE0 + sl], ((t >> 1) - 1) & 1, abort, a.err)) return false;
            store_tile(sbase + L::kK + sl * L::kTileKV, sbase + L::kKlo + sl * L::kTileKV, kc, kg, kflip);
            if (kRowScaled && dt < kKvTile) {
                ksc[(t & 3) * kKvTile + dt] = ks * c_k;   // the logit multiplier of token t
                vsc[(t & 3) * kKvTile + dt] = vs;
            }
            fence_proxy_async();
            mbar_arrive(&bars[B_KFULL0 + sl]);
            if (kRowScaled) mbar_arrive(&bars[B_SC0 + (t & 3)]);
            return true;
        };
        int blk_n[kVecsPerThread];                  // raw block ids of the tile after blk_k's
        fetch_ids(0, blk_k);
        load_codes(a.k_codes, a.k_scales, 0, kc, kg, blk_k);
        load_codes(a.v_codes, a.v_scales, 0, vc, vg, blk_k);
        if (kRowScaled) load_scales(0, ks, vs);
        put_k(0);
        fetch_ids(1, blk_k);
        fetch_raw(2, blk_n);
        load_codes(a.k_codes, a.k_scales, 1, kc, kg, blk_k);
        if (kRowScaled) load_scales(1, ks, vs);
        for (int j = 0; j < nkv; ++j) {
            const int sl = j & 1;
            const bool more = j + 1 < nkv;
            if (more) {
                if (!put_k(j + 1)) break;
#pragma unroll
                for (int it = 0; it < kVecsPerThread; ++it) {
                    blk_v[it] = blk_k[it];   // tile j+1
                    blk_k[it] = blk_n[it];   // tile j+2, loaded an iteration ago
                }
                check_ids(blk_k);
                fetch_raw(j + 3, blk_n);
                load_codes(a.k_codes, a.k_scales, j + 2, kc, kg, blk_k);
                if (kRowScaled) load_scales(j + 2, ks, vs);
            }
            if (j >= 2 && !wait_or_abort(&bars[B_VFREE0 + sl], ((j >> 1) - 1) & 1, abort, a.err)) break;
            store_tile(sbase + L::kV + sl * L::kTileKV, sbase + L::kVlo + sl * L::kTileKV, vc, vg, 0u);
            fence_proxy_async();
            mbar_arrive(&bars[B_VFULL0 + sl]);
            if (more) load_codes(a.v_codes, a.v_scales, j + 1, vc, vg, blk_v);
        }
    } else {
        // ------------------------------------------------------ softmax ----
        // Warps 0-3 serve query tile 0, warps 4-7 query tile 1; thread r of a
        // group owns row r (tensor-memory lane r, reached by warp % 4).
        const int g = warp >> 2, r = tid & 127;
        const int nq_g = g ? nq[1] : nq[0], nkv_me = g ? nkv_g[1] : nkv_g[0];
        const bool rv = r < TQ * G && r / G < nq_g;
        const int pos = rv ? (g ? p_first[1] : p_first[0]) + r / G : (g ? p_last[1] : p_last[0]);
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16) + g * kColsPerTile;
        {
            // stage query row r of tile g = (query (2 * pair + g) * TQ + r / G,
            // head kvh * G + r % G) into the 128-byte-swizzled A operand (zeros
            // for rows without a query), while the dequant warps fetch the first
            // K / V tiles
            const uint4* src = reinterpret_cast<const uint4*>(
                a.q + ((size_t)(q0 + (2 * pair + g) * TQ + (rv ? r / G : 0)) * Hq + kvh * G + r % G) * D);
#pragma unroll
            for (int c0 = 0; c0 < kChunks; c0 += 8) {   // eight 16-byte loads in flight at a time
                uint4 v[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) v[c] = rv ? src[c0 + c] : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(sbase + L::kQ + g * L::kTileQ + tile_off(L::kBlkQ, r, c0 + c), v[c]);
            }
            fence_proxy_async();
            mbar_arrive(&bars[B_QREADY]);
        }
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv_me && ok; ++j) {
            const int sl = j & 1;
            if (!wait_or_abort(&bars[B_SFULL00 + 2 * g + sl], (j >> 1) & 1, abort, a.err)) { ok = false; break; }
            tc_fence_after();
            if (kRowScaled && !wait_or_abort(&bars[B_SC0 + (j & 3)], (j >> 2) & 1, abort, a.err)) {
                ok = false;
                break;
            }
            const float* ks = ksc + (j & 3) * kKvTile;
            const float* vs = vsc + (j & 3) * kKvTile;
            const uint32_t srow = trow + sl * kKvTile;   // this tile's S / P columns
            const int lim = pos - j * kKvTile;           // columns u <= lim attend
            // lane 0 holds the warp's first position: past it no column is masked
            const bool full = __shfl_sync(0xFFFFFFFFu, lim, 0) >= kKvTile - 1;
            // pass 1: the tile's row maximum; the second TMEM load overlaps the first chunk's work
            float mx = -INFINITY;
            // Both passes exist in two copies: tiles past the warp's first
            // position carry no masking code at all (masked tiles are the last
            // one or two of a query tile's walk).
            auto chunk_max = [&](const uint32_t (&sv)[32], int ch, auto masked) {
                // four independent three-input max chains of 8 values each (a
                // single chain of 64 two-input maxima was 14% slower on the 70B chunk)
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int q = 0; q < 32; q += 2) {
                    const int u = ch * 32 + q;
                    float x0 = kRowScaled ? __uint_as_float(sv[q]) * ks[u] : __uint_as_float(sv[q]);
                    float x1 = kRowScaled ? __uint_as_float(sv[q + 1]) * ks[u + 1] : __uint_as_float(sv[q + 1]);
                    if constexpr (decltype(masked)::value) {
                        x0 = u <= lim ? x0 : -INFINITY;
                        x1 = u + 1 <= lim ? x1 : -INFINITY;
                    }
                    m4[(q >> 1) & 3] = fmax3(m4[(q >> 1) & 3], x0, x1);
                }
                mx = fmax3(mx, fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            };
            auto pass1 = [&](auto masked) {
                uint32_t sa[32], sb[32];
                tmem_ld32(srow, sa);
                tc_wait_ld();
                reg_fence32(sa);
                tmem_ld32(srow + 32, sb);
                chunk_max(sa, 0, masked);
                tc_wait_ld();
                reg_fence32(sb);
                chunk_max(sb, 1, masked);
            };
            if (full) pass1(std::false_type{});
            else pass1(std::true_type{});
            if (!kRowScaled) mx *= c_k;
            const float m_new = fmaxf(m_used, mx);
            float alpha = 1.f;
            bool resc = false;
            if (m_new > m_used + kRescaleLog2) {
                alpha = fast_exp2(m_used - m_new);
                m_used = m_new;
                resc = true;
            }
            if (j > 0 && __any_sync(0xFFFFFFFFu, resc)) {
                // O must hold every earlier tile's product before it is rescaled
                const int jp = j - 1;
                if (!wait_or_abort(&bars[B_VFREE0 + (jp & 1)], (jp >> 1) & 1, abort, a.err)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int ch = 0; ch < D / 32; ++ch) {
                    uint32_t o[32];
                    tmem_ld32(trow + kColO + ch * 32, o);
                    tc_wait_ld();
                    reg_fence32(o);
#pragma unroll
                    for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
                    tmem_st32(trow + kColO + ch * 32, o);
                }
            }
            l *= alpha;
            // pass 2: weights, written over their logits as fp16 hi + residual
            const float neg_m = -m_used;
            float l2 = 0.f;                         // second partial sum (shorter add chains)
            auto chunk_p = [&](const uint32_t (&sv)[16], int ch, auto masked) {
                uint32_t hi[8], lo[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float pv[2], ev[2];
#pragma unroll
                    for (int z = 0; z < 2; ++z) {
                        const int u = ch * 16 + 2 * q + z;
                        float e = fast_exp2(fmaf(__uint_as_float(sv[2 * q + z]), kRowScaled ? ks[u] : c_k, neg_m));
                        if constexpr (decltype(masked)::value) {
                            if (u > lim) e = 0.f;
                        }
                        ev[z] = e;
                        pv[z] = kRowScaled ? e * vs[u] : e;
                    }
                    l += ev[0];
                    l2 += ev[1];
                    hi[q] = pack_f16x2(pv[0], pv[1]);
                    lo[q] = residual_f16x2(hi[q], pv[0], pv[1]);
                }
                // tokens 16c .. 16c+15 (read from columns 16c .. 16c+15) -> hi in
                // columns 16c .. 16c+7, lo in 16c+8 .. 16c+15
                tmem_st8(srow + ch * 16, hi);
                tmem_st8(srow + ch * 16 + 8, lo);
            };
            auto pass2 = [&](auto masked) {
                uint32_t sa[16], sb[16];
                tmem_ld16(srow, sa);
                tc_wait_ld();
                reg_fence16(sa);
                tmem_ld16(srow + 16, sb);
                chunk_p(sa, 0, masked);
                tc_wait_ld();
                reg_fence16(sb);
                tmem_ld16(srow + 32, sa);
                chunk_p(sb, 1, masked);
                tc_wait_ld();
                reg_fence16(sa);
                tmem_ld16(srow + 48, sb);
                chunk_p(sa, 2, masked);
                tc_wait_ld();
                reg_fence16(sb);
                chunk_p(sb, 3, masked);
            };
            if (full) pass2(std::false_type{});
            else pass2(std::true_type{});
            l += l2;
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(&bars[B_PFULL00 + 2 * g + sl]);
        }

        if (ok && nq_g > 0 && wait_or_abort(&bars[B_OFINAL], 0, abort, a.err)) {
            tc_fence_after();
            const float inv = s_fp8 / l;
            const int qi = r / G;
            uint16_t* orow =
                a.out + ((size_t)(q0 + (2 * pair + g) * TQ + (rv ? qi : 0)) * Hq + kvh * G + r % G) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t o[32];
                tmem_ld32(trow + kColO + ch * 32, o);
                tc_wait_ld();
                reg_fence32(o);
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

template <int FMT, int D, bool GRP>
cudaError_t launch_t(const PrefillArgs& x, cudaStream_t s) {
    constexpr uint32_t smem = SmemLayout<D, GRP>::kAlloc;
    static_assert(smem <= 227 * 1024, "shared memory of one CTA");
    auto kern = prefill_kernel<FMT, D, GRP>;
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
    p.ngroups = x.cache.ngroups;
    const int G = x.num_q_heads / x.cache.num_kv_heads;
    const int TQ = kRows / G;
    const int tiles = (x.max_query_len + TQ - 1) / TQ;
    const dim3 grid((unsigned)((tiles + 1) / 2), (unsigned)x.cache.num_kv_heads, (unsigned)x.batch);
    return launch_pdl(kern, grid, dim3(threads_for(GRP)), smem, s, p);
}

}  // namespace

int prefill_rows_per_tile() { return kRows; }

cudaError_t launch_prefill(const PrefillArgs& x, cudaStream_t s) {
    const int D = x.cache.head_dim;
    switch (x.cache.fmt) {
        case E4M3: return D == 64 ? launch_t<E4M3, 64, false>(x, s) : launch_t<E4M3, 128, false>(x, s);
        case E5M2: return D == 64 ? launch_t<E5M2, 64, false>(x, s) : launch_t<E5M2, 128, false>(x, s);
        case INT4:
            if (x.cache.ngroups > 1)
                return D == 64 ? launch_t<INT4, 64, true>(x, s) : launch_t<INT4, 128, true>(x, s);
            return D == 64 ? launch_t<INT4, 64, false>(x, s) : launch_t<INT4, 128, false>(x, s);
        default:
            if (x.cache.ngroups > 1)
                return D == 64 ? launch_t<INT8, 64, true>(x, s) : launch_t<INT8, 128, true>(x, s);
            return D == 64 ? launch_t<INT8, 64, false>(x, s) : launch_t<INT8, 128, false>(x, s);
    }
}

}  // namespace kvq
