// Internal interface between the C-ABI layer (kvq_api.cu) and the kernel
// translation units.  Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#ifdef __CUDACC__
#define KVQ_HD __host__ __device__
#else
#define KVQ_HD
#endif

namespace kvq {

// Tokens per work unit of the decode kernel (two 16-row TMA boxes); the
// host sizes chunks and workspaces in these units.
constexpr int kDecodeTileTokens = 32;

struct CacheView {
    uint8_t* k_codes;
    uint8_t* v_codes;
    float* k_scales;
    float* v_scales;
    int32_t num_blocks, block_size, num_kv_heads, head_dim, fmt;
    int32_t ngroups;  // scales per row: 1, or 2 / 4 for group quantization (FP8: 1)
};

struct AppendArgs {
    const uint16_t* k;  // fp16 bits [T][Hkv][D]
    const uint16_t* v;
    CacheView cache;
    const int64_t* slot_mapping;
    int64_t num_tokens;
    const float* scale;  // device, may be null (= 1.0)
    unsigned long long* err;
};

struct DequantArgs {
    CacheView cache;
    const int64_t* slots;
    int64_t num_slots;
    const float* scale;
    float* out_k;
    float* out_v;
    unsigned long long* err;
};

struct DecodeArgs {
    const uint16_t* q;  // fp16 bits [B][Hq][D]
    CacheView cache;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    int32_t batch, num_q_heads, max_context_len;
    const float* scale;  // device, may be null (= 1.0); FP8 only
    float sm_scale;      // resolved (> 0)
    uint16_t* out;       // fp16 bits [B][Hq][D]
    float* ws;           // chunk partials (layout below)
    int32_t chunk_tiles; // C: 32-token tiles per context chunk
    int32_t num_chunks;  // chunks per sequence at max_context_len
    int32_t kernel;      // 1 = CUDA-core, 2 = tensor-core
    unsigned long long* err;
    cudaEvent_t ev_begin, ev_end;  // optional: recorded around the main kernel
    const uint16_t* k_new;  // optional fp16 [B][Hkv][D]: newest token's K/V, appended in the launch
    const uint16_t* v_new;
    // q-heads of each kv-head's group served by one stream launch: heads
    // head_off .. head_off + heads - 1 (all of them unless the tensor-core
    // consumer needs more than one pass; set by launch_decode)
    int32_t head_off, heads;
};

struct PrefillArgs {
    const uint16_t* q;  // fp16 bits [num_q_tokens][Hq][D]
    CacheView cache;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    const int32_t* query_start;  // [batch + 1]
    int64_t num_q_tokens;
    int32_t batch, num_q_heads, max_query_len;
    const float* scale;  // device, may be null (= 1.0); FP8 only
    float sm_scale;      // resolved (> 0)
    uint16_t* out;       // fp16 bits [num_q_tokens][Hq][D]
    unsigned long long* err;
};

#ifdef __CUDACC__
// Launch with programmatic stream serialization: the kernel may be scheduled
// while the previous kernel on the stream finishes; it must call
// griddep_wait() before reading anything that kernel may have written.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
#endif

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);
cudaError_t launch_dequant(const DequantArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);
int prefill_rows_per_tile();  // (query, q-head) rows per CTA of the prefill kernel

// Workspace layout: every context chunk of every (sequence, q-head) has two
// partial slots (a chunk is streamed by at most two warps).  acc fp32
// [B][Hq][chunks][2][D] followed (256-byte aligned) by (m, l) fp32 pairs
// [B][Hq][chunks][2].
KVQ_HD inline size_t ws_acc_bytes(int64_t B, int64_t Hq, int64_t NCH, int64_t D) {
    return ((size_t)(B * Hq * NCH * 2 * D) * 4 + 255) / 256 * 256;
}
KVQ_HD inline size_t ws_bytes(int64_t B, int64_t Hq, int64_t NCH, int64_t D) {
    return ws_acc_bytes(B, Hq, NCH, D) + ((size_t)(B * Hq * NCH * 2) * 8 + 255) / 256 * 256;
}

}  // namespace kvq
