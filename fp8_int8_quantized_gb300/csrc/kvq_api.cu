// C ABI of the kvq library: argument validation, status codes, workspace
// sizing, context-split choice and the per-device error word.  Every entry
// point validates before it launches anything, so a call that returns an
// error has written nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "../../include/kvq.h"
#include "kvq_device.cuh"
#include "kvq_launch.h"

namespace kvq {
// The debug FP8 encoder's launcher (kvq_dequant.cu).
cudaError_t launch_encode_fp8(const float* x, uint8_t* codes, int64_t n, int fmt, cudaStream_t s);
}  // namespace kvq

namespace {

// First error a kernel met on this device: code << 56 | detail.
__device__ unsigned long long g_kvq_err = 0;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned long long* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
std::atomic<int> g_decode_kernel{0};
cudaEvent_t g_ev_begin = nullptr, g_ev_end = nullptr;

constexpr int kMaxChunkTokens = 65536;
constexpr int kMaxBatch = 4096;   // the decode kernel scans the context lengths in shared memory

bool current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return false;
    return *dev >= 0 && *dev < kMaxDevices;
}

unsigned long long* err_word(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kvq_err) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned long long*>(p);
    }
    return g_err_ptr[dev];
}

int sm_count(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_sm_count[dev] = n;
    }
    return g_sm_count[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kvq_status check_cache(const kvq_cache* c, int32_t fmt) {
    if (!c) return KVQ_ERR_INVALID_ARG;
    if (fmt != KVQ_E4M3 && fmt != KVQ_E5M2 && fmt != KVQ_INT8 && fmt != KVQ_INT4) return KVQ_ERR_INVALID_ARG;
    if (c->fmt != fmt) return KVQ_ERR_INVALID_ARG;
    if (!c->k_codes || !c->v_codes || !aligned(c->k_codes, 16) || !aligned(c->v_codes, 16))
        return KVQ_ERR_INVALID_ARG;
    if (c->num_blocks <= 0 || c->num_kv_heads <= 0) return KVQ_ERR_INVALID_ARG;
    if (c->head_dim != 64 && c->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
    if (c->block_size != 16 && c->block_size != 32 && c->block_size != 64) return KVQ_ERR_UNSUPPORTED;
    if (fmt == KVQ_INT8 || fmt == KVQ_INT4) {
        if (!c->k_scales || !c->v_scales || !aligned(c->k_scales, 16) || !aligned(c->v_scales, 16))
            return KVQ_ERR_INVALID_ARG;
        const int32_t g = c->group_size;
        if (g != 0 && g != c->head_dim && g != c->head_dim / 2 && g != c->head_dim / 4) return KVQ_ERR_INVALID_ARG;
    } else if (c->group_size != 0) {
        return KVQ_ERR_INVALID_ARG;
    }
    // TMA row coordinates are 32-bit
    if ((int64_t)c->num_blocks * c->num_kv_heads * c->block_size > 0x7FFFFFFFll) return KVQ_ERR_UNSUPPORTED;
    return KVQ_OK;
}

kvq::CacheView view(const kvq_cache* c) {
    const int32_t ng = c->group_size > 0 ? c->head_dim / c->group_size : 1;
    return kvq::CacheView{static_cast<uint8_t*>(c->k_codes), static_cast<uint8_t*>(c->v_codes), c->k_scales,
                          c->v_scales, c->num_blocks, c->block_size, c->num_kv_heads, c->head_dim, c->fmt, ng};
}

// Decode tiles (kDecodeTileTokens tokens) per context chunk.  Every warp of the persistent decode
// kernel streams a contiguous range of the flat tile list that is at least one
// chunk long; chunks of about half a range keep every warp busy while the
// partial slots stay few (two per chunk).  Counts 16 warps per SM (the kernel
// runs 12, and 16 for INT4), so chunks come out at 0.4-0.5 of a range.
int32_t choose_chunk_tiles(int32_t batch, int32_t num_kv_heads, int32_t group, int32_t max_ctx, int sms) {
    constexpr int TT = kvq::kDecodeTileTokens;
    const int64_t tiles = (int64_t)batch * num_kv_heads * ((max_ctx + TT - 1) / TT);
    const int64_t warps = (int64_t)sms * 16;
    int64_t c = tiles / (2 * warps);
    // Small batches: short chunks spread the few tiles over many warps; the
    // partial slots a chunk writes (G q-heads x head_dim + 2 floats, twice)
    // stay below ~1/8 of its cache bytes with at least G / 2 tiles per chunk,
    // and one-tile chunks cost more in flushes than they gain (Llama-2-7B
    // shapes at batch 4: 31 us per step against 27 with two-tile chunks).
    const int64_t cmin = group > 4 ? group / 2 : 2;
    if (c < cmin) c = cmin;
    if (c > 256) c = 256;
    return (int32_t)c;
}

int32_t resolve_chunk_tiles(int32_t partition_size, int32_t batch, int32_t num_kv_heads, int32_t group,
                            int32_t max_ctx) {
    if (partition_size > 0) return partition_size / kvq::kDecodeTileTokens;
    int dev = 0;
    if (!current_device(&dev)) dev = 0;
    return choose_chunk_tiles(batch, num_kv_heads, group, max_ctx, sm_count(dev));
}

kvq_status decode_impl(const void* q, const void* k_new, const void* v_new, const kvq_cache* cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                       int32_t batch, int32_t num_q_heads, int32_t max_context_len, const float* scale, int32_t fmt,
                       float sm_scale, void* out, void* workspace, size_t workspace_bytes, int32_t partition_size,
                       kvq_stream_t stream) {
    kvq_status st = check_cache(cache, fmt);
    if (st != KVQ_OK) return st;
    if (batch < 0 || num_q_heads <= 0 || max_context_len < 0 || max_blocks_per_seq <= 0) return KVQ_ERR_INVALID_ARG;
    if (num_q_heads % cache->num_kv_heads) return KVQ_ERR_INVALID_ARG;
    const int G = num_q_heads / cache->num_kv_heads;
    if (G > 8) return KVQ_ERR_UNSUPPORTED;
    // (the tensor-core consumer carries one operand row per (q-head, scale
    // group), eight per launch: more take several launches over the same tiles)
    if ((int64_t)max_blocks_per_seq * cache->block_size < max_context_len) return KVQ_ERR_INVALID_ARG;
    if (batch > 65535 || cache->num_kv_heads > 65535 || num_q_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    if (batch == 0) return KVQ_OK;
    if (!q || !block_tables || !context_lens || !out || !aligned(q, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return KVQ_ERR_INVALID_ARG;
    if (scale && !aligned(scale, 4)) return KVQ_ERR_INVALID_ARG;
    if (!(sm_scale >= 0.f) || std::isinf(sm_scale)) return KVQ_ERR_INVALID_ARG;
    if (partition_size < 0 || partition_size % 64 || partition_size > kMaxChunkTokens) return KVQ_ERR_INVALID_ARG;
    if (batch > kMaxBatch) return KVQ_ERR_UNSUPPORTED;
    constexpr int TT = kvq::kDecodeTileTokens;
    if ((int64_t)batch * cache->num_kv_heads * ((max_context_len + TT - 1) / TT) >= 0x7FFFFFFFll)
        return KVQ_ERR_UNSUPPORTED;  // flat tile indices are 32-bit
    const int32_t C = resolve_chunk_tiles(partition_size, batch, cache->num_kv_heads, G, max_context_len);
    const int32_t nch = std::max<int32_t>(1, ((max_context_len + TT - 1) / TT + C - 1) / C);
    const size_t need = kvq::ws_bytes(batch, num_q_heads, nch, cache->head_dim);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return KVQ_ERR_WORKSPACE;
    int kind = g_decode_kernel.load();
    if (kind == 0) kind = 2;
    // CUDA-core kernel: 8-bit codes, G <= 4
    if (kind == 1 && (G > 4 || fmt == KVQ_INT4)) return KVQ_ERR_UNSUPPORTED;
    int dev;
    if (!current_device(&dev)) return KVQ_ERR_CUDA;
    unsigned long long* err = err_word(dev);
    if (!err) return KVQ_ERR_CUDA;
    kvq::DecodeArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.cache = view(cache);
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.max_context_len = max_context_len;
    a.scale = (fmt == KVQ_INT8 || fmt == KVQ_INT4) ? nullptr : scale;
    a.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt((float)cache->head_dim);
    a.out = static_cast<uint16_t*>(out);
    a.ws = static_cast<float*>(workspace);
    a.chunk_tiles = C;
    a.num_chunks = nch;
    a.kernel = kind;
    a.err = err;
    a.ev_begin = g_ev_begin;
    a.ev_end = g_ev_end;
    a.k_new = static_cast<const uint16_t*>(k_new);
    a.v_new = static_cast<const uint16_t*>(v_new);
    return kvq::launch_decode(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

}  // namespace

extern "C" {

int32_t kvq_abi_version(void) { return KVQ_ABI_VERSION; }

const char* kvq_status_string(kvq_status s) {
    switch (s) {
        case KVQ_OK: return "ok";
        case KVQ_ERR_INVALID_ARG: return "invalid argument";
        case KVQ_ERR_UNSUPPORTED: return "unsupported size (head_dim, block_size or group size)";
        case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
        case KVQ_ERR_OUT_OF_RANGE: return "a slot, block id or context length was outside the cache";
        case KVQ_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
        case KVQ_ERR_CUDA: return "CUDA runtime error";
        case KVQ_ERR_SCRATCH_LIMIT: return "needs more scratch than the library's fixed device array";
    }
    return "unknown status";
}

void kvq_set_decode_timing_events(void* ev_begin, void* ev_end) {
    if (ev_begin && ev_end) {
        g_ev_begin = static_cast<cudaEvent_t>(ev_begin);
        g_ev_end = static_cast<cudaEvent_t>(ev_end);
    } else {
        g_ev_begin = g_ev_end = nullptr;
    }
}

int32_t kvq_set_decode_kernel(int32_t kind) {
    if (kind < 0 || kind > 2) return -1;
    return g_decode_kernel.exchange(kind);
}

kvq_status kvq_append(const void* k, const void* v, const kvq_cache* cache, const int64_t* slot_mapping,
                      int64_t num_tokens, const float* scale, int32_t fmt, kvq_stream_t stream) {
    kvq_status st = check_cache(cache, fmt);
    if (st != KVQ_OK) return st;
    if (num_tokens < 0) return KVQ_ERR_INVALID_ARG;
    if (num_tokens == 0) return KVQ_OK;
    if (!k || !v || !slot_mapping || !aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8))
        return KVQ_ERR_INVALID_ARG;
    if (scale && !aligned(scale, 4)) return KVQ_ERR_INVALID_ARG;
    if (num_tokens * cache->num_kv_heads * (cache->head_dim / 16) / 256 >= 0x7FFFFFFFll) return KVQ_ERR_UNSUPPORTED;
    int dev;
    if (!current_device(&dev)) return KVQ_ERR_CUDA;
    unsigned long long* err = err_word(dev);
    if (!err) return KVQ_ERR_CUDA;
    kvq::AppendArgs a{static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), view(cache), slot_mapping,
                      num_tokens, (fmt == KVQ_INT8 || fmt == KVQ_INT4) ? nullptr : scale, err};
    return kvq::launch_append(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

size_t kvq_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t max_context_len, int32_t partition_size) {
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
    if (num_q_heads % num_kv_heads) return 0;
    const int32_t C = resolve_chunk_tiles(partition_size, batch, num_kv_heads, num_q_heads / num_kv_heads,
                                          max_context_len);
    if (C <= 0) return 0;
    constexpr int TT = kvq::kDecodeTileTokens;
    const int64_t nch = std::max<int64_t>(1, ((max_context_len + TT - 1) / TT + C - 1) / C);
    return kvq::ws_bytes(batch, num_q_heads, nch, head_dim);
}

kvq_status kvq_decode_attention(const void* q, const kvq_cache* cache, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
                                int32_t num_q_heads, int32_t max_context_len, const float* scale, int32_t fmt,
                                float sm_scale, void* out, void* workspace, size_t workspace_bytes,
                                int32_t partition_size, kvq_stream_t stream) {
    return decode_impl(q, nullptr, nullptr, cache, block_tables, max_blocks_per_seq, context_lens, batch,
                       num_q_heads, max_context_len, scale, fmt, sm_scale, out, workspace, workspace_bytes,
                       partition_size, stream);
}

kvq_status kvq_decode_attention_append(const void* q, const void* k_new, const void* v_new, const kvq_cache* cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                       int32_t max_context_len, const float* scale, int32_t fmt, float sm_scale,
                                       void* out, void* workspace, size_t workspace_bytes, int32_t partition_size,
                                       kvq_stream_t stream) {
    if (batch > 0 && (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16))) return KVQ_ERR_INVALID_ARG;
    return decode_impl(q, k_new, v_new, cache, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                       max_context_len, scale, fmt, sm_scale, out, workspace, workspace_bytes, partition_size,
                       stream);
}

kvq_status kvq_prefill_attention(const void* q, const kvq_cache* cache, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens, const int32_t* query_start,
                                 int32_t batch, int64_t num_q_tokens, int32_t num_q_heads, int32_t max_query_len,
                                 const float* scale,
                                 int32_t fmt, float sm_scale, void* out, kvq_stream_t stream) {
    kvq_status st = check_cache(cache, fmt);
    if (st != KVQ_OK) return st;
    if (batch < 0 || num_q_tokens < 0 || num_q_heads <= 0 || max_query_len < 0 || max_blocks_per_seq <= 0)
        return KVQ_ERR_INVALID_ARG;
    if (num_q_heads % cache->num_kv_heads) return KVQ_ERR_INVALID_ARG;
    if (num_q_heads / cache->num_kv_heads > kvq::prefill_rows_per_tile()) return KVQ_ERR_UNSUPPORTED;
    if (num_q_tokens > 0x7FFFFFFFll) return KVQ_ERR_UNSUPPORTED;   // query_start entries are int32
    if (batch > 65535 || cache->num_kv_heads > 65535) return KVQ_ERR_UNSUPPORTED;
    if (batch == 0 || max_query_len == 0 || num_q_tokens == 0) return KVQ_OK;
    if (!q || !block_tables || !context_lens || !query_start || !out || !aligned(q, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(query_start, 4))
        return KVQ_ERR_INVALID_ARG;
    if (scale && !aligned(scale, 4)) return KVQ_ERR_INVALID_ARG;
    if (!(sm_scale >= 0.f) || std::isinf(sm_scale)) return KVQ_ERR_INVALID_ARG;
    int dev;
    if (!current_device(&dev)) return KVQ_ERR_CUDA;
    unsigned long long* err = err_word(dev);
    if (!err) return KVQ_ERR_CUDA;
    kvq::PrefillArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.cache = view(cache);
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.batch = batch;
    a.num_q_tokens = num_q_tokens;
    a.num_q_heads = num_q_heads;
    a.max_query_len = max_query_len;
    a.scale = (fmt == KVQ_INT8 || fmt == KVQ_INT4) ? nullptr : scale;
    a.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt((float)cache->head_dim);
    a.out = static_cast<uint16_t*>(out);
    a.err = err;
    return kvq::launch_prefill(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_dequant(const kvq_cache* cache, const int64_t* slots, int64_t num_slots, const float* scale,
                       int32_t fmt, float* out_k, float* out_v, kvq_stream_t stream) {
    kvq_status st = check_cache(cache, fmt);
    if (st != KVQ_OK) return st;
    if (num_slots < 0) return KVQ_ERR_INVALID_ARG;
    if (num_slots == 0) return KVQ_OK;
    if (!slots || !out_k || !out_v || !aligned(slots, 8) || !aligned(out_k, 16) || !aligned(out_v, 16))
        return KVQ_ERR_INVALID_ARG;
    if (scale && !aligned(scale, 4)) return KVQ_ERR_INVALID_ARG;
    if (num_slots * cache->num_kv_heads * (cache->head_dim / 16) / 256 >= 0x7FFFFFFFll) return KVQ_ERR_UNSUPPORTED;
    int dev;
    if (!current_device(&dev)) return KVQ_ERR_CUDA;
    unsigned long long* err = err_word(dev);
    if (!err) return KVQ_ERR_CUDA;
    kvq::DequantArgs a{view(cache), slots, num_slots, (fmt == KVQ_INT8 || fmt == KVQ_INT4) ? nullptr : scale, out_k, out_v, err};
    return kvq::launch_dequant(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_encode_fp8(const float* x, void* codes, int64_t n, int32_t fmt, kvq_stream_t stream) {
    if (fmt != KVQ_E4M3 && fmt != KVQ_E5M2) return KVQ_ERR_INVALID_ARG;
    if (n < 0) return KVQ_ERR_INVALID_ARG;
    if (n == 0) return KVQ_OK;
    if (!x || !codes || !aligned(x, 16) || !aligned(codes, 16)) return KVQ_ERR_INVALID_ARG;
    return kvq::launch_encode_fp8(x, static_cast<uint8_t*>(codes), n, fmt,
                                  reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? KVQ_OK
               : KVQ_ERR_CUDA;
}

kvq_status kvq_device_error_check(kvq_stream_t stream, int64_t* detail) {
    int dev;
    if (!current_device(&dev)) return KVQ_ERR_CUDA;
    unsigned long long* err = err_word(dev);
    if (!err) return KVQ_ERR_CUDA;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return KVQ_ERR_CUDA;
    unsigned long long v = 0;
    if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
    if (v == 0) {
        if (detail) *detail = 0;
        return KVQ_OK;
    }
    const unsigned long long zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return KVQ_ERR_CUDA;
    int64_t d = (int64_t)(v & 0x00FFFFFFFFFFFFFFull);
    if (d & 0x0080000000000000ll) d |= (int64_t)0xFF00000000000000ull;  // sign-extend 56 bits
    if (detail) *detail = d;
    return (v >> 56) == kvq::DEV_ERR_TIMEOUT ? KVQ_ERR_TIMEOUT : KVQ_ERR_OUT_OF_RANGE;
}

}  // extern "C"
