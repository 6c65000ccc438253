// Decode attention for callers that cannot allocate device memory.
//
// kvq_decode_attention asks its caller for a workspace when a context is split
// across several CTAs (the per-partition partial results).  Some callers have
// no way to provide one: plugin hosts that hand an operator only its inputs and
// outputs while their own pool owns every other byte of device memory, and
// serving loops that must not allocate once they are running (an allocation can
// stall on the device or fail after a pool has reserved the memory).  This file
// gives them kvq_decode_attention_static_scratch, which takes its workspace from
// a fixed array that lives in the library's own device memory.
//
// The array is kvq_static_scratch_bytes() = 64 MiB.  Every GPU that loads this
// part of the library holds it until the process exits.  Its address is looked
// up once per device (cudaGetSymbolAddress, with that device current) by the
// first call on the device.  All calls share it and it keeps what the last call
// wrote; the decode kernels write every partial they later read, so nothing in
// it needs to start at zero.  (A call whose kernels record a device error -- a
// context length or block id out of range, a bounded wait that ran out -- may
// leave partials unwritten; its output is then undefined, as with a caller
// workspace.)  Two calls whose kernels overlap on the GPU (on different
// streams, or from different host threads) race on the array.  The arguments
// are checked before the size limit, so a bad argument gets the status
// kvq_decode_attention would give it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kvq.h"

namespace {

constexpr size_t kScratchBytes = (size_t)64 << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device; the name g_static_scratch
// in host code is only a host-side stand-in and must never reach a kernel.
void* scratch_ptr(int dev) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

size_t kvq_static_scratch_bytes(void) { return kScratchBytes; }

kvq_status kvq_decode_attention_static_scratch(const void* q, const kvq_cache* cache,
                                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                                               const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                               int32_t max_context_len, const float* scale, int32_t fmt,
                                               float sm_scale, void* out, int32_t partition_size,
                                               kvq_stream_t stream) {
    // The arguments are checked first, exactly as kvq_decode_attention checks
    // them: called without a workspace it validates everything, launches
    // nothing, and answers KVQ_ERR_WORKSPACE only when the arguments are good
    // and a workspace is needed.  Any other answer (an argument error, or OK
    // for an empty batch) is this call's answer too.
    const kvq_status st = kvq_decode_attention(q, cache, block_tables, max_blocks_per_seq, context_lens, batch,
                                               num_q_heads, max_context_len, scale, fmt, sm_scale, out, nullptr, 0,
                                               partition_size, stream);
    if (st != KVQ_ERR_WORKSPACE) return st;
    const size_t need = kvq_decode_workspace_size(batch, num_q_heads, cache->num_kv_heads, cache->head_dim,
                                                  max_context_len, partition_size);
    if (need == 0) return KVQ_ERR_INVALID_ARG;
    if (need > kScratchBytes) return KVQ_ERR_SCRATCH_LIMIT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
    void* ws = scratch_ptr(dev);
    if (!ws) return KVQ_ERR_CUDA;
    return kvq_decode_attention(q, cache, block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads,
                                max_context_len, scale, fmt, sm_scale, out, ws, kScratchBytes, partition_size,
                                stream);
}

}  // extern "C"
