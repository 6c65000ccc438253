/*
 * kvq.h -- C ABI of the GB300 (sm_103a) quantized paged KV cache.
 *
 * Two operations make up the hot path of an LLM server's quantized KV cache:
 *
 *   kvq_append            quantize-on-write of fp16 K/V into the paged cache;
 *   kvq_decode_attention  single-token decode attention that dequantizes the
 *                         cache on read and computes in fp16/fp32.
 *
 * Around them: kvq_decode_attention_append (the same decode with each
 * sequence's newest K/V row quantized into the cache in the same launch),
 * kvq_decode_attention_static_scratch (decode without a caller workspace),
 * kvq_prefill_attention (causal attention of a chunk of new queries per
 * sequence over the same cache), kvq_dequant (a debugging gather of the
 * fp32 values a kernel sees) and kvq_encode_fp8 (the append kernels' FP8
 * encoder on raw fp32 values, for checking it).  The operations follow these pages (cited by
 * title and section):
 *
 *   [TGI] "Accelerating Inference with FP8 KV Cache" (text-generation-inference
 *         docs).  Intro: the KV cache is stored in FP8 while computation runs in
 *         FP16.  "FP8 Formats: E4M3 and E5M2": E4M3 = 1 sign, 4 biased exponent,
 *         3 mantissa bits; E5M2 = 1 sign, 5 biased exponent, 2 mantissa bits;
 *         one fp32 scaling factor per quantized tensor (per-tensor scalar).
 *         "FP8 E4M3 KV Cache": a scale of 1.0 is used when none is given.
 *         "Checkpoint structure for KV scales": one kv_scale per attention layer,
 *         shared by K and V.  "Current Hardware Support": NVIDIA GPUs take
 *         E4M3 ("fp8") and E5M2 ("fp8_e5m2").
 *   [LMD] "[Feature] TurboMind support W8A8 or FP8 KV Cache" (lmdeploy issue
 *         1463): online KV-cache INT8 (quant-policy 8) as the alternative, and
 *         an INT4 implementation named beside it.
 *   [QQQ] "[QST] Scale factors and benchmarks" (QQQ issue 2): group
 *         quantization named for a 4-bit KV cache.
 *
 * Conventions for every call:
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except the
 *     kvq_cache descriptor itself (a host struct read during the call only).
 *     The library allocates no memory and frees none.
 *   - Calls are asynchronous on `stream` (NULL = the legacy default stream) and
 *     never synchronize the host, except kvq_device_error_check.
 *   - Arguments are validated before any launch; a call that returns an error
 *     status has launched nothing and written nothing.
 *   - fp16 tensors are IEEE binary16, row-major, 16-byte aligned.
 *   - A kernel that meets a slot or block id outside the cache skips that
 *     access and records it in a device error word; kvq_device_error_check
 *     reports it.  No kernel traps.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_ABI_VERSION 1

#if defined(__GNUC__)
#define KVQ_API __attribute__((visibility("default")))
#else
#define KVQ_API
#endif

/* Same object as cudaStream_t; declared here so the header needs no CUDA include. */
typedef struct CUstream_st* kvq_stream_t;

/* Cache formats.  [TGI] "Current Hardware Support": "fp8" = E4M3 (OCP
 * E4M3FN: no infinities, S.1111.111 = NaN, max 448) and "fp8_e5m2" = E5M2
 * (max 57344); [LMD]: online INT8, and the INT4 implementation the same
 * thread names beside it (read here as INT8 with 4 bits: codes in [-7, 7],
 * scale amax / 7 per row, two codes per byte, channel 2i in the low nibble). */
typedef enum {
    KVQ_E4M3 = 1,
    KVQ_E5M2 = 2,
    KVQ_INT8 = 3,
    KVQ_INT4 = 4
} kvq_fmt;

typedef enum {
    KVQ_OK = 0,
    KVQ_ERR_INVALID_ARG = 1,   /* null / misaligned pointer, bad size, fmt mismatch */
    KVQ_ERR_UNSUPPORTED = 2,   /* head_dim, block_size or q-group size not built */
    KVQ_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    KVQ_ERR_OUT_OF_RANGE = 4,  /* a kernel met a slot / block id outside the cache */
    KVQ_ERR_TIMEOUT = 5,       /* a kernel's bounded wait ran out (never expected) */
    KVQ_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed */
    KVQ_ERR_SCRATCH_LIMIT = 7  /* needs more scratch than the library's fixed array */
} kvq_status;

/* The paged cache: caller-owned device memory.
 *   k_codes, v_codes: [num_blocks][num_kv_heads][block_size][head_dim] bytes,
 *                     FP8 codes (u8) or INT8 codes (i8); for INT4
 *                     [..][head_dim / 2] bytes of packed codes; 16-byte aligned.
 *   k_scales, v_scales: INT8 and INT4, fp32 [num_blocks][num_kv_heads][block_size]
 *                     [head_dim / group_size] (one scale per group of channels of a
 *                     (token, kv-head) row; one per row when group_size is 0);
 *                     NULL for FP8.
 *   head_dim in {64, 128}; block_size in {16, 32, 64}; fmt a kvq_fmt.
 *   group_size: INT8 / INT4 group quantization (the QQQ page "[QST] Scale
 *     factors and benchmarks" names group quantization for a 4-bit KV cache):
 *     0 or head_dim = one scale per row; head_dim / 2 or head_dim / 4 = two or
 *     four groups of consecutive channels, each quantized as a row is (its own
 *     amax and scale).  Must be 0 for FP8; any other value is INVALID_ARG.
 *     Every entry point takes every group size.  Decode reads the cache once,
 *     except for INT4 kv-heads of head_dim 64 with 16-channel groups and more
 *     than 8 (q-head, scale group) pairs: those stream it ceil(G * 4 / 16)
 *     times. */
typedef struct {
    void* k_codes;
    void* v_codes;
    float* k_scales;
    float* v_scales;
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t fmt;
    int32_t group_size;
} kvq_cache;

/* Quantize-on-write ([TGI] intro and "FP8 Formats"; [LMD] online INT8).
 *   k, v: fp16 [num_tokens][num_kv_heads][head_dim].
 *   slot_mapping: int64 [num_tokens]; token t goes to block slot / block_size,
 *     row slot % block_size; slot -1 skips the token (padding).
 *   scale: FP8 only -- device pointer to ONE fp32 per-tensor scale shared by K
 *     and V, or NULL for the default 1.0 ([TGI] "FP8 E4M3 KV Cache").  Each
 *     element is stored as code = RNE-satfinite(fl32(x / scale)).  Ignored for
 *     INT8, where each (token, kv-head) row gets s = fl32(amax / 127) and codes
 *     clamp(rint(fl32(x / s)), -127, 127) (s = 0 and zero codes for a zero row);
 *     INT4 the same with s = fl32(amax / 7) and codes in [-7, 7].
 *   fmt must equal cache->fmt.  num_tokens == 0 is a no-op. */
KVQ_API kvq_status kvq_append(const void* k, const void* v, const kvq_cache* cache,
                      const int64_t* slot_mapping, int64_t num_tokens,
                      const float* scale, int32_t fmt, kvq_stream_t stream);

/* Bytes of workspace kvq_decode_attention needs for these sizes on the
 * current device (nonzero whenever batch > 0).  partition_size as below. */
KVQ_API size_t kvq_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_context_len,
                                 int32_t partition_size);

/* Single-token decode attention over the paged quantized cache ([TGI] intro:
 * stored quantized, computed in FP16; accumulation here is fp32).
 *   q:   fp16 [batch][num_q_heads][head_dim].
 *   block_tables: int32 [batch][max_blocks_per_seq]; entry i of sequence b is
 *     the physical block holding its tokens i*block_size .. (i+1)*block_size-1.
 *   context_lens: int32 [batch], each in [0, max_context_len]; every token
 *     t < context_len attends (the new token is appended first).  A sequence
 *     with context 0 gets a zero output.
 *   q-head h reads kv-head h / (num_q_heads / num_kv_heads); num_q_heads must be
 *     a multiple of num_kv_heads and the group size at most 8.
 *   INT4 caches are decoded by the tensor-core kernel (kvq_set_decode_kernel(1)
 *   with INT4 returns KVQ_ERR_UNSUPPORTED).
 *   batch at most 4096, and batch * num_kv_heads * ceil(max_context_len / 32)
 *     below 2^31 (KVQ_ERR_UNSUPPORTED otherwise).
 *   scale: FP8 per-tensor scale as in kvq_append (NULL = 1.0); ignored for INT8
 *     and INT4.
 *   sm_scale: softmax scale; 0 selects 1 / sqrt(head_dim).
 *   out: fp16 [batch][num_q_heads][head_dim] = softmax(sm_scale * q K^T) V.
 *   workspace: device scratch of kvq_decode_workspace_size() bytes, 256-byte
 *     aligned, holding the partial results of context chunks; contents are not
 *     preserved and nothing in it needs to be initialised.
 *   partition_size: tokens per context chunk whose partial result is kept
 *     (a multiple of 64, at most 65536), or 0 to let the library choose from
 *     the sizes and the device's SM count.  Results agree across choices up to
 *     fp32 summation order.
 *   When kvq_device_error_check reports an error recorded by this call (a
 *   context length or block id out of range, or a bounded wait that ran out),
 *   `out` is undefined for the whole call: a warp that stopped early may have
 *   left partial results unwritten, and the merge then reads whatever the
 *   workspace held. */
KVQ_API kvq_status kvq_decode_attention(const void* q, const kvq_cache* cache,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, int32_t batch,
                                int32_t num_q_heads, int32_t max_context_len,
                                const float* scale, int32_t fmt, float sm_scale, void* out,
                                void* workspace, size_t workspace_bytes,
                                int32_t partition_size, kvq_stream_t stream);

/* Decode step with the newest token's K/V appended inside the same launch:
 * the result -- cache bytes, INT8 / INT4 scales and out -- is bit-identical to
 * kvq_append of k_new / v_new followed by kvq_decode_attention with the same
 * arguments.  It follows the same passages as those two calls; fusing them is
 * a scheduling choice (one launch instead of two) that no page prescribes.
 *   k_new, v_new: fp16 [batch][num_kv_heads][head_dim], the K and V rows of
 *     each sequence's newest token, position context_lens[b] - 1, which goes to
 *     the cache slot block_tables[b][(ctx - 1) / block_size] * block_size +
 *     (ctx - 1) % block_size.  A sequence with context 0 appends nothing.
 *     The row is quantized exactly as kvq_append does (FP8 with `scale`, INT8
 *     and INT4 with the row's own scale, or its groups').
 *   Every other argument, the workspace and the errors are those of
 *   kvq_decode_attention; a block id outside the cache is recorded and its row
 *   is not written. */
KVQ_API kvq_status kvq_decode_attention_append(const void* q, const void* k_new, const void* v_new,
                                       const kvq_cache* cache, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t batch, int32_t num_q_heads, int32_t max_context_len,
                                       const float* scale, int32_t fmt, float sm_scale, void* out,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t partition_size, kvq_stream_t stream);

/* Decode attention for callers that cannot allocate device memory (no page
 * has a counterpart: this is a deployment variant).  Plugin hosts that give an
 * operator only its inputs and outputs while their own pool owns the rest of
 * device memory, and serving loops that must not allocate once running, have
 * no workspace to pass.  Same arguments and result as kvq_decode_attention
 * without workspace / workspace_bytes: the workspace is a fixed array of
 * kvq_static_scratch_bytes() (64 MiB) in the library's device memory, held by
 * every GPU that loads the library until the process exits.  The arguments
 * are checked first and give the statuses kvq_decode_attention gives; then
 * sizes whose kvq_decode_workspace_size() exceeds the array return
 * KVQ_ERR_SCRATCH_LIMIT with nothing launched.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress); make that first call before any stream
 * capture.  Calls share the array and it keeps the last call's contents;
 * nothing in it needs to start at zero.  Calls whose kernels overlap on the GPU
 * race on it.  Allocates nothing. */
KVQ_API kvq_status kvq_decode_attention_static_scratch(const void* q, const kvq_cache* cache,
                                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                       const int32_t* context_lens, int32_t batch,
                                                       int32_t num_q_heads, int32_t max_context_len,
                                                       const float* scale, int32_t fmt, float sm_scale,
                                                       void* out, int32_t partition_size, kvq_stream_t stream);
KVQ_API size_t kvq_static_scratch_bytes(void);

/* Causal attention of chunks of new queries over the paged quantized cache
 * (chunked prefill).  The pages define the cache formats and their scales
 * ([TGI] "FP8 Formats: E4M3 and E5M2", intro: stored quantized, computed in
 * FP16; [LMD] online INT8) but not the prefill step itself; this is the plain
 * causal attention that reads that cache, with fp16 x fp16 products and fp32
 * sums on the tensor cores.
 *   q:   fp16 [num_q_tokens][num_q_heads][head_dim]; sequence b owns rows
 *     query_start[b] .. query_start[b+1]-1 (n_b = query_start[b+1] -
 *     query_start[b] new queries, in position order).
 *   query_start: int32 [batch + 1], non-decreasing, 0 <= query_start[b] and
 *     query_start[batch] <= num_q_tokens (the rows q and out hold).
 *   context_lens: int32 [batch]: every cached token of b, the chunk's own
 *     included (append the chunk's K/V first).  Query i of the chunk sits at
 *     position context_lens[b] - n_b + i and attends to tokens 0 .. position.
 *   block_tables, max_blocks_per_seq, scale, fmt, sm_scale: as in
 *     kvq_decode_attention.  q-head h reads kv-head h / (num_q_heads /
 *     num_kv_heads); the group size may be at most 128.
 *   max_query_len: an upper bound of every n_b (sizes the launch).
 *   out: fp16 [num_q_tokens][num_q_heads][head_dim]; rows of sequences with
 *     n_b > context_lens[b], n_b > max_query_len, query_start[b] < 0,
 *     query_start[b+1] > num_q_tokens or context_lens[b] >
 *     max_blocks_per_seq * block_size are left unwritten and the sequence
 *     index is recorded for kvq_device_error_check (KVQ_ERR_OUT_OF_RANGE), as
 *     is a block id outside the cache (its tokens then count as zeros).
 *   Needs no workspace. */
KVQ_API kvq_status kvq_prefill_attention(const void* q, const kvq_cache* cache,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, const int32_t* query_start,
                                 int32_t batch, int64_t num_q_tokens, int32_t num_q_heads,
                                 int32_t max_query_len,
                                 const float* scale, int32_t fmt, float sm_scale, void* out,
                                 kvq_stream_t stream);

/* Debug gather + dequantize-on-read: for each of num_slots slots, fp32
 * [num_slots][num_kv_heads][head_dim] rows of K and V, each value
 * fl32(decode(code) * scale) (FP8) or fl32(code * s) (INT8, INT4), s the
 * scale of the value's row, or of its channel group when group_size > 0.
 * A slot outside the cache leaves its rows unwritten and is recorded for
 * kvq_device_error_check (KVQ_ERR_OUT_OF_RANGE). */
KVQ_API kvq_status kvq_dequant(const kvq_cache* cache, const int64_t* slots, int64_t num_slots,
                       const float* scale, int32_t fmt, float* out_k, float* out_v,
                       kvq_stream_t stream);

/* Debug: the FP8 encoder of the append kernels on raw fp32 values
 * ([TGI] "FP8 Formats: E4M3 and E5M2"; OCP E4M3FN / E5M2): codes[i] =
 * RNE-satfinite(x[i]) -- round to nearest, ties to even, |x| beyond the
 * format's largest finite value (Inf included) to +-that value, NaN to a NaN
 * code -- which is what kvq_append stores for an fp16 input once it has divided
 * it by the scale.  It exists so that the hardware conversion can be checked
 * on every fp32 input.
 *   x: fp32 [n]; codes: u8 [n]; both 16-byte aligned.  fmt: KVQ_E4M3 or
 *   KVQ_E5M2 (anything else is KVQ_ERR_INVALID_ARG).  n == 0 is a no-op. */
KVQ_API kvq_status kvq_encode_fp8(const float* x, void* codes, int64_t n, int32_t fmt, kvq_stream_t stream);

/* Decode kernel family used by kvq_decode_attention in this process:
 * 0 = automatic (tensor-core kernel), 1 = CUDA-core kernel (group size <= 4,
 * FP8 and INT8 only),
 * 2 = tensor-core kernel.  A tuning and cross-checking knob; returns the
 * previous value, or -1 for an unknown kind (nothing changes). */
KVQ_API int32_t kvq_set_decode_kernel(int32_t kind);

/* Measurement hook.  While set (both non-NULL), every kvq_decode_attention
 * call records ev_begin on its stream immediately before its main kernel and
 * ev_end immediately after it, so that kernel can be timed alone (the call
 * also launches a small reduce kernel).  Both are cudaEvent_t created by the
 * caller; NULL, NULL turns the hook off.  Process-wide, not thread-safe. */
KVQ_API void kvq_set_decode_timing_events(void* ev_begin, void* ev_end);

/* Synchronizes `stream`, then reads and clears the current device's error word.
 * Returns KVQ_OK, KVQ_ERR_OUT_OF_RANGE or KVQ_ERR_TIMEOUT (the first one
 * recorded); *detail (if not NULL) receives the offending slot / block id. */
KVQ_API kvq_status kvq_device_error_check(kvq_stream_t stream, int64_t* detail);

KVQ_API const char* kvq_status_string(kvq_status status);
KVQ_API int32_t kvq_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
