/*
 * pagedattn.h - C ABI of libpagedattn.so: one batched attention step over a
 * paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operations follow the vLLM inference notes ("AI Infra入门干货总结：大模型是
 * 如何高效推理的"):
 *   - §Paged Attention: the per-layer cache is [num_blocks, block_size,
 *     num_kv_heads, head_dim] for K and for V; block_table[b][i] is the
 *     physical block of logical block i of request b; slot_mapping tells the
 *     kernel where to write each new token's K/V; slot = block * block_size +
 *     offset, block = slot / block_size, offset = slot % block_size.
 *   - §LLM 推理全流程 3 (Attention): K/V are read discretely from the paged
 *     cache; Q is [query_lens, num_heads, head_dim]; GQA maps one KV head to a
 *     group of query heads by index, without copies; FlashAttention-style
 *     fusion with online softmax keeps S and P out of HBM.
 *   - §Continuous Batching: one step mixes requests; each schedules
 *     num_tokens - num_computed_tokens query tokens (decode tokens and
 *     chunked-prefill chunks alike).
 *
 * Conventions shared by every call:
 *   - Pointers marked (device) are CUDA device pointers on the current device;
 *     (host) are host pointers. The caller owns every buffer; the library
 *     allocates no device memory and frees nothing.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Calls enqueue work on it and return without synchronising.
 *   - Element data (q, key, value, the caches and out of one call) is one
 *     16-bit float type: bf16 (dtype PA_BF16) or IEEE fp16 (PA_FP16). The
 *     arithmetic is the same for both (fp32 accumulation, outputs rounded to
 *     nearest even in the element type). Indices are int32, except
 *     slot_mapping, which is int64.
 *   - Errors the host can see (null pointers, bad sizes, unsupported shapes,
 *     misalignment, small workspace) are returned before anything is
 *     launched. Errors only the device can see (a block id or slot out of
 *     range, lengths that contradict the host bounds) make the kernels skip
 *     the offending work and set bits in a device status word, which
 *     pa_debug_status() reads; outputs of the offending request are then
 *     undefined.
 *   - 8-bit caches (LLM-infra reading map, §4.2: the KV cache is stored in
 *     8 bits, quantised online as it is written and dequantised as attention
 *     reads it): the *_fp8 calls keep K and V caches of E4M3 codes (sign,
 *     4-bit exponent with bias 7, 3-bit fraction, no infinities, largest
 *     finite 448; 0x7F and 0xFF are NaN), one byte per element, with one
 *     float scale per cache. Writing stores code = E4M3(x / scale): the
 *     quotient in binary32 (correctly rounded), then rounded to the nearest
 *     code, ties to even, magnitudes beyond 448 saturating to 448. Reading
 *     uses code * scale. q, key, value and out stay bf16 or fp16.
 *   - Supported now: head_dim 64, 80, 96, 128 or 256; block_size 8, 16 or 32 (the
 *     reading map, §2.3, sweeps page sizes; the kernels stage K/V 16 keys at a
 *     time); num_heads a multiple of num_kv_heads with group size 1, 2, 4 or 8.
 *     pa_rope_reshape_and_cache and pa_copy_blocks take any block_size.
 *     The elements of one token's cache row (num_kv_heads * head_dim; for
 *     the rotary calls, its q, K and V rows together) must number fewer than
 *     2^31 (PA_ERR_UNSUPPORTED otherwise).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_NULL = -1,          /* a required pointer is NULL */
    PA_ERR_DIMS = -2,          /* a size is negative or sizes contradict each other */
    PA_ERR_UNSUPPORTED = -3,   /* dtype, head_dim, block_size or group size not built */
    PA_ERR_ALIGN = -4,         /* a pointer or stride breaks 16-byte vector alignment */
    PA_ERR_WORKSPACE = -5,     /* workspace NULL or smaller than pa_attention_workspace_size() */
    PA_ERR_LAUNCH = -6,        /* a kernel launch failed (the CUDA error is sticky or the config invalid) */
    PA_ERR_DEVICE_BOUNDS = -7, /* pa_debug_status: a kernel met an out-of-range index */
    PA_ERR_CUDA = -8           /* another CUDA runtime call failed */
} pa_status;

/* Element types. PA_FP8_E4M3 names 8-bit cache codes (the *_fp8 calls, and
 * pa_copy_blocks / pa_gather_kv on such caches). */
enum { PA_BF16 = 0, PA_FP16 = 1, PA_FP8_E4M3 = 2 };

/* Bits of the device status word (pa_debug_status). */
enum {
    PA_FLAG_SLOT_RANGE = 1u << 0,   /* reshape_and_cache: slot >= num_blocks * block_size */
    PA_FLAG_BLOCK_RANGE = 1u << 1,  /* a block_tables entry that must be read is outside [0, num_blocks) */
    PA_FLAG_LENGTHS = 1u << 2,      /* seq_len < query_len, seq_len > max_seq_len, query_len > max_query_len,
                                       or seq_len > max_blocks_per_seq * block_size */
    PA_FLAG_QUERY_LOC = 1u << 3,    /* query_start_loc not non-decreasing from 0 to total_q_tokens */
    PA_FLAG_TIMEOUT = 1u << 4,      /* a kernel gave up waiting for its own data copy (bounded wait) */
    PA_FLAG_POSITION_RANGE = 1u << 5 /* rope_reshape_and_cache: position outside [0, max_position) */
};

/*
 * Step 1 - reshape_and_cache: write this step's new K/V rows into the cache
 * (vLLM notes, §Paged Attention: slot_mapping names each new token's slot,
 * and a slot splits into block = slot / block_size and offset = slot %
 * block_size, which address the cache).
 *
 * For every token t in [0, num_tokens) with s = slot_mapping[t] >= 0:
 *   key_cache[s / block_size][s % block_size][:][:]   = key[t][:][:]
 *   value_cache[s / block_size][s % block_size][:][:] = value[t][:][:]
 * A negative slot means "padding token, write nothing". Two tokens of one
 * call must not name the same slot (which write wins is then unspecified).
 *
 *   key, value         (device) `dtype`, token t starts at key + t * key_token_stride
 *                      elements and holds [num_kv_heads, head_dim] contiguous
 *                      elements (so key may be a slice of a fused QKV output).
 *   key_token_stride,  elements between consecutive tokens (>= num_kv_heads * head_dim,
 *   value_token_stride a multiple of 8).
 *   key_cache,         (device) `dtype` [num_blocks, block_size, num_kv_heads, head_dim],
 *   value_cache        contiguous, updated in place.
 *   slot_mapping       (device) int64 [num_tokens].
 * All data pointers must be 16-byte aligned (PA_ERR_ALIGN otherwise).
 * A slot >= num_blocks * block_size is skipped and sets PA_FLAG_SLOT_RANGE.
 * num_tokens == 0 launches nothing.
 */
pa_status pa_reshape_and_cache(const void *key, const void *value,
                               int64_t key_token_stride, int64_t value_token_stride,
                               void *key_cache, void *value_cache,
                               const int64_t *slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int64_t num_blocks,
                               int32_t dtype, void *stream);

/*
 * reshape_and_cache into 8-bit caches: the same slots and arguments as
 * pa_reshape_and_cache (key and value are `dtype`, bf16 or fp16), but every
 * element is stored as the E4M3 code of x / k_scale (keys) or x / v_scale
 * (values). key_cache, value_cache: (device) uint8 [num_blocks, block_size,
 * num_kv_heads, head_dim], 16-byte aligned. k_scale and v_scale must be
 * finite and positive (PA_ERR_DIMS otherwise); a NaN element gives a NaN
 * code.
 */
pa_status pa_reshape_and_cache_fp8(const void *key, const void *value,
                                   int64_t key_token_stride, int64_t value_token_stride,
                                   void *key_cache, void *value_cache,
                                   const int64_t *slot_mapping, int32_t num_tokens,
                                   int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int64_t num_blocks,
                                   float k_scale, float v_scale, int32_t dtype, void *stream);

/*
 * Bytes of device workspace pa_attention_varlen or pa_attention_varlen_fp8 needs for these host-side
 * bounds (0 if the arguments are invalid). Pure host arithmetic; no CUDA call.
 * The workspace holds the work plan and the split-KV partial results.
 */
size_t pa_attention_workspace_size(int32_t num_seqs, int32_t total_q_tokens,
                                   int32_t max_query_len, int32_t max_seq_len,
                                   int32_t num_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size);

/*
 * How pa_attention_varlen (16-bit caches) will split KV for these bounds: the
 * partition size in tokens and the largest number of partitions of one
 * request. Host only. (pa_attention_varlen_fp8 runs more warps per SM, so it
 * may choose smaller partitions; the workspace size covers both.)
 */
pa_status pa_attention_plan_info(int32_t num_seqs, int32_t max_seq_len,
                                 int32_t num_heads, int32_t num_kv_heads,
                                 int32_t *partition_tokens, int32_t *max_partitions);

/*
 * Step 2 - attention over the paged cache, for a batch that may mix decode
 * tokens and chunked-prefill chunks (vLLM notes, §LLM 推理全流程 3: Q of
 * [query_lens, num_heads, head_dim] against K/V read through the block table
 * from the paged cache, GQA by index, FlashAttention-style online softmax;
 * §Continuous Batching: each request's query tokens are the ones between
 * num_computed_tokens and num_tokens; LLM-infra reading map, §6: long
 * contexts split over KV partitions whose partial results are merged by
 * their log-sum-exp, Flash-Decoding).
 *
 * Request b owns query tokens [query_start_loc[b], query_start_loc[b+1]) and
 * has seq_len = seq_lens[b] KV tokens, which include its new tokens (run
 * pa_reshape_and_cache first, on the same stream). With
 * query_len = query_start_loc[b+1] - query_start_loc[b] and
 * ctx = seq_len - query_len, query i of the request sits at position ctx + i
 * and attends to keys 0 .. ctx + i (causal, bottom-right aligned; a decode
 * token sees the whole sequence). Query head h reads KV head
 * h / (num_heads / num_kv_heads). Logical key j of request b lives at
 * block_tables[b * max_blocks_per_seq + j / block_size], row j % block_size.
 *
 *   out[t][h][:] = round_dtype( sum_j softmax_j(scale * q[t][h] . K[j]) * V[j] )
 *
 *   q                (device) `dtype`; token t at q + t * q_token_stride elements,
 *                    [num_heads, head_dim] contiguous; q_token_stride even.
 *   key_cache,       (device) `dtype` [num_blocks, block_size, num_kv_heads, head_dim].
 *   value_cache
 *   block_tables     (device) int32 [num_seqs, max_blocks_per_seq]; entries past
 *                    ceil(seq_len / block_size) are never read.
 *   seq_lens         (device) int32 [num_seqs].
 *   query_start_loc  (device) int32 [num_seqs + 1], starts at 0, non-decreasing,
 *                    ends at total_q_tokens.
 *   max_query_len,   (host) upper bounds of query_len and seq_len over the batch;
 *   max_seq_len      they size the launch and the workspace without a device read.
 *   scale            softmax scale (usually 1/sqrt(head_dim)).
 *   out              (device) `dtype` [total_q_tokens, num_heads, head_dim], contiguous.
 *   workspace        (device) at least pa_attention_workspace_size(...) bytes,
 *                    256-byte aligned; contents need no initialisation and are
 *                    scratch after the call.
 * Requests with query_len 0 are allowed and produce nothing. All work is
 * enqueued on `stream`: a planning kernel, the split-KV attention kernel (for
 * requests of at most 8 / (num_heads / num_kv_heads) query tokens), the
 * tensor-core prefill-tile kernel when some request is longer, and the
 * log-sum-exp merge kernel when some request is split.
 */
pa_status pa_attention_varlen(const void *q, int64_t q_token_stride,
                              const void *key_cache, const void *value_cache,
                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                              const int32_t *seq_lens, const int32_t *query_start_loc,
                              int32_t num_seqs, int32_t total_q_tokens,
                              int32_t max_query_len, int32_t max_seq_len,
                              int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int64_t num_blocks, float scale,
                              void *out, void *workspace, size_t workspace_bytes,
                              int32_t dtype, void *stream);

/*
 * Attention over 8-bit caches: the same operation and arguments as
 * pa_attention_varlen (same workspace size), with key_cache and value_cache
 * holding E4M3 codes (uint8 [num_blocks, block_size, num_kv_heads, head_dim],
 * 16-byte aligned) whose values are code * k_scale and code * v_scale:
 *   out[t][h][:] = round( sum_j softmax_j(scale * q[t][h] . (k_scale * Kc[j]))
 *                         * (v_scale * Vc[j]) )
 * q and out are `dtype` (bf16 or fp16). k_scale and v_scale must be finite and
 * positive (PA_ERR_DIMS otherwise). Each code is widened exactly and the
 * products accumulate in fp32, as for 16-bit caches: the tensor cores take
 * fp16 operands (a bf16 q row or column whose largest |q| reaches 2^15 is
 * scaled by a power of two first, and its scores scaled back).
 */
pa_status pa_attention_varlen_fp8(const void *q, int64_t q_token_stride,
                                  const void *key_cache, const void *value_cache,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *seq_lens, const int32_t *query_start_loc,
                                  int32_t num_seqs, int32_t total_q_tokens,
                                  int32_t max_query_len, int32_t max_seq_len,
                                  int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int64_t num_blocks, float scale,
                                  float k_scale, float v_scale,
                                  void *out, void *workspace, size_t workspace_bytes,
                                  int32_t dtype, void *stream);

/*
 * Rotary position embedding fused with reshape_and_cache (vLLM notes, §LLM
 * 推理全流程 2: a token's position is a rotation angle, with a precomputed
 * cos_sin_cache of shape [max_position, rotary_dim]). For every token t with
 * positions[t] in [0, max_position):
 *   - every head of q[t] is rotated in place;
 *   - if slot_mapping[t] >= 0, key[t] rotated and value[t] unchanged are
 *     written to the slot, exactly as pa_reshape_and_cache writes them (key
 *     and value themselves are not modified).
 * Row p of cos_sin_cache (device, fp32, 16-byte aligned) holds
 * cos(p * theta_i) for i < rotary_dim / 2 followed by sin(p * theta_i) for the
 * same i. A rotated pair (x1, x2) becomes (x1 cos - x2 sin, x2 cos + x1 sin),
 * computed in fp32 and rounded once to the element type. Pairs are element
 * i with i + rotary_dim / 2 (is_neox != 0) or elements 2i and 2i + 1
 * (is_neox == 0), for i < rotary_dim / 2; elements at rotary_dim and above
 * pass through. rotary_dim must be a multiple of 16, at most head_dim and at
 * most 512; head_dim a multiple of 8.
 *   q (device): [num_tokens, num_heads, head_dim], token stride q_token_stride
 *       elements (a multiple of 8, >= num_heads * head_dim), 16-byte aligned.
 *   key, value, caches, slot_mapping: as for pa_reshape_and_cache (any
 *       block_size).
 *   positions (device): int64 [num_tokens].
 * A token whose position is out of range is skipped entirely (q unrotated,
 * nothing cached) and sets PA_FLAG_POSITION_RANGE; a slot out of range sets
 * PA_FLAG_SLOT_RANGE.
 */
pa_status pa_rope_reshape_and_cache(void *q, int64_t q_token_stride, const void *key, const void *value,
                                    int64_t key_token_stride, int64_t value_token_stride,
                                    void *key_cache, void *value_cache, const int64_t *slot_mapping,
                                    const int64_t *positions, const float *cos_sin_cache,
                                    int32_t max_position, int32_t rotary_dim, int32_t is_neox,
                                    int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                    int32_t dtype, void *stream);

/*
 * The same rotation into 8-bit caches: q is rotated in place as above; the
 * rotated key row (rounded once to `dtype`, exactly as above) and the value
 * row are stored as the E4M3 codes of x / k_scale and x / v_scale, as
 * pa_reshape_and_cache_fp8 stores them. key_cache, value_cache: (device)
 * uint8 [num_blocks, block_size, num_kv_heads, head_dim], 16-byte aligned;
 * head_dim a multiple of 16; k_scale and v_scale finite and positive
 * (PA_ERR_DIMS otherwise). Other arguments and errors as above.
 */
pa_status pa_rope_reshape_and_cache_fp8(void *q, int64_t q_token_stride, const void *key, const void *value,
                                        int64_t key_token_stride, int64_t value_token_stride,
                                        void *key_cache, void *value_cache, const int64_t *slot_mapping,
                                        const int64_t *positions, const float *cos_sin_cache,
                                        int32_t max_position, int32_t rotary_dim, int32_t is_neox,
                                        int32_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                        float k_scale, float v_scale, int32_t dtype, void *stream);

/*
 * Copy-on-write block copy (LLM-infra reading map, §2.2: a physical block
 * shared by several requests is copied before one of them writes into it).
 * For each pair i < num_pairs, copy physical block block_mapping[2*i] to
 * physical block block_mapping[2*i + 1] in both caches: all block_size
 * tokens, all KV heads, raw bits: dtype PA_BF16 or PA_FP16 for 16-bit caches,
 * PA_FP8_E4M3 for 8-bit ones (head_dim a multiple of 16 then).
 *   key_cache, value_cache (device): [num_blocks, block_size, num_kv_heads,
 *       head_dim], 16-byte aligned, head_dim a multiple of 8.
 *   block_mapping (device): int64 [num_pairs, 2] = (source, destination).
 * Destinations must be distinct and no destination may also be a source in
 * the same call (the result is unspecified otherwise). A pair with an id
 * outside [0, num_blocks) is skipped and sets PA_FLAG_BLOCK_RANGE.
 * Returns PA_OK without launching when num_pairs == 0.
 */
pa_status pa_copy_blocks(void *key_cache, void *value_cache, const int64_t *block_mapping,
                         int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int64_t num_blocks, int32_t dtype, void *stream);

/*
 * Block-table addressing on its own: copy the seq_len logical K/V rows of one
 * request, read through its block-table row, into contiguous
 * [seq_len, num_kv_heads, head_dim] buffers (device, 16-byte aligned), raw
 * bits of `dtype` (PA_BF16, PA_FP16, or PA_FP8_E4M3 for 8-bit caches).
 * block_table_row is a device pointer to that request's row. Used to check
 * the addressing bit for bit.
 */
pa_status pa_gather_kv(const void *key_cache, const void *value_cache,
                       const int32_t *block_table_row, int32_t seq_len,
                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int64_t num_blocks, void *key_out, void *value_out,
                       int32_t dtype, void *stream);

/* Human-readable name of a pa_status value (static string). */
const char *pa_status_string(int32_t status);

/*
 * Synchronise `stream`, then read and clear the current device's status word.
 * *flags_out (host, may be NULL) receives the PA_FLAG_* bits that were set.
 * Returns PA_ERR_DEVICE_BOUNDS if any bit was set, PA_ERR_CUDA if the
 * synchronisation failed, PA_OK otherwise.
 */
pa_status pa_debug_status(void *stream, uint32_t *flags_out);

/* Number of kernels this library has launched in this process. */
uint64_t pa_launch_count(void);

/*
 * Name of the CUDA runtime error (a static string such as
 * "cudaErrorInvalidValue") behind the last PA_ERR_LAUNCH or PA_ERR_CUDA that
 * a call made by this host thread returned; "cudaSuccess" if there was none.
 * Makes no CUDA call that touches a device.
 */
const char *pa_last_cuda_error(void);

/*
 * Measurement hook: the next pa_attention_varlen call made by this host
 * thread records `start` (a cudaEvent_t) just before its split-KV attention
 * kernel and `stop` just after it, on the call's stream, then forgets them.
 * Pass NULL, NULL to cancel.
 */
pa_status pa_attention_set_timing_events(void *start, void *stop);

/*
 * The same for the prefill-tile (tensor-core) kernel of the next
 * pa_attention_varlen / pa_attention_varlen_fp8 call by this host thread; the
 * events are not recorded if that call launches no tile kernel (no request
 * has more than 8 / (num_heads / num_kv_heads) query tokens).
 */
pa_status pa_attention_set_tile_timing_events(void *start, void *stop);

/*
 * Attention without a caller-provided workspace, for callers that cannot
 * call cudaMalloc: a plugin inside a host framework that owns every device
 * allocation and hands the plugin only its inputs and outputs, or a serving
 * process whose device memory is all reserved up front by its own pool, so
 * that a further allocation would fail or fragment it. The pages describe no
 * such call; it exists only for these callers.
 *
 * Same arguments and result as pa_attention_varlen, minus `workspace` and
 * `workspace_bytes`: the split-KV plan and partials live in a scratch array
 * compiled into the library (PA_STATIC_WORKSPACE_BYTES bytes of device
 * memory, held on every GPU that loads the library until the process exits).
 * The call itself allocates nothing.
 *
 *   - A problem whose workspace exceeds PA_STATIC_WORKSPACE_BYTES is
 *     rejected with PA_ERR_WORKSPACE before anything is launched; use
 *     pa_attention_varlen for it. The size checked is that of the plan
 *     pa_attention_varlen makes for 16-bit caches (at most
 *     pa_attention_workspace_size(), which also covers 8-bit caches).
 *   - The first call on a device looks up that device's copy of the scratch
 *     array (with the device current); make that first call before any
 *     stream capture. Later calls only read the cached address. A lookup
 *     that fails returns PA_ERR_CUDA (pa_last_cuda_error() names the
 *     error) and is tried again by the next call.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind. Nothing in it needs to start at zero (the planning kernel
 *     rewrites every word that later kernels read), but calls whose kernels
 *     overlap on the GPU (different streams, no ordering between them) race
 *     on the array and produce garbage. Order such calls on one stream.
 */
#define PA_STATIC_WORKSPACE_BYTES (32u << 20)

pa_status pa_attention_varlen_static(const void *q, int64_t q_token_stride,
                                     const void *key_cache, const void *value_cache,
                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                     const int32_t *seq_lens, const int32_t *query_start_loc,
                                     int32_t num_seqs, int32_t total_q_tokens,
                                     int32_t max_query_len, int32_t max_seq_len,
                                     int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                     int32_t block_size, int64_t num_blocks, float scale,
                                     void *out, int32_t dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
