/*
 * qattn -- the attention step of a Qwen2 decoder layer over a block-paged KV
 * cache, as a C ABI over hand-written sm_103a CUDA kernels.
 *
 * The step (restated from the pages it comes from):
 *   1. rotate-half RoPE with rope_theta = 1e6 on the query and key heads of
 *      the fused QKV projection output -- get_rope(head_dim,
 *      rotary_dim=head_dim, max_position, base=rope_theta) in
 *      "Qwen2大模型架构解析与vLLM优化实践" section 2.2; the 1e6 default in
 *      "Qwen2 模型结构代码详解" section 2 (配置解析);
 *   2. the new K/V rows written into fixed-size cache blocks through a slot
 *      mapping -- PagedAttention block cache (vLLM-deploys-Qwen notes,
 *      gsyq.cn, section 2.1) and the per-sequence block_table plus
 *      prepare_prefill context of the nano-vllm Qwen3 skeleton page,
 *      section 5;
 *   3. grouped-query attention, num_heads / num_kv_heads query heads per KV
 *      head, scale head_dim ** -0.5 ("Qwen2 模型结构代码详解" section 2;
 *      Attention(...) in "Qwen2大模型架构解析与vLLM优化实践" section 4.1),
 *      gathering each sequence's blocks through its block table: decode, and
 *      causal varlen / chunked prefill (FlashAttention-2 varlen in the Qwen
 *      engineering notes, 0539edu.com, section 2.1).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers unless the argument says host.
 *     The caller owns every buffer; the library allocates no device memory
 *     and keeps no device state between calls -- with one exception,
 *     qattn_paged_decode_noalloc, whose split-KV scratch is a fixed array
 *     inside the library (see its declaration).
 *   - Any entry point may be called from several host threads, and for any
 *     device (the current device of the calling thread): the host-side
 *     caches (SM counts, encoded tensor maps, the kernels' shared-memory
 *     limits, set once per device; the shared-prefix calls' side stream and
 *     events, created once per device) are lock-protected.
 *   - bf16 everywhere for activations and cache; int32 for every index.
 *   - Cache layout: k_cache and v_cache are [num_blocks][num_kv_heads]
 *     [block_size][head_dim] bf16, contiguous.  Token slot s lives in block
 *     s / block_size at offset s % block_size.  Both base pointers must be
 *     16-byte aligned.
 *   - Query head h reads KV head h / (num_heads / num_kv_heads).
 *   - Row strides are in elements and must be multiples of 8 (16 bytes);
 *     head h of a row starts at element h * head_dim of the row.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  The return value reports host-side
 *     argument checks and launch errors only.
 *   - Data-dependent errors are found on the device: the offending element
 *     is skipped and a bit is OR-ed into *err_word (a device int32 that the
 *     caller zeroes; may be NULL).  Kernels never trap.  Outputs of a row
 *     that raised an error bit are unspecified.
 *   - Supported today: head_dim 128, block_size 16, 32 or 64, num_heads a multiple of
 *     num_kv_heads with at most 8 query heads per KV head, num_heads <= 128.
 *     Anything else returns QATTN_ERR_UNSUPPORTED without launching.
 *   - A call with zero tokens / zero sequences returns QATTN_OK and launches
 *     nothing.
 */
#ifndef QATTN_H_
#define QATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Model shape of one attention layer. */
typedef struct qattn_dims {
  int32_t num_heads;    /* H: query heads */
  int32_t num_kv_heads; /* Hkv: key/value heads (GQA group = H / Hkv) */
  int32_t head_dim;     /* D (128) */
  int32_t block_size;   /* tokens per cache block (16, 32 or 64) */
  float scale;          /* softmax scale; <= 0 selects head_dim ** -0.5 */
} qattn_dims;

/* Host-side return codes. */
enum {
  QATTN_OK = 0,
  QATTN_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad stride/alignment */
  QATTN_ERR_UNSUPPORTED = 2, /* shape outside the supported set above */
  QATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call or launch failed */
  QATTN_ERR_WORKSPACE = 4    /* workspace missing or smaller than required */
};

/* Bits OR-ed into the optional device error word. */
enum {
  QATTN_DEVERR_SLOT = 1,      /* slot_mapping entry >= num_blocks * block_size */
  QATTN_DEVERR_BLOCK = 2,     /* block_tables entry outside [0, num_blocks) */
  QATTN_DEVERR_CONTEXT = 4,   /* context_len <= 0, > max_context_len, or
                                 smaller than the sequence's query count;
                                 bad cu_seqlens_q */
  QATTN_DEVERR_TIMEOUT = 8,   /* a bounded wait inside a kernel gave up */
  QATTN_DEVERR_POSITION = 16, /* position outside [0, max_pos) */
  QATTN_DEVERR_PREFIX = 32    /* a block table does not start with the shared
                                 prefix blocks of row 0 */
};

/* Human-readable name of a return code (static storage). */
const char* qattn_status_string(int status);

/* Library version as major * 10000 + minor * 100 + patch. */
int qattn_version(void);

/* Build the RoPE cos/sin table on the HOST, once per model (the table that
 * get_rope(head_dim, rotary_dim=head_dim, max_position, base) owns;
 * "Qwen2大模型架构解析与vLLM优化实践" section 2.2).  host_cos_sin receives
 * [max_pos][head_dim] fp32: columns i < head_dim/2 hold
 * cos(pos * theta^(-2i/head_dim)) and column head_dim/2 + i the matching
 * sin, each evaluated in fp64 and rounded to fp32.  The caller copies it to
 * the device.  Returns QATTN_INVALID_ARG for a null pointer, max_pos <= 0,
 * an odd head_dim or theta <= 0. */
int qattn_rope_table_build(float* host_cos_sin, int32_t max_pos,
                           int32_t head_dim, double theta);

/* The same table with rope_scaling ("Qwen2大模型架构解析与vLLM优化实践"
 * section 7.1: rope_scaling = {type, factor, original_max_position}):
 *   QATTN_ROPE_SCALING_NONE     the table above;
 *   QATTN_ROPE_SCALING_LINEAR   position interpolation: angle =
 *                               (pos / factor) * theta^(-2i/D);
 *   QATTN_ROPE_SCALING_DYNAMIC  dynamic NTK: when max_pos exceeds
 *                               original_max_position the base becomes
 *                               theta * (factor * max_pos /
 *                               original_max_position - (factor - 1))
 *                               ^ (D / (D - 2)); otherwise unchanged.  max_pos
 *                               stands for the batch's sequence-length bound
 *                               (a longer batch builds a new table).
 * Angles in fp64, rounded to fp32.  QATTN_ERR_INVALID_ARG for a null pointer,
 * max_pos <= 0, head_dim odd or <= 2, theta <= 0, an unknown scaling,
 * factor < 1, or a dynamic table without original_max_position > 0. */
#define QATTN_ROPE_SCALING_NONE 0
#define QATTN_ROPE_SCALING_LINEAR 1
#define QATTN_ROPE_SCALING_DYNAMIC 2
int qattn_rope_table_build_scaled(float* host_cos_sin, int32_t max_pos,
                                  int32_t head_dim, double theta,
                                  int32_t scaling, double factor,
                                  int32_t original_max_position);

/* Step 1 + 2: rotate-half RoPE and cache append, one launch.
 *   q        [num_tokens, q_row_stride] bf16, rotated IN PLACE (heads
 *            0 .. num_heads-1 of each row);
 *   k, v     [num_tokens, *_row_stride] bf16, read only (num_kv_heads heads
 *            per row); k is rotated on the way into k_cache, v copied as is.
 *            For the fused QKV output [T, (H + 2 Hkv) * D] pass
 *            q = base, k = base + H*D, v = base + (H + Hkv)*D and the same
 *            row stride (H + 2 Hkv) * D for all three;
 *   positions    [num_tokens] int32 rotary position of each token;
 *   slot_mapping [num_tokens] int32 cache slot of each token, < 0 = padding
 *            (q is still rotated, nothing is written to the cache);
 *   cos_sin  [max_pos, head_dim] fp32 table from qattn_rope_table_build.
 * Rotation arithmetic, element pair (i, i + D/2):
 *   y_i = x_i c - x_{i+D/2} s,  y_{i+D/2} = x_{i+D/2} c + x_i s,
 * every product and sum rounded to fp32 (no fused multiply-add), the result
 * rounded to bf16 nearest-even -- so the cache contents are bit-reproducible.
 * Device errors: QATTN_DEVERR_POSITION (token skipped entirely),
 * QATTN_DEVERR_SLOT (cache write skipped).  Duplicate non-negative slots in
 * one call are undefined. */
int qattn_rope_cache_append(void* q, int64_t q_row_stride, const void* k,
                            int64_t k_row_stride, const void* v,
                            int64_t v_row_stride, const int32_t* positions,
                            const int32_t* slot_mapping, int32_t num_tokens,
                            void* k_cache, void* v_cache, int32_t num_blocks,
                            const float* cos_sin, int32_t max_pos,
                            qattn_dims dims, int32_t* err_word, void* stream);

/* qattn_rope_cache_append with two optional steps before the rotation, for
 * the layers whose projection output has not had them yet:
 *   qkv_bias       [(H + 2 Hkv) * head_dim] bf16 (q heads, then k, then v),
 *                  or NULL: x' = bf16(x + b), one rounding (the Qwen2 qkv
 *                  projection's bias=True, "Qwen2大模型架构解析与vLLM优化实践";
 *                  v too);
 *   q_norm_weight, k_norm_weight  [head_dim] bf16, or NULL: the Qwen3
 *                  attention's per-head RMSNorm of q and of k (nano-vllm Qwen3
 *                  skeleton page, module tree q_norm / k_norm), applied after
 *                  the bias: ss = the sum of squares of the head in fp32,
 *                  slice p = dims 8p .. 8p+7 then 64+8p .. 64+8p+7 summed in
 *                  order, the 8 slice sums as ((s0+s1)+(s2+s3))+((s4+s5)+
 *                  (s6+s7)); v = fp32(ss / head_dim + norm_eps), r = 1 /
 *                  sqrt(v) (correctly rounded fp32), y = bf16(fp32(fp32(x *
 *                  r) * w)), every fp32 step rounded, no fused multiply-add;
 *   norm_eps       rms_norm_eps (1e-6 for Qwen2/Qwen3), 0 <= eps < 1.
 * The cache stays bit-reproducible.  Pointers must be 16-byte aligned.
 * Same errors as qattn_rope_cache_append. */
int qattn_rope_cache_append_ex(void* q, int64_t q_row_stride, const void* k,
                               int64_t k_row_stride, const void* v,
                               int64_t v_row_stride, const int32_t* positions,
                               const int32_t* slot_mapping, int32_t num_tokens,
                               void* k_cache, void* v_cache, int32_t num_blocks,
                               const float* cos_sin, int32_t max_pos,
                               const void* qkv_bias, const void* q_norm_weight,
                               const void* k_norm_weight, float norm_eps,
                               qattn_dims dims, int32_t* err_word, void* stream);

/* ---- FP8 KV cache ----------------------------------------------------
 *
 * kv_cache_dtype "fp8": fp8_e4m3fn codes with one cache scale per tensor
 * (the K scale and the V scale of the layer), "Qwen2大模型架构解析与vLLM
 * 优化实践" sections 4.1 (KV cache quantisation), 4.2 (the cache scale
 * loaded per tensor, kv_cache_dtype="fp8") and 6.3 (fp8_e4m3fn).  The cache
 * has the bf16 cache's shape with 1-byte elements: [num_blocks][Hkv]
 * [block_size][head_dim] uint8, 16-byte aligned.  Element x of a bf16 cache
 * is stored as e4m3(x / scale): the fp32 quotient (correctly rounded)
 * rounded to the nearest e4m3fn value, ties to even, magnitudes past 448
 * saturated to 448.  The attention entry points read code * scale.  Decode
 * takes q . k on the codes themselves (e4m3 tensor-core products, fp32
 * accumulation), with each head's q as the sum of two e4m3 parts under a
 * power-of-two scale of that head: the sum equals the bf16 q exactly for
 * every element within a factor 2^9 of the head's largest |q|, and is off
 * by at most 2^-17 of that largest |q| for the others (q must be finite:
 * the e4m3 conversion saturates an infinite element to the format's range;
 * a NaN stays NaN).  P V in decode,
 * and both products of prefill and the shared-prefix pass, run on the
 * codes converted exactly (to f16 in decode, with the softmax weights
 * rounded to f16; to bf16 in prefill).  k_scale multiplies the logits'
 * scale and v_scale the output.
 * Scales must be finite, positive and normal fp32 (QATTN_ERR_INVALID_ARG
 * otherwise). */

/* qattn_rope_cache_append_ex into an FP8 cache: the bf16 key (after bias,
 * norm and RoPE) and value rows are stored as e4m3(x / k_scale) and
 * e4m3(x / v_scale).  q is rotated in place exactly as by the bf16 entry
 * points.  Same arguments and errors otherwise. */
int qattn_rope_cache_append_fp8(void* q, int64_t q_row_stride, const void* k,
                                int64_t k_row_stride, const void* v,
                                int64_t v_row_stride, const int32_t* positions,
                                const int32_t* slot_mapping, int32_t num_tokens,
                                void* k_cache, void* v_cache, int32_t num_blocks,
                                const float* cos_sin, int32_t max_pos,
                                const void* qkv_bias, const void* q_norm_weight,
                                const void* k_norm_weight, float norm_eps,
                                float k_scale, float v_scale, qattn_dims dims,
                                int32_t* err_word, void* stream);

/* Bytes of device workspace qattn_paged_decode needs (256-byte aligned
 * pointer, contents need not be initialised).  Depends only on the
 * arguments.  The workspace holds the split-KV partial results between the
 * decode kernel and the merge kernel of one call; two calls whose kernels
 * can overlap on the GPU must not share a workspace. */
size_t qattn_paged_decode_workspace_size(int32_t num_seqs,
                                         int32_t max_context_len,
                                         qattn_dims dims);

/* Testing hook for the decode kernel's failure path (the pages have no
 * counterpart).  Every decode launch after this call (qattn_paged_decode,
 * its FP8 and no-allocation variants, the decode rows of the varlen and
 * shared-prefix calls) limits each of its bounded waits to wait_limit_ns
 * (0 restores the default of 2 s; otherwise 1000 .. 2e9), and, if
 * skip_k_copy >= 0, the decode kernel's first CTA does not issue the copy of
 * its K tile number skip_k_copy, so that the waits on that tile run out.
 * Such a call still returns QATTN_OK; on the device every role of the
 * stalled CTA gives up, its copies and MMAs in flight are drained (at most
 * max(wait_limit_ns, 10 ms) each) and its tensor memory is freed, and
 * QATTN_DEVERR_TIMEOUT is set in the error word; that call's output is
 * unspecified, and the next call with the defaults restored is unaffected.
 * Process-wide state, not synchronised with calls in flight on other host
 * threads: for tests only.  Returns QATTN_ERR_INVALID_ARG for values out of
 * range. */
int qattn_debug_decode_faults(int64_t wait_limit_ns, int32_t skip_k_copy);

/* Step 3, decode: one query row per sequence.
 *   out          [num_seqs, num_heads, head_dim] bf16, contiguous;
 *   q            [num_seqs, q_row_stride] bf16 (already rotated);
 *   block_tables [num_seqs, max_blocks_per_seq] int32 physical block ids;
 *   context_lens [num_seqs] int32 tokens in the cache for each sequence,
 *                including the one appended this step (the query sits at
 *                position context_len - 1 and sees every cached token);
 *   max_context_len  host upper bound on context_lens (sizes the split
 *                workspace; a larger device value raises
 *                QATTN_DEVERR_CONTEXT).
 * out[b, h] = sum_j softmax_j(scale * q[b,h] . k_j) v_j over j <
 * context_lens[b], keys and values of KV head h / (H / Hkv).  Accumulation
 * is fp32; the work is split into fixed token ranges whose partial results
 * (normalised output and log-sum-exp) are merged by a second kernel in a
 * fixed order, so results are run-to-run bit-identical.  Rows with
 * context_len <= 0 are written as zeros with QATTN_DEVERR_CONTEXT. */
int qattn_paged_decode(void* out, const void* q, int64_t q_row_stride,
                       const void* k_cache, const void* v_cache,
                       int32_t num_blocks, const int32_t* block_tables,
                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                       int32_t num_seqs, int32_t max_context_len,
                       qattn_dims dims, void* workspace, size_t workspace_bytes,
                       int32_t* err_word, void* stream);

/* qattn_paged_decode over FP8 caches (uint8 e4m3 codes, see above):
 * out = attention over code * k_scale keys and code * v_scale values, on
 * the tensor-core kernel for every group size and block size.  Workspace
 * as qattn_paged_decode_workspace_size.  Same arguments and errors as
 * qattn_paged_decode, plus QATTN_ERR_INVALID_ARG for an invalid scale. */
int qattn_paged_decode_fp8(void* out, const void* q, int64_t q_row_stride,
                           const void* k_cache, const void* v_cache,
                           int32_t num_blocks, const int32_t* block_tables,
                           int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t num_seqs,
                           int32_t max_context_len, float k_scale, float v_scale,
                           qattn_dims dims, void* workspace, size_t workspace_bytes,
                           int32_t* err_word, void* stream);

/* Bytes of workspace qattn_paged_decode_shared_prefix needs (same rules as
 * qattn_paged_decode_workspace_size; room for the prefix parts too). */
size_t qattn_paged_decode_shared_prefix_workspace_size(int32_t num_seqs,
                                                       int32_t max_context_len,
                                                       qattn_dims dims);

/* qattn_paged_decode for a batch whose sequences share a cached prefix
 * (prefix caching, "Qwen2 模型结构代码详解" sections 3-4, over the shared
 * blocks of the PagedAttention cache, vLLM-deploys-Qwen notes section 2.1): tokens
 * 0 .. shared_prefix_len - 1 of EVERY sequence are the same cached tokens
 * in the same physical blocks, block_tables[b][j] == block_tables[0][j] for
 * j < shared_prefix_len / block_size.  Same arguments and result as
 * qattn_paged_decode, plus
 *   shared_prefix_len  host, a multiple of block_size, 0 <= it < every context_len
 *                      (0: plain decode), < max_context_len.
 * The prefix is attended once per kv head for the whole batch on tensor
 * cores (all sequences' query groups against the prefix tiles) on an eighth
 * of the SMs, at the same time as the decode kernel reads each sequence's
 * remaining tokens on the others, and the parts are merged in a fixed order
 * (deterministic).  The prefix pass runs on a stream of the library's own,
 * forked from and joined back into `stream` with events (one stream and two
 * events per device, created on the first call): the work is still ordered
 * on `stream`, and the call may be captured into a CUDA graph.  Device errors: those
 * of qattn_paged_decode, a context_len <= shared_prefix_len gives a zero row
 * and QATTN_DEVERR_CONTEXT, a table that does not start with row 0's prefix
 * blocks QATTN_DEVERR_PREFIX (its result is then unspecified). */
int qattn_paged_decode_shared_prefix(void* out, const void* q, int64_t q_row_stride,
                                     const void* k_cache, const void* v_cache,
                                     int32_t num_blocks, const int32_t* block_tables,
                                     int32_t max_blocks_per_seq, const int32_t* context_lens,
                                     int32_t num_seqs, int32_t max_context_len,
                                     int32_t shared_prefix_len, qattn_dims dims,
                                     void* workspace, size_t workspace_bytes,
                                     int32_t* err_word, void* stream);

/* qattn_paged_decode_shared_prefix over FP8 caches (uint8 e4m3 codes).  The
 * prefix blocks (those of table row 0) are copied into the workspace as bf16
 * values of their codes (exact) and the prefix pass runs on the copy; each
 * sequence's own tokens are read as codes by the FP8 decode.  Workspace:
 * qattn_paged_decode_shared_prefix_fp8_workspace_size(num_seqs,
 * max_context_len, shared_prefix_len, dims) bytes.  Same arguments and
 * errors as qattn_paged_decode_shared_prefix, plus the scales. */
size_t qattn_paged_decode_shared_prefix_fp8_workspace_size(int32_t num_seqs,
                                                           int32_t max_context_len,
                                                           int32_t shared_prefix_len,
                                                           qattn_dims dims);
int qattn_paged_decode_shared_prefix_fp8(void* out, const void* q, int64_t q_row_stride,
                                         const void* k_cache, const void* v_cache,
                                         int32_t num_blocks, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t num_seqs,
                                         int32_t max_context_len,
                                         int32_t shared_prefix_len, float k_scale,
                                         float v_scale, qattn_dims dims, void* workspace,
                                         size_t workspace_bytes, int32_t* err_word,
                                         void* stream);

/* qattn_paged_decode for callers that cannot allocate device memory (code
 * running inside someone else's CUDA-graph capture, a serving loop whose
 * memory pool is fixed at start-up, a host that only lends the tensors it
 * computes on).  Same arguments and results as qattn_paged_decode, without
 * the workspace: the split-KV partial results go to a 32 MiB scratch array
 * compiled into this library, which every GPU that loads the library keeps
 * until the process exits.  This entry point has no counterpart on the
 * pages; it exists only because of those callers.
 *   - Shapes whose qattn_paged_decode_workspace_size() exceeds 32 MiB
 *     (33554432 bytes) are refused with QATTN_ERR_WORKSPACE before any
 *     launch (e.g. 64 sequences x 4096 tokens x 28 heads needs ~16 MiB).
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress); make that first call
 *     before any stream capture.  No call allocates or frees memory.
 *   - All calls share the array and it keeps the previous call's contents;
 *     nothing in it needs to start at zero.  Calls whose kernels may run at
 *     the same time on the GPU (unordered streams) race on it: order them,
 *     or use qattn_paged_decode with workspaces of your own. */
int qattn_paged_decode_noalloc(void* out, const void* q, int64_t q_row_stride,
                               const void* k_cache, const void* v_cache,
                               int32_t num_blocks, const int32_t* block_tables,
                               int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t num_seqs,
                               int32_t max_context_len, qattn_dims dims,
                               int32_t* err_word, void* stream);

/* Bytes of device workspace qattn_varlen_prefill needs (same rules). */
size_t qattn_varlen_prefill_workspace_size(int32_t num_seqs,
                                           int32_t max_context_len,
                                           qattn_dims dims);

/* Step 3, causal varlen / chunked prefill over a mixed batch.
 *   out          [total_q, num_heads, head_dim] bf16, contiguous;
 *   q            [total_q, q_row_stride] bf16 (already rotated);
 *   cu_seqlens_q [num_seqs + 1] int32, cu_seqlens_q[0] = 0,
 *                cu_seqlens_q[num_seqs] = total_q: query rows of sequence b
 *                are cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1;
 *   max_q_len    host upper bound on any sequence's query count, at most
 *                49152 (QATTN_ERR_UNSUPPORTED above, before any launch);
 *   context_lens [num_seqs] tokens in the cache for each sequence after
 *                this step's append (cached + new).
 * Query i of sequence b (q_len = cu_seqlens_q[b+1] - cu_seqlens_q[b],
 * L = context_lens[b]) sits at position L - q_len + i and attends keys
 * 0 .. L - q_len + i (causal, aligned to the end of the context).
 * Sequences with q_len == 1 are decode rows and take the decode kernel's
 * path; longer ones use the tensor-core prefill kernel.  Both run on
 * `stream`.  Rows of a sequence with q_len > L or L <= 0 are zeroed with
 * QATTN_DEVERR_CONTEXT. */
int qattn_varlen_prefill(void* out, const void* q, int64_t q_row_stride,
                         const int32_t* cu_seqlens_q, int32_t num_seqs,
                         int32_t total_q, int32_t max_q_len,
                         const void* k_cache, const void* v_cache,
                         int32_t num_blocks, const int32_t* block_tables,
                         int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t max_context_len,
                         qattn_dims dims, void* workspace,
                         size_t workspace_bytes, int32_t* err_word,
                         void* stream);

/* qattn_varlen_prefill over FP8 caches (uint8 e4m3 codes, see above).  The
 * decode rows read the codes directly (as qattn_paged_decode_fp8); for the
 * prefill rows (two or more new queries) the sequences' blocks are first
 * copied into the workspace as bf16 values of the codes (exact: every e4m3
 * value is a bf16 number), then the bf16 tensor-core prefill runs on the
 * copy with k_scale folded into the logit scale and v_scale into the
 * output.
 *   num_prefill_seqs  host, an upper bound on the sequences with two or
 *                     more new queries (the copy's capacity, in sequences
 *                     of up to max_context_len tokens); a sequence beyond it
 *                     sets QATTN_DEVERR_CONTEXT and its rows are
 *                     unspecified.
 *   workspace         qattn_varlen_prefill_fp8_workspace_size(num_seqs,
 *                     num_prefill_seqs, max_context_len, dims) bytes.
 * Same arguments and errors as qattn_varlen_prefill otherwise. */
size_t qattn_varlen_prefill_fp8_workspace_size(int32_t num_seqs,
                                               int32_t num_prefill_seqs,
                                               int32_t max_context_len,
                                               qattn_dims dims);
int qattn_varlen_prefill_fp8(void* out, const void* q, int64_t q_row_stride,
                             const int32_t* cu_seqlens_q, int32_t num_seqs,
                             int32_t total_q, int32_t max_q_len,
                             const void* k_cache, const void* v_cache,
                             int32_t num_blocks, const int32_t* block_tables,
                             int32_t max_blocks_per_seq,
                             const int32_t* context_lens,
                             int32_t max_context_len, int32_t num_prefill_seqs,
                             float k_scale, float v_scale, qattn_dims dims,
                             void* workspace, size_t workspace_bytes,
                             int32_t* err_word, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QATTN_H_ */
