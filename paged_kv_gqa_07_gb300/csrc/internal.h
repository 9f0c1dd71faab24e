// Host-side launch interfaces between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/qattn.h"

namespace qattn {

// ---- rope + cache append (rope_append.cu) ----
struct RopeAppendArgs {
  void* q;
  int64_t q_row_stride;
  const void* k;
  int64_t k_row_stride;
  const void* v;
  int64_t v_row_stride;
  const int32_t* positions;
  const int32_t* slot_mapping;
  int32_t num_tokens;
  void* k_cache;
  void* v_cache;
  int32_t num_blocks;
  const float* cos_sin;
  int32_t max_pos;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t* err_word;
};
cudaError_t launch_rope_append(const RopeAppendArgs& a, cudaStream_t stream);

// ---- paged decode (paged_decode.cu) ----
// Decode-mode work comes in fixed chunks of 32 tokens (two cache blocks);
// every CTA of the persistent grid owns a contiguous run of at least
// kMinChunksPerCta chunks of the (sequence, kv head, chunk) space.
constexpr int kChunkTokens = 32;
constexpr int kMinChunksPerCta = 8;

struct DecodeWorkspace {
  int32_t* cum;    // [num_seqs] chunk-space offset of each sequence (+ header)
  float* lse;      // [num_seqs * Hkv * max_parts * group]
  float* part_o;   // [num_seqs * Hkv * max_parts * group * 128]
  int32_t max_parts;
};

size_t decode_workspace_bytes(int32_t num_seqs, int32_t max_context_len, int32_t num_kv_heads,
                              int32_t group);
DecodeWorkspace carve_decode_workspace(void* base, int32_t num_seqs, int32_t max_context_len,
                                       int32_t num_kv_heads, int32_t group);

struct DecodeArgs {
  void* out;               // [rows, H, D] bf16
  const void* q;           // rows strided by q_row_stride
  int64_t q_row_stride;
  const int32_t* cu_seqlens_q;  // null: decode mode (row b = sequence b)
  const int32_t* context_lens;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_blocks;
  int32_t max_context_len;
  int32_t num_heads;
  int32_t num_kv_heads;
  float scale_log2;        // softmax scale * log2(e)
  int32_t* err_word;
  DecodeWorkspace ws;
  int32_t tile_tokens;     // tokens per work unit of the kernel that ran (merge needs it)
};
// CUDA-core decode (K2): 32-token chunks, the GQA group on CUDA cores.
cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, int num_sms, cudaStream_t stream);
// Tensor-core decode (K2t): 128-token tiles, the GQA group as the MMA N dimension.
constexpr int kTcTileTokens = 128;
constexpr int kTcMinTilesPerCta = 2;
cudaError_t launch_paged_decode_tc(const DecodeArgs& a, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, const CUtensorMap& qmap,
                                   int num_sms, cudaStream_t stream);
// K2r for either decode kernel (reads a.tile_tokens).
cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t stream);

// ---- varlen prefill (varlen_prefill.cu) ----
struct PrefillArgs {
  void* out;
  const void* q;
  int64_t q_row_stride;
  const int32_t* cu_seqlens_q;
  const int32_t* context_lens;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_blocks;
  int32_t total_q;
  int32_t max_q_len;
  int32_t max_context_len;
  int32_t num_heads;
  int32_t num_kv_heads;
  float scale_log2;
  int32_t* err_word;
};
cudaError_t launch_varlen_prefill(const PrefillArgs& a, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, int num_sms, cudaStream_t stream);

}  // namespace qattn
