// Host-side launch interfaces between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/qattn.h"

namespace qattn {

// Launch with programmatic stream serialization (see grid_dep_wait).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// How a decode kernel cuts its list of T work units (chunks or tiles) into
// contiguous runs, one per CTA of a grid of P CTAs.  With T >= min_run * P
// the runs are balanced: CTA k owns [floor(k T / P), floor((k+1) T / P)),
// every run at least min_run long.  Otherwise runs are exactly min_run long
// and only the first ceil(T / min_run) CTAs work.  Either way a unit of n
// consecutive work items touches at most ceil(n / min_run) + 1 runs.
struct RunSplit {
  int total;    // T
  int ctas;     // P
  int min_run;  // minimum run length
  __host__ __device__ bool balanced() const {
    return static_cast<long long>(total) >= static_cast<long long>(min_run) * ctas;
  }
  __host__ __device__ int begin(int k) const {
    if (balanced()) return static_cast<int>(static_cast<long long>(k) * total / ctas);
    const long long b = static_cast<long long>(k) * min_run;
    return b < total ? static_cast<int>(b) : total;
  }
  // The CTA whose run holds work item u (0 <= u < total).
  __host__ __device__ int cta_of(int u) const {
    if (balanced())
      return static_cast<int>((static_cast<long long>(u + 1) * ctas - 1) / total);
    return u / min_run;
  }
};

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
  int32_t* cum;    // [num_seqs] work-list offset of each sequence, then a
                   // header: [num_seqs] = total, [num_seqs + 1] = grid size,
                   // [num_seqs + 2] = minimum run
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
#ifdef __CUDACC__
// Every CTA of a decode kernel touches the context lengths (planning) and,
// right after, a slice of the block tables it cannot know in advance.
// Prefetching both whole arrays into L2 at entry turns the second of those
// two dependent DRAM round trips into an L2 hit.  (Inputs only: these are
// never written by the previous kernel on the stream.)
__device__ __forceinline__ void prefetch_decode_metadata(const DecodeArgs& a) {
  const char* bt = reinterpret_cast<const char*>(a.block_tables);
  const int64_t bt_bytes = static_cast<int64_t>(a.num_seqs) * a.max_blocks_per_seq * 4;
  for (int64_t off = static_cast<int64_t>(threadIdx.x) * 128; off < bt_bytes;
       off += static_cast<int64_t>(blockDim.x) * 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(bt + off));
  const char* cl = reinterpret_cast<const char*>(a.context_lens);
  for (int64_t off = static_cast<int64_t>(threadIdx.x) * 128; off < a.num_seqs * 4LL;
       off += static_cast<int64_t>(blockDim.x) * 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(cl + off));
}

// Context length of decode sequence b if it is valid for a decode kernel
// (one query row; 1 <= L <= max_context_len; within the block table), else 0.
__device__ __forceinline__ int decode_len_eff(const DecodeArgs& a, int b) {
  const int L = a.context_lens[b];
  if (a.cu_seqlens_q != nullptr) {
    if (a.cu_seqlens_q[b + 1] - a.cu_seqlens_q[b] != 1) return 0;
  }
  if (L < 1 || L > a.max_context_len || L > a.max_blocks_per_seq * 16) return 0;
  return L;
}

// Called by one full warp of CTA 0 of a decode kernel: waits for the
// previous grid, then writes the work-list offset of every sequence (units
// of `unit_tokens` tokens, one list entry per (sequence, kv head, unit)) and
// the run-split header [total, grid size, minimum run] the merge kernel
// reads.  s_len: the kernel's shared copy of decode_len_eff per sequence, or
// null when the batch did not fit in it.
__device__ __forceinline__ void write_unit_offsets(const DecodeArgs& a, const int* s_len,
                                                   int total, int unit_tokens, int min_run) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  int run = 0;
  for (int base = 0; base < a.num_seqs; base += 32) {
    const int b = base + lane;
    int u = 0;
    if (b < a.num_seqs) {
      const int L = s_len != nullptr ? s_len[b] : decode_len_eff(a, b);
      u = a.num_kv_heads * ((L + unit_tokens - 1) / unit_tokens);
    }
    int incl = u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (b < a.num_seqs) a.ws.cum[b] = run + incl - u;
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (lane == 0) {
    a.ws.cum[a.num_seqs] = total;
    a.ws.cum[a.num_seqs + 1] = static_cast<int>(gridDim.x);
    a.ws.cum[a.num_seqs + 2] = min_run;
  }
}
#endif
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
