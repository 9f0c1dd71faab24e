// Host-side launch interfaces between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments here are already validated.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/qattn.h"

namespace qattn {

// Raises a kernel's dynamic shared memory limit to `bytes` (0: leaves it)
// and asks for the largest shared-memory carve-out, on the current device,
// once per (kernel, device): the attributes belong to the device's context,
// so a process driving several GPUs sets them on each.  Thread-safe.
cudaError_t set_max_dynamic_smem(const void* kernel, int bytes);

// cuTensorMapEncodeTiled from the driver, looked up once (nullptr if the
// driver lacks it).  Thread-safe.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();

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
  int32_t block_size;      // tokens per cache block: 16, 32 or 64
  int32_t* err_word;
  // FP8 cache: e4m3 codes of x / k_scale and x / v_scale
  int32_t kv_fp8;
  float k_scale, v_scale;
  // Optional steps before RoPE (null: skipped): the qkv projection bias
  // [(H + 2 Hkv) * 128] bf16, and Qwen3's per-head RMSNorm weights [128]
  // bf16 for q and for k, with eps.
  const void* bias;
  const void* q_norm_w;
  const void* k_norm_w;
  float norm_eps;
};
cudaError_t launch_rope_append(const RopeAppendArgs& a, cudaStream_t stream);

// ---- paged decode (paged_decode_tc.cu) and its merge (decode_merge.cu) ----
// Decode work comes in 128-token tiles; every CTA of the persistent grid owns
// a contiguous run of at least kTcMinTilesPerCta tiles of the (sequence, kv
// head, tile) list.
constexpr int kTcTileTokens = 128;
constexpr int kTcMinTilesPerCta = 2;

// Parts a unit of max_context_len tokens can leave in the workspace: a run
// of n tiles meets at most ceil(n / kTcMinTilesPerCta) + 1 CTAs.
__host__ __device__ inline int64_t decode_max_parts(int64_t max_context_len) {
  const int64_t tiles = (max_context_len + kTcTileTokens - 1) / kTcTileTokens;
  return (tiles + kTcMinTilesPerCta - 1) / kTcMinTilesPerCta + 1;
}

struct DecodeWorkspace {
  int32_t* nparts;  // [num_seqs * Hkv] parts of each (sequence, kv head) unit, written
                    // by the decode kernel (0: no valid context), read by the merge
  float* lse;       // [num_seqs * Hkv * max_parts * group] log2-sum-exp of each part
  float* part_o;    // [num_seqs * Hkv * max_parts * group * 128] normalised O of each part
  int32_t max_parts;
};

// extra_parts: part slots a unit needs beyond its own split (shared-prefix
// parts).
size_t decode_workspace_bytes(int32_t num_seqs, int32_t max_context_len, int32_t num_kv_heads,
                              int32_t group, int32_t extra_parts = 0);
DecodeWorkspace carve_decode_workspace(void* base, int32_t num_seqs, int32_t max_context_len,
                                       int32_t num_kv_heads, int32_t group,
                                       int32_t extra_parts = 0);

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
  int32_t block_size;      // tokens per cache block: 16, 32 or 64
  float scale_log2;        // softmax scale * log2(e) (* k_scale for an FP8 cache)
  int32_t kv_fp8;          // the caches hold e4m3 codes
  float v_scale;           // FP8: multiplies the output
  int32_t* err_word;
  DecodeWorkspace ws;
  // Shared-prefix (cascade) mode: the kernel attends only to tokens
  // prefix_len .. L - 1 of every sequence (the prefix is done elsewhere),
  // and writes every unit as parts part_base + i of the workspace instead of
  // output rows.  Plain decode: both 0.
  int32_t prefix_len;
  int32_t part_base;
  // Limits of the kernel's bounded waits: every wait while working, and the
  // drain of copies and MMAs in flight before exit (never below 10 ms, so
  // that a short test limit cannot cut a drain short).
  uint64_t wait_ns;
  uint64_t drain_ns;
  // Testing only: the first CTA skips the copy of its K tile with this
  // index (-1: none), so that the wait on it runs out.
  int32_t debug_skip_k;
};
// Tensor-core decode (K2t): 128-token tiles, the GQA group as the MMA N
// dimension, on a grid of num_sms CTAs; then the merge (K2r), after
// merge_after (an event of work on another stream that writes parts), if
// given.
cudaError_t launch_paged_decode_tc(const DecodeArgs& a, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, const CUtensorMap& qmap,
                                   int num_sms, cudaStream_t stream,
                                   cudaEvent_t merge_after = nullptr);
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

// Tokens of decode sequence b the kernel attends to (L - prefix_len) if the
// row is valid for a decode kernel (one query row; prefix_len < L <=
// max_context_len; within the block table), else 0.
__device__ __forceinline__ int decode_len_eff(const DecodeArgs& a, int b) {
  const int L = a.context_lens[b];
  if (a.cu_seqlens_q != nullptr) {
    if (a.cu_seqlens_q[b + 1] - a.cu_seqlens_q[b] != 1) return 0;
  }
  if (L <= a.prefix_len || L > a.max_context_len || L > a.max_blocks_per_seq * a.block_size)
    return 0;
  return L - a.prefix_len;
}

// Block-table entries of sequence b from its first attended token on.
__device__ __forceinline__ const int32_t* decode_block_row(const DecodeArgs& a, int b) {
  return a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq +
         a.prefix_len / a.block_size;
}

// A unit that straddles CTAs leaves one partial result per CTA (O
// normalised by its own sum, LSE in log2 units) -- the split-KV scheme of
// the decode pages -- and the merge kernel K2r combines them.  The CTA that
// holds a unit's first part records how many parts it has.
__device__ __forceinline__ void record_parts(const DecodeArgs& a, int64_t seg, int nparts) {
  a.ws.nparts[seg] = nparts;
}

// Whole CTA, before any early exit.  Sequences b = blockIdx.x (mod grid):
// a decode row with no valid context gets a zero output row, no parts and
// the CONTEXT error bit; an empty varlen sequence (no query rows) gets the
// bit alone.
// s_len: the kernel's shared copy of decode_len_eff, or null.  Output is
// written only after the previous grid on the stream, which may write the
// same rows, has finished.
__device__ __forceinline__ void finish_invalid_rows(const DecodeArgs& a, const int* s_len) {
  for (int b = blockIdx.x; b < a.num_seqs; b += gridDim.x) {
    int64_t row = b;
    if (a.cu_seqlens_q != nullptr) {
      const int ql = a.cu_seqlens_q[b + 1] - a.cu_seqlens_q[b];
      if (ql != 1) {
        if (ql < 1 && threadIdx.x == 0) set_err(a.err_word, QATTN_DEVERR_CONTEXT);
        continue;  // a prefill sequence: the prefill kernel owns it
      }
      row = a.cu_seqlens_q[b];
    }
    const int L = s_len != nullptr ? s_len[b] : decode_len_eff(a, b);
    if (L > 0) continue;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int g = threadIdx.x; g < a.num_kv_heads; g += blockDim.x)
      a.ws.nparts[static_cast<int64_t>(b) * a.num_kv_heads + g] = 0;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                          row * a.num_heads * kHeadDim);
    for (int i = threadIdx.x; i < a.num_heads * (kHeadDim / 8); i += blockDim.x)
      dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) set_err(a.err_word, QATTN_DEVERR_CONTEXT);
  }
}
#endif

// K2r: merge the parts of straddling units.
cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t stream);

// Tracing build (-DQATTN_TRACE): per-CTA %globaltimer stamps of the decode
// kernel (slots: entry, plan done, first scores, every copy issued, softmax
// done, CTA done) and of the merge kernel (entry, decode grid seen, done).
constexpr int kTraceCtas = 1024;
constexpr int kTraceSlots = 8;
constexpr int kTraceMergeCtas = 16384;
#ifdef QATTN_TRACE
cudaError_t read_decode_trace(unsigned long long* host, size_t n);
cudaError_t clear_decode_trace();
cudaError_t read_merge_trace(unsigned long long* host, size_t n);
cudaError_t clear_merge_trace();
#endif

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
  int32_t block_size;      // tokens per cache block: 16, 32 or 64
  float scale_log2;
  float out_scale;         // multiplies the output (v_scale over a dequantised FP8 cache)
  int32_t* err_word;
  // Shared-prefix pass (the same kernel, prefix_len > 0): every sequence's
  // query group against tokens 0 .. prefix_len - 1, held in the blocks of
  // table row 0; the result goes to the decode workspace as parts
  // 0 .. prefix_splits - 1 of every (sequence, kv head) unit.
  int32_t prefix_len;
  int32_t prefix_splits;
  DecodeWorkspace ws;
};
// A prefill launch plans at most this many (sequence, 128-row tile) pairs;
// larger calls are split into launches over sequence ranges, and a single
// sequence of more than kPrefillMaxPairs * 128 new tokens is unsupported.
constexpr int kPrefillMaxPairs = 384;
cudaError_t launch_varlen_prefill(const PrefillArgs& a, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, int num_sms, cudaStream_t stream);

// FP8 cache -> bf16 scratch cache for the sequences with two or more new
// queries (the prefill rows): the e4m3 code values (exact in bf16), block
// (b, j) of the k-th such sequence at scratch block k * blocks_per_seq + j,
// and a scratch block table [num_seqs][blocks_per_seq] (-1 where unused).
struct Fp8GatherArgs {
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  int32_t num_blocks;
  const int32_t* block_tables;
  int32_t max_blocks_per_seq;
  const int32_t* context_lens;
  const int32_t* cu_seqlens_q;
  int32_t num_seqs;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t blocks_per_seq;   // scratch table row length, ceil(max_context_len / block_size)
  int32_t capacity;         // prefill sequences the scratch holds
  __nv_bfloat16* k_out;
  __nv_bfloat16* v_out;
  int32_t* table_out;
  int32_t* err_word;
};
cudaError_t launch_fp8_gather(const Fp8GatherArgs& a, cudaStream_t stream);
// The shared prefix (blocks_per_seq = prefix blocks of table row 0) to
// scratch blocks 0 .., a scratch table of num_seqs identical rows, and the
// check that every table starts with row 0's blocks (QATTN_DEVERR_PREFIX).
cudaError_t launch_fp8_prefix_gather(const Fp8GatherArgs& a, cudaStream_t stream);
// The shared-prefix pass; qmap: the query rows as [rows][heads][128] with a
// box of 64 dims x G heads x (128 / G) rows.
constexpr int kMaxPrefixSplits = 32;
cudaError_t launch_shared_prefix(const PrefillArgs& a, const CUtensorMap& qmap,
                                 const CUtensorMap& kmap, const CUtensorMap& vmap, int num_sms,
                                 cudaStream_t stream);

}  // namespace qattn
