// Dequantising gather for prefill over an FP8 (e4m3) cache.
//
// The cache holds e4m3 codes with one scale per tensor ("Qwen2大模型架构解析
// 与vLLM优化实践" sections 4.1, 4.2, 6.3: kv_cache_dtype "fp8", the cache
// scale, fp8_e4m3fn).  Every e4m3 value is a bf16 number (3 mantissa bits,
// exponents 2^-9 .. 2^8), so the prefill rows can run the bf16 tensor-core
// prefill unchanged on a bf16 copy of the code values, with k_scale folded
// into the logit scale and v_scale into the output.  This kernel writes that
// copy for the sequences with two or more new queries: the k-th such
// sequence's block j goes to scratch block k * blocks_per_seq + j, and a
// scratch block table points there.  Prefill is compute-bound; this pass
// reads the prefill sequences' codes once and writes twice the bytes.
#include "common.cuh"
#include "internal.h"

namespace qattn {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerCta = 2;

// 16 e4m3 codes -> 16 bf16 values (exact: e4m3 -> f16 -> f32 -> bf16).
__device__ __forceinline__ void codes16_to_bf16(const uint4& c, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  uint32_t r[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t f = cvt_f16x2_from_e4m3x2(w[i] >> (16 * h));
      const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&f));
      const __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
      r[2 * i + h] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  lo = make_uint4(r[0], r[1], r[2], r[3]);
  hi = make_uint4(r[4], r[5], r[6], r[7]);
}

// grid (num_seqs, ceil(blocks_per_seq / kBlocksPerCta)): CTA (b, y) copies
// blocks y * kBlocksPerCta ... of sequence b; CTA (b, 0) writes b's table row.
__global__ void __launch_bounds__(kThreads) fp8_gather_kernel(const Fp8GatherArgs a) {
  __shared__ int s_count[kThreads / 32];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int q0 = a.cu_seqlens_q[b];
  const int ql = a.cu_seqlens_q[b + 1] - q0;
  if (ql < 2) return;  // decode rows read the codes directly
  // rank of b among the prefill sequences
  int cnt = 0;
  for (int i = tid; i < b; i += kThreads) cnt += (a.cu_seqlens_q[i + 1] - a.cu_seqlens_q[i]) >= 2;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((tid & 31) == 0) s_count[tid >> 5] = cnt;
  __syncthreads();
  int rank = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) rank += s_count[w];
  const int BS = a.block_size, bps = a.blocks_per_seq;
  const int L = a.context_lens[b];
  const int nb = L > 0 ? min((L + BS - 1) / BS, min(bps, a.max_blocks_per_seq)) : 0;
  const int* row = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
  const bool fits = rank < a.capacity;
  if (blockIdx.y == 0) {
    if (!fits && tid == 0) set_err(a.err_word, QATTN_DEVERR_CONTEXT);
    for (int j = tid; j < bps; j += kThreads) {
      int v = -1;
      if (fits && j < nb) {
        const int id = row[j];
        v = (id >= 0 && id < a.num_blocks) ? rank * bps + j : -1;  // -1: flagged by the prefill
      }
      a.table_out[static_cast<int64_t>(b) * bps + j] = v;
    }
  }
  if (!fits) return;
  const int j0 = blockIdx.y * kBlocksPerCta;
  const int j1 = min(nb, j0 + kBlocksPerCta);
  const int chunks = a.num_kv_heads * BS * (kHeadDim / 16);  // 16-code chunks per block
  for (int j = j0; j < j1; ++j) {
    const int id = row[j];
    if (id < 0 || id >= a.num_blocks) continue;
    const int64_t src = static_cast<int64_t>(id) * chunks;
    const int64_t dst = (static_cast<int64_t>(rank) * bps + j) * chunks;
    for (int c = tid; c < chunks; c += kThreads) {
      uint4 lo, hi;
      codes16_to_bf16(reinterpret_cast<const uint4*>(a.k_codes)[src + c], lo, hi);
      reinterpret_cast<uint4*>(a.k_out)[2 * (dst + c)] = lo;
      reinterpret_cast<uint4*>(a.k_out)[2 * (dst + c) + 1] = hi;
      codes16_to_bf16(reinterpret_cast<const uint4*>(a.v_codes)[src + c], lo, hi);
      reinterpret_cast<uint4*>(a.v_out)[2 * (dst + c)] = lo;
      reinterpret_cast<uint4*>(a.v_out)[2 * (dst + c) + 1] = hi;
    }
  }
}

// The shared prefix of a batch (blocks 0 .. blocks_per_seq - 1 of table row
// 0) to scratch blocks 0 .., every row of the scratch table pointing at them
// (the prefix pass reads row 0 and compares the others with it); the real
// check -- every sequence's table starts with row 0's prefix blocks -- is
// made here on the caller's tables.  grid.x: copy CTAs of kBlocksPerCta
// blocks; every CTA also takes a share of the (row, block) table entries.
__global__ void __launch_bounds__(kThreads) fp8_prefix_gather_kernel(const Fp8GatherArgs a) {
  const int pb = a.blocks_per_seq;
  const int tid = threadIdx.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + tid;
       i < static_cast<int64_t>(a.num_seqs) * pb; i += static_cast<int64_t>(gridDim.x) * kThreads) {
    const int b = static_cast<int>(i / pb), j = static_cast<int>(i % pb);
    const int id0 = a.block_tables[j];
    const bool ok0 = id0 >= 0 && id0 < a.num_blocks;
    if (b > 0 && a.block_tables[static_cast<int64_t>(b) * a.max_blocks_per_seq + j] != id0)
      set_err(a.err_word, QATTN_DEVERR_PREFIX);
    a.table_out[i] = ok0 ? j : -1;  // -1: flagged by the prefix pass
  }
  const int j0 = blockIdx.x * kBlocksPerCta;
  const int j1 = min(pb, j0 + kBlocksPerCta);
  const int chunks = a.num_kv_heads * a.block_size * (kHeadDim / 16);
  for (int j = j0; j < j1; ++j) {
    const int id = a.block_tables[j];
    if (id < 0 || id >= a.num_blocks) continue;
    const int64_t src = static_cast<int64_t>(id) * chunks;
    const int64_t dst = static_cast<int64_t>(j) * chunks;
    for (int c = tid; c < chunks; c += kThreads) {
      uint4 lo, hi;
      codes16_to_bf16(reinterpret_cast<const uint4*>(a.k_codes)[src + c], lo, hi);
      reinterpret_cast<uint4*>(a.k_out)[2 * (dst + c)] = lo;
      reinterpret_cast<uint4*>(a.k_out)[2 * (dst + c) + 1] = hi;
      codes16_to_bf16(reinterpret_cast<const uint4*>(a.v_codes)[src + c], lo, hi);
      reinterpret_cast<uint4*>(a.v_out)[2 * (dst + c)] = lo;
      reinterpret_cast<uint4*>(a.v_out)[2 * (dst + c) + 1] = hi;
    }
  }
}

}  // namespace

cudaError_t launch_fp8_prefix_gather(const Fp8GatherArgs& a, cudaStream_t stream) {
  if (a.num_seqs <= 0 || a.blocks_per_seq <= 0) return cudaSuccess;
  const int grid = (a.blocks_per_seq + kBlocksPerCta - 1) / kBlocksPerCta;
  const cudaError_t e =
      set_max_dynamic_smem(reinterpret_cast<const void*>(fp8_prefix_gather_kernel), 0);
  if (e != cudaSuccess) return e;
  fp8_prefix_gather_kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaPeekAtLastError();
}

cudaError_t launch_fp8_gather(const Fp8GatherArgs& a, cudaStream_t stream) {
  if (a.num_seqs <= 0 || a.blocks_per_seq <= 0) return cudaSuccess;
  const dim3 grid(a.num_seqs, (a.blocks_per_seq + kBlocksPerCta - 1) / kBlocksPerCta);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  const cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(fp8_gather_kernel), 0);
  if (e != cudaSuccess) return e;
  fp8_gather_kernel<<<grid, kThreads, 0, stream>>>(a);
  return cudaPeekAtLastError();
}

}  // namespace qattn
