// Kernel K2r and the decode workspace: the merge of split-KV parts.
//
// A (sequence, kv head) unit of the decode work list whose tiles are spread
// over several CTAs leaves one partial result per CTA: the output of its
// share of the keys normalised by its own softmax sum, and the log2 of that
// sum plus its running maximum.  This is the split-KV partition the decode
// kernel uses for long contexts (max_position_embeddings 32768,
// "Qwen2 模型结构代码详解" section 2); combining the parts with the
// log-sum-exp weights gives the unsplit softmax exactly up to rounding.
#include <math.h>

#include "common.cuh"
#include "internal.h"

#ifdef QATTN_TRACE
// Tracing build only: %globaltimer stamps of the merge CTAs (entry, the
// decode grid's completion seen, done).
__device__ unsigned long long g_qattn_merge_trace[qattn::kTraceMergeCtas * 4];
#define QATTN_MSTAMP(slot)                                                                  \
  do {                                                                                      \
    if (blockIdx.x < qattn::kTraceMergeCtas)                                                \
      g_qattn_merge_trace[blockIdx.x * 4 + (slot)] = qattn::globaltimer_ns();               \
  } while (0)
#else
#define QATTN_MSTAMP(slot) \
  do {                     \
  } while (0)
#endif

namespace qattn {
namespace {

// K2r: merge the parts of units that straddled CTAs.  One CTA per
// (sequence, kv head) unit, one warp per query head of its group, lane = 4
// dimensions:
//   out[row, g*G + h] = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M),
// folded in part order with a running maximum M (deterministic).  The first
// two parts are loaded with the part count, the rest kMergeBatch at a time.  The CTAs are small enough to become resident beside
// the decode kernel's (the launch is a programmatic dependent one) and wait
// there for its grid to finish.
constexpr int kMergeBatch = 8;

__device__ __forceinline__ void fold_one(float& m, float& den, float4& num, float lse,
                                         const float4& o) {
  const float mn = fmaxf(m, lse);
  const float sc = exp2f(m - mn);  // 0 for the first part
  const float f = exp2f(lse - mn);
  den = fmaf(den, sc, f);
  num.x = fmaf(num.x, sc, f * o.x);
  num.y = fmaf(num.y, sc, f * o.y);
  num.z = fmaf(num.z, sc, f * o.z);
  num.w = fmaf(num.w, sc, f * o.w);
  m = mn;
}

template <int G>
__global__ void __launch_bounds__(G * 32) decode_merge_kernel(const DecodeArgs a) {
  if (threadIdx.x == 0) QATTN_MSTAMP(0);
  grid_dep_wait();  // the parts come from the decode grid
  if (threadIdx.x == 0) QATTN_MSTAMP(1);
  const int Hkv = a.num_kv_heads;
  const int64_t seg = blockIdx.x;
  const int b = static_cast<int>(seg / Hkv), g = static_cast<int>(seg % Hkv);
  const int h = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t pbase = seg * a.ws.max_parts * G + h;  // part p at pbase + p * G
  const float* lse = a.ws.lse + pbase;
  const float* po = a.ws.part_o + pbase * kHeadDim + lane * 4;
  auto load = [&](int p, float& l, float4& o) {
    l = lse[static_cast<int64_t>(p) * G];
    o = *reinterpret_cast<const float4*>(po + static_cast<int64_t>(p) * G * kHeadDim);
  };
  float lv[kMergeBatch];
  float4 ov[kMergeBatch];
  // The first two parts (most units have at most two) are loaded with the
  // count; their slots exist whatever the count (max_parts >= 2).
  load(0, lv[0], ov[0]);
  load(1, lv[1], ov[1]);
  // The count comes from the decode kernel; a unit whose first part was
  // never finished (a CTA that gave up after a timeout) leaves whatever the
  // workspace held, so it is clamped to the unit's part slots: the output
  // of such a call is unspecified, but nothing is read out of bounds.
  const int nparts = min(a.ws.nparts[seg], a.ws.max_parts);
  int64_t row = b;
  int ql = 1;
  if (a.cu_seqlens_q != nullptr) {
    row = a.cu_seqlens_q[b];
    ql = a.cu_seqlens_q[b + 1] - static_cast<int>(row);
  }
  if (ql != 1 || nparts <= 1) {  // not a decode row, or written by the decode kernel
    if (threadIdx.x == 0) QATTN_MSTAMP(2);
    return;
  }
  float m = -INFINITY, den = 0.f;
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  // parts 2 .. kMergeBatch - 1 of the first batch, then whole batches
#pragma unroll
  for (int j = 2; j < kMergeBatch; ++j)
    if (j < nparts) load(j, lv[j], ov[j]);
  for (int p0 = 0;;) {
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)
      if (p0 + j < nparts) fold_one(m, den, num, lv[j], ov[j]);
    p0 += kMergeBatch;
    if (p0 >= nparts) break;
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)
      if (p0 + j < nparts) load(p0 + j, lv[j], ov[j]);
  }
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                        (row * a.num_heads + static_cast<int64_t>(g) * G + h) * kHeadDim + lane * 4;
  const float inv = 1.f / den;
  uint2 packed;
  packed.x = pack_bf16x2_rn(num.x * inv, num.y * inv);
  packed.y = pack_bf16x2_rn(num.z * inv, num.w * inv);
  *reinterpret_cast<uint2*>(orow) = packed;
  if (threadIdx.x == 0) QATTN_MSTAMP(2);
}

template <int G>
cudaError_t launch_merge_g(const DecodeArgs& a, cudaStream_t stream) {
  const int64_t units = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads;
  cudaError_t e = set_max_dynamic_smem(reinterpret_cast<const void*>(decode_merge_kernel<G>), 0);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_merge_kernel<G>, dim3(static_cast<unsigned>(units)),
                             dim3(G * 32), 0, stream, a);
  if (e != cudaSuccess) return e;
  return cudaPeekAtLastError();
}

}  // namespace

// Layout: nparts, lse, part_o; every section 256-byte aligned.
size_t decode_workspace_bytes(int32_t num_seqs, int32_t max_context_len, int32_t num_kv_heads,
                              int32_t group, int32_t extra_parts) {
  const int64_t max_parts = decode_max_parts(max_context_len) + extra_parts;
  auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t units = static_cast<int64_t>(num_seqs) * num_kv_heads * max_parts * group;
  return static_cast<size_t>(al(static_cast<int64_t>(num_seqs) * num_kv_heads * 4) +
                             al(units * 4) + al(units * kHeadDim * 4));
}

DecodeWorkspace carve_decode_workspace(void* base, int32_t num_seqs, int32_t max_context_len,
                                       int32_t num_kv_heads, int32_t group, int32_t extra_parts) {
  const int64_t max_parts = decode_max_parts(max_context_len) + extra_parts;
  auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t units = static_cast<int64_t>(num_seqs) * num_kv_heads * max_parts * group;
  uint8_t* p = static_cast<uint8_t*>(base);
  DecodeWorkspace w;
  w.nparts = reinterpret_cast<int32_t*>(p);
  p += al(static_cast<int64_t>(num_seqs) * num_kv_heads * 4);
  w.lse = reinterpret_cast<float*>(p);
  p += al(units * 4);
  w.part_o = reinterpret_cast<float*>(p);
  w.max_parts = static_cast<int32_t>(max_parts);
  return w;
}

cudaError_t launch_decode_merge(const DecodeArgs& a, cudaStream_t stream) {
  switch (a.num_heads / a.num_kv_heads) {
    case 1: return launch_merge_g<1>(a, stream);
    case 2: return launch_merge_g<2>(a, stream);
    case 3: return launch_merge_g<3>(a, stream);
    case 4: return launch_merge_g<4>(a, stream);
    case 5: return launch_merge_g<5>(a, stream);
    case 6: return launch_merge_g<6>(a, stream);
    case 7: return launch_merge_g<7>(a, stream);
    case 8: return launch_merge_g<8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

#ifdef QATTN_TRACE
cudaError_t read_merge_trace(unsigned long long* host, size_t n) {
  return cudaMemcpyFromSymbol(host, g_qattn_merge_trace, n * sizeof(unsigned long long));
}
cudaError_t clear_merge_trace() {
  static unsigned long long zero[kTraceMergeCtas * 4];
  return cudaMemcpyToSymbol(g_qattn_merge_trace, zero, sizeof(zero));
}
#endif

}  // namespace qattn
