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

namespace qattn {
namespace {

// K2r: merge the parts of units that straddled CTAs.  One CTA of four
// warps per (sequence, kv head, query head of the group); lane = 4
// dimensions.
//   out[row, g*G + h] = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M).
// A unit of up to kMergeBatch parts is folded by warp 0 alone, its parts
// loaded together with the part count (their addresses do not depend on
// it): one memory round trip.  Longer part lists (a long sequence spread
// over many CTAs) are cut into four consecutive ranges,
// one per warp, each folded in part order, kMergeBatch loads in flight; the
// four partial states are then combined in warp order through shared
// memory.  The order is fixed, so results are deterministic.
constexpr int kMergeBatch = 8;
constexpr int kMergeWarps = 4;

struct FoldState {
  float m, den;
  float4 num;
};

__device__ __forceinline__ void fold_one(FoldState& st, float lse, const float4& o) {
  const float mn = fmaxf(st.m, lse);
  const float sc = exp2f(st.m - mn);  // 0 for the first part
  const float f = exp2f(lse - mn);
  st.den = fmaf(st.den, sc, f);
  st.num.x = fmaf(st.num.x, sc, f * o.x);
  st.num.y = fmaf(st.num.y, sc, f * o.y);
  st.num.z = fmaf(st.num.z, sc, f * o.z);
  st.num.w = fmaf(st.num.w, sc, f * o.w);
  st.m = mn;
}

template <int G>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const DecodeArgs a) {
  __shared__ float s_m[kMergeWarps], s_den[kMergeWarps];
  __shared__ float4 s_num[kMergeWarps][32];
  grid_dep_wait();  // the parts come from the decode grid
  const int Hkv = a.num_kv_heads;
  const int64_t wid = blockIdx.x;
  const int h = static_cast<int>(wid % G);
  const int64_t seg = wid / G;
  const int b = static_cast<int>(seg / Hkv), g = static_cast<int>(seg % Hkv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t pbase = seg * a.ws.max_parts * G + h;  // part p at pbase + p * G
  const float* lse = a.ws.lse + pbase;
  const float* po = a.ws.part_o + pbase * kHeadDim + lane * 4;
  auto load = [&](int p, float& l, float4& o) {
    l = lse[static_cast<int64_t>(p) * G];
    o = *reinterpret_cast<const float4*>(po + static_cast<int64_t>(p) * G * kHeadDim);
  };
  float lv[kMergeBatch];
  float4 ov[kMergeBatch];
  if (warp == 0) {
#pragma unroll
    for (int j = 0; j < kMergeBatch; ++j)
      if (j < a.ws.max_parts) load(j, lv[j], ov[j]);  // inside this unit's part slots
  }
  // The count comes from the decode kernel; a unit whose first piece was
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
  if (ql != 1 || nparts <= 1) return;  // not a decode row, or written by the decode kernel
  const bool split = nparts > kMergeBatch;
  const int per = split ? (nparts + kMergeWarps - 1) / kMergeWarps : nparts;
  const int p_begin = warp * per;
  const int p_end = min(nparts, p_begin + per);
  FoldState st{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  if (warp == 0 || split) {
    for (int p0 = p_begin; p0 < p_end; p0 += kMergeBatch) {
      if (!(warp == 0 && p0 == 0)) {  // warp 0's first batch is already loaded
#pragma unroll
        for (int j = 0; j < kMergeBatch; ++j)
          if (p0 + j < p_end) load(p0 + j, lv[j], ov[j]);
      }
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j)
        if (p0 + j < p_end) fold_one(st, lv[j], ov[j]);
    }
  }
  if (split) {
    if (lane == 0) {
      s_m[warp] = st.m;
      s_den[warp] = st.den;
    }
    s_num[warp][lane] = st.num;
    __syncthreads();
    if (warp != 0) return;
    // warp 0 holds range 0; fold ranges 1..3 in order, each as a part of
    // log2-weight m + log2(den) and value num / den
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) {
      const float m = s_m[w], den = s_den[w];
      if (den > 0.f) {
        const float4 n = s_num[w][lane];
        const float mn = fmaxf(st.m, m);
        const float sa = exp2f(st.m - mn), sb = exp2f(m - mn);
        st.den = st.den * sa + den * sb;
        st.num.x = st.num.x * sa + n.x * sb;
        st.num.y = st.num.y * sa + n.y * sb;
        st.num.z = st.num.z * sa + n.z * sb;
        st.num.w = st.num.w * sa + n.w * sb;
        st.m = mn;
      }
    }
  } else if (warp != 0) {
    return;
  }
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                        (row * a.num_heads + static_cast<int64_t>(g) * G + h) * kHeadDim + lane * 4;
  const float inv = 1.f / st.den;
  uint2 packed;
  packed.x = pack_bf16x2_rn(st.num.x * inv, st.num.y * inv);
  packed.y = pack_bf16x2_rn(st.num.z * inv, st.num.w * inv);
  *reinterpret_cast<uint2*>(orow) = packed;
}

template <int G>
cudaError_t launch_merge_g(const DecodeArgs& a, cudaStream_t stream) {
  const int64_t ctas = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads * G;
  cudaError_t e = launch_pdl(decode_merge_kernel<G>, dim3(static_cast<unsigned>(ctas)),
                             dim3(kMergeWarps * 32), 0, stream, a);
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

}  // namespace qattn
