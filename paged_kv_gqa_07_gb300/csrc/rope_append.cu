// Kernel K1: rotate-half RoPE on the query and key heads of each new token,
// and the write of its key/value rows into the paged cache.
//
// Follows get_rope(head_dim, rotary_dim=head_dim, max_position, base) in
// "Qwen2大模型架构解析与vLLM优化实践" section 2.2 (full-width rotate-half,
// rope_theta = 1e6 per "Qwen2 模型结构代码详解" section 2), and the block
// cache written through a slot mapping (vLLM-deploys-Qwen notes section 2.1;
// nano-vllm Qwen3 skeleton page section 5).
//
// Work decomposition: one thread per (token, head, 8-pair slice).  A query
// or key head of 128 dims is 64 rotation pairs (i, i + 64); eight threads
// cover it, each loading two 16-byte vectors (dims i..i+7 and i+64..i+71)
// and the matching 32-byte cos and sin slices of the table row.  A value
// head is a plain 256-byte copy done by sixteen threads with 16-byte
// vectors.  All global accesses of a warp are contiguous 128-byte runs.
//
// The rotation is evaluated with explicitly rounded fp32 operations
// (__fmul_rn / __fsub_rn / __fadd_rn, no contraction into FMA) and rounded
// to bf16 nearest-even, so the cache contents are bit-reproducible.
//
// Optional steps before RoPE (the Qwen2 qkv projection's bias=True,
// "Qwen2大模型架构解析与vLLM优化实践"; the Qwen3 attention's q_norm / k_norm
// RMSNorms, nano-vllm Qwen3 skeleton page, module tree), each a bf16 tensor
// operation: x' = bf16(x + b) rounded once; RMSNorm over the head's 128
// values around the exact sum of their squares (integer arithmetic, see
// rmsnorm_group), v = fp32(mean + eps), r = 1 / sqrt(v) with correctly
// rounded fp32 sqrt and division, y = bf16(fp32(fp32(x * r) * w)).
//
// FP8 cache (kv_cache_dtype "fp8", fp8_e4m3fn with a cache scale per tensor,
// "Qwen2大模型架构解析与vLLM优化实践" sections 4.1, 4.2, 6.3): the bf16 key
// and value rows above are stored as e4m3(x / scale) -- fp32 division
// rounded to nearest, then the hardware conversion to e4m3 with
// round-to-nearest-even and saturation to +-448.
#include "common.cuh"
#include "internal.h"

namespace qattn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void rotate8(const uint4& x1, const uint4& x2, const float* c,
                                        const float* s, uint4& y1, uint4& y2) {
  const uint32_t* a = reinterpret_cast<const uint32_t*>(&x1);
  const uint32_t* b = reinterpret_cast<const uint32_t*>(&x2);
  uint32_t* o1 = reinterpret_cast<uint32_t*>(&y1);
  uint32_t* o2 = reinterpret_cast<uint32_t*>(&y2);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    float lo1[2] = {bf16lo_to_f32(a[w]), bf16hi_to_f32(a[w])};
    float hi1[2] = {bf16lo_to_f32(b[w]), bf16hi_to_f32(b[w])};
    float r1[2], r2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float cc = c[2 * w + e], ss = s[2 * w + e];
      r1[e] = __fsub_rn(__fmul_rn(lo1[e], cc), __fmul_rn(hi1[e], ss));
      r2[e] = __fadd_rn(__fmul_rn(hi1[e], cc), __fmul_rn(lo1[e], ss));
    }
    o1[w] = pack_bf16x2_rn(r1[0], r1[1]);
    o2[w] = pack_bf16x2_rn(r2[0], r2[1]);
  }
}

// 8 bf16 + 8 bf16 -> 8 bf16, each sum rounded once.
__device__ __forceinline__ uint4 add_bias8(const uint4& x, const __nv_bfloat16* b) {
  const uint4 bb = *reinterpret_cast<const uint4*>(b);
  const uint32_t* xs = reinterpret_cast<const uint32_t*>(&x);
  const uint32_t* bs = reinterpret_cast<const uint32_t*>(&bb);
  uint4 y;
  uint32_t* ys = reinterpret_cast<uint32_t*>(&y);
#pragma unroll
  for (int w = 0; w < 4; ++w)
    ys[w] = pack_bf16x2_rn(__fadd_rn(bf16lo_to_f32(xs[w]), bf16lo_to_f32(bs[w])),
                           __fadd_rn(bf16hi_to_f32(xs[w]), bf16hi_to_f32(bs[w])));
  return y;
}

// Exponent key of a bf16 value for the exact sum of squares: a value is
// sig * 2^(e - 134) with an 8-bit significand sig and e = max(exponent
// field, 1) (subnormals share e = 1, sig without the implicit bit).
__device__ __forceinline__ int bf16_sq_exp(uint32_t bits) {
  const int ef = static_cast<int>((bits >> 7) & 0xffu);
  return (bits & 0x7fffu) != 0u ? max(ef, 1) : 0;
}

// sig^2 * 2^(2 (e - emax) + 41): an integer for e >= emax - 20; smaller
// squares (below 2^-40 of the largest) are truncated.  At most 2^57 each,
// so the 128 terms of a head fit in 64 bits.
__device__ __forceinline__ uint64_t bf16_sq_term(uint32_t bits, int emax) {
  const uint32_t ef = (bits >> 7) & 0xffu;
  const uint32_t sig = (bits & 0x7fu) | (ef != 0u ? 0x80u : 0u);
  const uint64_t sq = static_cast<uint64_t>(sig * sig);
  const int sh = 2 * (max(static_cast<int>(ef), 1) - emax) + 41;
  if (sh >= 0) return sq << sh;
  return sh > -64 ? sq >> (-sh) : 0ull;
}

// RMSNorm of one head whose 128 values are spread over the 8 lanes of an
// aligned lane group (x1: dims 8p .. 8p+7, x2: dims 64+8p .. 64+8p+7 of
// lane p of the group).  The mean square is formed from the exact sum of
// the squares: each square as a 64-bit integer multiple of a power of two
// fixed by the head's largest exponent, summed in integers (exact, so the
// order of the lanes does not matter), then scaled to fp64 -- the value an
// fp64 sum of the squares gives whenever that sum is exact.  Then
// v = fp32(ss / 128 + eps), r = 1 / sqrt(v) with correctly rounded fp32
// sqrt and division, y = bf16(fp32(fp32(x * r) * w)).
__device__ __forceinline__ void rmsnorm_group(uint4& x1, uint4& x2, const __nv_bfloat16* w,
                                              int part, float eps) {
  const uint32_t mask = 0xffu << ((threadIdx.x & 31) & 24);
  uint32_t* u1 = reinterpret_cast<uint32_t*>(&x1);
  uint32_t* u2 = reinterpret_cast<uint32_t*>(&x2);
  uint32_t h[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    h[2 * i] = u1[i] & 0xffffu;
    h[2 * i + 1] = u1[i] >> 16;
    h[8 + 2 * i] = u2[i] & 0xffffu;
    h[8 + 2 * i + 1] = u2[i] >> 16;
  }
  int emax = 0;
  bool nan = false, inf = false;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    emax = max(emax, bf16_sq_exp(h[i]));
    const bool special = (h[i] & 0x7f80u) == 0x7f80u;
    nan = nan || (special && (h[i] & 0x7fu) != 0u);
    inf = inf || (special && (h[i] & 0x7fu) == 0u);
  }
  emax = max(emax, __shfl_xor_sync(mask, emax, 1));
  emax = max(emax, __shfl_xor_sync(mask, emax, 2));
  emax = max(emax, __shfl_xor_sync(mask, emax, 4));
  nan = __any_sync(mask, nan);
  inf = __any_sync(mask, inf);
  uint64_t acc = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) acc += bf16_sq_term(h[i], emax);
  acc += __shfl_xor_sync(mask, acc, 1);
  acc += __shfl_xor_sync(mask, acc, 2);
  acc += __shfl_xor_sync(mask, acc, 4);
  double ss;
  if (nan) {
    ss = __longlong_as_double(0x7ff8000000000000ll);
  } else if (inf) {
    ss = __longlong_as_double(0x7ff0000000000000ll);
  } else {
    // x^2 = term * 2^(2 emax - 309); emax in 1..254 keeps the scale normal
    const int k = emax > 0 ? 2 * emax - 309 : 0;
    ss = __dmul_rn(__ull2double_rn(acc),
                   __longlong_as_double(static_cast<long long>(k + 1023) << 52));
  }
  const float v = __double2float_rn(__dadd_rn(__dmul_rn(ss, 1.0 / 128.0),
                                              static_cast<double>(eps)));
  const float r = __fdiv_rn(1.0f, __fsqrt_rn(v));
  const uint4 w1 = *reinterpret_cast<const uint4*>(w + part * 8);
  const uint4 w2 = *reinterpret_cast<const uint4*>(w + 64 + part * 8);
  const uint32_t* ws1 = reinterpret_cast<const uint32_t*>(&w1);
  const uint32_t* ws2 = reinterpret_cast<const uint32_t*>(&w2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    u1[i] = pack_bf16x2_rn(__fmul_rn(__fmul_rn(bf16lo_to_f32(u1[i]), r), bf16lo_to_f32(ws1[i])),
                           __fmul_rn(__fmul_rn(bf16hi_to_f32(u1[i]), r), bf16hi_to_f32(ws1[i])));
    u2[i] = pack_bf16x2_rn(__fmul_rn(__fmul_rn(bf16lo_to_f32(u2[i]), r), bf16lo_to_f32(ws2[i])),
                           __fmul_rn(__fmul_rn(bf16hi_to_f32(u2[i]), r), bf16hi_to_f32(ws2[i])));
  }
}

// 8 bf16 values -> 8 e4m3 codes of x / s (byte i = value i).
__device__ __forceinline__ uint2 quantize8_e4m3(const uint4& x, float s) {
  const uint32_t* xs = reinterpret_cast<const uint32_t*>(&x);
  uint32_t pr[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float lo = __fdiv_rn(bf16lo_to_f32(xs[w]), s);
    const float hi = __fdiv_rn(bf16hi_to_f32(xs[w]), s);
    pr[w] = cvt_e4m3x2(lo, hi);
  }
  return make_uint2(pr[0] | (pr[1] << 16), pr[2] | (pr[3] << 16));
}

// kExtras: bias and/or norms present (the plain step compiles without them);
// kFp8: the caches hold e4m3 codes.
template <bool kExtras, bool kFp8>
__global__ void __launch_bounds__(kThreads) rope_append_kernel(RopeAppendArgs a,
                                                               int tasks_per_token) {
  // A following decode kernel may start its set-up now; it reads nothing
  // this kernel writes before its own grid_dep_wait().
  grid_dep_launch();
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t t = gid / tasks_per_token;
  if (t >= a.num_tokens) return;
  const int r = static_cast<int>(gid - t * tasks_per_token);
  const int H = a.num_heads, Hkv = a.num_kv_heads;
  const int nrot = (H + Hkv) * 8;

  const int pos = a.positions[t];
  if (pos < 0 || pos >= a.max_pos) {
    if (r == 0) set_err(a.err_word, QATTN_DEVERR_POSITION);
    return;
  }
  const int slot = a.slot_mapping[t];
  const int BS = a.block_size;
  const int64_t num_slots = static_cast<int64_t>(a.num_blocks) * BS;
  bool write_cache = slot >= 0;
  if (write_cache && slot >= num_slots) {
    if (r == 0) set_err(a.err_word, QATTN_DEVERR_SLOT);
    write_cache = false;
  }
  int64_t cache_row = 0;  // element offset of (block, kv head 0, offset) in the cache
  if (write_cache) {
    const int blk = slot / BS, off = slot % BS;
    cache_row = (static_cast<int64_t>(blk) * Hkv * BS + off) * kHeadDim;
  }

  if (r < nrot) {
    const int head = r >> 3;
    const int part = r & 7;
    const float* row = a.cos_sin + static_cast<int64_t>(pos) * kHeadDim;
    float c[8], s[8];
    {
      const float4 c0 = __ldg(reinterpret_cast<const float4*>(row + part * 8));
      const float4 c1 = __ldg(reinterpret_cast<const float4*>(row + part * 8 + 4));
      const float4 s0 = __ldg(reinterpret_cast<const float4*>(row + 64 + part * 8));
      const float4 s1 = __ldg(reinterpret_cast<const float4*>(row + 64 + part * 8 + 4));
      c[0] = c0.x; c[1] = c0.y; c[2] = c0.z; c[3] = c0.w;
      c[4] = c1.x; c[5] = c1.y; c[6] = c1.z; c[7] = c1.w;
      s[0] = s0.x; s[1] = s0.y; s[2] = s0.z; s[3] = s0.w;
      s[4] = s1.x; s[5] = s1.y; s[6] = s1.z; s[7] = s1.w;
    }
    // bias and norm first (head = q head h, or H + kv head g: also the
    // head's row in the bias)
    const __nv_bfloat16* bias =
        kExtras && a.bias
            ? static_cast<const __nv_bfloat16*>(a.bias) + static_cast<int64_t>(head) * kHeadDim
            : nullptr;
    if (head < H) {
      __nv_bfloat16* src = static_cast<__nv_bfloat16*>(a.q) + t * a.q_row_stride +
                           static_cast<int64_t>(head) * kHeadDim;
      uint4* p1 = reinterpret_cast<uint4*>(src + part * 8);
      uint4* p2 = reinterpret_cast<uint4*>(src + 64 + part * 8);
      uint4 x1 = *p1, x2 = *p2;
      if (bias) {
        x1 = add_bias8(x1, bias + part * 8);
        x2 = add_bias8(x2, bias + 64 + part * 8);
      }
      if (kExtras && a.q_norm_w)
        rmsnorm_group(x1, x2, static_cast<const __nv_bfloat16*>(a.q_norm_w), part, a.norm_eps);
      uint4 y1, y2;
      rotate8(x1, x2, c, s, y1, y2);
      *p1 = y1;
      *p2 = y2;
    } else {
      if (!write_cache) return;  // the whole lane group: same token
      const int g = head - H;
      const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.k) + t * a.k_row_stride +
                                 static_cast<int64_t>(g) * kHeadDim;
      uint4 x1 = *reinterpret_cast<const uint4*>(src + part * 8);
      uint4 x2 = *reinterpret_cast<const uint4*>(src + 64 + part * 8);
      if (bias) {
        x1 = add_bias8(x1, bias + part * 8);
        x2 = add_bias8(x2, bias + 64 + part * 8);
      }
      if (kExtras && a.k_norm_w)
        rmsnorm_group(x1, x2, static_cast<const __nv_bfloat16*>(a.k_norm_w), part, a.norm_eps);
      uint4 y1, y2;
      rotate8(x1, x2, c, s, y1, y2);
      const int64_t dst = cache_row + static_cast<int64_t>(g) * BS * kHeadDim;
      if (kFp8) {
        uint8_t* d8 = static_cast<uint8_t*>(a.k_cache) + dst;
        *reinterpret_cast<uint2*>(d8 + part * 8) = quantize8_e4m3(y1, a.k_scale);
        *reinterpret_cast<uint2*>(d8 + 64 + part * 8) = quantize8_e4m3(y2, a.k_scale);
      } else {
        __nv_bfloat16* d16 = static_cast<__nv_bfloat16*>(a.k_cache) + dst;
        *reinterpret_cast<uint4*>(d16 + part * 8) = y1;
        *reinterpret_cast<uint4*>(d16 + 64 + part * 8) = y2;
      }
    }
  } else {
    if (!write_cache) return;
    const int r2 = r - nrot;
    const int g = r2 >> 4, part = r2 & 15;
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(a.v) + t * a.v_row_stride +
                               static_cast<int64_t>(g) * kHeadDim;
    const int64_t dst = cache_row + static_cast<int64_t>(g) * BS * kHeadDim + part * 8;
    uint4 x = *reinterpret_cast<const uint4*>(src + part * 8);
    if (kExtras && a.bias)
      x = add_bias8(x, static_cast<const __nv_bfloat16*>(a.bias) +
                           static_cast<int64_t>(H + Hkv + g) * kHeadDim + part * 8);
    if (kFp8)
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.v_cache) + dst) =
          quantize8_e4m3(x, a.v_scale);
    else
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.v_cache) + dst) = x;
  }
}

}  // namespace

cudaError_t launch_rope_append(const RopeAppendArgs& a, cudaStream_t stream) {
  const int tasks_per_token = (a.num_heads + a.num_kv_heads) * 8 + a.num_kv_heads * 16;
  const int64_t total = static_cast<int64_t>(a.num_tokens) * tasks_per_token;
  const int64_t blocks = (total + kThreads - 1) / kThreads;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  const bool extras = a.bias != nullptr || a.q_norm_w != nullptr || a.k_norm_w != nullptr;
  const dim3 grid(static_cast<unsigned>(blocks));
  const void* fn =
      a.kv_fp8 ? (extras ? reinterpret_cast<const void*>(rope_append_kernel<true, true>)
                         : reinterpret_cast<const void*>(rope_append_kernel<false, true>))
               : (extras ? reinterpret_cast<const void*>(rope_append_kernel<true, false>)
                         : reinterpret_cast<const void*>(rope_append_kernel<false, false>));
  const cudaError_t e = set_max_dynamic_smem(fn, 0);
  if (e != cudaSuccess) return e;
  if (a.kv_fp8) {
    if (extras)
      rope_append_kernel<true, true><<<grid, kThreads, 0, stream>>>(a, tasks_per_token);
    else
      rope_append_kernel<false, true><<<grid, kThreads, 0, stream>>>(a, tasks_per_token);
  } else {
    if (extras)
      rope_append_kernel<true, false><<<grid, kThreads, 0, stream>>>(a, tasks_per_token);
    else
      rope_append_kernel<false, false><<<grid, kThreads, 0, stream>>>(a, tasks_per_token);
  }
  return cudaPeekAtLastError();
}

}  // namespace qattn
