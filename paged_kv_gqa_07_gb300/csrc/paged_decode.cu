// Kernels K2 (paged GQA decode on CUDA cores, the default for groups of one
// or two query heads per KV head) and K2r (merge of split units).
//
// What is computed: for every decode sequence b and query head h, with KV
// head g = h / G (G = num_heads / num_kv_heads),
//     out[b, h] = sum_j softmax_j(scale * q[b, h] . k_j) v_j,  j < L_b,
// keys and values gathered through the sequence's block table -- the
// grouped-query attention with scaling head_dim ** -0.5 of
// "Qwen2 模型结构代码详解" section 2 over the PagedAttention block cache of
// the vLLM-deploys-Qwen notes section 2.1.
//
// Design (GB300): the decode step is bound by HBM bandwidth on KV bytes, so
// the kernel is built to read every KV byte exactly once, at full rate.
//   * Work space: the (sequence, kv head) units, each cut into chunks of 32
//     tokens (two 16-token blocks).  All chunks of all units form one
//     ordered list; a persistent grid of one CTA per SM gives every CTA an
//     equal contiguous run of the list (at least 8 chunks), so long and short
//     sequences balance.  A unit that straddles CTAs leaves one partial
//     result per CTA (normalised output plus log2-sum-exp); K2r merges them
//     in part order, so results are deterministic.
//   * One producer warp streams the run through a ring of shared-memory
//     stages with one 4-D TMA per (block, kv head) tile of K or V (16 rows x
//     256 B, 128-byte swizzle) and copies each unit's G query heads.  Four
//     consumer warps take chunks round-robin.  Stage hand-off uses
//     mbarriers (full: TMA byte count, empty: consumer release).
//   * A consumer warp holds the whole GQA group: QK^T is lane-per-token (lane
//     j owns token j's 256-byte key row, read conflict-free thanks to the
//     swizzle, and broadcast-reads the fp32 query heads, pre-scaled by
//     scale * log2 e), so each key byte serves all G heads with no shuffle
//     reduction; the chunk max per head is one 5-step shuffle tree; PV is
//     lane-per-dimension (4 dims per lane) with p broadcast from shared
//     memory.  Each warp keeps its own online-softmax state (running max m,
//     lane-partial sums l, output o) and the warps are merged at the end of
//     every unit.
//   * Every wait is bounded (see common.cuh); on a timeout the kernel raises
//     QATTN_DEVERR_TIMEOUT, drains its copies in flight and returns.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace qattn {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kStages = 11;
constexpr int kBoxBytes = kBlockSize * 128;     // 16 rows x 128 B
constexpr int kTileBytes = 2 * kBoxBytes;       // one (block, kv head) tile of K or V
constexpr int kKBytes = 2 * kTileBytes;         // two blocks of K
constexpr int kStageBytes = 2 * kKBytes;        // K + V of one chunk
constexpr int kMaxGroup = 8;

// Shared-memory layout (offsets from a 1024-byte aligned base).
constexpr int kOffStages = 0;
constexpr int kOffQStage = kOffStages + kStages * kStageBytes;       // 2 x [8][128] bf16
constexpr int kOffQf = kOffQStage + 2 * kMaxGroup * kHeadDim * 2;    // [8][128] fp32
constexpr int kOffP = kOffQf + kMaxGroup * kHeadDim * 4;             // [warps][8][32] fp32
constexpr int kOffMo = kOffP + kConsumerWarps * kMaxGroup * 32 * 4;  // [warps][8][128] fp32
constexpr int kOffMl = kOffMo + kConsumerWarps * kMaxGroup * kHeadDim * 4;  // [warps][8][2]
constexpr int kOffBars = kOffMl + kConsumerWarps * kMaxGroup * 2 * 4;
constexpr int kNumBars = 2 * kStages + 4 + 1;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kOffLens = kOffMisc + 64;                               // [kMaxSmemSeqs] int32
constexpr int kMaxSmemSeqs = 4096;
constexpr int kSmemBytes = kOffLens + kMaxSmemSeqs * 4 + 1024;  // + alignment slack

struct Misc {
  int abort;
  int total;
  int b0;
  int off0;
  int warp_sums[kConsumerWarps + 1];
};

// Context length of decode sequence b if it is valid for this kernel, else 0.
__device__ __forceinline__ int seq_len_eff(const DecodeArgs& a, int b) {
  return decode_len_eff(a, b);
}

// Chunks of sequence b (and its effective length), served from the
// shared-memory copy when the batch fits in it.
__device__ __forceinline__ int seq_chunks_cached(const DecodeArgs& a, const int* s_len, int b,
                                                 int* L_out) {
  const int L = a.num_seqs <= kMaxSmemSeqs ? s_len[b] : seq_len_eff(a, b);
  *L_out = L;
  return (L + kChunkTokens - 1) / kChunkTokens;
}

// Position in the chunk list: sequence b, kv head g, chunk i of nch.
struct Walk {
  int b, g, i, nch, L;
};

__device__ __forceinline__ void walk_next(Walk& w, const DecodeArgs& a, const int* s_len) {
  if (++w.i < w.nch) return;
  w.i = 0;
  if (++w.g < a.num_kv_heads) return;
  w.g = 0;
  for (;;) {
    ++w.b;
    if (w.b >= a.num_seqs) {
      w.nch = 0;
      return;
    }
    w.nch = seq_chunks_cached(a, s_len, w.b, &w.L);
    if (w.nch > 0) return;
  }
}

__device__ __forceinline__ Walk shfl_walk(const Walk& w, int src) {
  Walk r;
  r.b = __shfl_sync(0xffffffffu, w.b, src);
  r.g = __shfl_sync(0xffffffffu, w.g, src);
  r.i = __shfl_sync(0xffffffffu, w.i, src);
  r.nch = __shfl_sync(0xffffffffu, w.nch, src);
  r.L = __shfl_sync(0xffffffffu, w.L, src);
  return r;
}

__device__ __forceinline__ int64_t q_row_of(const DecodeArgs& a, int b) {
  return a.cu_seqlens_q != nullptr ? static_cast<int64_t>(a.cu_seqlens_q[b]) : b;
}

// Block-wide inclusive scan over all kThreads threads.
__device__ __forceinline__ int block_scan(int v, int* warp_sums, int* block_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kConsumerWarps + 1 ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kConsumerWarps + 1) warp_sums[lane] = w;
  }
  __syncthreads();
  const int add = warp > 0 ? warp_sums[warp - 1] : 0;
  *block_total = warp_sums[kConsumerWarps];
  __syncthreads();
  return v + add;
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* empty = full + kStages;
  uint64_t* qfull = empty + kStages;
  uint64_t* qempty = qfull + 2;
  uint64_t* cbar = qempty + 2;
  Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);
  int* s_len = reinterpret_cast<int*>(smem + kOffLens);
  volatile int* abort_flag = &misc->abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = a.num_kv_heads;
  const int B = a.num_seqs;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&qfull[s], 1);
      mbar_init(&qempty[s], 1);
    }
    mbar_init(cbar, kConsumerWarps);
    misc->abort = 0;
    misc->b0 = -1;
    misc->off0 = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }

  prefetch_decode_metadata(a);
  // ---- plan: total chunk count, this CTA's run [c0, c1), its first unit ----
  int local = 0;
  for (int b = tid; b < B; b += kThreads) {
    const int L = seq_len_eff(a, b);
    if (B <= kMaxSmemSeqs) s_len[b] = L;
    local += Hkv * ((L + kChunkTokens - 1) / kChunkTokens);
  }
  int total;
  block_scan(local, misc->warp_sums, &total);
  const RunSplit split{total, static_cast<int>(gridDim.x), kMinChunksPerCta};
  const int c0 = split.begin(blockIdx.x);
  const int c1 = split.begin(blockIdx.x + 1);
  int running = 0;
  for (int base = 0; base < B; base += kThreads) {
    const int b = base + tid;
    int L = 0;
    const int u = b < B ? Hkv * seq_chunks_cached(a, s_len, b, &L) : 0;
    int tile_total;
    const int incl = block_scan(u, misc->warp_sums, &tile_total);
    const int excl = running + incl - u;
    if (u > 0 && excl <= c0 && c0 < excl + u) {
      misc->b0 = b;
      misc->off0 = c0 - excl;
    }
    running += tile_total;
  }
  __syncthreads();
  // The next kernel on the stream may start its own set-up now.
  grid_dep_launch();
  finish_invalid_rows(a, B <= kMaxSmemSeqs ? s_len : nullptr);
  if (c0 >= c1) return;  // no work for this CTA (nothing issued yet)
  const int nloc = c1 - c0;

  Walk w0;
  w0.b = misc->b0;
  w0.nch = seq_chunks_cached(a, s_len, w0.b, &w0.L);
  w0.g = misc->off0 / w0.nch;
  w0.i = misc->off0 % w0.nch;

  const uint32_t smem_base = smem_u32(smem);
  if (warp == kProducerWarp) {
    // ================================ producer ================================
    // Chunks are handled in batches of 32: lane l owns chunk (batch start + l),
    // walks to it and loads its block ids; the next batch's walk and id loads
    // are issued before the current batch's copies so their latency hides.
    int n = 0, seg = -1, q_issued = 0;
    bool ok = true;
    auto prepare = [&](const Walk& start, int cnt, Walk& mw, int& id0, int& id1,
                       int64_t& qrow, int n_first) {
      mw = start;
      for (int k = 0; k < lane && k < cnt - 1; ++k) walk_next(mw, a, s_len);
      id0 = -1;
      id1 = -1;
      qrow = 0;
      if (lane < cnt) {
        const int ntok = min(kChunkTokens, mw.L - mw.i * kChunkTokens);
        const int* row = decode_block_row(a, mw.b);
        id0 = row[2 * mw.i];
        if (ntok > kBlockSize) id1 = row[2 * mw.i + 1];
        if (mw.i == 0 || n_first + lane == 0) qrow = q_row_of(a, mw.b);
      }
    };
    Walk mw;
    int id0, id1;
    int64_t qrow;
    int cnt = min(32, nloc);
    prepare(w0, cnt, mw, id0, id1, qrow, 0);
    // Queries and the cache may come from the previous kernel on the stream
    // (the RoPE + append step): nothing of theirs is read before this.
    grid_dep_wait();
    while (n < nloc && ok) {
      // next batch, issued ahead
      const int n_next = n + cnt;
      const int cnt2 = min(32, nloc - n_next);
      Walk mw2 = mw;
      int id0b = -1, id1b = -1;
      int64_t qrowb = 0;
      if (cnt2 > 0) {
        Walk start = shfl_walk(mw, cnt - 1);
        walk_next(start, a, s_len);
        prepare(start, cnt2, mw2, id0b, id1b, qrowb, n_next);
      }
      // validate this batch's ids (the loads have landed by now)
      if (lane < cnt) {
        const bool bad0 = id0 < 0 || id0 >= a.num_blocks;
        const int ntok = min(kChunkTokens, mw.L - mw.i * kChunkTokens);
        const bool bad1 = ntok > kBlockSize && (id1 < 0 || id1 >= a.num_blocks);
        if (bad0 || bad1) set_err(a.err_word, QATTN_DEVERR_BLOCK);
        if (bad0) id0 = -1;
        if (bad1) id1 = -1;
      }
      for (int c = 0; c < cnt; ++c) {
        const int g = __shfl_sync(0xffffffffu, mw.g, c);
        const int ci = __shfl_sync(0xffffffffu, mw.i, c);
        const int cid0 = __shfl_sync(0xffffffffu, id0, c);
        const int cid1 = __shfl_sync(0xffffffffu, id1, c);
        const int64_t cq = __shfl_sync(0xffffffffu, qrow, c);
        const int stage = n % kStages;
        if (lane == 0) {
          if (ci == 0 || n == 0) {
            ++seg;
            const int slot = seg & 1;
            if (!mbar_wait(&qempty[slot], ((seg >> 1) & 1) ^ 1, abort_flag)) {
              ok = false;
            } else {
              const __nv_bfloat16* qsrc = static_cast<const __nv_bfloat16*>(a.q) +
                                          cq * a.q_row_stride +
                                          static_cast<int64_t>(g) * G * kHeadDim;
              mbar_arrive_expect_tx(&qfull[slot], G * kHeadDim * 2);
              bulk_load(smem + kOffQStage + slot * kMaxGroup * kHeadDim * 2, qsrc,
                        G * kHeadDim * 2, &qfull[slot]);
              ++q_issued;
            }
          }
          if (ok && !mbar_wait(&empty[stage], ((n / kStages) & 1) ^ 1, abort_flag)) ok = false;
          if (ok) {
            const uint32_t bytes = (cid0 >= 0 ? kKBytes : 0) + (cid1 >= 0 ? kKBytes : 0);
            if (bytes == 0) {
              mbar_arrive(&full[stage]);
            } else {
              mbar_arrive_expect_tx(&full[stage], bytes);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // Lanes 0..3 each copy one whole 4 KB (block, kv head) tile: lane =
        // block j (bit 1), K or V (bit 0) -- one warp-wide instruction.
        if (lane < 4) {
          const int j = lane >> 1, isv = lane & 1;
          const int id = j ? cid1 : cid0;
          if (id >= 0) {
            uint8_t* dst = smem + kOffStages + stage * kStageBytes + isv * kKBytes + j * kTileBytes;
            tma_load_cache_tile(dst, isv ? &vmap : &kmap, id * Hkv + g, kBlockSize / 8,
                                &full[stage]);
          }
        }
        ++n;
      }
      mw = mw2;
      id0 = id0b;
      id1 = id1b;
      qrow = qrowb;
      cnt = cnt2;
    }
    // Drain: every stage's most recent load must land before the CTA exits.
    if (lane == 0) {
      const int issued = n;
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / kStages) * kStages;
        if (!mbar_wait_drain(&full[s], (last / kStages) & 1)) break;
      }
      // q copy k went to slot k & 1 with phase parity (k >> 1) & 1.
      for (int k = q_issued - 1; k >= 0 && k >= q_issued - 2; --k)
        mbar_wait_drain(&qfull[k & 1], (k >> 1) & 1);
      if (*abort_flag) set_err(a.err_word, QATTN_DEVERR_TIMEOUT);
    }
    return;
  }

  // ================================= consumers ================================
  const uint32_t qf_addr = smem_base + kOffQf;
  const uint32_t p_addr = smem_base + kOffP + warp * (kMaxGroup * 32 * 4);
  float* pbuf = reinterpret_cast<float*>(smem + kOffP) + warp * kMaxGroup * 32;
  float* mo = reinterpret_cast<float*>(smem + kOffMo);
  float* ml = reinterpret_cast<float*>(smem + kOffMl);
  int cphase = 0;

  // Online-softmax state of this warp for the current unit: running max m
  // (log2 domain), this lane's share of the sum l, and the output of this
  // lane's 4 dimensions kept as (even-token, odd-token) partial pairs.

  float m[G], l[G];
  float2 acc[G][4];
  Walk cw = w0;
  int seg = -1;
  bool ok = true;
  for (int n = 0; n < nloc && ok; ++n, walk_next(cw, a, s_len)) {
    const bool seg_start = (n == 0) || (cw.i == 0);
    const bool seg_end = (n == nloc - 1) || (cw.i == cw.nch - 1);
    if (seg_start) {
      ++seg;
      const int slot = seg & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&qfull[slot], (seg >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(
          smem + kOffQStage + slot * kMaxGroup * kHeadDim * 2);
      float* qfw = reinterpret_cast<float*>(smem + kOffQf);
      for (int e = tid; e < G * kHeadDim; e += kConsumerWarps * 32)
        qfw[e] = __bfloat162float(qs[e]) * a.scale_log2;
      __syncwarp();
      if (lane == 0) mbar_arrive(cbar);
      if (!__all_sync(0xffffffffu, mbar_wait(cbar, cphase & 1, abort_flag))) {
        ok = false;
        break;
      }
      ++cphase;
      if (tid == 0) mbar_arrive(&qempty[slot]);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = make_float2(0.f, 0.f);
      }
    }

    if (n % kConsumerWarps == warp) {
      const int stage = n % kStages;
      if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], (n / kStages) & 1, abort_flag))) {
        ok = false;
        break;
      }
      const uint32_t sK = smem_base + kOffStages + stage * kStageBytes;
      const uint32_t sV = sK + kKBytes;
      const int ntok = min(kChunkTokens, cw.L - cw.i * kChunkTokens);

      // ---- S = q . k, lane-per-token, packed pairs of dimensions ----
      float2 s2[G];
#pragma unroll
      for (int h = 0; h < G; ++h) s2[h] = make_float2(0.f, 0.f);
      {
        const int r = lane & 15;
        const uint32_t rowbase = sK + (lane >> 4) * kTileBytes;
#pragma unroll 4
        for (int c = 0; c < 16; ++c) {
          const uint32_t addr = rowbase + tile_chunk_offset(r, c);
          const uint4 kv = lds128(addr);
          const float2 k01 = make_float2(bf16lo_to_f32(kv.x), bf16hi_to_f32(kv.x));
          const float2 k23 = make_float2(bf16lo_to_f32(kv.y), bf16hi_to_f32(kv.y));
          const float2 k45 = make_float2(bf16lo_to_f32(kv.z), bf16hi_to_f32(kv.z));
          const float2 k67 = make_float2(bf16lo_to_f32(kv.w), bf16hi_to_f32(kv.w));
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float4 qa = lds128f(qf_addr + (h * kHeadDim + c * 8) * 4);
            const float4 qb = lds128f(qf_addr + (h * kHeadDim + c * 8 + 4) * 4);
            float2 t = s2[h];
            t = __ffma2_rn(make_float2(qa.x, qa.y), k01, t);
            t = __ffma2_rn(make_float2(qa.z, qa.w), k23, t);
            t = __ffma2_rn(make_float2(qb.x, qb.y), k45, t);
            t = __ffma2_rn(make_float2(qb.z, qb.w), k67, t);
            s2[h] = t;
          }
        }
      }

      // ---- online softmax (log2 domain) ----
      const bool valid = lane < ntok;
      float alpha[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float sv = valid ? s2[h].x + s2[h].y : -INFINITY;
        const float mnew = fmaxf(m[h], warp_max(sv));
        alpha[h] = exp2f(m[h] - mnew);
        const float p = exp2f(sv - mnew);
        l[h] = fmaf(l[h], alpha[h], p);
        m[h] = mnew;
        pbuf[h * 32 + lane] = p;
      }
      if (ntok < kChunkTokens) {
        // Rows past the end of the context hold stale or never-written
        // data; zero this lane's slice of them so 0 * garbage stays 0.
        for (int j = ntok; j < kChunkTokens; ++j) {
          const uint32_t addr = sV + (j >> 4) * kTileBytes +
                                tile_chunk_offset(j & 15, lane >> 1) + (lane & 1) * 8;
          asm volatile("st.shared.v2.u32 [%0], {%1, %1};" ::"r"(addr), "r"(0u) : "memory");
        }
      }
      __syncwarp();

      // ---- acc = alpha * acc + P V over token pairs, lane-per-4-dims ----
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float2 a2 = make_float2(alpha[h], alpha[h]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = __fmul2_rn(acc[h][e], a2);
      }
      // This lane's 4 dims are 16-byte chunk lane/2 of a row, bytes (lane&1)*8..
      const int vchunk = lane >> 1;
      const uint32_t vlane = sV + (lane & 1) * 8;
#pragma unroll 2
      for (int j4 = 0; j4 < 8; ++j4) {
        float4 p4[G];
#pragma unroll
        for (int h = 0; h < G; ++h) p4[h] = lds128f(p_addr + (h * 32 + j4 * 4) * 4);
#pragma unroll
        for (int pr = 0; pr < 2; ++pr) {
          const int j = j4 * 4 + pr * 2;  // tokens j, j + 1 (same block: j is even)
          const int r0 = j & 15, r1 = r0 + 1;
          const uint32_t vb = vlane + (j >> 4) * kTileBytes;
          const uint2 v0 = lds64(vb + tile_chunk_offset(r0, vchunk));
          const uint2 v1 = lds64(vb + tile_chunk_offset(r1, vchunk));
          const float2 d0 = make_float2(bf16lo_to_f32(v0.x), bf16lo_to_f32(v1.x));
          const float2 d1 = make_float2(bf16hi_to_f32(v0.x), bf16hi_to_f32(v1.x));
          const float2 d2 = make_float2(bf16lo_to_f32(v0.y), bf16lo_to_f32(v1.y));
          const float2 d3 = make_float2(bf16hi_to_f32(v0.y), bf16hi_to_f32(v1.y));
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float2 pp = pr == 0 ? make_float2(p4[h].x, p4[h].y)
                                      : make_float2(p4[h].z, p4[h].w);
            acc[h][0] = __ffma2_rn(pp, d0, acc[h][0]);
            acc[h][1] = __ffma2_rn(pp, d1, acc[h][1]);
            acc[h][2] = __ffma2_rn(pp, d2, acc[h][2]);
            acc[h][3] = __ffma2_rn(pp, d3, acc[h][3]);
          }
        }
      }
      if (ntok < kChunkTokens) fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }

    if (seg_end) {
      // ---- merge the warps' states for this unit ----
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float lt = warp_sum(l[h]);
        *reinterpret_cast<float4*>(&mo[((warp * kMaxGroup) + h) * kHeadDim + lane * 4]) =
            make_float4(acc[h][0].x + acc[h][0].y, acc[h][1].x + acc[h][1].y,
                        acc[h][2].x + acc[h][2].y, acc[h][3].x + acc[h][3].y);
        if (lane == 0) {
          ml[(warp * kMaxGroup + h) * 2 + 0] = m[h];
          ml[(warp * kMaxGroup + h) * 2 + 1] = lt;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(cbar);
      if (!__all_sync(0xffffffffu, mbar_wait(cbar, cphase & 1, abort_flag))) {
        ok = false;
        break;
      }
      ++cphase;
      const int gidx = c0 + n;
      const int u0 = gidx - cw.i;  // list index of this unit's first chunk
      const int first = split.cta_of(u0), last = split.cta_of(u0 + cw.nch - 1);
      const int nparts = last - first + 1;
      const int part = static_cast<int>(blockIdx.x) - first;
      const int64_t row = q_row_of(a, cw.b);
      const int64_t seg_id = static_cast<int64_t>(cw.b) * Hkv + cw.g;
      const bool fits = a.part_base + nparts <= a.ws.max_parts;
      const bool as_part = nparts > 1 || a.part_base > 0;
      if (!fits && tid == 0) set_err(a.err_word, QATTN_DEVERR_CONTEXT);
      for (int idx = tid; idx < G * 32; idx += kConsumerWarps * 32) {
        const int h = idx >> 5, d4 = idx & 31;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, ml[(w * kMaxGroup + h) * 2]);
        float den = 0.f;
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float f = exp2f(ml[(w * kMaxGroup + h) * 2] - M);
          den = fmaf(f, ml[(w * kMaxGroup + h) * 2 + 1], den);
          const float4 ov =
              *reinterpret_cast<const float4*>(&mo[((w * kMaxGroup) + h) * kHeadDim + d4 * 4]);
          num.x = fmaf(f, ov.x, num.x);
          num.y = fmaf(f, ov.y, num.y);
          num.z = fmaf(f, ov.z, num.z);
          num.w = fmaf(f, ov.w, num.w);
        }
        const float inv = 1.f / den;
        const float4 res = make_float4(num.x * inv, num.y * inv, num.z * inv, num.w * inv);
        const int head = cw.g * G + h;
        if (!as_part) {
          uint2 packed;
          packed.x = pack_bf16x2_rn(res.x, res.y);
          packed.y = pack_bf16x2_rn(res.z, res.w);
          *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) +
                                    (row * a.num_heads + head) * kHeadDim + d4 * 4) = packed;
        } else if (fits) {
          const int64_t pidx = seg_id * a.ws.max_parts + a.part_base + part;
          *reinterpret_cast<float4*>(a.ws.part_o + (pidx * G + h) * kHeadDim + d4 * 4) = res;
          if (d4 == 0) a.ws.lse[pidx * G + h] = M + log2f(den);
        }
      }
      if (part == 0 && tid == 0) record_parts(a, seg_id, fits ? a.part_base + nparts : 0);
    }
  }
  if (!ok && lane == 0) set_err(a.err_word, QATTN_DEVERR_TIMEOUT);
}

// K2r: merge the parts of units that straddled CTAs (either decode
// kernel).  One warp per (sequence, kv head) unit; lane = 4 dimensions.
//   out[row, g*G + h] = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M),
// folded in part order with a running maximum M (deterministic); the loads
// of a batch of NB parts (all heads) are issued together.
template <int G, int NB>
__device__ __forceinline__ void fold_parts(const float (&lv)[NB][G], const float4 (&ov)[NB][G],
                                           int count, float (&m)[G], float (&den)[G],
                                           float4 (&num)[G]) {
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    if (j < count) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mn = fmaxf(m[h], lv[j][h]);
        const float sc = exp2f(m[h] - mn);  // 0 for the first part
        const float f = exp2f(lv[j][h] - mn);
        den[h] = fmaf(den[h], sc, f);
        num[h].x = fmaf(num[h].x, sc, f * ov[j][h].x);
        num[h].y = fmaf(num[h].y, sc, f * ov[j][h].y);
        num[h].z = fmaf(num[h].z, sc, f * ov[j][h].z);
        num[h].w = fmaf(num[h].w, sc, f * ov[j][h].w);
        m[h] = mn;
      }
    }
  }
}

// K2r: merge the parts of units that straddled CTAs (either decode
// kernel).  One warp per (sequence, kv head) unit; lane = 4 dimensions.
//   out[row, g*G + h] = sum_p 2^(lse_p - M) o_p / sum_p 2^(lse_p - M),
// folded in part order with a running maximum M (deterministic).  The
// first NB parts are loaded together with the part count (their addresses
// do not depend on it), so the usual merge is one memory round trip.
template <int G, int NB>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeArgs a) {
  grid_dep_wait();  // the parts come from the decode grid
  const int Hkv = a.num_kv_heads;
  const int64_t seg = static_cast<int64_t>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (seg >= static_cast<int64_t>(a.num_seqs) * Hkv) return;
  const int b = static_cast<int>(seg / Hkv), g = static_cast<int>(seg % Hkv);
  const int lane = threadIdx.x & 31;
  const int64_t pbase = seg * a.ws.max_parts * G;
  const float* lse = a.ws.lse + pbase;
  const float* po = a.ws.part_o + pbase * kHeadDim + lane * 4;
  const int nparts = a.ws.nparts[seg];
  int64_t row = b;
  int ql = 1;
  if (a.cu_seqlens_q != nullptr) {
    row = a.cu_seqlens_q[b];
    ql = a.cu_seqlens_q[b + 1] - static_cast<int>(row);
  }
  float lv[NB][G];
  float4 ov[NB][G];
#pragma unroll
  for (int j = 0; j < NB; ++j) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (j < a.ws.max_parts) {  // inside this unit's part slots
        lv[j][h] = lse[j * G + h];
        ov[j][h] =
            *reinterpret_cast<const float4*>(po + static_cast<int64_t>(j * G + h) * kHeadDim);
      }
    }
  }
  if (ql != 1 || nparts <= 1) return;  // not a decode row, or written by the decode kernel
  float m[G], den[G];
  float4 num[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    den[h] = 0.f;
    num[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  fold_parts<G, NB>(lv, ov, nparts, m, den, num);
  for (int p0 = NB; p0 < nparts; p0 += NB) {
#pragma unroll
    for (int j = 0; j < NB; ++j) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (p0 + j < nparts) {
          const int k = (p0 + j) * G + h;
          lv[j][h] = lse[k];
          ov[j][h] = *reinterpret_cast<const float4*>(po + static_cast<int64_t>(k) * kHeadDim);
        }
      }
    }
    fold_parts<G, NB>(lv, ov, nparts - p0, m, den, num);
  }
  __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                        (row * a.num_heads + static_cast<int64_t>(g) * G) * kHeadDim + lane * 4;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float inv = 1.f / den[h];
    uint2 packed;
    packed.x = pack_bf16x2_rn(num[h].x * inv, num[h].y * inv);
    packed.y = pack_bf16x2_rn(num[h].z * inv, num[h].w * inv);
    *reinterpret_cast<uint2*>(orow + h * kHeadDim) = packed;
  }
}

template <int G>
cudaError_t launch_merge_g(const DecodeArgs& a, cudaStream_t stream) {
  const int64_t segs = static_cast<int64_t>(a.num_seqs) * a.num_kv_heads;
  cudaError_t e = launch_pdl(decode_merge_kernel<G, (G >= 4 ? 2 : 8 / G)>,
                             dim3(static_cast<unsigned>((segs + 3) / 4)), dim3(128), 0, stream, a);
  if (e != cudaSuccess) return e;
  return cudaPeekAtLastError();
}

template <int G>
cudaError_t launch_g(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     int num_sms, cudaStream_t stream) {
  cudaError_t e =
      set_max_dynamic_smem(reinterpret_cast<const void*>(paged_decode_kernel<G>), kSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(paged_decode_kernel<G>, dim3(num_sms), dim3(kThreads), kSmemBytes, stream, kmap,
                 vmap, a);
  if (e != cudaSuccess) return e;
  e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  return launch_decode_merge(a, stream);
}

}  // namespace

size_t decode_workspace_bytes(int32_t num_seqs, int32_t max_context_len, int32_t num_kv_heads,
                              int32_t group, int32_t extra_parts) {
  const int64_t nch = (static_cast<int64_t>(max_context_len) + kChunkTokens - 1) / kChunkTokens;
  const int64_t max_parts = (nch + kMinChunksPerCta - 1) / kMinChunksPerCta + 1 + extra_parts;
  auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t units = static_cast<int64_t>(num_seqs) * num_kv_heads * max_parts * group;
  return static_cast<size_t>(al(static_cast<int64_t>(num_seqs) * num_kv_heads * 4) +
                             al(units * 4) + al(units * kHeadDim * 4));
}

DecodeWorkspace carve_decode_workspace(void* base, int32_t num_seqs, int32_t max_context_len,
                                       int32_t num_kv_heads, int32_t group, int32_t extra_parts) {
  const int64_t nch = (static_cast<int64_t>(max_context_len) + kChunkTokens - 1) / kChunkTokens;
  const int64_t max_parts = (nch + kMinChunksPerCta - 1) / kMinChunksPerCta + 1 + extra_parts;
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

cudaError_t launch_paged_decode(const DecodeArgs& a, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, int num_sms, cudaStream_t stream) {
  switch (a.num_heads / a.num_kv_heads) {
    case 1: return launch_g<1>(a, kmap, vmap, num_sms, stream);
    case 2: return launch_g<2>(a, kmap, vmap, num_sms, stream);
    case 3: return launch_g<3>(a, kmap, vmap, num_sms, stream);
    case 4: return launch_g<4>(a, kmap, vmap, num_sms, stream);
    case 5: return launch_g<5>(a, kmap, vmap, num_sms, stream);
    case 6: return launch_g<6>(a, kmap, vmap, num_sms, stream);
    case 7: return launch_g<7>(a, kmap, vmap, num_sms, stream);
    case 8: return launch_g<8>(a, kmap, vmap, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qattn
