// Kernel K2t: paged GQA decode with the group's dot products on tcgen05.
//
// What is computed is the decode attention of the grouped-query layer
// ("Qwen2 模型结构代码详解" section 2: 28 query heads share 4 KV heads, scale
// head_dim ** -0.5) over the PagedAttention block cache (vLLM-deploys-Qwen
// notes section 2.1): for each decode sequence b and query head h with KV
// head g = h / G,  out[b, h] = sum_j softmax_j(scale * q[b,h] . k_j) v_j.
//
// Why tensor cores here.  All G query heads of a group read the same keys,
// so per KV tile the work is a dense product of the tile (tokens x 128) with
// the group (128 x G).  Done on CUDA cores that costs ~2400 warp
// instructions per 16 KB of KV for G = 7 (measured), which caps the kernel
// well below HBM speed; on tcgen05 the same tile is 16 instructions of one
// thread.  The layout puts tokens on the MMA M dimension (128) and the group
// on N (padded to 16), so the K tile straight from the cache is the K-major
// A operand and the V tile is the MN-major A operand of the transposed
// product -- nothing is re-laid:
//     S^T[tok, h]  = K[tok, :] . Q^T[:, h]           (M = 128, N = 16, K = 128)
//     O^T[d, h]   += V^T[d, tok] . P^T[tok, h]        (M = 128, N = 16, K = 128)
// The online-softmax state (per-head running max and sum over tokens) is
// reduced across the 128 token threads with warp shuffles plus one exchange
// between the four softmax warps per tile.
//
// Structure (one CTA per SM, persistent):
//   * work list: (sequence, kv head) units cut into 128-token tiles (eight
//     16-token blocks); each CTA takes an equal contiguous run of tiles
//     (>= 2); a unit that straddles CTAs leaves one partial result per CTA,
//     merged in part order by K2r (a round trip to memory inside this
//     kernel costs ~3 us while every SM streams, so the merge waits for the
//     grid to finish; K2r's CTAs launch early and wait on the grid).
//   * warp 4 issues TMA: Q^T of a unit (a G x 128 box of the query rows),
//     K and V tiles (16 x 64 boxes, 128-byte swizzle) into 3-deep K and V
//     rings; one thread of warp 5 issues the Q K^T MMAs and one of warp 6
//     the P V MMAs (two issuers: each MMA issue waits on the pipe); warps 0-3
//     (thread = token for S, thread = dimension for O) run the softmax and
//     write P^T as bf16 into swizzled shared memory; four epilogue warps (7-10,
//     FP8 11-14) finish each unit: O^T / l into the output, or the CTA's part
//     of a straddling unit (measured: done by the softmax warps, each unit's
//     epilogue took ~1.4 us of their time, and runs holding many short units
//     fell behind the others).
//   * O is rescaled lazily (only when a head's max grows by more than 2^8).
//   * keys past the context are masked in S and their V rows zeroed.
//   * every wait is bounded; on a timeout all roles unwind, drain their
//     copies and MMAs, and TMEM is freed.
//
// FP8 cache (kFp8; kv_cache_dtype "fp8", fp8_e4m3fn codes with a cache
// scale per tensor, "Qwen2大模型架构解析与vLLM优化实践" sections 4.1, 4.2,
// 6.3): the cache tiles are half the bytes (128 B per token row) and land
// by TMA in 4-deep 16 KB rings.  S^T = K . Q^T runs on the codes themselves
// (kind::f8f6f4, the K tile straight from the ring as the K-major e4m3 A):
// per unit four more warps (7-10) write Q^T as two e4m3 rows per head,
// hi = e4m3(q 2^e) and lo = e4m3(q 2^e - hi), with 2^e the power of two that
// puts the head's largest |q| in [128, 256).  hi + lo is the bf16 value
// exactly for every element within 2^9 of that maximum (hi keeps four
// significant bits, the residue at most four more, none of them below the
// e4m3 subnormal step 2^-9 while the scaled |q| >= 2^-2; smaller elements
// are off by at most 2^-10 scaled), so the score is the two columns' sum
// times 2^-e -- the bf16 path's dot product up to fp32 rounding.  The same warps dequantise V (e4m3 -> f16 is exact) into
// the swizzled MN-major f16 layout the bf16 path gets from TMA, with rows
// past the context written as zeros, and P V runs in f16 (P^T written as
// f16); k_scale is folded into the logit scale and v_scale into the
// epilogue.
#include <math.h>

#include "common.cuh"
#include "internal.h"

// Tracing build only (compiled with -DQATTN_TRACE, never in the library the
// entry points ship in): %globaltimer stamps per CTA at the kernel's phase
// boundaries, read back with qattn_trace_read (include/qattn_trace.h).
#ifdef QATTN_TRACE
__device__ unsigned long long g_qattn_decode_trace[qattn::kTraceCtas * qattn::kTraceSlots];
#define QATTN_STAMP(slot)                                                                   \
  do {                                                                                      \
    if (blockIdx.x < qattn::kTraceCtas)                                                     \
      g_qattn_decode_trace[blockIdx.x * qattn::kTraceSlots + (slot)] = qattn::globaltimer_ns(); \
  } while (0)
#else
#define QATTN_STAMP(slot) \
  do {                    \
  } while (0)
#endif

namespace qattn {
namespace {

constexpr int kTile = kTcTileTokens;  // 128 tokens
constexpr int kN = 16;                // MMA N: the query group padded to 16 heads
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;     // issues the Q K^T stream (and owns TMEM)
constexpr int kPvWarp = 6;      // issues the P V stream
constexpr int kConvWarp0 = 7;   // FP8 only: warps 7-10 dequantise
// The four epilogue warps (7-10 for bf16, 11-14 for FP8) cover the four
// tensor-memory lane quarters between them.
// A tile of 128 tokens lands as 8-token row groups 2 KB apart whatever the
// block size (a block's box is block_size / 8 such groups), so the code below
// addresses it in 16-token / 4 KB units.
constexpr int kCacheTileBytes = 16 * kHeadDim * 2;  // 16 tokens: 4 KB
constexpr int kTileBytes = kTile * kHeadDim * 2;    // 32 KB
constexpr int kSmallHalf = kN * 128;     // 16 rows x 128 B
constexpr int kSmallBytes = 2 * kSmallHalf;
constexpr int kQ8Bytes = kN * 128;      // FP8: Q^T as e4m3, 16 rows x 128 B
constexpr uint32_t kColO = 32;   // O^T of unit u at kColO + (u & 1) * kN
constexpr float kLazyRescale = 8.0f;
constexpr int kMaxSmemSeqs = 2048;

// Shared-memory layout.  bf16: 3 + 3 ring slots of 32 KB cache tiles.  FP8:
// 4 + 4 slots of 16 KB code tiles, then two 32 KB f16 V tiles; after the
// P^T buffers two slots of e4m3 Q^T and, after the epilogue's maxima, the
// per-head scales 2^-e of the two units those slots belong to.
template <bool kFp8>
struct Lay {
  static constexpr int kWarps = kFp8 ? 15 : 11;
  static constexpr int kEpiWarp0 = kFp8 ? 11 : 7;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kKStages = kFp8 ? 4 : 3;
  static constexpr int kVStages = kFp8 ? 4 : 3;
  static constexpr int kStageBytes = kFp8 ? kTile * kHeadDim : kTileBytes;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKStages * kStageBytes;
  static constexpr int kOffVc = kOffV + kVStages * kStageBytes;  // FP8: f16 V tiles
  static constexpr int kOffQ = kOffVc + (kFp8 ? 2 * kTileBytes : 0);  // 2 slots of Q^T
  static constexpr int kOffP = kOffQ + 2 * kSmallBytes;               // 2 buffers of P^T
  static constexpr int kOffQ8 = kOffP + 2 * kSmallBytes;              // FP8: 2 x e4m3 Q^T
  static constexpr int kOffRed = kOffQ8 + (kFp8 ? 2 * kQ8Bytes : 0);  // [2][4][16] fp32
  static constexpr int kOffEpiL = kOffRed + 2 * 4 * kN * 4;           // [2][4][16] fp32
  static constexpr int kOffEpiM = kOffEpiL + 2 * 4 * kN * 4;          // [2][16] fp32
  static constexpr int kOffQs = kOffEpiM + 2 * kN * 4;                // FP8: [2][16] fp32
  static constexpr int kOffBars = kOffQs + (kFp8 ? 2 * kN * 4 : 0);
  // k_full/k_empty[kKStages] v_full/v_empty[kVStages] q_full q_empty s_full
  // s_free p_full pv_done o_free epi_full epi_empty seg_done [2] rbar
  // mma_done; FP8 adds vc_full vc_empty qc_full sc_free [2]
  static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 2 * 10 + 2 + (kFp8 ? 8 : 0);
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kOffLens = kOffMisc + 128;  // Misc
  static constexpr int kSmemBytes = kOffLens + kMaxSmemSeqs * 4 + 1024;
  static constexpr uint32_t kTmemCols = 64;
};
static_assert(Lay<true>::kOffQ8 % 1024 == 0, "e4m3 Q^T slots on the 128-byte swizzle's period");
static_assert(Lay<true>::kSmemBytes <= 227 * 1024, "FP8 decode shared memory");
static_assert(Lay<false>::kSmemBytes <= 227 * 1024, "decode shared memory");

struct Misc {
  uint32_t tmem;
  int abort;
  int b0;
  int off0;
  int warp_sums[16];
};
static_assert(sizeof(Misc) <= 128, "Misc overlaps the context lengths");

__device__ __forceinline__ int seq_len_eff(const DecodeArgs& a, int b) {
  return decode_len_eff(a, b);
}

__device__ __forceinline__ int seq_len_cached(const DecodeArgs& a, const int* s_len, int b) {
  return a.num_seqs <= kMaxSmemSeqs ? s_len[b] : seq_len_eff(a, b);
}

struct Walk {
  int b, g, i, nt, L;  // sequence, kv head, tile i of nt, context length
};

__device__ __forceinline__ void walk_next(Walk& w, const DecodeArgs& a, const int* s_len) {
  if (++w.i < w.nt) return;
  w.i = 0;
  if (++w.g < a.num_kv_heads) return;
  w.g = 0;
  for (;;) {
    ++w.b;
    if (w.b >= a.num_seqs) {
      w.nt = 0;
      return;
    }
    w.L = seq_len_cached(a, s_len, w.b);
    w.nt = (w.L + kTile - 1) / kTile;
    if (w.nt > 0) return;
  }
}

__device__ __forceinline__ Walk shfl_walk_helper(const Walk& w, int src) {
  Walk r;
  r.b = __shfl_sync(0xffffffffu, w.b, src);
  r.g = __shfl_sync(0xffffffffu, w.g, src);
  r.i = __shfl_sync(0xffffffffu, w.i, src);
  r.nt = __shfl_sync(0xffffffffu, w.nt, src);
  r.L = __shfl_sync(0xffffffffu, w.L, src);
  return r;
}

__device__ __forceinline__ int64_t q_row_of(const DecodeArgs& a, int b) {
  return a.cu_seqlens_q != nullptr ? static_cast<int64_t>(a.cu_seqlens_q[b]) : b;
}

// Inclusive scan over the CTA's NW warps.
template <int NW>
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
    int w = lane < NW ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < NW) warp_sums[lane] = w;
  }
  __syncthreads();
  const int add = warp > 0 ? warp_sums[warp - 1] : 0;
  *block_total = warp_sums[NW - 1];
  __syncthreads();
  return v + add;
}

template <int G, bool kFp8>
__global__ void __launch_bounds__(Lay<kFp8>::kThreads, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap,
                           const __grid_constant__ CUtensorMap qmap, const DecodeArgs a) {
  using L = Lay<kFp8>;
  constexpr int kThreads = L::kThreads;
  // The FP8 kernel (fifteen warps in six roles) is sensitive to its code
  // size: its MMA loops are unrolled by 4 (measured against 2 and 8: b64
  // 51.8 / 53.3 / 55.7 us); bf16 unrolls all eight.
  constexpr int kMmaUnroll = kFp8 ? 4 : 8;
  constexpr int kKStages = L::kKStages;
  constexpr int kVStages = L::kVStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBars);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + kKStages;
  uint64_t* v_full = k_empty + kKStages;
  uint64_t* v_empty = v_full + kVStages;
  uint64_t* q_full = v_empty + kVStages;
  uint64_t* q_empty = q_full + 2;
  uint64_t* s_full = q_empty + 2;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  // pv_done[b]: one phase per P V group that read P^T buffer b (tiles of
  // parity b).  Waiters are never more than one phase behind on either.
  uint64_t* pv_done = p_full + 2;
  // o_free[b]: the softmax has read O^T slot b (units of parity b).
  uint64_t* o_free = pv_done + 2;
  // epi_full[s] / epi_empty[s]: the softmax has handed segment k's maximum
  // and row sums (k & 1 == s) to the epilogue warps / they have read them;
  // seg_done[s]: segment k's last P V is complete (its O^T is final).
  uint64_t* epi_full = o_free + 2;
  uint64_t* epi_empty = epi_full + 2;
  uint64_t* seg_done = epi_empty + 2;
  uint64_t* rbar = seg_done + 2;
  uint64_t* mma_done = rbar + 1;
  // FP8: vc_full[b] -- the converters have written V of tile n as f16 (tiles
  // of parity b); vc_empty[b] -- the P V that read it is done; qc_full[s] --
  // the e4m3 Q^T and the scales of slot s are written; sc_free[s] -- the
  // softmax has read slot s's scales.
  uint64_t* vc_full = mma_done + 1;
  uint64_t* vc_empty = vc_full + 2;
  uint64_t* qc_full = vc_empty + 2;
  uint64_t* sc_free = qc_full + 2;
  Misc* misc = reinterpret_cast<Misc*>(smem + L::kOffMisc);
  int* s_len = reinterpret_cast<int*>(smem + L::kOffLens);
  float* red = reinterpret_cast<float*>(smem + L::kOffRed);
  float* epi_l = reinterpret_cast<float*>(smem + L::kOffEpiL);
  float* epi_m = reinterpret_cast<float*>(smem + L::kOffEpiM);
  float* q_inv = reinterpret_cast<float*>(smem + L::kOffQs);  // FP8: 2^-e per head
  volatile int* abort_flag = &misc->abort;
  const uint32_t sbase = smem_u32(smem);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) QATTN_STAMP(0);  // entry
  const int Hkv = a.num_kv_heads;
  const int B = a.num_seqs;
  const int bpt = kTile / a.block_size;    // cache blocks per tile: 8, 4 or 2
  const int groups = a.block_size / 8;     // 8-row groups per block box
  const uint32_t blk_bytes = static_cast<uint32_t>(a.block_size) * kHeadDim * (kFp8 ? 1 : 2);

  prefetch_decode_metadata(a);
  // Barriers and the zeroed Q^T / P^T buffers do not depend on the plan:
  // set them up while the context lengths are on their way (the last
  // thread, whose share of the plan is smallest, initialises the barriers;
  // the barrier after the plan publishes them).
  if (tid == kThreads - 1) {
    // K slots are released by the MMA; V slots by the MMA (bf16) or the four
    // converter warps (FP8).
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], kFp8 ? 4 : 1);
    }
    if (kFp8) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(&vc_full[s], 4);
        mbar_init(&vc_empty[s], 1);
        mbar_init(&qc_full[s], 4);
        mbar_init(&sc_free[s], 4);
      }
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 4);
      mbar_init(&p_full[s], 4);
      mbar_init(&pv_done[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&o_free[s], 4);     // the four epilogue warps
      mbar_init(&epi_full[s], 4);   // the four softmax warps
      mbar_init(&epi_empty[s], 4);  // the four epilogue warps
      mbar_init(&seg_done[s], 1);   // the P V thread's commit
    }
    mbar_init(rbar, 4);
    mbar_init(mma_done, 2);  // one commit per MMA-issuing thread
    fence_barrier_init();
  }
  // Rows >= G of Q^T (and the e4m3 rows of no head) stay zero.
  for (int i = tid; i < (4 * kSmallBytes + (kFp8 ? 2 * kQ8Bytes : 0)) / 16; i += kThreads)
    sts128(sbase + L::kOffQ + i * 16, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  // ---- plan: tile count, this CTA's run [c0, c1), its first unit ----
  if (tid == 0) {
    misc->abort = 0;
    misc->b0 = -1;
    misc->off0 = 0;
  }
  int total, c0, c1;
  RunSplit split;
  if (B <= kThreads) {
    // one sequence per thread: a single scan gives the total and each
    // sequence's first tile
    const int b = tid;
    int u = 0;
    if (b < B) {
      const int L = seq_len_eff(a, b);
      if (B <= kMaxSmemSeqs) s_len[b] = L;
      u = Hkv * ((L + kTile - 1) / kTile);
    }
    const int incl = block_scan<L::kWarps>(u, misc->warp_sums, &total);
    split = RunSplit{total, static_cast<int>(gridDim.x), kTcMinTilesPerCta};
    c0 = split.begin(blockIdx.x);
    c1 = split.begin(blockIdx.x + 1);
    const int excl = incl - u;
    if (u > 0 && excl <= c0 && c0 < excl + u) {
      misc->b0 = b;
      misc->off0 = c0 - excl;
    }
  } else {
    int local = 0;
    for (int b = tid; b < B; b += kThreads) {
      const int L = seq_len_eff(a, b);
      if (B <= kMaxSmemSeqs) s_len[b] = L;
      local += Hkv * ((L + kTile - 1) / kTile);
    }
    block_scan<L::kWarps>(local, misc->warp_sums, &total);
    split = RunSplit{total, static_cast<int>(gridDim.x), kTcMinTilesPerCta};
    c0 = split.begin(blockIdx.x);
    c1 = split.begin(blockIdx.x + 1);
    int running = 0;
    for (int base = 0; base < B; base += kThreads) {
      const int b = base + tid;
      const int L = b < B ? seq_len_cached(a, s_len, b) : 0;
      const int u = Hkv * ((L + kTile - 1) / kTile);
      int tile_total;
      const int incl = block_scan<L::kWarps>(u, misc->warp_sums, &tile_total);
      const int excl = running + incl - u;
      if (u > 0 && excl <= c0 && c0 < excl + u) {
        misc->b0 = b;
        misc->off0 = c0 - excl;
      }
      running += tile_total;
    }
  }
  __syncthreads();
  if (tid == 0) QATTN_STAMP(1);  // plan done
  // The next kernel on the stream may start its own set-up now.
  grid_dep_launch();
  finish_invalid_rows(a, B <= kMaxSmemSeqs ? s_len : nullptr);
  if (c0 >= c1) return;  // nothing for this CTA: no copy or TMEM in use yet
  const int nloc = c1 - c0;

  // ---- set-up: TMEM ----
  if (warp == kMmaWarp) {
    tmem_alloc(&misc->tmem, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem;

  Walk w0;
  w0.b = misc->b0;
  w0.L = seq_len_cached(a, s_len, w0.b);
  w0.nt = (w0.L + kTile - 1) / kTile;
  w0.g = misc->off0 / w0.nt;
  w0.i = misc->off0 % w0.nt;

  if (warp == kProducerWarp) {
    // ================================ producer ================================
    // Batches of 32 tiles: lane l walks to tile (batch start + l) and loads
    // its block ids (up to eight); lane 0 then issues the copies tile by tile.
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      tma_prefetch_desc(&qmap);
    }
    Walk bw = w0;
    // V of a tile is issued one tile after its K (order K0 K1 V0 K2 V1 ...):
    // V lands about when P V needs it instead of idling in its ring slot
    // while the softmax runs, and at start-up the first K tiles are served
    // ahead of the V burst.
    // The KV tiles are read once: evict-first in L2, so that they do not
    // push out the parts the merge kernel reads back, the query rows and
    // the block tables.
    const uint64_t kv_policy = policy_evict_first();
    int n = 0, seg = -1, nv = 0;
    int prev_id = -1, prev_g = 0;
    uint32_t prev_nvalid = 0;
    bool ok = true;
    auto issue_v = [&](int j, int id_lane, int gg, uint32_t nval) -> bool {
      const int vs = j % kVStages;
      bool okv = true;
      if (lane == 0) {
        okv = mbar_wait(&v_empty[vs], ((j / kVStages) & 1) ^ 1, abort_flag, a.wait_ns);
        if (okv) mbar_arrive_expect_tx(&v_full[vs], nval * blk_bytes);
      }
      okv = __shfl_sync(0xffffffffu, okv, 0);
      if (!okv) return false;
      if (lane < bpt && id_lane >= 0) {
        uint8_t* dst = smem + L::kOffV + vs * L::kStageBytes + lane * blk_bytes;
        if constexpr (kFp8)
          tma_load_2d_hint(dst, &vmap, 0, (id_lane * Hkv + gg) * a.block_size, &v_full[vs], kv_policy);
        else
          tma_load_cache_tile_hint(dst, &vmap, id_lane * Hkv + gg, groups, &v_full[vs], kv_policy);
      }
      ++nv;
      return true;
    };
    // Queries and the cache may come from the previous kernel on the stream
    // (the RoPE + append step): nothing of theirs is read before this.
    grid_dep_wait();
    while (n < nloc && ok) {
      const int cnt = min(32, nloc - n);
      Walk mw = bw;
      for (int k = 0; k < lane && k < cnt - 1; ++k) walk_next(mw, a, s_len);
      int ids[8];
      int64_t qrow = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) ids[j] = -1;
      if (lane < cnt) {
        const int ntok = min(kTile, mw.L - mw.i * kTile);
        const int nblk = (ntok + a.block_size - 1) / a.block_size;
        const int* row = decode_block_row(a, mw.b) + mw.i * bpt;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < nblk) ids[j] = row[j];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j < nblk && (ids[j] < 0 || ids[j] >= a.num_blocks)) {
            set_err(a.err_word, QATTN_DEVERR_BLOCK);
            ids[j] = -1;
          }
        }
        if (mw.i == 0 || n + lane == 0) qrow = q_row_of(a, mw.b);
      }
      for (int c = 0; c < cnt && ok; ++c) {
        const int g = __shfl_sync(0xffffffffu, mw.g, c);
        const int ci = __shfl_sync(0xffffffffu, mw.i, c);
        const int64_t cq = __shfl_sync(0xffffffffu, qrow, c);
        // Lane j (< blocks per tile) issues block j's box itself: one
        // warp-wide TMA instruction then moves the tile's boxes (a single lane
        // issuing all 32 boxes of a tile was measured at ~55 ns per box).
        int myid = -1;
        uint32_t nvalid = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int v = __shfl_sync(0xffffffffu, ids[j], c);
          if (lane == j) myid = v;
          nvalid += v >= 0 ? 1u : 0u;
        }
        if (lane == 0 && (ci == 0 || n == 0)) {
          ++seg;
          const int qs = seg & 1;
          ok = mbar_wait(&q_empty[qs], ((seg >> 1) & 1) ^ 1, abort_flag, a.wait_ns);
          if (ok) {
            mbar_arrive_expect_tx(&q_full[qs], 2 * G * 128);
            uint8_t* qdst = smem + L::kOffQ + qs * kSmallBytes;
            tma_load_3d(qdst, &qmap, 0, g * G, static_cast<int32_t>(cq), &q_full[qs]);
            tma_load_3d(qdst + kSmallHalf, &qmap, 64, g * G, static_cast<int32_t>(cq),
                        &q_full[qs]);
          }
        }
        const int ks = n % kKStages;
        if (lane == 0 && ok) {
          ok = mbar_wait(&k_empty[ks], ((n / kKStages) & 1) ^ 1, abort_flag, a.wait_ns);
          if (ok) mbar_arrive_expect_tx(&k_full[ks], nvalid * blk_bytes);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        // (a test may ask the first CTA to skip one copy: its K barrier
        // then never completes and the waits on it run out)
        const bool skip = blockIdx.x == 0 && n == a.debug_skip_k;
        if (lane < bpt && myid >= 0 && !skip) {
          uint8_t* dst = smem + L::kOffK + ks * L::kStageBytes + lane * blk_bytes;
          if constexpr (kFp8)
            tma_load_2d_hint(dst, &kmap, 0, (myid * Hkv + g) * a.block_size, &k_full[ks], kv_policy);
          else
            tma_load_cache_tile_hint(dst, &kmap, myid * Hkv + g, groups, &k_full[ks], kv_policy);
        }
        ++n;  // K(n) issued
        if (n >= 2 && !issue_v(n - 2, prev_id, prev_g, prev_nvalid)) {
          ok = false;
          break;
        }
        prev_id = myid;
        prev_g = g;
        prev_nvalid = nvalid;
      }
      bw = shfl_walk_helper(mw, cnt - 1);
      walk_next(bw, a, s_len);
    }
    if (lane == 0) QATTN_STAMP(3);  // every copy issued
    if (ok && n > 0 && nv < n) issue_v(n - 1, prev_id, prev_g, prev_nvalid);
    // Drain: the most recent K, V and Q copies land before the CTA exits.
    if (lane == 0) {
      const int nk = n;
      for (int j = nk - 1; j >= 0 && j >= nk - kKStages; --j)
        mbar_wait_drain(&k_full[j % kKStages], (j / kKStages) & 1, a.drain_ns);
      for (int j = nv - 1; j >= 0 && j >= nv - kVStages; --j)
        mbar_wait_drain(&v_full[j % kVStages], (j / kVStages) & 1, a.drain_ns);
      for (int s = seg; s >= 0 && s >= seg - 1; --s) mbar_wait_drain(&q_full[s & 1], (s >> 1) & 1, a.drain_ns);
      if (*abort_flag) set_err(a.err_word, QATTN_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ============================= MMA issuers ===============================
    // Warp 5 issues Q K^T(n) as soon as K(n) is in and S buffer n & 1 is
    // free; warp 6 issues P V(j) as soon as P(j) and V(j) are in (it frees
    // V's ring slot, the resource the producer waits on longest).  A thread
    // issuing tcgen05.mma waits for the pipe to take each instruction (~90
    // cycles even at N = 16, measured), so with one issuer each stream
    // waited behind the other's eight MMAs.  The streams share no tensor
    // memory (S vs O^T) and each thread's commits track its own MMAs.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = kFp8 ? idesc_e4m3_f32(kTile, kN)
                                         : idesc_bf16_f32(kTile, kN, false, false);
      constexpr uint32_t idesc_pv = kFp8 ? idesc_f16_f32(kHeadDim, kN, false, true)
                                         : idesc_bf16_f32(kHeadDim, kN, false, true);
      bool ok = true;
      uint64_t idle_since = 0;
      // No progress for the wait limit (or the abort flag): give up.
      auto idle = [&](bool progressed) {
        if (progressed) {
          idle_since = 0;
        } else {
          const uint64_t now = globaltimer_ns();
          if (idle_since == 0) {
            idle_since = now;
          } else if (*abort_flag || now - idle_since > a.wait_ns) {
            *abort_flag = 1;
            ok = false;
          }
        }
      };
      if (warp == kPvWarp) {
        Walk pw = w0;
        int pn = 0, pseg = -1;
        while (pn < nloc && ok) {
          bool progressed = false;
          const bool first = (pn == 0) || (pw.i == 0);
          const bool last = (pn == nloc - 1) || (pw.i == pw.nt - 1);
          const int seg_j = pseg + (first ? 1 : 0);
          const int pb = pn & 1;
          bool ready = mbar_test(&p_full[pb], (pn >> 1) & 1) &&
                       (kFp8 ? mbar_test(&vc_full[pn & 1], (pn >> 1) & 1)
                             : mbar_test(&v_full[pn % kVStages], (pn / kVStages) & 1));
          // A unit's first P V overwrites O^T slot seg_j & 1, last read
          // for unit seg_j - 2.
          if (ready && first && seg_j >= 2)
            ready = mbar_test(&o_free[seg_j & 1], ((seg_j >> 1) - 1) & 1);
          if (ready) {
            tc_fence_after();
            const uint32_t sv = kFp8 ? sbase + L::kOffVc + (pn & 1) * kTileBytes
                                     : sbase + L::kOffV + (pn % kVStages) * kTileBytes;
            const uint32_t sp = sbase + L::kOffP + pb * kSmallBytes;
#pragma unroll(kMmaUnroll)
            for (int k = 0; k < kTile / 16; ++k) {
              // V tile as the MN-major A: the two 64-dim halves 1 KB apart
              // (LBO), 8-token groups 2 KB apart (SBO); K step k = tokens
              // 16k..16k+15.
              const uint64_t ad = sdesc_sw128(sv + k * 4096, 1024, 2048);
              const uint64_t bd =
                  sdesc_sw128(sp + (k >> 2) * kSmallHalf + (k & 3) * 32, 16, 1024);
              mma_bf16_ss(tmem + kColO + (seg_j & 1) * kN, ad, bd, idesc_pv,
                          (first && k == 0) ? 0u : 1u);
            }
            mma_commit(&pv_done[pb]);
            mma_commit(kFp8 ? &vc_empty[pn & 1] : &v_empty[pn % kVStages]);
            if (last) mma_commit(&seg_done[seg_j & 1]);
            if (first) pseg = seg_j;
            ++pn;
            walk_next(pw, a, s_len);
            progressed = true;
          }
          idle(progressed);
        }
      } else {
        Walk qw = w0;
        int qn = 0, qseg = -1;
        while (qn < nloc && ok) {
          bool progressed = false;
          const bool first = (qn == 0) || (qw.i == 0);
          const bool last = (qn == nloc - 1) || (qw.i == qw.nt - 1);
          const int seg_q = qseg + (first ? 1 : 0);
          const int ks = qn % kKStages, sb = qn & 1;
          bool ready = mbar_test(&k_full[ks], (qn / kKStages) & 1);
          if (ready && qn >= 2) ready = mbar_test(&s_free[sb], ((qn >> 1) & 1) ^ 1);
          if (ready && first)
            ready = mbar_test(kFp8 ? &qc_full[seg_q & 1] : &q_full[seg_q & 1], (seg_q >> 1) & 1);
          if (ready) {
            tc_fence_after();
            const uint32_t sk = sbase + L::kOffK + ks * L::kStageBytes;
            if constexpr (kFp8) {
              // The code tile as the K-major e4m3 A: 128-byte token rows,
              // 8-row groups 1 KB apart; K step k = dims 32k..32k+31 (32 B
              // into the swizzle row).  B: the slot's e4m3 Q^T, hi rows
              // 0..G-1 and lo rows 8..8+G-1, in the same layout.
              const uint32_t sq = sbase + L::kOffQ8 + (seg_q & 1) * kQ8Bytes;
#pragma unroll(kMmaUnroll)
              for (int k = 0; k < kHeadDim / 32; ++k) {
                const uint64_t ad = sdesc_sw128(sk + k * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(sq + k * 32, 16, 1024);
                mma_e4m3_ss(tmem + sb * kN, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
              }
            } else {
              const uint32_t sq = sbase + L::kOffQ + (seg_q & 1) * kSmallBytes;
#pragma unroll(kMmaUnroll)
              for (int k = 0; k < kHeadDim / 16; ++k) {
                const uint64_t bd =
                    sdesc_sw128(sq + (k >> 2) * kSmallHalf + (k & 3) * 32, 16, 1024);
                // K tile as the K-major A: dim half k/4 at +1 KB, 8-token
                // groups 2 KB apart.
                const uint64_t ad = sdesc_sw128(sk + (k >> 2) * 1024 + (k & 3) * 32, 16, 2048);
                mma_bf16_ss(tmem + sb * kN, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
              }
            }
            mma_commit(&s_full[sb]);
            mma_commit(&k_empty[ks]);
            if (last) mma_commit(&q_empty[seg_q & 1]);
            if (first) qseg = seg_q;
            ++qn;
            walk_next(qw, a, s_len);
            progressed = true;
          }
          idle(progressed);
        }
      }
      // Drain: every MMA of both threads completes before TMEM is released.
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0, a.drain_ns);
    }
    __syncwarp();
  } else if (warp >= L::kEpiWarp0) {
    // ============================== epilogue ================================
    // Thread = dimension row d of O^T (warp w reads TMEM lanes 32 (w % 4) ..
    // 32 (w % 4) + 31).  For each segment (a unit's tiles in this CTA's run):
    // wait for the softmax's maximum and row sums and for the segment's last
    // P V, read O^T, release its TMEM slot, and write out = O / l -- or, when
    // the unit straddles CTAs, this CTA's normalised part and its log2-sum-exp
    // for the merge kernel.  Off the softmax warps, a unit boundary costs the
    // softmax only its row-sum hand-over.
    const int d = ((warp & 3) << 5) | lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    bool ok = true;
    Walk ew = w0;
    int seg = -1;
    for (int j = 0; j < nloc && ok; ++j) {
      const bool first = (j == 0) || (ew.i == 0);
      const bool last = (j == nloc - 1) || (ew.i == ew.nt - 1);
      if (first) ++seg;
      if (last) {
        const int es = seg & 1;
        bool w_ok = mbar_wait(&epi_full[es], (seg >> 1) & 1, abort_flag, a.wait_ns);
        if (w_ok) w_ok = mbar_wait(&seg_done[es], (seg >> 1) & 1, abort_flag, a.wait_ns);
        if (!__all_sync(0xffffffffu, w_ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float o[kN];
        tmem_ld16(lane_addr + kColO + es * kN, o);
        float ltot[G], mu[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float* el = epi_l + es * 4 * kN + h;
          ltot[h] = (el[0 * kN] + el[1 * kN]) + (el[2 * kN] + el[3 * kN]);
          mu[h] = epi_m[es * kN + h];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&o_free[es]);
          mbar_arrive(&epi_empty[es]);
        }
        const int u0 = c0 + j - ew.i;  // list index of the unit's first tile
        const int first_cta = split.cta_of(u0), last_cta = split.cta_of(u0 + ew.nt - 1);
        const int nparts = last_cta - first_cta + 1;
        const int part = static_cast<int>(blockIdx.x) - first_cta;
        const int64_t row = q_row_of(a, ew.b);
        const int64_t seg_id = static_cast<int64_t>(ew.b) * Hkv + ew.g;
        const bool fits = a.part_base + nparts <= a.ws.max_parts;
        // O / l, times v_scale for an FP8 cache
        auto out_val = [&](float ov, float l) -> float {
          if constexpr (kFp8)
            return (ov / l) * a.v_scale;
          else
            return ov / l;
        };
        if (nparts == 1 && a.part_base == 0) {
          __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                                (row * a.num_heads + static_cast<int64_t>(ew.g) * G) * kHeadDim;
#pragma unroll
          for (int h = 0; h < G; ++h)
            orow[h * kHeadDim + d] = __float2bfloat16_rn(out_val(o[h], ltot[h]));
        } else if (fits) {
          const int64_t pidx = seg_id * a.ws.max_parts + a.part_base + part;
#pragma unroll
          for (int h = 0; h < G; ++h)
            a.ws.part_o[(pidx * G + h) * kHeadDim + d] = out_val(o[h], ltot[h]);
          if (d < G) {
#pragma unroll
            for (int h = 0; h < G; ++h)
              if (h == d) a.ws.lse[pidx * G + h] = mu[h] + log2f(ltot[h]);
          }
        } else if (d == 0) {
          set_err(a.err_word, QATTN_DEVERR_CONTEXT);
        }
        if (part == 0 && d == 0) record_parts(a, seg_id, fits ? a.part_base + nparts : 0);
      }
      walk_next(ew, a, s_len);
    }
    if (!ok && lane == 0) set_err(a.err_word, QATTN_DEVERR_TIMEOUT);
  } else if (kFp8 && warp >= kConvWarp0) {
    // ============================ FP8 converters =============================
    // Per unit, Q^T as e4m3 pairs (warp w takes heads w and w + 4, lane =
    // dims 4 lane .. 4 lane + 3); per tile, V as f16 (thread = token row).
    // Order: the Q^T of the unit tile n starts, then V(n-1) -- the
    // producer's issue order.
    const int row = ((warp & 3) << 5) | lane;
    const int cw = warp - kConvWarp0;  // 0..3
    bool ok = true;
    Walk kw = w0, vw = w0;
    int seg = -1;
    // Q^T of the next unit into e4m3 slot seg & 1 (row h = hi, row 8 + h =
    // lo, 128-byte swizzle) and 2^-e of each head into q_inv, once the bf16
    // Q^T has landed and the softmax has read the slot's previous scales.
    auto conv_q = [&]() -> bool {
      ++seg;
      const int qs = seg & 1;
      bool w_ok = mbar_wait(&q_full[qs], (seg >> 1) & 1, abort_flag, a.wait_ns);
      if (w_ok && seg >= 2)
        w_ok = mbar_wait(&sc_free[qs], ((seg >> 1) & 1) ^ 1, abort_flag, a.wait_ns);
      if (!__all_sync(0xffffffffu, w_ok)) return false;
      for (int h = cw; h < G; h += 4) {
        // bf16 Q^T row h: dims 64 (lane / 16) + 4 (lane % 16) .. + 3, i.e.
        // 4 lane .. 4 lane + 3, in the 128-byte-swizzled half lane / 16
        const uint2 x = lds64(sbase + L::kOffQ + qs * kSmallBytes + (lane >> 4) * kSmallHalf +
                              h * 128 + ((((lane & 15) >> 1) ^ (h & 7)) << 4) + (lane & 1) * 8);
        float v[4] = {bf16lo_to_f32(x.x), bf16hi_to_f32(x.x), bf16lo_to_f32(x.y),
                      bf16hi_to_f32(x.y)};
        const float mx = warp_max(fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])),
                                        fmaxf(fabsf(v[2]), fabsf(v[3]))));
        // 2^e with the maximum's exponent E: max |q| 2^e in [128, 256)
        int e = 7 - (static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127);
        e = max(-126, min(126, e));
        const float up = __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] *= up;  // exact: a power of two
        const uint32_t h01 = cvt_e4m3x2(v[0], v[1]), h23 = cvt_e4m3x2(v[2], v[3]);
        const uint32_t c01 = cvt_f16x2_from_e4m3x2(h01), c23 = cvt_f16x2_from_e4m3x2(h23);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&c01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&c23));
        const uint32_t l01 = cvt_e4m3x2(v[0] - f01.x, v[1] - f01.y);
        const uint32_t l23 = cvt_e4m3x2(v[2] - f23.x, v[3] - f23.y);
        const uint32_t dst = sbase + L::kOffQ8 + qs * kQ8Bytes + ((((lane >> 2) ^ (h & 7))) << 4) +
                             (lane & 3) * 4;
        sts32(dst + h * 128, h01 | (h23 << 16));
        sts32(dst + (8 + h) * 128, l01 | (l23 << 16));
        if (lane == 0) q_inv[qs * kN + h] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qc_full[qs]);
      return true;
    };
    // V(j): the code row as f16 into the swizzled MN-major tile (chunk c of
    // 8 dims at tile_chunk_offset), zeros for rows past the context.
    auto conv_v = [&](int j) -> bool {
      const int vs = j % kVStages;
      const int nvalid_tok = min(kTile, vw.L - vw.i * kTile);
      bool w_ok = mbar_wait(&v_full[vs], (j / kVStages) & 1, abort_flag, a.wait_ns);
      if (w_ok && j >= 2) w_ok = mbar_wait(&vc_empty[j & 1], ((j >> 1) & 1) ^ 1, abort_flag, a.wait_ns);
      if (!__all_sync(0xffffffffu, w_ok)) return false;
      const uint32_t src = sbase + L::kOffV + vs * L::kStageBytes + row * 128;
      const uint32_t dst = sbase + L::kOffVc + (j & 1) * kTileBytes + (row >> 4) * kCacheTileBytes;
      const bool valid = row < nvalid_tok;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (valid) x = lds128(src + ((c ^ (row & 7)) << 4));
        sts128(dst + tile_chunk_offset(row & 15, 2 * c), cvt_f16x2_from_e4m3x2(x.x),
               cvt_f16x2_from_e4m3x2(x.x >> 16), cvt_f16x2_from_e4m3x2(x.y),
               cvt_f16x2_from_e4m3x2(x.y >> 16));
        sts128(dst + tile_chunk_offset(row & 15, 2 * c + 1), cvt_f16x2_from_e4m3x2(x.z),
               cvt_f16x2_from_e4m3x2(x.z >> 16), cvt_f16x2_from_e4m3x2(x.w),
               cvt_f16x2_from_e4m3x2(x.w >> 16));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&v_empty[vs]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&vc_full[j & 1]);
      return true;
    };
    for (int n = 0; n <= nloc && ok; ++n) {
      if (n < nloc) {
        if (n == 0 || kw.i == 0) ok = conv_q();
        walk_next(kw, a, s_len);
        if (!ok) break;
      }
      if (n >= 1) {
        ok = conv_v(n - 1);
        walk_next(vw, a, s_len);
      }
    }
    if (!ok && lane == 0) set_err(a.err_word, QATTN_DEVERR_TIMEOUT);
  } else {
    // =============================== softmax ================================
    const int t = tid;  // token row of S^T / dimension row of O^T = TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m_used[G], l_t[G];
    // FP8: the logit scale of head h for the current unit, scale_log2 * 2^-e
    float qsc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) qsc[h] = a.scale_log2;
    int rphase = 0;
    // PV(j) completes phase j >> 1 of pv_done[j & 1].  Tile n always waits
    // for PV(n-2) (P^T buffer reuse), so when it later waits for PV(n-1)
    // (rescale) neither barrier is two phases behind -- the condition a
    // parity wait needs.
    auto wait_pv = [&](int j) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(&pv_done[j & 1], (j >> 1) & 1, abort_flag, a.wait_ns));
    };
    bool ok = true;
    Walk sw = w0;
    int seg = -1;
    // A step is one tile, or two consecutive tiles of the same unit: the
    // per-step latencies (S wait, the 4-warp max exchange, the P buffer
    // wait, proxy fence) are then paid once per 256 tokens.
    for (int n = 0; n < nloc;) {
      const int cnt = (n + 1 < nloc && sw.i + 1 < sw.nt) ? 2 : 1;
      const int nl = n + cnt - 1;  // the step's last tile
      Walk lw = sw;
      lw.i += cnt - 1;
      const bool seg_start = (n == 0) || (sw.i == 0);
      const bool seg_end = (nl == nloc - 1) || (lw.i == lw.nt - 1);
      if (seg_start) {
        ++seg;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          m_used[h] = -INFINITY;
          l_t[h] = 0.f;
        }
        if constexpr (kFp8) {
          // the unit's 2^-e per head (written with its e4m3 Q^T); slot
          // seg & 1 is rewritten for unit seg + 2 only after this read
          if (!__all_sync(0xffffffffu, mbar_wait(&qc_full[seg & 1], (seg >> 1) & 1, abort_flag,
                                                 a.wait_ns))) {
            ok = false;
            break;
          }
#pragma unroll
          for (int h = 0; h < G; ++h) qsc[h] = a.scale_log2 * q_inv[(seg & 1) * kN + h];
          __syncwarp();
          if (lane == 0) mbar_arrive(&sc_free[seg & 1]);
        }
      }
      const int nv0 = min(kTile, sw.L - sw.i * kTile);
      const int nv1 = cnt == 2 ? min(kTile, sw.L - (sw.i + 1) * kTile) : 0;
      const int nv_last = cnt == 2 ? nv1 : nv0;  // only a unit's last tile is partial

      float s[2][kN];
      bool w_ok = true;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j < cnt) {
          const int nj = n + j;
          w_ok = w_ok && __all_sync(0xffffffffu,
                                    mbar_wait(&s_full[nj & 1], (nj >> 1) & 1, abort_flag, a.wait_ns));
          if (w_ok) {
            tc_fence_after();
            tmem_ld16(lane_addr + (nj & 1) * kN, s[j]);
          }
        }
      }
      if (!w_ok) {
        ok = false;
        break;
      }
      if (n == 0 && t == 0) QATTN_STAMP(2);  // first scores
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        for (int j = 0; j < cnt; ++j) mbar_arrive(&s_free[(n + j) & 1]);

      // per-head max over the step's tokens: shuffle tree, then 4 warps
      float* rd = red + (rphase & 1) * 4 * kN;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if constexpr (kFp8) {  // hi column h plus lo column 8 + h
          s[0][h] = t < nv0 ? (s[0][h] + s[0][8 + h]) * qsc[h] : -INFINITY;
          s[1][h] = t < nv1 ? (s[1][h] + s[1][8 + h]) * qsc[h] : -INFINITY;
        } else {
          s[0][h] = t < nv0 ? s[0][h] * a.scale_log2 : -INFINITY;
          s[1][h] = t < nv1 ? s[1][h] * a.scale_log2 : -INFINITY;
        }
        const float wm = warp_max(fmaxf(s[0][h], s[1][h]));
        if (lane == 0) rd[warp * kN + h] = wm;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(rbar);
      if (!__all_sync(0xffffffffu, mbar_wait(rbar, rphase & 1, abort_flag, a.wait_ns))) {
        ok = false;
        break;
      }
      ++rphase;
      // P^T buffer of tile n + j was last read by PV(n + j - 2).
      if (n >= 2 && !wait_pv(n - 2)) {
        ok = false;
        break;
      }
      if (cnt == 2 && n >= 1 && !wait_pv(n - 1)) {
        ok = false;
        break;
      }
      float alpha[G];
      bool any_rescale = false;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float tmax =
            fmaxf(fmaxf(rd[0 * kN + h], rd[1 * kN + h]), fmaxf(rd[2 * kN + h], rd[3 * kN + h]));
        alpha[h] = 1.f;
        if (seg_start) {
          m_used[h] = tmax;
        } else if (tmax > m_used[h] + kLazyRescale) {
          alpha[h] = exp2f(m_used[h] - tmax);
          m_used[h] = tmax;
          any_rescale = true;
        }
      }
      if (any_rescale) {
        // O^T holds the unit's tiles so far: wait for PV(n-1), scale row t.
        if (cnt == 1 && !wait_pv(n - 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float o[kN];
        tmem_ld16(lane_addr + kColO + (seg & 1) * kN, o);
#pragma unroll
        for (int h = 0; h < G; ++h) o[h] *= alpha[h];
        tmem_st16(lane_addr + kColO + (seg & 1) * kN, o);
#pragma unroll
        for (int h = 0; h < G; ++h) l_t[h] *= alpha[h];
      }
      // P^T row h, token t into buffer (n + j) & 1: bf16, or f16 for an FP8
      // cache (whose V^T is f16).  The row sums add the rounded weights the
      // MMA multiplies, so numerator and denominator of O / l use the same
      // weights (a consistent softmax; summing the fp32 values would leave a
      // 2^-9 relative mismatch per key).
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        if (j < cnt) {
          unsigned short pbits[G];
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float p = fast_exp2(s[j][h] - m_used[h]);
            if constexpr (kFp8) {
              const __half ph = __float2half_rn(p);
              pbits[h] = __half_as_ushort(ph);
              l_t[h] += __half2float(ph);
            } else {
              pbits[h] = __bfloat16_as_ushort(__float2bfloat16_rn(p));
              l_t[h] += __uint_as_float(static_cast<uint32_t>(pbits[h]) << 16);
            }
          }
          const uint32_t pbase =
              sbase + L::kOffP + ((n + j) & 1) * kSmallBytes + (t >> 6) * kSmallHalf;
          const int c = t & 63;
#pragma unroll
          for (int h = 0; h < kN; ++h) {
            const uint32_t addr = pbase + h * 128 + ((((c >> 3) ^ (h & 7))) << 4) + (c & 7) * 2;
            const unsigned short bits = h < G ? pbits[h < G ? h : 0] : 0;
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(bits) : "memory");
          }
        }
      }
      if (!kFp8 && nv_last < kTile) {
        // V rows of tokens past the context (only the unit's last tile, the
        // step's last): zero them before P V reads them, once V(nl) has
        // landed (the FP8 converters write them as zero).  PV(nl-2) is done,
        // hence V(nl-3) landed: this slot's barrier is at most one phase
        // behind.
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&v_full[nl % kVStages], (nl / kVStages) & 1, abort_flag, a.wait_ns))) {
          ok = false;
          break;
        }
        if (t >= nv_last) {
          const uint32_t vtile = sbase + L::kOffV + (nl % kVStages) * kTileBytes +
                                 (t >> 4) * kCacheTileBytes;
#pragma unroll
          for (int c = 0; c < 16; ++c) sts128(vtile + tile_chunk_offset(t & 15, c), 0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0)
        for (int j = 0; j < cnt; ++j) mbar_arrive(&p_full[(n + j) & 1]);

      if (seg_end) {
        // Hand the segment's per-head maximum and the four warps' row sums
        // to the epilogue warps (its O^T / l and the output or part are
        // theirs), once they have taken the segment two before out of this
        // slot.
        const int es = seg & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&epi_empty[es], ((seg >> 1) & 1) ^ 1, abort_flag,
                                               a.wait_ns))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float ws = warp_sum(l_t[h]);
          if (lane == 0) epi_l[(es * 4 + warp) * kN + h] = ws;
        }
        if (warp == 0 && lane == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) epi_m[es * kN + h] = m_used[h];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&epi_full[es]);
      }
      n += cnt;
      for (int j = 0; j < cnt; ++j) walk_next(sw, a, s_len);
    }
    if (t == 0) QATTN_STAMP(4);  // softmax done
    if (!ok && lane == 0) set_err(a.err_word, QATTN_DEVERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) QATTN_STAMP(5);  // CTA done
  if (warp == kMmaWarp) tmem_dealloc(tmem, L::kTmemCols);
}

template <int G, bool kFp8>
cudaError_t launch_tc_gf(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         const CUtensorMap& qmap, int num_sms, cudaStream_t stream,
                         cudaEvent_t merge_after) {
  using L = Lay<kFp8>;
  cudaError_t e = set_max_dynamic_smem(
      reinterpret_cast<const void*>(paged_decode_tc_kernel<G, kFp8>), L::kSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(paged_decode_tc_kernel<G, kFp8>, dim3(num_sms), dim3(L::kThreads),
                             L::kSmemBytes, stream, kmap, vmap, qmap, a);
  if (e != cudaSuccess) return e;
  e = cudaPeekAtLastError();
  if (e != cudaSuccess) return e;
  if (merge_after != nullptr) {  // parts that work on another stream writes
    e = cudaStreamWaitEvent(stream, merge_after, 0);
    if (e != cudaSuccess) return e;
  }
  return launch_decode_merge(a, stream);
}

template <int G>
cudaError_t launch_tc_g(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                        const CUtensorMap& qmap, int num_sms, cudaStream_t stream,
                        cudaEvent_t merge_after) {
  return a.kv_fp8 ? launch_tc_gf<G, true>(a, kmap, vmap, qmap, num_sms, stream, merge_after)
                  : launch_tc_gf<G, false>(a, kmap, vmap, qmap, num_sms, stream, merge_after);
}

}  // namespace

cudaError_t launch_paged_decode_tc(const DecodeArgs& a, const CUtensorMap& kmap,
                                   const CUtensorMap& vmap, const CUtensorMap& qmap, int num_sms,
                                   cudaStream_t stream, cudaEvent_t merge_after) {
  switch (a.num_heads / a.num_kv_heads) {
    case 1: return launch_tc_g<1>(a, kmap, vmap, qmap, num_sms, stream, merge_after);
    case 2: return launch_tc_g<2>(a, kmap, vmap, qmap, num_sms, stream, merge_after);
    case 3: return launch_tc_g<3>(a, kmap, vmap, qmap, num_sms, stream, merge_after);
    case 4: return launch_tc_g<4>(a, kmap, vmap, qmap, num_sms, stream, merge_after);
    case 5: return launch_tc_g<5>(a, kmap, vmap, qmap, num_sms, stream, merge_after);
    case 6: return launch_tc_g<6>(a, kmap, vmap, qmap, num_sms, stream, merge_after);
    case 7: return launch_tc_g<7>(a, kmap, vmap, qmap, num_sms, stream, merge_after);
    case 8: return launch_tc_g<8>(a, kmap, vmap, qmap, num_sms, stream, merge_after);
    default: return cudaErrorInvalidValue;
  }
}

#ifdef QATTN_TRACE
cudaError_t read_decode_trace(unsigned long long* host, size_t n) {
  return cudaMemcpyFromSymbol(host, g_qattn_decode_trace, n * sizeof(unsigned long long));
}
cudaError_t clear_decode_trace() {
  static unsigned long long zero[kTraceCtas * kTraceSlots];
  return cudaMemcpyToSymbol(g_qattn_decode_trace, zero, sizeof(zero));
}
#endif

}  // namespace qattn
