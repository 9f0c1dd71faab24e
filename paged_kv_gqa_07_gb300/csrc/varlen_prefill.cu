// Kernel K3: causal varlen / chunked prefill on tcgen05 tensor cores.
//
// What is computed: for a sequence b with q_len new tokens (rows
// cu_seqlens_q[b] ..) and context L (cached + new, already appended),
// query i sits at position L - q_len + i and attends keys 0 .. L - q_len + i
// of KV head h / G through the block table, with softmax scale
// head_dim ** -0.5 -- the FlashAttention-2 varlen causal attention of the Qwen
// engineering notes (0539edu.com) section 2.1 over the PagedAttention block
// cache (vLLM-deploys-Qwen notes section 2.1), chunked prefill mixing with
// decode rows as in continuous batching (same notes, section 2.1).
//
// Design (GB300): the prefill tiles are dense contractions, so they run on
// the 5th-generation tensor cores with the accumulators in tensor memory.
//   * Work: items (sequence, 128-row query tile, query head).  A persistent
//     grid of one CTA per SM; every CTA builds the same list of (sequence,
//     row tile) pairs, ranks them by KV tile count (largest first) and takes
//     items in a snake order over the ranked list, heads innermost (the G
//     heads of a KV group then run side by side and share the KV tiles in
//     L2).  Decode rows (one query) are left to the decode kernel.
//   * Warp roles: warp 8 copies Q of an item and its K tiles (eight 16-token
//     blocks gathered through the block table, one 4 KB TMA box per (block,
//     kv head), 128-byte swizzle) into a 2-deep ring; warp 10 copies the V
//     tiles into their own ring; one thread of warp 9 issues the Q K^T
//     stream (S into one of two TMEM S buffers) and one of warp 11 the P V
//     stream (O += P V into the item's TMEM O slot), each as soon as its
//     operands are ready -- two issuers, since a thread issuing tcgen05.mma
//     waits for the pipe to take each one; warps 0-7 do the
//     online softmax, two per TMEM lane quarter (rows 32q .. 32q + 31), one
//     per half of the 128 keys of a tile: S half-row from TMEM, causal mask
//     (only on tiles that cross the diagonal), half-row max swapped with the
//     partner warp through TMEM, exp2, P as bf16 into one of two
//     shared-memory P buffers (K-major, swizzled: the A operand of P V).
//     With two S, two P and two O slots, S(n+1) and P V(n) run on the tensor
//     cores while the softmax works on tile n, and an item's last P V and
//     epilogue overlap the next item's first tile.  The epilogue stages each
//     warp's bf16 output rows in the P buffer that last P V released, so
//     every store instruction writes whole 128-byte half-rows.
//   * O is rescaled lazily: the running max is only moved when the new max
//     exceeds it by more than 8 (log2 units), so most tiles skip the TMEM
//     round trip; P values stay <= 2^8, well inside bf16.
//   * Keys at or beyond L (the tail of the last block, unloaded blocks) are
//     masked in S and their V rows zeroed before P V, so stale cache contents
//     cannot leak in as 0 * NaN.
//   * Every wait is bounded; on a timeout all roles unwind, copies and
//     tensor-core work in flight are drained, TMEM is freed.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace qattn {
namespace {

constexpr int kM = 128;                 // query rows per tile
constexpr int kN = 128;                 // keys per KV tile
constexpr int kSoftmaxWarps = 8;        // two per TMEM lane quarter: column halves
constexpr int kProducerWarp = 8;        // Q and K copies
constexpr int kMmaWarp = 9;
constexpr int kVProducerWarp = 10;      // V copies
constexpr int kPvWarp = 11;             // issues the P V stream (warp 9: Q K^T)
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kHalfBytes = 128 * 128;   // 128 rows x 128 B (Q and P: [half][row])
constexpr int kTileBytes = 2 * kHalfBytes;
// A 128-token K/V tile lands as 8-token row groups 2 KB apart whatever the
// block size (each block's box is block_size / 8 groups); the V zeroing below
// addresses it in 16-token / 4 KB units.
constexpr int kCacheTileBytes = 16 * kHeadDim * 2;  // 16 tokens: 4 KB
constexpr uint32_t kTmemCols = 512;     // S[2] at 0 / 128, O[2] at 256 / 384
constexpr uint32_t kColO = 256;
constexpr float kLazyRescale = 8.0f;

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;          // 2 stages
constexpr int kOffV = kOffK + 2 * kTileBytes;      // 2 stages
constexpr int kOffP = kOffV + 2 * kTileBytes;      // 2 buffers
constexpr int kOffPairs = kOffP + 2 * kTileBytes;  // int[kPrefillMaxPairs], ranked
constexpr int kOffDesc = kOffPairs + kPrefillMaxPairs * 4;  // ItemDesc[2]
constexpr int kOffBars = kOffDesc + 2 * 64;
// q_full q_empty desc_full[2] desc_empty[2] k_full[2] k_empty[2] v_full[2]
// v_empty[2] s_full[2] s_free[2] p_full[2] pv_done[2] o_free[2] mma_done
// pair[4]
constexpr int kNumBars = 2 + 2 * 11 + 1 + 4;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 64 + 1024;
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct ItemDesc {
  int64_t row0;  // prefill: first query row of the tile
  int rows;      // valid rows (<= 128)
  int pos0;      // prefill: position of row 0 (row t sees keys <= pos0 + t)
  int nkv;       // KV tiles it attends
  int kt0;       // first of them (shared-prefix splits)
  int b;         // prefill: sequence; shared prefix: first sequence of the tile
  int h;         // prefill: query head; shared prefix: kv head
  int L;         // keys >= L do not exist
  int part;      // shared prefix: split index = part number in the workspace
  int causal;
};
static_assert(sizeof(ItemDesc) <= 64, "descriptor slot");

struct Misc {
  uint32_t tmem;
  int abort;
  int npairs;
  int nitems;
  int warp_sums[kWarps];
};

__device__ __forceinline__ bool prefill_ctx_ok(const PrefillArgs& a, int L, int ql) {
  return L >= ql && L <= a.max_context_len && L <= a.max_blocks_per_seq * a.block_size;
}

// Inclusive scan over the CTA's threads.
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
    int w = lane < kWarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kWarps) warp_sums[lane] = w;
  }
  __syncthreads();
  const int add = warp > 0 ? warp_sums[warp - 1] : 0;
  *block_total = warp_sums[kWarps - 1];
  __syncthreads();
  return v + add;
}

// Item r of this CTA: index into the ranked (pair, head) list, snake order.
__device__ __forceinline__ int item_index(int r) {
  const int P = gridDim.x, k = blockIdx.x;
  return r * P + ((r & 1) ? (P - 1 - k) : k);
}

// 12 warps: 3 on each of the four SM sub-partitions, so at most 168
// registers a thread.
__global__ void __launch_bounds__(kThreads, 1)
    varlen_prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                          const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* desc_full = bars + 2;
  uint64_t* desc_empty = bars + 4;
  uint64_t* k_full = bars + 6;
  uint64_t* k_empty = bars + 8;
  uint64_t* v_full = bars + 10;
  uint64_t* v_empty = bars + 12;
  uint64_t* s_full = bars + 14;
  uint64_t* s_free = bars + 16;
  uint64_t* p_full = bars + 18;
  uint64_t* pv_done = bars + 20;  // PV(n) completes phase n >> 1 of pv_done[n & 1]
  uint64_t* o_free = bars + 22;   // the softmax has read O slot r & 1 of item r
  uint64_t* mma_done = bars + 24;
  // pair[q]: the two softmax warps of lane quarter q have swapped their
  // partial row statistics (one phase per KV tile, plus one at the end)
  uint64_t* pair = bars + 25;
  Misc* misc = reinterpret_cast<Misc*>(smem + kOffMisc);
  ItemDesc* desc = reinterpret_cast<ItemDesc*>(smem + kOffDesc);
  int* pairs = reinterpret_cast<int*>(smem + kOffPairs);
  volatile int* abort_flag = &misc->abort;
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.num_seqs, H = a.num_heads;
  const int G = H / a.num_kv_heads;

  const bool prefix_mode = a.prefix_len > 0;
  // Shared-prefix pass: rows of a tile are (sequence, head of the group)
  // pairs, R sequences a tile; items (kv head, split, row tile).
  const int R = kM / G;
  const int MT = (B + R - 1) / R;
  const int TP = (a.prefix_len + kN - 1) / kN;  // prefix KV tiles
  const int S = a.prefix_splits;

  // ---- plan: the (sequence, row tile) pairs, ranked by KV tiles ----
  // (scratch for the unranked list: the P buffers, unused until the loop)
  int* sp = reinterpret_cast<int*>(smem + kOffP);
  int* sc = sp + kPrefillMaxPairs;
  int running = 0;
  for (int base = 0; base < B && !prefix_mode; base += kThreads) {
    const int b = base + tid;
    int np = 0, ql = 0, L = 0;
    if (b < B) {
      ql = a.cu_seqlens_q[b + 1] - a.cu_seqlens_q[b];
      L = a.context_lens[b];
      if (ql >= 2 && prefill_ctx_ok(a, L, ql)) np = (ql + kM - 1) / kM;
    }
    int tot;
    const int incl = block_scan(np, misc->warp_sums, &tot);
    for (int mt = 0; mt < np; ++mt) {
      const int idx = running + incl - np + mt;
      if (idx < kPrefillMaxPairs) {
        const int rows = min(kM, ql - mt * kM);
        const int pos0 = L - ql + mt * kM;
        sp[idx] = (b << 11) | mt;
        sc[idx] = (pos0 + rows - 1) / kN + 1;
      }
    }
    running += tot;
  }
  __syncthreads();
  const int NP = min(running, kPrefillMaxPairs);
  if (running > kPrefillMaxPairs && blockIdx.x == 0 && tid == 0)
    set_err(a.err_word, QATTN_DEVERR_CONTEXT);
  for (int i = tid; i < NP && !prefix_mode; i += kThreads) {
    const int ci = sc[i];
    int rank = 0;
    for (int j = 0; j < NP; ++j) {
      const int cj = sc[j];
      rank += (cj > ci || (cj == ci && j < i)) ? 1 : 0;
    }
    pairs[rank] = sp[i];
  }
  if (tid == 0) {
    const int NI = prefix_mode ? a.num_kv_heads * S * MT : NP * H;
    int n = 0;
    while (item_index(n) < NI) ++n;
    misc->nitems = n;
    misc->abort = 0;
  }
  __syncthreads();

  if (prefix_mode) {
    // Every sequence's table must start with row 0's prefix blocks.
    const int nb = a.prefix_len / a.block_size;
    const int64_t pairs_total = static_cast<int64_t>(B - 1) * nb;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + tid; i < pairs_total;
         i += static_cast<int64_t>(gridDim.x) * kThreads) {
      const int b = 1 + static_cast<int>(i / nb), j = static_cast<int>(i % nb);
      if (a.block_tables[static_cast<int64_t>(b) * a.max_blocks_per_seq + j] != a.block_tables[j])
        set_err(a.err_word, QATTN_DEVERR_PREFIX);
    }
  }
  // Prefill sequences with an invalid context: zero rows and the CONTEXT bit.
  for (int b = blockIdx.x; b < B && !prefix_mode; b += gridDim.x) {
    const int q0 = a.cu_seqlens_q[b];
    const int ql = a.cu_seqlens_q[b + 1] - q0;
    if (ql < 2 || prefill_ctx_ok(a, a.context_lens[b], ql)) continue;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                          static_cast<int64_t>(q0) * H * kHeadDim);
    for (int64_t i = tid; i < static_cast<int64_t>(ql) * H * (kHeadDim / 8); i += kThreads)
      dst[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) set_err(a.err_word, QATTN_DEVERR_CONTEXT);
  }
  const int nitems = misc->nitems;
  if (nitems == 0) return;  // no barrier, copy or TMEM in use yet

  // ---- set-up: barriers, TMEM ----
  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&desc_full[s], 1);
      mbar_init(&desc_empty[s], 2 + kSoftmaxWarps);  // the two MMA threads, the softmax warps
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], kSoftmaxWarps);
      mbar_init(&p_full[s], kSoftmaxWarps);
      mbar_init(&pv_done[s], 1);
      mbar_init(&o_free[s], kSoftmaxWarps);
    }
    mbar_init(mma_done, 2);
    for (int q = 0; q < 4; ++q) mbar_init(&pair[q], 2);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&misc->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem;

  if (warp == kProducerWarp || warp == kVProducerWarp) {
    // =============================== producers ================================
    // Warp 8 writes the item descriptors and copies Q and the K tiles; warp
    // 10 copies the V tiles on its own, so a K copy never waits behind a V
    // ring slot (V slots free only after P V, one tile after K slots).
    const bool is_v = warp == kVProducerWarp;
    uint64_t* full = is_v ? v_full : k_full;
    uint64_t* empty = is_v ? v_empty : k_empty;
    const CUtensorMap* map = is_v ? &vmap : &kmap;
    uint8_t* ring = smem + (is_v ? kOffV : kOffK);
    const int bpt = 128 / a.block_size;   // cache blocks per tile: 8, 4 or 2
    const int groups = a.block_size / 8;  // 8-row groups per block box
    const uint32_t blk_bytes = static_cast<uint32_t>(a.block_size) * kHeadDim * 2;
    if (lane == 0) {
      tma_prefetch_desc(map);
      if (!is_v) tma_prefetch_desc(&qmap);
    }
    int n = 0;       // tiles whose copies were issued (all items)
    int qn = 0;      // Q copies issued
    bool ok = true;
    for (int r = 0; r < nitems && ok; ++r) {
      const int idx = item_index(r);
      int b, mt, h, g, L, rows, pos0, nkv, kt0 = 0, part = 0;
      int64_t row0 = 0;
      if (prefix_mode) {
        // item = ((g * S + split) * MT + mt): row tiles of one (kv head,
        // split) run side by side and share its KV tiles in L2
        mt = idx % MT;
        part = (idx / MT) % S;
        g = idx / (MT * S);
        h = g;
        b = mt * R;
        L = a.prefix_len;
        rows = min(R, B - b) * G;
        pos0 = 0;
        kt0 = static_cast<int>(static_cast<int64_t>(part) * TP / S);
        nkv = static_cast<int>(static_cast<int64_t>(part + 1) * TP / S) - kt0;
      } else {
        const int pr = pairs[idx / H];
        b = pr >> 11;
        mt = pr & 2047;
        h = idx % H;
        g = h / G;
        const int q0 = a.cu_seqlens_q[b];
        const int ql = a.cu_seqlens_q[b + 1] - q0;
        L = a.context_lens[b];
        rows = min(kM, ql - mt * kM);
        pos0 = L - ql + mt * kM;
        nkv = (pos0 + rows - 1) / kN + 1;
        row0 = static_cast<int64_t>(q0) + mt * kM;
      }
      if (!is_v && lane == 0) {
        // descriptor slot r & 1 was last read for item r - 2
        ok = r < 2 || mbar_wait(&desc_empty[r & 1], ((r >> 1) & 1) ^ 1, abort_flag);
        if (ok) {
          ItemDesc& d = desc[r & 1];
          d.row0 = row0;
          d.rows = rows;
          d.pos0 = pos0;
          d.nkv = nkv;
          d.kt0 = kt0;
          d.b = b;
          d.h = h;
          d.L = L;
          d.part = part;
          d.causal = prefix_mode ? 0 : 1;
          mbar_arrive(&desc_full[r & 1]);
        }
        // Q buffer: the previous item's last Q K^T is done
        ok = ok && (r == 0 || mbar_wait(q_empty, (r - 1) & 1, abort_flag));
        if (ok && prefix_mode) {
          // R sequences x the G heads of kv head g: rows (sequence, head),
          // 128 B each; rows past the batch read as zeros
          mbar_arrive_expect_tx(q_full, 2 * 128 * R * G);
          tma_load_3d(smem + kOffQ, &qmap, 0, g * G, b, q_full);
          tma_load_3d(smem + kOffQ + kHalfBytes, &qmap, 64, g * G, b, q_full);
          ++qn;
        } else if (ok) {
          mbar_arrive_expect_tx(q_full, kTileBytes);
          tma_load_2d(smem + kOffQ, &qmap, h * kHeadDim, static_cast<int32_t>(row0), q_full);
          tma_load_2d(smem + kOffQ + kHalfBytes, &qmap, h * kHeadDim + 64,
                      static_cast<int32_t>(row0), q_full);
          ++qn;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      // the shared prefix lives in the blocks of table row 0
      const int* bt = a.block_tables + (prefix_mode ? 0 : static_cast<int64_t>(b) * a.max_blocks_per_seq);
      const int nblk = (L + a.block_size - 1) / a.block_size;
      for (int kt = 0; kt < nkv && ok; ++kt) {
        const int st = n & 1;
        int id = -1;
        if (lane < bpt) {
          const int bi = (kt0 + kt) * bpt + lane;
          if (bi < nblk) {
            id = bt[bi];
            if (id < 0 || id >= a.num_blocks) {
              if (!is_v) set_err(a.err_word, QATTN_DEVERR_BLOCK);
              id = -1;
            }
          }
        }
        const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, id >= 0));
        if (lane == 0) {
          ok = n < 2 || mbar_wait(&empty[st], ((n >> 1) & 1) ^ 1, abort_flag);
          if (ok) mbar_arrive_expect_tx(&full[st], nvalid * blk_bytes);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (id >= 0)
          tma_load_cache_tile(ring + st * kTileBytes + lane * blk_bytes, map,
                              id * a.num_kv_heads + g, groups, &full[st]);
        ++n;
      }
    }
    // Drain: the copies of the last (up to two) tiles and of the last Q land
    // before the CTA exits.
    if (lane == 0) {
      for (int j = n - 1; j >= 0 && j >= n - 2; --j) mbar_wait_drain(&full[j & 1], (j >> 1) & 1);
      if (qn > 0) mbar_wait_drain(q_full, (qn - 1) & 1);
      if (*abort_flag) set_err(a.err_word, QATTN_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ============================= MMA issuers ===============================
    // Warp 9 issues the Q K^T stream and warp 11 the P V stream: a thread
    // issuing tcgen05.mma waits for the tensor pipe to take each one (~85
    // cycles for 128 x 128 x 16), so with one issuer a ready Q K^T waited
    // behind a tile's P V and the other way round.  The streams share no
    // tensor memory (S vs O) and each thread's commits track its own MMAs.
    if (lane == 0) {
      bool ok = true;
      uint64_t idle_since = 0;
      // No progress for kWaitTimeoutNs (or the abort flag): give up.
      auto idle = [&](bool progressed) {
        if (progressed) {
          idle_since = 0;
        } else {
          const uint64_t now = globaltimer_ns();
          if (idle_since == 0) {
            idle_since = now;
          } else if (*abort_flag || now - idle_since > kWaitTimeoutNs) {
            *abort_flag = 1;
            ok = false;
          }
        }
      };
      if (warp == kMmaWarp) {
        constexpr uint32_t idesc_qk = idesc_bf16_f32(kM, kN, false);
        const uint32_t sq = sbase + kOffQ;
        int qr = 0, qkt = 0, q_nkv = 0;  // item, its tile, its length
        int qn = 0;                      // KV tiles so far
        while (qr < nitems && ok) {
          bool progressed = false;
          if (q_nkv == 0 && mbar_test(&desc_full[qr & 1], (qr >> 1) & 1)) {
            q_nkv = desc[qr & 1].nkv;
            mbar_arrive(&desc_empty[qr & 1]);
            progressed = true;
          }
          if (q_nkv > 0) {
            bool ready = mbar_test(&k_full[qn & 1], (qn >> 1) & 1);
            if (ready && qn >= 2) ready = mbar_test(&s_free[qn & 1], ((qn >> 1) & 1) ^ 1);
            if (ready && qkt == 0) ready = mbar_test(q_full, qr & 1);
            if (ready) {
              tc_fence_after();
              const uint32_t sk = sbase + kOffK + (qn & 1) * kTileBytes;
              // (both MMA loops unrolled by 4: measured 0-1.4 % faster than 8)
#pragma unroll 4
              for (int k = 0; k < kHeadDim / 16; ++k) {
                const uint64_t ad =
                    sdesc_sw128(sq + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024);
                // K tile as the K-major B: dim half k/4 at +1 KB, 8-key groups 2 KB apart.
                const uint64_t bd = sdesc_sw128(sk + (k >> 2) * 1024 + (k & 3) * 32, 16, 2048);
                mma_bf16_ss(tmem + (qn & 1) * kN, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
              }
              mma_commit(&s_full[qn & 1]);
              mma_commit(&k_empty[qn & 1]);
              if (qkt == q_nkv - 1) mma_commit(q_empty);
              ++qn;
              if (++qkt == q_nkv) {
                qkt = 0;
                q_nkv = 0;
                ++qr;
              }
              progressed = true;
            }
          }
          idle(progressed);
        }
      } else {
        constexpr uint32_t idesc_pv = idesc_bf16_f32(kM, kHeadDim, true);
        int pr = 0, pkt = 0, p_nkv = 0;  // item, its tile, its length
        int pn = 0;                      // KV tiles so far
        while (pr < nitems && ok) {
          bool progressed = false;
          if (p_nkv == 0 && mbar_test(&desc_full[pr & 1], (pr >> 1) & 1)) {
            p_nkv = desc[pr & 1].nkv;
            mbar_arrive(&desc_empty[pr & 1]);
            progressed = true;
          }
          if (p_nkv > 0) {
            const bool first = pkt == 0;
            bool ready = mbar_test(&p_full[pn & 1], (pn >> 1) & 1) &&
                         mbar_test(&v_full[pn & 1], (pn >> 1) & 1);
            // an item's first P V overwrites O slot pr & 1, last read for item pr - 2
            if (ready && first && pr >= 2) ready = mbar_test(&o_free[pr & 1], ((pr >> 1) - 1) & 1);
            if (ready) {
              tc_fence_after();
              const uint32_t sv = sbase + kOffV + (pn & 1) * kTileBytes;
              const uint32_t sp_ = sbase + kOffP + (pn & 1) * kTileBytes;
#pragma unroll 4
              for (int k = 0; k < kN / 16; ++k) {
                const uint64_t ad =
                    sdesc_sw128(sp_ + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024);
                // V tile as the MN-major B: dim halves 1 KB apart (LBO), 8-key
                // groups 2 KB apart (SBO); K step k = keys 16k..16k+15.
                const uint64_t bd = sdesc_sw128(sv + k * 4096, 1024, 2048);
                mma_bf16_ss(tmem + kColO + (pr & 1) * kHeadDim, ad, bd, idesc_pv,
                            (first && k == 0) ? 0u : 1u);
              }
              mma_commit(&pv_done[pn & 1]);
              mma_commit(&v_empty[pn & 1]);
              ++pn;
              if (++pkt == p_nkv) {
                pkt = 0;
                p_nkv = 0;
                ++pr;
              }
              progressed = true;
            }
          }
          idle(progressed);
        }
      }
      // Drain: every MMA of both threads completes before TMEM is released.
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
    __syncwarp();
  } else {
    // =============================== softmax ================================
    // Warp w owns TMEM lane quarter w & 3 (query rows t) and column half
    // hf = w >> 2: keys 64 hf .. 64 hf + 63 of every S tile, P columns of
    // that half, O dims of that half.  The two warps of a quarter swap their
    // half-row max (and, at an item's end, half-row sums) through two spare
    // TMEM columns of the S buffer they both just read.
    const int q4 = warp & 3, hf = warp >> 2;
    const int t = q4 * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    auto wait_pv = [&](int j) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(&pv_done[j & 1], (j >> 1) & 1, abort_flag));
    };
    // Swap (a, b) with the partner warp through TMEM columns `col` (own
    // half) / `col` of the other half; phase `ph` of the pair barrier.
    auto swap2 = [&](uint32_t col_base, int ph, float a, float b, float& pa, float& pb) -> bool {
      tmem_st2(lane_addr + col_base + 64 * hf, a, b);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pair[q4]);
      if (!__all_sync(0xffffffffu, mbar_wait(&pair[q4], ph & 1, abort_flag))) return false;
      tc_fence_after();
      tmem_ld2(lane_addr + col_base + 64 * (1 - hf), pa, pb);
      return true;
    };
    // Epilogue of item pr (last tile pn, row sum l): this half's O dims / l.
    // Epilogue of item pr (last tile pn, row max m and sum l): this half's O
    // dims / l -- bf16 output rows (prefill), or the item's split-KV part
    // (normalised O, log2-sum-exp) of each (sequence, head) row (shared
    // prefix).
    struct Pending {
      int64_t row0;
      int rows, h, b, part, n, r;
      float m, l;
    };
    auto finish = [&](const Pending& pd, float l) -> bool {
      if (!wait_pv(pd.n)) return false;
      tc_fence_after();
      const float inv = a.out_scale / l;
      const bool valid = t < pd.rows;
      const uint32_t col = kColO + (pd.r & 1) * kHeadDim + 64 * hf;
      if (prefix_mode) {
        const int j = t % G;
        const int64_t seg = static_cast<int64_t>(pd.b + t / G) * a.num_kv_heads + pd.h;
        const int64_t pidx = seg * a.ws.max_parts + pd.part;
        float* optr = a.ws.part_o + (pidx * G + j) * kHeadDim + 64 * hf;
#pragma unroll 1
        for (int c4 = 0; c4 < 2; ++c4) {
          float o[32];
          tmem_ld32(lane_addr + col + c4 * 32, o);
          if (valid) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<float4*>(optr + c4 * 32 + q * 4) =
                  make_float4(o[q * 4] * inv, o[q * 4 + 1] * inv, o[q * 4 + 2] * inv,
                              o[q * 4 + 3] * inv);
          }
        }
        if (valid && hf == 0) a.ws.lse[pidx * G + j] = pd.m + log2f(l);
      } else {
        // The bf16 half-rows go through this warp's 4 KB of the P buffer
        // that P V(pd.n) has released (the rows it writes P into; swizzled
        // like P), then out four whole 128-byte half-rows per store
        // instruction: written straight from the TMEM lanes, every store
        // touched 32 rows 7 KB apart.
        const uint32_t stage =
            sbase + kOffP + (pd.n & 1) * kTileBytes + hf * kHalfBytes + q4 * 32 * 128;
#pragma unroll 1
        for (int c4 = 0; c4 < 2; ++c4) {
          float o[32];
          tmem_ld32(lane_addr + col + c4 * 32, o);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            sts128(stage + lane * 128 + (((c4 * 4 + q) ^ (lane & 7)) << 4),
                   pack_bf16x2_rn(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv),
                   pack_bf16x2_rn(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv),
                   pack_bf16x2_rn(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv),
                   pack_bf16x2_rn(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv));
        }
        __syncwarp();
        const int cc = lane & 7;
#pragma unroll 4
        for (int i = 0; i < 8; ++i) {
          const int rr = i * 4 + (lane >> 3);  // row q4 * 32 + rr of the tile
          const uint4 v = lds128(stage + rr * 128 + ((cc ^ (rr & 7)) << 4));
          if (q4 * 32 + rr < pd.rows)
            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                      ((pd.row0 + q4 * 32 + rr) * H + pd.h) * kHeadDim +
                                      64 * hf + cc * 8) = v;
        }
        __syncwarp();  // the staging rows are P rows again from here
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[pd.r & 1]);
      return true;
    };
    bool pend = false;
    Pending pending{};  // pending.l: this half's row sum of the pending item
    int n = 0;  // KV tiles consumed (all items) = pair barrier phases so far
    bool ok = true;
    for (int r = 0; r < nitems && ok; ++r) {
      if (!__all_sync(0xffffffffu, mbar_wait(&desc_full[r & 1], (r >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      const int64_t d_row0 = desc[r & 1].row0;
      const int d_rows = desc[r & 1].rows, d_h = desc[r & 1].h;
      const int d_nkv = desc[r & 1].nkv, d_L = desc[r & 1].L;
      const int d_kt0 = desc[r & 1].kt0, d_b = desc[r & 1].b, d_part = desc[r & 1].part;
      // keys <= key_lim are visible
      const int key_lim = desc[r & 1].causal ? (t < d_rows ? desc[r & 1].pos0 + t : 0) : d_L - 1;
      __syncwarp();
      if (lane == 0) mbar_arrive(&desc_empty[r & 1]);
      const uint32_t o_col = kColO + (r & 1) * kHeadDim + 64 * hf;  // this item's O, my dims
      float m_run = -INFINITY, l_run = 0.f;
      for (int kt = 0; kt < d_nkv; ++kt, ++n) {
        const int sb = n & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (n >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        float s[64];
        tmem_ld64(lane_addr + sb * kN + 64 * hf, s);

        // Half-row max of the raw scores (scale > 0 commutes with max), eight
        // accumulators; keys past the causal limit are -inf.
        const int kbase = (d_kt0 + kt) * kN + 64 * hf;
        if (kbase + 63 > key_lim) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (kbase + c > key_lim) s[c] = -INFINITY;
        }
        float mx8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(s[i], s[56 + i]);
#pragma unroll
        for (int c = 8; c < 56; c += 16) {
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + 8 + i]);
        }
        const float mh = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                               fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
        float mh2, lp2;
        if (!swap2(sb * kN, n, mh, pend ? pending.l : 0.f, mh2, lp2)) {
          ok = false;
          break;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[sb]);
        const float mx = fmaxf(mh, mh2) * a.scale_log2;

        // P buffer sb was last read by PV(n-2).
        if (n >= 2 && !wait_pv(n - 2)) {
          ok = false;
          break;
        }
        if (kt == 0) {
          m_run = mx;
        } else {
          const bool rescale = mx > m_run + kLazyRescale;
          if (__any_sync(0xffffffffu, rescale)) {
            // O holds the item's tiles so far: wait for PV(n-1), scale my dims.
            if (!wait_pv(n - 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const float alpha = rescale ? exp2f(m_run - mx) : 1.f;
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
              float o[16];
              tmem_ld16(lane_addr + o_col + c4 * 16, o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] *= alpha;
              tmem_st16(lane_addr + o_col + c4 * 16, o);
            }
            if (rescale) {
              l_run *= alpha;
              m_run = mx;
            }
          }
        }
        // p = 2^(scale_log2 * s - m): one FMA (packed two at a time) and one
        // exp2 per score; eight partial sums (packed adds); P half hf of row
        // t, swizzled K-major.
        float2 sum2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sum2[i] = make_float2(0.f, 0.f);
        const uint32_t sp_row = sbase + kOffP + sb * kTileBytes + hf * kHalfBytes + t * 128;
        const float2 scale2 = make_float2(a.scale_log2, a.scale_log2);
        const float2 neg_m2 = make_float2(-m_run, -m_run);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          float p[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 x =
                __ffma2_rn(make_float2(s[cc * 8 + 2 * i], s[cc * 8 + 2 * i + 1]), scale2, neg_m2);
            p[2 * i] = fast_exp2(x.x);
            p[2 * i + 1] = fast_exp2(x.y);
            sum2[i] = __fadd2_rn(sum2[i], make_float2(p[2 * i], p[2 * i + 1]));
          }
          sts128(sp_row + ((cc ^ (t & 7)) << 4), pack_bf16x2_rn(p[0], p[1]),
                 pack_bf16x2_rn(p[2], p[3]), pack_bf16x2_rn(p[4], p[5]),
                 pack_bf16x2_rn(p[6], p[7]));
        }
        l_run += ((sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y)) +
                 ((sum2[2].x + sum2[2].y) + (sum2[3].x + sum2[3].y));
        if ((d_kt0 + kt) * kN + kN > d_L) {
          // The tile reaches past the context: zero V rows of keys >= L once
          // V(n) has landed (PV(n-2) is done, so this barrier is at most one
          // phase behind); this warp zeroes its half of each such row.
          if (!__all_sync(0xffffffffu, mbar_wait(&v_full[sb], (n >> 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          if ((d_kt0 + kt) * kN + t >= d_L) {
            const uint32_t vtile = sbase + kOffV + sb * kTileBytes + (t >> 4) * kCacheTileBytes;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              sts128(vtile + tile_chunk_offset(t & 15, 8 * hf + c), 0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
        if (pend) {  // the previous item ended at tile n - 1; its sums came with the swap
          if (!finish(pending, pending.l + lp2)) {
            ok = false;
            break;
          }
          pend = false;
        }
      }
      if (!ok) break;
      // The item's epilogue waits for its last P V: it runs after the next
      // item's first tile (O has a slot per item parity).
      pend = true;
      pending.row0 = d_row0;
      pending.rows = d_rows;
      pending.h = d_h;
      pending.b = d_b;
      pending.part = d_part;
      pending.m = m_run;
      pending.l = l_run;
      pending.n = n - 1;
      pending.r = r;
    }
    if (ok && pend) {
      // The last item: swap the half-row sums through S buffer 0 (no Q K^T
      // is left to write it), then its epilogue.
      float unused, lp2;
      ok = swap2(0, n, 0.f, pending.l, unused, lp2) && finish(pending, pending.l + lp2);
    }
    if (!ok && lane == 0) set_err(a.err_word, QATTN_DEVERR_TIMEOUT);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// The queries [total_q][q_row_stride] seen as a 2-D tensor of total_q rows by
// num_heads * 128 columns; a box is 128 rows x 64 columns (one half of one
// head's 128-row tile), 128-byte swizzled.
bool encode_q_map(CUtensorMap* map, const void* q, int64_t q_row_stride, int total_q,
                  int num_heads) {
  const EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(num_heads) * kHeadDim,
                              static_cast<cuuint64_t>(total_q)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(q_row_stride) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kM)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {
cudaError_t set_smem_attr() {
  return set_max_dynamic_smem(reinterpret_cast<const void*>(varlen_prefill_kernel), kSmemBytes);
}
}  // namespace

cudaError_t launch_shared_prefix(const PrefillArgs& a, const CUtensorMap& qmap,
                                 const CUtensorMap& kmap, const CUtensorMap& vmap, int num_sms,
                                 cudaStream_t stream) {
  cudaError_t e = set_smem_attr();
  if (e != cudaSuccess) return e;
  const int G = a.num_heads / a.num_kv_heads;
  const int R = kM / G;
  const int64_t items =
      static_cast<int64_t>(a.num_kv_heads) * a.prefix_splits * ((a.num_seqs + R - 1) / R);
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  varlen_prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, a);
  return cudaPeekAtLastError();
}

cudaError_t launch_varlen_prefill(const PrefillArgs& a, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, int num_sms, cudaStream_t stream) {
  cudaError_t es = set_smem_attr();
  if (es != cudaSuccess) return es;
  CUtensorMap qmap;
  if (!encode_q_map(&qmap, a.q, a.q_row_stride, a.total_q, a.num_heads))
    return cudaErrorInvalidValue;
  // A launch plans at most kPrefillMaxPairs (sequence, 128-row tile) pairs:
  // batches of sequences keep every launch within that.
  const int tiles_per_seq = (a.max_q_len + kM - 1) / kM;
  if (tiles_per_seq > kPrefillMaxPairs) return cudaErrorNotSupported;
  const int batch = kPrefillMaxPairs / tiles_per_seq;
  for (int s0 = 0; s0 < a.num_seqs; s0 += batch) {
    PrefillArgs p = a;
    p.num_seqs = a.num_seqs - s0 < batch ? a.num_seqs - s0 : batch;
    p.cu_seqlens_q = a.cu_seqlens_q + s0;
    p.context_lens = a.context_lens + s0;
    p.block_tables = a.block_tables + static_cast<int64_t>(s0) * a.max_blocks_per_seq;
    varlen_prefill_kernel<<<num_sms, kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, p);
    const cudaError_t e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace qattn
