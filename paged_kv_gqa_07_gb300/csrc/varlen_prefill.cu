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
//   * One CTA = one (sequence, query head, 128-row query tile).  Rows are
//     query tokens; the K/V tiles are 128 keys = eight 16-token blocks,
//     gathered through the block table with 2-D TMA (16 x 64 boxes, 128-byte
//     swizzle) into [d-half][key][64] shared-memory tiles -- exactly the
//     K-major layout tcgen05 reads for B of S = Q K^T and the MN-major layout
//     it reads for B of O = P V, so no data is re-laid.
//   * Warp roles: warp 4 issues TMA (Q once, then K and V per tile through a
//     2-stage ring), one thread of warp 5 issues tcgen05.mma (S = Q K^T into
//     one of two 128-column S buffers in TMEM, O += P V into a third), warps
//     0-3 own TMEM lanes 0-127 = the 128 query rows and do the online softmax:
//     S row from TMEM, causal mask (only on tiles that cross the diagonal),
//     row max, exp2, P written as bf16 into shared memory in the swizzled
//     K-major layout.  S(kt+1) is computed while softmax(kt) runs.
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
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = 6 * 32;
constexpr int kHalfBytes = 128 * 128;   // 128 rows x 128 B (Q and P: [half][row])
constexpr int kTileBytes = 2 * kHalfBytes;
constexpr int kCacheTileBytes = kBlockSize * kHeadDim * 2;  // one (block, kv head): 4 KB
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;
constexpr float kLazyRescale = 8.0f;

constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffP = kOffV + kStages * kTileBytes;
constexpr int kOffBars = kOffP + kTileBytes;
// barriers: q_full, k_full[2], v_full[2], kv_empty[2], s_full[2], s_free[2],
//           p_full, o_done, mma_done
constexpr int kNumBars = 14;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;

__device__ __forceinline__ void zero_rows(const PrefillArgs& a, int64_t row0, int rows, int h) {
  for (int i = threadIdx.x; i < rows * (kHeadDim / 8); i += blockDim.x) {
    const int r = i / (kHeadDim / 8), c = i % (kHeadDim / 8);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                              ((row0 + r) * a.num_heads + h) * kHeadDim + c * 8) =
        make_uint4(0, 0, 0, 0);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    varlen_prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                          const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  const int mt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int q0 = a.cu_seqlens_q[b];
  const int q_len = a.cu_seqlens_q[b + 1] - q0;
  if (q_len < 2 || mt * kM >= q_len) return;  // decode rows take the decode kernel
  const int L = a.context_lens[b];
  const int rows = min(kM, q_len - mt * kM);
  const int64_t row0 = static_cast<int64_t>(q0) + mt * kM;
  const int G = a.num_heads / a.num_kv_heads;
  const int g = h / G;
  if (L < q_len || L > a.max_context_len || L > a.max_blocks_per_seq * kBlockSize) {
    zero_rows(a, row0, rows, h);
    if (tid == 0 && h == 0 && mt == 0) set_err(a.err_word, QATTN_DEVERR_CONTEXT);
    return;
  }
  const int pos0 = L - q_len + mt * kM;  // position of tile row 0
  const int n_kv = (pos0 + rows - 1) / kN + 1;
  const int nblk = (L + kBlockSize - 1) / kBlockSize;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* q_full = bars + 0;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = bars + 3;
  uint64_t* kv_empty = bars + 5;
  uint64_t* s_full = bars + 7;
  uint64_t* s_free = bars + 9;
  uint64_t* p_full = bars + 11;
  uint64_t* o_done = bars + 12;
  uint64_t* mma_done = bars + 13;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const uint32_t sbase = smem_u32(smem);

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], 4);
    }
    mbar_init(p_full, 4);
    mbar_init(o_done, 1);
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp) {
    // ================================ producer ================================
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_2d(smem + kOffQ, &qmap, h * kHeadDim, static_cast<int32_t>(row0), q_full);
      tma_load_2d(smem + kOffQ + kHalfBytes, &qmap, h * kHeadDim + 64,
                  static_cast<int32_t>(row0), q_full);
    }
    const int* bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
    int issued = 0;
    bool ok = true;
    for (int kt = 0; kt < n_kv; ++kt) {
      const int st = kt & 1;
      int id = -1;
      if (lane < 8) {
        const int bi = kt * 8 + lane;
        if (bi < nblk) {
          id = bt[bi];
          if (id < 0 || id >= a.num_blocks) {
            set_err(a.err_word, QATTN_DEVERR_BLOCK);
            id = -1;
          }
        }
      }
      const int nvalid = __popc(__ballot_sync(0xffffffffu, id >= 0));
      if (lane == 0 && kt >= kStages)
        ok = mbar_wait(&kv_empty[st], ((kt >> 1) & 1) ^ 1, abort_flag);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      uint8_t* kdst = smem + kOffK + st * kTileBytes + lane * kCacheTileBytes;
      uint8_t* vdst = smem + kOffV + st * kTileBytes + lane * kCacheTileBytes;
      if (lane == 0) mbar_arrive_expect_tx(&k_full[st], nvalid * 2 * kBlockSize * 128);
      __syncwarp();
      if (id >= 0) {
        tma_load_cache_tile(kdst, &kmap, id * a.num_kv_heads + g, &k_full[st]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&v_full[st], nvalid * 2 * kBlockSize * 128);
      __syncwarp();
      if (id >= 0) {
        tma_load_cache_tile(vdst, &vmap, id * a.num_kv_heads + g, &v_full[st]);
      }
      ++issued;
    }
    // Drain: the copies of the last (up to two) issued tiles and of Q.
    if (lane == 0) {
      for (int j = issued - 1; j >= 0 && j >= issued - kStages; --j) {
        mbar_wait_drain(&k_full[j & 1], (j >> 1) & 1);
        mbar_wait_drain(&v_full[j & 1], (j >> 1) & 1);
      }
      mbar_wait_drain(q_full, 0);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ============================== MMA issuer ===============================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(kM, kN, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(kM, kHeadDim, true);
      const uint32_t sq = sbase + kOffQ, sp = sbase + kOffP;
      bool ok = mbar_wait(q_full, 0, abort_flag);
      auto issue_pv = [&](int j) {
        ok = ok && mbar_wait(p_full, j & 1, abort_flag);
        ok = ok && mbar_wait(&v_full[j & 1], (j >> 1) & 1, abort_flag);
        if (!ok) return;
        tc_fence_after();
        const uint32_t sv = sbase + kOffV + (j & 1) * kTileBytes;
#pragma unroll
        for (int k = 0; k < kN / 16; ++k) {
          const uint64_t ad = sdesc_sw128(sp + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024);
          // V tile as the MN-major B: dim halves 1 KB apart (LBO), 8-key
          // groups 2 KB apart (SBO); K step k = keys 16k..16k+15.
          const uint64_t bd = sdesc_sw128(sv + k * 4096, 1024, 2048);
          mma_bf16_ss(tmem + kColO, ad, bd, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit(o_done);
        mma_commit(&kv_empty[j & 1]);
      };
      for (int kt = 0; kt < n_kv && ok; ++kt) {
        const int st = kt & 1;
        ok = mbar_wait(&k_full[st], (kt >> 1) & 1, abort_flag);
        if (ok && kt >= kStages) ok = mbar_wait(&s_free[st], ((kt >> 1) & 1) ^ 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sk = sbase + kOffK + st * kTileBytes;
#pragma unroll
        for (int k = 0; k < kHeadDim / 16; ++k) {
          const uint64_t ad = sdesc_sw128(sq + (k >> 2) * kHalfBytes + (k & 3) * 32, 16, 1024);
          // K tile as the K-major B: dim half k/4 at +1 KB, 8-key groups 2 KB apart.
          const uint64_t bd = sdesc_sw128(sk + (k >> 2) * 1024 + (k & 3) * 32, 16, 2048);
          mma_bf16_ss(tmem + st * kN, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[st]);
        if (kt > 0) issue_pv(kt - 1);
      }
      if (ok) issue_pv(n_kv - 1);
      // Drain: every MMA issued above completes before TMEM is released.
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
    __syncwarp();
  } else {
    // =============================== softmax ================================
    const int r = tid;  // tile row = TMEM lane
    const bool row_valid = r < rows;
    const int key_lim = row_valid ? pos0 + r : 0;  // keys <= key_lim are visible
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t sp_row = sbase + kOffP + r * 128;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int kt = 0; kt < n_kv; ++kt) {
      const int sb = kt & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (kt >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kN];
#pragma unroll
      for (int c4 = 0; c4 < kN / 32; ++c4) {
        float t[32];
        tmem_ld32(lane_addr + sb * kN + c4 * 32, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c4 * 32 + i] = t[i];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[sb]);

      const int kbase = kt * kN;
      float mx = -INFINITY;
      if (kbase + kN - 1 > key_lim) {
#pragma unroll
        for (int c = 0; c < kN; ++c) {
          s[c] = (kbase + c <= key_lim) ? s[c] * a.scale_log2 : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kN; ++c) {
          s[c] *= a.scale_log2;
          mx = fmaxf(mx, s[c]);
        }
      }
      // PV(kt-1) must be done before O is rescaled or P is overwritten.
      if (kt > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(o_done, (kt - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const float m_new = fmaxf(m_run, mx);
      if (kt == 0) {
        m_run = m_new;
      } else {
        const bool rescale = m_new > m_run + kLazyRescale;
        if (__any_sync(0xffffffffu, rescale)) {
          const float alpha = rescale ? exp2f(m_run - m_new) : 1.f;
#pragma unroll
          for (int c4 = 0; c4 < kHeadDim / 32; ++c4) {
            float o[32];
            tmem_ld32(lane_addr + kColO + c4 * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(lane_addr + kColO + c4 * 32, o);
          }
          if (rescale) {
            l_run *= alpha;
            m_run = m_new;
          }
        }
      }
      float sum = 0.f;
#pragma unroll
      for (int cc = 0; cc < kN / 8; ++cc) {
        float p[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          p[i] = exp2f(s[cc * 8 + i] - m_run);
          sum += p[i];
        }
        const int half = cc >> 3, chunk = cc & 7;
        sts128(sp_row + half * kHalfBytes + ((chunk ^ (r & 7)) << 4), pack_bf16x2_rn(p[0], p[1]),
               pack_bf16x2_rn(p[2], p[3]), pack_bf16x2_rn(p[4], p[5]),
               pack_bf16x2_rn(p[6], p[7]));
      }
      l_run += sum;
      if (kbase + kN > L) {
        // The tile reaches past the context: zero V rows of keys >= L.
        if (!__all_sync(0xffffffffu, mbar_wait(&v_full[sb], (kt >> 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        if (kbase + r >= L) {
          const uint32_t vtile = sbase + kOffV + sb * kTileBytes + (r >> 4) * kCacheTileBytes;
#pragma unroll
          for (int c = 0; c < 16; ++c) sts128(vtile + tile_chunk_offset(r & 15, c), 0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(o_done, (n_kv - 1) & 1, abort_flag))) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(a.out) +
                            ((row0 + r) * a.num_heads + h) * kHeadDim;
#pragma unroll
      for (int c4 = 0; c4 < kHeadDim / 32; ++c4) {
        float o[32];
        tmem_ld32(lane_addr + kColO + c4 * 32, o);
        if (row_valid) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16x2_rn(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv);
            v.y = pack_bf16x2_rn(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv);
            v.z = pack_bf16x2_rn(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv);
            v.w = pack_bf16x2_rn(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv);
            *reinterpret_cast<uint4*>(orow + c4 * 32 + q * 8) = v;
          }
        }
      }
    } else {
      ok = false;
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
  using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                     const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                     const cuuint32_t*, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion,
                                     CUtensorMapFloatOOBfill);
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) != cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
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

cudaError_t launch_varlen_prefill(const PrefillArgs& a, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, int /*num_sms*/, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(varlen_prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap qmap;
  if (!encode_q_map(&qmap, a.q, a.q_row_stride, a.total_q, a.num_heads))
    return cudaErrorInvalidValue;
  const int mtiles = (a.max_q_len + kM - 1) / kM;
  if (a.num_seqs > 65535 || a.num_heads > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(mtiles, a.num_heads, a.num_seqs);
  varlen_prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(qmap, kmap, vmap, a);
  return cudaPeekAtLastError();
}

}  // namespace qattn
