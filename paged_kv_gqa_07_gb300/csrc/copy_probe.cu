// Tracing build only: the decode's cache copies with nothing consuming them.
//
// One warp per SM walks an even share of a tile list in the decode's order
// and issues, per 128-token tile, the same TMA boxes the decode kernel's
// producer issues (one per cache block of the tile, K and V, through the
// same tensor maps) into a ring of `stages` slots; a slot is reused as soon
// as its copies have landed.  The time of a pass is the copy time of the
// decode's access pattern alone -- the ceiling the decode's stream phase can
// reach -- measured on the same tiles (paged blocks at random places).
#ifdef QATTN_TRACE
#include "common.cuh"
#include "internal.h"

namespace qattn {
namespace {

template <bool kFp8>
__global__ void __launch_bounds__(32, 1)
    copy_stream_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const int32_t* tiles,
                       int32_t num_tiles, int32_t num_kv_heads, int32_t num_blocks,
                       int32_t block_size, int32_t stages, int32_t* err_word) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kTileBytes = kTcTileTokens * kHeadDim * (kFp8 ? 1 : 2);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + stages * 2 * kTileBytes);
  const int lane = threadIdx.x;
  if (lane == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncwarp();
  const uint32_t blk_bytes = static_cast<uint32_t>(block_size) * kHeadDim * (kFp8 ? 1 : 2);
  const int bpt = kTcTileTokens / block_size;
  const int c0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * num_tiles / gridDim.x);
  const int c1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * num_tiles / gridDim.x);
  bool ok = true;
  for (int n = c0; n < c1 && ok; ++n) {
    const int i = n - c0, s = i % stages;
    // slot s last held tile i - stages: its copies must have landed
    if (i >= stages && lane == 0) ok = mbar_wait_drain(&bars[s], ((i / stages) - 1) & 1);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    const int g = tiles[static_cast<int64_t>(n) * 9];
    int id = lane < bpt ? tiles[static_cast<int64_t>(n) * 9 + 1 + lane] : -1;
    if (id >= num_blocks || g < 0 || g >= num_kv_heads) {
      set_err(err_word, QATTN_DEVERR_BLOCK);
      id = -1;
    }
    const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, id >= 0));
    if (lane == 0) mbar_arrive_expect_tx(&bars[s], 2 * nvalid * blk_bytes);
    __syncwarp();
    if (id >= 0) {
      uint8_t* dk = smem + s * 2 * kTileBytes + lane * blk_bytes;
      uint8_t* dv = dk + kTileBytes;
      if constexpr (kFp8) {
        tma_load_2d(dk, &kmap, 0, (id * num_kv_heads + g) * block_size, &bars[s]);
        tma_load_2d(dv, &vmap, 0, (id * num_kv_heads + g) * block_size, &bars[s]);
      } else {
        tma_load_cache_tile(dk, &kmap, id * num_kv_heads + g, block_size / 8, &bars[s]);
        tma_load_cache_tile(dv, &vmap, id * num_kv_heads + g, block_size / 8, &bars[s]);
      }
    }
  }
  // the copies still in flight land before the CTA exits
  if (lane == 0) {
    const int cnt = c1 - c0;
    for (int i = cnt > stages ? cnt - stages : 0; i < cnt; ++i)
      if (!mbar_wait_drain(&bars[i % stages], (i / stages) & 1)) ok = false;
    if (!ok) set_err(err_word, QATTN_DEVERR_TIMEOUT);
  }
}

}  // namespace

int copy_stream_max_stages(bool kv_fp8) {
  const int tile = kTcTileTokens * kHeadDim * (kv_fp8 ? 1 : 2);
  return (227 * 1024 - 1024) / (2 * tile + 8);
}

cudaError_t launch_copy_stream(const CUtensorMap& kmap, const CUtensorMap& vmap, bool kv_fp8,
                               const int32_t* tiles, int32_t num_tiles, int32_t num_kv_heads,
                               int32_t num_blocks, int32_t block_size, int32_t stages,
                               int32_t* err_word, int num_sms, cudaStream_t stream) {
  const int tile = kTcTileTokens * kHeadDim * (kv_fp8 ? 1 : 2);
  const size_t smem = static_cast<size_t>(stages) * (2 * tile + 8) + 1024;
  const void* fn = kv_fp8 ? reinterpret_cast<const void*>(copy_stream_kernel<true>)
                          : reinterpret_cast<const void*>(copy_stream_kernel<false>);
  // the limit is set once per device: set it for the deepest ring
  const int most = copy_stream_max_stages(kv_fp8) * (2 * tile + 8) + 1024;
  cudaError_t e = set_max_dynamic_smem(fn, most);
  if (e != cudaSuccess) return e;
  if (kv_fp8)
    copy_stream_kernel<true><<<num_sms, 32, smem, stream>>>(
        kmap, vmap, tiles, num_tiles, num_kv_heads, num_blocks, block_size, stages, err_word);
  else
    copy_stream_kernel<false><<<num_sms, 32, smem, stream>>>(
        kmap, vmap, tiles, num_tiles, num_kv_heads, num_blocks, block_size, stages, err_word);
  return cudaPeekAtLastError();
}

}  // namespace qattn
#endif  // QATTN_TRACE
