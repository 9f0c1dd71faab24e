// C-ABI layer of the qattn library: argument validation, launch sizing,
// tensor-map encoding and status strings.  No device memory is allocated
// here; every buffer belongs to the caller.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "internal.h"

using namespace qattn;

#ifdef QATTN_TRACE
// The copy probe of the tracing build (copy_probe.cu).
namespace qattn {
int copy_stream_max_stages(bool kv_fp8);
cudaError_t launch_copy_stream(const CUtensorMap& kmap, const CUtensorMap& vmap, bool kv_fp8,
                               const int32_t* tiles, int32_t num_tiles, int32_t num_kv_heads,
                               int32_t num_blocks, int32_t block_size, int32_t stages,
                               int32_t* err_word, int num_sms, cudaStream_t stream);
}  // namespace qattn
#endif

namespace {

constexpr int kVersion = 100;  // 0.1.0

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const qattn_dims& d) {
  if (d.num_heads <= 0 || d.num_kv_heads <= 0 || d.head_dim <= 0 || d.block_size <= 0)
    return QATTN_ERR_INVALID_ARG;
  if (d.head_dim != kHeadDim) return QATTN_ERR_UNSUPPORTED;
  if (d.block_size != 16 && d.block_size != 32 && d.block_size != 64) return QATTN_ERR_UNSUPPORTED;
  if (d.num_heads % d.num_kv_heads != 0) return QATTN_ERR_UNSUPPORTED;
  if (d.num_heads / d.num_kv_heads > 8 || d.num_heads > 128) return QATTN_ERR_UNSUPPORTED;
  if (!(d.scale == d.scale) || isinf(d.scale)) return QATTN_ERR_INVALID_ARG;
  return QATTN_OK;
}

float scale_of(const qattn_dims& d) {
  return d.scale > 0.f ? d.scale : 1.0f / sqrtf(static_cast<float>(d.head_dim));
}

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------ device info --

int num_sms_current() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lk(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    cached[dev] = n;
  }
  return cached[dev];
}

// ------------------------------------------------------------ side stream --
//
// The shared-prefix calls run their prefix pass on a stream of the
// library's own, beside the decode of the sequences' own tokens on the
// caller's stream (the two kernels take disjoint sets of SMs), forked from
// and joined back into the caller's stream with two events: one stream and
// two events per device, created on first use.  The lock is held from the
// fork to the join, so that calls from several host threads do not
// interleave their records.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;

SideStream* side_stream_current() {  // with g_side_mu held
  static SideStream per_dev[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream& ss = per_dev[dev];
  if (ss.stream == nullptr) {
    if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess ||
        cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking) != cudaSuccess)
      return nullptr;
  }
  return &ss;
}

// ------------------------------------------------------------ tensor maps --

}  // namespace

EncodeTiledFn qattn::encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

cudaError_t qattn::set_max_dynamic_smem(const void* kernel, int bytes) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;  // (kernel, device)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& d : done)
    if (d.first == kernel && d.second == dev) return cudaSuccess;
  if (bytes > 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  // Every kernel of the library asks for the largest shared-memory carve-out,
  // so that an SM need not change its L1 / shared split between the decode
  // and prefill kernels (which need almost all of it) and the kernels around
  // them.
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess) done.emplace_back(kernel, dev);
  return e;
}

namespace {

// The paged cache [num_blocks][Hkv][BS][128] bf16 (BS = block size) seen as a
// 4-D tensor (64 columns, 8 rows, 2 column halves, num_blocks * Hkv * BS / 8
// row groups): element (c, r, h, m) is row 8m + r, column 64h + c of the 2-D
// [num_blocks * Hkv * BS][128] view.  A box of (64, 8, 2, BS / 8) is one whole
// (block, kv head) tile -- BS * 256 bytes in one copy -- and lands in shared
// memory as [row group][column half][8 rows][128 B] with the 128-byte
// swizzle: each 8-row x 128-byte atom sits on its own 1 KB, the two halves of
// a row group 1 KB apart and consecutive row groups 2 KB apart, which is the
// K-major (and, for V, MN-major) operand layout the tensor-core kernels
// describe with an 8-row-group stride of 2 KB, and what the CUDA-core kernel
// addresses directly.  Blocks placed one after another in shared memory thus
// form one uniform run of row groups whatever BS is.
bool encode_cache_map(CUtensorMap* map, const void* cache, int32_t num_blocks,
                      int32_t num_kv_heads, int32_t block_size) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {
      64, 8, 2, static_cast<cuuint64_t>(num_blocks) * num_kv_heads * (block_size / 8)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(kHeadDim) * 2,  // next row
                                 128,                                     // next half
                                 static_cast<cuuint64_t>(kHeadDim) * 2 * 8};  // next group
  const cuuint32_t box[4] = {64, 8, 2, static_cast<cuuint32_t>(block_size / 8)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An FP8 (e4m3) cache [num_blocks][Hkv][BS][128] uint8 seen as a 2-D tensor
// of 128-byte token rows; a box of (128, BS) is one (block, kv head) tile,
// landing as BS rows of 128 B with the 128-byte swizzle (row r's 16-byte
// chunk c at c ^ (r & 7)).
bool encode_cache_map_fp8(CUtensorMap* map, const void* cache, int32_t num_blocks,
                          int32_t num_kv_heads, int32_t block_size) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {
      static_cast<cuuint64_t>(kHeadDim),
      static_cast<cuuint64_t>(num_blocks) * num_kv_heads * block_size};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kHeadDim)};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kHeadDim),
                             static_cast<cuuint32_t>(block_size)};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A small cache of encoded maps: the same caches are used call after call.
struct MapEntry {
  const void* ptr;
  int32_t num_blocks;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t fp8;
  CUtensorMap map;
};

bool cached_cache_map(CUtensorMap* out, const void* cache, int32_t num_blocks,
                      int32_t num_kv_heads, int32_t block_size, int32_t fp8 = 0) {
  static std::mutex mu;
  static MapEntry entries[16];
  static int used = 0, next = 0;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < used; ++i) {
    if (entries[i].ptr == cache && entries[i].num_blocks == num_blocks &&
        entries[i].num_kv_heads == num_kv_heads && entries[i].block_size == block_size &&
        entries[i].fp8 == fp8) {
      *out = entries[i].map;
      return true;
    }
  }
  MapEntry e;
  e.ptr = cache;
  e.num_blocks = num_blocks;
  e.num_kv_heads = num_kv_heads;
  e.block_size = block_size;
  e.fp8 = fp8;
  if (!(fp8 ? encode_cache_map_fp8(&e.map, cache, num_blocks, num_kv_heads, block_size)
            : encode_cache_map(&e.map, cache, num_blocks, num_kv_heads, block_size)))
    return false;
  entries[next] = e;
  next = (next + 1) % 16;
  if (used < 16) ++used;
  *out = e.map;
  return true;
}

// The query rows seen as a 3-D tensor [rows][num_heads][128]; a box is one
// row's G consecutive heads x 64 columns (half a head), 128-byte swizzled:
// the tensor-core decode loads a KV head's query group with two boxes.
bool encode_q_group_map(CUtensorMap* map, const void* q, int64_t q_row_stride, int32_t rows,
                        int32_t num_heads, int32_t group, int32_t rows_per_box = 1) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim),
                              static_cast<cuuint64_t>(num_heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                                 static_cast<cuuint64_t>(q_row_stride) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group),
                             static_cast<cuuint32_t>(rows_per_box)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int check_cache(const void* k_cache, const void* v_cache, int32_t num_blocks,
                const qattn_dims& d) {
  if (k_cache == nullptr || v_cache == nullptr || num_blocks <= 0) return QATTN_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return QATTN_ERR_INVALID_ARG;
  // TMA coordinates are 32-bit.
  if (static_cast<int64_t>(num_blocks) * d.num_kv_heads * d.block_size >= (1ll << 31))
    return QATTN_ERR_UNSUPPORTED;
  return QATTN_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? QATTN_OK : QATTN_ERR_CUDA; }

// Testing hook state (qattn_debug_decode_faults): the decode kernel's wait
// limit (0: the default) and the K copy its first CTA skips (-1: none).
std::atomic<long long> g_debug_wait_ns{0};
std::atomic<int> g_debug_skip_k{-1};

constexpr uint64_t kMinDrainNs = 10000000ull;  // 10 ms

// A cache scale: finite, positive and normal (its reciprocal stays finite).
bool valid_scale(float s) { return s == s && !isinf(s) && s >= 1.17549435e-38f; }

}  // namespace

extern "C" {

const char* qattn_status_string(int status) {
  switch (status) {
    case QATTN_OK: return "ok";
    case QATTN_ERR_INVALID_ARG: return "invalid argument";
    case QATTN_ERR_UNSUPPORTED: return "unsupported shape";
    case QATTN_ERR_CUDA: return "CUDA error";
    case QATTN_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int qattn_version(void) { return kVersion; }

int qattn_rope_table_build(float* host_cos_sin, int32_t max_pos, int32_t head_dim,
                           double theta) {
  if (host_cos_sin == nullptr || max_pos <= 0 || head_dim <= 0 || (head_dim & 1) ||
      !(theta > 0.0))
    return QATTN_ERR_INVALID_ARG;
  const int32_t half = head_dim / 2;
  for (int32_t i = 0; i < half; ++i) {
    const double inv_freq = pow(theta, -(2.0 * i) / head_dim);
    for (int32_t pos = 0; pos < max_pos; ++pos) {
      const double ang = static_cast<double>(pos) * inv_freq;
      host_cos_sin[static_cast<int64_t>(pos) * head_dim + i] = static_cast<float>(cos(ang));
      host_cos_sin[static_cast<int64_t>(pos) * head_dim + half + i] =
          static_cast<float>(sin(ang));
    }
  }
  return QATTN_OK;
}

int qattn_rope_table_build_scaled(float* host_cos_sin, int32_t max_pos, int32_t head_dim,
                                  double theta, int32_t scaling, double factor,
                                  int32_t original_max_position) {
  if (host_cos_sin == nullptr || max_pos <= 0 || head_dim <= 2 || (head_dim & 1) ||
      !(theta > 0.0))
    return QATTN_ERR_INVALID_ARG;
  if (scaling < QATTN_ROPE_SCALING_NONE || scaling > QATTN_ROPE_SCALING_DYNAMIC)
    return QATTN_ERR_INVALID_ARG;
  if (scaling != QATTN_ROPE_SCALING_NONE && !(factor >= 1.0)) return QATTN_ERR_INVALID_ARG;
  if (scaling == QATTN_ROPE_SCALING_DYNAMIC && original_max_position <= 0)
    return QATTN_ERR_INVALID_ARG;
  const int32_t half = head_dim / 2;
  double base = theta;
  if (scaling == QATTN_ROPE_SCALING_DYNAMIC && max_pos > original_max_position) {
    const double grow = factor * static_cast<double>(max_pos) / original_max_position -
                        (factor - 1.0);
    base = theta * pow(grow, static_cast<double>(head_dim) / (head_dim - 2));
  }
  for (int32_t i = 0; i < half; ++i) {
    const double inv_freq = pow(base, -(2.0 * i) / head_dim);
    for (int32_t pos = 0; pos < max_pos; ++pos) {
      const double p =
          scaling == QATTN_ROPE_SCALING_LINEAR ? static_cast<double>(pos) / factor : pos;
      const double ang = p * inv_freq;
      host_cos_sin[static_cast<int64_t>(pos) * head_dim + i] = static_cast<float>(cos(ang));
      host_cos_sin[static_cast<int64_t>(pos) * head_dim + half + i] =
          static_cast<float>(sin(ang));
    }
  }
  return QATTN_OK;
}

// The append into a bf16 cache (kv_fp8 = 0) or an e4m3 cache.
static int append_common(void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                         const void* v, int64_t v_row_stride, const int32_t* positions,
                         const int32_t* slot_mapping, int32_t num_tokens, void* k_cache,
                         void* v_cache, int32_t num_blocks, const float* cos_sin,
                         int32_t max_pos, const void* qkv_bias, const void* q_norm_weight,
                         const void* k_norm_weight, float norm_eps, int kv_fp8, float k_scale,
                         float v_scale, qattn_dims dims, int32_t* err_word, void* stream) {
  int st = check_dims(dims);
  if (st != QATTN_OK) return st;
  if (num_tokens < 0) return QATTN_ERR_INVALID_ARG;
  if (num_tokens == 0) return QATTN_OK;
  if (q == nullptr || k == nullptr || v == nullptr || positions == nullptr ||
      slot_mapping == nullptr || cos_sin == nullptr || max_pos <= 0)
    return QATTN_ERR_INVALID_ARG;
  st = check_cache(k_cache, v_cache, num_blocks, dims);
  if (st != QATTN_OK) return st;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(cos_sin))
    return QATTN_ERR_INVALID_ARG;
  if (q_row_stride % 8 || k_row_stride % 8 || v_row_stride % 8) return QATTN_ERR_INVALID_ARG;
  if (!aligned16(qkv_bias) || !aligned16(q_norm_weight) || !aligned16(k_norm_weight))
    return QATTN_ERR_INVALID_ARG;
  if ((q_norm_weight != nullptr || k_norm_weight != nullptr) &&
      !(norm_eps >= 0.0f && norm_eps < 1.0f))
    return QATTN_ERR_INVALID_ARG;
  if (q_row_stride < static_cast<int64_t>(dims.num_heads) * kHeadDim ||
      k_row_stride < static_cast<int64_t>(dims.num_kv_heads) * kHeadDim ||
      v_row_stride < static_cast<int64_t>(dims.num_kv_heads) * kHeadDim)
    return QATTN_ERR_INVALID_ARG;
  RopeAppendArgs a;
  a.q = q;
  a.q_row_stride = q_row_stride;
  a.k = k;
  a.k_row_stride = k_row_stride;
  a.v = v;
  a.v_row_stride = v_row_stride;
  a.positions = positions;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.num_blocks = num_blocks;
  a.cos_sin = cos_sin;
  a.max_pos = max_pos;
  a.num_heads = dims.num_heads;
  a.num_kv_heads = dims.num_kv_heads;
  a.block_size = dims.block_size;
  a.err_word = err_word;
  a.bias = qkv_bias;
  a.q_norm_w = q_norm_weight;
  a.k_norm_w = k_norm_weight;
  a.norm_eps = norm_eps;
  a.kv_fp8 = kv_fp8;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return cuda_status(launch_rope_append(a, static_cast<cudaStream_t>(stream)));
}

int qattn_rope_cache_append_ex(void* q, int64_t q_row_stride, const void* k,
                               int64_t k_row_stride, const void* v, int64_t v_row_stride,
                               const int32_t* positions, const int32_t* slot_mapping,
                               int32_t num_tokens, void* k_cache, void* v_cache,
                               int32_t num_blocks, const float* cos_sin, int32_t max_pos,
                               const void* qkv_bias, const void* q_norm_weight,
                               const void* k_norm_weight, float norm_eps, qattn_dims dims,
                               int32_t* err_word, void* stream) {
  return append_common(q, q_row_stride, k, k_row_stride, v, v_row_stride, positions,
                       slot_mapping, num_tokens, k_cache, v_cache, num_blocks, cos_sin, max_pos,
                       qkv_bias, q_norm_weight, k_norm_weight, norm_eps, 0, 1.0f, 1.0f, dims,
                       err_word, stream);
}

int qattn_rope_cache_append_fp8(void* q, int64_t q_row_stride, const void* k,
                                int64_t k_row_stride, const void* v, int64_t v_row_stride,
                                const int32_t* positions, const int32_t* slot_mapping,
                                int32_t num_tokens, void* k_cache, void* v_cache,
                                int32_t num_blocks, const float* cos_sin, int32_t max_pos,
                                const void* qkv_bias, const void* q_norm_weight,
                                const void* k_norm_weight, float norm_eps, float k_scale,
                                float v_scale, qattn_dims dims, int32_t* err_word,
                                void* stream) {
  if (!valid_scale(k_scale) || !valid_scale(v_scale)) return QATTN_ERR_INVALID_ARG;
  return append_common(q, q_row_stride, k, k_row_stride, v, v_row_stride, positions,
                       slot_mapping, num_tokens, k_cache, v_cache, num_blocks, cos_sin, max_pos,
                       qkv_bias, q_norm_weight, k_norm_weight, norm_eps, 1, k_scale, v_scale,
                       dims, err_word, stream);
}

int qattn_rope_cache_append(void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride,
                            const void* v, int64_t v_row_stride, const int32_t* positions,
                            const int32_t* slot_mapping, int32_t num_tokens, void* k_cache,
                            void* v_cache, int32_t num_blocks, const float* cos_sin,
                            int32_t max_pos, qattn_dims dims, int32_t* err_word, void* stream) {
  return qattn_rope_cache_append_ex(q, q_row_stride, k, k_row_stride, v, v_row_stride,
                                    positions, slot_mapping, num_tokens, k_cache, v_cache,
                                    num_blocks, cos_sin, max_pos, nullptr, nullptr, nullptr,
                                    0.0f, dims, err_word, stream);
}

#ifdef QATTN_TRACE
// Tracing build only (include/qattn_trace.h).
int qattn_trace_dims(int32_t* decode_ctas, int32_t* decode_slots, int32_t* merge_ctas) {
  if (decode_ctas == nullptr || decode_slots == nullptr || merge_ctas == nullptr)
    return QATTN_ERR_INVALID_ARG;
  *decode_ctas = kTraceCtas;
  *decode_slots = kTraceSlots;
  *merge_ctas = kTraceMergeCtas;
  return QATTN_OK;
}

int qattn_trace_clear(void) {
  if (clear_decode_trace() != cudaSuccess || clear_merge_trace() != cudaSuccess)
    return QATTN_ERR_CUDA;
  return QATTN_OK;
}

int qattn_trace_copy_stream(const void* k_cache, const void* v_cache, int32_t num_blocks,
                            qattn_dims dims, int32_t kv_fp8, const int32_t* tiles,
                            int32_t num_tiles, int32_t stages, int32_t* err_word, void* stream) {
  int st = check_dims(dims);
  if (st != QATTN_OK) return st;
  if (tiles == nullptr || num_tiles < 0 || num_blocks <= 0 || (kv_fp8 != 0 && kv_fp8 != 1) ||
      stages < 2 || stages > copy_stream_max_stages(kv_fp8 != 0))
    return QATTN_ERR_INVALID_ARG;
  st = check_cache(k_cache, v_cache, num_blocks, dims);
  if (st != QATTN_OK) return st;
  if (num_tiles == 0) return QATTN_OK;
  CUtensorMap kmap, vmap;
  if (!cached_cache_map(&kmap, k_cache, num_blocks, dims.num_kv_heads, dims.block_size, kv_fp8) ||
      !cached_cache_map(&vmap, v_cache, num_blocks, dims.num_kv_heads, dims.block_size, kv_fp8))
    return QATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return QATTN_ERR_CUDA;
  return cuda_status(launch_copy_stream(kmap, vmap, kv_fp8 != 0, tiles, num_tiles,
                                        dims.num_kv_heads, num_blocks, dims.block_size, stages,
                                        err_word, sms, static_cast<cudaStream_t>(stream)));
}

int qattn_trace_read(uint64_t* decode_host, uint64_t* merge_host) {
  if (decode_host == nullptr || merge_host == nullptr) return QATTN_ERR_INVALID_ARG;
  if (read_decode_trace(reinterpret_cast<unsigned long long*>(decode_host),
                        static_cast<size_t>(kTraceCtas) * kTraceSlots) != cudaSuccess ||
      read_merge_trace(reinterpret_cast<unsigned long long*>(merge_host),
                       static_cast<size_t>(kTraceMergeCtas) * 4) != cudaSuccess)
    return QATTN_ERR_CUDA;
  return QATTN_OK;
}
#endif

int qattn_debug_decode_faults(int64_t wait_limit_ns, int32_t skip_k_copy) {
  if (wait_limit_ns < 0 || (wait_limit_ns > 0 && wait_limit_ns < 1000) ||
      wait_limit_ns > static_cast<int64_t>(kWaitTimeoutNs) || skip_k_copy < -1)
    return QATTN_ERR_INVALID_ARG;
  g_debug_wait_ns.store(wait_limit_ns);
  g_debug_skip_k.store(skip_k_copy);
  return QATTN_OK;
}

size_t qattn_paged_decode_workspace_size(int32_t num_seqs, int32_t max_context_len,
                                         qattn_dims dims) {
  if (check_dims(dims) != QATTN_OK || num_seqs < 0 || max_context_len < 0) return 0;
  return decode_workspace_bytes(num_seqs, max_context_len, dims.num_kv_heads,
                                dims.num_heads / dims.num_kv_heads);
}

namespace {

int decode_common(void* out, const void* q, int64_t q_row_stride, int32_t q_rows,
                  const int32_t* cu_seqlens_q,
                  const void* k_cache, const void* v_cache, int32_t num_blocks,
                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                  const int32_t* context_lens, int32_t num_seqs, int32_t max_context_len,
                  const qattn_dims& dims, void* workspace, size_t workspace_bytes,
                  int32_t* err_word, cudaStream_t stream, const CUtensorMap& kmap,
                  const CUtensorMap& vmap, int num_sms, int32_t prefix_len = 0,
                  int32_t part_base = 0, int32_t extra_parts = 0, int32_t kv_fp8 = 0,
                  float k_scale = 1.0f, float v_scale = 1.0f,
                  cudaEvent_t merge_after = nullptr) {
  const size_t need = decode_workspace_bytes(num_seqs, max_context_len, dims.num_kv_heads,
                                             dims.num_heads / dims.num_kv_heads, extra_parts);
  if (workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return QATTN_ERR_WORKSPACE;
  DecodeArgs a;
  a.out = out;
  a.q = q;
  a.q_row_stride = q_row_stride;
  a.cu_seqlens_q = cu_seqlens_q;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_blocks = num_blocks;
  a.max_context_len = max_context_len;
  a.num_heads = dims.num_heads;
  a.num_kv_heads = dims.num_kv_heads;
  a.block_size = dims.block_size;
  a.scale_log2 = scale_of(dims) * kLog2e * (kv_fp8 ? k_scale : 1.0f);
  a.kv_fp8 = kv_fp8;
  a.v_scale = kv_fp8 ? v_scale : 1.0f;
  a.err_word = err_word;
  a.ws = carve_decode_workspace(workspace, num_seqs, max_context_len, dims.num_kv_heads,
                                dims.num_heads / dims.num_kv_heads, extra_parts);
  a.prefix_len = prefix_len;
  a.part_base = part_base;
  const long long w = g_debug_wait_ns.load();
  a.wait_ns = w > 0 ? static_cast<uint64_t>(w) : kWaitTimeoutNs;
  a.drain_ns = a.wait_ns < kMinDrainNs ? kMinDrainNs
                                        : (a.wait_ns > kWaitTimeoutNs ? kWaitTimeoutNs : a.wait_ns);
  a.debug_skip_k = g_debug_skip_k.load();
  const int group = dims.num_heads / dims.num_kv_heads;
  CUtensorMap qmap;
  if (!encode_q_group_map(&qmap, q, q_row_stride, q_rows, dims.num_heads, group))
    return QATTN_ERR_CUDA;
  return cuda_status(launch_paged_decode_tc(a, kmap, vmap, qmap, num_sms, stream, merge_after));
}

// The shared-prefix pass beside the decode: the prefix in splits of at most
// 16 KV tiles (an item then takes ~20 us), on at most an eighth of the SMs;
// the decode of the sequences' own tokens keeps the rest.
void prefix_plan(int sms, int num_kv_heads, int row_tiles, int prefix_tiles, int* splits,
                 int* grid) {
  int sp = (prefix_tiles + 15) / 16;
  if (sp > kMaxPrefixSplits) sp = kMaxPrefixSplits;
  if (sp < 1) sp = 1;
  const int64_t items = static_cast<int64_t>(num_kv_heads) * row_tiles * sp;
  int g = sms / 8 > 1 ? sms / 8 : 1;
  if (items < g) g = static_cast<int>(items);
  *splits = sp;
  *grid = g;
}

int check_attention_args(void* out, const void* q, int64_t q_row_stride, const void* k_cache,
                         const void* v_cache, int32_t num_blocks, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                         int32_t max_context_len, const qattn_dims& dims) {
  if (out == nullptr || q == nullptr || block_tables == nullptr || context_lens == nullptr)
    return QATTN_ERR_INVALID_ARG;
  if (max_blocks_per_seq <= 0 || max_context_len <= 0) return QATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || q_row_stride % 8 ||
      q_row_stride < static_cast<int64_t>(dims.num_heads) * kHeadDim)
    return QATTN_ERR_INVALID_ARG;
  return check_cache(k_cache, v_cache, num_blocks, dims);
}

}  // namespace

int qattn_paged_decode(void* out, const void* q, int64_t q_row_stride, const void* k_cache,
                       const void* v_cache, int32_t num_blocks, const int32_t* block_tables,
                       int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                       int32_t max_context_len, qattn_dims dims, void* workspace,
                       size_t workspace_bytes, int32_t* err_word, void* stream) {
  int st = check_dims(dims);
  if (st != QATTN_OK) return st;
  if (num_seqs < 0) return QATTN_ERR_INVALID_ARG;
  if (num_seqs == 0) return QATTN_OK;
  st = check_attention_args(out, q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                            max_blocks_per_seq, context_lens, max_context_len, dims);
  if (st != QATTN_OK) return st;
  CUtensorMap kmap, vmap;
  if (!cached_cache_map(&kmap, k_cache, num_blocks, dims.num_kv_heads, dims.block_size) ||
      !cached_cache_map(&vmap, v_cache, num_blocks, dims.num_kv_heads, dims.block_size))
    return QATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return QATTN_ERR_CUDA;
  return decode_common(out, q, q_row_stride, num_seqs, nullptr, k_cache, v_cache, num_blocks,
                       block_tables,
                       max_blocks_per_seq, context_lens, num_seqs, max_context_len, dims,
                       workspace, workspace_bytes, err_word, static_cast<cudaStream_t>(stream),
                       kmap, vmap, sms);
}

int qattn_paged_decode_fp8(void* out, const void* q, int64_t q_row_stride, const void* k_cache,
                           const void* v_cache, int32_t num_blocks, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t num_seqs, int32_t max_context_len, float k_scale,
                           float v_scale, qattn_dims dims, void* workspace,
                           size_t workspace_bytes, int32_t* err_word, void* stream) {
  int st = check_dims(dims);
  if (st != QATTN_OK) return st;
  if (num_seqs < 0 || !valid_scale(k_scale) || !valid_scale(v_scale))
    return QATTN_ERR_INVALID_ARG;
  if (num_seqs == 0) return QATTN_OK;
  st = check_attention_args(out, q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                            max_blocks_per_seq, context_lens, max_context_len, dims);
  if (st != QATTN_OK) return st;
  CUtensorMap kmap, vmap;
  if (!cached_cache_map(&kmap, k_cache, num_blocks, dims.num_kv_heads, dims.block_size, 1) ||
      !cached_cache_map(&vmap, v_cache, num_blocks, dims.num_kv_heads, dims.block_size, 1))
    return QATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return QATTN_ERR_CUDA;
  return decode_common(out, q, q_row_stride, num_seqs, nullptr, k_cache, v_cache, num_blocks,
                       block_tables, max_blocks_per_seq, context_lens, num_seqs,
                       max_context_len, dims, workspace, workspace_bytes, err_word,
                       static_cast<cudaStream_t>(stream), kmap, vmap, sms, 0, 0, 0, 1, k_scale,
                       v_scale);
}

size_t qattn_paged_decode_shared_prefix_workspace_size(int32_t num_seqs,
                                                       int32_t max_context_len,
                                                       qattn_dims dims) {
  if (check_dims(dims) != QATTN_OK || num_seqs < 0 || max_context_len < 0) return 0;
  return decode_workspace_bytes(num_seqs, max_context_len, dims.num_kv_heads,
                                dims.num_heads / dims.num_kv_heads, kMaxPrefixSplits);
}

int qattn_paged_decode_shared_prefix(void* out, const void* q, int64_t q_row_stride,
                                     const void* k_cache, const void* v_cache,
                                     int32_t num_blocks, const int32_t* block_tables,
                                     int32_t max_blocks_per_seq, const int32_t* context_lens,
                                     int32_t num_seqs, int32_t max_context_len,
                                     int32_t shared_prefix_len, qattn_dims dims,
                                     void* workspace, size_t workspace_bytes, int32_t* err_word,
                                     void* stream) {
  int st = check_dims(dims);
  if (st != QATTN_OK) return st;
  if (num_seqs < 0) return QATTN_ERR_INVALID_ARG;
  if (num_seqs == 0) return QATTN_OK;
  st = check_attention_args(out, q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                            max_blocks_per_seq, context_lens, max_context_len, dims);
  if (st != QATTN_OK) return st;
  if (shared_prefix_len < 0 || shared_prefix_len % dims.block_size != 0 ||
      shared_prefix_len >= max_context_len ||
      shared_prefix_len > static_cast<int64_t>(max_blocks_per_seq) * dims.block_size)
    return QATTN_ERR_INVALID_ARG;
  const size_t need =
      qattn_paged_decode_shared_prefix_workspace_size(num_seqs, max_context_len, dims);
  if (workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return QATTN_ERR_WORKSPACE;
  CUtensorMap kmap, vmap;
  if (!cached_cache_map(&kmap, k_cache, num_blocks, dims.num_kv_heads, dims.block_size) ||
      !cached_cache_map(&vmap, v_cache, num_blocks, dims.num_kv_heads, dims.block_size))
    return QATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return QATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (shared_prefix_len == 0)
    return decode_common(out, q, q_row_stride, num_seqs, nullptr, k_cache, v_cache, num_blocks,
                         block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         max_context_len, dims, workspace, workspace_bytes, err_word, s, kmap,
                         vmap, sms, 0, 0, kMaxPrefixSplits);
  // Pass 1: the prefix, once per kv head for all sequences (tensor cores),
  // as parts 0 .. splits - 1 of every unit, on the side stream; pass 2
  // beside it: each sequence's own tokens (the decode kernel, parts from
  // `splits` on) on the other SMs; then, once both are done, the merge of
  // all parts.
  const int group = dims.num_heads / dims.num_kv_heads;
  const int rows_per_tile = 128 / group;
  const int row_tiles = (num_seqs + rows_per_tile - 1) / rows_per_tile;
  const int prefix_tiles = (shared_prefix_len + 127) / 128;
  int splits = 1, pgrid = 1;
  prefix_plan(sms, dims.num_kv_heads, row_tiles, prefix_tiles, &splits, &pgrid);
  CUtensorMap qmap;
  if (!encode_q_group_map(&qmap, q, q_row_stride, num_seqs, dims.num_heads, group,
                          rows_per_tile))
    return QATTN_ERR_CUDA;
  PrefillArgs p{};
  p.q = q;
  p.q_row_stride = q_row_stride;
  p.context_lens = context_lens;
  p.block_tables = block_tables;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_blocks = num_blocks;
  p.total_q = num_seqs;
  p.max_q_len = 1;
  p.max_context_len = max_context_len;
  p.num_heads = dims.num_heads;
  p.num_kv_heads = dims.num_kv_heads;
  p.block_size = dims.block_size;
  p.scale_log2 = scale_of(dims) * kLog2e;
  p.out_scale = 1.0f;
  p.err_word = err_word;
  p.prefix_len = shared_prefix_len;
  p.prefix_splits = splits;
  p.ws = carve_decode_workspace(workspace, num_seqs, max_context_len, dims.num_kv_heads, group,
                                kMaxPrefixSplits);
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStream* ss = side_stream_current();
  if (ss == nullptr || cudaEventRecord(ss->fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(ss->stream, ss->fork, 0) != cudaSuccess)
    return QATTN_ERR_CUDA;
  st = cuda_status(launch_shared_prefix(p, qmap, kmap, vmap, pgrid, ss->stream));
  if (st != QATTN_OK) return st;
  if (cudaEventRecord(ss->join, ss->stream) != cudaSuccess) return QATTN_ERR_CUDA;
  return decode_common(out, q, q_row_stride, num_seqs, nullptr, k_cache, v_cache, num_blocks,
                       block_tables, max_blocks_per_seq, context_lens, num_seqs,
                       max_context_len, dims, workspace, workspace_bytes, err_word, s, kmap,
                       vmap, sms - pgrid, shared_prefix_len, splits, kMaxPrefixSplits, 0, 1.0f,
                       1.0f, ss->join);
}

size_t qattn_varlen_prefill_workspace_size(int32_t num_seqs, int32_t max_context_len,
                                           qattn_dims dims) {
  return qattn_paged_decode_workspace_size(num_seqs, max_context_len, dims);
}

int qattn_varlen_prefill(void* out, const void* q, int64_t q_row_stride,
                         const int32_t* cu_seqlens_q, int32_t num_seqs, int32_t total_q,
                         int32_t max_q_len, const void* k_cache, const void* v_cache,
                         int32_t num_blocks, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                         int32_t max_context_len, qattn_dims dims, void* workspace,
                         size_t workspace_bytes, int32_t* err_word, void* stream) {
  int st = check_dims(dims);
  if (st != QATTN_OK) return st;
  if (num_seqs < 0 || total_q < 0 || max_q_len < 0) return QATTN_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0) return QATTN_OK;
  if (cu_seqlens_q == nullptr || max_q_len == 0) return QATTN_ERR_INVALID_ARG;
  if ((max_q_len + 127) / 128 > kPrefillMaxPairs) return QATTN_ERR_UNSUPPORTED;
  st = check_attention_args(out, q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                            max_blocks_per_seq, context_lens, max_context_len, dims);
  if (st != QATTN_OK) return st;
  CUtensorMap kmap, vmap;
  if (!cached_cache_map(&kmap, k_cache, num_blocks, dims.num_kv_heads, dims.block_size) ||
      !cached_cache_map(&vmap, v_cache, num_blocks, dims.num_kv_heads, dims.block_size))
    return QATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return QATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Decode rows (one query) of the batch.
  st = decode_common(out, q, q_row_stride, total_q, cu_seqlens_q, k_cache, v_cache, num_blocks,
                     block_tables, max_blocks_per_seq, context_lens, num_seqs, max_context_len,
                     dims, workspace, workspace_bytes, err_word, s, kmap, vmap, sms);
  if (st != QATTN_OK || max_q_len < 2) return st;
  // Prefill rows (two or more queries): tensor-core kernel.
  PrefillArgs p;
  p.out = out;
  p.q = q;
  p.q_row_stride = q_row_stride;
  p.cu_seqlens_q = cu_seqlens_q;
  p.context_lens = context_lens;
  p.block_tables = block_tables;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_blocks = num_blocks;
  p.total_q = total_q;
  p.max_q_len = max_q_len;
  p.max_context_len = max_context_len;
  p.num_heads = dims.num_heads;
  p.num_kv_heads = dims.num_kv_heads;
  p.block_size = dims.block_size;
  p.scale_log2 = scale_of(dims) * kLog2e;
  p.out_scale = 1.0f;
  p.err_word = err_word;
  p.prefix_len = 0;
  p.prefix_splits = 0;
  p.ws = DecodeWorkspace{};
  const cudaError_t e = launch_varlen_prefill(p, kmap, vmap, sms, s);
  return e == cudaErrorNotSupported ? QATTN_ERR_UNSUPPORTED : cuda_status(e);
}

}  // extern "C"

namespace {

// FP8 prefill scratch behind the decode workspace: the scratch block table
// [num_seqs][bps] and the bf16 copies of the prefill sequences' blocks.
struct Fp8Scratch {
  size_t decode_bytes, table_off, k_off, v_off, total;
  int32_t bps;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

Fp8Scratch fp8_scratch_layout(int32_t num_seqs, int32_t num_prefill_seqs,
                              int32_t max_context_len, const qattn_dims& d) {
  Fp8Scratch f;
  f.decode_bytes = align256(decode_workspace_bytes(num_seqs, max_context_len, d.num_kv_heads,
                                                   d.num_heads / d.num_kv_heads));
  f.bps = (max_context_len + d.block_size - 1) / d.block_size;
  const size_t block_bytes = static_cast<size_t>(d.num_kv_heads) * d.block_size * kHeadDim * 2;
  const size_t blocks = static_cast<size_t>(num_prefill_seqs) * f.bps;
  f.table_off = f.decode_bytes;
  f.k_off = f.table_off + align256(static_cast<size_t>(num_seqs) * f.bps * 4);
  f.v_off = f.k_off + align256(blocks * block_bytes);
  f.total = f.v_off + align256(blocks * block_bytes);
  return f;
}

}  // namespace

extern "C" {

size_t qattn_varlen_prefill_fp8_workspace_size(int32_t num_seqs, int32_t num_prefill_seqs,
                                               int32_t max_context_len, qattn_dims dims) {
  if (check_dims(dims) != QATTN_OK || num_seqs < 0 || max_context_len < 0 ||
      num_prefill_seqs < 0 || num_prefill_seqs > num_seqs)
    return 0;
  return fp8_scratch_layout(num_seqs, num_prefill_seqs, max_context_len, dims).total;
}

int qattn_varlen_prefill_fp8(void* out, const void* q, int64_t q_row_stride,
                             const int32_t* cu_seqlens_q, int32_t num_seqs, int32_t total_q,
                             int32_t max_q_len, const void* k_cache, const void* v_cache,
                             int32_t num_blocks, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                             int32_t max_context_len, int32_t num_prefill_seqs, float k_scale,
                             float v_scale, qattn_dims dims, void* workspace,
                             size_t workspace_bytes, int32_t* err_word, void* stream) {
  int st = check_dims(dims);
  if (st != QATTN_OK) return st;
  if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || !valid_scale(k_scale) ||
      !valid_scale(v_scale) || num_prefill_seqs < 0 || num_prefill_seqs > num_seqs)
    return QATTN_ERR_INVALID_ARG;
  if (num_seqs == 0 || total_q == 0) return QATTN_OK;
  if (cu_seqlens_q == nullptr || max_q_len == 0) return QATTN_ERR_INVALID_ARG;
  if ((max_q_len + 127) / 128 > kPrefillMaxPairs) return QATTN_ERR_UNSUPPORTED;
  st = check_attention_args(out, q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                            max_blocks_per_seq, context_lens, max_context_len, dims);
  if (st != QATTN_OK) return st;
  const Fp8Scratch f = fp8_scratch_layout(num_seqs, num_prefill_seqs, max_context_len, dims);
  if (workspace == nullptr || workspace_bytes < f.total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return QATTN_ERR_WORKSPACE;
  CUtensorMap kmap, vmap;
  if (!cached_cache_map(&kmap, k_cache, num_blocks, dims.num_kv_heads, dims.block_size, 1) ||
      !cached_cache_map(&vmap, v_cache, num_blocks, dims.num_kv_heads, dims.block_size, 1))
    return QATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return QATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Decode rows (one query): the FP8 decode kernel reads the codes.
  st = decode_common(out, q, q_row_stride, total_q, cu_seqlens_q, k_cache, v_cache, num_blocks,
                     block_tables, max_blocks_per_seq, context_lens, num_seqs, max_context_len,
                     dims, workspace, f.decode_bytes, err_word, s, kmap, vmap, sms, 0, 0, 0, 1,
                     k_scale, v_scale);
  if (st != QATTN_OK || max_q_len < 2 || num_prefill_seqs == 0) return st;
  // Prefill rows: bf16 copies of the code values, then the bf16 prefill.
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Fp8GatherArgs g;
  g.k_codes = static_cast<const uint8_t*>(k_cache);
  g.v_codes = static_cast<const uint8_t*>(v_cache);
  g.num_blocks = num_blocks;
  g.block_tables = block_tables;
  g.max_blocks_per_seq = max_blocks_per_seq;
  g.context_lens = context_lens;
  g.cu_seqlens_q = cu_seqlens_q;
  g.num_seqs = num_seqs;
  g.num_kv_heads = dims.num_kv_heads;
  g.block_size = dims.block_size;
  g.blocks_per_seq = f.bps;
  g.capacity = num_prefill_seqs;
  g.k_out = reinterpret_cast<__nv_bfloat16*>(ws + f.k_off);
  g.v_out = reinterpret_cast<__nv_bfloat16*>(ws + f.v_off);
  g.table_out = reinterpret_cast<int32_t*>(ws + f.table_off);
  g.err_word = err_word;
  cudaError_t e = launch_fp8_gather(g, s);
  if (e != cudaSuccess) return cuda_status(e);
  const int32_t scratch_blocks = num_prefill_seqs * f.bps;
  CUtensorMap skmap, svmap;
  if (!cached_cache_map(&skmap, g.k_out, scratch_blocks, dims.num_kv_heads, dims.block_size) ||
      !cached_cache_map(&svmap, g.v_out, scratch_blocks, dims.num_kv_heads, dims.block_size))
    return QATTN_ERR_CUDA;
  PrefillArgs p;
  p.out = out;
  p.q = q;
  p.q_row_stride = q_row_stride;
  p.cu_seqlens_q = cu_seqlens_q;
  p.context_lens = context_lens;
  p.block_tables = g.table_out;
  p.max_blocks_per_seq = f.bps;
  p.num_seqs = num_seqs;
  p.num_blocks = scratch_blocks;
  p.total_q = total_q;
  p.max_q_len = max_q_len;
  p.max_context_len = max_context_len;
  p.num_heads = dims.num_heads;
  p.num_kv_heads = dims.num_kv_heads;
  p.block_size = dims.block_size;
  p.scale_log2 = scale_of(dims) * kLog2e * k_scale;
  p.out_scale = v_scale;
  p.err_word = err_word;
  p.prefix_len = 0;
  p.prefix_splits = 0;
  p.ws = DecodeWorkspace{};
  e = launch_varlen_prefill(p, skmap, svmap, sms, s);
  return e == cudaErrorNotSupported ? QATTN_ERR_UNSUPPORTED : cuda_status(e);
}

size_t qattn_paged_decode_shared_prefix_fp8_workspace_size(int32_t num_seqs,
                                                           int32_t max_context_len,
                                                           int32_t shared_prefix_len,
                                                           qattn_dims dims) {
  if (check_dims(dims) != QATTN_OK || num_seqs < 0 || max_context_len < 0 ||
      shared_prefix_len < 0 || shared_prefix_len % dims.block_size != 0)
    return 0;
  const int32_t pb = shared_prefix_len / dims.block_size;
  const size_t block_bytes =
      static_cast<size_t>(dims.num_kv_heads) * dims.block_size * kHeadDim * 2;
  return align256(qattn_paged_decode_shared_prefix_workspace_size(num_seqs, max_context_len,
                                                                  dims)) +
         align256(static_cast<size_t>(num_seqs) * pb * 4) + 2 * align256(pb * block_bytes);
}

int qattn_paged_decode_shared_prefix_fp8(void* out, const void* q, int64_t q_row_stride,
                                         const void* k_cache, const void* v_cache,
                                         int32_t num_blocks, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t num_seqs,
                                         int32_t max_context_len, int32_t shared_prefix_len,
                                         float k_scale, float v_scale, qattn_dims dims,
                                         void* workspace, size_t workspace_bytes,
                                         int32_t* err_word, void* stream) {
  int st = check_dims(dims);
  if (st != QATTN_OK) return st;
  if (num_seqs < 0 || !valid_scale(k_scale) || !valid_scale(v_scale))
    return QATTN_ERR_INVALID_ARG;
  if (num_seqs == 0) return QATTN_OK;
  st = check_attention_args(out, q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                            max_blocks_per_seq, context_lens, max_context_len, dims);
  if (st != QATTN_OK) return st;
  if (shared_prefix_len < 0 || shared_prefix_len % dims.block_size != 0 ||
      shared_prefix_len >= max_context_len ||
      shared_prefix_len > static_cast<int64_t>(max_blocks_per_seq) * dims.block_size)
    return QATTN_ERR_INVALID_ARG;
  const size_t need = qattn_paged_decode_shared_prefix_fp8_workspace_size(
      num_seqs, max_context_len, shared_prefix_len, dims);
  if (workspace == nullptr || workspace_bytes < need ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return QATTN_ERR_WORKSPACE;
  CUtensorMap kmap, vmap;
  if (!cached_cache_map(&kmap, k_cache, num_blocks, dims.num_kv_heads, dims.block_size, 1) ||
      !cached_cache_map(&vmap, v_cache, num_blocks, dims.num_kv_heads, dims.block_size, 1))
    return QATTN_ERR_CUDA;
  const int sms = num_sms_current();
  if (sms <= 0) return QATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t decode_bytes =
      align256(qattn_paged_decode_shared_prefix_workspace_size(num_seqs, max_context_len, dims));
  if (shared_prefix_len == 0)
    return decode_common(out, q, q_row_stride, num_seqs, nullptr, k_cache, v_cache, num_blocks,
                         block_tables, max_blocks_per_seq, context_lens, num_seqs,
                         max_context_len, dims, workspace, decode_bytes, err_word, s, kmap,
                         vmap, sms, 0, 0, kMaxPrefixSplits, 1, k_scale, v_scale);
  // On the side stream: the prefix as bf16 values of its codes (exact), then
  // the prefix pass on the copy with the scales folded in; beside them, each
  // sequence's own tokens from the codes; then the merge of all parts.
  const int32_t pb = shared_prefix_len / dims.block_size;
  const size_t block_bytes =
      static_cast<size_t>(dims.num_kv_heads) * dims.block_size * kHeadDim * 2;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Fp8GatherArgs g{};
  g.k_codes = static_cast<const uint8_t*>(k_cache);
  g.v_codes = static_cast<const uint8_t*>(v_cache);
  g.num_blocks = num_blocks;
  g.block_tables = block_tables;
  g.max_blocks_per_seq = max_blocks_per_seq;
  g.num_seqs = num_seqs;
  g.num_kv_heads = dims.num_kv_heads;
  g.block_size = dims.block_size;
  g.blocks_per_seq = pb;
  g.table_out = reinterpret_cast<int32_t*>(ws + decode_bytes);
  const size_t k_off = decode_bytes + align256(static_cast<size_t>(num_seqs) * pb * 4);
  g.k_out = reinterpret_cast<__nv_bfloat16*>(ws + k_off);
  g.v_out = reinterpret_cast<__nv_bfloat16*>(ws + k_off + align256(pb * block_bytes));
  g.err_word = err_word;
  CUtensorMap skmap, svmap;
  if (!cached_cache_map(&skmap, g.k_out, pb, dims.num_kv_heads, dims.block_size) ||
      !cached_cache_map(&svmap, g.v_out, pb, dims.num_kv_heads, dims.block_size))
    return QATTN_ERR_CUDA;
  const int group = dims.num_heads / dims.num_kv_heads;
  const int rows_per_tile = 128 / group;
  const int row_tiles = (num_seqs + rows_per_tile - 1) / rows_per_tile;
  const int prefix_tiles = (shared_prefix_len + 127) / 128;
  int splits = 1, pgrid = 1;
  prefix_plan(sms, dims.num_kv_heads, row_tiles, prefix_tiles, &splits, &pgrid);
  CUtensorMap qmap;
  if (!encode_q_group_map(&qmap, q, q_row_stride, num_seqs, dims.num_heads, group,
                          rows_per_tile))
    return QATTN_ERR_CUDA;
  PrefillArgs p{};
  p.q = q;
  p.q_row_stride = q_row_stride;
  p.context_lens = context_lens;
  p.block_tables = g.table_out;
  p.max_blocks_per_seq = pb;
  p.num_seqs = num_seqs;
  p.num_blocks = pb;
  p.total_q = num_seqs;
  p.max_q_len = 1;
  p.max_context_len = max_context_len;
  p.num_heads = dims.num_heads;
  p.num_kv_heads = dims.num_kv_heads;
  p.block_size = dims.block_size;
  p.scale_log2 = scale_of(dims) * kLog2e * k_scale;
  p.out_scale = v_scale;
  p.err_word = err_word;
  p.prefix_len = shared_prefix_len;
  p.prefix_splits = splits;
  p.ws = carve_decode_workspace(workspace, num_seqs, max_context_len, dims.num_kv_heads, group,
                                kMaxPrefixSplits);
  std::lock_guard<std::mutex> lk(g_side_mu);
  SideStream* ss = side_stream_current();
  if (ss == nullptr || cudaEventRecord(ss->fork, s) != cudaSuccess ||
      cudaStreamWaitEvent(ss->stream, ss->fork, 0) != cudaSuccess)
    return QATTN_ERR_CUDA;
  cudaError_t e = launch_fp8_prefix_gather(g, ss->stream);
  if (e != cudaSuccess) return cuda_status(e);
  st = cuda_status(launch_shared_prefix(p, qmap, skmap, svmap, pgrid, ss->stream));
  if (st != QATTN_OK) return st;
  if (cudaEventRecord(ss->join, ss->stream) != cudaSuccess) return QATTN_ERR_CUDA;
  return decode_common(out, q, q_row_stride, num_seqs, nullptr, k_cache, v_cache, num_blocks,
                       block_tables, max_blocks_per_seq, context_lens, num_seqs,
                       max_context_len, dims, workspace, decode_bytes, err_word, s, kmap, vmap,
                       sms - pgrid, shared_prefix_len, splits, kMaxPrefixSplits, 1, k_scale,
                       v_scale, ss->join);
}

}  // extern "C"
