// qattn_paged_decode_noalloc: the paged decode for callers that cannot
// allocate device memory.
//
// Who needs this: code that runs where a cudaMalloc is not allowed or not
// safe -- inside a region being captured into a CUDA graph by someone else's
// framework, in a real-time serving loop whose memory pool was sized once at
// start-up, or in a host that hands this library only the tensors it
// computes on.  Such a caller cannot provide the split-KV workspace that
// qattn_paged_decode asks for.  This entry point uses a fixed scratch array
// that lives in this library's device image instead.
//
// The scratch: kScratchBytes (32 MiB) of device memory in a file-scope
// __device__ array.  Every GPU that loads the library holds it until the
// process exits.  It has room for the split-KV partial results of, for
// example, 64 sequences of up to 4096 tokens with 28 query heads, or 8
// sequences of 32768 tokens; qattn_paged_decode_workspace_size() tells the
// need of any other shape, and a need above kScratchBytes is refused with
// QATTN_ERR_WORKSPACE before anything is launched.
//
// In host code the array's name is only a stand-in, not a device address:
// the device address is looked up with cudaGetSymbolAddress on the first
// call made while a device is current, and again whenever the calling
// thread's current context on that device is not the one the address was
// taken in (after cudaDeviceReset, or from a context the caller created
// itself); each context has its own copy of the array.  The lookup may load
// the library's device code, so make the first call in a context outside
// any stream capture.
//
// All calls share the one array and it keeps whatever the last call left
// in it.  Nothing in it has to start at zero: the decode kernels write every
// scratch word before they read it.  Two calls whose kernels overlap on the
// GPU (different streams, no ordering between them) race on the array and
// give wrong results; order such calls, or use qattn_paged_decode with a
// workspace of your own.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace qattn {
namespace {

constexpr size_t kScratchBytes = 32ull << 20;

static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent from the driver, looked up once (nullptr if unavailable).
CtxGetCurrentFn ctx_get_current() {
  static std::once_flag once;
  static CtxGetCurrentFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_decode_scratch in the current context of the current
// device (looked up again when that context changes), or nullptr if the
// lookup failed.
void* scratch_on_current_device() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  static CUcontext owner[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (get == nullptr || get(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (ctx != nullptr && addr[dev] != nullptr && owner[dev] == ctx) return addr[dev];
  // (the lookup also makes the device's primary context current if no
  // context was)
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
  if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return nullptr;
  addr[dev] = p;
  owner[dev] = ctx;
  return p;
}

}  // namespace
}  // namespace qattn

extern "C" int qattn_paged_decode_noalloc(void* out, const void* q, int64_t q_row_stride,
                                          const void* k_cache, const void* v_cache,
                                          int32_t num_blocks, const int32_t* block_tables,
                                          int32_t max_blocks_per_seq,
                                          const int32_t* context_lens, int32_t num_seqs,
                                          int32_t max_context_len, qattn_dims dims,
                                          int32_t* err_word, void* stream) {
  if (num_seqs < 0 || max_context_len < 0) return QATTN_ERR_INVALID_ARG;
  if (num_seqs == 0) return QATTN_OK;
  const size_t need = qattn_paged_decode_workspace_size(num_seqs, max_context_len, dims);
  if (need == 0) {
    // Shape rejected by the size computation: let the regular entry point
    // report why, without a workspace.
    return qattn_paged_decode(out, q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                              max_blocks_per_seq, context_lens, num_seqs, max_context_len, dims,
                              nullptr, 0, err_word, stream);
  }
  if (need > qattn::kScratchBytes) return QATTN_ERR_WORKSPACE;
  void* scratch = qattn::scratch_on_current_device();
  if (scratch == nullptr) return QATTN_ERR_CUDA;
  return qattn_paged_decode(out, q, q_row_stride, k_cache, v_cache, num_blocks, block_tables,
                            max_blocks_per_seq, context_lens, num_seqs, max_context_len, dims,
                            scratch, qattn::kScratchBytes, err_word, stream);
}
