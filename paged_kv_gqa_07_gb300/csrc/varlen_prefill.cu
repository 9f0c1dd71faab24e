// Kernel K3: causal varlen / chunked prefill on tcgen05 tensor cores.
// (Placeholder until the tensor-core kernel lands: reports "not supported".)
#include "common.cuh"
#include "internal.h"

namespace qattn {

cudaError_t launch_varlen_prefill(const PrefillArgs&, const CUtensorMap&, const CUtensorMap&,
                                  int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace qattn
