// Tensor-core SimHash of bf16 prefill keys (tcgen05): placeholder until the
// tcgen05 kernel lands; reports that it did not run so the caller hashes on CUDA cores.
#include "mp_internal.h"

namespace mp {

cudaError_t launch_hash_keys_tc(const Geometry&, const void*, int, const TablesPtrs&, cudaStream_t,
                                bool* used) {
  *used = false;
  return cudaSuccess;
}

}  // namespace mp
